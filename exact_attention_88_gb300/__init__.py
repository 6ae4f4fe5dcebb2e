"""Python binding of libfa (exact attention for GB300 / sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libfa.so.  The C functions keep their names (`fa_fwd`, `fa_bwd`,
...); each takes device pointers (ints or torch CUDA tensors) and raises
`FaError` on a non-OK status.  `forward` / `backward` are conveniences that
allocate the outputs with torch and call the same C functions; they accept
[B, H, N, d] views of any layout whose last dimension is contiguous (for
example a [B, N, H, d] buffer transposed to [B, H, N, d]) and pass each
tensor's strides to the *_ex calls, so nothing is copied; they also take
dropout (probability, seed, offset).

Importing this package fails loudly if libfa.so has not been built
(`python -c "import __graft_entry__ as g; g.build()"`): there is no fallback.
"""
import ctypes
import os

__all__ = [
    "FaError", "FaMask", "FaLayout", "FaLayouts", "FaDropout", "FaBias", "FaOptions", "layout_of",
    "bias_of",
    "make_layouts", "make_options", "fa_fwd_ex", "fa_bwd_ex", "fa_fwd_fp32_ex", "fa_bwd_fp32_ex",
    "fa_bwd_preprocess_ex", "fa_bwd_dkdv_ex", "fa_bwd_dq_ex",
    "lib", "fa_fwd", "fa_bwd", "fa_bwd_workspace_size",
    "fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq", "fa_fwd_fp32", "fa_bwd_fp32",
    "fa_bwd_noalloc", "NOALLOC_SCRATCH_BYTES", "fa_status_string", "fa_get_device_status", "fa_debug_wait_timeout",
    "make_mask", "forward", "backward", "LIB_PATH",
    "fa_block_mask_order", "fa_block_mask_order_len", "block_mask_order",
    "FA_MASK_NONE", "FA_MASK_KEY_PADDING", "FA_MASK_BLOCK_SPARSE", "STATUS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

FA_MASK_NONE, FA_MASK_KEY_PADDING, FA_MASK_BLOCK_SPARSE = 0, 1, 2
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_ALIGNMENT",
          4: "FA_ERR_WORKSPACE", 5: "FA_ERR_CUDA", 6: "FA_ERR_TIMEOUT"}


class FaError(RuntimeError):
    def __init__(self, code, where, detail=None):
        self.code = code
        msg = "%s returned %s" % (where, STATUS.get(code, code))
        if detail:
            msg += " (%s)" % detail
        super().__init__(msg)


class FaMask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("kv_len", ctypes.c_void_p),
                ("block_mask", ctypes.c_void_p), ("block_size", ctypes.c_int),
                ("tile_order", ctypes.c_void_p)]


class FaLayout(ctypes.Structure):
    """Element strides of one [B, H, N, d] tensor (fa_layout)."""
    _fields_ = [("batch", ctypes.c_int64), ("head", ctypes.c_int64), ("row", ctypes.c_int64)]


_LAYOUT_NAMES = ("q", "k", "v", "o", "dO", "dq", "dk", "dv")


class FaLayouts(ctypes.Structure):
    """Layouts of the tensors of one call (fa_layouts)."""
    _fields_ = [(n, FaLayout) for n in _LAYOUT_NAMES]


class FaDropout(ctypes.Structure):
    """Dropout of a call (fa_dropout): probability, generator seed, offset."""
    _fields_ = [("p", ctypes.c_float), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint32)]


class FaBias(ctypes.Structure):
    """Additive score bias (fa_bias): fp32 device pointer and element strides."""
    _fields_ = [("ptr", ctypes.c_void_p), ("batch", ctypes.c_int64), ("head", ctypes.c_int64),
                ("row", ctypes.c_int64)]


class FaOptions(ctypes.Structure):
    """Options of the *_ex calls (fa_options)."""
    _fields_ = [("layouts", ctypes.POINTER(FaLayouts)), ("dropout", ctypes.POINTER(FaDropout)),
                ("bias", ctypes.POINTER(FaBias))]


if not os.path.exists(LIB_PATH):
    raise ImportError("libfa.so is not built (expected at %s); run "
                      "__graft_entry__.build() first" % LIB_PATH)
lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
_mp = ctypes.POINTER(FaMask)
_op = ctypes.POINTER(FaOptions)

_SIGS = {
    "fa_fwd": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _f, _i, _mp, _p],
    "fa_fwd_fp32": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _f, _i, _mp, _p],
    "fa_bwd_workspace_size": [_i, _i, _i, _i],
    "fa_bwd": [_p] * 10 + [_sz, _i, _i, _i, _i, _f, _i, _mp, _p],
    "fa_bwd_fp32": [_p] * 10 + [_sz, _i, _i, _i, _i, _f, _i, _mp, _p],
    "fa_bwd_preprocess": [_p, _p, _p, _i, _i, _i, _i, _p],
    "fa_bwd_dkdv": [_p] * 8 + [_i, _i, _i, _i, _f, _i, _mp, _p],
    "fa_bwd_dq": [_p] * 7 + [_i, _i, _i, _i, _f, _i, _mp, _p],
    "fa_status_string": [_i],
    "fa_get_device_status": [_p, ctypes.POINTER(ctypes.c_int)],
    "fa_debug_wait_timeout": [ctypes.c_uint, _p],
    "fa_bwd_noalloc": [_p] * 9 + [_i, _i, _i, _i, _f, _i, _mp, _p],
    "fa_last_cuda_error": [],
    "fa_fwd_ex": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _f, _i, _mp, _op, _p],
    "fa_fwd_fp32_ex": [_p, _p, _p, _p, _p, _i, _i, _i, _i, _f, _i, _mp, _op, _p],
    "fa_bwd_ex": [_p] * 10 + [_sz, _i, _i, _i, _i, _f, _i, _mp, _op, _p],
    "fa_bwd_fp32_ex": [_p] * 10 + [_sz, _i, _i, _i, _i, _f, _i, _mp, _op, _p],
    "fa_bwd_preprocess_ex": [_p, _p, _p, _i, _i, _i, _i, _op, _p],
    "fa_bwd_dkdv_ex": [_p] * 8 + [_i, _i, _i, _i, _f, _i, _mp, _op, _p],
    "fa_bwd_dq_ex": [_p] * 7 + [_i, _i, _i, _i, _f, _i, _mp, _op, _p],
    "fa_block_mask_order_len": [_i],
    "fa_block_mask_order": [_p, _i, _i, _p, _p],
}
for _name, _args in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
lib.fa_status_string.restype = ctypes.c_char_p
lib.fa_last_cuda_error.restype = ctypes.c_char_p


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _check(code, where):
    if code != 0:
        detail = lib.fa_last_cuda_error().decode() if code == 5 else None
        raise FaError(code, where, detail)


def make_mask(kv_len=None, block_mask=None, block_size=128, tile_order=None):
    """A pointer to an fa_mask for key padding (kv_len) or a block-sparse tile
    mask (device tensors), or None for no mask.  tile_order: the block mask's
    work order (block_mask_order), or None for the default order."""
    if kv_len is not None and block_mask is not None:
        raise ValueError("one mask kind at a time")
    if tile_order is not None and block_mask is None:
        raise ValueError("tile_order belongs to a block mask")
    if kv_len is not None:
        return ctypes.pointer(FaMask(FA_MASK_KEY_PADDING, _ptr(kv_len), None, block_size, None))
    if block_mask is not None:
        return ctypes.pointer(FaMask(FA_MASK_BLOCK_SPARSE, None, _ptr(block_mask), block_size,
                                     _ptr(tile_order)))
    return None


def layout_of(t):
    """FaLayout of a 4-D [B, H, N, d] tensor whose last dimension is contiguous."""
    if t.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    if t.stride(3) != 1 and t.shape[3] > 1:
        raise ValueError("the d elements of a row must be contiguous (stride(3) == 1)")
    return FaLayout(t.stride(0), t.stride(1), t.stride(2))


def make_layouts(**tensors):
    """An FaLayouts holding layout_of(t) for each named tensor (names: q, k,
    v, o, dO, dq, dk, dv); entries not given stay zero, which the calls that
    read them reject."""
    unknown = set(tensors) - set(_LAYOUT_NAMES)
    if unknown:
        raise ValueError("unknown tensor names: %s" % sorted(unknown))
    ls = FaLayouts()
    for name, t in tensors.items():
        setattr(ls, name, layout_of(t))
    return ls


def bias_of(t):
    """FaBias of a CUDA fp32 tensor broadcastable to [B, H, N, N] (4-D, last
    dimension contiguous); dimensions of size 1 are broadcast (stride 0)."""
    if t.dim() != 4:
        raise ValueError("the bias must be 4-D: [B or 1, H or 1, N, N]")
    if t.stride(3) != 1:
        raise ValueError("the bias columns must be contiguous")
    st = [0 if t.shape[i] == 1 else t.stride(i) for i in range(3)]
    return FaBias(t.data_ptr(), st[0], st[1], st[2])


def make_options(layouts=None, dropout_p=0.0, seed=0, offset=0, bias=None):
    """A pointer to an FaOptions: `layouts` an FaLayouts (or None: dense),
    dropout with probability dropout_p (0: none), generator seed and offset,
    `bias` an FaBias (or None).  The pointer keeps its members alive."""
    opt = FaOptions()
    keep = []
    if bias is not None:
        keep.append(bias)
        opt.bias = ctypes.pointer(bias)
    if layouts is not None:
        keep.append(layouts)
        opt.layouts = ctypes.pointer(layouts)
    if dropout_p:
        dr = FaDropout(dropout_p, seed, offset)
        keep.append(dr)
        opt.dropout = ctypes.pointer(dr)
    ptr = ctypes.pointer(opt)
    ptr._keep = keep
    return ptr


def fa_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, mask=None, options=None,
              stream=None):
    _check(lib.fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                         int(causal), mask, options, _stream(stream)), "fa_fwd_ex")


def fa_fwd_fp32_ex(q, k, v, o, lse, B, H, N, d, scale, causal, mask=None, options=None,
                   stream=None):
    _check(lib.fa_fwd_fp32_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                              int(causal), mask, options, _stream(stream)), "fa_fwd_fp32_ex")


def fa_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale,
              causal, mask=None, options=None, stream=None):
    _check(lib.fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                         _ptr(dk), _ptr(dv), _ptr(workspace), workspace_bytes, B, H, N, d, scale,
                         int(causal), mask, options, _stream(stream)), "fa_bwd_ex")


def fa_bwd_fp32_ex(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d,
                   scale, causal, mask=None, options=None, stream=None):
    _check(lib.fa_bwd_fp32_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), _ptr(workspace), workspace_bytes, B, H, N, d,
                              scale, int(causal), mask, options, _stream(stream)),
           "fa_bwd_fp32_ex")


def fa_bwd_preprocess_ex(o, dO, D, B, H, N, d, options=None, stream=None):
    _check(lib.fa_bwd_preprocess_ex(_ptr(o), _ptr(dO), _ptr(D), B, H, N, d, options,
                                    _stream(stream)), "fa_bwd_preprocess_ex")


def fa_bwd_dkdv_ex(q, k, v, dO, lse, D, dk, dv, B, H, N, d, scale, causal, mask=None,
                   options=None, stream=None):
    _check(lib.fa_bwd_dkdv_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D), _ptr(dk),
                              _ptr(dv), B, H, N, d, scale, int(causal), mask, options,
                              _stream(stream)), "fa_bwd_dkdv_ex")


def fa_bwd_dq_ex(q, k, v, dO, lse, D, dq, B, H, N, d, scale, causal, mask=None, options=None,
                 stream=None):
    _check(lib.fa_bwd_dq_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D), _ptr(dq),
                            B, H, N, d, scale, int(causal), mask, options, _stream(stream)),
           "fa_bwd_dq_ex")


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, mask=None, stream=None):
    _check(lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                      int(causal), mask, _stream(stream)), "fa_fwd")


def fa_fwd_fp32(q, k, v, o, lse, B, H, N, d, scale, causal, mask=None, stream=None):
    _check(lib.fa_fwd_fp32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                           int(causal), mask, _stream(stream)), "fa_fwd_fp32")


def fa_bwd_workspace_size(B, H, N, d):
    return lib.fa_bwd_workspace_size(B, H, N, d)


def fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale,
           causal, mask=None, stream=None):
    _check(lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                      _ptr(dk), _ptr(dv), _ptr(workspace), workspace_bytes, B, H, N, d, scale,
                      int(causal), mask, _stream(stream)), "fa_bwd")


def fa_bwd_fp32(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale,
                causal, mask=None, stream=None):
    _check(lib.fa_bwd_fp32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(workspace), workspace_bytes, B, H, N, d,
                           scale, int(causal), mask, _stream(stream)), "fa_bwd_fp32")


def fa_bwd_preprocess(o, dO, D, B, H, N, d, stream=None):
    _check(lib.fa_bwd_preprocess(_ptr(o), _ptr(dO), _ptr(D), B, H, N, d, _stream(stream)),
           "fa_bwd_preprocess")


def fa_bwd_dkdv(q, k, v, dO, lse, D, dk, dv, B, H, N, d, scale, causal, mask=None, stream=None):
    _check(lib.fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D), _ptr(dk),
                           _ptr(dv), B, H, N, d, scale, int(causal), mask, _stream(stream)),
           "fa_bwd_dkdv")


def fa_bwd_dq(q, k, v, dO, lse, D, dq, B, H, N, d, scale, causal, mask=None, stream=None):
    _check(lib.fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D), _ptr(dq),
                         B, H, N, d, scale, int(causal), mask, _stream(stream)), "fa_bwd_dq")


NOALLOC_SCRATCH_BYTES = 32 << 20   # FA_NOALLOC_SCRATCH_BYTES


def fa_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, mask=None,
                   stream=None):
    """fa_bwd without a workspace argument, for callers that cannot allocate
    device memory: the library's fixed scratch array is used instead (sizes
    whose workspace exceeds NOALLOC_SCRATCH_BYTES raise FaError)."""
    _check(lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, H, N, d, scale, int(causal), mask,
                              _stream(stream)), "fa_bwd_noalloc")


def fa_block_mask_order_len(T):
    return lib.fa_block_mask_order_len(T)


def fa_block_mask_order(block_mask, T, causal, tile_order, stream=None):
    _check(lib.fa_block_mask_order(_ptr(block_mask), T, int(causal), _ptr(tile_order),
                                   _stream(stream)), "fa_block_mask_order")


def block_mask_order(block_mask, causal=False, stream=None):
    """The work order of a [T, T] uint8 CUDA block mask (an int32 CUDA
    tensor of fa_block_mask_order_len(T) entries), for make_mask(tile_order=)."""
    import torch
    T = int(block_mask.shape[0])
    n = fa_block_mask_order_len(T)
    if n == 0 or block_mask.numel() != T * T:
        raise ValueError("expected a [T, T] block mask with 1 <= T <= 4096")
    out = torch.empty(n, dtype=torch.int32, device=block_mask.device)
    fa_block_mask_order(block_mask, T, causal, out, stream)
    return out


def fa_status_string(code):
    return lib.fa_status_string(code).decode()


def fa_get_device_status(stream=None):
    """(status code, site) after synchronizing `stream`."""
    site = ctypes.c_int(0)
    code = lib.fa_get_device_status(_stream(stream), ctypes.byref(site))
    return code, site.value


def fa_debug_wait_timeout(limit_us, stream=None):
    _check(lib.fa_debug_wait_timeout(limit_us, _stream(stream)), "fa_debug_wait_timeout")


# ---------------------------------------------------------------------------
# conveniences: allocate outputs with torch, call the C functions
# ---------------------------------------------------------------------------

def _shape(q, *others):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d]")
    for t in others:
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device:
            raise ValueError("every tensor must match q in shape, dtype and device")
    return tuple(int(x) for x in q.shape)


def forward(q, k, v, scale=None, causal=False, kv_len=None, block_mask=None, stream=None,
            dropout_p=0.0, seed=0, offset=0, bias=None, tile_order=None):
    """(O, lse) for CUDA tensors q, k, v [B,H,N,d] (bf16 or fp32) of any layout
    whose last dimension is contiguous; O takes q's layout where torch can
    keep it (torch.empty_like).  dropout_p > 0 drops attention probabilities
    (bf16 only); the backward needs the same dropout_p, seed and offset.
    bias: fp32 tensor broadcastable to [B, H, N, N] added to the scaled
    scores (bf16 only); the backward needs it too.  tile_order: the block
    mask's work order (block_mask_order), optional."""
    import torch
    B, H, N, d = _shape(q, k, v)
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    mask = make_mask(kv_len, block_mask, tile_order=tile_order)
    opt = make_options(make_layouts(q=q, k=k, v=v, o=o), dropout_p, seed, offset,
                       None if bias is None else bias_of(bias))
    fn = fa_fwd_ex if q.dtype == torch.bfloat16 else fa_fwd_fp32_ex
    fn(q, k, v, o, lse, B, H, N, d, scale, causal, mask, opt, stream)
    return o, lse


def backward(q, k, v, o, do, lse, scale=None, causal=False, kv_len=None, block_mask=None,
             stream=None, workspace=None, dropout_p=0.0, seed=0, offset=0, bias=None,
             tile_order=None):
    """(dQ, dK, dV) for the forward above and output gradient do; each
    gradient takes the layout of its input where torch can keep it."""
    import torch
    B, H, N, d = _shape(q, k, v, o, do)
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    mask = make_mask(kv_len, block_mask, tile_order=tile_order)
    layouts = make_layouts(q=q, k=k, v=v, o=o, dO=do, dq=dq, dk=dk, dv=dv)
    opt = make_options(layouts, dropout_p, seed, offset, None if bias is None else bias_of(bias))
    fn = fa_bwd_ex if q.dtype == torch.bfloat16 else fa_bwd_fp32_ex
    fn(q, k, v, o, do, lse, dq, dk, dv, workspace, ws_bytes, B, H, N, d, scale, causal, mask,
       opt, stream)
    return dq, dk, dv
