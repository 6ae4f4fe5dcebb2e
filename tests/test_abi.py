"""C ABI checks that need no GPU: the library loads, exports every function
include/fa.h declares, and rejects bad arguments on the host before touching
the CUDA runtime."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    # These calls pass fake (never dereferenced) pointers that validation must
    # reject; keep them off machines with a GPU so that a validation bug can
    # never turn into a launch with bad pointers.
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only validation tests run on machines without a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_88_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
                     "fa_get_device_status", "fa_fwd_fp32", "fa_bwd_fp32"):
        assert required in names


def test_every_declared_symbol_is_exported(fa):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(\S+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(fa.lib, n)


def test_status_strings(fa):
    for code, name in fa.STATUS.items():
        assert fa.fa_status_string(code).startswith(name)
    assert "unknown" in fa.fa_status_string(99)


def test_workspace_size(fa):
    B, H, N, d = 2, 3, 1000, 128
    rows = B * H * N
    r256 = lambda x: (x + 255) // 256 * 256
    # D (fp32 per row, padded to 256 bytes), then 256 bytes for the work counter
    assert fa.fa_bwd_workspace_size(B, H, N, d) == r256(rows * 4) + 256
    assert fa.fa_bwd_workspace_size(0, 1, 1, 64) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 1, 96) == 0


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: validation fails first


def fwd(fa, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125,
             causal=0, mask=None)
    a.update(kw)
    return fa.lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                         a["d"], a["scale"], a["causal"], a["mask"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(lse=0), 1), (dict(B=0), 1), (dict(N=0), 1), (dict(N=-5), 1),
    (dict(d=96), 2), (dict(d=256), 2), (dict(B=300, H=300), 2),
    (dict(causal=2), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(q=FAKE + 8), 3), (dict(o=FAKE + 2), 3), (dict(lse=FAKE + 2), 3),
    # the size limits, on both sides: B*H <= 65535, B*H*N*d <= 2^40 elements
    # (5 = FA_ERR_CUDA: the arguments passed, and the launch found no GPU here)
    (dict(B=257, H=255), 5), (dict(B=65535), 5), (dict(B=65536), 2), (dict(B=256, H=256), 2),
    (dict(B=1024, N=1 << 24, d=64), 5),          # exactly 2^40 elements
    (dict(B=1024, N=(1 << 24) + 1, d=64), 2),
])
def test_fwd_rejects_bad_arguments(fa, kw, code):
    assert fwd(fa, **kw) == code
    assert fa.lib.fa_fwd_fp32(kw.get("q", FAKE), FAKE, FAKE, kw.get("o", FAKE),
                              kw.get("lse", FAKE), kw.get("B", 1), kw.get("H", 1),
                              kw.get("N", 128), kw.get("d", 64), kw.get("scale", 0.125),
                              kw.get("causal", 0), None, None) == code


def test_fwd_rejects_bad_masks(fa):
    m = ctypes.pointer(fa.FaMask(7, None, None, 128))
    assert fwd(fa, mask=m) == 1
    m = ctypes.pointer(fa.FaMask(fa.FA_MASK_KEY_PADDING, None, None, 0))
    assert fwd(fa, mask=m) == 1   # NULL kv_len
    m = ctypes.pointer(fa.FaMask(fa.FA_MASK_KEY_PADDING, FAKE + 2, None, 0))
    assert fwd(fa, mask=m) == 1   # misaligned kv_len
    m = ctypes.pointer(fa.FaMask(fa.FA_MASK_BLOCK_SPARSE, FAKE, None, 128))
    assert fwd(fa, mask=m) == 1   # NULL block mask
    m = ctypes.pointer(fa.FaMask(fa.FA_MASK_BLOCK_SPARSE, None, FAKE, 64))
    assert fwd(fa, mask=m) == 2   # only 128-wide tiles
    m = ctypes.pointer(fa.FaMask(fa.FA_MASK_BLOCK_SPARSE, None, FAKE, 128))
    assert fwd(fa, mask=m, N=4096 * 128) == 5       # T = 4096: valid (no CUDA here)
    assert fwd(fa, mask=m, N=4096 * 128 + 1) == 2   # T = 4097: beyond the tile bitmap
    m = ctypes.pointer(fa.FaMask(fa.FA_MASK_BLOCK_SPARSE, None, FAKE, 128, FAKE + 2))
    assert fwd(fa, mask=m) == 3   # misaligned work order
    assert bwd(fa, mask=m) == 3
    m = ctypes.pointer(fa.FaMask(fa.FA_MASK_BLOCK_SPARSE, None, FAKE, 128, FAKE))
    assert fwd(fa, mask=m) == 5   # valid (no CUDA here)


def test_block_mask_order_rules(fa):
    # 2T entries for 1 <= T <= 4096 (the block-mask limit), else 0
    assert [fa.fa_block_mask_order_len(t) for t in (1, 2, 3, 128, 4096)] == [
        2, 4, 6, 256, 8192]
    assert fa.fa_block_mask_order_len(0) == 0 and fa.fa_block_mask_order_len(4097) == 0
    call = lambda bm=FAKE, T=8, causal=0, out=FAKE: fa.lib.fa_block_mask_order(
        bm, T, causal, out, None)
    assert call(bm=0) == 1 and call(out=0) == 1
    assert call(T=0) == 1 and call(T=4097) == 1 and call(causal=2) == 1
    assert call(out=FAKE + 2) == 3
    assert call(T=4096) == 5   # valid: the launch finds no GPU here
    with pytest.raises(ValueError):
        fa.make_mask(kv_len=FAKE, tile_order=FAKE)


def bwd(fa, **kw):
    B, H, N, d = kw.get("B", 1), kw.get("H", 1), kw.get("N", 128), kw.get("d", 64)
    ws = kw.get("ws_bytes", fa.fa_bwd_workspace_size(1, 1, 128, 64))
    return fa.lib.fa_bwd(kw.get("q", FAKE), FAKE, FAKE, FAKE, kw.get("dO", FAKE), FAKE,
                         kw.get("dq", FAKE), FAKE, FAKE, kw.get("ws", FAKE), ws, B, H, N, d,
                         kw.get("scale", 0.125), kw.get("causal", 0), kw.get("mask"), None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(dO=0), 1), (dict(dq=FAKE + 4), 3), (dict(d=32), 2),
    (dict(ws=0), 4), (dict(ws_bytes=100), 4), (dict(ws=FAKE + 8), 3), (dict(scale=-0.1), 1),
    (dict(ws_bytes=512), 4),  # room for D (128 rows) but not for the work counter
])
def test_bwd_rejects_bad_arguments(fa, kw, code):
    assert bwd(fa, **kw) == code


def noalloc(fa, **kw):
    B, H, N, d = kw.get("B", 1), kw.get("H", 1), kw.get("N", 128), kw.get("d", 64)
    return fa.lib.fa_bwd_noalloc(kw.get("q", FAKE), FAKE, FAKE, FAKE, kw.get("dO", FAKE), FAKE,
                                 kw.get("dq", FAKE), FAKE, FAKE, B, H, N, d,
                                 kw.get("scale", 0.125), kw.get("causal", 0), kw.get("mask"),
                                 None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(dO=0), 1), (dict(dq=FAKE + 4), 3), (dict(d=32), 2), (dict(d=0), 1),
    (dict(d=-1), 1), (dict(B=0), 1), (dict(scale=-0.1), 1), (dict(causal=3), 1),
    (dict(B=300, H=300), 2),
])
def test_noalloc_rejects_what_fa_bwd_rejects(fa, kw, code):
    """The allocation-free backward checks its arguments as fa_bwd does, with
    the same codes, before any CUDA runtime call (no GPU here)."""
    assert noalloc(fa, **kw) == code
    assert bwd(fa, **kw) == code


def test_noalloc_rejects_sizes_beyond_its_scratch(fa):
    # D alone needs 64 MiB for 16 x 16 heads of 65536 rows: more than the
    # fixed 32 MiB scratch; valid arguments otherwise
    assert fa.fa_bwd_workspace_size(16, 16, 65536, 128) > fa.NOALLOC_SCRATCH_BYTES
    assert noalloc(fa, B=16, H=16, N=65536, d=128) == 2
    m = ctypes.pointer(fa.FaMask(7, None, None, 128))
    assert noalloc(fa, mask=m) == 1


def test_substeps_reject_bad_arguments(fa):
    assert fa.lib.fa_bwd_preprocess(0, FAKE, FAKE, 1, 1, 128, 64, None) == 1
    assert fa.lib.fa_bwd_preprocess(FAKE, FAKE, FAKE + 2, 1, 1, 128, 64, None) == 3
    assert fa.lib.fa_bwd_dkdv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128,
                              80, 0.1, 0, None, None) == 2
    assert fa.lib.fa_bwd_dq(0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.1, 0, None,
                            None) == 1
    assert fa.lib.fa_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, 1, 1, 128, 64, 0.1, 0,
                            None, None) == 3
    assert fa.lib.fa_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.1, 2,
                            None, None) == 1
    assert fa.lib.fa_debug_wait_timeout(0, None) == 1
    assert fa.lib.fa_debug_wait_timeout(2000000, None) == 1


def strided(fa, fp32=False, bwd=False, B=2, H=2, N=128, d=64, dropout=0.0, **lay):
    """Calls an *_ex entry point with fake pointers; `lay` overrides the
    (batch, head, row) strides of named tensors, the rest dense."""
    ls = fa.FaLayouts()
    for name in ("q", "k", "v", "o", "dO", "dq", "dk", "dv"):
        setattr(ls, name, fa.FaLayout(*lay.get(name, (H * N * d, N * d, d))))
    L = fa.make_options(ls, dropout, 1, 2)
    if dropout != dropout:   # NaN: make_options treats it as set
        L.contents.dropout = ctypes.pointer(fa.FaDropout(dropout, 1, 2))
    if not bwd:
        fn = fa.lib.fa_fwd_fp32_ex if fp32 else fa.lib.fa_fwd_ex
        return fn(FAKE, FAKE, FAKE, FAKE, FAKE, B, H, N, d, 0.125, 0, None, L, None)
    fn = fa.lib.fa_bwd_fp32_ex if fp32 else fa.lib.fa_bwd_ex
    ws = fa.fa_bwd_workspace_size(B, H, N, d)
    return fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, B, H, N, d, 0.125, 0,
              None, L, None)


@pytest.mark.parametrize("bwd", [False, True])
@pytest.mark.parametrize("fp32", [False, True])
def test_strided_layout_rules(fa, fp32, bwd):
    B, H, N, d = 2, 2, 128, 64
    name = "dv" if bwd else "o"
    # valid layouts pass validation and reach the CUDA runtime (absent here)
    assert strided(fa, fp32, bwd) == 5
    assert strided(fa, fp32, bwd, q=(N * H * d, d, H * d)) == 5          # [B,N,H,d]
    assert strided(fa, fp32, bwd, **{name: (N * 3 * H * d, d, 3 * H * d)}) == 5  # packed QKV
    # a zero, negative or overlapping stride is not supported
    assert strided(fa, fp32, bwd, k=(H * N * d, 0, d)) == 2
    assert strided(fa, fp32, bwd, v=(-H * N * d, N * d, d)) == 2
    assert strided(fa, fp32, bwd, **{name: (H * N * d, N * d, d - 8)}) == 2
    assert strided(fa, fp32, bwd, q=(1 << 40, N * d, d)) == 2
    # strides must be multiples of 16 bytes
    assert strided(fa, fp32, bwd, q=(H * N * d, N * d + 2, d)) == 3
    assert strided(fa, fp32, bwd, **{name: (H * N * d + 4, N * d, d)}) == (5 if fp32 else 3)
    # the strides of size-1 dimensions are ignored
    assert strided(fa, fp32, bwd, B=1, q=(0, N * d, d), k=(-5, N * d, d)) == 5
    assert strided(fa, fp32, bwd, H=1, N=1, q=(N * d, 3, 7)) == 5


def test_strided_backward_needs_every_layout(fa):
    # the forward ignores dO, dq, dk, dv; the backward rejects them when unset
    ls = fa.FaLayouts()
    for name in ("q", "k", "v", "o"):
        setattr(ls, name, fa.FaLayout(2 * 128 * 64, 128 * 64, 64))
    L = fa.make_options(ls)
    assert fa.lib.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 64, 0.125, 0, None, L,
                            None) == 5
    ws = fa.fa_bwd_workspace_size(2, 2, 128, 64)
    assert fa.lib.fa_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, 2,
                            2, 128, 64, 0.125, 0, None, L, None) == 2


def test_layout_of_reads_torch_strides(fa):
    import torch
    x = torch.zeros(2, 5, 3, 64).transpose(1, 2)   # [B,N,H,d] buffer seen as [B,H,N,d]
    lo = fa.layout_of(x)
    assert (lo.batch, lo.head, lo.row) == (5 * 3 * 64, 64, 3 * 64)
    with pytest.raises(ValueError):
        fa.layout_of(torch.zeros(2, 3, 64, 5).transpose(2, 3))   # d not contiguous
    with pytest.raises(ValueError):
        fa.make_layouts(x=x)


@pytest.mark.parametrize("bwd", [False, True])
def test_dropout_rules(fa, bwd):
    assert strided(fa, bwd=bwd, dropout=0.5) == 5            # valid (no CUDA here)
    assert strided(fa, bwd=bwd, dropout=0.999) == 5
    assert strided(fa, bwd=bwd, dropout=1.0) == 1
    assert strided(fa, bwd=bwd, dropout=-0.25) == 1
    assert strided(fa, bwd=bwd, dropout=float("nan")) == 1
    assert strided(fa, fp32=True, bwd=bwd, dropout=0.5) == 2  # fp32 path: no dropout
    assert strided(fa, fp32=True, bwd=bwd, dropout=0.0) == 5
    # p that rounds to a zero threshold is no dropout, also for fp32
    assert strided(fa, fp32=True, bwd=bwd, dropout=1e-6) == 5
    opt = fa.make_options(None, 0.5, 1, 2)
    assert fa.lib.fa_bwd_dkdv_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64,
                                 0.1, 0, None, opt, None) == 5
    bad = fa.make_options(None, 0.5, 1, 2)
    bad.contents.dropout.contents.p = 1.5
    assert fa.lib.fa_bwd_dq_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 0.1, 0,
                               None, bad, None) == 1


def test_diagnostics_stay_out_of_the_product_abi(fa):
    """The layout GEMM and the dropout-mask writer live in the test-only
    libfa_diag.so; libfa.so exports neither, and the test library rejects bad
    arguments on the host."""
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    assert "fa_diag_" not in out and "fa_debug_umma" not in out and "dropout_mask" not in out
    import _diag
    assert _diag.lib.fa_diag_umma_gemm(FAKE, FAKE, FAKE, 64, 128, 64, 0, 0, 0, 0, None) == 2
    assert _diag.lib.fa_diag_umma_gemm(FAKE, FAKE, FAKE, 128, 128, 64, 1, 0, 1, 0, None) == 1
    assert _diag.lib.fa_diag_umma_gemm(FAKE, FAKE, FAKE, 128, 128, 64, 0, 0, 2, 0, None) == 1
    dr = ctypes.byref(fa.FaDropout(0.5, 1, 2))
    assert _diag.lib.fa_diag_dropout_mask(None, 1, 1, 64, dr, 0, None) == 1
    assert _diag.lib.fa_diag_dropout_mask(FAKE, 1, 1, 64, None, 0, None) == 1
    assert _diag.lib.fa_diag_dropout_mask(FAKE, 1, 1, 5000, dr, 0, None) == 2
    assert _diag.lib.fa_diag_dropout_mask(FAKE, 1, 1, 64, dr, 2, None) == 1
    assert _diag.lib.fa_diag_dropout_mask(FAKE, 1, 1, 64, ctypes.byref(fa.FaDropout(1.0, 1, 2)),
                                          0, None) == 1


def test_bias_rules(fa):
    def call(fp32=False, bwd=False, N=128, **bkw):
        b = dict(ptr=FAKE, batch=0, head=0, row=N)
        b.update(bkw)
        bias = fa.FaBias(b["ptr"], b["batch"], b["head"], b["row"])
        opt = fa.make_options(None, 0.0, 0, 0, bias)
        if not bwd:
            fn = fa.lib.fa_fwd_fp32_ex if fp32 else fa.lib.fa_fwd_ex
            return fn(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, N, 64, 0.125, 0, None, opt, None)
        ws = fa.fa_bwd_workspace_size(1, 2, N, 64)
        fn = fa.lib.fa_bwd_fp32_ex if fp32 else fa.lib.fa_bwd_ex
        return fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, 1, 2, N, 64, 0.125,
                  0, None, opt, None)
    for bwd in (False, True):
        assert call(bwd=bwd) == 5                          # valid: reaches CUDA (none here)
        assert call(bwd=bwd, head=128 * 128, row=128) == 5
        assert call(bwd=bwd, ptr=None) == 1
        assert call(bwd=bwd, ptr=FAKE + 4) == 3
        assert call(bwd=bwd, row=130) == 3                  # not a multiple of 4 elements
        assert call(bwd=bwd, row=64) == 2                   # rows overlap (row < N)
        assert call(bwd=bwd, head=-128) == 2
        assert call(bwd=bwd, row=0) == 5                    # one row for every query
        assert call(fp32=True, bwd=bwd) == 2                # fp32 path: no bias
