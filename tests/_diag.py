"""Loader of libfa_diag.so, the test-only diagnostics built beside libfa.so
(not part of libfa's C ABI): the tensor-core operand-layout GEMM and the
dropout-mask writer, both running the attention kernels' own device code."""
import ctypes
import os

import exact_attention_88_gb300 as fa

DIAG_PATH = os.path.join(os.path.dirname(fa.LIB_PATH), "libfa_diag.so")
if not os.path.exists(DIAG_PATH):
    raise ImportError("libfa_diag.so is not built (expected at %s)" % DIAG_PATH)
lib = ctypes.CDLL(DIAG_PATH)

_p, _i = ctypes.c_void_p, ctypes.c_int
lib.fa_diag_umma_gemm.argtypes = [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p]
lib.fa_diag_dropout_mask.argtypes = [_p, _i, _i, _i, ctypes.POINTER(fa.FaDropout), _i, _p]
lib.fa_diag_status.argtypes = [_p, ctypes.POINTER(ctypes.c_int)]
for _fn in (lib.fa_diag_umma_gemm, lib.fa_diag_dropout_mask, lib.fa_diag_status):
    _fn.restype = ctypes.c_int


def _ptr(x):
    return None if x is None else (x.data_ptr() if hasattr(x, "data_ptr") else int(x))


def umma_gemm(a, b, d, M, N, K, a_mn_major=0, b_mn_major=0, a_in_tmem=0, use_tma=0):
    code = lib.fa_diag_umma_gemm(_ptr(a), _ptr(b), _ptr(d), M, N, K, a_mn_major, b_mn_major,
                                 a_in_tmem, use_tma, None)
    if code != 0:
        raise fa.FaError(code, "fa_diag_umma_gemm")


def dropout_mask(out, B, H, N, p, seed, offset, path):
    dr = fa.FaDropout(p, seed, offset)
    code = lib.fa_diag_dropout_mask(_ptr(out), B, H, N, ctypes.byref(dr), path, None)
    if code != 0:
        raise fa.FaError(code, "fa_diag_dropout_mask")


def status():
    """(code, site) of the diagnostics after a device synchronisation."""
    site = ctypes.c_int(0)
    return lib.fa_diag_status(None, ctypes.byref(site)), site.value
