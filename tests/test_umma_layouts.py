"""Tensor-core operand layouts on the GPU: the test-only diagnostic GEMM
(libfa_diag.so) stages A and B exactly as the attention kernels do
(128-byte-swizzled K-major or MN-major shared-memory tiles, TMA or plain
loads, A optionally in tensor memory) and must reproduce A B^T.  Also the
failure path of libfa's bounded waits."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    b = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = a.double() @ b.double().T
    return a.cuda(), b.cuda(), ref


def _run(fa, M, N, K, a_mn, b_mn, a_tmem, use_tma, seed=0):
    import _diag
    a, b, ref = _case(M, N, K, seed)
    d = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    _diag.umma_gemm(a, b, d, M, N, K, a_mn, b_mn, a_tmem, use_tma)
    torch.cuda.synchronize()
    code, site = _diag.status()
    assert code == 0, (code, site)
    err = (d.double().cpu() - ref).abs().max().item()
    return err, ref.abs().max().item()


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_smem_operands(fa, N, K, a_mn, b_mn):
    err, scale = _run(fa, 128, N, K, a_mn, b_mn, 0, 0)
    assert err <= 1e-4 * max(1.0, scale), err


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("K", [64, 128])
def test_tma_k_major_operands(fa, N, K):
    err, scale = _run(fa, 128, N, K, 0, 0, 0, 1)
    assert err <= 1e-4 * max(1.0, scale), err


@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("K", [64, 128])
def test_a_from_tensor_memory(fa, N, K):
    # A in TMEM as the kernels keep P, P^T, dS and dS^T: two bf16 per 32-bit
    # column, even k in the low half
    err, scale = _run(fa, 128, N, K, 0, 0, 1, 0)
    assert err <= 1e-4 * max(1.0, scale), err


def test_wait_timeout_is_reported(fa):
    """A wait that can never complete gives up after its limit; the kernel
    returns and the host reads FA_ERR_TIMEOUT (no hang, no fault)."""
    fa.fa_debug_wait_timeout(20000)   # 20 ms
    code, site = fa.fa_get_device_status()
    assert code == 6 and site == 9100, (code, site)
    # the status is cleared by the read and the context stays usable
    assert fa.fa_get_device_status() == (0, 0)
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
