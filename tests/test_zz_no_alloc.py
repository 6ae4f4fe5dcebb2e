"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (for example a plugin whose host framework has reserved all device
memory for its own pool, or latency-critical code that must not call
cudaMalloc because it can synchronize the device).  It works in a fixed
scratch array inside the library instead of a caller-provided workspace.

Checked through the C ABI against fa_bwd with an allocated workspace, on two
calls in a row with different inputs and sizes (the scratch keeps the first
call's contents, so the second call must not depend on them)."""
import numpy as np
import pytest
import torch

from workloads import random_case
from _gpu_helpers import TOL, f64, rel_fro, to_device

pytestmark = pytest.mark.gpu


def _reference_and_noalloc(fa, B, H, N, d, causal, seed):
    case = random_case(B, H, N, d, seed=seed)
    t = to_device(case, "bf16")
    scale = d ** -0.5
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal)
    ref = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal)
    got = [torch.full_like(t["q"], float("nan")) for _ in range(3)]
    fa.fa_bwd_noalloc(t["q"], t["k"], t["v"], o, t["do"], lse, got[0], got[1], got[2],
                      B, H, N, d, scale, causal)
    torch.cuda.synchronize()
    code, site = fa.fa_get_device_status()
    assert code == 0, (code, site)
    return ref, got


def test_noalloc_backward_matches_fa_bwd_twice(fa):
    tol = TOL["bf16"][2]
    # first call: 2 x 4 heads of 1000 tokens, causal (32 KB of scratch)
    ref, got = _reference_and_noalloc(fa, 2, 4, 1000, 64, True, seed=31)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert rel_fro(f64(g), f64(r)) <= tol, name
    # second call right after: other inputs, other size, non-causal
    ref, got = _reference_and_noalloc(fa, 1, 3, 777, 128, False, seed=32)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(f64(g))), name
        assert rel_fro(f64(g), f64(r)) <= tol, name


def test_noalloc_rejects_sizes_beyond_its_scratch(fa):
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(16, dtype=torch.float32, device="cuda")
    B, H, N, d = 64, 16, 16384, 128   # D alone needs 64 MiB: more than the fixed scratch
    assert fa.fa_bwd_workspace_size(B, H, N, d) > fa.NOALLOC_SCRATCH_BYTES
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd_noalloc(x, x, x, x, x, lse, x, x, x, B, H, N, d, 0.1, True)
    assert e.value.code == 2   # FA_ERR_UNSUPPORTED, rejected before any launch
