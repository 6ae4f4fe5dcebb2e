"""Consecutive calls on one stream.  The kernels are launched with
programmatic dependent launch: a kernel's CTAs may become resident while the
kernel ahead of it on the stream is still running, and each waits for that
kernel before its first global-memory access.  A missing wait would read a
predecessor's outputs (O, lse, D, the work order, the workspace counter)
before they are complete.  Several forward + backward steps, each on its own
inputs and into its own outputs, are queued with no synchronisation and must
give bit for bit what the same steps give one at a time with a device
synchronisation after every call."""
import numpy as np
import pytest
import torch

from workloads import block_mask_pattern, random_case
from _gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def step(fa, t, scale, causal, kv_len, block_mask, order, ws, sync):
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal, kv_len=kv_len,
                        block_mask=block_mask, tile_order=order)
    if sync:
        torch.cuda.synchronize()
    g = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal, kv_len=kv_len,
                    block_mask=block_mask, tile_order=order, workspace=ws)
    if sync:
        torch.cuda.synchronize()
    return (o, lse) + tuple(g)


CASES = [  # d, causal, mask
    (128, True, "none"),      # persistent dQ CTAs (workspace counter)
    (64, True, "none"),
    (64, False, "padding"),
    (128, False, "sparse"),   # work order computed on the stream each step
]


@pytest.mark.parametrize("d,causal,mask", CASES)
def test_queued_steps_match_synchronised_steps(fa, d, causal, mask):
    B, H, N, steps = 2, 4, 1536, 4
    T = (N + 127) // 128
    scale = d ** -0.5
    inputs = []
    for s in range(steps):
        kv = bm = None
        if mask == "padding":
            kv = np.array([N - 200 * s - 1, 300 + 100 * s], np.int32)
        if mask == "sparse":
            bm = block_mask_pattern("random", T, np.random.default_rng(s), p=0.3)
        case = random_case(B, H, N, d, seed=500 + 10 * s + d, kv_len=kv, block_mask=bm)
        inputs.append(to_device(case, "bf16"))
    ws = [torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
          for _ in range(steps)]

    def run_all(sync):
        outs = []
        for s, t in enumerate(inputs):
            order = None
            if mask == "sparse":
                order = fa.block_mask_order(t["block_mask"], causal)
            outs.append(step(fa, t, scale, causal, t["kv_len"], t["block_mask"], order, ws[s],
                             sync))
        torch.cuda.synchronize()
        return outs

    ref = run_all(sync=True)
    for _ in range(2):
        got = run_all(sync=False)
        code, site = fa.fa_get_device_status()
        assert code == 0, "device status %d at site %d" % (code, site)
        for s in range(steps):
            for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), got[s], ref[s]):
                assert torch.equal(a, b), (s, name)


def test_one_workspace_reused_back_to_back(fa):
    """The same workspace (D and the work counter) for every step: each step's
    preprocess rewrites D and zeroes the counter only after the previous
    step's backward kernel has finished with them."""
    B, H, N, d, steps = 2, 4, 2048, 128, 5
    scale = d ** -0.5
    inputs = [to_device(random_case(B, H, N, d, seed=700 + s), "bf16") for s in range(steps)]
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    ref = [step(fa, t, scale, True, None, None, None, ws, True) for t in inputs]
    torch.cuda.synchronize()
    got = [step(fa, t, scale, True, None, None, None, ws, False) for t in inputs]
    torch.cuda.synchronize()
    for s in range(steps):
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), got[s], ref[s]):
            assert torch.equal(a, b), (s, name)
