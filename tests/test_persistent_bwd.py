"""The combined backward with persistent dQ CTAs (d = 128 without a block mask,
key padding, dropout or a bias: after the one-per-unit dK/dV CTAs, one CTA
per SM takes dQ query tiles from a counter in the workspace) against the
one-CTA-per-unit kernels of the split calls (fa_bwd_preprocess, fa_bwd_dkdv,
fa_bwd_dq), which run the same arithmetic per unit: the gradients must be
bit-identical.  The shapes give each persistent CTA several units (so that
the hand-offs between units -- one Q/dO buffer, the accumulator read out
while the next unit starts -- run), a ragged last tile, both masks and a
strided layout; the oracle comparison of the same path is in test_parity.py."""
import numpy as np
import pytest
import torch

from workloads import random_case
from _gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def split_backward(fa, t, o, lse, scale, causal):
    B, H, N, d = t["q"].shape
    D = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
    fa.fa_bwd_preprocess(o, t["do"], D, B, H, N, d)
    fa.fa_bwd_dkdv(t["q"], t["k"], t["v"], t["do"], lse, D, dk, dv, B, H, N, d, scale,
                   int(causal))
    fa.fa_bwd_dq(t["q"], t["k"], t["v"], t["do"], lse, D, dq, B, H, N, d, scale,
                 int(causal))
    return dq, dk, dv


# (B, H, N, causal): units = 2 T B H against 152 SMs
SHAPES = [(2, 8, 2048, True),      # 512 units, 16 tiles a head
          (1, 16, 4096 - 57, False),  # 1024 units, ragged last tile
          (4, 12, 1024, True),     # 768 units, all heads in one grid-order group
          (1, 2, 200, True)]       # 8 units: fewer than the SMs


@pytest.mark.parametrize("B,H,N,causal", SHAPES)
def test_persistent_matches_split_kernels(fa, B, H, N, causal):
    case = random_case(B, H, N, 128, seed=N + B + causal)
    t = to_device(case, "bf16")
    scale = 128 ** -0.5
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal)
    g1 = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal)
    g2 = split_backward(fa, t, o, lse, scale, causal)
    g3 = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal)
    torch.cuda.synchronize()
    code, site = fa.fa_get_device_status()
    assert code == 0, "device status %d at site %d" % (code, site)
    for name, a, b, c in zip(("dq", "dk", "dv"), g1, g2, g3):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
        assert torch.equal(a.view(torch.int16), c.view(torch.int16)), name + " (second run)"


def test_persistent_with_strided_layouts(fa):
    """Inputs in [B, N, H, d] order (every tensor read and written through its
    strides) give the dense call's gradients bit for bit."""
    B, H, N, d = 2, 8, 1536, 128
    case = random_case(B, H, N, d, seed=77)
    t = to_device(case, "bf16")
    scale = d ** -0.5
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, True)
    ref = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, True)
    bnhd = {n: t[n].transpose(1, 2).contiguous().transpose(1, 2) for n in ("q", "k", "v", "do")}
    o_s = o.transpose(1, 2).contiguous().transpose(1, 2)
    got = fa.backward(bnhd["q"], bnhd["k"], bnhd["v"], o_s, bnhd["do"], lse, scale, True)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(a.contiguous().view(torch.int16), b.view(torch.int16)), name
