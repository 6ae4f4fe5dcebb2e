"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
run the library through its C ABI, compare with the oracle."""
import numpy as np
import torch

TOL = {
    # O max-abs, lse max-abs, dQ/dK/dV relative Frobenius
    "bf16": (1e-2, 1e-3, 2e-2),
    "fp32": (1e-3, 1e-4, 2e-3),
}


def to_device(case, dtype):
    out = {}
    for n in ("q", "k", "v", "do"):
        if dtype == "bf16":
            out[n] = torch.from_numpy(case[n + "_bits"].view(np.int16)).view(torch.bfloat16).cuda()
        else:
            out[n] = torch.from_numpy(np.ascontiguousarray(case[n])).cuda()
    out["kv_len"] = None if case.get("kv_len") is None else torch.from_numpy(case["kv_len"]).cuda()
    out["block_mask"] = (None if case.get("block_mask") is None
                         else torch.from_numpy(np.ascontiguousarray(case["block_mask"])).cuda())
    return out


def run(fa, t, scale, causal, with_bwd=True):
    o, lse = fa.forward(t["q"], t["k"], t["v"], scale, causal, kv_len=t["kv_len"],
                        block_mask=t["block_mask"])
    grads = None
    if with_bwd:
        grads = fa.backward(t["q"], t["k"], t["v"], o, t["do"], lse, scale, causal,
                            kv_len=t["kv_len"], block_mask=t["block_mask"])
    torch.cuda.synchronize()
    code, site = fa.fa_get_device_status()
    assert code == 0, "device status %d at site %d" % (code, site)
    return o, lse, grads


def f64(x):
    return x.float().cpu().numpy().astype(np.float64)


def max_abs(a, b, finite_only=False):
    with np.errstate(invalid="ignore"):   # -inf - -inf where both rows are empty
        d = np.abs(a - b)
    if finite_only:
        both_inf = np.isneginf(a) & np.isneginf(b)
        d = np.where(both_inf, 0.0, d)
    return float(np.max(d)) if d.size else 0.0


def rel_fro(a, b):
    den = np.linalg.norm(b)
    if den == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / den)
