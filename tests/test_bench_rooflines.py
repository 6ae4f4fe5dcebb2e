"""bench.py's tensor-pipe figure (CPU only): the activity of the kernels a
timed step launches (the forward, the preprocess and the combined backward),
weighted by their times, and its algorithmic share; the split dK/dV and dQ
kernels of the per-kernel pass do not enter it, and a constant cleared after a
kernel changed gives no figure at all."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PER_KERNEL = {"fwd": 0.72, "bwd_preprocess": 0.026, "bwd_dkdv": 1.6, "bwd_dq": 1.05,
              "bwd": 2.63, "bwd_combined": 2.604}


def test_step_kernels_weighted_by_time():
    fwd = 1.0995e12
    act = bench.TENSOR_PIPE_ACTIVE["long_causal_d128"]
    got = bench.tensor_pipe_share("long_causal_d128", PER_KERNEL, 3.5 * fwd, fwd)
    step = ("fwd", "bwd_preprocess", "bwd_combined")
    assert tuple(bench.STEP_KERNELS) == step
    busy = sum(act[k] * PER_KERNEL[k] for k in step) / sum(PER_KERNEL[k] for k in step)
    assert abs(got["active_time_weighted"] - round(busy, 4)) < 1e-12
    # the kernels execute fwd (2 GEMMs), dK/dV (4) and dQ (3) = 4.5 forwards of
    # GEMM work; the metric counts 3.5
    assert abs(got["executed_tflop"] - round(4.5 * fwd / 1e12, 4)) < 1e-12
    assert abs(got["algorithmic_active"] - round(busy * 3.5 / 4.5, 4)) < 1e-12
    assert set(got["per_kernel_active"]) == set(step)


def test_split_kernels_do_not_enter_the_weighting():
    fwd = 1.0995e12
    a = bench.tensor_pipe_share("long_causal_d128", PER_KERNEL, 3.5 * fwd, fwd)
    other = dict(PER_KERNEL, bwd_dkdv=9.0, bwd_dq=9.0, bwd=99.0)
    b = bench.tensor_pipe_share("long_causal_d128", other, 3.5 * fwd, fwd)
    assert a == b


def test_no_figure_without_captures(monkeypatch):
    fwd = 1.0
    assert bench.tensor_pipe_share("gpt2_causal", PER_KERNEL, 3.5 * fwd, fwd) is None
    cleared = {"long_causal_d128": dict(bench.TENSOR_PIPE_ACTIVE["long_causal_d128"], fwd=None)}
    monkeypatch.setattr(bench, "TENSOR_PIPE_ACTIVE", cleared)
    assert bench.tensor_pipe_share("long_causal_d128", PER_KERNEL, 3.5 * fwd, fwd) is None
