"""Host-side logic of bench.py's multi-GPU path (replicas), on CPU ranks over
gloo: the job's time is the slowest rank's, its work the sum over ranks, and
only rank 0 reports (the reference arm does no work on other ranks)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, dist, "cpu")
        out[rank] = (job_ms, bench.whole_job_tflops(1e12, 4, job_ms, world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    job_ms, tflops = res[0]
    assert job_ms == 15.0
    # 2 replicas x 4 steps x 1 TFLOP in 15 ms
    assert tflops == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_collective():
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5
    assert bench.whole_job_tflops(2e12, 10, 20.0, 1) == pytest.approx(1000.0)


def test_reference_arm_does_no_work_off_rank_0():
    class Args:
        workload = "long_causal_d128"
        steps = 1
        warmup = 0
        reference_rows = 8
    assert bench.run_reference(Args(), rank=1) is None


def test_cpu_sample_is_clamped_to_the_sequence():
    """A sample of more query rows than the sequence has times all N rows
    (it once indexed rows before the start of the sequence)."""
    from workloads import WORKLOADS, generate
    w = WORKLOADS["tiny_fp32_causal"]
    case = generate(w, seed=0, samples=1)
    sec, fl, n, slices = bench.oracle_sample(w, case, 8192)
    assert n == w.N and slices == 1 and sec > 0
    # causal: N (N + 1) / 2 visible pairs, 3.5 x (4 d) FLOPs per pair
    assert fl == pytest.approx(3.5 * 4 * w.d * w.N * (w.N + 1) / 2)
    # several slices: the work adds up; more slices than the workload has are capped
    _, fl2, _, slices2 = bench.oracle_sample(w, case, 8192, heads=5)
    assert slices2 == w.B * w.H and fl2 == pytest.approx(slices2 * fl)
    res = bench.cpu_baseline(w, case, 8192, 2)
    assert "last %d query rows of each of the first 2" % w.N in res["sample"]
    assert res["value"] > 0


def test_reference_arm_line_on_rank_0():
    """The reference arm's line: the oracle's throughput with the keys of the
    GPU arm's line, a cpu_baseline describing the run, and an e2e equal to
    the value with no host-device bytes."""
    class Args:
        workload = "tiny_fp32_causal"
        steps = 2
        warmup = 1
        reference_rows = 64
    res = bench.run_reference(Args(), rank=0)
    assert res["impl"] == "reference" and res["value"] > 0 and res["dtype"] == "f64"
    assert res["steps"] == 2 and res["warmup"] == 1 and res["higher_is_better"] is True
    assert res["config"]["workload"] == "tiny_fp32_causal"
    cpu = res["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == res["value"] and cpu["cores"] >= 1
    assert res["e2e"] == {"value": res["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
