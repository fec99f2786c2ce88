"""Host logic of bench.py's N > 1 path (replicas only), on CPU: two gloo ranks
reduce their timings to the maximum, and the reference arm's non-zero ranks
exit cleanly without printing."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports [r, 10 - r, 2r + 1]: the maxima are [1, 10, 3]
        got = bench.max_over_ranks([rank, 10 - rank, 2 * rank + 1], world)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()  # both ranks rendezvous on it
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        assert out[0] == [1.0, 10.0, 3.0] and out[1] == [1.0, 10.0, 3.0]


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3, 1.5], 1) == [3.0, 1.5]


def test_reference_arm_nonzero_rank_prints_nothing():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_gpus_flag_without_launcher_is_an_error():
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "torchrun" in (r.stderr + r.stdout)


def test_reference_arm_line_has_the_contract_keys(monkeypatch):
    """The reference arm (the fp64 oracle on the host cores) prints the bench
    contract's line: metric, unit, a positive value, the CPU baseline it measured
    and an e2e entry without host-device copies."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 1.0)
    line = bench.run_reference(argparse.Namespace(steps=2, warmup=3), 0, 1)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert bench.run_reference(argparse.Namespace(steps=2, warmup=3), 1, 2) is None  # other ranks: no work
