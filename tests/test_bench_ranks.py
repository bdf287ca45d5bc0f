"""The benchmark's multi-rank host logic, on CPU with the gloo backend (world size 2).

On more than one GPU the benchmark runs independent replicas: each rank times its own copy of the
step, the job time is the slowest rank's, and the whole-job rate counts every rank's tokens."""
import contextlib
import importlib.util
import io
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    # rank r measured (step ms, decode ms) = (1 + r, 5 - r): the job sees the slowest of each
    got = b.max_over_ranks([1.0 + rank, 5.0 - rank], dist, "cpu")
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(" ".join(str(v) for v in got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        vals = [float(x) for x in open(tmp_path / f"r{r}.txt").read().split()]
        assert vals == [2.0, 5.0]


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]


def test_whole_job_rate_counts_every_replica():
    b = _bench()
    one = b.whole_job_rate(524288, 1, 0.25)
    assert abs(one - 524288 / 0.25e-3) < 1e-3
    assert abs(b.whole_job_rate(524288, 4, 0.25) - 4 * one) < 1e-3


def test_reference_arm_is_silent_on_other_ranks():
    b = _bench()

    class Args:
        workload = b.DEFAULT_WORKLOAD
        steps = 1
        warmup = 3
        gpus = 2

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert b.run_reference(Args(), rank=1, world=2) is None
    assert buf.getvalue() == ""
