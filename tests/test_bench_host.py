"""Host-side logic of bench.py (CPU): the max-over-ranks reduction with two gloo ranks, the
clock-sample parsing, the measured-peak lookup and the argument defaults."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.reduce_max(1.5 + rank)
    bench.barrier()
    q.put((rank, v, bench.dist_env()))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [2.5, 2.5]
    assert [g[2][:2] for g in got] == [(0, 2), (1, 2)]


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max(3.25) == 3.25


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1965, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "0, 1980, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s["sm_mhz"] == 1972.5 and s["sm_max_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 2


def test_measured_peaks_and_defaults():
    p = bench.measured_peaks()
    assert p["bf16_tflops"] > 100 and p["hbm_gbs"] > 1000
    a = bench.parse_args([])
    assert a.gpus == 1 and a.steps >= 1 and a.warmup >= 3 and a.impl == "ours"


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` without a launcher starts two ranks through torch.distributed.run; on
    this CPU-only host both reach the multi-rank set-up (gloo) and then stop for lack of a GPU, so
    the run exits non-zero and never prints a one-GPU line."""
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR",
                                                            "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, bench.__file__, "--gpus", "2", "--steps", "1", "--warmup", "3",
                        "--no-cpu-baseline"], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode != 0
    assert '"n_gpus": 1' not in r.stdout
    assert "rank 0 of 2" in r.stderr and "rank 1 of 2" in r.stderr, r.stderr[-2000:]


def test_gpus_flag_must_match_the_launcher():
    env_keep = {k: os.environ.get(k) for k in ("WORLD_SIZE",)}
    os.environ["WORLD_SIZE"] = "3"
    try:
        with pytest.raises(SystemExit) as e:
            bench.main(["--gpus", "2"])
        assert "3 ranks" in str(e.value)
    finally:
        for k, v in env_keep.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
