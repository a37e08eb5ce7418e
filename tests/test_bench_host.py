"""Host-side logic of bench.py without a GPU: the replica aggregation over ranks (world size 2,
gloo), the reference arm's JSON line, and the clock-record parser."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    bench.dist_setup("gloo")
    ms = 1.0 + rank                       # rank 1 is the slowest
    worst = bench.dist_max(ms, None)
    bench.dist_barrier()
    q.put((rank, worst, bench.aggregate_us_per_layer(worst, 40, world)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replicas_take_the_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    assert got[0][1] == got[1][1] == 2.0
    # 2 ranks x 40 layers in 2 ms: 25 us per layer for the whole job
    assert abs(got[0][2] - 2.0 * 1000 / 80) < 1e-9


def test_clock_parser(tmp_path):
    p = tmp_path / "c.csv"
    p.write_text("0, 1965, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
                 "0, 1980, 2070, 950.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")

    class P:
        def terminate(self): pass
        def wait(self, timeout=None): pass
    f = open(tmp_path / "dummy", "w")
    got = bench.stop_clock_sampler(P(), f, str(p))
    assert got["sm_mhz"] == 1972.5 and got["sm_max_mhz"] == 2070 and got["reasons"] == ["sw_power_cap"]


def test_reference_arm_prints_its_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "us/layer" and line["higher_is_better"] is False
    assert line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    # at least 3 untimed warm-up steps, whatever was asked; the timed steps asked for, within the budget
    assert line["warmup"] >= 3 and line["steps"] == 1
    # each step is a whole 40-layer pass, timed: the line's time per step and per layer agree
    assert abs(line["ms_per_step"] * 1000 / 40 - line["value"]) <= 1e-3 * line["value"] + 1e-3
    assert line["ms_per_step"] / 1000 <= line["config"]["timed_s"] + 0.01   # timed_s is rounded


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """A kernel's traffic comes from its committed ncu summary only while the kernel source is
    the one the counters were taken on."""
    src = tmp_path / "attend.cu"
    src.write_bytes(b"kernel v1")
    import hashlib
    h = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    prof = tmp_path / "p.md"
    prof.write_text(f"# x\n\ntraffic_bytes: 123\nsource_sha256_16: {h}\n")
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.profiled_traffic("p.md", "attend.cu") == 123
    src.write_bytes(b"kernel v2")
    assert bench.profiled_traffic("p.md", "attend.cu") is None
    assert bench.profiled_traffic("missing.md", "attend.cu") is None


def test_committed_profiles_match_the_kernel_sources():
    """The committed ncu summaries the bench line takes `traffic` from were captured on the
    kernel sources as they stand: a kernel changed without a new capture reports no traffic."""
    assert bench.profiled_traffic("attend_swa_window512.md", "attend.cu") is not None
    assert bench.profiled_traffic("attend_full_8k_resident.md", "attend.cu") is not None
    assert bench.profiled_traffic("accept_17x131072.md", "accept.cu") is not None
