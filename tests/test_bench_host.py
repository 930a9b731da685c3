"""Host-side logic of bench.py: the multi-rank reduction (world size 2 over gloo,
on CPU) and the workload arithmetic the JSON line reports."""
import json
import math
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    dist.init_process_group("gloo")
    try:
        bench.barrier(world)
        # rank r pretends its timed region took 10 + r ms and processed (r + 1) units
        t = bench.max_over_ranks(10.0 + rank, world)
        n = bench.sum_over_ranks(float(rank + 1), world)
        q.put((rank, t, n))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_summed_work_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    # every rank sees the slowest rank's time and the whole job's work
    assert got == [(0, 11.0, 3.0), (1, 11.0, 3.0)]


def test_useful_flops_matches_the_window_volume_formula():
    sys.path.insert(0, ROOT)
    import bench
    # 3-D video latent: 4 * 24 heads * 115200 queries * 24576 keys * 128
    assert bench.useful_flops(1, 24, (30, 48, 80), (16, 32, 48), 128) == 4.0 * 24 * 115200 * 24576 * 128
    assert math.isclose(bench.useful_flops(1, 24, (30, 48, 80), (16, 32, 48), 128) / 1e12, 34.79, rel_tol=1e-3)
    # dense = window equal to the grid
    assert math.isclose(bench.useful_flops(1, 24, (30, 48, 80), (30, 48, 80), 128) / 1e12, 163.07, rel_tol=1e-3)


def test_reference_arm_other_ranks_print_nothing(capsys):
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.reference_arm(a, rank=1, world=2)
    assert capsys.readouterr().out == ""


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--dims", "4,16,16", "--window", "2,5,5", "--heads", "2",
                        "--head-dim", "32", "--ref-seconds", "1"], capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # the same config object as the GPU arm builds for these arguments (both call run_config)
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse_args(["--dims", "4,16,16", "--window", "2,5,5", "--heads", "2", "--head-dim", "32"])
    assert line["config"] == bench.run_config(a, 1)


def test_traffic_record_applies_only_to_the_captured_workload():
    """The committed ncu DRAM bytes scale with (b, head) planes of the captured
    workload and layout; any other workload reports null rather than a guess."""
    sys.path.insert(0, ROOT)
    import bench
    rec = json.load(open(bench.TRAFFIC_FILE))
    m = rec["match"]
    base = ["--dims", ",".join(map(str, m["dims"])), "--window", ",".join(map(str, m["window"])),
            "--stride", ",".join(map(str, m["stride"])), "--head-dim", str(m["head_dim"]), "--dtype", m["dtype"]]
    t1 = bench.kernel_traffic(bench.parse_args(base + ["--heads", "1"]))
    if t1 is None:        # the kernel source changed since the capture: nothing may be reported
        assert bench.kernel_traffic(bench.parse_args(base)) is None
        return
    assert t1 == rec["layouts"]["tiled"]["bytes_per_plane"]
    assert bench.kernel_traffic(bench.parse_args(base + ["--heads", "6", "--batch", "2"])) == 12 * t1
    raster = bench.kernel_traffic(bench.parse_args(base + ["--heads", "1", "--layout", "raster"]))
    if "raster" in rec["layouts"]:
        assert raster == rec["layouts"]["raster"]["bytes_per_plane"]
    else:                 # a layout without its own capture reports nothing
        assert raster is None
    other = "fp8" if m["dtype"] == "bf16" else "bf16"
    assert bench.kernel_traffic(bench.parse_args(base[:-1] + [other])) is None
    assert bench.kernel_traffic(bench.parse_args(base + ["--window", "1,1,1"])) is None
