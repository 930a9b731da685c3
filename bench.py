"""Benchmark of the GNA forward hot path on B300.

One step = one pass of the whole path over one batch of synthetic input:
    permute Q, K (raster -> 128-token tiles) and V (-> feature-major tiles)
    ->  fused GNA forward
    ->  unpermute O and lse (tiles -> raster)
or, with ``--layout raster``, permute V -> the forward reading Q, K and
writing O, lse in the raster layout, or with ``--layout raster_all`` the forward
alone on every tensor in the raster layout (no permute), on the 720p-video latent workload (30 x 48 x 80 tokens, 24 heads, head_dim 128,
window 16 x 32 x 48, bf16), the configuration the GNA page's video results and
its Blackwell kernel throughput are about.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
bounded samples of the same workload instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--stride 1,1,1] [--heads 24]
    torchrun --nproc-per-node N bench.py --gpus N ...
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "GNA fwd useful TFLOP/s on 1 B300 and % of dense tensor peak; speedup vs dense attn"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gna_fwd_traffic.json")
E4M3_PEAK_FILE = os.path.join(ROOT, "profiles", "e4m3_gemm_peak.json")
FWD_SOURCE = os.path.join(ROOT, "dimensional_sparse_attention_gna_b300", "csrc", "gna_fwd.cu")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--dims", default="30,48,80")
    ap.add_argument("--window", default="16,32,48")
    ap.add_argument("--stride", default="1,1,1")
    ap.add_argument("--heads", type=int, default=24)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp8"])
    ap.add_argument("--layout", default="tiled", choices=["tiled", "raster", "raster_all"],
                    help="tiled: permute Q, K, V and unpermute O, lse around gna_forward; "
                         "raster: permute V only, gna_forward_raster on raster Q, K, O, lse; "
                         "raster_all: no permute, gna_forward_raster_all on raster Q, K, V, O, lse (bf16, d 128)")
    ap.add_argument("--tiles", default="default", choices=["default", "planned"],
                    help="default: one tile for Q and KV (gna_tile_shape); planned: the query and key/value "
                         "tiles gna_plan_tiles picks (they may differ; forward only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--sustain", type=float, default=0.0,
                    help="also run the forward back to back for this many seconds and report the sustained rate")
    ap.add_argument("--backward", action="store_true",
                    help="also time the backward pass (delta, dq, dk/dv kernels; bf16, tiled layout)")
    ap.add_argument("--measure-host-link", action="store_true",
                    help="only measure the pinned host <-> device copy rate of the end-to-end step's sizes")
    ap.add_argument("--measure-e4m3-gemm", action="store_true",
                    help="only time a dense e4m3 GEMM (torch._scaled_mm, 8192^3, bf16 out) as a burst and "
                         "for 4 s back to back, print one JSON line and exit")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: total oracle time over warm-up and timed steps")
    a = ap.parse_args(argv)
    a.dims = tuple(int(x) for x in a.dims.split(","))
    a.window = tuple(int(x) for x in a.window.split(","))
    a.stride = tuple(int(x) for x in a.stride.split(","))
    return a


def useful_flops(B, heads, dims, window, d) -> float:
    """GNA page §1.2: every query processes prod(window) keys: 2 flops per MAC, QK^T and PV."""
    return 4.0 * B * heads * math.prod(dims) * math.prod(window) * d


def workload_name(a) -> str:
    kind = "3-D video" if a.dims[0] > 1 else "2-D image"
    return (f"{kind} GNA forward {'x'.join(map(str, a.dims))} tokens, {a.heads} heads, d={a.head_dim}, "
            f"window {'x'.join(map(str, a.window))}, stride {'x'.join(map(str, a.stride))}, B={a.batch}, {a.dtype}")


def run_config(a, world: int = 1) -> dict:
    """The ``config`` object of both arms' JSON lines (identical keys)."""
    esz = 2 if a.dtype == "bf16" else 1
    return {"workload": workload_name(a), "dims": list(a.dims), "window": list(a.window),
            "stride": list(a.stride), "heads": a.heads, "B": a.batch, "head_dim": a.head_dim,
            "layout": a.layout, "tiles": a.tiles,
            "l2": "inputs larger than L2 (3 x %.0f MB raster + tiled copies)" % (
                a.batch * math.prod(a.dims) * a.heads * a.head_dim * esz / 1e6),
            "parallelism": f"replicas x{world}: every rank runs the full workload on its own data"}


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


def load_e4m3_peak():
    """The dense e4m3 GEMM rate measured on the B300s by ``--measure-e4m3-gemm``
    (recorded in profiles/), or None."""
    try:
        with open(E4M3_PEAK_FILE) as f:
            rec = json.load(f)
        return float(rec["e4m3_tflops"]), float(rec["e4m3_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        return None


def measure_host_link(h2d_bytes: int = 2123366400, d2h_bytes: int = 718848000, reps: int = 5) -> dict:
    """The host link the end-to-end figure rides on: one pinned host -> device copy
    of the bench step's upload size alone, and the same with a device -> host copy
    of the step's download size running concurrently on another stream (CUDA events,
    best of `reps`)."""
    dev = torch.device("cuda")
    h = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    ho = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    do = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(both: bool) -> float:
        best = float("inf")
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(s_in)
            s_out.wait_event(e0)
            with torch.cuda.stream(s_in):
                d.copy_(h, non_blocking=True)
            e1.record(s_in)
            if both:
                with torch.cuda.stream(s_out):
                    ho.copy_(do, non_blocking=True)
            e2.record(s_out)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return best

    alone, with_down = timed(False), timed(True)
    return {"h2d_gbs_alone": h2d_bytes / (alone / 1e3) / 1e9, "h2d_gbs_with_d2h": h2d_bytes / (with_down / 1e3) / 1e9,
            "h2d_bytes": h2d_bytes, "d2h_bytes": d2h_bytes,
            "how": f"pinned host -> device copy of the step's upload size, alone and with a device -> host copy of "
                   f"the step's download size on another stream; best of {reps}, CUDA events"}


def measure_e4m3_gemm(n: int = 8192, seconds: float = 4.0) -> dict:
    """Dense e4m3 x e4m3 -> bf16 GEMM through torch._scaled_mm (cuBLASLt): the
    fp8 counterpart of the measured bf16 cuBLAS figures (2 n^3 flops per GEMM;
    best of 10 as the burst rate, then back to back for `seconds`)."""
    dev = torch.device("cuda")
    a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()      # column-major operand
    one = torch.ones((), device=dev)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps, t0 = 0, time.time()
        e0.record()
        while time.time() - t0 < seconds:
            for _ in range(20):
                mm()
            reps += 20
            torch.cuda.synchronize()
        e1.record()
        torch.cuda.synchronize()
    flops = 2.0 * n ** 3
    return {"e4m3_tflops": flops / (best / 1e3) / 1e12,
            "e4m3_tflops_sustained": flops / (e0.elapsed_time(e1) / reps / 1e3) / 1e12,
            "how": f"torch._scaled_mm e4m3 x e4m3 -> bf16, {n}^3 (2 n^3 flops): best of 10 (burst) and back "
                   f"to back for {seconds:.0f} s (sustained), CUDA events",
            "gpu_name": torch.cuda.get_device_name(), "clocks_sustained": clk.summary()}


def kernel_traffic(a) -> int | None:
    """DRAM bytes per forward launch from the committed ncu capture, scaled to this
    launch by (b, head) planes; None unless the workload (grid, window, stride,
    head_dim, dtype) and layout are the captured ones and the kernel source is
    unchanged since the capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        with open(FWD_SOURCE, "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    m = rec.get("match", {})
    same = (list(a.dims) == m.get("dims") and list(a.window) == m.get("window") and list(a.stride) == m.get("stride")
            and a.head_dim == m.get("head_dim") and a.dtype == m.get("dtype"))
    if rec.get("source_sha256") != h or not same or a.layout not in rec.get("layouts", {}) or a.tiles != "default":
        return None
    return rec["layouts"][a.layout]["bytes_per_plane"] * a.heads * a.batch


# ------------------------------------------------------------------ distributed plumbing

def dist_setup(a):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of ``x`` over all ranks (the job's wall time is its slowest rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            # start timing only once the sampler is producing lines
            t0 = time.time()
            while time.time() - t0 < 2.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.02)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ CPU oracle baseline

def oracle_rate(a, seconds: float, cores: int, seed_offset: int = 0):
    """Time the C oracle on a bounded random sample of the workload's queries.

    Returns (useful flops processed, seconds, n_queries)."""
    import oracle
    from synthetic_inputs import exact_f32, qkv_normal, quantize_e4m3, to_bf16, normal_raster

    dims, heads, d, B = a.dims, a.heads, a.head_dim, a.batch
    # One head's worth of keys is all a sampled query touches; generate a
    # 1-head raster of the same geometry (same per-query work) to bound memory.
    q, k, v = qkv_normal(2 + seed_offset, B, dims, 1, d)
    if a.dtype == "bf16":
        qf, kf, vf = (exact_f32(to_bf16(x)) for x in (q, k, v))
        scales = (1.0, 1.0, 1.0)
    else:
        qs = [quantize_e4m3(x) for x in (q, k, v)]
        qf, kf, vf = (exact_f32(c) for c, _ in qs)
        scales = tuple(s for _, s in qs)
    per_query = 4.0 * math.prod(a.window) * d
    rng = np.random.default_rng(7 + seed_offset)
    n_all = B * math.prod(dims)

    def run(n):
        sel = rng.integers(0, n_all, n).astype(np.int64)
        t0 = time.perf_counter()
        oracle.forward_c(qf, kf, vf, dims, a.window, a.stride, tensor_scales=scales, sel=sel, threads=cores)
        return time.perf_counter() - t0

    n = max(cores, 8)
    dt = run(n)
    while dt < 0.5:
        n *= 4
        dt = run(n)
    n_final = max(1, int(n * seconds / dt))
    dt = run(n_final)
    return per_query * n_final, dt, n_final


def reference_arm(a, rank, world):
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    per_step = a.ref_seconds / max(1, a.steps + a.warmup)     # keep the whole run near a minute
    for _ in range(a.warmup):
        oracle_rate(a, per_step, cores)
    flops = secs = 0.0
    nq = 0
    for i in range(a.steps):
        f, s, n = oracle_rate(a, per_step, cores, seed_offset=i)
        flops += f
        secs += s
        nq += n
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000.0 * secs / a.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: iid N(0,1) Q/K/V, rounded to the GPU input type",
        "config": run_config(a, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{nq} random queries of the workload over {a.steps} steps "
                                   "(plain C oracle, float64, one thread per core)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def gpu_arm(a, rank, world, local):
    from dimensional_sparse_attention_gna_b300 import gna as G

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, heads, dims, d = a.batch, a.heads, a.dims, a.head_dim
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float8_e4m3fn
    stream = torch.cuda.current_stream()

    # inputs: iid N(0,1) drawn on the device (identical recipe to the tests'
    # host generator in distribution; the bench times the path, not the draw)
    gen = torch.Generator(device=dev).manual_seed(20261204 + rank)
    raster_shape = (B,) + dims + (heads, d)
    descale = None
    xs = []
    for _ in range(3):
        x = torch.randn(raster_shape, device=dev, generator=gen, dtype=torch.float32)
        if a.dtype == "bf16":
            xs.append(x.to(torch.bfloat16))
        else:
            s = float(x.abs().max()) / 448.0
            xs.append((x / s).to(torch.float8_e4m3fn))
            descale = (descale or []) + [s]
        del x
    ds = None if descale is None else torch.tensor(descale, dtype=torch.float32, device=dev)
    raster = a.layout in ("raster", "raster_all")
    raster_v = a.layout == "raster_all"
    # query tile and key/value tile (None: the default tile for both)
    tq = tkv = None
    if a.tiles == "planned":
        tq, tkv, _, _ = G.gna_plan_tiles(dims, a.window, a.stride)
    shp = G.tiled_shape(B, heads, dims, d, tq)
    shp_kv = G.tiled_shape(B, heads, dims, d, tkv)
    if not raster:                      # the raster path has no tiled Q, K, O or lse
        qt = torch.empty(shp, dtype=dt, device=dev)
        kt = torch.empty(shp_kv, dtype=dt, device=dev)
        out_t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
        lse_t = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
    if not raster_v:                    # the all-raster path reads V as it is
        vt = torch.empty(G.value_shape(B, heads, dims, d, tkv), dtype=dt, device=dev)
    out = torch.empty(raster_shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(raster_shape[:-1] + (1,), dtype=torch.float32, device=dev)

    def forward(window, stride, q_in, k_in, o_dst, lse_dst, v_in=None):
        """One forward launch of the bench's layout (raster tensors in, raster out)."""
        if raster_v:
            G.gna_forward_raster_all(q_in, k_in, xs[2] if v_in is None else v_in, o_dst, lse_dst[..., 0], B, heads,
                                     dims, window, stride, d, tile=tq, tile_kv=tkv, stream=stream)
        elif raster:
            G.gna_forward_raster(q_in, k_in, vt, o_dst, lse_dst[..., 0], B, heads, dims, window, stride, d,
                                 descale=ds, tile=tq, tile_kv=tkv, stream=stream)
        else:
            G.gna_forward(qt, kt, vt, out_t, lse_t, B, heads, dims, window, stride, d, descale=ds, tile=tq,
                          tile_kv=tkv, stream=stream)

    def permute_in(q_in, k_in, v_in):
        if not raster:
            G.gna_permute(q_in, qt, B, heads, dims, d, tile=tq, stream=stream)
            G.gna_permute(k_in, kt, B, heads, dims, d, tile=tkv, stream=stream)
        if not raster_v:
            G.gna_permute_v(v_in, vt, B, heads, dims, d, tile=tkv, stream=stream)

    def unpermute_out(o_dst, lse_dst):
        if not raster:
            G.gna_unpermute(out_t, o_dst, B, heads, dims, d, tile=tq, stream=stream)
            G.gna_unpermute(lse_t.unsqueeze(-1), lse_dst, B, heads, dims, 1, tile=tq, stream=stream)

    ev = {"fwd": [], "perm": [], "unperm": []}

    def step(record=False):
        if record:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
        permute_in(*xs)
        if record:
            e[1].record(stream)
        forward(a.window, a.stride, xs[0], xs[1], out, lse)
        if record:
            e[2].record(stream)
        unpermute_out(out, lse)
        if record:
            e[3].record(stream)
            ev["perm"].append((e[0], e[1]))
            ev["fwd"].append((e[1], e[2]))
            ev["unperm"].append((e[2], e[3]))
    launches_per_step = 1 if raster_v else 2 if raster else 6

    # the first step of the process, timed on the host on its own: it also pays
    # the one-time set-up (kernel attributes, TMA descriptor encoding, module load)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    step()
    torch.cuda.synchronize()
    first_step_ms = (time.perf_counter() - h0) * 1e3
    for _ in range(max(0, a.warmup - 1)):
        step()
    G.gna_get_status(stream)

    barrier(world)
    torch.cuda.synchronize()
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except ValueError:
            gpu_index = local
    with ClockSampler(gpu_index) as clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(a.steps):
            step(record=True)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    G.gna_get_status(stream)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)
    fwd_ms = statistics.mean(s.elapsed_time(e) for s, e in ev["fwd"])
    perm_ms = statistics.mean(s.elapsed_time(e) for s, e in ev["perm"])
    unperm_ms = statistics.mean(s.elapsed_time(e) for s, e in ev["unperm"])
    flops_rank = useful_flops(B, heads, dims, a.window, d)
    total_flops = sum_over_ranks(flops_rank * a.steps, world)
    value = total_flops / (elapsed_ms / 1e3) / 1e12
    kernel_tflops = flops_rank / (fwd_ms / 1e3) / 1e12
    esz = torch.tensor([], dtype=dt).element_size()
    perm_bytes = (0 if raster_v else 1 if raster else 3) * 2 * B * math.prod(dims) * heads * d * esz
    unperm_bytes = 0 if raster else 2 * B * math.prod(dims) * heads * (d * 2 + 4)

    peaks, peaks_kind = load_peaks()
    # Denominators: the measured cuBLAS bf16 GEMM rates (fp8 takes twice the
    # bf16 rate, the nominal 4.5 / 2.25 PFLOP/s ratio).  The timed region is
    # well under a second, before the board reaches its average power cap, so
    # the burst figure is the matching one; the sustained one is reported too.
    mult = 2.0 if a.dtype == "fp8" else 1.0
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * mult
    peak_sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]) * mult
    peak_source = f"{peaks_kind} {'bf16' if a.dtype == 'bf16' else 'fp8 (2x bf16)'} burst"
    e4m3 = load_e4m3_peak() if a.dtype == "fp8" else None
    if e4m3 is not None:
        # the e4m3 GEMM rate measured on the same pool replaces the 2x bf16 ratio
        peak_burst, peak_sustained = e4m3
        peak_source = "measured e4m3 cuBLASLt GEMM burst (profiles/e4m3_gemm_peak.json)"

    # tile-level work of the launch (what the tensor cores execute)
    visited, partial, nq = G.gna_tile_stats(dims, a.window, a.stride, tq, tile_kv=tkv)
    tile_flops = 4.0 * B * heads * visited * 128 * 128 * d

    # dense attention through the same kernel on the same tokens (window = grid)
    # (same warm-up and step count as the GNA launches, clocks sampled alike, so
    # that the speedup can also be compared at equal clock: time x median MHz)
    speedup = None
    dense_ms = None
    dense_clk = None
    speedup_clock_normalised = None
    if not a.no_dense:
        dense = lambda: forward(dims, (1, 1, 1), xs[0], xs[1], out, lse)  # noqa: E731
        if tq is not None:
            # with planned tiles, dense attention still runs on the default tile
            # (its own best tiling: no padding of the grid beyond it), from its
            # own permuted copies, made outside the timed region
            if raster_v:
                dense = lambda: G.gna_forward_raster_all(xs[0], xs[1], xs[2], out, lse[..., 0], B, heads, dims,  # noqa: E731
                                                         dims, (1, 1, 1), d, stream=stream)
            else:
                vd = torch.empty(G.value_shape(B, heads, dims, d), dtype=dt, device=dev)
                G.gna_permute_v(xs[2], vd, B, heads, dims, d, stream=stream)
                if raster:
                    dense = lambda: G.gna_forward_raster(xs[0], xs[1], vd, out, lse[..., 0], B, heads, dims,  # noqa: E731
                                                         dims, (1, 1, 1), d, descale=ds, stream=stream)
                else:
                    qd, kd = (torch.empty(G.tiled_shape(B, heads, dims, d), dtype=dt, device=dev) for _ in range(2))
                    G.gna_permute(xs[0], qd, B, heads, dims, d, stream=stream)
                    G.gna_permute(xs[1], kd, B, heads, dims, d, stream=stream)
                    od = torch.empty(qd.shape, dtype=torch.bfloat16, device=dev)
                    ld = torch.empty(qd.shape[:-1], dtype=torch.float32, device=dev)
                    dense = lambda: G.gna_forward(qd, kd, vd, od, ld, B, heads, dims, dims, (1, 1, 1), d,  # noqa: E731
                                                  descale=ds, stream=stream)
        for _ in range(a.warmup):
            dense()
        torch.cuda.synchronize()
        dense_ev = []
        with ClockSampler(gpu_index) as dclocks:
            for _ in range(a.steps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dense()
                e1.record(stream)
                dense_ev.append((e0, e1))
            torch.cuda.synchronize()
        G.gna_get_status(stream)
        dense_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in dense_ev)
        speedup = dense_ms / fwd_ms
        dense_clk = dclocks.summary()

    # end to end through the public API with host buffers: every step copies its
    # Q, K, V from pinned host memory, runs the step's kernels and copies O and
    # lse back.  Copies run on their own streams so that step k+1's
    # upload and step k-1's download overlap step k's kernels (two buffer sets).
    e2e = None
    if not a.no_e2e:
        host_in = [x.cpu().pin_memory() for x in xs]
        host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        host_lse = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
        dev_in = [[torch.empty_like(x) for x in xs] for _ in range(2)]
        dev_out = [out, torch.empty_like(out)]
        dev_lse = [lse, torch.empty_like(lse)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in_ready", "perm_done", "comp_done", "out_done")}
        used = {name: [False, False] for name in ev}

        def e2e_step(k):
            b = k % 2
            if used["perm_done"][b]:
                s_in.wait_event(ev["perm_done"][b])       # inputs of step k-2 consumed
            with torch.cuda.stream(s_in):
                for h, dv in zip(host_in, dev_in[b]):
                    dv.copy_(h, non_blocking=True)
            ev["in_ready"][b].record(s_in)
            stream.wait_event(ev["in_ready"][b])
            permute_in(*dev_in[b])
            if not raster:
                ev["perm_done"][b].record(stream)
            if used["out_done"][b]:
                stream.wait_event(ev["out_done"][b])      # results of step k-2 downloaded
            forward(a.window, a.stride, dev_in[b][0], dev_in[b][1], dev_out[b], dev_lse[b], dev_in[b][2])
            if raster:
                ev["perm_done"][b].record(stream)         # the forward read the raster Q, K
            used["perm_done"][b] = True
            unpermute_out(dev_out[b], dev_lse[b])
            ev["comp_done"][b].record(stream)
            s_out.wait_event(ev["comp_done"][b])
            with torch.cuda.stream(s_out):
                host_out[b].copy_(dev_out[b], non_blocking=True)
                host_lse[b].copy_(dev_lse[b], non_blocking=True)
            ev["out_done"][b].record(s_out)
            used["out_done"][b] = True
        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps = a.steps
        e0.record(s_in)
        for k in range(e2e_steps):
            e2e_step(k)
        e1.record(s_out)
        torch.cuda.synchronize()
        barrier(world)
        G.gna_get_status(stream)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        e2e_val = sum_over_ranks(flops_rank * e2e_steps, world) / (e2e_ms / 1e3) / 1e12
        e2e = {"value": e2e_val, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(sum(x.numel() * x.element_size() for x in host_in)),
               "d2h_bytes_per_step": int(host_out[0].numel() * host_out[0].element_size()
                                         + host_lse[0].numel() * host_lse[0].element_size()),
               "ms_per_step": e2e_ms / e2e_steps,
               "pipelining": "uploads, kernels and downloads of consecutive steps on three streams"}

    clk = clocks.summary()
    if speedup is not None and clk and dense_clk and clk.get("sm_mhz") and dense_clk.get("sm_mhz"):
        # cycles instead of seconds: each arm's time x its median SM clock
        speedup_clock_normalised = (dense_ms * dense_clk["sm_mhz"]) / (fwd_ms * clk["sm_mhz"])

    # optional: the forward launched back to back for several seconds, long
    # enough for the board to reach its average power cap
    sustained = None
    if a.sustain > 0:
        with ClockSampler(gpu_index) as sclk:
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n_sus, t_wall = 0, time.time()
            s0.record(stream)
            while time.time() - t_wall < a.sustain:
                for _ in range(5):
                    forward(a.window, a.stride, xs[0], xs[1], out, lse)
                n_sus += 5
                stream.synchronize()
            s1.record(stream)
            torch.cuda.synchronize()
        G.gna_get_status(stream)
        sus_ms = s0.elapsed_time(s1) / n_sus
        sustained = {"value": flops_rank / (sus_ms / 1e3) / 1e12, "unit": "TFLOP/s", "launches": n_sus,
                     "forward_ms": sus_ms, "seconds": a.sustain, "clocks": sclk.summary(),
                     "frac_of_sustained_peak": flops_rank / (sus_ms / 1e3) / 1e12 / peak_sustained}
    # optional: the backward pass on the same workload, inputs resident (tiled
    # q, k, v, dout; k in the value layout; the forward's out and lse)
    backward = None
    if a.backward and a.dtype == "bf16" and d in (32, 64, 128) and not raster and a.tiles == "default":
        v_tiled = torch.empty(shp, dtype=dt, device=dev)
        k_val = torch.empty_like(vt)
        G.gna_permute(xs[2], v_tiled, B, heads, dims, d, stream=stream)
        G.gna_permute_v(xs[1], k_val, B, heads, dims, d, stream=stream)
        dout_t = torch.randn(shp, device=dev, generator=gen, dtype=torch.float32).to(dt)
        delta = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
        dq_t, dk_t, dv_t = (torch.empty(shp, dtype=dt, device=dev) for _ in range(3))
        G.gna_forward(qt, kt, vt, out_t, lse_t, B, heads, dims, a.window, a.stride, d, stream=stream)

        def bwd(ev3=None):
            if ev3:
                ev3[0].record(stream)
            G.gna_backward_delta(out_t, dout_t, delta, B, heads, dims, d, stream=stream)
            G.gna_backward_dq(qt, kt, k_val, v_tiled, dout_t, lse_t, delta, dq_t, B, heads, dims, a.window, a.stride,
                              d, stream=stream)
            if ev3:
                ev3[1].record(stream)
            G.gna_backward_dkdv(qt, kt, v_tiled, dout_t, lse_t, delta, dk_t, dv_t, B, heads, dims, a.window,
                                a.stride, d, stream=stream)
            if ev3:
                ev3[2].record(stream)
        for _ in range(2):
            bwd()
        runs = []
        for _ in range(3):
            ev3 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            bwd(ev3)
            runs.append(ev3)
        torch.cuda.synchronize()
        G.gna_get_status(stream)
        dq_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in runs)
        dkdv_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in runs)
        bwd_ms = dq_ms + dkdv_ms
        # five window-restricted matmuls (S, dP, dV, dK, dQ), 2 flops per MAC
        bwd_flops = 2.5 * flops_rank
        backward = {"ms": bwd_ms, "useful_tflops": bwd_flops / (bwd_ms / 1e3) / 1e12,
                    "frac_of_burst_peak": bwd_flops / (bwd_ms / 1e3) / 1e12 / peak_burst,
                    "kernels_ms": {"delta_and_dq": dq_ms, "dk_dv": dkdv_ms},
                    "flops": "10 * B * heads * N * |window| * d (S, dP, dV, dK, dQ restricted to the window)"}
        del v_tiled, k_val, dout_t, delta, dq_t, dk_t, dv_t
    traffic = kernel_traffic(a)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cores = os.cpu_count() or 1
        f, s, n = oracle_rate(a, a.cpu_seconds, cores)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} random queries of the workload (one synthetic head), plain C oracle, float64, "
                         f"{s:.1f} s on {cores} threads"}

    if rank != 0:
        return
    n_ratio = math.prod(dims) / math.prod(a.window)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": elapsed_ms / a.steps, "first_step_ms": first_step_ms,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": a.dtype,
        "data": "synthetic: iid N(0,1) Q/K/V drawn on the device per rank",
        "config": run_config(a, world), "tile": list(tq or G.gna_tile_shape(dims)),
        "tile_kv": list(tkv or tq or G.gna_tile_shape(dims)),
        "roofline": {"bound": "tensor", "achieved": kernel_tflops, "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": kernel_tflops / peak_burst, "traffic": traffic,
                     "peak_source": peak_source,
                     "frac_of_sustained_peak": kernel_tflops / peak_sustained,
                     "tile_work_tflops": tile_flops / (fwd_ms / 1e3) / 1e12,
                     "tile_overhead": tile_flops / flops_rank, "partial_tile_share": partial / visited},
        "kernels_ms": {("permute_v" if raster else "permute_qkv"): None if raster_v else perm_ms, "forward": fwd_ms,
                       "unpermute_o_lse": None if raster else unperm_ms},
        "permute_gbps": None if raster_v else perm_bytes / (perm_ms / 1e3) / 1e9,
        "permute_frac_of_hbm": None if raster_v else perm_bytes / (perm_ms / 1e3) / 1e9 / peaks.get("hbm_gbs", 6400.0),
        "unpermute_gbps": None if raster else unperm_bytes / (unperm_ms / 1e3) / 1e9,
        "dense_forward_ms": dense_ms, "speedup_vs_dense": speedup,
        "dense_clocks": dense_clk, "speedup_vs_dense_clock_normalised": speedup_clock_normalised,
        "flop_sparsity_ratio": n_ratio,
        # dense attention's tile pairs on the default tile over this launch's visited pairs
        "speedup_bound_at_equal_tile_rate": (math.prod(-(-L // t) for L, t in zip(dims, G.gna_tile_shape(dims))) ** 2
                                             / visited),
        "speedup_over_ratio": None if speedup is None else speedup / n_ratio,
        "e2e": e2e, "gpu_launches": launches_per_step * a.steps, "clocks": clk, "cpu_baseline": cpu,
        "sustained": sustained, "backward": backward,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    a = parse_args(argv)
    if a.measure_host_link:
        print(json.dumps(measure_host_link()), flush=True)
        return
    if a.measure_e4m3_gemm:
        print(json.dumps(measure_e4m3_gemm()), flush=True)
        return
    rank, world, local = dist_setup(a)
    try:
        if a.impl == "reference":
            reference_arm(a, rank, world)
        else:
            gpu_arm(a, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
