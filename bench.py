"""Benchmark of the ternary FFN decode step on GB300.

One "step" is one full FFN layer decode step (rotate+quantise x -> gate/up
ternary GEMVs + SiLU*up -> rotate+quantise h -> down GEMV) at hidden 5120,
intermediate 17408, batch 1, 2-bit ternary weights: the dense-FFN shape of a
27B ternary model.  Inputs are seeded synthetic data (see
ternary_weight_dp4a_gb300/synth.py).  The headline value is weight bytes
streamed per second (GB/s) with inputs resident in HBM; eight independently
seeded weight sets (568 MB, more than 4x the 129 MB L2) are used in rotation so
every step streams its weights from HBM.

Prints ONE JSON line on rank 0.  Launch with torchrun for N > 1 GPUs: each rank
runs an independent replica (the decode FFN needs no exchange between GPUs).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HIDDEN, INTER = 5120, 17408
N_SETS = 8
SWEEP_ROWS = (1, 2, 4, 8, 16, 32, 64)
METRIC = "ternary FFN decode step: weight GB/s & % HBM roofline, µs/token at batch 1/2/4/8"
WORKLOAD = "ffn_layer_h5120_i17408_ternary2"
BLOCK = 128


NOMINAL_HBM_GBS = 8000.0     # the nominal GB300 HBM3e figure the scope's roofline quotes
SMS = 152
INT_LANES_PER_CLK = 64       # integer pipe (prmt, lop3, shf, dp4a) per SM and clock, measured


ENGINES = {"tcgen05": 2, "dp4a": 1}
PASS_ROWS = {"tcgen05": 8, "dp4a": 4}


def int_ops_per_weight(fmt: int, rows: int, engine: str = "dp4a") -> float:
    """Integer-pipe ops per weight in one pass of ``rows`` activation rows.
    dp4a kernel (decode and dot products): 2-bit, 7 ops (3 shifts, 4 prmt) per
    16 weights plus one dp4a per 4 weights and row; 1-bit, a shift and a mask
    per 4 weights plus one dp4a per 4 weights and row.  Tensor-core kernel
    (the decode alone; the tensor core takes the products): 2-bit, the same 7
    ops per 16 weights; 1-bit, 15 ops (7 shifts, 8 masks) per 32 weights."""
    if engine == "tcgen05":
        return 7 / 16 if fmt == 0 else 15 / 32
    return (7 + 4 * rows) / 16 if fmt == 0 else (2 + rows) / 4


def alu_bound_us(fmt: int, m: int, weights: int, sm_mhz: float, engine: str = "dp4a") -> float:
    """Time the integer pipe needs for ``weights`` weights at m rows (passes of
    at most 4 rows on the dp4a kernel, 8 on the tensor-core kernel, each
    decoding every weight again) on every SM at ``sm_mhz``: a lower bound
    beside the HBM bound."""
    per = PASS_ROWS[engine]
    ops = 0.0
    for r0 in range(0, m, per):
        ops += int_ops_per_weight(fmt, min(per, m - r0), engine)
    return weights * ops / (SMS * INT_LANES_PER_CLK * sm_mhz * 1e6) * 1e6


def layer_bytes(hidden: int, inter: int, fmt: int) -> int:
    """Algorithmic bytes of one FFN layer: packed codes + fp16 scales of gate, up, down."""
    per = 4 if fmt == 0 else 8
    one = inter * hidden // per + 2 * inter * (hidden // BLOCK)
    return 3 * one


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# host-only sources that cannot change what a kernel does on the device
HOST_ONLY_SOURCES = ("tq_lifecycle.cu",)


def source_hash() -> str:
    """Hash of the sources the kernels are built from (recorded traffic is
    reported only while it matches)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ternary_weight_dp4a_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")) and f not in HOST_ONLY_SOURCES:
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary, or None
    if there is none or the kernel sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("source_hash") != source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        loaded = [r for r in rows if num(r[3]) is not None and num(r[3]) > 300.0] or rows
        sm_loaded = [num(r[1]) for r in loaded if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm_loaded or sm) if (sm_loaded or sm) else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": reasons, "samples": len(rows),
                "samples_under_load": len(loaded),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def dist_setup():
    """Rank, world size and local rank from the launcher's environment; a
    process group for N > 1 (NCCL on GPUs, gloo where CUDA is absent)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cuda = torch.cuda.is_available()
    if cuda:
        torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        if cuda:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_weights(fmt: int, sets: int, hidden: int, inter: int, seed_layer0: int = 0):
    """``sets`` independently seeded FFN layers, packed on the device."""
    import torch
    from ternary_weight_dp4a_gb300 import synth, tq
    layers = []
    for l in range(sets):
        mats = []
        for j, (n, k) in enumerate([(inter, hidden), (inter, hidden), (hidden, inter)]):
            codes, scales = synth.weight(n, k, fmt, synth.ffn_weight_seed(seed_layer0 + l, j),
                                         device="cuda")
            mats.append(tq.pack_weights(codes, fmt, scales))
            del codes
        layers.append(mats)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return layers


def _capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def time_steps(step_fns, steps: int, warmup: int, world: int, sampler_gpu=None):
    """Time exactly ``steps`` calls of the step functions in rotation
    (step_fns[0], step_fns[1], ..., wrapping), after exactly ``warmup``
    untimed ones: one CUDA graph per full pass over the list, replayed, and one
    of the first (steps mod n) functions for the remainder.  Returns (ms over
    the timed region between CUDA events on the replaying stream, clock
    summary sampled meanwhile)."""
    import torch
    n = len(step_fns)

    def part(r):
        def f():
            for fn in step_fns[:r]:
                fn()
        return f
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        part(n)()                       # eager warm-up of the code paths, outside capture
    torch.cuda.current_stream().wait_stream(s)
    graphs = {n: _capture(part(n))}
    for r in {steps % n, warmup % n} - {0}:
        graphs[r] = _capture(part(r))

    def run(count):
        for _ in range(count // n):
            graphs[n].replay()
        if count % n:
            graphs[count % n].replay()
    run(warmup)
    torch.cuda.synchronize()
    clocks = None
    ctx = ClockSampler(sampler_gpu) if sampler_gpu is not None else None
    if ctx:
        ctx.__enter__()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a ~100 us device sleep ahead of the start event: the host enqueues the
    # event and the replays meanwhile, so the timed region holds the steps
    # back to back and not the latency of the first launch after the sync
    torch.cuda._sleep(200000)
    start.record()
    run(steps)
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    if ctx:
        ctx.__exit__(None, None, None)
        clocks = ctx.summary()
    return start.elapsed_time(end), clocks


def set_engine(name: str) -> None:
    from ternary_weight_dp4a_gb300 import tq
    tq.set_engine(ENGINES[name])


# Standalone GEMV shapes (n, k): the tiny config, the FFN's gate/up and down
# matrices, the full-attention projections of the model family the pages
# describe (head_dim 256, 8:1 GQA with 2 KV heads: q 16 x 256 = 4096, k and
# v 2 x 256 = 512 each, o back to 5120), and a wide GEMV at LM-head scale
# (N = 131072; the pages give no vocabulary size).
GEMV_SHAPES = (("tiny_n512_k256", 512, 256), ("ffn_gate_n17408_k5120", 17408, 5120),
               ("ffn_down_n5120_k17408", 5120, 17408), ("attn_q_n4096_k5120", 4096, 5120),
               ("attn_kv_n512_k5120", 512, 5120), ("attn_o_n5120_k4096", 5120, 4096),
               ("wide_n131072_k5120", 131072, 5120))


def gemv_sweep(peak: float, fmt: int = 0, ms=(1, 8)):
    """tq_gemv time per call for each shape, row count and kernel, graph-replayed
    over enough independent weight copies to exceed the 129 MB L2 (at most 64
    copies: the smallest shapes stay partly L2-resident, said per entry)."""
    import torch
    from ternary_weight_dp4a_gb300 import synth, tq
    out = {}
    l2 = 129 * 2**20
    for name, n, k in GEMV_SHAPES:
        wbytes = n * k // (4 if fmt == 0 else 8) + 2 * n * (k // 128)
        copies = max(1, min(64, -(-2 * l2 // wbytes)))
        ws = []
        for c in range(copies):
            codes, scales = synth.weight(n, k, fmt, 7000 + c, device="cuda")
            ws.append(tq.pack_weights(codes, fmt, scales))
            del codes
        ent = {"n": n, "k": k, "weight_bytes": wbytes, "copies": copies,
               "l2_resident": copies * wbytes < l2}
        for m in ms:
            x = synth.activation(m, k, synth.SEED_ACT_BASE, 0.01, device="cuda")
            q, sc = tq.rotate_quant(x)
            y = torch.empty((m, n), dtype=torch.float32, device="cuda")
            wsp = tq.gemv_workspace(m, n, k)
            calls = max(copies, min(4000, 400 * copies // max(1, wbytes // 2**20 // 8 + 1)))
            for eng in ENGINES:
                set_engine(eng)
                fns = [lambda w=w: tq.gemv(w, q, sc, y=y, workspace=wsp) for w in ws]
                t, _ = time_steps(fns, calls, copies, 1)
                us = t * 1e3 / calls
                ent[f"m{m}_{eng}"] = {"us_per_call": round(us, 3), "weight_gbs": round(wbytes / us / 1e3, 1),
                                      "hbm_frac": round(wbytes / us / 1e3 / peak, 4)}
            set_engine("tcgen05")
        out[name] = ent
        del ws
        torch.cuda.empty_cache()
    set_engine("tcgen05")
    return out


def run_ours(args, rank, world, local):
    import torch
    from ternary_weight_dp4a_gb300 import build as tqbuild
    from ternary_weight_dp4a_gb300 import synth, tq

    tqbuild.build()
    tq.load()
    fmt = tq.FMT_TERNARY2
    peak, peak_kind = load_peaks()
    lb = layer_bytes(HIDDEN, INTER, fmt)
    layers = make_weights(fmt, N_SETS, HIDDEN, INTER)
    xs = {m: synth.activation(m, HIDDEN, synth.SEED_ACT_BASE, 0.01, device="cuda")
          for m in SWEEP_ROWS}
    ys = {m: torch.empty((m, HIDDEN), dtype=torch.float32, device="cuda") for m in xs}
    wss = {m: tq.ffn_workspace(m, HIDDEN, INTER) for m in xs}

    def step_fns(m):
        return [lambda g=g, u=u, d=d: tq.ffn_step(g, u, d, xs[m], y=ys[m], workspace=wss[m])
                for g, u, d in layers]

    # --- headline: m = 1, exactly K steps after exactly W warm-up steps, on
    #     the library's default kernel (dp4a: the faster, see the sweep) ---
    engine = "dp4a"
    set_engine(engine)
    ms, clocks = time_steps(step_fns(1), args.steps, args.warmup, world, sampler_gpu=local)
    ms = max_over_ranks(ms, world)
    ms_step = ms / args.steps
    value = world * lb / (ms_step * 1e-3) / 1e9
    # the integer-pipe bound uses the SM clock sampled under load (max clock if none)
    sm_mhz = float((clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or 2070.0)
    layer_w = 3 * HIDDEN * INTER

    # --- the same over a long run (a steady-state figure beside the K-step one) ---
    steady_steps = max(2000, args.steps)
    t_st, _ = time_steps(step_fns(1), steady_steps, N_SETS, world)
    t_st = max_over_ranks(t_st, world)
    steady = {"steps": steady_steps, "us_per_step": round(t_st * 1e3 / steady_steps, 3),
              "weight_gbs": round(lb / (t_st * 1e3 / steady_steps) / 1e3, 1),
              "hbm_frac": round(lb / (t_st * 1e3 / steady_steps) / 1e3 / peak, 4)}

    # --- batch sweep on both kernels: packed decode steps m = 1, 2, 4, 8 and
    #     verify-sized blocks m = 16, 32, 64 (same weights; one weight stream
    #     per pass of 8 rows on the tensor-core kernel, 4 on the dp4a kernel).
    #     This is the measured comparison that decides the kernel. ---
    sweep = {}
    for m in SWEEP_ROWS:
        for eng in ENGINES:
            set_engine(eng)
            passes = -(-m // PASS_ROWS[eng])
            n_steps = max(N_SETS, min(2000, 2000 // passes))
            t, _ = time_steps(step_fns(m), n_steps, N_SETS, world)
            t = max_over_ranks(t, world)
            us = t * 1e3 / n_steps
            ent = {"us_per_step": round(us, 3), "weight_gbs": round(lb / us / 1e3, 1),
                   "tokens_per_s": round(m * 1e6 / us, 1), "hbm_frac": round(lb / us / 1e3 / peak, 4),
                   "alu_bound_us": round(alu_bound_us(0, m, layer_w, sm_mhz, eng), 3), "steps": n_steps}
            ent["alu_frac"] = round(ent["alu_bound_us"] / us, 4)
            sweep[f"m{m}_{eng}"] = ent
    set_engine(engine)

    # --- roofline: at m = 1 a step is one launch of the step kernel (gate/up,
    #     SiLU*up, rotation of h, down), so the dominant kernel's average launch
    #     duration is the headline's timed region over its launches (CUDA
    #     events on the replaying stream).  The figure includes the gap between
    #     consecutive launches, so `achieved` is a lower bound.  Algorithmic
    #     bytes per launch: the layer's codes and scales, each read once. ---
    launches = args.steps                    # one kernel launch per m = 1 step
    k_us = ms * 1e3 / launches
    k_achieved = lb / (k_us * 1e-6) / 1e9
    kernel_name = ("tq::tc::tc_kernel<0,1> (tensor-core step: gate/up + SiLU*up + h rotation + down)"
                   if engine == "tcgen05" else
                   "tq::tq_kernel<0,1,false> (dp4a step: gate/up + SiLU*up + h rotation + down)")

    # --- end to end through the public API with pinned host buffers: every step
    #     copies x host->device, runs the step, copies y device->host.  The
    #     per-step sequence is captured as CUDA graphs and replayed. ---
    x_host = xs[1].cpu().pin_memory()
    y_host = torch.empty((1, HIDDEN), dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(xs[1])

    def e2e_fns():
        def one(g, u, d):
            x_dev.copy_(x_host, non_blocking=True)
            tq.ffn_step(g, u, d, x_dev, y=ys[1], workspace=wss[1])
            y_host.copy_(ys[1], non_blocking=True)
        return [lambda g=g, u=u, d=d: one(g, u, d) for g, u, d in layers]

    # at least 2000 steps (as the steady figure), whatever --steps is
    e2e_steps = max(2000, min(args.steps, 4000))
    t_e2e, _ = time_steps(e2e_fns(), e2e_steps, N_SETS, world)
    e2e_ms = max_over_ranks(t_e2e, world) / e2e_steps
    e2e_value = world * lb / (e2e_ms * 1e-3) / 1e9
    # the same with one eager Python call per step (host launch overhead included)
    fns = e2e_fns()
    for f in fns:
        f()
    torch.cuda.synchronize()
    eager_steps = N_SETS * (1000 // N_SETS)        # 1000 eager calls, whatever --steps is
    t0 = time.perf_counter()
    for i in range(eager_steps):
        fns[i % N_SETS]()
    torch.cuda.synchronize()
    eager_ms = (time.perf_counter() - t0) * 1e3 / eager_steps

    # --- the 64-layer stacks (2-bit m = 1; 1-bit m = 1, 2, 4, 8) on both kernels ---
    stacks = {}
    if not args.no_stack:
        del layers
        torch.cuda.empty_cache()
        for sfmt, sms in ((0, (1,)), (1, (1, 2, 4, 8))):
            stack_layers = make_weights(sfmt, 64, HIDDEN, INTER)
            sb = 64 * layer_bytes(HIDDEN, INTER, sfmt)
            for m in sms:
                xm = synth.activation(m, HIDDEN, synth.SEED_ACT_BASE, 0.01, device="cuda")
                ym = torch.empty((m, HIDDEN), dtype=torch.float32, device="cuda")
                wsm = tq.ffn_workspace(m, HIDDEN, INTER)
                for eng in ENGINES:
                    set_engine(eng)
                    fn = [lambda: tq.ffn_stack(stack_layers, xm, 1e-6, y=ym, workspace=wsm)]
                    t, _ = time_steps(fn, args.stack_reps, 2, world)
                    t = max_over_ranks(t, world)
                    us = t * 1e3 / args.stack_reps
                    alu = alu_bound_us(sfmt, m, 64 * layer_w, sm_mhz, eng)
                    stacks[f"{'ternary2' if sfmt == 0 else 'binary1'}_64L_m{m}_{eng}"] = {
                        "us_per_token_step": round(us, 2), "bytes_per_step": sb,
                        "weight_gbs": round(sb / us / 1e3, 1), "hbm_frac": round(sb / us / 1e3 / peak, 4),
                        "tokens_per_s": round(m * 1e6 / us, 1),
                        "alu_bound_us": round(alu, 2), "alu_frac": round(alu / us, 4)}
            del stack_layers
            torch.cuda.empty_cache()
        set_engine(engine)

    # --- standalone GEMV shapes (tq_gemv; weights rotated past L2 where they fit) ---
    gemv = {} if args.no_gemv else gemv_sweep(peak)
    set_engine(engine)

    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 6),
        "us_per_token_m1": round(ms_step * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8xternary2->f32",
        "data": "synthetic (seeded; ternary p0=0.4, fp16 scales U[0.01,0.05], bf16 N(0,1) x, 1% x10 outliers)",
        "config": {"workload": WORKLOAD, "hidden": HIDDEN, "intermediate": INTER, "m": 1,
                   "weight_format": "2-bit ternary, 128-blocks, fp16 scales",
                   "bytes_per_step": lb, "weight_sets": N_SETS, "kernel": engine,
                   "l2": f"{N_SETS} weight sets rotated ({N_SETS * lb / 1e6:.0f} MB > 129 MB L2)",
                   "timing": "CUDA graphs over the weight sets (a full pass, replayed, and the remainder), "
                             "exactly --steps timed after exactly --warmup; CUDA events",
                   "parallelism": f"replicas x{world}"},
        "hbm_frac": round(value / world / peak, 4),
        "steady": steady,
        "sweep": sweep,
        "roofline": {"bound": "hbm",
                     "kernel": kernel_name,
                     "achieved": round(k_achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(k_achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal": round(k_achieved / NOMINAL_HBM_GBS, 4),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "alu_bound_us": round(alu_bound_us(0, 1, layer_w, sm_mhz, engine), 3),
                     "bytes_per_launch": lb, "avg_launch_us": round(k_us, 3),
                     "launches_timed": launches,
                     "traffic": recorded_traffic(f"step_m1_{engine}")},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                "us_per_step": round(e2e_ms * 1e3, 3),
                "h2d_bytes_per_step": HIDDEN * 2, "d2h_bytes_per_step": HIDDEN * 4,
                "how": "pinned H2D copy + tq_ffn_step + D2H copy per step, graph-replayed",
                "eager_us_per_step": round(eager_ms * 1e3, 3)},
        "stack": stacks,
        "gemv": gemv,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    return result


def profile_steps(n: int, engine: str = "dp4a", m: int = 1, fmt: str = "2bit"):
    """n eager m-row steps over the weight sets (no timing, no JSON line)."""
    import torch
    from ternary_weight_dp4a_gb300 import build as tqbuild
    from ternary_weight_dp4a_gb300 import synth, tq
    tqbuild.build()
    tq.load()
    set_engine(engine)
    layers = make_weights(tq.FMT_TERNARY2 if fmt == "2bit" else tq.FMT_BINARY1, N_SETS, HIDDEN, INTER)
    x = synth.activation(m, HIDDEN, synth.SEED_ACT_BASE, 0.01, device="cuda")
    y = torch.empty((m, HIDDEN), dtype=torch.float32, device="cuda")
    ws = tq.ffn_workspace(m, HIDDEN, INTER)
    for i in range(n):
        g, u, d = layers[i % N_SETS]
        tq.ffn_step(g, u, d, x, y=y, workspace=ws)
    torch.cuda.synchronize()


def profile_gemv(n: int, engine: str = "dp4a"):
    """n eager m = 1 tq_gemv calls on the 17408 x 5120 gate shape, rotating
    over the weight sets' gate matrices (no timing, no JSON line)."""
    import torch
    from ternary_weight_dp4a_gb300 import build as tqbuild
    from ternary_weight_dp4a_gb300 import synth, tq
    tqbuild.build()
    tq.load()
    set_engine(engine)
    layers = make_weights(tq.FMT_TERNARY2, N_SETS, HIDDEN, INTER)
    x = synth.activation(1, HIDDEN, synth.SEED_ACT_BASE, 0.01, device="cuda")
    q, s = tq.rotate_quant(x)
    y = torch.empty((1, INTER), dtype=torch.float32, device="cuda")
    wsp = tq.gemv_workspace(1, INTER, HIDDEN)
    for i in range(n):
        tq.gemv(layers[i % N_SETS][0], q, s, y=y, workspace=wsp)
    torch.cuda.synchronize()


def host_info() -> dict:
    """Core count and CPU model of this host, read at run time."""
    import platform
    import subprocess
    model = ""
    try:
        for line in open("/proc/cpuinfo"):
            key, _, val = line.partition(":")
            if key.strip().lower() in ("model name", "cpu model"):
                model = val.strip()
                break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


def _time_calls(fn, budget_s: float):
    """Seconds per call of fn over about budget_s seconds (at least one call)."""
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el / n * (n + 1) > 2 * budget_s:
            return el / n, n


def _ffn_mats_host(fmt: int, layer: int = 0):
    from oracle import oracle
    from ternary_weight_dp4a_gb300 import synth
    mats = []
    for j, (n, k) in enumerate([(INTER, HIDDEN), (INTER, HIDDEN), (HIDDEN, INTER)]):
        codes, scales = synth.weight(n, k, fmt, synth.ffn_weight_seed(layer, j))
        mats.extend([oracle.pack(codes, fmt), scales])
        del codes
    return mats


def cpu_oracle_baseline(budget_s: float, fmt: int = 0, m: int = 1, extras: bool = False):
    """Time the oracle's FFN step on the host cores on a bounded sample: as many
    full layer steps (m rows) as fit in about ``budget_s`` seconds.  With
    ``extras`` also: the same step on 1 and on cores - 2 threads, the tiny GEMV,
    and per-token estimates of the 64-layer stacks from a sample of layers."""
    from oracle import oracle
    from ternary_weight_dp4a_gb300 import synth
    oracle.build()
    mats = _ffn_mats_host(fmt)
    x = synth.activation(m, HIDDEN, synth.SEED_ACT_BASE, 0.01)
    lb = layer_bytes(HIDDEN, INTER, fmt)
    threads = oracle.get_threads()
    sec, steps = _time_calls(lambda: oracle.ffn_step(*mats, fmt, HIDDEN, INTER, x), budget_s)
    out = {"value": round(lb / sec / 1e9, 4), "unit": "GB/s",
           "cores": threads, "kind": "oracle",
           "sample": f"{steps} full FFN layer step(s), m={m}, hidden {HIDDEN}, "
                     f"intermediate {INTER}, 2-bit; {sec * steps:.1f} s",
           "us_per_step": round(sec * 1e6, 1)}
    if not extras:
        return out
    out["host"] = host_info()
    # the same step on 1 thread, cores - 2 threads (cores left to the OS) and all
    scan = []
    for t in sorted({1, max(1, threads - 2), threads}):
        oracle.set_threads(t)
        st, n = _time_calls(lambda: oracle.ffn_step(*mats, fmt, HIDDEN, INTER, x),
                            min(3.0, budget_s / 3))
        scan.append({"threads": t, "us_per_step": round(st * 1e6, 1),
                     "weight_gbs": round(lb / st / 1e9, 4), "steps": n})
    oracle.set_threads(threads)
    out["threads_scan"] = scan
    configs = {}
    # tiny GEMV, K = 256, N = 512 (2-bit)
    codes, scales = synth.weight(512, 256, 0, synth.SEED_TINY_WEIGHT)
    packed = oracle.pack(codes, 0)
    q, s = oracle.rotate_quant(synth.activation(1, 256, synth.SEED_ACT_BASE, 0.0))
    st, n = _time_calls(lambda: oracle.gemv(packed, scales, 0, 512, 256, q, s), 0.5)
    tb = 512 * 256 // 4 + 2 * 512 * 2
    configs["tiny_gemv_n512_k256"] = {"us_per_call": round(st * 1e6, 2), "weight_gbs": round(tb / st / 1e9, 4),
                                      "sample": f"{n} calls"}
    # 64-layer stacks: one layer (step + RMS-normalise) timed, times 64
    for sfmt, ms in ((0, (1,)), (1, (1, 2, 4, 8))):
        smats = mats if sfmt == fmt else _ffn_mats_host(sfmt)
        for mm in ms:
            xm = synth.activation(mm, HIDDEN, synth.SEED_ACT_BASE, 0.01)

            def layer():
                y = oracle.ffn_step(*smats, sfmt, HIDDEN, INTER, xm)["y"]
                oracle.rmsnorm_bf16(y, 1e-6)
            st, n = _time_calls(layer, 0.5)
            sb = 64 * layer_bytes(HIDDEN, INTER, sfmt)
            configs[f"{'ternary2' if sfmt == 0 else 'binary1'}_64L_m{mm}"] = {
                "us_per_token_step": round(64 * st * 1e6, 1), "weight_gbs": round(sb / (64 * st) / 1e9, 4),
                "sample": f"{n} layer(s) timed, x 64"}
        del smats
    out["configs"] = configs
    return out


def reference_arm(steps: int, warmup: int, budget_s: float = 120.0):
    """The oracle as it stands, on the host cores: exactly ``warmup`` untimed
    and ``steps`` timed steps of the headline workload.  A step is the full FFN
    layer step when ``steps`` of them fit in about ``budget_s`` seconds, else
    the same fraction of every matrix's rows (rotate x, gate and up rows, SiLU
    times up, down rows on the h of one full step taken first), so that any
    --steps ends within a few minutes.  GB/s = weight bytes the timed steps
    read / their time."""
    from oracle import oracle
    from ternary_weight_dp4a_gb300 import synth
    oracle.build()
    mats = _ffn_mats_host(0)
    x = synth.activation(1, HIDDEN, synth.SEED_ACT_BASE, 0.01)
    t0 = time.perf_counter()
    full = oracle.ffn_step(*mats, 0, HIDDEN, INTER, x)
    t_full = time.perf_counter() - t0
    frac = min(1.0, budget_s / max(steps, 1) / t_full)
    if frac >= 1.0:
        def step():
            oracle.ffn_step(*mats, 0, HIDDEN, INTER, x)
        step_bytes = layer_bytes(HIDDEN, INTER, 0)
        sample = "full FFN layer steps"
    else:
        rg, rd = max(1, int(INTER * frac)), max(1, int(HIDDEN * frac))
        gate, gate_s, up, up_s, down, down_s = mats
        g_p, g_s, u_p, u_s = gate[:rg], gate_s[:rg], up[:rg], up_s[:rg]
        d_p, d_s = down[:rd], down_s[:rd]

        def step():
            q, s = oracle.rotate_quant(x)
            g = oracle.gemv(g_p, g_s, 0, rg, HIDDEN, q, s)
            u = oracle.gemv(u_p, u_s, 0, rg, HIDDEN, q, s)
            oracle.silu_mul_bf16(g, u)
            oracle.gemv(d_p, d_s, 0, rd, INTER, full["qh"], full["sh"])
        step_bytes = 2 * rg * (HIDDEN // 4 + 2 * HIDDEN // 128) + rd * (INTER // 4 + 2 * INTER // 128)
        sample = (f"{rg} of {INTER} gate/up rows and {rd} of {HIDDEN} down rows per step "
                  f"(the same fraction {frac:.4f} of every matrix)")
    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    sec = (time.perf_counter() - t0) / max(steps, 1)
    return {"value": round(step_bytes / sec / 1e9, 4), "unit": "GB/s", "cores": oracle.get_threads(),
            "kind": "oracle", "sample": f"{steps} timed steps after {warmup} untimed: {sample}, m=1, "
                                        f"hidden {HIDDEN}, intermediate {INTER}, 2-bit",
            "us_per_step": round(sec * 1e6, 1), "bytes_per_step": step_bytes}


def run_probe(name: str):
    """Build csrc/probes/<name>.cu for sm_103a into a temporary directory and
    run it.  tq_mma_rate: time per tcgen05.mma (kind::f8f6f4, M = 128,
    K = 32) at N = 16..256 with A in tensor or shared memory.  tq_lut_rate:
    weights per cycle per SM of the 1-bit dp4a inner loop against 16- and
    256-entry lookup tables."""
    import shutil
    import subprocess
    import tempfile
    src = os.path.join(ROOT, "ternary_weight_dp4a_gb300", "csrc", "probes", name + ".cu")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, name)
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        print(r.stdout, end="")
        if r.returncode != 0:
            print(r.stderr, end="")
            raise SystemExit(r.returncode)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--stack-reps", type=int, default=100)
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--no-gemv", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many eager steps of the headline workload and exit "
                         "(a small, untimed case for a profiler to capture)")
    ap.add_argument("--profile-gemv", type=int, default=0,
                    help="run this many eager m = 1 GEMVs on the 17408 x 5120 gate shape and exit")
    ap.add_argument("--profile-engine", choices=list(ENGINES), default="dp4a",
                    help="kernel for --profile-steps / --profile-gemv (default: the default engine's)")
    ap.add_argument("--profile-rows", type=int, default=1, help="rows per step for --profile-steps")
    ap.add_argument("--profile-fmt", choices=["2bit", "1bit"], default="2bit",
                    help="weight format for --profile-steps")
    ap.add_argument("--probe-mma-rate", action="store_true",
                    help="build and run the tcgen05.mma throughput probe (csrc/probes/tq_mma_rate.cu) and exit")
    ap.add_argument("--probe-lut-rate", action="store_true",
                    help="build and run the 1-bit dp4a vs lookup-table probe (csrc/probes/tq_lut_rate.cu) and exit")
    args = ap.parse_args()
    if args.probe_mma_rate:
        run_probe("tq_mma_rate")
        return
    if args.probe_lut_rate:
        run_probe("tq_lut_rate")
        return
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        # the reference arm is the CPU oracle, timed on rank 0's host cores only
        if rank != 0:
            return
        base = reference_arm(args.steps, args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": base["value"], "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(base["us_per_step"] / 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int8xternary2->f32",
                "data": "synthetic (seeded)",
                "config": {"workload": WORKLOAD, "hidden": HIDDEN, "intermediate": INTER, "m": 1},
                "cpu_baseline": base,
                "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    rank, world, local = dist_setup()
    if args.profile_steps > 0:
        profile_steps(args.profile_steps, args.profile_engine, args.profile_rows, args.profile_fmt)
        return
    if args.profile_gemv > 0:
        profile_gemv(args.profile_gemv, args.profile_engine)
        return
    result = run_ours(args, rank, world, local)
    if rank == 0:
        result["cpu_baseline"] = cpu_oracle_baseline(args.cpu_budget, extras=True)
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
