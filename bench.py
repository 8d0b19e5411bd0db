"""Benchmark of the fp8 MoE decode / speculative-verify layer on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload verify8]
                [--impl ours|reference]

One step = one pass of the whole layer (route, union, dispatch, gate/up GEMM,
down GEMM, combine) over one batch of seeded synthetic inputs already
resident in HBM: one moe_layer call, its kernels chained by programmatic
dependent launch, CUDA events at the step boundaries on the launching stream.
L2 is flushed (a 256 MB write) before every step, outside the events.
`value` = rows processed by all ranks / max over ranks of the step time.  A
second pass runs the step-by-step entry points with an event between every two
kernels: it gives each kernel's device time (`phase_ms`) and the roofline of
the dominant kernel.  Under torchrun every rank runs its own replica (the
layer has no exchange step on one GPU): scaling "weak".

`e2e` measures the same metric through moe_layer with host buffers: per step
the rows go from pinned host memory to the device, the layer runs, and the
bf16 output comes back to pinned host memory; `e2e.graph_replay` is the same
step with moe_layer captured once in a CUDA graph and replayed.

`--impl reference` times the CPU oracle (the plain restatement the tests
check the kernels against) on the host cores, on a bounded sample of the same
workload, and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = ("MoE-layer rows/s and achieved HBM GB/s (% of 8 TB/s) at 8-row verify; "
          "fp8 TFLOPS at 4096")
PHASES = ["router", "union", "dispatch", "ffn", "combine"]


def kernels_per_step(R: int) -> int:
    """Kernels of one moe_layer call: router logits, selection + union (one
    kernel up to 64 rows, two above), dispatch, expert GEMMs (one fused launch
    up to 64 rows, gate/up and down above), combine."""
    return 5 if R <= 64 else 7
# DRAM bytes (read + write) of the fused expert GEMM per algorithmic byte at
# the 16-row tile (calls of up to 64 rows), from one ncu capture of that kernel
# at 8 rows on 32 experts of the same shape (dram__bytes_read.sum +
# dram__bytes_write.sum over the launch's algorithmic bytes); traffic grows
# with the weight bytes streamed, so a full launch's traffic is this ratio
# times its algorithmic bytes.  The capture holds only for the kernel source it
# was taken on: `kernel_sha16` is the hash of that source (ffn_source_sha16()),
# and a bench run on other source reports the traffic as null.
FFN_TRAFFIC = {"per_alg_byte": 1.0031, "profile": "profiles/ffn_fused_profile8.md",
               "kernel_sha16": "51438ff6819ee307"}
FFN_SOURCES = ("moe_speculative_verify_gb300/csrc/ffn.cu",
               "moe_speculative_verify_gb300/csrc/common.cuh")
HOST_AHEAD_CYCLES = 400_000   # GPU sleep before each step so the host enqueues it whole
FLUSH_BYTES = 256 << 20       # > 129 MB L2


def ffn_source_sha16() -> str:
    """Hash of the expert GEMM's source files (what a profile was taken on)."""
    h = hashlib.sha256()
    for f in FFN_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def peaks():
    """Roofline denominators: measured HBM copy GB/s and dense bf16 TFLOP/s
    (burst); fp8 dense is taken as 2x bf16, the nominal ratio of the two
    tensor rates (4.5 vs 2.25 PFLOP/s)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        out = {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
               "source": "measured"}
    else:
        out = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}
    out["fp8_tflops"] = 2.0 * out["bf16_tflops"]
    return out


def fp8_roofline(flops: float, nbytes: float, ms: float, pk: dict) -> dict:
    """fp8 tensor-pipe figures of a phase: achieved TFLOP/s, its fraction of
    the fp8 dense peak, and its fraction of the intensity-bound ceiling
    min(peak, AI * HBM bandwidth) with AI = flops / algorithmic bytes."""
    tf = flops / (ms / 1e3) / 1e12
    ai = flops / nbytes
    ceiling = min(pk["fp8_tflops"], ai * pk["hbm_gbs"] / 1e3)
    return {"tflops": round(tf, 1), "fp8_peak_tflops": round(pk["fp8_tflops"], 1),
            "fp8_frac_of_peak": round(tf / pk["fp8_tflops"], 4),
            "ai_flop_per_byte": round(ai, 1), "ai_ceiling_tflops": round(ceiling, 1),
            "frac_of_ai_ceiling": round(tf / ceiling, 4)}


# ------------------------------------------------------------------ ranks --
def max_over_ranks(x: float) -> float:
    """Largest value of x over the ranks of the default process group (x itself
    without one).  The job's step time is the slowest replica's."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank: int, world: int, step_ms_max: float) -> float:
    """Whole-job throughput: every replica processes rows_per_rank rows per step."""
    return world * rows_per_rank / (step_ms_max / 1e3)


# ----------------------------------------------------------- algorithmics --
def algorithmic(wl, ids: np.ndarray, valid: np.ndarray) -> dict:
    """Bytes each kernel must move at minimum and the layer's fp8 MMA flops."""
    s = wl.shape
    H, I, E, K, S = s.hidden, s.inter, s.n_experts, s.topk, s.n_shared
    R = wl.rows
    Rv = int(valid.sum())
    U = len(np.unique(ids[ids >= 0]))
    T = Rv * (K + S)
    ent = U + (S if Rv else 0)
    w_gu = ent * (2 * I * H + 2 * (I // 128) * (H // 128) * 4)
    w_dn = ent * (H * I + (H // 128) * (I // 128) * 4)
    b = {
        "router": E * H * 4 + R * H * 2 + E * 4 + 2 * R * E * 4 + R * K * 8,
        "union": R * K * 4 + (R * (K + S) * 2) * 4,
        "dispatch": Rv * H * 2 + T * H + T * (H // 128) * 4,
        "ffn": (w_gu + T * H + T * (H // 128) * 4 + T * I + T * (I // 128) * 4) +
               (w_dn + T * I + T * (I // 128) * 4 + T * H * 4),
        "combine": Rv * (K + S) * H * 4 + Rv * K * 4 + R * H * 2,
    }
    flops = 2 * T * (2 * I * H) + 2 * T * (H * I)
    return {"bytes": b, "total_bytes": sum(b.values()), "flops": flops, "U": U, "T": T,
            "Rv": Rv, "weights_bytes": w_gu + w_dn}


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi samples (every 20 ms) of SM clock, power and throttle reasons.

    Started before the warm-up; stop(t0, t1) keeps the samples taken inside the
    timed region [t0, t1] (wall clock), widening the window symmetrically until
    it holds at least 3 samples when the region is shorter than the sampling
    period, and reports the window used."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", gpu_index, "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]),
                             [n for n, v in zip(names, parts[6:10]) if v.lower() == "active"]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        half = 0.0
        while True:
            sel = [r for r in rows if t0 - half <= r[0] <= t1 + half]
            if len(sel) >= 3 or half > 5.0:
                break
            half += 0.02
        if not sel:
            sel = rows
        reasons = sorted({n for r in sel for n in r[4]})
        return {"sm_mhz": statistics.median(r[1] for r in sel),
                "sm_max_mhz": max(r[2] for r in sel),
                "power_w_max": max(r[3] for r in sel), "samples": len(sel),
                "window_s": round((t1 - t0) + 2 * half, 3), "reasons": reasons}


# ------------------------------------------------------------------ oracle --
def oracle_baseline(wl, t_dev: dict, target_s: float = 12.0) -> dict:
    """The CPU oracle, as it stands, on a bounded sample of the workload's rows."""
    import oracle
    host = {k: (v.detach().cpu().view(torch.int16).numpy().view(np.uint16)
                if v.dtype == torch.bfloat16 else v.detach().cpu().numpy())
            for k, v in t_dev.items()}
    cores = oracle.num_threads()
    valid = np.nonzero(host["row_valid"])[0]
    t0 = time.perf_counter()
    oracle.moe_layer(wl.shape, host, rows=valid[:1])
    one = max(time.perf_counter() - t0, 1e-3)
    # about target_s of CPU work: the valid rows, cycled when there are fewer
    n = int(max(1, target_s / one))
    rows = np.resize(valid, n) if n > len(valid) else \
        valid[np.linspace(0, len(valid) - 1, n).astype(int)]
    t0 = time.perf_counter()
    oracle.moe_layer(wl.shape, host, rows=rows)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} row evaluations over the {len(valid)} valid rows of {wl.name} "
                      f"(cycled), full layer per row (routing + {wl.shape.topk} routed + "
                      f"{wl.shape.n_shared} shared experts), {dt:.1f} s"}


def run_reference(args, wl) -> None:
    """Reference arm: the CPU oracle on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    t0 = time.perf_counter()
    # inputs only: generated where it is quick, then handed to the oracle on the host
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    host = synth.to_numpy(synth.make_layer(wl, device=gen_dev))
    if gen_dev == "cuda":
        torch.cuda.empty_cache()
    valid = np.nonzero(host["row_valid"])[0]
    cores = oracle.num_threads()
    # each step: a bounded sample of rows, sized so the whole run takes about 2 minutes
    per_step = max(1.0, min(10.0, 120.0 / max(1, args.steps)))
    t1 = time.perf_counter()
    oracle.moe_layer(wl.shape, host, rows=valid[:1])
    one = max(time.perf_counter() - t1, 1e-3)
    n = int(max(1, per_step / one))
    rows = np.resize(valid, n)          # the valid rows, cycled when there are fewer
    if args.warmup > 0:
        oracle.moe_layer(wl.shape, host, rows=rows[:1])
    times = []
    for _ in range(args.steps):
        t1 = time.perf_counter()
        oracle.moe_layer(wl.shape, host, rows=rows)
        times.append(time.perf_counter() - t1)
    step = statistics.mean(times)
    value = n / step
    line = {"metric": METRIC, "value": value, "unit": "rows/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp32 dequant / fp64 accumulate (CPU)",
            "data": "synthetic (seeded)",
            "config": {"workload": wl.name, "rows": wl.rows, "sample_rows": n},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} row evaluations per step over the "
                                       f"{len(valid)} valid rows of {wl.name} (cycled)"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "setup_s": round(t1 - t0, 1)}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ extras --
def measure_extras(m, cfg, wl, bufs, dev, steps) -> dict:
    """Greedy verify of one 8-row span over a GLM-sized vocabulary, and the
    combine fused with the residual add + RMSNorm against the plain combine,
    on the verify step's own expert outputs."""
    out = {}
    stream = torch.cuda.current_stream()
    flush = bufs["flush"]
    R, H = wl.rows, wl.shape.hidden

    def timed(fn):
        ts = []
        for _ in range(max(3, steps)):
            flush.zero_()
            torch.cuda._sleep(HOST_AHEAD_CYCLES // 4)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.mean(ts[1:])

    V = 151552
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    logits = torch.randn((8, V), generator=g, device=dev).to(torch.bfloat16)
    draft = torch.randint(0, V, (8,), generator=g, device=dev, dtype=torch.int32)
    nd = torch.full((1,), 7, dtype=torch.int32, device=dev)
    am = torch.empty(8, dtype=torch.int32, device=dev)
    acc = torch.empty(1, dtype=torch.int32, device=dev)
    toks = torch.empty(8, dtype=torch.int32, device=dev)
    ms = timed(lambda: m.moe_greedy_verify(logits, draft, nd, am, acc, toks))
    nbytes = logits.numel() * 2
    out["greedy_verify"] = {"rows": 8, "vocab": V, "dtype": "bf16", "us": round(ms * 1e3, 2),
                            "gbs": round(nbytes / (ms / 1e3) / 1e9, 1)}
    residual = torch.randn((R, H), generator=g, device=dev).to(torch.bfloat16)
    gamma = torch.rand((H,), generator=g, device=dev) + 0.5
    ro = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    no = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    ms_plain = timed(lambda: m.moe_combine(cfg, bufs["y_slots"], bufs["y_sh"], bufs["wts"],
                                           bufs["ub"], y))
    ms_fused = timed(lambda: m.moe_combine_add_rmsnorm(cfg, bufs["y_slots"], bufs["y_sh"],
                                                       bufs["wts"], bufs["ub"], residual, gamma,
                                                       1e-5, ro, no))
    K, S = wl.shape.topk, wl.shape.n_shared
    b_fused = R * (K + S) * H * 4 + R * H * 2 * 3 + H * 4
    out["combine_add_rmsnorm"] = {"rows": R, "us": round(ms_fused * 1e3, 2),
                                  "plain_combine_us": round(ms_plain * 1e3, 2),
                                  "gbs": round(b_fused / (ms_fused / 1e3) / 1e9, 1)}
    return out


def measure_w8a16(m, cfg, W, wl, dev, steps, flush) -> dict:
    """The layer at 1, 2, 4 and 8 rows with the w8a16 expert FFNs against the
    fp8 ones (moe_layer_w8a16 vs moe_layer), same weights and routing mix,
    L2 flushed before every call; microseconds per call."""
    stream = torch.cuda.current_stream()
    out = {}
    for R in (1, 2, 4, 8):
        wr = synth.Workload(f"{wl.name}_r{R}", wl.shape, rows=R, routing=wl.routing,
                            hot_per_group=wl.hot_per_group, hot_delta=wl.hot_delta)
        ri = synth.make_router_inputs(wr, device=dev)
        ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
        y = torch.empty((R, wl.shape.hidden), dtype=torch.bfloat16, device=dev)
        ids = torch.empty((R, wl.shape.topk), dtype=torch.int32, device=dev)
        res = {}
        for name, fn in (("fp8", m.moe_layer), ("w8a16", m.moe_layer_w8a16)):
            ts = []
            for i in range(max(3, steps) + 3):
                flush.zero_()
                torch.cuda._sleep(HOST_AHEAD_CYCLES // 4)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn(cfg, ri["x"], ri["wr"], ri["bias"], W, ri["row_valid"], y, ws, topk_ids=ids)
                b.record(stream)
                b.synchronize()
                if i >= 3:
                    ts.append(a.elapsed_time(b))
            assert m.moe_get_device_error(ws) == 0
            res[name] = statistics.mean(ts)
        U = len(np.unique(ids.cpu().numpy()))
        nbytes = (U + wl.shape.n_shared) * 3 * wl.shape.hidden * wl.shape.inter
        out[str(R)] = {"distinct_experts": U, "fp8_us": round(res["fp8"] * 1e3, 2),
                       "w8a16_us": round(res["w8a16"] * 1e3, 2),
                       "w8a16_weight_gbs": round(nbytes / (res["w8a16"] / 1e3) / 1e9, 1),
                       "w8a16_over_fp8": round(res["w8a16"] / res["fp8"], 3)}
    return out


# -------------------------------------------------------------------- ours --
def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="verify8", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", default="verify64,decode512,prefill4096",
                    help="other workloads measured on the same weights (summary only); "
                         "\"none\" for none")
    args = ap.parse_args()
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import moe_speculative_verify_gb300 as m
    m.build()
    m.load()

    # row-major codes (the oracle's layout), and the same codes in 16 KB
    # 128x128 blocks: the layout the layer is given (its GEMMs then read each
    # weight stream sequentially)
    weights = synth.make_expert_weights(wl, device=dev)
    tiled = m.tile_weights(weights)
    W = m.Weights.from_tensors(tiled, m.LAYOUT_TILED)
    W_rm = m.Weights.from_tensors(weights)
    cfg = m.Config.from_shape(wl.shape)
    pk = peaks()

    def measure(wl_m, steps, warmup, record_clocks):
        R = wl_m.rows
        s = wl_m.shape
        ri = synth.make_router_inputs(wl_m, device=dev)
        ids = torch.empty((R, s.topk), dtype=torch.int32, device=dev)
        wts = torch.empty((R, s.topk), dtype=torch.float32, device=dev)
        logits = torch.empty((R, s.n_experts), dtype=torch.float32, device=dev)
        ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
        ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
        y_slots = torch.empty((R * s.topk, s.hidden), dtype=torch.float32, device=dev)
        y_sh = torch.empty((R, s.hidden), dtype=torch.float32, device=dev)
        out = torch.empty((R, s.hidden), dtype=torch.bfloat16, device=dev)
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream()

        def step(ev=None):
            def mark(i):
                if ev is not None:
                    ev[i].record(stream)
            mark(0)
            m.moe_route(cfg, ri["x"], ri["wr"], ri["bias"], ri["row_valid"], ids, wts, logits)
            mark(1)
            m.moe_build_union(cfg, ids, ub)
            mark(2)
            m.moe_dispatch(cfg, ri["x"], ub, ws)
            mark(3)
            # the GEMM launches moe_layer makes at this row count
            if R <= 64:
                m.moe_expert_gemms_fp8(cfg, W, ub, R, y_slots, y_sh, ws)
            else:
                m.moe_gate_up_fp8(cfg, W, ub, R, ws)
                m.moe_down_fp8(cfg, W, ub, R, y_slots, y_sh, ws)
            mark(4)
            m.moe_combine(cfg, y_slots, y_sh, wts, ub, out)
            mark(5)

        lws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)

        def layer_step():
            # the product call: one moe_layer (selection and union in one
            # kernel at R <= 64)
            m.moe_layer(cfg, ri["x"], ri["wr"], ri["bias"], W, ri["row_valid"], out, lws,
                        topk_ids=ids, topk_w=wts)

        def prologue():
            # flush L2, then keep the GPU busy while the host enqueues the step
            flush.zero_()
            torch.cuda._sleep(HOST_AHEAD_CYCLES)

        clk = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
            if record_clocks else None
        for _ in range(warmup):
            prologue()
            layer_step()
        for _ in range(warmup):
            prologue()
            step()
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        assert m.moe_get_device_error(lws) == 0
        # timed region: events at the step boundaries only, so consecutive
        # kernels keep overlapping their launch with the predecessor's tail
        ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        t_start = time.time()
        torch.cuda.nvtx.range_push(f"timed_{wl_m.name}")
        for i in range(steps):
            prologue()
            ev0[i].record(stream)
            layer_step()
            ev1[i].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        t_end = time.time()
        if world > 1:
            torch.distributed.barrier()
        clocks = clk.stop(t_start, t_end) if clk else None
        err = m.moe_get_device_error(lws)
        assert err == 0, err
        tot = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
        out_layer = out.clone()
        # breakdown pass: an event between every two kernels (this serialises
        # the kernel boundaries, so it is reported beside, not as, the step)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        for i in range(steps):
            prologue()
            step(evs[i])
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        stepwise_same = bool(torch.equal(out, out_layer))
        ph = {p: [] for p in PHASES}
        for e in evs:
            for i, p in enumerate(PHASES):
                ph[p].append(e[i].elapsed_time(e[i + 1]))
        alg = algorithmic(wl_m, ids.cpu().numpy(), ri["row_valid"].cpu().numpy())
        return {"ri": ri, "phase_ms": {p: statistics.mean(v) for p, v in ph.items()},
                "step_ms": statistics.mean(tot), "step_ms_min": min(tot), "wall_s": wall,
                "alg": alg, "clocks": clocks, "out": out_layer, "stepwise_same": stepwise_same,
                "bufs": {"y_slots": y_slots, "y_sh": y_sh, "wts": wts, "ub": ub, "flush": flush}}

    res = measure(wl, args.steps, max(args.warmup, 3), True)
    step_ms = max_over_ranks(res["step_ms"])
    alg = res["alg"]
    R = wl.rows
    value = job_rows_per_s(R, world, step_ms)
    layer_gbs = alg["total_bytes"] / (step_ms / 1e3) / 1e9
    tflops = alg["flops"] / (step_ms / 1e3) / 1e12

    # roofline of the dominant kernel (the expert GEMMs: all weight bytes)
    dom = max(res["phase_ms"], key=res["phase_ms"].get)
    dom_ms = res["phase_ms"][dom]
    dom_bytes = alg["bytes"][dom]
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    ffn_name = ("ffn_kernel<NT, fused> (gate/up + SiLU*mul + down)" if R <= 64 else
                "ffn_kernel<NT, gate/up> + ffn_kernel<NT, down> (the two launches together)")
    sha = ffn_source_sha16()
    traffic, traffic_src = None, None
    if dom == "ffn" and R <= 64:
        if FFN_TRAFFIC["kernel_sha16"] == sha:
            traffic = round(dom_bytes * FFN_TRAFFIC["per_alg_byte"])
            traffic_src = (f"{FFN_TRAFFIC['profile']}: ncu DRAM read + write per algorithmic "
                           f"byte of the same kernel and tile at 8 rows on 32 experts "
                           f"({FFN_TRAFFIC['per_alg_byte']}), times this launch's algorithmic "
                           f"bytes; kernel source {sha}")
        else:
            traffic_src = (f"null: the kernel source ({sha}) differs from the one profiled in "
                           f"{FFN_TRAFFIC['profile']} ({FFN_TRAFFIC['kernel_sha16']})")
    roofline = {"kernel": {"ffn": ffn_name}
                .get(dom, dom), "bound": "hbm", "achieved": round(achieved, 1),
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": traffic, "traffic_source": traffic_src,
                "peak_source": pk["source"], "kernel_source_sha16": sha,
                "algorithmic_bytes_per_launch": dom_bytes}

    extra = {}
    if rank == 0 and args.extra:
        for name in [n for n in args.extra.split(",") if n not in ("", "none", wl.name)]:
            wl2 = synth.WORKLOADS[name]
            r2 = measure(wl2, max(20, args.steps), 3, False)
            a2 = r2["alg"]
            ffn_ms = r2["phase_ms"]["ffn"]
            extra[name] = {
                "rows": wl2.rows, "rows_per_s": round(wl2.rows / (r2["step_ms"] / 1e3), 1),
                "ms_per_step": round(r2["step_ms"], 4), "steps": max(20, args.steps),
                "hbm_gbs": round(a2["total_bytes"] / (r2["step_ms"] / 1e3) / 1e9, 1),
                "hbm_frac_of_measured": round(a2["total_bytes"] / (r2["step_ms"] / 1e3) / 1e9
                                              / pk["hbm_gbs"], 4),
                "fp8_tflops": round(a2["flops"] / (r2["step_ms"] / 1e3) / 1e12, 1),
                "distinct_experts": a2["U"],
                "phase_ms": {k: round(v, 4) for k, v in r2["phase_ms"].items()},
                "ffn_gbs": round(a2["bytes"]["ffn"] / (ffn_ms / 1e3) / 1e9, 1),
                # fp8 MMA throughput of the expert GEMMs alone (their event-timed
                # phase) and of the whole step, against the fp8 dense peak
                # (2 x the measured bf16 burst, the nominal fp8 : bf16 ratio)
                # and against min(peak, AI x measured HBM)
                "ffn_fp8": fp8_roofline(a2["flops"], a2["bytes"]["ffn"], ffn_ms, pk),
                "step_fp8": fp8_roofline(a2["flops"], a2["total_bytes"], r2["step_ms"], pk)}
            del r2

    # the verify-step extras, each timed alone with events on its stream
    if rank == 0:
        extra.update(measure_extras(m, cfg, wl, res["bufs"], dev, args.steps))
        if wl.rows <= m.W8A16_MAX_ROWS:
            extra["w8a16_vs_fp8"] = measure_w8a16(m, cfg, W, wl, dev, args.steps,
                                                  res["bufs"]["flush"])

    # end to end through moe_layer with host buffers
    import moe_speculative_verify_gb300 as m2
    ri = res["ri"]
    x_host = ri["x"].cpu().pin_memory()
    v_host = ri["row_valid"].cpu().pin_memory()
    out_host = torch.empty((R, wl.shape.hidden), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(ri["x"])
    v_dev = torch.empty_like(ri["row_valid"])
    out_dev = torch.empty((R, wl.shape.hidden), dtype=torch.bfloat16, device=dev)
    lws = torch.zeros(m2.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        v_dev.copy_(v_host, non_blocking=True)
        m2.moe_layer(cfg, x_dev, ri["wr"], ri["bias"], W, v_dev, out_dev, lws)
        out_host.copy_(out_dev, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        flush.zero_()
        e2e_step()
    e2e_times = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = statistics.mean(e2e_times)
    e2e_same = bool(torch.equal(out_host.to(dev), res["out"]))

    # the same end to end step with moe_layer captured once in a CUDA graph
    # and replayed (how a serving loop calls it: the row count fixes the
    # launches, the valid mask is read at kernel time), the copies outside it
    gstream = torch.cuda.Stream()
    gstream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gstream):
        m2.moe_layer(cfg, x_dev, ri["wr"], ri["bias"], W, v_dev, out_dev, lws, stream=gstream)
    gstream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        m2.moe_layer(cfg, x_dev, ri["wr"], ri["bias"], W, v_dev, out_dev, lws, stream=gstream)
    torch.cuda.synchronize()

    def e2e_graph_step():
        x_dev.copy_(x_host, non_blocking=True)
        v_dev.copy_(v_host, non_blocking=True)
        graph.replay()
        out_host.copy_(out_dev, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        flush.zero_()
        e2e_graph_step()
    g_times = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_graph_step()
        g_times.append(time.perf_counter() - t0)
    e2e_graph_s = statistics.mean(g_times)
    e2e_graph_same = bool(torch.equal(out_host.to(dev), res["out"]))
    del graph
    # the same layer on the row-major codes gives the same bits
    m2.moe_layer(cfg, x_dev, ri["wr"], ri["bias"], W_rm, v_dev, out_dev, lws)
    torch.cuda.synchronize()
    layout_same = bool(torch.equal(out_dev, res["out"]))

    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline:
        t_all = dict(res["ri"])
        t_all.update(weights)
        cpu = oracle_baseline(wl, t_all)

    if rank == 0:
        clocks = res["clocks"]
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8_e4m3 (fp32 accumulate; bf16 in/out)", "data": "synthetic (seeded)",
            "config": {"workload": wl.name, "rows": R, "valid_rows": alg["Rv"],
                       "hidden": wl.shape.hidden, "inter": wl.shape.inter,
                       "experts": wl.shape.n_experts, "groups": wl.shape.n_groups,
                       "topk_groups": wl.shape.topk_groups, "topk": wl.shape.topk,
                       "shared": wl.shape.n_shared, "distinct_experts": alg["U"],
                       "l2": "flushed before every step (256 MB write, outside the events)",
                       "weight_layout": "tiled (each 128x128 e4m3 block as 16 KB, "
                                        "row-block-major)",
                       "parallelism": f"replicas x{world}"},
            "hbm": {"achieved_gbs": round(layer_gbs, 1),
                    "frac_of_measured": round(layer_gbs / pk["hbm_gbs"], 4),
                    "frac_of_8tbs": round(layer_gbs / 8000.0, 4),
                    "algorithmic_bytes_per_step": alg["total_bytes"]},
            "fp8_tflops": round(tflops, 2),
            "phase_ms": {k: round(v, 4) for k, v in res["phase_ms"].items()},
            "phase_note": "separate pass through the step-by-step entry points (route, union, "
                          "dispatch, expert GEMMs, combine) with an event between every two "
                          "kernels; the timed pass is one moe_layer call per step",
            "stepwise_bit_identical": res["stepwise_same"],
            "row_major_layout_bit_identical": layout_same,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(world * R / e2e_s, 1), "unit": "rows/s",
                    "h2d_bytes_per_step": x_host.numel() * 2 + v_host.numel(),
                    "d2h_bytes_per_step": out_host.numel() * 2,
                    "note": "moe_layer, pinned host x -> device -> pinned host out, per step",
                    "bit_identical_to_step_path": e2e_same,
                    "graph_replay": {"value": round(world * R / e2e_graph_s, 1),
                                     "unit": "rows/s",
                                     "note": "the same step with moe_layer captured once in a "
                                             "CUDA graph and replayed, copies outside it",
                                     "bit_identical_to_step_path": e2e_graph_same}},
            "gpu_launches": kernels_per_step(R) * args.steps,
            "clocks": clocks,
            "also": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
