"""Benchmark of the bit-exact int8-QAT linear hot path on GB300.

One step = one pass of the whole hot path over one batch of the workload
(default: one GQA decoder block's four linears, 4 micro-batches of 16,384
tokens, TreeFold over R = 6 replicas): weight scales and int8 weights, then per
micro-batch and linear the activation scale, int8 activations, exact int8
forward, canonical-order fp32 dX and dW with dW accumulated in micro-batch
order, and finally TreeFold.  Inputs are seeded synthetic tensors resident in
HBM (about 8 GB, far larger than L2) when the timed region starts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload block|attn_out|gate_up|down_accum|tiny]

Prints one JSON line (rank 0).  N > 1 runs one independent replica per GPU
("replicas only": the step has no collective on its data path); `value` is the
tokens of all ranks divided by the slowest rank's time.  `--impl reference`
times the CPU oracle on a bounded slice of the same workload's step.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bitwise_reproducible_int8_gb300 import inputs  # noqa: E402

METRIC = "tokens/s bit-exact int8-QAT linear fwd+bwd (1 GB300); % of int8/FP32/HBM roofline"

# DRAM bytes (read + write) per backward launch, averaged over the 160 backward
# launches of the block workload's 4 captured steps, from one ncu capture of
# dram__bytes_read.sum + dram__bytes_write.sum (single pass) on a GB300.  Valid only
# for that kernel and workload; anything else reports null.
# DRAM bytes per backward launch: mean over the block step's eight launch shapes,
# from one ncu capture (-k regex:k_bwd_tma -c 8, dram__bytes_read.sum +
# dram__bytes_write.sum) of the one-micro-batch profiling case block_1mb
BWD_TRAFFIC_PER_LAUNCH = {("block", "k_bwd_tma"): 1678.0e6, ("block_1mb", "k_bwd_tma"): 1678.0e6}
BWD_TRAFFIC_SOURCE = ("profiles/k_bwd_tma_traffic_block.md: ncu -k regex:k_bwd_tma -c 8 "
                      "--metrics dram__bytes_read.sum,dram__bytes_write.sum on block_1mb "
                      "(the block step's eight backward shapes), mean per launch")
UNIT = "tokens/s"


# ---------------------------------------------------------------- helpers

def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_workload(wl, rank: int):
    """Replicas only: rank r processes its own micro-batches (the pages' data
    ownership: window m belongs to rank m mod R), so its seeds are offset by
    r times the micro-batch count; weights are shared."""
    return dataclasses.replace(wl, x_seed_base=wl.x_seed_base + rank * wl.microbatches)


def max_over_ranks(ms: float, world: int, device) -> float:
    """Slowest rank's time (all_reduce MAX; a no-op for one rank)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank_step: int, steps: int, world: int,
                           ms_max: float) -> float:
    """Tokens of all ranks over the slowest rank's time."""
    return tokens_per_rank_step * steps * world / (ms_max / 1000.0)


# ---------------------------------------------------------------- oracle leg

class OracleSample:
    """The oracle, as it stands, timed on samples of one step's work, part by
    part, each part's time divided by the fraction of that part's work its
    sample holds, so that the estimate of a whole step does not depend on the
    sample size.  Every sample is a run of consecutive output elements (the
    first 1/2^k of each tensor in row-major order), computed through the
    oracle's calls for given elements, which parallelise over elements:
      weights      weight scale + codes of the first 1/2^k of every weight;
      activations  activation scale + codes of the first 1/2^k of every X;
      forward      the first 1/2^k of every Y (fraction weighted by K);
      dx           the first 1/2^k of every dX (weighted by N);
      dw           the first 1/2^k of every dW (each output reduces all M tokens);
      accumulate   the micro-batch accumulation of that dW sample;
      treefold     TreeFold over that sample of the gradient.
    The sampled outputs need every token's codes: prepare() computes them with
    the oracle once, untimed."""

    PARTS = ("weights", "activations", "forward", "dx", "dw", "accumulate", "treefold")

    def __init__(self, wl, host):
        import oracle as orc
        orc.build()
        self.orc, self.wl, self.host = orc, wl, host
        self.prepared = False

    def prepare(self):
        orc, wl, h = self.orc, self.wl, self.host
        L, J = len(wl.linears), wl.microbatches
        self.s_w = [orc.wscale(h.W[i], 0) for i in range(L)]
        self.wq = [orc.quant_i8(h.W[i], self.s_w[i]) for i in range(L)]
        self.s_x = [[orc.wscale(h.X[i][j], 1) for j in range(J)] for i in range(L)]
        self.xq = [[orc.quant_i8(h.X[i][j], self.s_x[i][j]) for j in range(J)] for i in range(L)]
        self.prepared = True

    def run(self, frac_log2: int, threads: int | None = None) -> dict:
        """Times one sampled step; returns {"parts": {name: (sec, fraction)},
        "timed_s": seconds spent, "step_s": extrapolated seconds of a whole step}."""
        import time as _t
        orc, wl, h = self.orc, self.wl, self.host
        if not self.prepared:
            self.prepare()
        saved = orc.threads()
        if threads:
            orc.set_threads(threads)
        f = 1 << frac_log2
        L, J, M = len(wl.linears), wl.microbatches, wl.tokens
        lins = wl.linears
        cut = lambda total: max(1, -(-total // f))  # noqa: E731
        sy = [cut(M * l.n_out) for l in lins]          # sampled outputs of Y
        sx = [cut(M * l.k_in) for l in lins]           # of dX (and of X's codes)
        sg = [cut(l.n_out * l.k_in) for l in lins]     # of dW (and of W's codes)
        flat = lambda cnt, cols: (np.arange(cnt, dtype=np.int64) // cols,  # noqa: E731
                                  np.arange(cnt, dtype=np.int64) % cols)
        iy = [flat(sy[i], lins[i].n_out) for i in range(L)]
        ix = [flat(sx[i], lins[i].k_in) for i in range(L)]
        ig = [flat(sg[i], lins[i].k_in) for i in range(L)]
        W_s = [np.ascontiguousarray(h.W[i].reshape(-1)[:sg[i]]) for i in range(L)]
        X_s = [[np.ascontiguousarray(h.X[i][j].reshape(-1)[:sx[i]]) for j in range(J)]
               for i in range(L)]
        t = dict.fromkeys(self.PARTS, 0.0)
        try:
            t0 = _t.perf_counter()
            for i in range(L):
                orc.quant_i8(W_s[i], orc.wscale(W_s[i], 0))
            t["weights"] = _t.perf_counter() - t0
            G = [None] * L
            for j in range(J):
                for i in range(L):
                    xq, s_x, wq, s_w = self.xq[i][j], self.s_x[i][j], self.wq[i], self.s_w[i]
                    dY = h.dY[i][j]
                    t0 = _t.perf_counter()
                    orc.quant_i8(X_s[i][j], orc.wscale(X_s[i][j], 1))
                    t1 = _t.perf_counter()
                    orc.linear_fwd_at(xq, wq, s_x, s_w, *iy[i])
                    t2 = _t.perf_counter()
                    orc.linear_bwd_dx_at(dY, wq, s_w, *ix[i])
                    t3 = _t.perf_counter()
                    dw = orc.linear_bwd_dw_at(dY, xq, s_x, *ig[i])
                    t4 = _t.perf_counter()
                    G[i] = dw if G[i] is None else orc.grad_accum(G[i], dw)
                    t5 = _t.perf_counter()
                    t["activations"] += t1 - t0
                    t["forward"] += t2 - t1
                    t["dx"] += t3 - t2
                    t["dw"] += t4 - t3
                    t["accumulate"] += t5 - t4
            if wl.replicas > 1:
                g = np.concatenate(G)
                offs = np.cumsum([0] + [l.n_out * l.k_in for l in lins])
                idx = np.concatenate([offs[i] + np.arange(sg[i]) for i in range(L)])
                parts = [g] + [orc.grad_accum(g, h.noise[r][idx]) for r in range(1, wl.replicas)]
                t0 = _t.perf_counter()
                orc.treefold(parts)
                t["treefold"] = _t.perf_counter() - t0
        finally:
            orc.set_threads(saved)
        nk = sum(l.n_out * l.k_in for l in lins)
        mk = sum(M * l.k_in for l in lins)
        frac = {"weights": sum(sg) / nk, "activations": sum(sx) / mk,
                "forward": sum(sy[i] * lins[i].k_in for i in range(L)) / (M * nk),
                "dx": sum(sx[i] * lins[i].n_out for i in range(L)) / (M * nk),
                "dw": sum(sg) / nk, "accumulate": sum(sg) / nk, "treefold": sum(sg) / nk}
        if J < 2:
            frac["accumulate"] = 1.0   # nothing to accumulate: zero time, any fraction
        if wl.replicas <= 1:
            frac["treefold"] = 1.0
        parts = {k: (t[k], frac[k]) for k in self.PARTS}
        return {"parts": parts, "timed_s": sum(t.values()),
                "step_s": sum(sec / fr for sec, fr in parts.values()),
                "threads": threads or saved}


def _sample_text(wl, frac_log2, r) -> str:
    parts = ", ".join(f"{k} {sec:.2f} s / {fr:.2e}" for k, (sec, fr) in r["parts"].items())
    if frac_log2 == 0:
        parts = ", ".join(f"{k} {sec:.3f} s" for k, (sec, _) in r["parts"].items())
        return (f"{wl.name}: the whole step, every output of every call; parts: {parts}; "
                f"{r['timed_s']:.3f} s on {r['threads']} threads")
    return (f"{wl.name}: the first 1/{1 << frac_log2} of the outputs of every call of one step "
            f"(Y, dX, dW, codes, the gradient's accumulation and TreeFold), each part of the "
            f"step timed on its own sample and divided by that sample's fraction of the part's "
            f"work (multiply-adds or elements); parts [time / fraction]: {parts}; "
            f"{r['timed_s']:.2f} s timed on {r['threads']} threads, a whole step extrapolated to "
            f"{r['step_s']:.0f} s")


def cpu_baseline(wl, host, frac_log2: int, one_core_extra_log2: int = 2) -> dict:
    """The oracle on every host core (the reported value), and on one core.  A
    small step (under 2^30 multiply-adds, the single-linear 64-token case) runs
    whole both times; a larger one is sampled, the one-core sample 2^-extra the
    size of the all-core one, both extrapolated part by part."""
    smp = OracleSample(wl, host)
    smp.prepare()
    tokens = wl.tokens * wl.microbatches
    macs = tokens * sum(l.n_out * l.k_in for l in wl.linears)
    small = macs < (1 << 30)   # a sample's fixed per-call costs would swamp it: run it whole
    if small:
        frac_log2 = 0
    r = smp.run(frac_log2)
    one_log2 = 0 if small else frac_log2 + one_core_extra_log2
    r1 = smp.run(one_log2, threads=1)
    return {"value": tokens / r["step_s"], "unit": UNIT, "cores": r["threads"], "kind": "oracle",
            "sample": _sample_text(wl, frac_log2, r),
            "one_core": {"value": tokens / r1["step_s"], "unit": UNIT, "cores": 1,
                         "sample": _sample_text(wl, one_log2, r1),
                         "extrapolated": one_log2 > 0}}


def run_reference(args, wl):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from bitwise_reproducible_int8_gb300 import step as S
    host = S.generate_host_inputs(wl)
    smp = OracleSample(wl, host)
    smp.prepare()                       # every token's codes, once, untimed
    for _ in range(args.warmup):
        smp.run(args.ref_frac_log2)
    runs = [smp.run(args.ref_frac_log2) for _ in range(args.steps)]
    step_s = sum(r["step_s"] for r in runs) / len(runs)
    timed = sum(r["timed_s"] for r in runs)
    value = wl.tokens * wl.microbatches / step_s
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * timed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i8/f32",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": wl.name, "tokens_per_step": wl.tokens * wl.microbatches,
                   "sample_fraction": 1.0 / (1 << args.ref_frac_log2),
                   "ms_per_step_is": "the sampled slices' timed ms; value extrapolates each part "
                                     "of the step by its own fraction",
                   "extrapolated_s_per_full_step": step_s,
                   "parallelism": "replicas only"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": runs[0]["threads"],
                         "kind": "oracle", "sample": _sample_text(wl, args.ref_frac_log2, runs[-1])},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    from bitwise_reproducible_int8_gb300 import build_lib
    from bitwise_reproducible_int8_gb300 import repro as R
    from bitwise_reproducible_int8_gb300 import step as S

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if args.bwd_kernel >= 0 or args.fwd_path >= 0:
        R.repro_set_launch_cfg(bwd_kernel=args.bwd_kernel, fwd_path=args.fwd_path)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or not os.path.exists(build_lib.LIB):
        build_lib.build()
    if world > 1:
        dist.barrier()
    wl_r = replica_workload(wl, rank)
    host = S.generate_host_inputs(wl_r)
    hp = S.HotPathStep(wl_r, host, fused_accum=not args.unfused_accum,
                       dw_stream=False if args.no_dw_stream else None)
    inputs_sha256 = hp.input_digest()   # untimed, before any step changes the weights
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        if wl_r.replicas > 1 or wl_r.shards > 1:
            hp.prepare(stream)
        for _ in range(args.warmup):
            hp.run(stream)
    stream.synchronize()
    if R.repro_device_check(stream) != 0:
        raise RuntimeError("device error during warm-up")
    graph, graph_launches = None, 0
    if args.graph:
        # the step captured once into a CUDA graph, replayed per step
        l0 = R.repro_launch_count()
        graph = hp.capture(stream)
        graph_launches = R.repro_launch_count() - l0
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()

    # ---- device-timed region: K steps, inputs resident in HBM
    timers = {}
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = R.repro_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                hp.run(stream, timers=timers)
        t_end.record(stream)
    stream.synchronize()
    launches = R.repro_launch_count() - launches0
    if graph is not None:
        launches = graph_launches * args.steps
    clk = clocks.stop()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end)
    if R.repro_device_check(stream) != 0:
        raise RuntimeError("device error during the timed steps")
    if graph is not None:
        # graph replays carry no per-call events: split the step by call from
        # the same number of eager steps, timed call by call
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                hp.run(stream, timers=timers)
        stream.synchronize()
    pairs = timers.pop("bwd_pair", None)
    pair_ms = n_pairs = None
    if pairs:
        pair_ms = sum(max(f.elapsed_time(dx), f.elapsed_time(dw)) for f, dx, dw in pairs)
        n_pairs = len(pairs)
    per_class = {k: sum(a.elapsed_time(b) for a, b in v) for k, v in timers.items()}
    launch_counts = {k: len(v) for k, v in timers.items()}

    ms_max = max_over_ranks(ms, world, "cuda")
    value = whole_job_tokens_per_s(hp.tokens(), args.steps, world, ms_max)

    # ---- end to end: host inputs copied in, result copied out, every step
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(hp, host, args.steps, stream, world)

    if rank == 0:
        peaks = load_peaks()
        sms = torch.cuda.get_device_properties(local).multi_processor_count
        fl = hp.flops()
        bwd_ops = (fl["bwd_dx_fp32_ops"] + fl["bwd_dw_fp32_ops"]) * args.steps
        if pair_ms is not None:
            # dX and dW of a linear run concurrently: the unit is the pair, timed
            # from the fork to the later of its two ends (the forward launched
            # between them included, so the rate errs low)
            bwd_ms, n_units = pair_ms, n_pairs
        else:
            bwd_ms = per_class.get("bwd_dx", 0.0) + per_class.get("bwd_dw", 0.0)
            n_units = None
        fp32_peak = sms * 128 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        achieved = bwd_ops / (bwd_ms / 1000.0) / 1e12 if bwd_ms > 0 else 0.0
        nb = launch_counts.get("bwd_dx", 0) + launch_counts.get("bwd_dw", 0)
        kname = {1: "k_bwd_prefetch", 8: "k_bwd_tma"}[args.bwd_kernel if args.bwd_kernel >= 0 else 8]
        traffic = BWD_TRAFFIC_PER_LAUNCH.get((wl.name, kname))
        unit_note = None
        if n_units:
            unit_note = ("one unit = the dX and dW launches of one linear and micro-batch, run "
                         "concurrently on two streams; its time runs from the fork to the later "
                         "of the two ends and includes the forward launched between them; "
                         "traffic is the two launches' (each measured alone under ncu)")
            traffic = 2 * traffic if traffic is not None else None
        per_unit = n_units if n_units else nb
        roofline = {
            "bound": "alu", "kernel": f"{kname} (dX and dW, canonical-order fp32)",
            "achieved": achieved, "peak": fp32_peak, "unit": "TFLOP/s",
            "frac": achieved / fp32_peak if fp32_peak else None,
            "peak_note": f"FP32 pipe: {sms} SMs x 128 lanes x {peaks.get('sm_max_mhz', 2070.0):.0f} MHz,"
                         " one FMUL or FADD per lane per clock (no FMA may be used)",
            # the same work as a FLOP fraction of the peak that counts an FFMA as
            # two FLOPs; without FMA this can reach at most 0.5
            "flop_frac_of_ffma_peak": achieved / (2 * fp32_peak) if fp32_peak else None,
            "traffic": traffic,
            "traffic_source": BWD_TRAFFIC_SOURCE if traffic is not None else None,
            "launches": nb,
            "flops_per_launch": bwd_ops / per_unit if per_unit else None,
            "avg_launch_ms": bwd_ms / per_unit if per_unit else None,
        }
        if unit_note:
            roofline["units"] = n_units
            roofline["unit_note"] = unit_note
        other = {}
        fwd_ms = per_class.get("fwd", 0.0)
        if fwd_ms > 0:
            tops = fl["fwd_int_ops"] * args.steps / (fwd_ms / 1e3) / 1e12
            # the codes run on the bf16 tensor path (exact K-slices), so the
            # denominator is the measured bf16 dense burst peak; the time includes
            # the two int8 -> bf16 widening passes of every call
            other["fwd_int8"] = {"achieved_tops": tops, "ms_per_step": fwd_ms / args.steps,
                                 "frac_bf16_peak": tops / peaks["bf16_tflops"],
                                 "peak_tflops": peaks["bf16_tflops"]}
            if hp.s_dw is not None:
                other["fwd_int8"]["note"] = ("overlaps a dW on the other stream: a lower bound; "
                                             "--no-dw-stream times it alone")
        gbytes = hbm_bytes(hp)
        for cls, nbytes in gbytes.items():
            c_ms = per_class.get(cls, 0.0)
            if c_ms > 0:
                gbs = nbytes * args.steps / (c_ms / 1e3) / 1e9
                other[cls] = {"achieved_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                              "ms_per_step": c_ms / args.steps}
                if cls == "state_hash":
                    other[cls]["bound"] = "alu (SHA-256 compressions on the integer pipe)"
        if "wscale_w" in other and "treefold" in other:
            # a step opens with the weights' scale, right after the previous
            # step's TreeFold, whose output is still partly dirty in L2: that
            # write-back shares the scale's DRAM time, so the pair is reported too
            tw = per_class["treefold"] + per_class["wscale_w"]
            both = (gbytes["treefold"] + gbytes["wscale_w"]) * args.steps / (tw / 1e3) / 1e9
            other["wscale_w"]["note"] = ("follows the previous step's TreeFold, whose output is "
                                         "written back from L2 meanwhile; see treefold_then_wscale_w")
            other["treefold_then_wscale_w"] = {"achieved_gbs": both, "frac_hbm": both / peaks["hbm_gbs"],
                                               "ms_per_step": tw / args.steps}

        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(wl_r, host, args.cpu_frac_log2)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "i8/f32", "data": "synthetic",
            "config": {"workload": wl.name, "tokens_per_step": hp.tokens(),
                       "micro_batches": wl.microbatches, "micro_batch_tokens": wl.tokens,
                       "linears": [f"{l.name} {l.n_out}x{l.k_in}" for l in wl.linears],
                       "replicas": wl.replicas, "shards": wl.shards,
                       "parallelism": "replicas only",
                       "streams": "dW on a second stream, concurrent with the forward and dX"
                       if hp.s_dw is not None else "one stream",
                       "accumulation": "unfused repro_grad_accum" if args.unfused_accum
                       else "fused into the dW epilogue",
                       "l2": (f"inputs larger than L2: {resident_gb(hp):.1f} GB resident, "
                              "streamed once per step") if resident_gb(hp) > 0.129 else
                             (f"inputs fit in L2 ({resident_gb(hp) * 1e3:.1f} MB resident): a "
                              "launch-latency case, L2 not flushed"),
                       "launch": "one CUDA graph replay per step" if graph is not None
                       else "eager calls",
                       "inputs_sha256": inputs_sha256,
                       "inputs_sha256_of": "RFC 6962 Merkle root (SHA-256, 4 KB leaves) of rank 0's "
                                           "flat weights, then X and dY per linear, micro-batch "
                                           "by micro-batch"},
            "roofline": roofline, "other_kernels": other,
            "ms_per_step_by_call": {k: v / args.steps for k, v in per_class.items()},
            "overlapping_calls": ["bwd_dw", "fwd", "bwd_dx"] if hp.s_dw is not None else [],
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk, "peaks_source": peaks["source"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def resident_gb(hp) -> float:
    tot = sum(x.numel() * 4 for i in range(len(hp.X)) for x in hp.X[i])
    tot += sum(x.numel() * 4 for i in range(len(hp.dY)) for x in hp.dY[i])
    return tot / 1e9


def hbm_bytes(hp) -> dict:
    """Algorithmic HBM bytes per step of the streaming call classes."""
    wl = hp.wl
    J = wl.microbatches
    nw = sum(w.numel() for w in hp.W)
    nx = sum(x.numel() for i in range(len(hp.X)) for x in hp.X[i])
    out = {"wscale_w": 4 * nw, "quant_w": 5 * nw, "wscale_x": 4 * nx, "quant_x": 5 * nx}
    if hp.TF is not None:
        out["treefold"] = 4 * (wl.replicas + 1) * hp.n_grad
    if hp.G2 is not None:
        out["running_sum"] = 4 * (wl.shards + 1) * hp.n_grad
    if hp.use_optimizer:
        out["sumsq"] = 4 * hp.n_grad
        out["adamw"] = 28 * hp.n_grad
        out["state_hash"] = 12 * hp.n_grad   # parameters + two moments read once
    if hp.dW_tmp is not None:
        out["accum"] = 12 * nw * (J - 1)
    return out


def measure_e2e(hp, host, steps, stream, world):
    """Same steps through the public API with host buffers: every step copies
    its inputs from pinned host memory (micro-batch 0's X and dY, the weights,
    then the other micro-batches, on a copy stream) and reads the result back.  X and dY are double
    buffered across steps: step s+1 copies into the set step s-1 used, as soon
    as step s-1 has read each buffer for the last time, so its copies overlap
    step s.  The weights are one buffer, refilled once the previous step's
    scale and quantise calls have read them (with the optimizer on, once the
    whole previous step is done, since it updates them)."""
    import torch
    L, J = len(hp.wl.linears), hp.wl.microbatches
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    hW = [pin(host.W[i]) for i in range(L)]
    hX = [[pin(host.X[i][j]) for j in range(J)] for i in range(L)]
    hdY = [[pin(host.dY[i][j]) for j in range(J)] for i in range(L)]
    res = hp.result()
    out_host = torch.empty(res.shape, dtype=res.dtype, pin_memory=True)
    h2d = sum(t.numel() * 4 for t in hW) + sum(t.numel() * 4 for r in hX for t in r) + \
        sum(t.numel() * 4 for r in hdY for t in r)
    d2h = res.numel() * 4
    copy = torch.cuda.Stream()
    sets = [(hp.X, hp.dY),
            ([[torch.empty_like(t) for t in row] for row in hp.X],
             [[torch.empty_like(t) for t in row] for row in hp.dY])]
    torch.cuda.synchronize()
    released = [None, None]   # per buffer set: the release events of its last step
    w_released = [None]
    count = [0]
    # the TreeFold output is rewritten only at the end of the next step, so its
    # read-back runs on a stream of its own and that step's TreeFold waits for it
    down = torch.cuda.Stream() if hp.TF is not None else None
    read_done = [None]

    def one_step():
        k = count[0]
        count[0] += 1
        hp.X, hp.dY = sets[k % 2]
        prev = released[k % 2]
        evs = [None] * J
        done = [None] * (J + 1)
        with torch.cuda.stream(copy):
            if k == 0:
                copy.wait_stream(stream)
            for j in range(J):
                if prev is not None:
                    for ev in prev[j]:
                        copy.wait_event(ev)
                for i in range(L):
                    hp.X[i][j].copy_(hX[i][j], non_blocking=True)
                    hp.dY[i][j].copy_(hdY[i][j], non_blocking=True)
                if j == 0:
                    # the weights right after micro-batch 0: the step starts with them
                    if hp.use_optimizer:
                        copy.wait_stream(stream)
                    elif w_released[0] is not None:
                        for ev in w_released[0]:
                            copy.wait_event(ev)
                    for i in range(L):
                        hp.W[i].copy_(hW[i], non_blocking=True)
                evs[j] = torch.cuda.Event()
                evs[j].record(copy)
        hp.run(stream, wait_events=evs, done_events=done,
               fold_wait_events=[read_done[0]] if read_done[0] is not None else None)
        released[k % 2] = done
        w_released[0] = done[J]
        if down is None:
            with torch.cuda.stream(stream):
                out_host.copy_(res, non_blocking=True)
        else:
            step_end = torch.cuda.Event()
            step_end.record(stream)
            with torch.cuda.stream(down):
                down.wait_event(step_end)
                out_host.copy_(res, non_blocking=True)
                read_done[0] = torch.cuda.Event()
                read_done[0].record(down)

    # the inputs are the same every step, so every step's result must equal
    # the device-resident step's, bit for bit (a refill that raced a read
    # would show here); without the optimizer only, which changes W
    expect = None if hp.use_optimizer else res.detach().cpu().clone()
    with torch.cuda.stream(stream):
        one_step()
    stream.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        one_step()
    if read_done[0] is not None:
        stream.wait_event(read_done[0])   # the last read-back is inside the timed region
    b.record(stream)
    stream.synchronize()
    if expect is not None and not torch.equal(out_host.view(torch.int32), expect.view(torch.int32)):
        raise RuntimeError("end-to-end steps changed the result bits")
    ms = max_over_ranks(a.elapsed_time(b), world, "cuda")
    return {"value": whole_job_tokens_per_s(hp.tokens(), steps, world, ms), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms / steps}


# ---------------------------------------------------------------- attention leg

def attn_pairs(aw) -> int:
    """Valid (query, key) pairs per step: sum over rows of min(i + 1, W)."""
    T, W = aw.seq_len, aw.window
    if W <= 0 or W >= T:
        per_seq = T * (T + 1) // 2
    else:
        per_seq = W * (W + 1) // 2 + (T - W) * W
    return per_seq * aw.sequences * aw.heads_q


def attn_oracle_sample(aw, q, k, v, do, frac_log2: int) -> tuple:
    """The oracle on a uniform 2^-k sample of one step's rows: V's scale and
    codes in full, the forward of 1/2^k of the query rows, dQ of 1/2^k of the
    query rows and dK, dV of 1/2^k of the key rows.  Returns (s, tokens)."""
    import oracle as orc
    f = 1 << frac_log2
    nq, nk = aw.tokens * aw.heads_q, aw.tokens * aw.heads_kv
    rng = np.random.default_rng(12345)
    qrows = np.sort(rng.choice(nq, max(1, nq // f), replace=False))
    krows = np.sort(rng.choice(nk, max(1, nk // f), replace=False))
    t0 = time.perf_counter()
    s_v = orc.wscale(v, 1)
    vq = orc.quant_i8(v, s_v).reshape(v.shape)
    o_s, m_s, l_s = orc.attn_fwd_rows(q, k, vq, s_v, aw.window, qrows)
    sec = time.perf_counter() - t0
    # the backward reads o, m, l of every row it touches: the sampled query
    # rows carry their own from the timed forward; the other rows (reached by
    # dK/dV) get placeholder statistics -- the same work per row, values unchecked
    o = np.zeros((aw.tokens * aw.heads_q, q.shape[-1]), np.float32)
    m = np.zeros(aw.tokens * aw.heads_q, np.float32)
    l = np.ones(aw.tokens * aw.heads_q, np.float32)
    o[qrows], m[qrows], l[qrows] = o_s, m_s, l_s
    t1 = time.perf_counter()
    orc.attn_bwd_rows(q, k, vq, s_v, o.reshape(q.shape), do, m.reshape(q.shape[:3]),
                      l.reshape(q.shape[:3]), aw.window, qrows, krows)
    sec += time.perf_counter() - t1
    return sec, aw.tokens / f


def _attn_sample_text(aw, frac_log2, toks, sec=None):
    t = (f"{aw.name}: 1/{1 << frac_log2} of one step's rows -- forward and dQ of "
         f"{max(1, aw.tokens * aw.heads_q >> frac_log2)} query rows, dK and dV of "
         f"{max(1, aw.tokens * aw.heads_kv >> frac_log2)} key rows (dK/dV of unsampled query "
         f"rows use placeholder statistics: same work, not checked), V's scale and codes in "
         f"full; credited {toks:.1f} tokens")
    return t + (f"; {sec:.2f} s" if sec is not None else "")


def run_attn(args, aw):
    import torch

    from bitwise_reproducible_int8_gb300 import build_lib
    from bitwise_reproducible_int8_gb300 import repro as R

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or not os.path.exists(build_lib.LIB):
        build_lib.build()
    if world > 1:
        dist.barrier()
    aw_r = dataclasses.replace(aw, seed=aw.seed + 1000 * rank)   # replicas only: own data
    q, k, v, do = inputs.attn_inputs(aw_r)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    dev = torch.device("cuda", local)
    tq, tk, tv, tdo = (torch.from_numpy(x).to(dev) for x in (q, k, v, do))
    vq = torch.empty(v.shape, dtype=torch.int8, device=dev)
    s_v = torch.zeros(1, device=dev)
    o = torch.empty(q.shape, device=dev)
    m = torch.empty(q.shape[:3], device=dev)
    l = torch.empty(q.shape[:3], device=dev)
    dq = torch.empty(q.shape, device=dev)
    dk = torch.empty(k.shape, device=dev)
    dv = torch.empty(k.shape, device=dev)
    ws_s = torch.empty(max(R.repro_wscale_ws_bytes(v.size), 16), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(R.repro_attn_bwd_ws_bytes(B, T, Hq, aw.window), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(max(R.repro_attn_fwd_ws_bytes(B, T, Hq, aw.window), 16), dtype=torch.uint8,
                       device=dev)   # the forward's logit cache
    dev_bufs = (tq, tk, tv, tdo, dq, dk, dv)
    d32 = torch.empty(32, dtype=torch.uint8, device=dev)
    R.repro_state_hash([tq, tk, tv, tdo], d32)   # untimed record of the inputs
    torch.cuda.synchronize()
    inputs_sha256 = bytes(d32.cpu().numpy()).hex()
    torch.cuda.synchronize()   # s_v's fill ran on the default stream
    stream = torch.cuda.Stream()
    timers = {}

    def ev(cls):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        timers.setdefault(cls, []).append([e, None])

    def end(cls):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        timers[cls][-1][1] = e

    def one_step(timed, bufs=None):
        tq, tk, tv, tdo, dq, dk, dv = bufs if bufs is not None else dev_bufs
        if timed:
            ev("vscale")
        R.repro_wscale(tv, R.REPRO_SCALE_ACT_AMAX, s_v, ws=ws_s, stream=stream)
        if timed:
            end("vscale")
            ev("vquant")
        R.repro_quant_i8(tv, s_v, vq, stream=stream)
        if timed:
            end("vquant")
            ev("attn_fwd")
        R.repro_attn_fwd(tq, tk, vq, s_v, o, m, l, aw.window, ws=ws_f, stream=stream)
        if timed:
            end("attn_fwd")
            ev("attn_bwd")
        R.repro_attn_bwd(tq, tk, vq, s_v, o, tdo, m, l, dq, dk, dv, aw.window, ws=ws_b,
                         fwd_ws=ws_f, stream=stream)
        if timed:
            end("attn_bwd")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step(False)
    stream.synchronize()
    if R.repro_device_check(stream) != 0:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = R.repro_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            one_step(True)
        t_end.record(stream)
    stream.synchronize()
    launches = R.repro_launch_count() - launches0
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    if R.repro_device_check(stream) != 0:
        raise RuntimeError("device error during the timed steps")
    per_class = {kk: sum(a.elapsed_time(b) for a, b in vv) for kk, vv in timers.items()}
    ms_max = max_over_ranks(ms, world, "cuda")
    value = whole_job_tokens_per_s(aw.tokens, args.steps, world, ms_max)

    # e2e: every step copies q, k, v, dO from pinned host memory and reads dq,
    # dk, dv back, through the same calls.  Inputs and outputs are double
    # buffered across steps: step s+1's uploads (copy stream) overlap step s,
    # step s's downloads (a third stream) overlap step s+1, and a buffer set is
    # refilled or rewritten only once step s-1 (its last user) is done with it
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (torch.from_numpy(x).pin_memory() for x in (q, k, v, do))
        hdq = torch.empty(dq.shape).pin_memory()
        hdk = torch.empty(dk.shape).pin_memory()
        hdv = torch.empty(dv.shape).pin_memory()
        # the inputs are the same every step: the last download must equal the
        # device-resident step's gradients, bit for bit
        expect = [t.detach().cpu().clone() for t in dev_bufs[4:]]
        sets = [dev_bufs, tuple(torch.empty_like(t) for t in dev_bufs)]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        in_free, out_free = [None, None], [None, None]
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        up.wait_stream(stream)
        last_down = None
        h2d_ev = []   # each step's uploads, from their start to their end
        for step in range(args.steps):
            cur = sets[step % 2]
            with torch.cuda.stream(up):
                if in_free[step % 2] is not None:
                    up.wait_event(in_free[step % 2])
                u0 = torch.cuda.Event(enable_timing=True)
                u0.record(up)
                for d, h in zip(cur[:4], (hq, hk, hv, hdo)):
                    d.copy_(h, non_blocking=True)
                ready = torch.cuda.Event(enable_timing=True)
                ready.record(up)
                h2d_ev.append((u0, ready))
            stream.wait_event(ready)
            if out_free[step % 2] is not None:
                stream.wait_event(out_free[step % 2])
            with torch.cuda.stream(stream):
                one_step(False, cur)
                done = torch.cuda.Event()
                done.record(stream)
            in_free[step % 2] = done
            with torch.cuda.stream(down):
                down.wait_event(done)
                for h, d in zip((hdq, hdk, hdv), cur[4:]):
                    h.copy_(d, non_blocking=True)
                last_down = torch.cuda.Event()
                last_down.record(down)
            out_free[step % 2] = last_down
        stream.wait_event(last_down)
        a1.record(stream)
        stream.synchronize()
        for h, e in zip((hdq, hdk, hdv), expect):
            if not torch.equal(h.view(torch.int32), e.view(torch.int32)):
                raise RuntimeError("end-to-end attention steps changed the gradient bits")
        e_ms = a0.elapsed_time(a1)
        e2e = {"value": whole_job_tokens_per_s(aw.tokens, args.steps, world,
                                               max_over_ranks(e_ms, world, "cuda")),
               "unit": UNIT,
               "h2d_bytes_per_step": int(4 * (q.size + k.size + v.size + do.size)),
               "d2h_bytes_per_step": int(4 * (dq.numel() + dk.numel() + dv.numel())),
               "ms_per_step": e_ms / args.steps}
        # the host link as these steps saw it: the uploads hide behind a step
        # only while they take less than it
        up_ms = sum(x.elapsed_time(y) for x, y in h2d_ev) / args.steps
        e2e["h2d_ms_per_step"] = up_ms
        e2e["h2d_gbs"] = e2e["h2d_bytes_per_step"] / (up_ms / 1e3) / 1e9 if up_ms > 0 else None

    if rank == 0:
        peaks = load_peaks()
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        fp32_peak = sms * 128 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        pairs = attn_pairs(aw)
        # algorithmic FP32 work per valid (query, key) pair: the logits once in
        # the forward (2 * 128), and in the backward the dA, dQ, dK and dV dot
        # products (4 * 2 * 128) -- the backward reads the forward's logits from
        # its cache instead of recomputing them; P.V is integer work (dp4a)
        fwd_ops, bwd_ops = 2 * D * pairs, 8 * D * pairs
        f_ms, b_ms = per_class.get("attn_fwd", 0.0), per_class.get("attn_bwd", 0.0)
        ach = (fwd_ops + bwd_ops) * args.steps / ((f_ms + b_ms) / 1e3) / 1e12
        roofline = {
            "bound": "alu", "kernel": "k_attn_fwd + k_attn_bwd (canonical-order fp32 logits, "
                                      "softmax and gradients; int8 P.V)",
            "achieved": ach, "peak": fp32_peak, "unit": "TFLOP/s", "frac": ach / fp32_peak,
            "peak_note": f"FP32 pipe: {sms} SMs x 128 lanes x {peaks.get('sm_max_mhz', 2070.0):.0f}"
                         " MHz, one FMUL or FADD per lane per clock (no FMA may be used)",
            "traffic": None, "launches": 4 * args.steps,
            "flops_per_launch": (fwd_ops + bwd_ops) / 2,
            "avg_launch_ms": (f_ms + b_ms) / (2 * args.steps),
            "fwd_frac": fwd_ops * args.steps / (f_ms / 1e3) / 1e12 / fp32_peak if f_ms else None,
            "bwd_frac": bwd_ops * args.steps / (b_ms / 1e3) / 1e12 / fp32_peak if b_ms else None,
        }
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            import oracle as orc
            orc.build()
            sec, toks = attn_oracle_sample(aw_r, q, k, v, do, args.cpu_frac_log2)
            cpu = {"value": toks / sec, "unit": UNIT, "cores": orc.threads(), "kind": "oracle",
                   "sample": _attn_sample_text(aw, args.cpu_frac_log2, toks, sec)}
        line = {
            "metric": "tokens/s bit-exact int8 P.V attention fwd+bwd (1 GB300); % of FP32 roofline",
            "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32/i8", "data": "synthetic",
            "config": {"workload": aw.name, "tokens_per_step": aw.tokens,
                       "sequences": aw.sequences, "seq_len": aw.seq_len, "heads_q": aw.heads_q,
                       "heads_kv": aw.heads_kv, "head_dim": D, "window": aw.window,
                       "pairs_per_step": pairs, "parallelism": "replicas only",
                       "l2": "inputs larger than L2: q, k, v, dO and outputs ~0.7 GB",
                       "inputs_sha256": inputs_sha256,
                       "inputs_sha256_of": "RFC 6962 Merkle root (SHA-256, 4 KB leaves) of rank 0's "
                                           "q, k, v and dO"},
            "roofline": roofline,
            "ms_per_step_by_call": {kk: vv / args.steps for kk, vv in per_class.items()},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk, "peaks_source": peaks["source"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_attn_reference(args, aw):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle as orc
    orc.build()
    q, k, v, do = inputs.attn_inputs(aw)
    for _ in range(args.warmup):
        attn_oracle_sample(aw, q, k, v, do, args.ref_frac_log2)
    runs = [attn_oracle_sample(aw, q, k, v, do, args.ref_frac_log2) for _ in range(args.steps)]
    total = sum(r[0] for r in runs)
    toks = sum(r[1] for r in runs)
    value = toks / total
    line = {
        "metric": "tokens/s bit-exact int8 P.V attention fwd+bwd (1 GB300); % of FP32 roofline",
        "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32/i8", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": aw.name, "tokens_per_step": aw.tokens,
                   "sample_fraction": 1.0 / (1 << args.ref_frac_log2),
                   "parallelism": "replicas only"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.threads(), "kind": "oracle",
                         "sample": _attn_sample_text(aw, args.ref_frac_log2, toks / args.steps)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="block",
                    choices=sorted(inputs.WORKLOADS) + sorted(inputs.ATTN_WORKLOADS))
    ap.add_argument("--unfused-accum", action="store_true",
                    help="accumulate dW with repro_grad_accum instead of the fused epilogue")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-dw-stream", action="store_true",
                    help="run each dW after its dX on the one stream (default: dW on a "
                         "second stream, concurrent with the forward and dX, for linears of "
                         "at least 2^30 multiply-adds)")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step into a CUDA graph and time its replays "
                         "(launch-bound workloads; not with the optimizer)")
    ap.add_argument("--bwd-kernel", type=int, default=-1,
                    help="backward kernel (launch-configuration hook; -1: default 8, the "
                         "tensor-copy-fed kernel; 1: the register-prefetch kernel)")
    ap.add_argument("--fwd-path", type=int, default=-1,
                    help="forward path (launch-configuration hook; -1: default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-frac-log2", type=int, default=10,
                    help="the oracle's timed sample is 2^-k of one step's work")
    ap.add_argument("--ref-frac-log2", type=int, default=12,
                    help="each reference-arm step is 2^-k of one step's work")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload in inputs.ATTN_WORKLOADS:
        aw = inputs.ATTN_WORKLOADS[args.workload]
        if args.impl == "reference":
            return run_attn_reference(args, aw)
        return run_attn(args, aw)
    wl = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
