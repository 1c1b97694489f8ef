"""Benchmark of the sequence-parallel DiT attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input
already resident in HBM: Ulysses seq->head layout -> attention partials ->
merge (when R > 1) -> head->seq layout -> CFG combine.  The layout steps run
as one pass each (--exchange direct, the default: on one memory the
all-to-all aliases receive and send blocks) or as pack -> simulated
all-to-all -> unpack (--exchange a2a, the calls a multi-GPU build keeps).
The default workload is the FLUX-1024-like one (B=1, S=4608, H=24, D=128,
U=4, R=1; CFG on [2,4608,3072] bf16, g=3.5).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--U U]
    python bench.py --impl reference ...     # the fp64 CPU oracle, timed

Prints one JSON line (rank 0).  `value` is attention TFLOP/s over the whole
step (algorithmic 4*B*H*S^2*D flops / step time, summed over ranks);
`e2e` is the same through the public API with pinned host buffers and the
host<->device copies inside the timed region.  L2 is flushed (a 256 MiB
write) before every timed step; only the step itself is inside the events
(one at its start, one at its end); a second pass with events between the
phases gives the per-phase split in `kernels`.  The block of K timed steps
is repeated back to back until it has run for at least half a second, so
that the clock sampler (nvidia-smi, 20 ms period) takes its samples inside
the timed region; `value` is the mean over every timed step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DiT attn TFLOP/s & % bf16 TC peak (S=4608,H=24,D=128); pack/CFG GB/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ATTN_SRC = os.path.join(ROOT, "sequence_attention_gb300", "csrc", "attn_tc.cu")
TRAFFIC_NOTE = os.path.join(ROOT, "profiles", "attn_tc_flux1024.md")
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


# ---------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def init_dist(backend: str):
    import torch.distributed as dist
    rank, _, ws = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return dist


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- peaks, clocks
def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None
        self.start = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi takes a while to start: hold the timed region back
            # until its first sample has come in, so the samples after this
            # point are the region's own
            t0 = time.time()
            while not self.lines and self.proc.poll() is None and time.time() - t0 < 10:
                time.sleep(0.005)
        except OSError:
            self.proc = None
        self.start = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        inside = self.lines[self.start:]
        # a region shorter than the sampling interval: the sample taken just
        # before it started
        lines = inside if inside else self.lines[max(self.start - 1, 0):self.start]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_region": len(inside)}


def traffic_per_launch(kernel_src: str, note: str):
    """dram bytes per launch recorded by an ncu capture, if the kernel source
    has not changed since (the note stores the source's sha256)."""
    try:
        text = open(note).read()
        sha = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_launch_full:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_b) or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


# ---------------------------------------------------------------- workload
def bench_config(w, U: int):
    """The workload part of the JSON line's config, the same for both arms."""
    return {"workload": f"{w.name}-like: B={w.B} S={w.S} H={w.H} D={w.D}, Ulysses U={U}, "
                        f"ring R={w.R}; CFG [2,{','.join(map(str, w.cfg_shape[1:]))}] "
                        f"{w.cfg_in}->{w.cfg_out} g={w.g}",
            "B": w.B, "S": w.S, "H": w.H, "D": w.D, "U": U, "R": w.R,
            "parallelism": f"virtual ranks U{U}xR{w.R} on one GPU; replicas across GPUs"}


def workload_config(name: str, U: int):
    import synth
    w = synth.WORKLOADS[name]
    if U is None:
        U = max(w.U)
    return w, U


class OracleStep:
    """The oracle's work on a workload, for the CPU baselines.

    full():      the whole step as the oracle composes it (USP layout as an
                 index permutation, attention partials of every rank, the
                 log-sum-exp merge, the inverse layout) and the CFG combine.
    attention(): plain fp64 attention of the given query rows (all heads)
                 against every key, the oracle's definition of the result.
    cfg():       the CFG combine of a leading fraction of the elements."""

    def __init__(self, w, U: int):
        import synth
        from oracle import layout as olayout
        self.w, self.U = w, U
        self.L = olayout.make_layout(w.B, w.S, w.H, w.D, U, w.R)
        q, k, v = w.qkv()
        self.qkv = [synth.as_f64(t) for t in (q, k, v)]
        self.pred = synth.as_bits(w.cfg_pair()).reshape(2, -1)

    def full(self):
        from oracle import cfg as ocfg
        from oracle import usp as ousp
        o, _ = ousp.usp_attention(self.L, *self.qkv)
        c = ocfg.cfg_combine_bits(self.pred, self.w.cfg_in, self.w.g, self.w.cfg_out)
        return o, c

    def rows(self, n: int, seed: int):
        import numpy as np
        return np.sort(np.random.default_rng(seed).choice(self.w.S, size=min(n, self.w.S), replace=False))

    def attention(self, rows) -> float:
        from oracle import attention as oatt
        w = self.w
        q, k, v = self.qkv
        for b in range(w.B):
            oatt.attention(q[b:b + 1, rows], k[b:b + 1], v[b:b + 1])
        return 4.0 * w.B * w.H * len(rows) * w.S * w.D

    def cfg(self, frac: float):
        from oracle import cfg as ocfg
        n = max(1, int(self.pred.shape[1] * frac))
        ocfg.cfg_combine_bits(self.pred[:, :n], self.w.cfg_in, self.w.g, self.w.cfg_out)


def oracle_baseline(w, U: int, budget_s: float):
    """The oracle's attention timed on the host cores: every query row when
    that fits budget_s (estimated from 64 rows), else a seeded sample of rows
    sized to the budget, with the full time extrapolated from the sampled
    rate and labelled as such."""
    st = OracleStep(w, U)
    t0 = time.perf_counter()
    st.attention(st.rows(64, 5))
    est = (time.perf_counter() - t0) * w.S / min(64, w.S)
    cores = blas_threads()
    full = est <= budget_s
    rows = st.rows(w.S if full else max(16, int(w.S * budget_s / est)), 6)
    t0 = time.perf_counter()
    fl = st.attention(rows)
    dt = time.perf_counter() - t0
    rate = fl / dt / 1e12
    res = {"value": round(rate, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle"}
    if full:
        res["sample"] = (f"full fp64 oracle attention: all {w.S} query rows x {w.H} heads x B={w.B} against all "
                         f"{w.S} keys, {dt:.2f} s on the host cores")
        res["full_s"] = round(dt, 3)
    else:
        res["sample"] = (f"fp64 oracle attention of {len(rows)} seeded query rows x {w.H} heads x B={w.B} against "
                         f"all {w.S} keys, {dt:.1f} s on the host cores")
        res["per_row_ms"] = round(dt / len(rows) * 1e3, 3)
        res["extrapolated_full_s"] = round(w.attn_flops / (rate * 1e12), 1)
    return res


def cpu_oracle_kernels(budget_s: float = 30.0):
    """The oracle's bandwidth steps timed on the host on the FLUX-like
    workload (U=4; the merge on FLUX-1008's R=2 partials): GB/s of the same
    algorithmic bytes the GPU lines count.  Stops once the budget is spent."""
    import numpy as np
    import synth
    from oracle import attention as oatt
    from oracle import cfg as ocfg
    from oracle import fp8 as ofp8
    from oracle import layout as olayout
    from oracle import rope as orope
    from oracle import ulysses as ou
    w = synth.WORKLOADS["flux1024"]
    L = olayout.make_layout(w.B, w.S, w.H, w.D, 4, 1)
    planes = [synth.as_bits(t) for t in w.qkv()]
    eb = 2
    plane_bytes = w.B * w.S * w.H * w.D * eb
    res = {}
    t_all = time.perf_counter()

    def timed(name, nbytes, fn):
        if time.perf_counter() - t_all > budget_s:
            return None
        t0 = time.perf_counter()
        out = fn()
        dt = time.perf_counter() - t0
        res[name + "_GBs"] = round(nbytes / dt / 1e9, 3)
        return out

    send = timed("s2h_pack", 6 * plane_bytes, lambda: ou.s2h_pack(L, planes, "bf16", "bf16"))
    recv = None if send is None else timed("a2a", 6 * plane_bytes, lambda: ou.a2a(L, "s2h", 3, send))
    if recv is not None:
        timed("s2h_unpack", 6 * plane_bytes, lambda: ou.s2h_unpack(L, recv, "bf16", ("bf16", "bf16", "f16")))
    w8 = synth.WORKLOADS["flux1008"]
    L8 = olayout.make_layout(w8.B, w8.S, w8.H, w8.D, 4, w8.R)
    Sr = L8.ring_len[0]
    rng = np.random.default_rng(0)
    parts = [(rng.standard_normal((1, Sr, w8.H, w8.D)), rng.standard_normal((1, w8.H, Sr))) for _ in range(2)]
    timed("merge", Sr * w8.H * (2 * (w8.D * 4 + 4) + w8.D * 2), lambda: oatt.merge(parts))
    if recv is not None:
        cos, sin = (t.double().numpy() for t in synth.rope_tables_joint(w.S_txt, w.S, w.D))
        timed("receive_prep_rope", 6 * plane_bytes + 4 * w.S * w.D,
              lambda: orope.receive_prep(L, recv, "bf16", ["bf16", "bf16", "f16"], cos, sin, 0b011))
    pred = synth.as_bits(w.cfg_pair())
    n = pred.size // 2
    timed("cfg", 3 * n * eb, lambda: ocfg.cfg_combine_bits(pred, "bf16", w.g, "bf16"))
    timed("e4m3_pack_qv", 2 * plane_bytes + 2 * w.B * w.S * L.Hp * (w.D + 16),
          lambda: ofp8.s2h_pack(L, [planes[0], planes[2]], "bf16"))
    res["seconds"] = round(time.perf_counter() - t_all, 2)
    return res


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    rank, local_rank, ws = dist_env()
    torch.cuda.set_device(local_rank)
    if ws > 1:
        init_dist("nccl")
    dev = torch.device("cuda", local_rank)
    import synth
    import sequence_attention_gb300 as sa
    from sequence_attention_gb300.usp import UspPlan

    w, U = workload_config(args.workload, args.U)
    host_qkv, host_pred = w.qkv(), w.cfg_pair()
    inputs_sha = synth.digest(*host_qkv, host_pred)
    q, k, v = (t.to(dev) for t in host_qkv)
    pred = host_pred.to(dev)
    del host_qkv, host_pred
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device=dev)
    cfg_out = torch.empty(w.cfg_shape[1:], dtype=synth.torch_dtype(w.cfg_out), device=dev)
    plan = UspPlan(w.B, w.S, w.H, w.D, U, w.R, in_dtype=synth.torch_dtype(w.dtype), device=str(dev),
                   exchange=args.exchange, ring_merge=args.ring_merge)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    names = plan.steps() + ["cfg"]
    n_cfg_kernels = 1 if (pred.numel() // 2) % 8 == 0 else 2

    def step(ev=None, phases=True):
        # ev: 6 events to record (phases=True: between every two phases;
        # False: at the step's start and end only, events 0 and 5)
        def mark(i):
            if ev is not None and (phases or i in (0, 5)):
                ev[i].record(stream)
        mark(0)
        plan.layout_in(q, k, v)
        mark(1)
        plan.partials(out=out)  # writes out itself when the plan can (no layout-out pass then)
        mark(2)
        plan.merge()            # nothing when R = 1
        mark(3)
        plan.layout_out(out)
        mark(4)
        sa.dit_cfg_combine(pred, cfg_out, w.g)
        mark(5)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)

    K = args.steps
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0] or 0) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local_rank
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]

    def block(phases):
        barrier()
        torch.cuda.synchronize(dev)
        for i in range(K):
            flush.zero_()
            step(evs[i], phases)
        torch.cuda.synchronize(dev)
        barrier()

    # repeats of the K-step block: enough for >= 0.5 s of wall time, so that
    # the clock samples fall inside the timed region (the same count on
    # every rank)
    t0 = time.perf_counter()
    block(False)
    block_s = max(time.perf_counter() - t0, 1e-4)
    reps = int(max_over_ranks(float(max(1, math.ceil(args.min_timed_s / block_s))), dev))

    def timed(phases, nrep):
        ms = []
        with ClockSampler(gpu_index) as cs:
            for _ in range(nrep):
                block(phases)
                if phases:
                    ms.append([[e[i].elapsed_time(e[i + 1]) for e in evs] for i in range(5)])
                else:
                    ms.extend(e[0].elapsed_time(e[5]) for e in evs)
        return cs.summary(), ms

    # The timed steps: events at each step's start and end only (an event
    # between two phases breaks their launch overlap); L2 flushed between
    # steps, outside the events.
    clocks, step_ms = timed(False, reps)
    if any(r in clocks["reasons"] for r in BAD_REASONS):
        clocks, step_ms = timed(False, reps)   # rejected once: measure again
        clocks["remeasured"] = True
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, dev)
    # A second pass with events between the phases gives the split below:
    # ms per segment: layout-in, attention partials, merge, layout-out, CFG
    _, split_blocks = timed(True, 1)
    seg = split_blocks[0]
    split_ms = statistics.mean([sum(x) for x in zip(*seg)])
    attn_ms = statistics.mean(seg[1])          # the partial-attention launch alone
    flops = w.attn_flops
    value = ws * flops / (ms_max * 1e-3) / 1e12

    # bytes of the bandwidth steps (real elements read + written; the head
    # layout's padded heads are written, so they count)
    L = plan.L
    eb = 2 if w.dtype != "f32" else 4
    qkv_bytes = 3 * w.B * w.S * w.H * w.D * eb
    wire3 = 3 * w.B * w.S * L.Hp * w.D * eb
    o_bytes = w.B * w.S * w.H * w.D * 2
    wire1 = w.B * w.S * L.Hp * w.D * 2
    out_in_place = plan.direct_out(out)              # the attention writes out: no layout-out pass
    if plan.exchange == "direct":
        layout_in_bytes = qkv_bytes + wire3          # sequence planes in, head layout out
        layout_out_bytes = 0 if out_in_place else o_bytes + o_bytes   # real heads in, output out
    else:
        layout_in_bytes = (qkv_bytes + wire3) + 2 * wire3 + (wire3 + wire3)
        layout_out_bytes = (o_bytes + wire1) + 2 * wire1 + (wire1 + o_bytes)
    cfg_n = pred.numel() // 2
    cfg_bytes = cfg_n * (2 * pred.element_size() + cfg_out.element_size())

    peaks, peak_src = load_peaks()
    achieved = flops / (attn_ms * 1e-3) / 1e12
    # the ncu note covers the attention launch of the default FLUX-like workload
    traffic = traffic_per_launch(ATTN_SRC, TRAFFIC_NOTE) if (w.name == "flux1024" and w.R == 1) else None
    attn_kernel = f"attn_f32_kernel<{w.D}>" if w.dtype == "f32" else f"attn_tc_kernel<{w.D},false>"
    # merge bytes: R partials (in the plan's partial type) and their LSE per
    # real row and head, the output written once (16-bit)
    pb = plan.parts.element_size() if plan.parts is not None else 4
    merge_bytes = w.B * w.S * w.H * (w.R * (w.D * pb + 4) + w.D * 2)

    # one step alone, launched call by call and replayed from its own CUDA
    # graph (L2 flushed before each, median of 20): the cost of the launches
    one = plan.capture(q, k, v, out, extra=lambda: sa.dit_cfg_combine(pred, cfg_out, w.g))

    def one_step(fn):
        ts = []
        for i in range(25):
            flush.zero_()
            ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ga.record(stream)
            fn()
            gb.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 5:
                ts.append(ga.elapsed_time(gb))
        return statistics.median(ts)
    graph_ms = one_step(one.replay)
    eager_ms = one_step(lambda: step(None, False))
    del one
    other = {}
    if out_in_place:
        # the same step with the output exchange as a pass of its own: the
        # attention writes the head layout, the one-pass head->seq follows
        def step_pass():
            plan.layout_in(q, k, v)
            plan.partials()
            plan.merge()
            plan.layout_out(out)
            sa.dit_cfg_combine(pred, cfg_out, w.g)
        step_pass()
        other["step_layout_out_pass_ms"] = round(one_step(step_pass), 4)
    if w.R > 1:
        # the other form of the ring merge, one step alone (same launches)
        alt = "partials" if plan.ring_merge == "fold" else "fold"
        plan2 = UspPlan(w.B, w.S, w.H, w.D, U, w.R, in_dtype=synth.torch_dtype(w.dtype), device=str(dev),
                        exchange=args.exchange, ring_merge=alt)

        def step2():
            plan2.run(q, k, v, out)
            sa.dit_cfg_combine(pred, cfg_out, w.g)
        step2()
        other[f"step_{alt}_ms"] = round(one_step(step2), 4)
        del plan2

    # end to end through the public API: pinned host inputs in, results out
    e2e = run_e2e(plan, w, q, k, v, pred, out, cfg_out, dev, args)
    extra = {} if args.no_extra else {**back_to_back(w, U, dev), **bandwidth_at_scale(dev, flush, peaks),
                                      **receive_prep_at_scale(dev, flush),
                                      **fp8_wire_at_scale(dev, flush)}

    if "merge_step_f16" in extra.get("back_to_back", {}):
        # the merge launch alone (40 in a row, inputs out of L2): the step's
        # split above adds the launch latency its events expose
        extra["merge_kernel_us"] = extra["back_to_back"]["merge_step_f16"]["us"]
        extra["merge_kernel_GBs"] = extra["back_to_back"]["merge_step_f16"]["GBs"]
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_max, 4),
        "repeats": reps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)*0.5 bf16 Q/K/V, N(0,1) CFG branches)",
        "config": {**bench_config(w, U),
                   "exchange": plan.exchange,
                   **({"ring_merge": plan.ring_merge} if w.R > 1 else {}),
                   "l2": "flushed before every timed step (256 MiB write, outside the events)",
                   "timing": f"CUDA events around each step; the block of {K} steps repeated {reps} times "
                             f"back to back (>= {args.min_timed_s} s, so the clock samples fall inside); "
                             f"value = mean over all {K * reps} timed steps",
                   "inputs_sha256": inputs_sha},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks.get("bf16_tflops"), "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": traffic, "kernel": f"{attn_kernel} (dit_attn_partial)",
                     "peak_source": f"{peak_src} bf16 burst",
                     "frac_of_sustained": round(achieved / peaks.get("bf16_tflops_sustained",
                                                                      peaks["bf16_tflops"]), 4)},
        "kernels": {
            "layout_in_ms": round(statistics.mean(seg[0]), 4),
            "layout_in_GBs": round(layout_in_bytes / (statistics.mean(seg[0]) * 1e-3) / 1e9, 1),
            "attention_ms": round(attn_ms, 4), "attention_TFLOPs": round(achieved, 1),
            **({"merge_ms": round(statistics.mean(seg[2]), 4),
                "merge_GBs": round(merge_bytes / (statistics.mean(seg[2]) * 1e-3) / 1e9, 1)}
               if plan.parts is not None else {}),
            "layout_out_ms": round(statistics.mean(seg[3]), 4),
            "layout_out_GBs": (round(layout_out_bytes / (statistics.mean(seg[3]) * 1e-3) / 1e9, 1)
                               if layout_out_bytes else None),
            "layout_out": "in the attention's output view" if out_in_place else "a pass of its own",
            "cfg_ms": round(statistics.mean(seg[4]), 4),
            "cfg_GBs": round(cfg_bytes / (statistics.mean(seg[4]) * 1e-3) / 1e9, 1),
            "hbm_peak_GBs": peaks.get("hbm_gbs"),
            "step_graph_ms": round(graph_ms, 4),
            "step_eager_ms": round(eager_ms, 4),
            "step_split_ms": round(split_ms, 4),     # the same steps with events between phases
            **other,
            **extra,
        },
        "e2e": e2e,
        "gpu_launches": K * reps * (len(names) - 1 + n_cfg_kernels),
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = oracle_baseline(w, U, args.cpu_budget)
        if not args.no_extra:
            res["cpu_baseline"]["bandwidth_steps"] = cpu_oracle_kernels()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bandwidth_at_scale(dev, flush, peaks):
    """The merge (not in the R = 1 step) and CFG on the Wan-like shapes,
    each launch timed alone with L2 flushed before it (median of 10)."""
    import torch
    import sequence_attention_gb300 as sa
    import synth
    w = synth.WORKLOADS["wan"]
    R, H, D = w.R, w.H, w.D
    L = sa.dit_sp_layout_init(w.B, w.S, H, D, max(w.U), R)
    cap = L.S_cap
    parts = torch.randn((R, R, w.B, cap, H, D), dtype=torch.float32, device=dev)
    lse = torch.randn((R, R, w.B, H, cap), dtype=torch.float32, device=dev)
    out = torch.empty((R, w.B, cap, H, D), dtype=torch.bfloat16, device=dev)
    rl = L.ring_len
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ts = []
        for i in range(13):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                ts.append(s.elapsed_time(e))
        return statistics.median(ts)

    res = {}
    ms = timed(lambda: sa.dit_attn_merge_lse(parts, lse, out, None, rl))
    rows = sum(rl) * w.B
    nbytes = rows * H * (R * D * 4 + R * 4 + D * 2)
    res["merge_wan_ms"] = round(ms, 4)
    res["merge_wan_GBs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    del parts, lse, out
    pred = torch.randn(w.cfg_shape, dtype=torch.bfloat16, device=dev)
    cfg = torch.empty(w.cfg_shape[1:], dtype=torch.bfloat16, device=dev)
    ms = timed(lambda: sa.dit_cfg_combine(pred, cfg, w.g))
    res["cfg_wan_ms"] = round(ms, 4)
    res["cfg_wan_GBs"] = round(3 * cfg.numel() * 2 / (ms * 1e-3) / 1e9, 1)
    del pred, cfg
    torch.cuda.empty_cache()
    return res


def back_to_back(w, U, dev):
    """Each bandwidth kernel of the step on its own: 40 launches in a row on
    one stream (consecutive launches overlap their launch latency through
    programmatic dependent launch, as inside a model), rotating over enough
    buffer sets that every launch reads inputs last touched more than three
    L2 capacities earlier; one event pair around the 40 launches.  The step's
    own split (events between its phases) includes a launch gap per phase,
    which weighs most on the short CFG launch."""
    import torch
    import sequence_attention_gb300 as sa
    import synth
    L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, U, w.R)
    dt = torch.bfloat16 if w.dtype != "f32" else torch.float32
    eb = 2 if w.dtype != "f32" else 4
    shp, hs = (w.B, w.S, w.H, w.D), L.head_shape()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.current_stream(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)

    def rnd(shape, dtype=dt):
        return torch.randn(shape, generator=gen, dtype=torch.float32, device=dev).to(dtype)

    def timed(nbytes_in, make, launch, nbytes):
        nsets = max(2, -(-3 * l2 // max(nbytes_in, 1)))
        sets = [make() for _ in range(nsets)]
        for i in range(6):
            launch(sets[i % nsets])
        torch.cuda.synchronize(dev)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 40
        s.record(stream)
        for i in range(n):
            launch(sets[i % nsets])
        e.record(stream)
        torch.cuda.synchronize(dev)
        ms = s.elapsed_time(e) / n
        del sets
        torch.cuda.empty_cache()
        return {"us": round(ms * 1e3, 2), "GBs": round(nbytes / (ms * 1e-3) / 1e9, 1)}

    plane = w.B * w.S * w.H * w.D * eb
    wire1 = L.wire_elems(1) * eb
    wire3 = L.wire_elems(3) * eb
    S2H, H2S = sa.DIT_SEQ_TO_HEAD, sa.DIT_HEAD_TO_SEQ
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    v_dt = torch.float16 if dt == torch.bfloat16 else dt
    res = {}
    res["pack_s2h"] = timed(3 * plane, lambda: ([rnd(shp) for _ in range(3)], torch.empty(L.wire_elems(3), dtype=dt, device=dev)),
                            lambda x: sa.dit_ulysses_pack(L, S2H, x[0], x[1]), 3 * plane + wire3)
    res["a2a_s2h"] = timed(wire3, lambda: (rnd(L.wire_elems(3)), torch.empty(L.wire_elems(3), dtype=dt, device=dev)),
                           lambda x: sa.dit_a2a_sim(L, S2H, 3, x[0], x[1]), 2 * wire3)
    res["unpack_s2h"] = timed(wire3, lambda: (rnd(L.wire_elems(3)), [torch.empty(hs, dtype=t, device=dev) for t in (dt, dt, v_dt)]),
                              lambda x: sa.dit_ulysses_unpack(L, S2H, x[0], x[1], flag), 2 * wire3)
    res["pack_h2s"] = timed(wire1, lambda: (rnd(hs), torch.empty(L.wire_elems(1), dtype=dt, device=dev)),
                            lambda x: sa.dit_ulysses_pack(L, H2S, [x[0]], x[1]), plane + wire1)
    res["a2a_h2s"] = timed(wire1, lambda: (rnd(L.wire_elems(1)), torch.empty(L.wire_elems(1), dtype=dt, device=dev)),
                           lambda x: sa.dit_a2a_sim(L, H2S, 1, x[0], x[1]), 2 * wire1)
    res["unpack_h2s"] = timed(wire1, lambda: (rnd(L.wire_elems(1)), torch.empty(shp, dtype=dt, device=dev)),
                              lambda x: sa.dit_ulysses_unpack(L, H2S, x[0], [x[1]]), wire1 + plane)
    # the one-pass layout steps of the default step (no wire buffers)
    res["seq_to_head"] = timed(3 * plane, lambda: ([rnd(shp) for _ in range(3)],
                                                   [torch.empty(hs, dtype=t, device=dev) for t in (dt, dt, v_dt)]),
                               lambda x: sa.dit_ulysses_seq_to_head(L, x[0], x[1], flag), 3 * plane + wire3)
    res["head_to_seq"] = timed(wire1, lambda: (rnd(hs), torch.empty(shp, dtype=dt, device=dev)),
                               lambda x: sa.dit_ulysses_head_to_seq(L, x[0], x[1]), 2 * plane)
    cfg_in = {"f32": torch.float32, "bf16": torch.bfloat16}[w.cfg_in]
    cfg_out = {"f32": torch.float32, "bf16": torch.bfloat16}[w.cfg_out]
    n = 1
    for d in w.cfg_shape[1:]:
        n *= d
    ib, ob = (4 if cfg_in == torch.float32 else 2), (4 if cfg_out == torch.float32 else 2)
    res["cfg"] = timed(2 * n * ib, lambda: (rnd(w.cfg_shape, cfg_in), torch.empty(w.cfg_shape[1:], dtype=cfg_out, device=dev)),
                       lambda x: sa.dit_cfg_combine(x[0], x[1], w.g), n * (2 * ib + ob))
    # the receive preparation with RoPE on Q and K, and the e4m3 wire of Q
    # and V (records of D + 16 bytes per token and head), on these shapes
    cos, sin = synth.rope_tables_linear(w.S, w.D)
    cos, sin = cos.to(dev), sin.to(dev)
    res["seq_to_head_rope"] = timed(
        3 * plane, lambda: ([rnd(shp) for _ in range(3)], [torch.empty(hs, dtype=t, device=dev) for t in (dt, dt, v_dt)]),
        lambda x: sa.dit_ulysses_seq_to_head(L, x[0], x[1], flag, rope=(cos, sin)), 3 * plane + wire3 + 2 * w.S * w.D * 4)
    res["unpack_rope_s2h"] = timed(
        wire3, lambda: (rnd(L.wire_elems(3)), [torch.empty(hs, dtype=t, device=dev) for t in (dt, dt, v_dt)]),
        lambda x: sa.dit_ulysses_unpack_rope(L, x[0], x[1], cos, sin, 0b011, flag), 2 * wire3 + 2 * w.S * w.D * 4)
    rec = 2 * w.B * L.S_pad * L.Hp * (w.D + 16)
    nrec = L.wire_bytes_e4m3(2)
    res["pack_e4m3_qv"] = timed(2 * plane, lambda: ([rnd(shp), rnd(shp)], torch.empty(nrec, dtype=torch.uint8, device=dev)),
                                lambda x: sa.dit_ulysses_pack(L, S2H, x[0], x[1]), 2 * plane + rec)
    res["a2a_e4m3_qv"] = timed(nrec, lambda: (torch.randint(0, 120, (nrec,), dtype=torch.uint8, device=dev),
                                              torch.empty(nrec, dtype=torch.uint8, device=dev)),
                               lambda x: sa.dit_a2a_sim(L, S2H, 2, x[0], x[1]), 2 * rec)
    def packed_records():
        src = [rnd(shp), rnd(shp)]
        buf = torch.empty(nrec, dtype=torch.uint8, device=dev)
        sa.dit_ulysses_pack(L, S2H, src, buf)
        return (buf, [torch.empty(hs, dtype=dt, device=dev), torch.empty(hs, dtype=v_dt, device=dev)])
    res["unpack_e4m3_qv"] = timed(nrec, packed_records, lambda x: sa.dit_ulysses_unpack(L, S2H, x[0], x[1]),
                                  rec + 2 * (wire3 // 3))
    # the ring merge on the FLUX-1008-like partials (R = 2, the step's only
    # R > 1 bandwidth kernel at this scale): fp32 parts and LSE in, bf16 out
    wm = synth.WORKLOADS["flux1008"]
    Lm = sa.dit_sp_layout_init(wm.B, wm.S, wm.H, wm.D, max(wm.U), wm.R)
    R, cap, rl = wm.R, Lm.S_cap, Lm.ring_len
    mbytes = sum(rl) * wm.B * wm.H * (R * (wm.D * 4 + 4) + wm.D * 2)
    res["merge_flux1008"] = timed(
        R * R * wm.B * cap * wm.H * wm.D * 4,
        lambda: (torch.randn((R, R, wm.B, cap, wm.H, wm.D), generator=gen, device=dev),
                 torch.randn((R, R, wm.B, wm.H, cap), generator=gen, device=dev),
                 torch.empty((R, wm.B, cap, wm.H, wm.D), dtype=torch.bfloat16, device=dev)),
        lambda x: sa.dit_attn_merge_lse(x[0], x[1], x[2], None, rl), mbytes)
    # the merge of this workload's own step (f16 partials, bf16 out) when it has one
    if w.R > 1:
        Lw = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, U, w.R)
        Rw, capw, rlw = w.R, Lw.S_cap, Lw.ring_real
        res["merge_step_f16"] = timed(
            Rw * Rw * w.B * capw * w.H * w.D * 2,
            lambda: (torch.randn((Rw, Rw, w.B, capw, w.H, w.D), generator=gen, device=dev).half(),
                     torch.randn((Rw, Rw, w.B, w.H, capw), generator=gen, device=dev),
                     torch.empty((Rw, w.B, capw, w.H, w.D), dtype=torch.bfloat16, device=dev)),
            lambda x: sa.dit_attn_merge_lse(x[0], x[1], x[2], None, rlw),
            sum(rlw) * w.B * w.H * (Rw * (w.D * 2 + 4) + w.D * 2))
    # ... and with the step's own f16 partials
    mbytes16 = sum(rl) * wm.B * wm.H * (R * (wm.D * 2 + 4) + wm.D * 2)
    res["merge_flux1008_f16"] = timed(
        R * R * wm.B * cap * wm.H * wm.D * 2,
        lambda: (torch.randn((R, R, wm.B, cap, wm.H, wm.D), generator=gen, device=dev).half(),
                 torch.randn((R, R, wm.B, wm.H, cap), generator=gen, device=dev),
                 torch.empty((R, wm.B, cap, wm.H, wm.D), dtype=torch.bfloat16, device=dev)),
        lambda x: sa.dit_attn_merge_lse(x[0], x[1], x[2], None, rl), mbytes16)
    return {"back_to_back": res}


def receive_prep_at_scale(dev, flush):
    """The receive preparation with RoPE on Q and K against the plain
    seq->head unpack, on the FLUX-like (U=4) and Wan-like (U=8, R=4) shapes,
    and the paired text/image pack against the plain pack on the FLUX-like
    shape; each launch timed alone with L2 flushed before it (median of 10).
    Bytes: the wire read, the head-layout planes written and, with RoPE, the
    two float32 angle tables read once."""
    import torch
    import sequence_attention_gb300 as sa
    import synth
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ts = []
        for i in range(13):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                ts.append(s.elapsed_time(e))
        return statistics.median(ts)

    res = {}
    for name, U in (("flux1024", 4), ("wan", 8)):
        w = synth.WORKLOADS[name]
        L = sa.dit_sp_layout_init(w.B, w.S, w.H, w.D, U, w.R)
        recv = torch.randn(L.wire_elems(3), dtype=torch.bfloat16, device=dev)
        heads = [torch.empty(L.head_shape(), dtype=t, device=dev)
                 for t in (torch.bfloat16, torch.bfloat16, torch.float16)]
        cos, sin = (t.to(dev) for t in synth.rope_tables_joint(w.S_txt, w.S, w.D))
        moved = 2 * 3 * w.B * w.S * L.Hp * w.D * 2
        tables = 2 * w.S * (w.D // 2) * 4
        tag = "flux" if name == "flux1024" else name
        ms = timed(lambda: sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, recv, heads))
        res[f"unpack_{tag}_ms"] = round(ms, 4)
        res[f"unpack_{tag}_GBs"] = round(moved / (ms * 1e-3) / 1e9, 1)
        ms = timed(lambda: sa.dit_ulysses_unpack_rope(L, recv, heads, cos, sin, 0b011))
        res[f"unpack_rope_{tag}_ms"] = round(ms, 4)
        res[f"unpack_rope_{tag}_GBs"] = round((moved + tables) / (ms * 1e-3) / 1e9, 1)
        if w.S_txt > 0:
            joint = [torch.randn((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
            txt = [j[:, :w.S_txt].contiguous() for j in joint]
            img = [j[:, w.S_txt:].contiguous() for j in joint]
            send = torch.empty(L.wire_elems(3), dtype=torch.bfloat16, device=dev)
            pmoved = 3 * w.B * w.S * (w.H + L.Hp) * w.D * 2
            ms = timed(lambda: sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, joint, send))
            res[f"pack_{tag}_ms"] = round(ms, 4)
            res[f"pack_{tag}_GBs"] = round(pmoved / (ms * 1e-3) / 1e9, 1)
            ms = timed(lambda: sa.dit_ulysses_pack_joint(L, txt, img, send))
            res[f"pack_joint_{tag}_ms"] = round(ms, 4)
            res[f"pack_joint_{tag}_GBs"] = round(pmoved / (ms * 1e-3) / 1e9, 1)
            del joint, txt, img, send
        del recv, heads
        torch.cuda.empty_cache()
    return res


def fp8_wire_at_scale(dev, flush):
    """The e4m3 wire of Q and V (cache-dit's Async FP8 Ulysses Attention) on
    the FLUX-like (U=4) and Wan-like (U=8, R=4) shapes: the quantizing pack,
    the exchange of the records and the decoding unpack, each launch timed
    alone with L2 flushed before it (median of 10), and the whole seq->head
    layout step (K on its own 16-bit exchange) against the all-16-bit one.
    Bytes: real elements read and records written (D + 16 bytes per token
    and head) and the reverse for the unpack."""
    import torch
    import sequence_attention_gb300 as sa
    import synth
    from sequence_attention_gb300.usp import UspPlan
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ts = []
        for i in range(13):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                ts.append(s.elapsed_time(e))
        return statistics.median(ts)

    res = {}
    for name, U in (("flux1024", 4), ("wan", 8)):
        w = synth.WORKLOADS[name]
        tag = "flux" if name == "flux1024" else name
        q, k, v = (torch.randn((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device=dev) for _ in range(3))
        plan16 = UspPlan(w.B, w.S, w.H, w.D, U, w.R, device=str(dev), exchange="a2a")
        plan1 = UspPlan(w.B, w.S, w.H, w.D, U, w.R, device=str(dev), exchange="direct")
        plan8 = UspPlan(w.B, w.S, w.H, w.D, U, w.R, device=str(dev), fp8_qv=True)
        L = plan8.L
        rec = 2 * w.B * w.S * L.Hp * (w.D + 16)
        real = 2 * w.B * w.S * w.H * w.D * 2
        heads = 2 * w.B * w.S * L.Hp * w.D * 2
        ms = timed(lambda: sa.dit_ulysses_pack(L, sa.DIT_SEQ_TO_HEAD, [q, v], plan8.send_qv))
        res[f"pack_e4m3_{tag}_GBs"] = round((real + rec) / (ms * 1e-3) / 1e9, 1)
        ms = timed(lambda: sa.dit_a2a_sim(L, sa.DIT_SEQ_TO_HEAD, 2, plan8.send_qv, plan8.recv_qv))
        res[f"a2a_e4m3_{tag}_GBs"] = round(2 * rec / (ms * 1e-3) / 1e9, 1)
        ms = timed(lambda: sa.dit_ulysses_unpack(L, sa.DIT_SEQ_TO_HEAD, plan8.recv_qv, [plan8.q_h, plan8.v_h]))
        res[f"unpack_e4m3_{tag}_GBs"] = round((rec + heads) / (ms * 1e-3) / 1e9, 1)
        res[f"layout_in_bf16_{tag}_ms"] = round(timed(lambda: plan16.layout_in(q, k, v)), 4)
        res[f"layout_in_e4m3_qv_{tag}_ms"] = round(timed(lambda: plan8.layout_in(q, k, v)), 4)
        res[f"layout_in_direct_{tag}_ms"] = round(timed(lambda: plan1.layout_in(q, k, v)), 4)
        res[f"wire_bytes_ratio_{tag}"] = round((rec + w.B * w.S * L.Hp * w.D * 2) /
                                               (3 * w.B * w.S * L.Hp * w.D * 2), 4)
        del q, k, v, plan16, plan8, plan1
        torch.cuda.empty_cache()
    return res


def run_sweep(args):
    """One JSON line per workload: the full step (layout, attention partials,
    merge, layout back, CFG) with per-segment times, on one GPU."""
    import torch
    import synth
    import sequence_attention_gb300 as sa
    from sequence_attention_gb300.usp import UspPlan
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cases = [("tiny", 2), ("flux1024", 2), ("flux1024", 4), ("flux1008", 4), ("flux1008_4480", 4),
             ("qwen1328", 5), ("wan", 8)]
    for name, U in cases:
        w = synth.WORKLOADS[name]
        q, k, v = (t.to(dev) for t in w.qkv())
        pred = w.cfg_pair().to(dev)
        out = torch.empty((w.B, w.S, w.H, w.D), dtype=q.dtype, device=dev)
        cfg_out = torch.empty(w.cfg_shape[1:], dtype=synth.torch_dtype(w.cfg_out), device=dev)
        plan = UspPlan(w.B, w.S, w.H, w.D, U, w.R, in_dtype=synth.torch_dtype(w.dtype), device=str(dev),
                       exchange=args.exchange, ring_merge=args.ring_merge)
        stream = torch.cuda.current_stream(dev)
        reps = 3 if name == "wan" else 10
        seg = [[] for _ in range(5)]
        for i in range(reps + 3):
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            ev[0].record(stream)
            plan.layout_in(q, k, v)
            ev[1].record(stream)
            plan.partials(out=out)
            ev[2].record(stream)
            plan.merge()
            ev[3].record(stream)
            plan.layout_out(out)
            ev[4].record(stream)
            sa.dit_cfg_combine(pred, cfg_out, w.g)
            ev[5].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                for j in range(5):
                    seg[j].append(ev[j].elapsed_time(ev[j + 1]))
        med = [statistics.median(x) for x in seg]
        fl = w.attn_flops
        tf = fl / (med[1] * 1e-3) / 1e12
        tfm = fl / ((med[1] + med[2]) * 1e-3) / 1e12
        L = plan.L
        # merge bytes: R partials (O in the plan's partial type, and LSE) of
        # every ring block read, the output written
        rows = w.B * w.S * w.H
        pb = plan.parts.element_size() if plan.parts is not None else 0
        merge_bytes = rows * (w.R * (w.D * pb + 4) + w.D * plan.o_h.element_size()) if plan.parts is not None else 0
        res = {"workload": name, "U": U, "R": w.R, "B": w.B, "S": w.S, "H": w.H, "D": w.D, "dtype": w.dtype,
               "step_ms": round(sum(med), 4), "layout_in_ms": round(med[0], 4),
               "attention_ms": round(med[1], 4), "attention_TFLOPs": round(tf, 1),
               "attention_frac_of_measured_peak": round(tf / peaks["bf16_tflops"], 4) if w.dtype != "f32" else None,
               "merge_ms": round(med[2], 4),
               "merge_GBs": round(merge_bytes / (med[2] * 1e-3) / 1e9, 1) if plan.parts is not None else None,
               "ring_merge": plan.ring_merge,
               "attention_plus_merge_TFLOPs": round(tfm, 1),
               "layout_out_ms": round(med[3], 4), "cfg_ms": round(med[4], 4),
               "layout_out": "in the attention's output view" if plan.direct_out(out) else "a pass of its own",
               "heads_padded": L.Hp - w.H, "status": int(plan.status.item()),
               "range_flag": int(plan.range_flag.item()), "exchange": plan.exchange}
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = oracle_baseline(w, U, args.cpu_budget)
        print(json.dumps(res), flush=True)
        del q, k, v, pred, out, cfg_out, plan
        torch.cuda.empty_cache()


def run_e2e(plan, w, q, k, v, pred, out, cfg_out, dev, args):
    """End to end through the public API: every step copies its inputs from
    pinned host memory and reads both results back.  Copies run on their own
    streams and overlap the neighbouring steps' kernels (inputs and outputs
    are double-buffered); all of them are inside the timed region."""
    import torch
    import sequence_attention_gb300 as sa
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hp = pred.cpu().pin_memory()
    ho = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    hc = [torch.empty(cfg_out.shape, dtype=cfg_out.dtype).pin_memory() for _ in range(2)]
    din = [(q, k, v, pred)] + [tuple(torch.empty_like(t) for t in (q, k, v, pred))]
    dout = [(out, cfg_out), (torch.empty_like(out), torch.empty_like(cfg_out))]
    comp = torch.cuda.current_stream(dev)
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    for e in in_free + out_free:
        e.record(comp)

    def upload(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            h2d.wait_event(in_free[b])
            for dst, src in zip(din[b], (hq, hk, hv, hp)):
                dst.copy_(src, non_blocking=True)
            in_ready[b].record(h2d)

    def run(n):
        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            comp.wait_event(in_ready[b])
            comp.wait_event(out_free[b])
            dq, dk, dv, dp = din[b]
            o, c = dout[b]
            plan.run(dq, dk, dv, o)
            sa.dit_cfg_combine(dp, c, w.g)
            in_free[b].record(comp)
            out_ready[b].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(out_ready[b])
                ho[b].copy_(o, non_blocking=True)
                hc[b].copy_(c, non_blocking=True)
                out_free[b].record(d2h)
        comp.wait_stream(d2h)

    run(3)
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, 50))
    barrier()
    torch.cuda.synchronize(dev)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(comp)
    run(n)
    e.record(comp)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(s.elapsed_time(e) / n, dev)
    _, _, ws = dist_env()
    h2d_b = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hp))
    d2h_b = ho[0].numel() * ho[0].element_size() + hc[0].numel() * hc[0].element_size()
    return {"value": round(ws * w.attn_flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b, "ms_per_step": round(ms, 4),
            "note": "inputs H2D and results D2H every step on copy streams overlapping adjacent steps"}


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle as it stands, timed on the host cores on this arm's
    workload.  Each step is one measured slice of the workload: fp64
    attention of a seeded sample of query rows (all heads, every key) and
    the CFG combine of the same fraction of the prediction tensors, the
    sample sized so that the W + K steps take about --ref-budget seconds (a
    whole oracle step, with its layout permutations, takes longer than the
    run may: about half a minute at the FLUX-like size).  ms_per_step and
    value are the timed steps' own wall time and work; nothing is
    extrapolated."""
    rank, _, ws = dist_env()
    if rank != 0:
        return
    w, U = workload_config(args.workload, args.U)
    st = OracleStep(w, U)
    W = max(args.warmup, 3)
    per_step = args.ref_budget / (args.steps + W)
    n = min(64, w.S)
    # warm-up steps, each resizing the sample from the last one's cost
    for i in range(W):
        t0 = time.perf_counter()
        st.attention(st.rows(n, 10 + i))
        st.cfg(n / w.S)
        dt = max(time.perf_counter() - t0, 1e-6)
        # the cost grows faster than the row count (numpy temporaries), so
        # the resize is damped and bounded
        n = max(16, min(w.S, 4 * n, max(n // 4, int(n * (per_step / dt) ** 0.7))))
    frac = n / w.S
    times, flops = [], 0.0
    for i in range(args.steps):
        rows = st.rows(n, 100 + i)
        t0 = time.perf_counter()
        flops += st.attention(rows)
        st.cfg(frac)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = flops / total / 1e12
    ms = total / max(args.steps, 1) * 1e3
    cores = blas_threads()
    sample = (f"each step: fp64 oracle attention of {n} seeded query rows ({100 * frac:.1f} % of {w.S}) x {w.H} "
              f"heads x B={w.B} against all {w.S} keys, and the oracle CFG combine of the same fraction of "
              f"[2,{','.join(map(str, w.cfg_shape[1:]))}]; value = the timed steps' attention flops / their wall time")
    res = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
           "steps": args.steps, "warmup": W, "ms_per_step": round(ms, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1)*0.5 bf16 Q/K/V, N(0,1) CFG branches)", "impl": "reference",
           "config": bench_config(w, U),
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="flux1024")
    ap.add_argument("--U", type=int, default=None)
    ap.add_argument("--cpu-budget", type=float, default=12.0, dest="cpu_budget",
                    help="seconds of oracle work for the cpu_baseline (a whole step when it fits)")
    ap.add_argument("--ref-budget", type=float, default=120.0, dest="ref_budget",
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the Wan-size merge/CFG timings")
    ap.add_argument("--sweep", action="store_true", help="one line per workload instead of the bench line")
    ap.add_argument("--exchange", choices=("direct", "a2a"), default="direct",
                    help="layout steps in one pass (direct) or as pack / exchange / unpack (a2a)")
    ap.add_argument("--ring-merge", choices=("fold", "partials"), default=None, dest="ring_merge",
                    help="R > 1: key blocks folded in the attention kernel, or partials then the merge kernel "
                         "(default: the plan's choice, fold on 16-bit inputs)")
    ap.add_argument("--min-timed-s", type=float, default=0.5, dest="min_timed_s",
                    help="repeat the K-step block until the timed region lasts this long")
    args = ap.parse_args(argv)
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
