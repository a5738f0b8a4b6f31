#!/usr/bin/env python
"""Benchmark of the quantized-KV speculative decode-attention hot path.

One step = one pass over every stage of the path for one layer of a
Llama-2-7B-shaped model (32 heads, head_dim 128, hierarchical INT8/INT4 cache
with G = 128, 8K quantized context):
  1. INT8 verify attention: gamma = 8 causal query tokens over the quantized
     cache, the bf16 residual buffer and the 8 pending speculative tokens
     (split-K dequant + QK^T + online softmax + PV, bf16 tail, fused combine);
  2. top-64 per KV head under the INT4 (upper-nibble) keys, for the last query token;
  3. quantize-append of the 8 accepted tokens.  This includes a flush of G tokens
     from the 2G residual buffer into the quantized cache.
The host counters are restored after each step, so every step is identical.
Each step runs as one CUDA-graph replay of the C-ABI calls.  The steps rotate
over 4 cache copies (4 x 76 MB > L2), so no step reads L2-resident inputs.

``--impl reference`` times the CPU oracle on the same workload and metric.
Under torchrun with N > 1, each rank runs an independent replica.  The path
has no cross-GPU exchange.
"""
import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import kvq_inputs as ki  # noqa: E402

METRIC = "quant-KV decode attention: ms/call, KV tok/s, HBM GB/s (% of ~8 TB/s)"
UNIT = "KV tok/s"
WORKLOAD = "llama7b-layer-verify-8k"


# --------------------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------------------

class Spec:
    B, Hq, Hkv, D, G = 1, 32, 32, 128, 128
    Lq = 8192
    r0 = 2 * 128 - 4            # residual fill before the step: the append flushes a group
    gamma = 8
    P = 8                       # pending speculative tokens (all visible causally)
    top_k = 64
    n_accept = 8
    copies = 4

    @property
    def n_prefill(self):
        return self.Lq + self.r0

    @property
    def kv_tokens_per_step(self):
        return self.B * (self.Lq + self.r0 + self.P)

    def attend_bytes(self):
        """Algorithmic bytes of the INT8 verify call: both nibble planes of
        keys and values, key/value scale+zero, and the bf16 residual tokens."""
        per_tok = 4 * self.D // 2 + 2 * self.D * 4 // self.G + 2 * 4 * (self.D // self.G)
        return self.B * self.Hkv * (self.Lq * per_tok + self.r0 * 2 * self.D * 2)

    def topk_bytes(self):
        per_tok = self.D // 2 + 2 * self.D * 4 // self.G
        return self.B * self.Hkv * self.Lq * per_tok


def make_inputs(spec: Spec, seed: int = 0):
    K, V = ki.kv_stream(seed, spec.B, spec.Hkv, spec.n_prefill + spec.n_accept, spec.D)
    q = ki.queries(seed, spec.B, spec.gamma, spec.Hq, spec.D)
    pk, pv = ki.pending(seed, spec.B, spec.Hkv, spec.P, spec.D)
    return dict(K=K[:, :, :spec.n_prefill], V=V[:, :, :spec.n_prefill],
                Knew=K[:, :, spec.n_prefill:], Vnew=V[:, :, spec.n_prefill:], q=q, pk=pk, pv=pv)


# --------------------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------------------
# device arm
# --------------------------------------------------------------------------------------

def run_device(args, rank, world):
    import quantized_kv_speculative_gb300 as kvq
    from quantized_kv_speculative_gb300 import _build
    if rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    lib = kvq.load_library()
    spec = Spec()
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = make_inputs(spec)
    up = lambda x: ki.f32_to_bf16_tensor(x, dev)
    K, V = up(inp["K"]), up(inp["V"])
    q, pk, pv = up(inp["q"]), up(inp["pk"]), up(inp["pv"])
    kn, vn = up(inp["Knew"]), up(inp["Vnew"])
    q_spec = q[:, -1].contiguous()
    caches, wss = [], []
    for _ in range(spec.copies):
        c = kvq.QuantizedKVCache(spec.B, spec.Hkv, spec.D, spec.G, "hier8", spec.Lq + 2 * spec.G)
        kvq.kvq_quantize_append(c, K, V)                      # bulk cache build (prefill)
        caches.append(c)
        wss.append(kvq.make_workspace(c, spec.Hq, spec.gamma, spec.top_k))
    torch.cuda.synchronize()
    assert caches[0].state() == (spec.Lq, spec.r0, 0), caches[0].state()
    out = torch.empty_like(q)
    lse = torch.empty((spec.B, spec.gamma, spec.Hq), dtype=torch.float32, device=dev)
    idx = torch.empty((spec.B, spec.Hkv, spec.top_k), dtype=torch.int32, device=dev)
    sc = torch.empty((spec.B, spec.Hkv, spec.top_k), dtype=torch.float32, device=dev)

    # The top-k reads only the quantized keys, so it runs on a second stream,
    # concurrent with the attention (which reads the residual buffer the append
    # then rewrites, so the append follows it on the first stream).
    side = torch.cuda.Stream()

    def step(i, stream=None):
        s0 = stream if stream is not None else torch.cuda.current_stream()
        c = caches[i % spec.copies]
        ws = wss[i % spec.copies]
        st = c.state()
        fork = torch.cuda.Event()
        fork.record(s0)
        side.wait_event(fork)
        kvq.kvq_attend(c, "int8", q, pk, pv, out=out, lse=lse, workspace=ws, stream=s0)
        kvq.kvq_topk(c, "int4", q_spec, spec.top_k, idx_out=idx, score_out=sc, workspace=ws, stream=side)
        join = torch.cuda.Event()
        join.record(side)
        kvq.kvq_quantize_append(c, kn, vn, stream=s0)
        s0.wait_event(join)
        c.set_state(st)

    # attend, top-k, then the append: one flush kernel when the residual buffer
    # reaches 2G (it also writes the new residual rows), else one residual-write
    # kernel
    T = spec.r0 + spec.n_accept
    f = 0 if T < 2 * spec.G else T // spec.G - 1
    launches_per_step = 2 + (1 if f > 0 else 0) + (1 if (T - max(spec.r0, f * spec.G)) > 0 and f == 0 else 0)
    # warm-up eagerly (also sets kernel attributes outside any capture)
    for i in range(max(args.warmup, spec.copies)):
        step(i)
    torch.cuda.synchronize()
    for ws in wss:
        assert kvq.kvq_workspace_status(ws) == 0

    # one graph per cache copy
    cap_stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(cap_stream):
        for j in range(spec.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                step(j, stream=cap_stream)
            graphs.append(g)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        graphs[i % spec.copies].replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    for i in range(args.steps):
        graphs[i % spec.copies].replay()
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    value = whole_job_rate(spec.kv_tokens_per_step, world, ms_step * 1e-3)

    # ---- dominant kernel: INT8 verify attention, back-to-back launches ----
    def per_call_ms(fn, reps=64, rounds=8):
        gk = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(gk, stream=cap_stream):
                for i in range(reps):
                    fn(i, cap_stream)
        torch.cuda.synchronize()
        gk.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(rounds):
            gk.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * rounds)

    def attend_only(i, s):
        kvq.kvq_attend(caches[i % spec.copies], "int8", q, pk, pv, out=out, lse=lse,
                       workspace=wss[i % spec.copies], stream=s)

    def topk_only(i, s):
        kvq.kvq_topk(caches[i % spec.copies], "int4", q_spec, spec.top_k, idx_out=idx, score_out=sc,
                     workspace=wss[i % spec.copies], stream=s)

    def append_only(i, s):
        c = caches[i % spec.copies]
        st = c.state()
        kvq.kvq_quantize_append(c, kn, vn, stream=s)
        c.set_state(st)

    att_ms = per_call_ms(attend_only)
    topk_ms = per_call_ms(topk_only)
    app_ms = per_call_ms(append_only)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured"
    if not peak:
        peak, peak_src = 6800.0, "fallback"
    att_gbs = spec.attend_bytes() / (att_ms * 1e-3) / 1e9
    traffic = measured_traffic()

    # ---- e2e: public API with pinned host inputs and a host read of the results ----
    # The step's inputs (q, pending K/V, the appended K/V) sit in one pinned
    # host buffer and go up in one copy; the outputs and top-k indices come
    # back in two copies; the host then waits for them.
    parts = [ki.to_bf16_bits(inp[k]).view(np.int16).reshape(-1) for k in ("q", "pk", "pv", "Knew", "Vnew")]
    h_in = torch.from_numpy(np.concatenate(parts)).view(torch.bfloat16).pin_memory()
    d_in = torch.empty_like(h_in, device=dev)
    views, o = [], 0
    for x in (q, pk, pv, kn, vn):
        views.append(d_in[o:o + x.numel()].view(x.shape))
        o += x.numel()
    d_q, d_pk, d_pv, d_kn, d_vn = views
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_idx = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
    d_qs = d_q[:, -1] if spec.B == 1 else torch.empty_like(q_spec)   # B = 1: the last query row is contiguous
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size() + h_idx.numel() * h_idx.element_size()
    n_e2e = max(10, min(args.steps, 400))
    e2e_side = torch.cuda.Stream()

    def e2e_step(i):
        s0 = torch.cuda.current_stream()
        d_in.copy_(h_in, non_blocking=True)
        if spec.B != 1:
            d_qs.copy_(d_q[:, -1])
        c = caches[i % spec.copies]
        ws = wss[i % spec.copies]
        st = c.state()
        fork = torch.cuda.Event()
        fork.record(s0)
        e2e_side.wait_event(fork)
        kvq.kvq_attend(c, "int8", d_q, d_pk, d_pv, out=out, lse=lse, workspace=ws, stream=s0)
        kvq.kvq_topk(c, "int4", d_qs, spec.top_k, idx_out=idx, score_out=sc, workspace=ws, stream=e2e_side)
        join = torch.cuda.Event()
        join.record(e2e_side)
        kvq.kvq_quantize_append(c, d_kn, d_vn, stream=s0)
        c.set_state(st)
        s0.wait_event(join)
        h_out.copy_(out, non_blocking=True)
        h_idx.copy_(idx, non_blocking=True)
        s0.synchronize()

    for i in range(3):
        e2e_step(i)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, dev)
    for ws in wss:
        assert kvq.kvq_workspace_status(ws) == 0, "device status word set"

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 codes, f16 mma / fp32 accumulate, bf16 io",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q, 4 of 128 key channels x8 per head)",
        "config": {"workload": WORKLOAD, "batch": spec.B, "q_heads": spec.Hq, "kv_heads": spec.Hkv,
                   "head_dim": spec.D, "group": spec.G, "quantized_tokens": spec.Lq, "residual_tokens": spec.r0,
                   "gamma": spec.gamma, "pending": spec.P, "top_k": spec.top_k, "append_per_step": spec.n_accept,
                   "step": "int8 verify attend and int4 top-k on two streams, then quantize-append with one group flush",
                   "timing": "CUDA graph per step, CUDA events over the K steps",
                   "l2": f"rotating {spec.copies} cache copies of {spec.attend_bytes() / 1e6:.1f} MB each (> L2)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "calls": {"attend_int8_verify_ms": att_ms, "attend_gbs": att_gbs,
                  "topk_int4_ms": topk_ms, "topk_gbs": spec.topk_bytes() / (topk_ms * 1e-3) / 1e9,
                  "append_8_with_flush_ms": app_ms, "hbm_gbs_step": (spec.attend_bytes() + spec.topk_bytes()) / (ms_step * 1e-3) / 1e9},
        "roofline": {"kernel": "attend_kernel<INT8,128,1> (verify, gamma=8)", "bound": "hbm", "achieved": att_gbs,
                     "peak": peak, "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s", "frac": att_gbs / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": spec.attend_bytes(),
                     "timing": "64 back-to-back launches over 4 rotating caches, CUDA events"},
        "e2e": {"value": whole_job_rate(spec.kv_tokens_per_step, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    return result, spec, inp


# --------------------------------------------------------------------------------------
# oracle (CPU) arm
# --------------------------------------------------------------------------------------

def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest of the ranks' values of x (each rank's timed seconds or ms),
    through the default process group; x itself with one rank."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, world: int, seconds_per_step: float) -> float:
    """Whole-job throughput: every rank's units of one step over the slowest
    rank's time per step (replicas: per-rank work is fixed as ranks grow)."""
    return units_per_rank_step * world / seconds_per_step


def kernel_source_hash() -> str:
    """sha256 over the sources the attention kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    for f in ("kvq_attend.cu", "kvq_modes.cuh", "kvq_device.cuh", "kvq_internal.h"):
        h.update(open(os.path.join(ROOT, "quantized_kv_speculative_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def measured_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None if there is none or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "attend_int8_verify_8k.json")
    try:
        rec = json.load(open(path))
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


class OracleSample:
    """The CPU oracle on a bounded sample of the workload: every query row of a
    few KV heads, over the first ``lq`` quantized tokens of the same context plus
    the residual and pending tokens, then their top-k and the 8-token append."""

    def __init__(self, spec: Spec, inp, units=(0,), lq=None):
        import oracle
        self.oracle = oracle
        self.spec = spec
        self.units = list(units)
        self.lq = spec.Lq if lq is None else lq
        h = self.units
        n = self.lq + spec.r0
        self.c = oracle.OracleCache(1, len(h), spec.D, spec.G, "hier8", self.lq + 2 * spec.G)
        self.c.append(inp["K"][:, h, :n], inp["V"][:, h, :n])
        hg = spec.Hq // spec.Hkv
        qh = [x for u in h for x in range(u * hg, (u + 1) * hg)]
        self.q = inp["q"][:, :, qh]
        self.pk, self.pv = inp["pk"][:, h], inp["pv"][:, h]
        self.kn, self.vn = inp["Knew"][:, h], inp["Vnew"][:, h]

    def run_once(self):
        o = self.oracle
        o.attend(self.c, "int8", self.q, self.pk, self.pv)
        o.topk(self.c, "int4", self.q[:, -1], self.spec.top_k)
        saved = (self.c.Lq, self.c.r, self.c.res_k.copy(), self.c.res_v.copy())
        self.c.append(self.kn, self.vn)
        self.c.Lq, self.c.r, self.c.res_k, self.c.res_v = saved

    def kv_tok_per_s(self, seconds):
        """KV tokens/s in the workload's units (one KV token = all B*Hkv heads):
        unit-tokens processed by the sample / (B*Hkv) / time."""
        unit_tokens = len(self.units) * (self.lq + self.spec.r0 + self.spec.P)
        return unit_tokens / (self.spec.B * self.spec.Hkv) / seconds


def cpu_baseline(spec, inp, budget_s=12.0):
    s = OracleSample(spec, inp, units=(0,))
    s.run_once()
    n, t0 = 0, time.perf_counter()
    while True:
        s.run_once()
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 50:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": s.kv_tok_per_s(dt), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"1 of {spec.Hkv} KV heads: all {spec.gamma} query rows over the full context, its top-k "
                      f"and 8-token append; {n} repetitions; numpy single-threaded; scaled by the head fraction"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    spec = Spec()
    inp = make_inputs(spec)
    s = OracleSample(spec, inp, units=(0,))
    t0 = time.perf_counter()
    s.run_once()
    t_full = time.perf_counter() - t0
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    if per_step < t_full:
        lq = max(spec.G, int(spec.Lq * per_step / t_full) // spec.G * spec.G)
        s = OracleSample(spec, inp, units=(0,), lq=lq)
    for _ in range(args.warmup):
        s.run_once()
    times = []
    t_start = time.perf_counter()
    for i in range(args.steps):
        t1 = time.perf_counter()
        s.run_once()
        times.append(time.perf_counter() - t1)
        if time.perf_counter() - t_start > 1.3 * budget:
            break
    dt = sum(times) / len(times)
    v = s.kv_tok_per_s(dt)
    sample = (f"per step: 1 of {spec.Hkv} KV heads, all {spec.gamma} query rows over {s.lq} quantized "
              f"+ {spec.r0} residual + {spec.P} pending tokens, its top-{spec.top_k} and the 8-token append; "
              f"numpy single-threaded; tokens scaled to the workload's KV-token unit")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 0,
            "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": spec.kv_tokens_per_step / v * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 quantizer, f64 attention", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------------------
# other workloads (one JSON line each; the default run above is the headline)
# --------------------------------------------------------------------------------------

def _graph(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn(stream)
    torch.cuda.synchronize()
    return g


def _time_graph(g, reps):
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _peak():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"], "measured"
    except Exception:
        return 6800.0, "fallback"


def _bytes_per_token(mode, D, G):
    """Algorithmic bytes per quantized token per KV head read by a mode."""
    codes = {"int8": D, "int4": D // 2, "int2": D // 4, "int1": D // 8}[mode]   # keys + values
    return 2 * codes + 2 * D * 4 // G + 2 * 4 * (D // G)


def run_multilayer_spec(layers, lq, r0, gamma, drafts, append, reps=3, seed=0):
    """A 32-layer QuantSpec cycle: `drafts` INT4 draft steps (gamma = 1, the
    drafts so far pending) over every layer, one INT8 verify over every layer,
    and optionally the quantize-append of the accepted tokens."""
    import quantized_kv_speculative_gb300 as kvq
    from quantized_kv_speculative_gb300 import _build
    _build.build()
    B, H, D, G = 1, 32, 128, 128
    dev = torch.device("cuda")
    caches, wss = [], []
    n = lq + r0
    for layer in range(layers):
        K, V = ki.kv_stream_torch(seed + layer, B, H, n, D)
        c = kvq.QuantizedKVCache(B, H, D, G, "hier8", lq + 2 * G * (1 + append // G + 1))
        kvq.kvq_quantize_append(c, K, V)
        del K, V
        caches.append(c)
        wss.append(kvq.make_workspace(c, H, gamma, 0))
    torch.cuda.synchronize()
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 999)
    rnd = lambda *shape: torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
    qd = rnd(B, 1, H, D)
    qv = rnd(B, gamma, H, D)
    pk, pv = rnd(B, H, max(gamma, drafts), D), rnd(B, H, max(gamma, drafts), D)
    kn, vn = rnd(B, H, max(append, 1), D), rnd(B, H, max(append, 1), D)
    out_d, out_v = torch.empty_like(qd), torch.empty_like(qv)
    lse_d = torch.empty((B, 1, H), device=dev)
    lse_v = torch.empty((B, gamma, H), device=dev)
    pend = [(pk[:, :, :j].contiguous(), pv[:, :, :j].contiguous()) for j in range(1, drafts + 1)]
    pver = (pk[:, :, :gamma].contiguous(), pv[:, :, :gamma].contiguous())
    s = torch.cuda.Stream()

    def draft_step(j):
        def f(st):
            for L in range(layers):
                kvq.kvq_attend(caches[L], "int4", qd, pend[j][0], pend[j][1], out=out_d, lse=lse_d,
                               workspace=wss[L], stream=st)
        return f

    def verify(st):
        for L in range(layers):
            kvq.kvq_attend(caches[L], "int8", qv, pver[0], pver[1], out=out_v, lse=lse_v, workspace=wss[L], stream=st)

    def commit(st):
        for L in range(layers):
            c = caches[L]
            sv = c.state()
            kvq.kvq_quantize_append(c, kn[:, :, :append].contiguous(), vn[:, :, :append].contiguous(), stream=st)
            c.set_state(sv)

    # eager warm-up (kernel attributes are set outside any capture)
    draft_step(0)(None)
    verify(None)
    if append:
        commit(None)
    torch.cuda.synchronize()
    gd = [_graph(draft_step(j), s) for j in range(drafts)]
    gv = _graph(verify, s)
    gc_ = _graph(commit, s) if append else None
    t_draft = [_time_graph(g, reps) for g in gd]
    t_ver = _time_graph(gv, reps)
    t_app = _time_graph(gc_, reps) if append else 0.0
    for ws in wss:
        assert kvq.kvq_workspace_status(ws) == 0
    peak, src = _peak()
    res_b = r0 * 2 * D * 2 * H * B
    b_draft = layers * (B * H * lq * _bytes_per_token("int4", D, G) + res_b)
    b_ver = layers * (B * H * lq * _bytes_per_token("int8", D, G) + res_b)
    td = statistics.mean(t_draft)
    cycle_ms = sum(t_draft) + t_ver + t_app
    toks = B * layers * (sum(lq + r0 + j for j in range(1, drafts + 1)) + (lq + r0 + gamma))
    return {
        "draft_step_ms": td, "draft_step_gbs": b_draft / (td * 1e-3) / 1e9,
        "draft_frac": b_draft / (td * 1e-3) / 1e9 / peak,
        "draft_call_ms": td / layers,
        "verify_ms": t_ver, "verify_gbs": b_ver / (t_ver * 1e-3) / 1e9, "verify_frac": b_ver / (t_ver * 1e-3) / 1e9 / peak,
        "verify_call_ms": t_ver / layers,
        "append_ms": t_app, "cycle_ms": cycle_ms, "kv_tok_per_s": toks / (cycle_ms * 1e-3),
        "peak_gbs": peak, "peak_source": src, "launches_per_cycle": layers * (drafts + 1 + (2 if append else 0)),
    }


def run_specache(fmt, seed=0, reps=20):
    """SpeCache-style batched decode: batch 36, 32 q / 8 kv heads, D 128, G 32,
    32768 quantized + 32 residual tokens; top-64 from the speculative token,
    the fetch of those 64 tokens' 16-bit K/V from the full cache in pinned host
    memory, then attention (gamma = 2) with them at 16 bits."""
    import quantized_kv_speculative_gb300 as kvq
    from quantized_kv_speculative_gb300 import _build
    _build.build()
    B, Hq, H, D, G, lq, r0, k = 36, 32, 8, 128, 32, 32768, 32, 64
    K, V = ki.kv_stream_torch(seed, B, H, lq + r0, D)
    c = kvq.QuantizedKVCache(B, H, D, G, fmt, lq + 2 * G)
    kvq.kvq_quantize_append(c, K, V)
    ws = kvq.make_workspace(c, Hq, 2, k)
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 5)
    q = torch.randn((B, 2, Hq, D), generator=gen, device=dev).to(torch.bfloat16)
    pk = torch.randn((B, H, 2, D), generator=gen, device=dev).to(torch.bfloat16)
    pv = torch.randn((B, H, 2, D), generator=gen, device=dev).to(torch.bfloat16)
    qs = q[:, 1].contiguous()
    idx, sc = kvq.kvq_topk(c, fmt, qs, k, workspace=ws)
    # the full 16-bit cache, offloaded to pinned host memory
    hk = torch.empty(K.shape, dtype=torch.bfloat16, pin_memory=True)
    hv = torch.empty(V.shape, dtype=torch.bfloat16, pin_memory=True)
    hk.copy_(K)
    hv.copy_(V)
    sk, sv = kvq.kvq_gather_selected(hk, hv, idx)
    gi = idx.long().clamp_min(0)[..., None].expand(-1, -1, -1, D)
    assert torch.equal(sk, torch.gather(K, 2, gi)) and torch.equal(sv, torch.gather(V, 2, gi))
    del K, V, gi
    out = torch.empty_like(q)
    lse = torch.empty((B, 2, Hq), device=dev)
    s = torch.cuda.Stream()
    kvq.kvq_attend(c, fmt, q, pk, pv, idx, sk, sv, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    ga = _graph(lambda st: kvq.kvq_attend(c, fmt, q, pk, pv, idx, sk, sv, out=out, lse=lse, workspace=ws, stream=st), s)
    gt = _graph(lambda st: kvq.kvq_topk(c, fmt, qs, k, idx_out=idx, score_out=sc, workspace=ws, stream=st), s)
    # the fetch over 16 independent index sets (150 MB of rows > L2), per fetch
    nset = 16
    sets = [torch.randint(0, lq, (B, H, k), generator=gen, device=dev, dtype=torch.int32) for _ in range(nset)]
    sk2, sv2 = torch.empty_like(sk), torch.empty_like(sv)
    ta, tt = _time_graph(ga, reps), _time_graph(gt, reps)
    try:
        gg = _graph(lambda st: [kvq.kvq_gather_selected(hk, hv, ix, sel_k=sk2, sel_v=sv2, stream=st) for ix in sets], s)
        tg, fetch_err = _time_graph(gg, reps) / nset, None
    except Exception as ex:   # reported in the line instead of ending the run
        torch.cuda.synchronize()
        tg, fetch_err = float("nan"), f"{type(ex).__name__}: {ex}"[:200]
    assert kvq.kvq_workspace_status(ws) == 0
    # One SpeCache step: attention with the rows fetched the step before, the
    # top-k of the speculative token, and the fetch of the next step's rows.
    # Timed as one graph under three schedules: all on one stream; top-k and
    # fetch on a second stream beside the attention; top-k first, then the
    # attention with only the fetch beside it.  step_ms is the fastest.
    side = torch.cuda.Stream()
    idx_n, sc_n = torch.empty_like(idx), torch.empty_like(sc)
    sk_n, sv_n = torch.empty_like(sk), torch.empty_like(sv)
    att = lambda st: kvq.kvq_attend(c, fmt, q, pk, pv, idx, sk, sv, out=out, lse=lse, workspace=ws, stream=st)
    tpk = lambda st: kvq.kvq_topk(c, fmt, qs, k, idx_out=idx_n, score_out=sc_n, workspace=ws, stream=st)
    fch = lambda st: kvq.kvq_gather_selected(hk, hv, idx_n, sel_k=sk_n, sel_v=sv_n, stream=st)

    def forked(st, before, on_side, on_main):
        before(st)
        fork = torch.cuda.Event()
        fork.record(st)
        side.wait_event(fork)
        on_side(side)
        on_main(st)
        join = torch.cuda.Event()
        join.record(side)
        st.wait_event(join)
    schedules = {
        "one_stream": lambda st: (att(st), tpk(st), fch(st)),
        "topk_fetch_beside_attention": lambda st: forked(st, lambda x: None, lambda x: (tpk(x), fch(x)), att),
        "fetch_beside_attention": lambda st: forked(st, tpk, fch, att),
    }
    step_by = {}
    step_err = None
    for name, fn in schedules.items():
        try:
            fn(torch.cuda.current_stream())
            torch.cuda.synchronize()
            step_by[name] = _time_graph(_graph(fn, s), reps)
        except Exception as ex:   # reported in the line instead of ending the run
            torch.cuda.synchronize()
            step_err = f"{name}: {type(ex).__name__}: {ex}"[:200]
    best = min(step_by, key=step_by.get) if step_by else None
    t_step = step_by[best] if best else float("nan")
    assert kvq.kvq_workspace_status(ws) == 0
    # the link's measured rate for a plain copy: 1 GiB pinned host -> device
    hb = hk.view(-1)[: 1 << 29]
    db = torch.empty_like(hb, device=dev)
    db.copy_(hb, non_blocking=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(3):
        db.copy_(hb, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    h2d_gbs = 3 * hb.numel() * 2 / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del db, hk, hv
    peak, src = _peak()
    mode = fmt
    ba = B * H * (lq * _bytes_per_token(mode, D, G) + r0 * 2 * D * 2)
    codes_k = {"int2": D // 4, "int1": D // 8}[mode]
    bt = B * H * lq * (codes_k + 2 * D * 4 // G)
    return {"attend_ms": ta, "attend_gbs": ba / (ta * 1e-3) / 1e9, "attend_frac": ba / (ta * 1e-3) / 1e9 / peak,
            "attend_bytes": ba, "sel_kv_bytes": B * H * k * 2 * D * 2,
            "topk_ms": tt, "topk_gbs": bt / (tt * 1e-3) / 1e9, "topk_frac": bt / (tt * 1e-3) / 1e9 / peak,
            "fetch_ms": tg, "fetch_error": fetch_err, "fetch_gbs": B * H * k * 2 * D * 2 / (tg * 1e-3) / 1e9,
            "fetch_frac_of_h2d_copy": B * H * k * 2 * D * 2 / (tg * 1e-3) / 1e9 / h2d_gbs, "h2d_copy_gbs": h2d_gbs,
            "step_ms": t_step, "step_schedule": best, "step_ms_by_schedule": step_by, "step_error": step_err,
            "calls_sum_ms": ta + tt + tg,
            "kv_tok_per_s": B * (lq + r0 + 2) / (t_step * 1e-3),
            "peak_gbs": peak, "peak_source": src}


def run_sweep(seed=0):
    """Single-layer INT4 draft attention (gamma = 1, r = 128) over 8K..256K."""
    import quantized_kv_speculative_gb300 as kvq
    from quantized_kv_speculative_gb300 import _build
    _build.build()
    B, H, D, G = 1, 32, 128, 128
    dev = torch.device("cuda")
    peak, src = _peak()
    rows = []
    for lq in ki.SWEEP_CONTEXTS:
        n = lq + 128 + 128
        per_copy = B * H * lq * _bytes_per_token("int4", D, G)
        copies = max(1, min(8, math.ceil(4 * 129e6 / (B * H * lq * _bytes_per_token("int8", D, G)))))
        K, V = ki.kv_stream_torch(seed, B, H, n, D)
        caches = []
        for _ in range(copies):
            c = kvq.QuantizedKVCache(B, H, D, G, "hier8", lq + 2 * G)
            kvq.kvq_quantize_append(c, K, V)
            caches.append(c)
        del K, V
        wss = [kvq.make_workspace(c, H, 1, 0) for c in caches]
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed + lq)
        q = torch.randn((B, 1, H, D), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        lse = torch.empty((B, 1, H), device=dev)
        for i in range(copies):
            kvq.kvq_attend(caches[i], "int4", q, out=out, lse=lse, workspace=wss[i])
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        reps_in = 8 * copies

        def f(st):
            for i in range(reps_in):
                kvq.kvq_attend(caches[i % copies], "int4", q, out=out, lse=lse, workspace=wss[i % copies], stream=st)
        g = _graph(f, s)
        t = _time_graph(g, 5) / reps_in
        b = per_copy + B * H * 128 * 2 * D * 2
        rows.append({"context": lq, "ms": t, "gbs": b / (t * 1e-3) / 1e9, "frac": b / (t * 1e-3) / 1e9 / peak,
                     "copies_rotated": copies, "kv_tok_per_s": B * (lq + 128) / (t * 1e-3)})
        del caches, wss, g
        torch.cuda.empty_cache()
    return {"rows": rows, "peak_gbs": peak, "peak_source": src}


def run_profile_case(name, launches):
    """A few eager launches of one call, for ncu captures (no graphs, no timing)."""
    import quantized_kv_speculative_gb300 as kvq
    from quantized_kv_speculative_gb300 import _build
    _build.build()
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    rnd = lambda *shape: torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
    if name in ("attend-int8-verify-8k", "attend-int4-draft-32k", "topk-int4-8k"):
        B, H, D, G = 1, 32, 128, 128
        lq, r0 = (8192, 252) if name != "attend-int4-draft-32k" else (32768, 128)
        copies = 4
        K, V = ki.kv_stream_torch(0, B, H, lq + r0, D)
        caches = []
        for _ in range(copies):
            c = kvq.QuantizedKVCache(B, H, D, G, "hier8", lq + 2 * G)
            kvq.kvq_quantize_append(c, K, V)
            caches.append(c)
        gamma = 8 if name == "attend-int8-verify-8k" else 1
        ws = [kvq.make_workspace(c, H, gamma, 64) for c in caches]
        q = rnd(B, gamma, H, D)
        pk, pv = rnd(B, H, gamma, D), rnd(B, H, gamma, D)
        out = torch.empty_like(q)
        lse = torch.empty((B, gamma, H), device=dev)
        idx = torch.empty((B, H, 64), dtype=torch.int32, device=dev)
        for i in range(launches):
            c = caches[i % copies]
            if name == "topk-int4-8k":
                kvq.kvq_topk(c, "int4", q[:, 0].contiguous(), 64, idx_out=idx, workspace=ws[i % copies])
            else:
                mode = "int8" if gamma == 8 else "int4"
                kvq.kvq_attend(c, mode, q, pk, pv, out=out, lse=lse, workspace=ws[i % copies])
    elif name in ("attend-int2-specache-32k", "topk-int2-specache-32k"):
        B, Hq, H, D, G, lq, r0, k = 36, 32, 8, 128, 32, 32768, 32, 64
        K, V = ki.kv_stream_torch(0, B, H, lq + r0, D)
        c = kvq.QuantizedKVCache(B, H, D, G, "int2", lq + 2 * G)
        kvq.kvq_quantize_append(c, K, V)
        ws = kvq.make_workspace(c, Hq, 2, k)
        q = rnd(B, 2, Hq, D)
        pk, pv = rnd(B, H, 2, D), rnd(B, H, 2, D)
        idx, _ = kvq.kvq_topk(c, "int2", q[:, 1].contiguous(), k, workspace=ws)
        gi = idx.long().clamp_min(0)[..., None].expand(-1, -1, -1, D)
        sk, sv = torch.gather(K, 2, gi).contiguous(), torch.gather(V, 2, gi).contiguous()
        del K, V
        for i in range(launches):
            if name.startswith("topk"):
                kvq.kvq_topk(c, "int2", q[:, 1].contiguous(), k, idx_out=idx, workspace=ws)
            else:
                kvq.kvq_attend(c, "int2", q, pk, pv, idx, sk, sv, workspace=ws)
    elif name == "fetch-specache-host":
        # the SpeCache batch's fetch: 36 x 8 heads x 64 selected rows out of a
        # pinned host store of 4096 tokens per head (600 MB per K and V)
        B, H, D, N, k = 36, 8, 128, 4096, 64
        hk = torch.zeros((B, H, N, D), dtype=torch.bfloat16, pin_memory=True)
        hv = torch.zeros((B, H, N, D), dtype=torch.bfloat16, pin_memory=True)
        sets = [torch.randint(0, N, (B, H, k), generator=gen, device=dev, dtype=torch.int32) for _ in range(4)]
        for i in range(launches):
            kvq.kvq_gather_selected(hk, hv, sets[i % 4])
    else:
        raise SystemExit(f"unknown profile case {name}")
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": name, "launches": launches}))


def run_workload(name):
    t0 = time.perf_counter()
    if name == "llama7b-32l-spec-32k":
        r = run_multilayer_spec(32, 32768, 128, 8, 8, 0)
    elif name == "llama7b-32l-spec-128k":
        r = run_multilayer_spec(32, 131072, 253, 6, 6, 6)
    elif name in ("specache-b36-32k-int2", "specache-b36-32k-int1"):
        r = run_specache(name.split("-")[-1])
    elif name == "sweep-int4":
        r = run_sweep()
    else:
        raise SystemExit(f"unknown workload {name}")
    r["workload"] = name
    r["wall_s"] = time.perf_counter() - t0
    return r


# --------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", default=None, help="eager launches of one call for ncu captures")
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--workload", default=None,
                    help="extra measurement instead of the headline step: llama7b-32l-spec-32k, "
                         "llama7b-32l-spec-128k, specache-b36-32k-int2, specache-b36-32k-int1, sweep-int4, all")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    torch.cuda.set_device(local)
    if args.profile_case:
        run_profile_case(args.profile_case, args.launches)
        return
    if args.workload:
        names = (["llama7b-32l-spec-32k", "specache-b36-32k-int2", "specache-b36-32k-int1", "sweep-int4",
                  "llama7b-32l-spec-128k"] if args.workload == "all" else [args.workload])
        for nm in names:
            print(json.dumps(run_workload(nm)), flush=True)
            torch.cuda.empty_cache()
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    res, spec, inp = run_device(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(spec, inp)
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
