#!/usr/bin/env python
"""Benchmark of the quantized-KV speculative decode-attention hot path.

One step = one QuantSpec speculation cycle of a Llama-2-7B-shaped model at a
128K context: 32 layers, each with 32 heads x head_dim 128 of hierarchical
INT8/INT4 KV cache (G = 128) over 131072 quantized tokens plus 253 bf16
residual tokens.  Per layer:
  1. six INT4 draft attentions (1 query token each, the drafts so far pending:
     draft j sees j pending tokens), layer by layer for each draft step;
  2. one INT8 verify attention of the 6 draft tokens (gamma = 6, causal);
  3. the quantize-append of the 6 accepted tokens, which flushes one group of
     G tokens from the 2G residual buffer into the quantized cache.
The host counters are restored after each step, so every step is identical.
The three phases run as three CUDA graphs of the C-ABI calls (192 + 32 + 32
launches), with CUDA events between them, so the INT4 draft kernel's average
launch time is measured inside the timed region.  The 36.5 GB of quantized
cache (1.14 GB per layer) is far larger than L2, so no step reads L2-resident
data and no flush is needed.

The line also carries the single-layer 8K verify step (INT8 verify + INT4
top-64 + 8-token append) as an extra figure, and the CPU oracle timed on the
host cores (one core, then all cores) on a sample of the same cycle.

``--impl reference`` times the CPU oracle on all host cores on the same
workload and metric.  Under torchrun with N > 1, each rank runs an independent
replica; the path has no cross-GPU exchange.
"""
import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import multiprocessing  # noqa: E402
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
WORKLOAD = "llama7b-32l-spec-cycle-128k"


def _bytes_per_token(mode, D, G):
    """Algorithmic bytes per quantized token per KV head read by a mode: the
    mode's key and value code planes plus fp32 key and value scale/zero."""
    codes = {"int8": D, "int4": D // 2, "int2": D // 4, "int1": D // 8}[mode]   # keys + values
    return 2 * codes + 2 * D * 4 // G + 2 * 4 * (D // G)


# --------------------------------------------------------------------------------------
# workload: the 128K speculation cycle
# --------------------------------------------------------------------------------------

class CycleSpec:
    layers, B, H, D, G = 32, 1, 32, 128, 128
    Lq = 131072
    r0 = 253                    # residual fill before the cycle: the append of 6 flushes one group
    drafts = 6                  # INT4 draft steps, one query token each
    gamma = 6                   # INT8 verify query tokens (all drafts pending, causal)
    n_accept = 6

    def capacity(self):
        return self.Lq + 2 * self.G

    def kv_tokens_per_step(self):
        """KV tokens read per step (one KV token = all heads of one layer of one
        sequence): quantized + residual + pending tokens of every call."""
        per_layer = sum(self.Lq + self.r0 + j for j in range(1, self.drafts + 1)) + (self.Lq + self.r0 + self.gamma)
        return self.layers * self.B * per_layer

    def residual_bytes(self):
        return self.B * self.H * self.r0 * 2 * self.D * 2

    def draft_bytes_per_launch(self):
        return self.B * self.H * self.Lq * _bytes_per_token("int4", self.D, self.G) + self.residual_bytes()

    def verify_bytes_per_launch(self):
        return self.B * self.H * self.Lq * _bytes_per_token("int8", self.D, self.G) + self.residual_bytes()

    def launches_per_step(self):
        T = self.r0 + self.n_accept
        f = 0 if T < 2 * self.G else T // self.G - 1
        append = 1 if f > 0 else (1 if T > self.r0 else 0)   # the flush kernel also writes the new residual rows
        return self.layers * (self.drafts + 1 + append)

    # step inputs of one layer, in bf16 elements of one flat buffer:
    # draft queries [drafts][B,1,H,D], verify queries [B,gamma,H,D], pending K and V
    # of draft j = 1..drafts [B,H,j,D] each, appended K and V [B,H,n_accept,D] each
    def layer_input_elems(self):
        t = self.B * self.H * self.D
        return t * (self.drafts + self.gamma + 2 * sum(range(1, self.drafts + 1)) + 2 * self.n_accept)

    def layer_output_elems(self):
        return self.B * self.H * self.D * (self.drafts + self.gamma)


def _cycle_views(spec: CycleSpec, d_in, d_out):
    """Per-layer tensors viewed in the flat step input / output buffers."""
    B, H, D = spec.B, spec.H, spec.D
    layers = []
    for L in range(spec.layers):
        o = L * spec.layer_input_elems()
        take = lambda n, shape: (d_in[o:o + n].view(shape), o + n)
        qd = []
        for j in range(spec.drafts):
            x, o = take(B * H * D, (B, 1, H, D))
            qd.append(x)
        qv, o = take(B * spec.gamma * H * D, (B, spec.gamma, H, D))
        pend = []
        for j in range(1, spec.drafts + 1):
            pk, o = take(B * H * j * D, (B, H, j, D))
            pv, o = take(B * H * j * D, (B, H, j, D))
            pend.append((pk, pv))
        kn, o = take(B * H * spec.n_accept * D, (B, H, spec.n_accept, D))
        vn, o = take(B * H * spec.n_accept * D, (B, H, spec.n_accept, D))
        oo = L * spec.layer_output_elems()
        od = [d_out[oo + j * B * H * D: oo + (j + 1) * B * H * D].view(B, 1, H, D) for j in range(spec.drafts)]
        ob = oo + spec.drafts * B * H * D
        ov = d_out[ob: ob + B * spec.gamma * H * D].view(B, spec.gamma, H, D)
        layers.append(dict(qd=qd, qv=qv, pend=pend, kn=kn, vn=vn, od=od, ov=ov))
    return layers


def _cycle_host_inputs(spec: CycleSpec, seed=0):
    """Seeded bf16 step inputs (pinned host memory), N(0,1) like the cache."""
    g = ki.rng(seed, 9000)
    n = spec.layers * spec.layer_input_elems()
    x = g.standard_normal(n, dtype=np.float32)
    return torch.from_numpy(ki.to_bf16_bits(x).view(np.int16)).view(torch.bfloat16).pin_memory()


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


def _peak():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"], "measured"
    except Exception:
        return 6800.0, "fallback"


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
    for f in ("kvq_attend_kernel.cuh", "kvq_modes.cuh", "kvq_device.cuh", "kvq_internal.h"):
        h.update(open(os.path.join(ROOT, "quantized_kv_speculative_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def measured_traffic(name):
    """DRAM bytes per launch of a kernel from its committed ncu summary
    (profiles/<name>.json), or None if there is none or the kernel's sources
    changed since the counters were taken."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", name + ".json")))
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------------------
# device arm: the 128K cycle
# --------------------------------------------------------------------------------------

def run_device(args, rank, world):
    import quantized_kv_speculative_gb300 as kvq
    from quantized_kv_speculative_gb300 import _build
    if rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    kvq.load_library()
    spec = CycleSpec()
    dev = torch.device("cuda", torch.cuda.current_device())
    caches, wss = [], []
    for L in range(spec.layers):
        K, V = ki.kv_stream_torch(1000 + L, spec.B, spec.H, spec.Lq + spec.r0, spec.D)
        c = kvq.QuantizedKVCache(spec.B, spec.H, spec.D, spec.G, "hier8", spec.capacity())
        kvq.kvq_quantize_append(c, K, V)                      # bulk cache build (prefill)
        del K, V
        caches.append(c)
        wss.append(kvq.make_workspace(c, spec.H, spec.gamma, 0))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    assert caches[0].state() == (spec.Lq, spec.r0, 0), caches[0].state()
    h_in = _cycle_host_inputs(spec)
    d_in = torch.empty_like(h_in, device=dev)
    d_in.copy_(h_in)
    d_out = torch.empty(spec.layers * spec.layer_output_elems(), dtype=torch.bfloat16, device=dev)
    h_out = torch.empty(d_out.shape, dtype=d_out.dtype).pin_memory()
    views = _cycle_views(spec, d_in, d_out)
    lse_d = torch.empty((spec.B, 1, spec.H), dtype=torch.float32, device=dev)
    lse_v = torch.empty((spec.B, spec.gamma, spec.H), dtype=torch.float32, device=dev)

    def drafts(st):
        for j in range(spec.drafts):
            for L in range(spec.layers):
                v = views[L]
                kvq.kvq_attend(caches[L], "int4", v["qd"][j], v["pend"][j][0], v["pend"][j][1], out=v["od"][j],
                               lse=lse_d, workspace=wss[L], stream=st)

    def verify(st):
        for L in range(spec.layers):
            v = views[L]
            kvq.kvq_attend(caches[L], "int8", v["qv"], v["pend"][-1][0], v["pend"][-1][1], out=v["ov"],
                           lse=lse_v, workspace=wss[L], stream=st)

    def commit(st):
        for L in range(spec.layers):
            c = caches[L]
            saved = c.state()
            kvq.kvq_quantize_append(c, views[L]["kn"], views[L]["vn"], stream=st)
            c.set_state(saved)

    phases = (drafts, verify, commit)
    # warm-up eagerly (sets kernel attributes outside any capture)
    for _ in range(2):
        for ph in phases:
            ph(None)
    torch.cuda.synchronize()
    for ws in wss:
        assert kvq.kvq_workspace_status(ws) == 0
    cap = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(cap):
        for ph in phases:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                ph(cap)
            graphs.append(g)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()

    # ---- timed region: K steps, events between the phases on the launching stream ----
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    marks = [[mk() for _ in range(4)] for _ in range(args.steps)]
    e0, e1 = mk(), mk()
    t0 = time.perf_counter()
    e0.record()
    for i in range(args.steps):
        m = marks[i]
        m[0].record()
        for k, g in enumerate(graphs):
            g.replay()
            m[k + 1].record()
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    value = whole_job_rate(spec.kv_tokens_per_step(), world, ms_step * 1e-3)
    phase_ms = [sum(m[k].elapsed_time(m[k + 1]) for m in marks) / args.steps for k in range(3)]
    draft_launch_ms = phase_ms[0] / (spec.drafts * spec.layers)
    verify_launch_ms = phase_ms[1] / spec.layers
    peak, peak_src = _peak()
    draft_gbs = spec.draft_bytes_per_launch() / (draft_launch_ms * 1e-3) / 1e9
    verify_gbs = spec.verify_bytes_per_launch() / (verify_launch_ms * 1e-3) / 1e9
    for ws in wss:
        assert kvq.kvq_workspace_status(ws) == 0, "device status word set"

    # ---- e2e: the public API, eager, with the step's inputs uploaded from pinned
    # host memory and the step's attention outputs read back every step ----
    def e2e_step():
        s0 = torch.cuda.current_stream()
        d_in.copy_(h_in, non_blocking=True)
        for ph in phases:
            ph(s0)
        h_out.copy_(d_out, non_blocking=True)
        s0.synchronize()

    n_e2e = max(3, min(args.steps, 10))
    e2e_step()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t1) / n_e2e, world, dev)
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    for ws in wss:
        assert kvq.kvq_workspace_status(ws) == 0, "device status word set"
    del caches, wss, graphs
    torch.cuda.empty_cache()

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8/int4 codes, f16 mma / fp32 accumulate, bf16 io",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q, 4 of 128 key channels x8 per head)",
        "config": {"workload": WORKLOAD, "layers": spec.layers, "batch": spec.B, "q_heads": spec.H,
                   "kv_heads": spec.H, "head_dim": spec.D, "group": spec.G, "quantized_tokens": spec.Lq,
                   "residual_tokens": spec.r0, "draft_steps": spec.drafts, "verify_gamma": spec.gamma,
                   "append_per_step": spec.n_accept,
                   "step": "per layer: 6 INT4 draft attentions (gamma 1, 1..6 pending), INT8 verify (gamma 6, "
                           "6 pending, causal), quantize-append of 6 tokens with one group flush",
                   "timing": "3 CUDA graphs per step (drafts, verify, append), CUDA events over the K steps "
                             "and between the phases",
                   "l2": "no flush: 36.5 GB of quantized cache per step (> L2)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "calls": {"draft_int4_launch_ms": draft_launch_ms, "draft_int4_gbs": draft_gbs,
                  "draft_int4_frac": draft_gbs / peak,
                  "verify_int8_launch_ms": verify_launch_ms, "verify_int8_gbs": verify_gbs,
                  "verify_int8_frac": verify_gbs / peak,
                  "append_6_with_flush_ms_per_layer": phase_ms[2] / spec.layers,
                  "phase_ms": {"drafts": phase_ms[0], "verify": phase_ms[1], "append": phase_ms[2]}},
        "roofline": {"kernel": "attend_kernel<INT4,128,1,1> (draft, gamma=1, 128K)", "bound": "hbm",
                     "achieved": draft_gbs, "peak": peak, "peak_source": f"{peak_src} hbm_gbs (of {peak_src})",
                     "unit": "GB/s", "frac": draft_gbs / peak,
                     "traffic": measured_traffic("attend_int4_draft_128k"),
                     "algorithmic_bytes_per_launch": spec.draft_bytes_per_launch(),
                     "timing": "draft phase of every timed step (192 launches), CUDA events on the graph stream"},
        "e2e": {"value": whole_job_rate(spec.kv_tokens_per_step(), world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "steps": n_e2e, "how": "eager C-ABI calls through the Python binding; step inputs uploaded "
                                      "from pinned host memory, attention outputs read back, every step"},
        "gpu_launches": spec.launches_per_step() * args.steps,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    return result


# --------------------------------------------------------------------------------------
# extra figure: the single-layer 8K verify step
# --------------------------------------------------------------------------------------

class LayerSpec:
    B, Hq, Hkv, D, G = 1, 32, 32, 128, 128
    Lq = 8192
    r0 = 2 * 128 - 4            # residual fill before the step: the append flushes a group
    gamma = 8
    P = 8
    top_k = 64
    n_accept = 8
    copies = 4

    @property
    def kv_tokens_per_step(self):
        return self.B * (self.Lq + self.r0 + self.P)

    def attend_bytes(self):
        per_tok = _bytes_per_token("int8", self.D, self.G)
        return self.B * self.Hkv * (self.Lq * per_tok + self.r0 * 2 * self.D * 2)

    def topk_bytes(self):
        per_tok = self.D // 2 + 2 * self.D * 4 // self.G
        return self.B * self.Hkv * self.Lq * per_tok


def run_layer_verify_8k(steps=2000, warmup=20):
    """One Llama-2-7B-shaped layer at 8K: INT8 verify (gamma 8) and INT4 top-64
    on two streams, then the 8-token append with a flush; one CUDA graph per
    step, rotating over 4 cache copies (4 x 76 MB > L2)."""
    import quantized_kv_speculative_gb300 as kvq
    spec = LayerSpec()
    dev = torch.device("cuda", torch.cuda.current_device())
    K, V = ki.kv_stream_torch(0, spec.B, spec.Hkv, spec.Lq + spec.r0 + spec.n_accept, spec.D)
    n = spec.Lq + spec.r0
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    q = torch.randn((spec.B, spec.gamma, spec.Hq, spec.D), generator=gen, device=dev).to(torch.bfloat16)
    pk = torch.randn((spec.B, spec.Hkv, spec.P, spec.D), generator=gen, device=dev).to(torch.bfloat16)
    pv = torch.randn((spec.B, spec.Hkv, spec.P, spec.D), generator=gen, device=dev).to(torch.bfloat16)
    kn, vn = K[:, :, n:].contiguous(), V[:, :, n:].contiguous()
    q_spec = q[:, -1].contiguous()
    caches, wss = [], []
    for _ in range(spec.copies):
        c = kvq.QuantizedKVCache(spec.B, spec.Hkv, spec.D, spec.G, "hier8", spec.Lq + 2 * spec.G)
        kvq.kvq_quantize_append(c, K[:, :, :n].contiguous(), V[:, :, :n].contiguous())
        caches.append(c)
        wss.append(kvq.make_workspace(c, spec.Hq, spec.gamma, spec.top_k))
    del K, V
    out = torch.empty_like(q)
    lse = torch.empty((spec.B, spec.gamma, spec.Hq), dtype=torch.float32, device=dev)
    idx = torch.empty((spec.B, spec.Hkv, spec.top_k), dtype=torch.int32, device=dev)
    sc = torch.empty((spec.B, spec.Hkv, spec.top_k), dtype=torch.float32, device=dev)
    side = torch.cuda.Stream()

    def step(i, s0):
        c, ws = caches[i % spec.copies], wss[i % spec.copies]
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

    for i in range(spec.copies):
        step(i, torch.cuda.current_stream())
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(cap):
        for j in range(spec.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                step(j, cap)
            graphs.append(g)
    torch.cuda.synchronize()
    for i in range(warmup):
        graphs[i % spec.copies].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        graphs[i % spec.copies].replay()
    e1.record()
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / steps

    def per_call_ms(fn, reps=64, rounds=8):
        gk = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(gk, stream=cap):
                for i in range(reps):
                    fn(i, cap)
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

    att_ms = per_call_ms(lambda i, s: kvq.kvq_attend(caches[i % spec.copies], "int8", q, pk, pv, out=out, lse=lse,
                                                     workspace=wss[i % spec.copies], stream=s))
    topk_ms = per_call_ms(lambda i, s: kvq.kvq_topk(caches[i % spec.copies], "int4", q_spec, spec.top_k,
                                                    idx_out=idx, score_out=sc, workspace=wss[i % spec.copies],
                                                    stream=s))
    for ws in wss:
        assert kvq.kvq_workspace_status(ws) == 0
    peak, src = _peak()
    att_gbs = spec.attend_bytes() / (att_ms * 1e-3) / 1e9
    topk_gbs = spec.topk_bytes() / (topk_ms * 1e-3) / 1e9
    del caches, wss, graphs
    torch.cuda.empty_cache()
    return {"workload": "llama7b-layer-verify-8k", "value": spec.kv_tokens_per_step / (ms_step * 1e-3),
            "unit": UNIT, "ms_per_step": ms_step, "steps": steps,
            "step": "INT8 verify (gamma 8) and INT4 top-64 on two streams, then an 8-token append with a flush; "
                    "one CUDA graph per step over 4 rotating cache copies",
            "attend_int8_verify_ms": att_ms, "attend_gbs": att_gbs, "attend_frac": att_gbs / peak,
            "topk_int4_ms": topk_ms, "topk_gbs": topk_gbs, "topk_frac": topk_gbs / peak,
            "attend_traffic": measured_traffic("attend_int8_verify_8k"), "peak_gbs": peak, "peak_source": src}


# --------------------------------------------------------------------------------------
# oracle (CPU) arm: the same cycle on sampled (layer, head) units
# --------------------------------------------------------------------------------------
# Worker processes are forked before the first CUDA call (a process forked after
# CUDA is initialised can hang), each builds one (layer, head) unit of the 128K
# cache with the oracle, then all run their cycle at once behind a barrier.

_POOL_BARRIER = None
_UNIT = None


def _oracle_unit(unit_id):
    """The oracle's cache of one (layer, head) unit of the cycle, plus its step
    inputs (same distributions as the device run)."""
    import oracle
    spec = CycleSpec()
    K, V = ki.kv_stream(unit_id, 1, 1, spec.Lq + spec.r0 + spec.n_accept, spec.D)
    n = spec.Lq + spec.r0
    c = oracle.OracleCache(1, 1, spec.D, spec.G, "hier8", spec.capacity())
    c.append(K[:, :, :n], V[:, :, :n])
    q = ki.queries(unit_id, 1, spec.gamma, 1, spec.D)
    pk, pv = ki.pending(unit_id, 1, 1, spec.gamma, spec.D)
    return dict(c=c, q=q, pk=pk, pv=pv, kn=K[:, :, n:], vn=V[:, :, n:])


def _oracle_cycle(u):
    """One cycle of one unit: 6 INT4 drafts, the INT8 verify, the 6-token append
    (the cache state is restored afterwards, as on the device)."""
    import oracle
    spec = CycleSpec()
    c = u["c"]
    for j in range(1, spec.drafts + 1):
        oracle.attend(c, "int4", u["q"][:, j - 1:j], u["pk"][:, :, :j], u["pv"][:, :, :j])
    oracle.attend(c, "int8", u["q"], u["pk"], u["pv"])
    saved = (c.Lq, c.r, c.res_k.copy(), c.res_v.copy())
    c.append(u["kn"], u["vn"])
    c.Lq, c.r, c.res_k, c.res_v = saved


def _pool_init(barrier):
    global _POOL_BARRIER
    _POOL_BARRIER = barrier


def _pool_build_and_run(unit_id):
    """Build the unit (untimed), wait for every worker, run one cycle (timed)."""
    global _UNIT
    _UNIT = _oracle_unit(unit_id)
    _POOL_BARRIER.wait(timeout=900)
    t0 = time.perf_counter()
    _oracle_cycle(_UNIT)
    return t0, time.perf_counter()


def _pool_run(_):
    """One more cycle of this worker's unit, started with the other workers'."""
    _POOL_BARRIER.wait(timeout=900)
    t0 = time.perf_counter()
    _oracle_cycle(_UNIT)
    return t0, time.perf_counter()


class OraclePool:
    """``n`` forked worker processes, one (layer, head) unit each.  Create it
    before any CUDA call."""

    def __init__(self, n):
        ctx = multiprocessing.get_context("fork")
        self.n = n
        self.barrier = ctx.Barrier(n)
        self.pool = ctx.Pool(n, initializer=_pool_init, initargs=(self.barrier,))

    def first(self):
        """Every worker builds its unit, then all run one cycle together."""
        return self.pool.map(_pool_build_and_run, range(self.n), chunksize=1)

    def again(self):
        return self.pool.map(_pool_run, range(self.n), chunksize=1)

    def close(self):
        self.pool.terminate()
        self.pool.join()


def _unit_kv_tokens(spec: CycleSpec, units):
    """KV tokens (all heads of a layer = one) that `units` (layer, head) units of
    one cycle amount to."""
    return spec.kv_tokens_per_step() / (spec.layers * spec.H) * units


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def pool_size():
    return max(1, min(host_cores(), 32))


def cpu_baseline(pool: "OraclePool"):
    """The oracle on the host: one (layer, head) unit on one core, then one unit
    per core at once.  Throughput is scaled to the workload's KV-token unit."""
    spec = CycleSpec()
    u = _oracle_unit(0)
    t0 = time.perf_counter()
    _oracle_cycle(u)
    single_s = time.perf_counter() - t0
    del u
    spans = pool.first()
    wall = max(b for a, b in spans) - min(a for a, b in spans)
    v_all = _unit_kv_tokens(spec, pool.n) / wall
    v_one = _unit_kv_tokens(spec, 1) / single_s
    cpu = ""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                cpu = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"value": v_all, "unit": UNIT, "cores": pool.n, "kind": "oracle",
            "sample": f"one 128K cycle (6 INT4 drafts, INT8 verify, 6-token append) of {pool.n} (layer, head) "
                      f"units, one per worker process, run at once ({wall:.2f} s wall); KV tokens scaled from "
                      f"units to whole layers (1 of {spec.layers * spec.H} units = 1/{spec.layers * spec.H} of a "
                      f"step); numpy, one BLAS thread per process",
            "single_core": {"value": v_one, "cores": 1, "seconds_per_unit_cycle": single_s},
            "nproc": host_cores(), "cpu": cpu}


def run_reference(args, rank, world, pool):
    """The oracle on all host cores: each step is one cycle of one (layer, head)
    unit per worker, run at once.  Steps stop early once about 150 s are spent,
    and the line reports the steps actually timed."""
    if rank != 0:
        return None
    spec = CycleSpec()
    spans = pool.first()                       # builds the units; counts as the first warm-up step
    for _ in range(max(0, args.warmup - 1)):
        pool.again()
    times, t_start = [], time.perf_counter()
    for _ in range(args.steps):
        sp = pool.again()
        times.append(max(b for a, b in sp) - min(a for a, b in sp))
        if time.perf_counter() - t_start > 150.0:
            break
    dt = sum(times) / len(times)
    v = _unit_kv_tokens(spec, pool.n) / dt
    sample = (f"per step: one 128K cycle (6 INT4 drafts, INT8 verify, 6-token append) of {pool.n} (layer, head) "
              f"units of the {spec.layers}-layer x {spec.H}-head cache, one per worker process, at once; "
              f"value = those units' KV tokens (1/{spec.layers * spec.H} of a step's each) per second")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 0,
            "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "ms_per_step_is": "measured wall time of one sampled step",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 quantizer, f64 attention", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample, "first_cycle_s":
                       max(b for a, b in spans) - min(a for a, b in spans)},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": pool.n, "kind": "oracle", "sample": sample},
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
    memory, then attention (gamma = 2) with them at 16 bits.  Each call is
    timed on its own; the step time is their sum."""
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
    # attention fused with the next step's top-k (one read of the low-bit keys),
    # scored by the speculative token (row 1) and by the output token (row 0)
    idx_f, sc_f = torch.empty_like(idx), torch.empty_like(sc)
    fused = {}
    for row in (1, 0):
        gf = _graph(lambda st: kvq.kvq_attend_topk(c, fmt, q, k, row, pk, pv, idx, sk, sv, out=out, lse=lse,
                                                   next_idx=idx_f, next_score=sc_f, workspace=ws, stream=st), s)
        fused[row] = _time_graph(gf, reps)
    kvq.kvq_topk(c, fmt, qs, k, idx_out=idx, score_out=sc, workspace=ws)
    torch.cuda.synchronize()
    fused_same = bool(torch.equal(idx_f, kvq.kvq_topk(c, fmt, q[:, 0].contiguous(), k, workspace=ws)[0]))
    try:
        gg = _graph(lambda st: [kvq.kvq_gather_selected(hk, hv, ix, sel_k=sk2, sel_v=sv2, stream=st) for ix in sets], s)
        tg, fetch_err = _time_graph(gg, reps) / nset, None
    except Exception as ex:   # reported in the line instead of ending the run
        torch.cuda.synchronize()
        tg, fetch_err = float("nan"), f"{type(ex).__name__}: {ex}"[:200]
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
            "fused_attend_topk_ms": fused[1], "fused_attend_topk_row0_ms": fused[0],
            "fused_matches_separate_topk": fused_same,
            "step_ms": fused[1] + tg, "step": "fused attention + top-k, then the fetch, each timed on its own",
            "step_separate_ms": ta + tt + tg,
            "kv_tok_per_s": B * (lq + r0 + 2) / ((fused[1] + tg) * 1e-3),
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
    elif name in ("attend-int4-draft-128k", "attend-int8-verify-128k"):
        # one layer of the 128K cycle (1.14 GB of cache; the launch is the same
        # as each layer's in the 32-layer step)
        spec = CycleSpec()
        K, V = ki.kv_stream_torch(1000, spec.B, spec.H, spec.Lq + spec.r0, spec.D)
        c = kvq.QuantizedKVCache(spec.B, spec.H, spec.D, spec.G, "hier8", spec.capacity())
        kvq.kvq_quantize_append(c, K, V)
        del K, V
        torch.cuda.empty_cache()
        gamma = 1 if "draft" in name else spec.gamma
        ws = kvq.make_workspace(c, spec.H, spec.gamma, 0)
        q = rnd(spec.B, gamma, spec.H, spec.D)
        pk, pv = rnd(spec.B, spec.H, spec.gamma, spec.D), rnd(spec.B, spec.H, spec.gamma, spec.D)
        out = torch.empty_like(q)
        for _ in range(launches):
            kvq.kvq_attend(c, "int4" if gamma == 1 else "int8", q, pk, pv, out=out, workspace=ws)
    elif name in ("attend-int2-specache-32k", "topk-int2-specache-32k", "attend-topk-int2-specache-32k"):
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
        del K, V, gi
        torch.cuda.empty_cache()
        nidx = torch.empty_like(idx)
        for i in range(launches):
            if name.startswith("topk"):
                kvq.kvq_topk(c, "int2", q[:, 1].contiguous(), k, idx_out=idx, workspace=ws)
            elif name.startswith("attend-topk"):
                kvq.kvq_attend_topk(c, "int2", q, k, 1, pk, pv, idx, sk, sv, next_idx=nidx, workspace=ws)
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
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the single-layer 8K figure")
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
        if rank == 0:
            pool = OraclePool(pool_size())
            try:
                res = run_reference(args, rank, world, pool)
            finally:
                pool.close()
            print(json.dumps(res), flush=True)
        return
    # the oracle's worker processes are forked before the first CUDA call
    pool = None
    if rank == 0 and not (args.no_cpu_baseline or args.profile_case or args.workload):
        pool = OraclePool(pool_size())
    try:
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
        res = run_device(args, rank, world)
        if rank == 0:
            if not args.no_extra:
                res["extra"] = {"llama7b-layer-verify-8k": run_layer_verify_8k()}
            if pool is not None:
                res["cpu_baseline"] = cpu_baseline(pool)
            print(json.dumps(res), flush=True)
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
    finally:
        if pool is not None:
            pool.close()


if __name__ == "__main__":
    main()
