"""Seeded synthetic inputs shared by the oracle-side tests and the device-side runs.

This module only *draws* inputs.  It holds none of the method's arithmetic: no
quantizer, no dequantizer, no attention, no scoring.  Both the CPU oracle and the
CUDA library receive the arrays it returns.

Every tensor the method consumes is bf16.  Values are drawn in fp32 from a seeded
PCG64 stream, then rounded to bf16 with round-to-nearest-even.  They are returned
as float32 arrays that hold exactly those bf16 values (``to_bf16_bits`` gives the
raw 16-bit patterns for upload).

The workload shapes follow the pages' own workloads: 7B-class attention layers
(32 heads x head_dim 128), contexts of 8K to 256K tokens, speculation lengths up to
8, and SpeCache's batch of 36 with 4:1 grouped-query attention.  The pages'
datasets are not available here.  These seeded normal tensors stand in for them,
with the same shapes and a few outlier key channels.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# --------------------------------------------------------------------------------
# bf16 helpers (input preparation only)
# --------------------------------------------------------------------------------


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even) and return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    out = ((u + rounding) >> np.uint64(16)).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 array holding the bf16-rounded values of ``x``."""
    return bf16_bits_to_f32(to_bf16_bits(x))


# --------------------------------------------------------------------------------
# Draws
# --------------------------------------------------------------------------------


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def normal_bf16(g: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    return round_bf16(g.standard_normal(shape, dtype=np.float32) * np.float32(scale))


def kv_stream(
    seed: int,
    batch: int,
    num_kv_heads: int,
    n_tokens: int,
    head_dim: int,
    outlier_channels: int = 4,
    outlier_gain: float = 8.0,
    stream: int = 0,
):
    """Keys and values ``[B, Hkv, N, D]`` ~ N(0,1) in bf16.

    A fixed, seeded set of ``outlier_channels`` key channels per (b, kv head) is
    multiplied by ``outlier_gain`` (KIVI-style per-channel key outliers).
    """
    g = rng(seed, 1000 + stream)
    k = g.standard_normal((batch, num_kv_heads, n_tokens, head_dim), dtype=np.float32)
    v = g.standard_normal((batch, num_kv_heads, n_tokens, head_dim), dtype=np.float32)
    if outlier_channels > 0:
        for b in range(batch):
            for h in range(num_kv_heads):
                ch = g.choice(head_dim, size=outlier_channels, replace=False)
                k[b, h, :, ch] *= np.float32(outlier_gain)
    return round_bf16(k), round_bf16(v)


def queries(seed: int, batch: int, gamma: int, num_q_heads: int, head_dim: int, stream: int = 0):
    """Query tokens ``[B, gamma, Hq, D]`` ~ N(0,1) in bf16."""
    g = rng(seed, 2000 + stream)
    return normal_bf16(g, (batch, gamma, num_q_heads, head_dim))


def pending(seed: int, batch: int, num_kv_heads: int, n_pend: int, head_dim: int, stream: int = 0):
    """Speculative (not yet committed) keys/values ``[B, Hkv, P, D]``."""
    g = rng(seed, 3000 + stream)
    return (normal_bf16(g, (batch, num_kv_heads, n_pend, head_dim)),
            normal_bf16(g, (batch, num_kv_heads, n_pend, head_dim)))


def plant_needles(
    k: np.ndarray,
    q: np.ndarray,
    seed: int,
    n_needles: int = 8,
    gain: float = 3.0,
    limit: Optional[int] = None,
):
    """Make attention peaked: overwrite ``n_needles`` keys per (b, kv head) with a
    scaled copy of the group's first query head direction, so those tokens' logits
    sit several units above the rest.  ``k`` is ``[B, Hkv, N, D]``, ``q`` is
    ``[B, gamma, Hq, D]``.  Returns a new key array and the needle positions."""
    B, Hkv, N, D = k.shape
    Hq = q.shape[2]
    hg = Hq // Hkv
    g = rng(seed, 4000)
    k = k.copy()
    lim = N if limit is None else min(limit, N)
    pos = np.zeros((B, Hkv, n_needles), dtype=np.int64)
    for b in range(B):
        for h in range(Hkv):
            p = g.choice(lim, size=n_needles, replace=False)
            pos[b, h] = np.sort(p)
            qdir = q[b, -1, h * hg].astype(np.float32)
            qdir = qdir / np.float32(np.linalg.norm(qdir) + 1e-6)
            for t in p:
                k[b, h, t] = qdir * np.float32(gain * np.sqrt(D)) + g.standard_normal(D).astype(np.float32) * np.float32(0.1)
    return round_bf16(k), pos


# --------------------------------------------------------------------------------
# Workload shapes (the pages' workloads, restated as named shapes)
# --------------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    group_size: int
    fmt: str                 # "hier8", "int2", "int1"
    n_tokens: int            # tokens committed to the cache (quantized + residual)
    gamma: int               # query tokens per call
    n_pend: int              # speculative tokens passed alongside the cache
    layers: int = 1
    top_k: int = 0
    outlier_channels: int = 4
    outlier_gain: float = 8.0

    @property
    def quantized_len(self) -> int:
        G = self.group_size
        return 0 if self.n_tokens < 2 * G else G * (self.n_tokens // G - 1)

    @property
    def residual_len(self) -> int:
        return self.n_tokens - self.quantized_len


def _n_for(lq: int, r: int) -> int:
    return lq + r


WORKLOADS = {
    # Tiny correctness case: 4 heads, head_dim 64, 512 quantized + 32 residual tokens.
    "tiny-d64-g32": Workload("tiny-d64-g32", 1, 4, 4, 64, 32, "hier8", _n_for(512, 32), 1, 1,
                             outlier_channels=4, outlier_gain=10.0),
    # One Llama-2-7B-shaped layer, verify step: 8K quantized context, gamma = 8 causal queries.
    "llama7b-layer-verify-8k": Workload("llama7b-layer-verify-8k", 1, 32, 32, 128, 128, "hier8",
                                        _n_for(8192, 128), 8, 8),
    # 7B-shaped 32-layer draft/verify cycle at 32K.
    "llama7b-32l-spec-32k": Workload("llama7b-32l-spec-32k", 1, 32, 32, 128, 128, "hier8",
                                     _n_for(32768, 128), 8, 8, layers=32),
    # SpeCache-style batched low-bit decode: batch 36, GQA 4:1, 2 query tokens, top-64.
    "specache-b36-32k-int2": Workload("specache-b36-32k-int2", 36, 32, 8, 128, 32, "int2",
                                      _n_for(32768, 32), 2, 2, top_k=64),
    "specache-b36-32k-int1": Workload("specache-b36-32k-int1", 36, 32, 8, 128, 32, "int1",
                                      _n_for(32768, 32), 2, 2, top_k=64),
    # Long-context stress case: 32 layers at 128K, gamma = 6.
    "llama7b-32l-spec-128k": Workload("llama7b-32l-spec-128k", 1, 32, 32, 128, 128, "hier8",
                                      _n_for(131072, 253), 6, 6, layers=32),
}

# Single-layer INT4 draft-attention sweep over context lengths (gamma = 1).
SWEEP_CONTEXTS = (8192, 16384, 32768, 65536, 131072, 262144)


# --------------------------------------------------------------------------------
# Device-side draws for the large workloads (seeded torch generator on the GPU).
# The oracle side downloads the slices it needs; those are inputs, not results.
# --------------------------------------------------------------------------------


def kv_stream_torch(seed: int, batch: int, num_kv_heads: int, n_tokens: int, head_dim: int,
                    outlier_channels: int = 4, outlier_gain: float = 8.0, device="cuda"):
    """bf16 ``[B, Hkv, N, D]`` keys and values ~ N(0,1) drawn on ``device``.  A
    seeded set of ``outlier_channels`` key channels per (b, kv head) is scaled by
    ``outlier_gain``."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    shape = (batch, num_kv_heads, n_tokens, head_dim)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outlier_channels > 0:
        cpu = np.random.Generator(np.random.PCG64([seed, 77]))
        gain = torch.ones((batch, num_kv_heads, 1, head_dim), device=device)
        for b in range(batch):
            for h in range(num_kv_heads):
                ch = cpu.choice(head_dim, size=outlier_channels, replace=False)
                gain[b, h, 0, torch.as_tensor(ch, device=device)] = outlier_gain
        k.mul_(gain)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def bf16_tensor_to_f32(t) -> np.ndarray:
    """Download a bf16 torch tensor as float32 numpy (exact widening)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32)


def f32_to_bf16_tensor(x: np.ndarray, device="cuda"):
    """Upload bf16-valued float32 numpy data as a bf16 torch tensor."""
    import torch
    bits = to_bf16_bits(x)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(device)
