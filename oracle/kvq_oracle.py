"""Plain, slow CPU oracle for quantized-KV speculative decode attention.

TEST INFRASTRUCTURE ONLY.  The library's product path never imports, calls or
links anything in this package.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg do.  This package shares no code with the CUDA
library: no kernels, headers, helpers or tables.  It computes the method the way
the pages state it, step by step:

* Quantizer.  KIVI-style asymmetric min/max quantization.  Keys are grouped per
  channel over G tokens; values per token over G channels.  The code is
  round-half-even((x - min) * (1/scale)), computed in fp32 and clamped.
  (SpeCache page, Approach / Measured effects: "2-bit KIVI (g=32)", "1-bit
  KIVI"; QuantSpec page, Experimental setup: builds on KIVI.)
* Hierarchical INT8 code.  The upper nibble is the INT4 draft code; upper plus
  lower nibble rebuild the INT8 target code.  No separate draft copy is stored.
  (QuantSpec page, Approach.)  A second INT4 reading puts the draft code at the
  middle of the 8-bit codes it stands for (lower nibble read as 8).
* Centred 1-bit reading.  The 1-bit KIVI codes read with the two levels at the
  centres of the two halves of each group's range.  SpeCache (Approach) gives
  1-bit KIVI a new zero point and scale without a formula; this reading is the
  library's, pinned against its own closed form, so its agreement with the
  pages' variant is unknown.
* Double full-precision buffer of 2G tokens.  It keeps recent tokens in bf16.
  When full, the oldest G tokens are quantized.  (QuantSpec page, Approach.)
* Attention.  Softmax attention, in fp64, over the dequantized cache plus the
  bf16 residual tokens plus gamma causal speculative tokens.  Selected tokens
  use their 16-bit K/V in place of the low-bit copy.  (SpeCache page,
  Approach; QuantSpec page, Approach.)
* Top-k.  Per KV head, the k tokens that score highest under the low-bit keys,
  scored with the speculative token's query.  (SpeCache page, Approach.)

Where the pages are silent, the reading taken is stated at the function.  Those
readings are also listed in the repository's design notes.  The "parity
unpinned" functions are named in the module docstring of ``tests/test_oracle_pins.py``
(none at present).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np

F32 = np.float32

FORMAT_BITS = {"hier8": 8, "int2": 2, "int1": 1}
# mode -> (storage format it reads, code bits seen by the mode, scale multiplier)
MODES = {
    "int8": ("hier8", 8, 1),
    "int4": ("hier8", 4, 16),
    "int4mid": ("hier8", 4, 16),
    "int2": ("int2", 2, 1),
    "int1": ("int1", 1, 1),
    "int1c": ("int1", 1, 0.5),
}
# The midpoint reading of the INT4 draft code: the upper nibble hi stands for
# the 8-bit codes 16 hi .. 16 hi + 15, and "int4mid" reconstructs it at the
# middle of that range, 16 hi + MID_NIBBLE, instead of at its bottom.
MID_NIBBLE = 8
# The centred reading of the 1-bit KIVI code (SpeCache page, Approach: 1-bit
# KIVI gets a new zero point and scale; the pages give no formula).  Plain
# 1-bit min/max puts the two levels at the group's min and max.  "int1c"
# reads the same codes (1 above the midpoint of [min, max]) with the levels at
# the centres of the two halves, min + r/4 and min + 3r/4 (r = max - min, the
# stored scale): zero point z + CENTER_SHIFT s and scale s/2.  For values
# spread evenly over [min, max] that cuts the mean squared error by four.
CENTER_SHIFT = 0.25
SLAB = 32  # tokens per value-plane slab (storage layout, see pack_v_plane)


# ================================================================================
# Quantizer
# ================================================================================


def quantize_minmax(x: np.ndarray, bits: int, axis: int):
    """Asymmetric min/max quantization of ``x`` along ``axis``.

    Follows the KIVI-style quantizer the pages build on (SpeCache page, Approach
    and Measured effects table; QuantSpec page, Experimental setup).  Every step
    is an fp32 operation rounded to nearest even.  No step is fused.

      1. mn = min(x) + 0, mx = max(x) + 0      (the + 0 turns -0 into +0)
      2. scale = (mx - mn) / (2^bits - 1)
      3. inv = 0 if scale == 0 else 1 / scale  (a constant group gets codes 0)
      4. code = clamp(rint((x - mn) * inv), 0, 2^bits - 1), with half-even rint
      5. zero point = mn

    Returns (codes uint8, scale f32, zero f32); the reduced axis is dropped from
    scale and zero.  Non-finite inputs are rejected.
    """
    x = np.asarray(x, dtype=F32)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite input to the quantizer")
    levels = F32(2 ** bits - 1)
    mn = (x.min(axis=axis, keepdims=True) + F32(0)).astype(F32)
    mx = (x.max(axis=axis, keepdims=True) + F32(0)).astype(F32)
    scale = ((mx - mn) / levels).astype(F32)
    with np.errstate(divide="ignore"):
        inv = np.where(scale == F32(0), F32(0), (F32(1) / scale)).astype(F32)
    t = ((x - mn).astype(F32) * inv).astype(F32)
    codes = np.clip(np.rint(t), F32(0), levels).astype(np.uint8)
    return codes, np.squeeze(scale, axis=axis), np.squeeze(mn, axis=axis)


def quantize_key_group(kg: np.ndarray, bits: int):
    """Keys of one token group ``[..., G, D]``: one (scale, zero) per channel over
    the G tokens.  Returns codes ``[..., G, D]``, scale/zero ``[..., D]``."""
    return quantize_minmax(kg, bits, axis=-2)


def quantize_value_group(vg: np.ndarray, bits: int, G: int):
    """Values ``[..., T, D]``: one (scale, zero) per token per block of G channels.
    Returns codes ``[..., T, D]``, scale/zero ``[..., T, D/G]``."""
    shp = vg.shape
    D = shp[-1]
    x = vg.reshape(shp[:-1] + (D // G, G))
    c, s, z = quantize_minmax(x, bits, axis=-1)
    return c.reshape(shp), s, z


def split_hierarchical(codes8: np.ndarray):
    """Hierarchical INT8 code -> (upper nibble, lower nibble).  The upper nibble
    is the INT4 draft code (QuantSpec page, Approach)."""
    c = codes8.astype(np.uint8)
    return (c >> 4).astype(np.uint8), (c & 15).astype(np.uint8)


def mode_codes_scale(mode: str, codes: np.ndarray, scale: np.ndarray):
    """The (code, scale) pair a read mode sees.

    INT8 reads the full hierarchical code with its scale.  INT4 reads only the
    upper nibble, with 16 x scale.  So INT4 dequant equals INT8 dequant with the
    lower nibble zeroed (QuantSpec page, Approach).  INT4-mid reads the same
    nibble and scale (its zero point moves, see mode_zero).  INT2/INT1 read
    their own codes and scale; INT1-centred reads the 1-bit codes with half
    the scale.
    """
    _, _, mult = MODES[mode]
    if mode in ("int4", "int4mid"):
        return (codes >> 4).astype(np.uint8), scale.astype(np.float64) * 16.0
    return codes, scale.astype(np.float64) * mult


def mode_zero(mode: str, zero: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """The zero point a read mode sees, in fp64.  INT4-mid adds MID_NIBBLE
    steps of the 8-bit scale, so that its dequant equals INT8 dequant with the
    lower nibble set to MID_NIBBLE: (16 hi + 8) s + z = hi (16 s) + (z + 8 s).
    INT1-centred adds a quarter of the 1-bit scale (the range).  Every other
    mode reads the stored zero point."""
    z = zero.astype(np.float64)
    if mode == "int4mid":
        return z + MID_NIBBLE * scale.astype(np.float64)
    if mode == "int1c":
        return z + CENTER_SHIFT * scale.astype(np.float64)
    return z


# ================================================================================
# Packed storage layout (the bytes the device library stores)
# ================================================================================


def pack_k_plane(codes: np.ndarray, pb: int) -> np.ndarray:
    """Key plane, token-major: row t holds the D channel codes of token t.  Each
    byte j packs channels (8/pb)*j + e at bits [pb*e, pb*e + pb).
    ``codes [..., T, D]`` (values < 2^pb) -> ``[..., T, D*pb/8]`` uint8."""
    per = 8 // pb
    c = codes.astype(np.uint8)
    shp = c.shape
    c = c.reshape(shp[:-1] + (shp[-1] // per, per))
    out = np.zeros(c.shape[:-1], dtype=np.uint8)
    for e in range(per):
        out |= (c[..., e] << (pb * e)).astype(np.uint8)
    return out


def pack_v_plane(codes: np.ndarray, pb: int) -> np.ndarray:
    """Value plane, in 32-token slabs: slab s, row d holds the codes of channel d
    for tokens 32s..32s+31.  Each byte j packs tokens 32s + (8/pb)*j + e at bits
    [pb*e, pb*e + pb).  ``codes [..., T, D]`` (T a multiple of 32) ->
    ``[..., T/32, D, 32*pb/8]`` uint8."""
    per = 8 // pb
    c = codes.astype(np.uint8)
    *lead, T, D = c.shape
    c = c.reshape(tuple(lead) + (T // SLAB, SLAB, D))
    c = np.swapaxes(c, -1, -2)                         # [..., T/32, D, 32]
    c = c.reshape(c.shape[:-1] + (SLAB // per, per))
    out = np.zeros(c.shape[:-1], dtype=np.uint8)
    for e in range(per):
        out |= (c[..., e] << (pb * e)).astype(np.uint8)
    return out


# ================================================================================
# The cache: quantized history + 2G bf16 residual buffer
# ================================================================================


class OracleCache:
    """One layer's cache for ``batch`` sequences and ``num_kv_heads`` KV heads.

    State (Lq, r).  Lq counts quantized tokens, a multiple of G.  r counts
    residual bf16 tokens, 0 <= r < 2G.  The residual buffer is linear: slot 0
    holds the oldest token.  Appending one token goes like this (QuantSpec page,
    Approach: a double full-precision buffer of size 2G):

      1. write it to slot r; r += 1
      2. if r == 2G: quantize slots [0, G) as token group [Lq, Lq + G);
         move slots [G, 2G) to [0, G); Lq += G; r = G

    So once N >= 2G tokens have arrived, at least G recent tokens stay in bf16.
    Closed form: Lq = G*(floor(N/G) - 1), r = N - Lq.  Keys and values are both
    quantized when their group is flushed.
    """

    def __init__(self, batch: int, num_kv_heads: int, head_dim: int, group_size: int,
                 fmt: str, capacity: int):
        if fmt not in FORMAT_BITS:
            raise ValueError(fmt)
        if capacity % group_size:
            raise ValueError("capacity must be a multiple of the group size")
        if head_dim % group_size:
            raise ValueError("value groups span G channels: G must divide head_dim")
        self.B, self.H, self.D, self.G = batch, num_kv_heads, head_dim, group_size
        self.fmt, self.bits, self.capacity = fmt, FORMAT_BITS[fmt], capacity
        B, H, D, G = self.B, self.H, self.D, self.G
        self.k_codes = np.zeros((B, H, capacity, D), np.uint8)
        self.v_codes = np.zeros((B, H, capacity, D), np.uint8)
        self.k_scale = np.zeros((B, H, capacity // G, D), F32)
        self.k_zero = np.zeros((B, H, capacity // G, D), F32)
        self.v_scale = np.zeros((B, H, capacity, D // G), F32)
        self.v_zero = np.zeros((B, H, capacity, D // G), F32)
        self.res_k = np.zeros((B, H, 2 * G, D), F32)
        self.res_v = np.zeros((B, H, 2 * G, D), F32)
        self.Lq = 0
        self.r = 0

    # -- appending ---------------------------------------------------------------

    def _flush(self):
        G, L = self.G, self.Lq
        if L + G > self.capacity:
            raise OverflowError("quantized capacity exceeded")
        kc, ks, kz = quantize_key_group(self.res_k[:, :, :G], self.bits)
        vc, vs, vz = quantize_value_group(self.res_v[:, :, :G], self.bits, G)
        self.k_codes[:, :, L:L + G] = kc
        self.k_scale[:, :, L // G] = ks
        self.k_zero[:, :, L // G] = kz
        self.v_codes[:, :, L:L + G] = vc
        self.v_scale[:, :, L:L + G] = vs
        self.v_zero[:, :, L:L + G] = vz
        self.res_k[:, :, :G] = self.res_k[:, :, G:].copy()
        self.res_v[:, :, :G] = self.res_v[:, :, G:].copy()
        self.Lq += G
        self.r = G

    def append_token(self, k1: np.ndarray, v1: np.ndarray):
        """Append one token: ``k1, v1`` are ``[B, Hkv, D]`` bf16-valued float32."""
        self.res_k[:, :, self.r] = k1
        self.res_v[:, :, self.r] = v1
        self.r += 1
        if self.r == 2 * self.G:
            self._flush()

    def append(self, k_new: np.ndarray, v_new: np.ndarray):
        """Append ``n`` tokens (``[B, Hkv, n, D]``) as n single-token steps."""
        n = k_new.shape[2]
        T = self.r + n
        f = 0 if T < 2 * self.G else T // self.G - 1
        if self.Lq + f * self.G > self.capacity:
            raise OverflowError("quantized capacity exceeded")
        for i in range(n):
            self.append_token(k_new[:, :, i], v_new[:, :, i])

    # -- views -------------------------------------------------------------------

    def residual(self):
        return self.res_k[:, :, :self.r], self.res_v[:, :, :self.r]

    def packed_k_planes(self):
        """Stored key planes ``[B, Hkv, Lq, rowbytes]``: [upper, lower] nibble
        planes for the hierarchical format, [codes] otherwise."""
        c = self.k_codes[:, :, :self.Lq]
        if self.fmt == "hier8":
            hi, lo = split_hierarchical(c)
            return [pack_k_plane(hi, 4), pack_k_plane(lo, 4)]
        return [pack_k_plane(c, self.bits)]

    def packed_v_planes(self):
        """Stored value planes ``[B, Hkv, Lq/32, D, slabbytes]``."""
        c = self.v_codes[:, :, :self.Lq]
        if self.fmt == "hier8":
            hi, lo = split_hierarchical(c)
            return [pack_v_plane(hi, 4), pack_v_plane(lo, 4)]
        return [pack_v_plane(c, self.bits)]

    def dequant_unit(self, mode: str, b: int, h: int):
        """Dequantized keys and values of (b, kv head h) in fp64, ``[Lq, D]`` each:
        x_hat = code * scale + zero under the mode's (code, scale)."""
        fmt, _, _ = MODES[mode]
        if fmt != self.fmt:
            raise ValueError(f"mode {mode} cannot read format {self.fmt}")
        L, G, D = self.Lq, self.G, self.D
        kc, ks = mode_codes_scale(mode, self.k_codes[b, h, :L], self.k_scale[b, h, :L // G])
        vc, vs = mode_codes_scale(mode, self.v_codes[b, h, :L], self.v_scale[b, h, :L])
        kz = mode_zero(mode, self.k_zero[b, h, :L // G], self.k_scale[b, h, :L // G])
        vz = mode_zero(mode, self.v_zero[b, h, :L], self.v_scale[b, h, :L])
        khat = kc.astype(np.float64) * np.repeat(ks, G, axis=0) + np.repeat(kz, G, axis=0)
        vhat = (vc.astype(np.float64).reshape(L, D // G, G) * vs[:, :, None] + vz[:, :, None]).reshape(L, D)
        return khat, vhat


# ================================================================================
# Attention (fp64)
# ================================================================================


def _units(B: int, H: int, units: Optional[Iterable]):
    if units is None:
        return [(b, h) for b in range(B) for h in range(H)]
    return list(units)


def attend(cache: OracleCache, mode: str, q: np.ndarray,
           pend_k: Optional[np.ndarray] = None, pend_v: Optional[np.ndarray] = None,
           sel_idx: Optional[np.ndarray] = None, sel_k: Optional[np.ndarray] = None,
           sel_v: Optional[np.ndarray] = None, sm_scale: Optional[float] = None,
           units: Optional[Sequence] = None):
    """Decode attention of gamma query tokens over the cache, in fp64.

    ``q [B, gamma, Hq, D]``.  Query head h uses KV head floor(h / (Hq/Hkv)),
    i.e. consecutive grouping.  Query token i sees these keys:

    * every quantized token t in [0, Lq), dequantized under ``mode``.  If t
      appears in ``sel_idx[b, kvh]``, the 16-bit ``sel_k/sel_v`` row replaces its
      low-bit copy (SpeCache page, Approach: the top-k 16-bit KV pairs).
      Entries outside [0, Lq) are ignored.  Valid entries must be distinct.
    * every residual bf16 token (QuantSpec page, Approach: the full-precision
      buffer keeps recent tokens unquantized).
    * pending speculative token p in [0, P) when p <= P - gamma + i.  That is
      causal masking among the gamma query tokens, which are the last gamma of
      the P pending tokens.

    logit = sm_scale * (q . k), with sm_scale = 1/sqrt(D) by default.
    Returns ``out [B, gamma, Hq, D]`` (fp64) and ``lse [B, gamma, Hq]``
    (natural log of the softmax denominator).  A query with no visible key gets
    out = 0 and lse = -inf.  Only the (b, kv head) pairs in ``units`` are
    computed; the rest stay 0 / -inf.
    """
    B, gamma, Hq, D = q.shape
    H = cache.H
    if Hq % H:
        raise ValueError("Hq must be a multiple of Hkv")
    hg = Hq // H
    P = 0 if pend_k is None else pend_k.shape[2]
    if P and P < gamma:
        raise ValueError("need at least gamma pending tokens")
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, gamma, Hq, D), np.float64)
    lse = np.full((B, gamma, Hq), -np.inf, np.float64)
    rk, rv = cache.residual()
    for (b, h) in _units(B, H, units):
        khat, vhat = cache.dequant_unit(mode, b, h)
        keep = np.ones(cache.Lq, bool)
        xk, xv = [], []
        if sel_idx is not None:
            for j in range(sel_idx.shape[2]):
                t = int(sel_idx[b, h, j])
                if 0 <= t < cache.Lq:
                    if not keep[t]:
                        raise ValueError("duplicate selected index")
                    keep[t] = False
                    xk.append(sel_k[b, h, j].astype(np.float64))
                    xv.append(sel_v[b, h, j].astype(np.float64))
        base_k = [khat[keep], rk[b, h].astype(np.float64)]
        base_v = [vhat[keep], rv[b, h].astype(np.float64)]
        if xk:
            base_k.append(np.stack(xk))
            base_v.append(np.stack(xv))
        for i in range(gamma):
            nvis = (P - gamma + i + 1) if P else 0
            keys = np.concatenate(base_k + [pend_k[b, h, :nvis].astype(np.float64)] if P else base_k)
            vals = np.concatenate(base_v + [pend_v[b, h, :nvis].astype(np.float64)] if P else base_v)
            if keys.shape[0] == 0:
                continue
            for hh in range(hg):
                hq = h * hg + hh
                logits = sm_scale * (keys @ q[b, i, hq].astype(np.float64))
                m = logits.max()
                e = np.exp(logits - m)
                s = e.sum()
                out[b, i, hq] = (e @ vals) / s
                lse[b, i, hq] = m + math.log(s)
    return out, lse


# ================================================================================
# Top-k under the low-bit keys (exact integer scoring)
# ================================================================================

W_BITS = 21          # magnitude bits of the integer-rounded folded query weights
Z_BITS = 40          # magnitude bits of the integer-rounded zero-point products
E_MIN = -100         # floor on the weight exponent (keeps the unit a normal fp32)


Z_EMIN = -80         # floor on the product exponent (keeps 2^(f - 40) a normal fp32)


def _exponent(M: float, floor: int = E_MIN) -> int:
    """e with M < 2^e (frexp's exponent), floored; 0 for M = 0."""
    e = math.frexp(M)[1] if M > 0 else 0
    return max(e, floor)


def score_group(qs: np.ndarray, scale_eff: np.ndarray, zero: np.ndarray,
                codes: np.ndarray) -> np.ndarray:
    """Top-k score of the G tokens of one key group for one summed query.

    The pages say only that the k tokens attended most, as predicted from the
    speculative token under the low-bit keys, are prefetched (SpeCache page,
    Approach).  The score is the logit qs . k_hat, with k_hat = code * scale +
    zero per channel.  It is computed so that any correct implementation gets
    the same fp32 value, bit for bit:

      w_d   = fp32(qs_d * scale_d)                           (folded weight)
      e     = exponent of max_d |w_d| (max|w| < 2^e), floored at -100
      W_d   = rint(w_d * 2^(21 - e))                         (|W_d| <= 2^21)
      S_t   = sum_d W_d * code_{t,d}                         (exact integer)
      p_d   = fp32(qs_d * z_d)                               (zero-point product)
      f     = exponent of max_d |p_d| (max|p| < 2^f), floored at -80
      Z     = sum_d rint(p_d * 2^(40 - f))                   (exact integer)
      beta  = fp32(Z) * 2^(f - 40)
      score = fp32( fp32(fp32(S_t) * 2^(e - 21)) + beta )

    Both sums are exact integers, so no summation order can change the
    score: every implementation, serial or parallel, reaches the same bits.
    The roundings are the weights' 2^-21 and the products' 2^-40 relative
    rounding to integers, fp32(S_t), fp32(Z), exact power-of-two scalings and
    the final add.
    """
    D = qs.shape[0]
    w = (qs.astype(F32) * scale_eff.astype(F32)).astype(F32)
    e = _exponent(float(np.max(np.abs(w)))) if D else 0
    W = np.rint(w.astype(np.float64) * (2.0 ** (W_BITS - e))).astype(np.int64)
    S = codes.astype(np.int64) @ W                       # exact integer dot products
    Sf = S.astype(np.float64).astype(F32)                # |S| < 2^53: one rounding
    unit = F32(2.0 ** (e - W_BITS))
    beta = zero_term(qs, zero)
    return ((Sf * unit).astype(F32) + beta).astype(F32)


def zero_term(qs: np.ndarray, zero: np.ndarray) -> np.float32:
    """beta = fp32(sum_d rint(p_d 2^(40-f))) * 2^(f-40), p_d = fp32(qs_d z_d),
    f the exponent of max|p| (floored at -80).  The sum of integers is exact
    (|each| <= 2^40, at most a few thousand terms), so its order is free."""
    p = (qs.astype(F32) * zero.astype(F32)).astype(F32)
    f = _exponent(float(np.max(np.abs(p))), Z_EMIN) if p.size else 0
    Z = int(np.sum(np.rint(p.astype(np.float64) * (2.0 ** (Z_BITS - f))).astype(np.int64)))
    return F32(F32(float(Z)) * F32(2.0 ** (f - Z_BITS)))


def score_group_inputs(cache: "OracleCache", mode: str, b: int, h: int, g: int):
    """(codes, effective scale, zero point) of key group g of (b, kv head h) as
    the top-k score reads them, all fp32: INT4 and INT4-mid read the upper
    nibble with fp32(16 s); INT4-mid's zero point is fp32(z + fp32(8 s)), one
    rounding (8 s is exact).  INT1-centred reads fp32(s / 2) and
    fp32(z + fp32(s / 4)) (both products exact)."""
    G = cache.G
    codes = cache.k_codes[b, h, g * G:(g + 1) * G]
    s = cache.k_scale[b, h, g].astype(F32)
    z = cache.k_zero[b, h, g].astype(F32)
    if mode == "int4mid":
        z = (z + (F32(MID_NIBBLE) * s).astype(F32)).astype(F32)
    if mode in ("int4", "int4mid"):
        codes = codes >> 4
        s = (s * F32(16)).astype(F32)
    if mode == "int1c":
        z = (z + (F32(CENTER_SHIFT) * s).astype(F32)).astype(F32)
        s = (s * F32(0.5)).astype(F32)
    return codes, s, z


def summed_query(q_spec_b: np.ndarray, h: int, hg: int) -> np.ndarray:
    """fp32 sum, ascending head order, of the speculative token's query heads
    that share KV head h.  Under MHA (hg = 1) it is that head's query.  The
    pages do not say how grouped heads are combined; the sum makes the score
    the summed logit of the group."""
    qs = np.zeros(q_spec_b.shape[-1], F32)
    for hh in range(hg):
        qs = (qs + q_spec_b[h * hg + hh].astype(F32)).astype(F32)
    return qs


def topk(cache: OracleCache, mode: str, q_spec: np.ndarray, k: int,
         units: Optional[Sequence] = None):
    """Per KV head, the k quantized tokens with the highest low-bit score.

    ``q_spec [B, Hq, D]`` is the speculative token's query (SpeCache page,
    Approach).  Candidates are the quantized tokens t in [0, Lq); residual
    tokens are already 16-bit on the device.  Tokens are ordered by (score
    descending, index ascending).  Slots beyond Lq get index -1 and score -inf.
    Returns ``idx [B, Hkv, k] int32`` and ``score [B, Hkv, k] float32``.
    """
    B, Hq, D = q_spec.shape
    H, G, L = cache.H, cache.G, cache.Lq
    hg = Hq // H
    fmt, _, mult = MODES[mode]
    if fmt != cache.fmt:
        raise ValueError(f"mode {mode} cannot read format {cache.fmt}")
    idx = np.full((B, H, k), -1, np.int32)
    score = np.full((B, H, k), -np.inf, F32)
    for (b, h) in _units(B, H, units):
        qs = summed_query(q_spec[b], h, hg)
        sc = np.empty(L, F32)
        for g in range(L // G):
            codes, s, z = score_group_inputs(cache, mode, b, h, g)
            sc[g * G:(g + 1) * G] = score_group(qs, s, z, codes)
        order = sorted(range(L), key=lambda t: (-float(sc[t]), t))[:k]
        idx[b, h, :len(order)] = order
        score[b, h, :len(order)] = sc[order]
    return idx, score


def all_scores(cache: OracleCache, mode: str, q_spec: np.ndarray, b: int, h: int) -> np.ndarray:
    """Scores of every quantized token of (b, kv head h) (used by tests)."""
    Hq = q_spec.shape[1]
    hg = Hq // cache.H
    qs = summed_query(q_spec[b], h, hg)
    G = cache.G
    out = np.empty(cache.Lq, F32)
    for g in range(cache.Lq // G):
        codes, s, z = score_group_inputs(cache, mode, b, h, g)
        out[g * G:(g + 1) * G] = score_group(qs, s, z, codes)
    return out


# ================================================================================
# Fetch of the selected 16-bit KV
# ================================================================================


def gather_selected(full_k: np.ndarray, full_v: np.ndarray, sel_idx: np.ndarray):
    """The selected tokens' 16-bit K/V out of the full-precision store.

    SpeCache keeps the whole 16-bit cache in CPU memory and, each step, fetches
    the top-k pairs the speculative token predicted (SpeCache page, Approach).
    ``full_k, full_v [B, Hkv, N, D]`` (any dtype), ``sel_idx [B, Hkv, k]``.
    Entry j of (b, h) is row ``sel_idx[b, h, j]`` of that head.  Reading: an
    index outside [0, N), such as the -1 that pads a short top-k list, gives a
    row of zeros (the attention ignores those entries).
    Returns ``sel_k, sel_v [B, Hkv, k, D]``.
    """
    B, H, N, D = full_k.shape
    k = sel_idx.shape[2]
    sel_k = np.zeros((B, H, k, D), full_k.dtype)
    sel_v = np.zeros((B, H, k, D), full_v.dtype)
    for b in range(B):
        for h in range(H):
            for j in range(k):
                t = int(sel_idx[b, h, j])
                if 0 <= t < N:
                    sel_k[b, h, j] = full_k[b, h, t]
                    sel_v[b, h, j] = full_v[b, h, t]
    return sel_k, sel_v
