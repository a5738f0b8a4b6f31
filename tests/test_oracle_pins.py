"""Pins of the CPU oracle against things other than itself.

Sources: hand-derived closed forms (tests/golden), brute force on tiny inputs,
invariants the pages state, and textbook or library special cases (torch's
scaled_dot_product_attention in fp64).  Each test says which plausible oracle
mistake it catches.  Every oracle function has a pin here; no function is
"parity unpinned".
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import kvq_inputs as ki
import oracle
from oracle import kvq_oracle as ko

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------------------------
# Quantizer
# ------------------------------------------------------------------------------------


@pytest.mark.parametrize("case", _golden("quantizer_examples.json")["cases"], ids=lambda c: c["name"])
def test_quantizer_golden(case):
    """Hand-derived codes, scales and zeros: catches a wrong level count, floor
    instead of half-even rounding, or a wrong zero point."""
    x = np.array(case["x"], F32)
    c, s, z = oracle.quantize_minmax(x, case["bits"], axis=0)
    assert c.tolist() == case["codes"]
    assert float(s) == pytest.approx(case["scale"], rel=0, abs=1e-12)
    assert float(z) == case["zero"]
    if "upper_nibble" in case:
        hi, lo = oracle.split_hierarchical(c)
        assert hi.tolist() == case["upper_nibble"]
        assert lo.tolist() == case["lower_nibble"]
    if "upper_plane_bytes" in case:
        hi, lo = oracle.split_hierarchical(c)
        assert oracle.pack_k_plane(hi[None, :], 4)[0].tolist() == case["upper_plane_bytes"]
        assert oracle.pack_k_plane(lo[None, :], 4)[0].tolist() == case["lower_plane_bytes"]


@pytest.mark.parametrize("bits", [8, 2, 1])
def test_quantizer_roundtrip_bound_and_bruteforce(bits):
    """Each code is the nearest level: error <= scale*(1/2 + 2^-12), and the code
    is the argmin over all 2^b levels except within fp32 noise of a half-tie.
    Catches scale = range/2^b, floor rounding, a wrong zero, a transposed axis."""
    g = ki.rng(7, bits)
    x = ki.normal_bf16(g, (64, 16))
    c, s, z = oracle.quantize_minmax(x, bits, axis=0)           # per column over 64 rows
    s64, z64 = s.astype(np.float64), z.astype(np.float64)
    xh = c.astype(np.float64) * s64 + z64
    err = np.abs(x.astype(np.float64) - xh)
    assert np.all(err <= s64 * (0.5 + 2.0 ** -12) + 1e-30)
    levels = np.arange(2 ** bits, dtype=np.float64)
    for j in range(x.shape[1]):
        d = np.abs(x[:, j, None].astype(np.float64) - (levels[None, :] * s64[j] + z64[j]))
        best = d.argmin(axis=1)
        second = np.sort(d, axis=1)[:, 1]
        near_tie = (second - d.min(axis=1)) <= 2.0 ** -11 * s64[j]
        assert np.all((best == c[:, j]) | near_tie)
    assert np.all(c <= 2 ** bits - 1)
    # extremes map to the end codes exactly
    assert np.all(c[x.argmin(axis=0), np.arange(16)] == 0)
    assert np.all(c[x.argmax(axis=0), np.arange(16)] == 2 ** bits - 1)


def test_quantizer_negative_zero_canonical():
    """A group of -0.0 values gets zero point +0.0 (bit pattern 0)."""
    x = np.array([-0.0, -0.0, -0.0, -0.0], F32)
    c, s, z = oracle.quantize_minmax(x, 8, 0)
    assert np.asarray(z, F32).view(np.uint32) == 0
    assert float(s) == 0.0 and c.tolist() == [0, 0, 0, 0]


@pytest.mark.parametrize("bits", [8, 2, 1])
def test_lossless_affine_grid_keys_per_channel_values_per_token(bits):
    """Lossless special case.  If each quantization group already lies on a
    power-of-two affine grid that uses both end levels, dequant returns the
    input exactly.  The key grid differs per channel and the value grid per
    (token, channel block).  So a key axis transposed to per-token, or a value
    axis transposed to per-channel, breaks exactness."""
    G, D = 32, 64
    g = ki.rng(11, bits)
    top = 2 ** bits - 1
    kcodes = g.integers(0, top + 1, (G, D))
    kcodes[0, :], kcodes[1, :] = 0, top
    ks = (2.0 ** g.integers(-4, 2, D)).astype(F32)
    kz = g.integers(-8, 8, D).astype(F32) * F32(0.25)
    K = (kcodes * ks[None, :] + kz[None, :]).astype(F32)
    c, s, z = oracle.quantize_key_group(K, bits)
    assert np.array_equal(c, kcodes) and np.array_equal(s, ks) and np.array_equal(z, kz)
    vcodes = g.integers(0, top + 1, (G, D))
    vcodes.reshape(G, D // G, G)[:, :, 0] = 0
    vcodes.reshape(G, D // G, G)[:, :, 1] = top
    vs = (2.0 ** g.integers(-4, 2, (G, D // G))).astype(F32)
    vz = g.integers(-8, 8, (G, D // G)).astype(F32) * F32(0.5)
    V = (vcodes.reshape(G, D // G, G) * vs[:, :, None] + vz[:, :, None]).reshape(G, D).astype(F32)
    c, s, z = oracle.quantize_value_group(V, bits, G)
    assert np.array_equal(c, vcodes) and np.array_equal(s, vs) and np.array_equal(z, vz)


def _cache_from_tokens(fmt, G, K, V, cap=None):
    B, H, N, D = K.shape
    cap = cap or (N // G + 1) * G
    c = oracle.OracleCache(B, H, D, G, fmt, cap)
    c.append(K, V)
    return c


def test_int4_is_int8_with_lower_nibble_zeroed():
    """The hierarchy invariant (QuantSpec page, Approach).  INT4 dequant equals
    INT8 dequant recomputed here with the lower nibble masked off.  Catches a
    missing 16x on the INT4 scale or a wrong nibble."""
    K, V = ki.kv_stream(3, 1, 2, 200, 64)
    c = _cache_from_tokens("hier8", 32, K, V)
    for h in range(2):
        k4, v4 = c.dequant_unit("int4", 0, h)
        L, G = c.Lq, c.G
        kc = (c.k_codes[0, h, :L] & 0xF0).astype(np.float64)
        ks = np.repeat(c.k_scale[0, h, :L // G].astype(np.float64), G, axis=0)
        kz = np.repeat(c.k_zero[0, h, :L // G].astype(np.float64), G, axis=0)
        np.testing.assert_array_equal(k4, kc * ks + kz)
        vc = (c.v_codes[0, h, :L] & 0xF0).astype(np.float64)
        vs = np.repeat(c.v_scale[0, h, :L].astype(np.float64), G, axis=1)
        vz = np.repeat(c.v_zero[0, h, :L].astype(np.float64), G, axis=1)
        np.testing.assert_array_equal(v4, vc * vs + vz)


# ------------------------------------------------------------------------------------
# The 2G double buffer
# ------------------------------------------------------------------------------------


@pytest.mark.parametrize("G,N", [(32, 0), (32, 1), (32, 63), (32, 64), (32, 65), (32, 95), (32, 96),
                                 (32, 544), (64, 1000), (128, 8320)])
def test_buffer_closed_form(G, N):
    """Closed form of the state after N tokens: Lq = G*(floor(N/G) - 1) once
    N >= 2G, r = N - Lq in [G, 2G); before that everything is residual.
    Catches flushing all 2G tokens, or flushing at 2G - 1."""
    D = max(64, G)
    K, V = ki.kv_stream(5, 1, 1, N, D, outlier_channels=0)
    c = _cache_from_tokens("hier8", G, K, V, cap=max(G, (N // G) * G))
    exp_lq = 0 if N < 2 * G else G * (N // G - 1)
    assert c.Lq == exp_lq and c.r == N - exp_lq
    if N:
        assert c.r < 2 * G


def test_buffer_contents_match_direct_group_quantization():
    """After N tokens appended in uneven chunks, each quantized group equals the
    quantizer applied directly to input tokens [gG, gG+G), and the residual
    holds the last r input tokens in order.  Catches off-by-one errors in the
    flush or move."""
    G, D, N = 32, 64, 421
    K, V = ki.kv_stream(9, 2, 2, N, D)
    c = oracle.OracleCache(2, 2, D, G, "int2", 448)
    pos = 0
    for n in [1, 5, 70, 0, 33, 200, 112]:
        c.append(K[:, :, pos:pos + n], V[:, :, pos:pos + n])
        pos += n
    assert pos == N
    for g in range(c.Lq // G):
        kc, ks, kz = oracle.quantize_key_group(K[:, :, g * G:(g + 1) * G], 2)
        vc, vs, vz = oracle.quantize_value_group(V[:, :, g * G:(g + 1) * G], 2, G)
        assert np.array_equal(c.k_codes[:, :, g * G:(g + 1) * G], kc)
        assert np.array_equal(c.k_scale[:, :, g], ks) and np.array_equal(c.k_zero[:, :, g], kz)
        assert np.array_equal(c.v_codes[:, :, g * G:(g + 1) * G], vc)
        assert np.array_equal(c.v_scale[:, :, g * G:(g + 1) * G], vs)
    rk, rv = c.residual()
    assert np.array_equal(rk, K[:, :, c.Lq:]) and np.array_equal(rv, V[:, :, c.Lq:])


def test_capacity_checked_before_any_write():
    K, V = ki.kv_stream(1, 1, 1, 200, 64)
    c = oracle.OracleCache(1, 1, 64, 32, "hier8", 64)
    with pytest.raises(OverflowError):
        c.append(K, V)
    assert c.Lq == 0 and c.r == 0


# ------------------------------------------------------------------------------------
# Packing (independent bit-level unpack)
# ------------------------------------------------------------------------------------


@pytest.mark.parametrize("pb", [4, 2, 1])
def test_pack_layouts_against_bitlevel_unpack(pb):
    """Unpack the packed planes bit by bit with np.unpackbits and compare them to
    the logical codes.  Catches a swapped nibble order or a transposed slab."""
    g = ki.rng(13, pb)
    T, D = 64, 64
    codes = g.integers(0, 2 ** pb, (T, D)).astype(np.uint8)
    kp = oracle.pack_k_plane(codes, pb)
    bitsk = np.unpackbits(kp, axis=-1, bitorder="little").reshape(T, D, pb)
    k_back = (bitsk * (1 << np.arange(pb))).sum(-1)
    assert np.array_equal(k_back, codes)
    vp = oracle.pack_v_plane(codes, pb)
    assert vp.shape == (T // 32, D, 32 * pb // 8)
    bitsv = np.unpackbits(vp, axis=-1, bitorder="little").reshape(T // 32, D, 32, pb)
    v_back = (bitsv * (1 << np.arange(pb))).sum(-1)          # [slab, d, tok]
    assert np.array_equal(v_back.transpose(0, 2, 1).reshape(T, D), codes)


# ------------------------------------------------------------------------------------
# Attention
# ------------------------------------------------------------------------------------


def _sdpa_reference(q, keys, vals, mask, scale):
    """torch fp64 scaled_dot_product_attention: one query, a key list."""
    qt = torch.from_numpy(q[None, None, None, :].astype(np.float64))
    kt = torch.from_numpy(keys[None, None].astype(np.float64))
    vt = torch.from_numpy(vals[None, None].astype(np.float64))
    mt = torch.from_numpy(mask[None, None, None, :])
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mt, scale=scale)
    return o[0, 0, 0].numpy()


def test_int4mid_is_int8_with_lower_nibble_eight():
    """The midpoint reading of the draft code: INT4-mid dequant equals INT8
    dequant recomputed here with the lower nibble replaced by 8, i.e. the
    middle of the sixteen 8-bit codes one upper nibble stands for.  Catches a
    wrong midpoint, a midpoint in units of the 16x scale, and a zero point
    that does not move."""
    K, V = ki.kv_stream(5, 1, 2, 260, 64)
    c = _cache_from_tokens("hier8", 32, K, V)
    for h in range(2):
        km, vm = c.dequant_unit("int4mid", 0, h)
        L, G = c.Lq, c.G
        kc = ((c.k_codes[0, h, :L] & 0xF0) | 8).astype(np.float64)
        ks = np.repeat(c.k_scale[0, h, :L // G].astype(np.float64), G, axis=0)
        kz = np.repeat(c.k_zero[0, h, :L // G].astype(np.float64), G, axis=0)
        ref_k = kc * ks + kz
        np.testing.assert_allclose(km, ref_k, rtol=0, atol=1e-14 * np.abs(ref_k).max())
        vc = ((c.v_codes[0, h, :L] & 0xF0) | 8).astype(np.float64)
        vs = np.repeat(c.v_scale[0, h, :L].astype(np.float64), G, axis=1)
        vz = np.repeat(c.v_zero[0, h, :L].astype(np.float64), G, axis=1)
        ref_v = vc * vs + vz
        np.testing.assert_allclose(vm, ref_v, rtol=0, atol=1e-14 * np.abs(ref_v).max())


def test_int4mid_error_bound_halves_int4():
    """Reconstruction error against the original bf16 values: the INT8 code is
    within half a step of x, and the lower nibble read as 8 is within 8 steps
    of the true lower nibble, so INT4-mid is within 8.5 steps of x, where the
    truncating INT4 reading can be 15.5 steps off (and is more than 8.5 steps
    off somewhere on these inputs)."""
    G, D = 32, 64
    K, V = ki.kv_stream(9, 1, 1, 8 * G + 5, D)
    c = _cache_from_tokens("hier8", G, K, V)
    L = c.Lq
    ks = np.repeat(c.k_scale[0, 0, :L // G].astype(np.float64), G, axis=0)
    km, _ = c.dequant_unit("int4mid", 0, 0)
    k4, _ = c.dequant_unit("int4", 0, 0)
    err_mid = np.abs(km - K[0, 0, :L])
    err_4 = np.abs(k4 - K[0, 0, :L])
    assert np.all(err_mid <= 8.5 * ks * (1 + 2.0 ** -10) + 1e-30)
    assert np.all(err_4 <= 15.5 * ks * (1 + 2.0 ** -10) + 1e-30)
    assert np.any(err_4 > 8.5 * ks * (1 + 2.0 ** -10))
    assert err_mid.mean() < err_4.mean()


def test_int4mid_topk_zero_point_moves_by_eight_steps():
    """The top-k score of INT4-mid reads zero point fp32(z + 8 s) with the
    8-bit scale s: equal to the INT4 score of a cache whose zero points were
    moved by hand."""
    G, D, N = 32, 64, 5 * 32 + 7
    K, V = ki.kv_stream(13, 1, 1, N, D)
    c = _cache_from_tokens("hier8", G, K, V)
    q = ki.queries(13, 1, 1, 1, D)[:, 0]
    mid = oracle.all_scores(c, "int4mid", q, 0, 0)
    c.k_zero[0, 0, :c.Lq // G] = (c.k_zero[0, 0, :c.Lq // G] + F32(8) * c.k_scale[0, 0, :c.Lq // G]).astype(F32)
    moved = oracle.all_scores(c, "int4", q, 0, 0)
    np.testing.assert_array_equal(mid.view(np.uint32), moved.view(np.uint32))


def test_int1c_levels_golden():
    """The centred 1-bit reading on a hand-worked key group: one channel over
    G = 32 tokens holds -1 (token 0), 3 (token 1) and 0 elsewhere.  Stored:
    min -1, scale (range) 4; codes round((x + 1) / 4): -1 -> 0, 0 -> 0 (0.25
    rounds down), 3 -> 1.  Plain 1-bit reads the levels -1 and 3; the centred
    reading reads -1 + 4/4 = 0 and -1 + 3 * 4/4 = 2, so the zeros come back
    exact and the outliers at 0 and 2.  Catches a shift of a half (levels 1
    and 3), an unhalved scale (0 and 4), and codes that moved."""
    G, D = 32, 64
    K = np.zeros((1, 1, 2 * G, D), F32)              # the first group flushes once 2G tokens arrived
    V = np.zeros((1, 1, 2 * G, D), F32)
    K[0, 0, 0, 5], K[0, 0, 1, 5] = -1.0, 3.0
    c = _cache_from_tokens("int1", G, K, V)
    assert c.Lq == G
    assert c.k_zero[0, 0, 0, 5] == F32(-1) and c.k_scale[0, 0, 0, 5] == F32(4)
    assert list(c.k_codes[0, 0, :3, 5]) == [0, 1, 0]
    k1, _ = c.dequant_unit("int1", 0, 0)
    kc, _ = c.dequant_unit("int1c", 0, 0)
    assert list(k1[:3, 5]) == [-1.0, 3.0, -1.0]
    assert list(kc[:3, 5]) == [0.0, 2.0, 0.0]
    assert np.all(kc[2:, 5] == 0.0)
    assert np.all(kc[:, :5] == 0.0)                    # constant channels stay exact


def test_int1c_quarters_the_error_on_evenly_spread_values():
    """For values spread evenly over [min, max] the two halves' centres are the
    best two levels given the midpoint threshold: the mean squared error drops
    from r^2/12 (levels at min and max) to r^2/48."""
    G, D = 32, 64
    g = ki.rng(71, 0)
    vals = np.linspace(0.0, 1.0, G, dtype=np.float64)
    K = np.stack([g.permutation(vals) for _ in range(D)], axis=1)[None, None].astype(F32)
    K = np.concatenate([K, K], axis=2)                 # 2G tokens: the first group flushes
    c = _cache_from_tokens("int1", G, K, np.zeros_like(K))
    assert c.Lq == G
    k1, _ = c.dequant_unit("int1", 0, 0)
    kc, _ = c.dequant_unit("int1c", 0, 0)
    e1 = float(np.mean((k1 - K[0, 0, :G]) ** 2))
    ec = float(np.mean((kc - K[0, 0, :G]) ** 2))
    # the 32 evenly spaced points make the ratio slightly above a quarter
    assert 0.2 < ec / e1 < 0.3


def test_int1c_is_int1_with_moved_levels():
    """Attention under the centred reading equals plain 1-bit attention on a
    cache whose zero points were moved by a quarter of the scale and whose
    scales were halved by hand; the top-k score reads the same fp32 zero point
    z + s/4 and scale s/2."""
    G, D, N = 32, 64, 4 * 32 + 9
    K, V = ki.kv_stream(23, 1, 2, N, D)
    c = _cache_from_tokens("int1", G, K, V)
    q = ki.queries(23, 1, 2, 4, D)
    out_c, lse_c = oracle.attend(c, "int1c", q)
    sc_c = oracle.all_scores(c, "int1c", q[:, 1], 0, 1)
    L = c.Lq
    c.k_zero[:, :, :L // G] = (c.k_zero[:, :, :L // G] + F32(0.25) * c.k_scale[:, :, :L // G]).astype(F32)
    c.k_scale[:, :, :L // G] = (c.k_scale[:, :, :L // G] * F32(0.5)).astype(F32)
    c.v_zero[:, :, :L] = (c.v_zero[:, :, :L] + F32(0.25) * c.v_scale[:, :, :L]).astype(F32)
    c.v_scale[:, :, :L] = (c.v_scale[:, :, :L] * F32(0.5)).astype(F32)
    out_1, lse_1 = oracle.attend(c, "int1", q)
    sc_1 = oracle.all_scores(c, "int1", q[:, 1], 0, 1)
    np.testing.assert_allclose(out_c, out_1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_c, lse_1, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(sc_c.view(np.uint32), sc_1.view(np.uint32))


@pytest.mark.parametrize("mode,fmt,G", [("int8", "hier8", 32), ("int4", "hier8", 32), ("int4mid", "hier8", 64),
                                        ("int2", "int2", 32), ("int1", "int1", 64), ("int1c", "int1", 32)])
def test_attention_equals_library_sdpa(mode, fmt, G):
    """The oracle equals torch's fp64 SDPA on the same key/value lists, for GQA
    with causal pending tokens and selected 16-bit overrides.  Catches a
    missing sm_scale, a wrong causal offset, a wrong GQA head map, or a
    selected token counted twice."""
    B, Hkv, Hq, D, N, gamma, P = 2, 2, 4, 64, 3 * G + 17, 3, 4
    K, V = ki.kv_stream(21, B, Hkv, N, D)
    c = _cache_from_tokens(fmt, G, K, V)
    q = ki.queries(21, B, gamma, Hq, D)
    pk, pv = ki.pending(21, B, Hkv, P, D)
    g = ki.rng(21, 5)
    ksel = 5
    sel = np.stack([np.stack([g.choice(c.Lq, ksel, replace=False) for _ in range(Hkv)]) for _ in range(B)])
    sel[0, 1, 2] = -1                                   # ignored entry
    sk = ki.normal_bf16(g, (B, Hkv, ksel, D))
    sv = ki.normal_bf16(g, (B, Hkv, ksel, D))
    out, lse = oracle.attend(c, mode, q, pk, pv, sel, sk, sv)
    scale = 1 / math.sqrt(D)
    rk, rv = c.residual()
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            kh, vh = c.dequant_unit(mode, b, kvh)
            kh, vh = kh.copy(), vh.copy()
            for j in range(ksel):
                t = sel[b, kvh, j]
                if t >= 0:
                    kh[t], vh[t] = sk[b, kvh, j], sv[b, kvh, j]
            keys = np.concatenate([kh, rk[b, kvh], pk[b, kvh]])
            vals = np.concatenate([vh, rv[b, kvh], pv[b, kvh]])
            for i in range(gamma):
                mask = np.ones(len(keys), bool)
                base = c.Lq + c.r
                mask[base + (P - gamma + i + 1):] = False
                ref = _sdpa_reference(q[b, i, h], keys, vals, mask, scale)
                np.testing.assert_allclose(out[b, i, h], ref, rtol=1e-10, atol=1e-12)
                lg = scale * (keys[mask] @ q[b, i, h].astype(np.float64))
                assert lse[b, i, h] == pytest.approx(np.logaddexp.reduce(lg), rel=1e-12)


def test_attention_lossless_equals_dense_over_original():
    """If the cache is lossless, attention over it equals dense attention over
    the original bf16 K/V.  Catches dequantization errors and scale/zero mixups
    that the SDPA pin, which reads the oracle's own dequant, cannot see."""
    G, D, N = 32, 64, 3 * 32 + 5
    g = ki.rng(31)
    ngroups = 2
    K = np.zeros((1, 1, N, D), F32)
    V = np.zeros((1, 1, N, D), F32)
    for grp in range(ngroups):
        kc = g.integers(0, 256, (G, D)); kc[0], kc[1] = 0, 255
        K[0, 0, grp * G:(grp + 1) * G] = kc * F32(2.0 ** -6) - F32(2.0)
        vc = g.integers(0, 256, (G, D)); vc.reshape(G, D // G, G)[:, :, 0] = 0
        vc.reshape(G, D // G, G)[:, :, 1] = 255
        V[0, 0, grp * G:(grp + 1) * G] = vc * F32(2.0 ** -7) - F32(1.0)
    K[0, 0, ngroups * G:] = ki.normal_bf16(g, (N - ngroups * G, D))
    V[0, 0, ngroups * G:] = ki.normal_bf16(g, (N - ngroups * G, D))
    c = _cache_from_tokens("hier8", G, K, V)
    assert c.Lq == ngroups * G
    q = ki.queries(31, 1, 1, 1, D)
    out, lse = oracle.attend(c, "int8", q)
    ref = _sdpa_reference(q[0, 0, 0], K[0, 0], V[0, 0], np.ones(N, bool), 1 / math.sqrt(D))
    np.testing.assert_allclose(out[0, 0, 0], ref, rtol=1e-12, atol=1e-13)


def test_attention_closed_forms():
    """Closed forms.  With every key identical, out is the mean of the values
    and lse = logit + log(n).  With no keys at all, out = 0 and lse = -inf."""
    G, D = 32, 64
    N = 2 * G + 7
    K = np.ones((1, 1, N, D), F32) * F32(0.5)
    g = ki.rng(41)
    V = ki.normal_bf16(g, (1, 1, N, D))
    c = _cache_from_tokens("hier8", G, K, V)
    q = ki.queries(41, 1, 1, 1, D)
    out, lse = oracle.attend(c, "int8", q)
    # Constant key groups have scale 0, so the dequantized keys equal the input.
    vh = c.dequant_unit("int8", 0, 0)[1]
    allv = np.concatenate([vh, c.residual()[1][0, 0]])
    np.testing.assert_allclose(out[0, 0, 0], allv.mean(0), rtol=1e-12, atol=1e-14)
    logit = 0.5 * q[0, 0, 0].astype(np.float64).sum() / math.sqrt(D)
    assert lse[0, 0, 0] == pytest.approx(logit + math.log(N), rel=1e-12)
    empty = oracle.OracleCache(1, 1, D, G, "hier8", 64)
    out, lse = oracle.attend(empty, "int8", q)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_attention_gamma_causal_equals_single_query_calls():
    """Query token i of a gamma-token causal call equals a one-token call that
    sees P - gamma + i + 1 pending tokens."""
    G, D, gamma, P = 32, 64, 4, 6
    K, V = ki.kv_stream(51, 1, 2, 150, D)
    c = _cache_from_tokens("hier8", G, K, V)
    q = ki.queries(51, 1, gamma, 2, D)
    pk, pv = ki.pending(51, 1, 2, P, D)
    out, lse = oracle.attend(c, "int4", q, pk, pv)
    for i in range(gamma):
        nv = P - gamma + i + 1
        o1, l1 = oracle.attend(c, "int4", q[:, i:i + 1], pk[:, :, :nv], pv[:, :, :nv])
        np.testing.assert_allclose(out[:, i], o1[:, 0], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[:, i], l1[:, 0], rtol=1e-13)


# ------------------------------------------------------------------------------------
# Top-k
# ------------------------------------------------------------------------------------


def _exact_logit(cache, mode, qs, b, h):
    """fp64 exact (fsum) logit of the summed query against the dequantized keys."""
    kh, _ = cache.dequant_unit(mode, b, h)
    q64 = qs.astype(np.float64)
    return np.array([math.fsum(q64 * kh[t]) for t in range(kh.shape[0])])


@pytest.mark.parametrize("grp", _golden("topk_score_examples.json")["groups"], ids=lambda g: g["name"])
def test_topk_score_golden(grp):
    """Hand-derived scores of tiny key groups (tests/golden/topk_score_examples.json).
    The first group fixes the order of the zero-point sum: added left to right
    its fp32 sum is 1, added right to left 1 + 2^-22, pairwise 1 + 2^-23.  The
    all-zero-code tokens score exactly beta.  Catches a reordered or pairwise
    beta, an fma-contracted product in the weights, a dropped beta and a wrong
    weight exponent."""
    qs = np.array(grp["qs"], np.float64).astype(F32)
    s = np.array(grp["scale"], np.float64).astype(F32)
    z = np.array(grp["zero"], np.float64).astype(F32)
    codes = np.array(grp["codes"], np.uint8)
    got = oracle.score_group(qs, s, z, codes)
    want = np.array(grp["scores"], np.float64).astype(F32)
    assert got.dtype == F32
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    zero_rows = np.flatnonzero(codes.sum(1) == 0)
    assert zero_rows.size and np.all(got[zero_rows] == F32(grp["beta"]))


def test_topk_score_does_not_depend_on_channel_order():
    """Both sums of the score are exact integers, so permuting the channels
    (the same permutation applied to the query, scales, zero points and code
    columns) leaves every score bit unchanged.  An fp32 running sum of the
    zero-point products fails this on these mixed-magnitude inputs."""
    g = ki.rng(404)
    D, G = 128, 32
    for trial in range(20):
        qs = (g.standard_normal(D) * np.exp2(g.integers(-6, 7, D))).astype(F32)
        s = np.abs(g.standard_normal(D) * 0.3).astype(F32) + F32(1e-3)
        z = (g.standard_normal(D) * np.exp2(g.integers(-8, 6, D))).astype(F32)
        codes = g.integers(0, 4, (G, D)).astype(np.uint8)
        perm = g.permutation(D)
        a = oracle.score_group(qs, s, z, codes)
        b = oracle.score_group(qs[perm], s[perm], z[perm], codes[:, perm])
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_zero_term_is_within_its_rounding_of_the_exact_sum():
    """beta against the exact sum of the fp32 products (math.fsum): within the
    2^-41 relative integer rounding of each product (at the largest product's
    unit) plus one fp32 rounding.  Catches a dropped product, a wrong unit or a
    wrong sign."""
    g = ki.rng(405)
    for trial in range(50):
        D = int(g.integers(1, 200))
        qs = (g.standard_normal(D) * np.exp2(g.integers(-4, 5, D))).astype(F32)
        z = (g.standard_normal(D) * np.exp2(g.integers(-10, 10, D))).astype(F32)
        p = (qs * z).astype(F32).astype(np.float64)
        exact = math.fsum(p)
        beta = float(ko.zero_term(qs, z))
        f = math.frexp(np.abs(p).max())[1]
        assert abs(beta - exact) <= D * 2.0 ** (f - 41) + 2.0 ** -24 * abs(exact) + 1e-300


@pytest.mark.parametrize("mode,fmt", [("int4", "hier8"), ("int4mid", "hier8"), ("int2", "int2"), ("int1", "int1")])
def test_topk_score_fidelity(mode, fmt):
    """The canonical score stays within its stated error of the exact logit
    qs . k_hat, with qs the sum of the group's query heads.  The error budget
    is the 2^-22 relative rounding of each folded weight, then fp32 rounding of
    the partial sums and of the final add.  Catches a dropped zero-point term
    (beta), a missing 16x INT4 scale, a wrong sign, or summing the wrong heads."""
    G, D, N = 32, 128, 6 * 32 + 9
    K, V = ki.kv_stream(61, 1, 2, N, D)
    c = _cache_from_tokens(fmt, G, K, V)
    q = ki.queries(61, 1, 1, 4, D)[:, 0]                  # [B, Hq, D], GQA 2:1
    for h in range(2):
        qs = q[0, 2 * h].astype(np.float64) + q[0, 2 * h + 1].astype(np.float64)
        ex = _exact_logit(c, mode, qs.astype(F32), 0, h)
        sc = oracle.all_scores(c, mode, q, 0, h).astype(np.float64)
        kc, ks = oracle.mode_codes_scale(mode, c.k_codes[0, h, :c.Lq], c.k_scale[0, h])
        for g in range(c.Lq // G):
            w = np.abs(qs * ks[g])
            zterm = np.abs(qs * oracle.mode_zero(mode, c.k_zero[0, h, g], c.k_scale[0, h, g])).sum()
            cw = (kc[g * G:(g + 1) * G].astype(np.float64) * w[None, :]).sum(1)
            bound = 2.0 ** -21 * w.max() * kc[g * G:(g + 1) * G].sum(1) + 2.0 ** -20 * (cw + zterm) \
                + 2.0 ** -23 * np.abs(ex[g * G:(g + 1) * G])
            assert np.all(np.abs(sc[g * G:(g + 1) * G] - ex[g * G:(g + 1) * G]) <= bound)


@pytest.mark.parametrize("mode,fmt", [("int4", "hier8"), ("int2", "int2")])
def test_topk_order_is_the_defined_total_order(mode, fmt):
    """Check the selection by counting, with no sort: each selected token's
    position equals the number of tokens with a strictly better (score,
    -index), and every unselected token is worse than every selected one.
    Catches ascending order, ties won by the higher index, and dropped tokens."""
    G, D, N = 32, 64, 8 * 32 + 40
    K, V = ki.kv_stream(71, 1, 2, N, D)
    q = ki.queries(71, 1, 1, 2, D)[:, 0]
    for h in range(2):                              # tokens 3 and 5: equal top scores (a tie)
        K[0, h, 3] = K[0, h, 5] = ki.round_bf16(4.0 * q[0, h])
    c = _cache_from_tokens(fmt, G, K, V)
    k = 17
    idx, sc = oracle.topk(c, mode, q, k)
    for h in range(2):
        allsc = oracle.all_scores(c, mode, q, 0, h)
        sel = idx[0, h]
        for pos, t in enumerate(sel):
            better = np.sum((allsc > allsc[t]) | ((allsc == allsc[t]) & (np.arange(c.Lq) < t)))
            assert better == pos
            assert sc[0, h, pos] == allsc[t]
    # the planted tie: equal scores, both selected, token 3 first
    for h in range(2):
        allsc = oracle.all_scores(c, mode, q, 0, h)
        assert allsc[3] == allsc[5]
        sel = idx[0, h].tolist()
        assert 3 in sel and 5 in sel and sel.index(3) < sel.index(5)


def test_topk_padding_and_mha():
    """k > Lq pads with index -1 and score -inf.  Under MHA the summed query is
    that head's query."""
    G, D = 32, 64
    K, V = ki.kv_stream(81, 1, 1, 2 * G + 3, D)
    c = _cache_from_tokens("int2", G, K, V)
    assert c.Lq == 32
    q = ki.queries(81, 1, 1, 1, D)[:, 0]
    idx, sc = oracle.topk(c, "int2", q, 40)
    assert sorted(idx[0, 0, :32].tolist()) == list(range(32))
    assert np.all(idx[0, 0, 32:] == -1) and np.all(np.isneginf(sc[0, 0, 32:]))
    qs = oracle.summed_query(q[0], 0, 1)
    assert np.array_equal(qs, q[0, 0])


def test_topk_agrees_with_exact_logit_topk_up_to_near_ties():
    """The top-k set from the canonical score equals the top-k of the exact fp64
    logits, except for tokens within the score error of the k-th value."""
    G, D, N = 32, 128, 40 * 32 + 33
    K, V = ki.kv_stream(91, 1, 1, N, D)
    c = _cache_from_tokens("int2", G, K, V)
    q = ki.queries(91, 1, 1, 1, D)[:, 0]
    k = 64
    idx, _ = oracle.topk(c, "int2", q, k)
    ex = _exact_logit(c, "int2", q[0, 0].astype(F32), 0, 0)
    order = np.argsort(-ex, kind="stable")
    kth = ex[order[k - 1]]
    diff = set(order[:k].tolist()) ^ set(idx[0, 0].tolist())
    for t in diff:
        assert abs(ex[t] - kth) <= 1e-4 * (1 + abs(kth))


# ------------------------------------------------------------------------------------
# Fetch of the selected 16-bit KV
# ------------------------------------------------------------------------------------


def test_gather_selected_rows_decode_to_their_source():
    """Every store value encodes its own (b, h, t, d) and (+0.5 for V), so each
    fetched row is decoded back to its source instead of being compared with
    another indexing expression.  Padding (-1) and an index past the end give
    zero rows.  Catches a wrong head or batch stride, K/V swapped, or padding
    that wraps around to the last row."""
    B, H, N, D, k = 2, 3, 11, 4, 5
    b_, h_, t_, d_ = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), np.arange(D), indexing="ij")
    full_k = (1000.0 * b_ + 100.0 * h_ + t_ + d_ / 8).astype(np.float64)
    full_v = full_k + 0.5
    g = ki.rng(41)
    sel = np.stack([np.stack([g.choice(N, k, replace=False) for _ in range(H)]) for _ in range(B)]).astype(np.int32)
    sel[0, 1, 3] = -1
    sel[1, 2, 0] = N
    sk, sv = oracle.gather_selected(full_k, full_v, sel)
    for b in range(B):
        for h in range(H):
            for j in range(k):
                t = int(sel[b, h, j])
                if not 0 <= t < N:
                    assert not sk[b, h, j].any() and not sv[b, h, j].any()
                    continue
                row = sk[b, h, j]
                assert int(row[0]) // 1000 == b and (int(row[0]) // 100) % 10 == h and int(row[0]) % 100 == t
                np.testing.assert_array_equal(row - row[0], np.arange(D) / 8)
                np.testing.assert_array_equal(sv[b, h, j], row + 0.5)


def test_gather_every_token_makes_attention_exact():
    """Selecting every quantized token and fetching its 16-bit rows from the
    original K/V turns the low-bit cache back into the original: attention then
    equals dense fp64 SDPA over the original bf16 K/V (SpeCache page, Approach:
    the selected pairs attend with their 16-bit values).  Catches a fetch that
    picks the wrong rows as well as an attention that ignores the overrides."""
    B, Hkv, Hq, D, G = 1, 2, 4, 64, 32
    N = 3 * G + 9
    K, V = ki.kv_stream(43, B, Hkv, N, D)
    c = _cache_from_tokens("int2", G, K, V)
    q = ki.queries(43, B, 1, Hq, D)
    sel = np.tile(np.arange(c.Lq, dtype=np.int32)[::-1], (B, Hkv, 1))
    sk, sv = oracle.gather_selected(K, V, sel)
    out, _ = oracle.attend(c, "int2", q, None, None, sel, sk, sv)
    for h in range(Hq):
        kvh = h // (Hq // Hkv)
        ref = _sdpa_reference(q[0, 0, h], K[0, kvh], V[0, kvh], np.ones(N, bool), 1 / math.sqrt(D))
        np.testing.assert_allclose(out[0, 0, h], ref, rtol=1e-10, atol=1e-12)
