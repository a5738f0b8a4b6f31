"""GPU parity on seeded random shapes: attention, top-k and the two fused,
through the C ABI, against the CPU oracle, over combinations that the
hand-picked cases do not enumerate (every read mode, head size, group size,
query rows per KV head, draft length, pending and selected tokens, context
length).

The shapes are drawn once from a fixed seed, so a run always tests the same
cases; the tolerances are those of the hand-picked parity tests.
"""
import numpy as np
import pytest
import torch

import kvq_inputs as ki
import oracle
import quantized_kv_speculative_gb300 as kvq
from quantized_kv_speculative_gb300 import _build

from kvq_testlib import assert_attention_close, build_pair, compare_cache, dev
from test_gpu_parity import _attn_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kvq.load_library()
    torch.cuda.init()


def _groups(D):
    return (32, 64) if D == 64 else (32, 64, 128)


def _attn_shapes(n, seed=2024):
    """(mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, needles) with at most
    eight query rows per KV head and pending tokens either none or at least
    gamma."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        mode = str(g.choice(["int8", "int4", "int4mid", "int2", "int1", "int1c"]))
        D = int(g.choice([64, 128]))
        G = int(g.choice(_groups(D)))
        HG = int(g.choice([1, 2, 4]))
        gammas = [x for x in (1, 2, 3, 4, 6, 8) if x * HG <= 8]
        gamma = int(g.choice(gammas))
        Hkv = int(g.integers(1, 4))
        B = int(g.integers(1, 3))
        N = int(g.integers(2 * G + 8, 3200))
        P = 0 if g.random() < 0.25 else gamma + int(g.integers(0, 3))
        top_k = int(g.choice([0, 0, 8, 16]))
        needles = bool(g.random() < 0.3)
        out.append((mode, B, Hkv, Hkv * HG, D, G, N, gamma, P, top_k, needles))
    return out


def _topk_shapes(n, seed=4048):
    """(mode, B, Hkv, Hq, D, G, N, k)."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        mode = str(g.choice(["int4", "int4mid", "int2", "int1", "int1c"]))
        D = int(g.choice([64, 128]))
        G = int(g.choice(_groups(D)))
        HG = int(g.choice([1, 2, 4]))
        Hkv = int(g.integers(1, 4))
        B = int(g.integers(1, 3))
        N = int(g.integers(G + 1, 12000))
        k = int(g.choice([1, 5, 17, 64, 100, 128, 200]))
        out.append((mode, B, Hkv, Hkv * HG, D, G, N, k))
    return out


def _fused_shapes(n, seed=8096):
    """(mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, next_k, row) for the
    attention fused with the next step's top-k (the top-k read modes only)."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        mode = str(g.choice(["int4", "int4mid", "int2", "int1", "int1c"]))
        D = int(g.choice([64, 128]))
        G = int(g.choice(_groups(D)))
        HG = int(g.choice([1, 2, 4]))
        gamma = int(g.choice([x for x in (1, 2, 3, 4, 6, 8) if x * HG <= 8]))
        Hkv = int(g.integers(1, 4))
        B = int(g.integers(1, 3))
        N = int(g.integers(2 * G + 8, 5000))
        P = gamma + int(g.integers(0, 2))
        top_k = int(g.choice([0, 8]))
        next_k = int(g.choice([1, 16, 64, 128]))
        row = int(g.integers(0, gamma))
        out.append((mode, B, Hkv, Hkv * HG, D, G, N, gamma, P, top_k, next_k, row))
    return out


def _append_patterns(n, seed=1234):
    """(fmt, B, Hkv, D, G, chunk sizes): appends of 1 token up to several
    groups at a time, crossing zero, one or many flushes per call."""
    g = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        fmt = ("hier8", "int2", "int1")[len(out) % 3]   # every format in turn
        D = int(g.choice([64, 128]))
        G = int(g.choice(_groups(D)))
        B = int(g.integers(1, 3))
        Hkv = int(g.integers(1, 4))
        chunks = [int(x) for x in g.choice([1, 2, 3, G - 1, G, G + 1, 3 * G + 5, 7 * G], size=int(g.integers(4, 9)))]
        out.append((fmt, B, Hkv, D, G, tuple(chunks)))
    return out


RANDOM_APPEND = _append_patterns(9)
RANDOM_ATTN = _attn_shapes(24)
RANDOM_TOPK = _topk_shapes(16)
RANDOM_FUSED = _fused_shapes(12)


@pytest.mark.parametrize("case", RANDOM_ATTN, ids=lambda c: "-".join(map(str, c)))
def test_attend_random_shapes(case):
    mode = case[0]
    gc, oc, q, pk, pv, sel, sk, sv = _attn_case(*case, seed=31)
    ref_out, ref_lse = oracle.attend(oc, mode, q, pk, pv, sel, sk, sv)
    out, lse = kvq.kvq_attend(gc, mode, dev(q), None if pk is None else dev(pk), None if pv is None else dev(pv),
                              None if sel is None else torch.from_numpy(sel).cuda(),
                              None if sk is None else dev(sk), None if sv is None else dev(sv))
    torch.cuda.synchronize()
    assert_attention_close(out, lse, ref_out, ref_lse, what=str(case))


@pytest.mark.parametrize("case", RANDOM_TOPK, ids=lambda c: "-".join(map(str, c)))
def test_topk_random_shapes(case):
    mode, B, Hkv, Hq, D, G, N, k = case
    fmt = kvq.MODE_FORMAT[mode]
    K, V = ki.kv_stream(41, B, Hkv, N, D)
    gc, oc = build_pair(fmt, B, Hkv, D, G, (N // G + 1) * G, K, V, [N])
    qspec = ki.queries(41, B, 1, Hq, D)[:, 0]
    ref_idx, ref_sc = oracle.topk(oc, mode, qspec, k)
    idx, sc = kvq.kvq_topk(gc, mode, dev(qspec), k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), ref_sc.view(np.uint32))


@pytest.mark.parametrize("case", RANDOM_FUSED, ids=lambda c: "-".join(map(str, c)))
def test_attend_topk_random_shapes(case):
    """The fused call: attention against the oracle, the next step's top-k
    bit-exact against the oracle and against kvq_topk on the same row."""
    mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, next_k, row = case
    gc, oc, q, pk, pv, sel, sk, sv = _attn_case(mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, False, seed=53)
    t = lambda x: None if x is None else dev(x)
    out, lse, idx, sc = kvq.kvq_attend_topk(gc, mode, dev(q), next_k, row, t(pk), t(pv),
                                           None if sel is None else torch.from_numpy(sel).cuda(), t(sk), t(sv))
    idx2, sc2 = kvq.kvq_topk(gc, mode, dev(q[:, row]), next_k)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attend(oc, mode, q, pk, pv, sel, sk, sv)
    assert_attention_close(out, lse, ref_out, ref_lse, what=str(case))
    ridx, rsc = oracle.topk(oc, mode, q[:, row], next_k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), rsc.view(np.uint32))
    np.testing.assert_array_equal(idx.cpu().numpy(), idx2.cpu().numpy())
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), sc2.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("case", RANDOM_APPEND, ids=lambda c: "-".join(map(str, c[:5])) + "-" + ".".join(map(str, c[5])))
def test_append_random_patterns(case):
    """Codes, scales, zero points and the residual buffer stay bit-exact after
    every append of a random chunk sequence."""
    fmt, B, Hkv, D, G, chunks = case
    N = sum(chunks)
    K, V = ki.kv_stream(61, B, Hkv, N, D)
    cap = (N // G + 1) * G
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, fmt, cap)
    oc = oracle.OracleCache(B, Hkv, D, G, fmt, cap)
    pos = 0
    for n in chunks:
        kvq.kvq_quantize_append(gc, dev(K[:, :, pos:pos + n]), dev(V[:, :, pos:pos + n]))
        oc.append(K[:, :, pos:pos + n], V[:, :, pos:pos + n])
        pos += n
        torch.cuda.synchronize()
        assert (gc.quantized_len, gc.residual_len) == (oc.Lq, oc.r)
        compare_cache(gc, oc)
