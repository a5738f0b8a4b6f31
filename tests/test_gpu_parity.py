"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

* Codes, scales, zero points and the residual buffer match bit for bit.
* Top-k indices and scores match bit for bit.
* Attention matches within |err| <= 2e-3 * max|ref| + 1e-3 over a call's output,
  and log-sum-exp matches within 1e-3 + 1e-4 |lse|.
Sizes span several tiles, warps and splits, plus a ragged tail.
"""
import numpy as np
import pytest
import torch

import kvq_inputs as ki
import oracle
import quantized_kv_speculative_gb300 as kvq
from quantized_kv_speculative_gb300 import _build

from kvq_testlib import assert_attention_close, build_pair, compare_cache, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kvq.load_library()
    torch.cuda.init()


# ------------------------------------------------------------------------------------
# quantize + append
# ------------------------------------------------------------------------------------

CACHE_SHAPES = [
    ("hier8", 64, 32), ("hier8", 128, 128), ("hier8", 128, 64), ("hier8", 64, 64),
    ("int2", 128, 32), ("int2", 64, 64), ("int2", 128, 128), ("int1", 128, 32), ("int1", 64, 32),
]


@pytest.mark.parametrize("fmt,D,G", CACHE_SHAPES)
def test_quantize_append_bit_exact(fmt, D, G):
    """Bulk prefill, then single tokens and chunks that cross flushes, in the
    same call pattern as a decode loop.  The state after every call matches the
    oracle's token-by-token buffer."""
    B, Hkv = 2, 3
    N = 5 * G + 7 + 1 + 3 + 2 * G + 1 + G + 5
    K, V = ki.kv_stream(100 + D + G, B, Hkv, N, D)
    chunks = [5 * G + 7, 1, 3, 2 * G + 1, G, 5]
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


def test_quantize_degenerate_groups_and_signed_zero():
    """Constant groups (scale 0), -0.0 values and extreme bf16 magnitudes."""
    B, Hkv, D, G = 1, 2, 64, 32
    N = 3 * G + 4
    K = np.zeros((B, Hkv, N, D), np.float32)
    V = np.zeros((B, Hkv, N, D), np.float32)
    K[0, 0] = -0.0
    K[0, 1, :, :8] = 3.5
    K[0, 1, :, 8:] = ki.normal_bf16(ki.rng(5), (N, D - 8))
    V[0, 0, :, :32] = -0.0
    V[0, 1] = ki.round_bf16(ki.rng(6).standard_normal((N, D)).astype(np.float32) * np.float32(1e30))
    for fmt in ("hier8", "int2", "int1"):
        gc, oc = build_pair(fmt, B, Hkv, D, G, 4 * G, K, V, [N])
        compare_cache(gc, oc)


# ------------------------------------------------------------------------------------
# attention
# ------------------------------------------------------------------------------------

ATTN_CASES = [
    # mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, needles
    ("int8", 1, 4, 4, 64, 32, 544, 1, 1, 0, False),         # tiny-d64-g32 shape
    ("int4", 1, 4, 4, 64, 32, 544, 1, 1, 0, False),
    ("int8", 2, 2, 8, 128, 128, 1150, 2, 3, 0, False),      # GQA 4:1, 8 rows, ragged residual
    ("int4", 2, 2, 8, 128, 128, 1150, 2, 3, 0, True),
    ("int8", 1, 3, 3, 128, 128, 4000, 8, 8, 0, True),       # gamma = 8 verify, MHA
    ("int4", 1, 3, 3, 128, 64, 2500, 1, 0, 0, False),       # no pending tokens
    ("int8", 1, 2, 6, 128, 64, 3100, 2, 2, 0, False),       # 6 rows
    ("int2", 3, 2, 8, 128, 32, 2100, 2, 2, 16, False),      # SpeCache shape, selected tokens
    ("int1", 3, 2, 8, 128, 32, 2100, 2, 2, 16, True),
    ("int2", 1, 2, 2, 64, 32, 900, 1, 1, 5, False),
    ("int1", 1, 2, 4, 64, 64, 1000, 2, 2, 0, False),
    ("int4", 2, 2, 8, 128, 32, 1700, 2, 2, 0, False),       # hierarchical format with G = 32
    ("int4mid", 1, 4, 4, 64, 32, 544, 1, 1, 0, False),      # the midpoint reading of the draft code
    ("int4mid", 1, 3, 3, 128, 128, 4000, 1, 1, 0, True),    # one row, needles
    ("int4mid", 2, 2, 8, 128, 64, 1700, 2, 2, 7, False),    # eight rows, selected tokens
    ("int1c", 3, 2, 8, 128, 32, 2100, 2, 2, 16, True),      # the centred 1-bit reading, SpeCache shape
    ("int1c", 1, 2, 4, 64, 64, 1000, 2, 2, 0, False),
    ("int1c", 1, 3, 3, 128, 32, 1500, 1, 1, 0, False),      # one row
    # one weight n-tile with two to four rows (rows past R up to a power of two stay zero)
    ("int8", 1, 2, 4, 128, 64, 1300, 1, 1, 0, False),       # 2 rows
    ("int2", 1, 1, 3, 128, 32, 1100, 1, 1, 4, False),       # 3 rows (padded to 4), selected tokens
    ("int4", 2, 2, 4, 128, 128, 1400, 2, 2, 0, False),      # 4 rows
    ("int1", 1, 2, 2, 128, 32, 900, 2, 2, 0, True),         # 2 rows, needles
]


def _attn_case(mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, needles, seed=0):
    fmt = kvq.MODE_FORMAT[mode]
    K, V = ki.kv_stream(seed + 7, B, Hkv, N, D)
    q = ki.queries(seed + 7, B, gamma, Hq, D)
    if needles:
        K, _ = ki.plant_needles(K, q, seed + 7, limit=N - 2 * G)
    cap = (N // G + 1) * G
    gc, oc = build_pair(fmt, B, Hkv, D, G, cap, K, V, [N - 3, 1, 2])
    pk = pv = None
    if P:
        pk, pv = ki.pending(seed + 7, B, Hkv, P, D)
    sel = sk = sv = None
    if top_k:
        g = ki.rng(seed + 7, 9)
        sel = np.stack([np.stack([g.choice(oc.Lq, top_k, replace=False) for _ in range(Hkv)]) for _ in range(B)])
        sel = sel.astype(np.int32)
        sel[0, 0, -1] = -1                       # padding entry
        sk = ki.normal_bf16(g, (B, Hkv, top_k, D))
        sv = ki.normal_bf16(g, (B, Hkv, top_k, D))
    return gc, oc, q, pk, pv, sel, sk, sv


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-Hkv{c[2]}-Hq{c[3]}-D{c[4]}-G{c[5]}-N{c[6]}-g{c[7]}-P{c[8]}-k{c[9]}{'-needle' if c[10] else ''}")
def test_attend_matches_oracle(case):
    mode = case[0]
    gc, oc, q, pk, pv, sel, sk, sv = _attn_case(*case)
    ref_out, ref_lse = oracle.attend(oc, mode, q, pk, pv, sel, sk, sv)
    out, lse = kvq.kvq_attend(gc, mode, dev(q), None if pk is None else dev(pk), None if pv is None else dev(pv),
                              None if sel is None else torch.from_numpy(sel).cuda(),
                              None if sk is None else dev(sk), None if sv is None else dev(sv))
    torch.cuda.synchronize()
    assert_attention_close(out, lse, ref_out, ref_lse, what=str(case))


# Enough (b, kvh) units that the plan stays within 16 CTAs per unit, and few
# enough that the clusters fit the device at once (on a 152-SM GB300 with two
# CTAs per SM, 28 clusters of 10 CTAs) and that the splits do not fill the
# first wave on their own, so the launch takes the cluster combine.
CLUSTER_CASES = [
    ("int8", 1, 16, 16, 128, 128, 1300, 8, 8, 0, True),     # verify, eight rows, 16 KV heads
    ("int4", 1, 32, 32, 128, 128, 1500, 1, 1, 0, False),    # draft, one row
    ("int2", 2, 8, 32, 128, 32, 1500, 2, 2, 16, False),     # SpeCache shape, selected tokens
    ("int1", 2, 8, 16, 64, 32, 1000, 2, 2, 0, False),
    ("int8", 2, 2, 8, 128, 128, 1150, 2, 3, 0, False),      # few units, ragged residual
    ("int4mid", 1, 32, 32, 128, 128, 1500, 1, 1, 0, False),
    ("int1c", 2, 8, 32, 128, 32, 1500, 2, 2, 16, False),
]


@pytest.mark.parametrize("case", CLUSTER_CASES, ids=lambda c: f"{c[0]}-N{c[6]}-g{c[7]}-k{c[9]}")
def test_attend_cluster_and_ticket_combines(case, monkeypatch):
    """The same call through both combines: one thread-block cluster per
    (b, kvh) merging in shared memory, and (KVQ_ATTEND_CLUSTERS=0) partials in
    the workspace merged by the last CTA.  The plan reports which one ran; both
    match the oracle."""
    mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, needles = case
    gc, oc, q, pk, pv, sel, sk, sv = _attn_case(*case)
    ref_out, ref_lse = oracle.attend(oc, mode, q, pk, pv, sel, sk, sv)
    args = (dev(q), None if pk is None else dev(pk), None if pv is None else dev(pv),
            None if sel is None else torch.from_numpy(sel).cuda(), None if sk is None else dev(sk),
            None if sv is None else dev(sv))
    monkeypatch.delenv("KVQ_ATTEND_CLUSTERS", raising=False)
    plan = kvq.kvq_attend_plan(gc, mode, Hq, gamma, P, top_k)
    assert plan["cluster"] and plan["quant_splits"] + plan["tail_splits"] <= 16, plan
    out_c, lse_c = kvq.kvq_attend(gc, mode, *args)
    monkeypatch.setenv("KVQ_ATTEND_CLUSTERS", "0")
    plan0 = kvq.kvq_attend_plan(gc, mode, Hq, gamma, P, top_k)
    assert not plan0["cluster"]
    assert (plan0["quant_splits"], plan0["tail_splits"], plan0["chunk_tokens"]) == \
        (plan["quant_splits"], plan["tail_splits"], plan["chunk_tokens"])
    out_t, lse_t = kvq.kvq_attend(gc, mode, *args)
    torch.cuda.synchronize()
    assert_attention_close(out_c, lse_c, ref_out, ref_lse, what=f"cluster {case}")
    assert_attention_close(out_t, lse_t, ref_out, ref_lse, what=f"ticket {case}")


@pytest.mark.parametrize("mode,Hq,gamma,P", [("int4", 1, 1, 1), ("int8", 4, 1, 2), ("int8", 4, 2, 2)])
def test_attend_many_splits_ticket_combine(mode, Hq, gamma, P):
    """One (b, kv head) over a long cache: the plan takes far more splits than
    the combine prefetches per lane (eight per lane, with one to eight lanes
    per output item), so the ticket combine's prefetched and streamed partials
    both take part.  One, four and eight rows."""
    B, Hkv, D, G, N = 1, 1, 128, 128, 20000
    case = (mode, B, Hkv, Hq, D, G, N, gamma, P, 0, False)
    gc, oc, q, pk, pv, _, _, _ = _attn_case(*case)
    plan = kvq.kvq_attend_plan(gc, mode, Hq, gamma, P, 0)
    assert not plan["cluster"] and plan["quant_splits"] + plan["tail_splits"] > 32, plan
    ref_out, ref_lse = oracle.attend(oc, mode, q, pk, pv)
    out, lse = kvq.kvq_attend(gc, mode, dev(q), dev(pk), dev(pv))
    torch.cuda.synchronize()
    assert_attention_close(out, lse, ref_out, ref_lse, what=f"{mode} rows {Hq * gamma}")


def test_attend_deterministic_and_split_independent():
    """Two calls give identical bytes.  The result does not depend on the
    workspace's history, because the ticket counters reset themselves."""
    case = ("int8", 2, 2, 8, 128, 128, 1150, 2, 3, 0, False)
    gc, oc, q, pk, pv, _, _, _ = _attn_case(*case)
    ws = kvq.make_workspace(gc, 8, 2, 0)
    outs = []
    for _ in range(3):
        o, l = kvq.kvq_attend(gc, "int8", dev(q), dev(pk), dev(pv), workspace=ws)
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(l, outs[0][1])
    assert kvq.kvq_workspace_status(ws) == 0


def test_selection_calls_deterministic():
    """Top-k and attention with selected 16-bit tokens over many CTAs: repeated
    calls give identical bytes (no call depends on thread timing)."""
    B, Hkv, Hq, D, G, N, k = 8, 8, 32, 128, 32, 8192 + 40, 64
    K, V = ki.kv_stream_torch(13, B, Hkv, N, D)
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, "int2", 8192 + 2 * G)
    kvq.kvq_quantize_append(gc, K, V)
    q = dev(ki.queries(13, B, 2, Hq, D))
    pk, pv = (dev(x) for x in ki.pending(13, B, Hkv, 2, D))
    ws = kvq.make_workspace(gc, Hq, 2, k)
    idx0, sc0 = kvq.kvq_topk(gc, "int2", q[:, 1].contiguous(), k, workspace=ws)
    gi = idx0.long().clamp_min(0)[..., None].expand(-1, -1, -1, D)
    sk, sv = torch.gather(K, 2, gi).contiguous(), torch.gather(V, 2, gi).contiguous()
    outs = []
    for _ in range(5):
        idx, sc = kvq.kvq_topk(gc, "int2", q[:, 1].contiguous(), k, workspace=ws)
        assert torch.equal(idx, idx0) and torch.equal(sc.view(torch.int32), sc0.view(torch.int32))
        o, l = kvq.kvq_attend(gc, "int2", q, pk, pv, idx0, sk, sv, workspace=ws)
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(l.view(torch.int32), outs[0][1].view(torch.int32))
    assert kvq.kvq_workspace_status(ws) == 0


def test_attend_edge_cases():
    """An empty cache gives out 0 and lse -inf.  Residual only (Lq = 0);
    pending == gamma; selected entries all padding; k > Lq."""
    D, G, Hkv = 64, 32, 2
    q = ki.queries(3, 1, 2, 2, D)
    gc = kvq.QuantizedKVCache(1, Hkv, D, G, "hier8", 256)
    out, lse = kvq.kvq_attend(gc, "int8", dev(q))
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0) and torch.all(torch.isneginf(lse))
    # residual only
    K, V = ki.kv_stream(4, 1, Hkv, 50, D)
    gc, oc = build_pair("hier8", 1, Hkv, D, G, 256, K, V, [50])
    assert oc.Lq == 0
    pk, pv = ki.pending(4, 1, Hkv, 2, D)
    ref = oracle.attend(oc, "int4", q, pk, pv)
    out, lse = kvq.kvq_attend(gc, "int4", dev(q), dev(pk), dev(pv))
    assert_attention_close(out, lse, *ref, what="residual only")
    # exactly one quantized group, all selected entries padding
    K, V = ki.kv_stream(5, 1, Hkv, 2 * G + 1, D)
    gc, oc = build_pair("int2", 1, Hkv, D, G, 256, K, V, [2 * G + 1])
    sel = -np.ones((1, Hkv, 3), np.int32)
    sk = ki.normal_bf16(ki.rng(1), (1, Hkv, 3, D))
    ref = oracle.attend(oc, "int2", q, pk, pv, sel, sk, sk)
    out, lse = kvq.kvq_attend(gc, "int2", dev(q), dev(pk), dev(pv), torch.from_numpy(sel).cuda(), dev(sk), dev(sk))
    assert_attention_close(out, lse, *ref, what="padding selection")


def test_bounded_wait_reports_timeout_without_hanging():
    """A kernel that waits on an mbarrier nothing arrives at gives up after its
    limit, records KVQ_ERR_DEVICE_TIMEOUT, and leaves the context usable."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    kvq.kvq_selftest_bounded_wait(ws, 100000)
    assert kvq.kvq_workspace_status(ws) == 6
    assert kvq.kvq_workspace_status(ws) == 0      # read clears it
    x = torch.ones(16, device="cuda")
    assert float(x.sum()) == 16.0


# ------------------------------------------------------------------------------------
# top-k
# ------------------------------------------------------------------------------------

TOPK_CASES = [
    # mode, B, Hkv, Hq, D, G, N, k
    ("int4", 1, 2, 2, 128, 128, 3000, 64),
    ("int4", 2, 2, 8, 64, 32, 1500, 17),
    ("int2", 3, 2, 8, 128, 32, 2100, 64),
    ("int2", 1, 1, 4, 128, 32, 20000, 100),     # several splits, ragged last chunk
    ("int1", 3, 2, 8, 128, 32, 2100, 64),
    ("int1", 1, 2, 2, 64, 64, 700, 1),
    ("int2", 1, 2, 2, 64, 32, 130, 80),         # k > Lq: padded with -1
    ("int4", 1, 2, 4, 128, 128, 6000, 128),     # the largest k of the warp-sort selection
    ("int4", 1, 2, 4, 128, 128, 6000, 300),     # k above it: radix selection on small chunks
    ("int2", 1, 1, 4, 128, 32, 30000, 1024),    # the largest k: 4 splits x 1024 candidates to merge
    ("int4mid", 1, 2, 2, 128, 128, 3000, 64),   # the midpoint reading: zero points moved by 8 steps
    ("int4mid", 2, 2, 8, 64, 32, 1500, 17),
    ("int1c", 3, 2, 8, 128, 32, 2100, 64),      # the centred 1-bit reading: zero point z + s/4, scale s/2
    ("int1c", 1, 2, 2, 64, 64, 700, 5),
]


@pytest.mark.parametrize("case", TOPK_CASES, ids=lambda c: "-".join(map(str, c)))
def test_topk_matches_oracle(case):
    mode, B, Hkv, Hq, D, G, N, k = case
    fmt = kvq.MODE_FORMAT[mode]
    K, V = ki.kv_stream(11, B, Hkv, N, D)
    K[:, :, 7] = K[:, :, 3]                       # a planted score tie
    gc, oc = build_pair(fmt, B, Hkv, D, G, (N // G + 1) * G, K, V, [N])
    qspec = ki.queries(11, B, 1, Hq, D)[:, 0]
    ref_idx, ref_sc = oracle.topk(oc, mode, qspec, k)
    idx, sc = kvq.kvq_topk(gc, mode, dev(qspec), k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), ref_sc.view(np.uint32))


@pytest.mark.parametrize("pattern,mode,G,N,k", [
    ("zero_query", "int4", 128, 9000, 64),     # every score equal: every key passes the lower bound
    ("zero_query", "int2", 32, 700, 17),
    ("two_keys", "int4", 128, 9000, 64),       # half of the tokens tie at the top score
    ("two_keys", "int2", 32, 3000, 100),
    ("two_keys", "int1", 64, 2000, 128),
])
def test_topk_heavy_ties(pattern, mode, G, N, k):
    """Massive score ties: the selection's lower bound admits far more
    candidates than k (a whole chunk, or half of it), so the sorted and the
    radix fallbacks run; ties still go to the lowest index, as in the oracle."""
    B, Hkv, Hq, D = 1, 2, 4, 128
    fmt = kvq.MODE_FORMAT[mode]
    K, V = ki.kv_stream(13, B, Hkv, N, D)
    if pattern == "two_keys":
        K[:, :, 2::2] = K[:, :, 0:1]
        K[:, :, 3::2] = K[:, :, 1:2]
    gc, oc = build_pair(fmt, B, Hkv, D, G, (N // G + 1) * G, K, V, [N])
    qspec = ki.queries(13, B, 1, Hq, D)[:, 0]
    if pattern == "zero_query":
        qspec = np.zeros_like(qspec)
    ref_idx, ref_sc = oracle.topk(oc, mode, qspec, k)
    idx, sc = kvq.kvq_topk(gc, mode, dev(qspec), k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), ref_sc.view(np.uint32))


def test_topk_then_attend_specache_step():
    """One SpeCache step: top-k from the speculative token (query row 1), then
    attention that uses those tokens at 16 bits.  Both match the oracle."""
    B, Hkv, Hq, D, G, N, k = 2, 2, 8, 128, 32, 2100, 32
    K, V = ki.kv_stream(12, B, Hkv, N, D)
    gc, oc = build_pair("int2", B, Hkv, D, G, (N // G + 1) * G, K, V, [N])
    q = ki.queries(12, B, 2, Hq, D)
    idx, _ = kvq.kvq_topk(gc, "int2", dev(q[:, 1]), k)
    ref_idx, _ = oracle.topk(oc, "int2", q[:, 1], k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    # the 16-bit rows come from the full store in pinned host memory
    sk, sv = oracle.gather_selected(K, V, ref_idx)
    hk, hv = (torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in (K, V))
    gk, gv = kvq.kvq_gather_selected(hk, hv, idx)
    torch.cuda.synchronize()
    assert torch.equal(gk.cpu(), torch.from_numpy(sk).to(torch.bfloat16))
    assert torch.equal(gv.cpu(), torch.from_numpy(sv).to(torch.bfloat16))
    pk, pv = ki.pending(12, B, Hkv, 2, D)
    ref = oracle.attend(oc, "int2", q, pk, pv, ref_idx, sk, sv)
    out, lse = kvq.kvq_attend(gc, "int2", dev(q), dev(pk), dev(pv), idx, gk, gv)
    assert_attention_close(out, lse, *ref, what="specache step")


@pytest.mark.parametrize("B,Hkv,N,D,k,where", [(3, 2, 2100, 128, 16, "host"), (2, 4, 700, 64, 33, "host"),
                                              (36, 8, 2048, 128, 64, "host"), (2, 2, 1500, 128, 7, "device")])
def test_gather_selected_bit_exact(B, Hkv, N, D, k, where):
    """The fetch of the selected 16-bit rows is a bit-exact copy, from pinned
    host memory or from device memory, with -1 padding and an index past the
    end giving zero rows; sizes cover several warps, a ragged last sweep and
    the SpeCache batch (36 x 8 heads x 64)."""
    g = ki.rng(51, B * 1000 + k)
    K = ki.normal_bf16(g, (B, Hkv, N, D))
    V = ki.normal_bf16(g, (B, Hkv, N, D))
    sel = np.stack([np.stack([g.choice(N, k, replace=False) for _ in range(Hkv)]) for _ in range(B)]).astype(np.int32)
    sel[0, 0, -1] = -1
    sel[-1, -1, 0] = N
    ref_k, ref_v = oracle.gather_selected(K, V, sel)
    tk, tv = (torch.from_numpy(x).to(torch.bfloat16) for x in (K, V))
    if where == "host":
        tk, tv = tk.pin_memory(), tv.pin_memory()
    else:
        tk, tv = tk.cuda(), tv.cuda()
    sk, sv = kvq.kvq_gather_selected(tk, tv, torch.from_numpy(sel).cuda())
    torch.cuda.synchronize()
    assert torch.equal(sk.cpu(), torch.from_numpy(ref_k).to(torch.bfloat16))
    assert torch.equal(sv.cpu(), torch.from_numpy(ref_v).to(torch.bfloat16))


def test_gather_selected_rejects_pageable_memory():
    """A store in pageable host memory is refused before any launch."""
    lib = kvq.load_library()
    K = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16)          # pageable
    sel = torch.zeros((1, 1, 4), dtype=torch.int32, device="cuda")
    out = torch.empty((1, 1, 4, 128), dtype=torch.bfloat16, device="cuda")
    st = lib.kvq_gather_selected(K.data_ptr(), K.data_ptr(), 64, 1, 1, 128, sel.data_ptr(), 4, out.data_ptr(),
                                 out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert kvq.STATUS[st] == "KVQ_ERR_INVALID_ARG"
    with pytest.raises(ValueError):
        kvq.kvq_gather_selected(K, K, sel)


# ------------------------------------------------------------------------------------
# attention fused with the next step's top-k
# ------------------------------------------------------------------------------------

FUSED_CASES = [
    # mode, B, Hkv, Hq, D, G, N, gamma, P, top_k (selected), next_k, score_row
    ("int2", 3, 2, 8, 128, 32, 2100, 2, 2, 16, 64, 1),      # SpeCache step: the speculative token scores
    ("int2", 3, 2, 8, 128, 32, 2100, 2, 2, 16, 64, 0),      # the output token scores (non-speculative fetch)
    ("int1", 2, 2, 8, 64, 32, 1500, 2, 2, 0, 17, 1),
    ("int4", 1, 3, 3, 128, 128, 4000, 1, 1, 0, 64, 0),      # MHA draft shape, one row
    ("int4mid", 2, 2, 8, 128, 64, 1700, 2, 2, 7, 33, 1),
    ("int1c", 3, 2, 8, 128, 32, 2100, 2, 2, 16, 64, 1),
    ("int2", 1, 1, 4, 128, 32, 20000, 2, 2, 0, 100, 1),     # several top-k splits
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: "-".join(map(str, c)))
def test_attend_topk_matches_oracle_and_topk(case):
    """kvq_attend_topk: the attention output matches the oracle, and the next
    step's top-k is identical (indices and score bits) to the oracle's and to
    kvq_topk on the same query row."""
    mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, next_k, row = case
    gc, oc, q, pk, pv, sel, sk, sv = _attn_case(mode, B, Hkv, Hq, D, G, N, gamma, P, top_k, False, seed=3)
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


def test_flush_counters_start_from_garbage():
    """The flush kernel's arrival counters are zeroed before the cache's first
    flush even when earlier appends flushed nothing: the cache memory is
    filled with 0xFF first, then tokens that only fill the residual buffer,
    then tokens that flush.  Bytes must match the oracle."""
    B, Hkv, D, G = 2, 3, 64, 32
    K, V = ki.kv_stream(19, B, Hkv, 4 * G + 9, D)
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, "int2", 6 * G)
    gc.storage.fill_(255)
    oc = oracle.OracleCache(B, Hkv, D, G, "int2", 6 * G)
    pos = 0
    for n in (5, G, 3 * G + 4):
        kvq.kvq_quantize_append(gc, dev(K[:, :, pos:pos + n]), dev(V[:, :, pos:pos + n]))
        oc.append(K[:, :, pos:pos + n], V[:, :, pos:pos + n])
        pos += n
    torch.cuda.synchronize()
    compare_cache(gc, oc)
