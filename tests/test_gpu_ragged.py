"""Ragged batches: every sequence of one cache keeps its own lengths.

Each sequence of a ragged device cache must hold the same bytes as a
batch-of-one oracle cache that appended the same tokens, and attention and
top-k over the whole ragged batch must match the oracle run per sequence
(SpeCache page, "Key results": batched decoding of 36 sequences at 32K, whose
real lengths differ).  Appends mix sequences that flush, that only fill their
residual buffer, and that append nothing, in one call.
"""
import numpy as np
import pytest
import torch

import kvq_inputs as ki
import oracle
import quantized_kv_speculative_gb300 as kvq
from quantized_kv_speculative_gb300 import _build

from kvq_testlib import assert_attention_close, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kvq.load_library()


def _compare_sequence(gc, b, oc):
    """Bit-exact codes, scales, zeros and residual tokens of sequence b."""
    Hkv, G = gc.desc.num_kv_heads, gc.desc.group_size
    lq, r, start = gc.seq_state(b)
    assert (lq, r) == (oc.Lq, oc.r), f"sequence {b}: state {(lq, r)} vs oracle {(oc.Lq, oc.r)}"
    kp, vp = oc.packed_k_planes(), oc.packed_v_planes()
    rk, rv = gc.residual()
    ork, orv = oc.residual()
    for h in range(Hkv):
        u = b * Hkv + h
        for i, plane in enumerate(kp):
            np.testing.assert_array_equal(gc.k_plane(i)[u, :lq].cpu().numpy(), plane[0, h], err_msg=f"seq {b} k{i}")
        for i, plane in enumerate(vp):
            np.testing.assert_array_equal(gc.v_plane(i)[u, :lq // 32].cpu().numpy(), plane[0, h],
                                          err_msg=f"seq {b} v{i}")
        ksz = gc.k_scale_zero()[u, :lq // G].cpu().numpy()
        np.testing.assert_array_equal(ksz[:, 0].view(np.uint32), oc.k_scale[0, h, :lq // G].view(np.uint32))
        np.testing.assert_array_equal(ksz[:, 1].view(np.uint32), oc.k_zero[0, h, :lq // G].view(np.uint32))
        vsz = gc.v_scale_zero()[u, :lq].cpu().numpy()
        np.testing.assert_array_equal(vsz[:, 0].view(np.uint32), oc.v_scale[0, h, :lq].view(np.uint32))
        np.testing.assert_array_equal(vsz[:, 1].view(np.uint32), oc.v_zero[0, h, :lq].view(np.uint32))
        slots = [(start + i) % (2 * G) for i in range(r)]
        if slots:
            np.testing.assert_array_equal(ki.bf16_tensor_to_f32(rk[u, slots]), ork[0, h])
            np.testing.assert_array_equal(ki.bf16_tensor_to_f32(rv[u, slots]), orv[0, h])


def _build_ragged(fmt, B, Hkv, D, G, steps, seed):
    """A ragged device cache and one oracle cache per sequence, fed the same
    tokens: `steps` is a list of per-sequence counts, one list per append."""
    totals = [sum(st[b] for st in steps) for b in range(B)]
    cap = (max(totals) // G + 1) * G
    K, V = ki.kv_stream(seed, B, Hkv, max(totals), D)
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, fmt, cap, ragged=True)
    ocs = [oracle.OracleCache(1, Hkv, D, G, fmt, cap) for _ in range(B)]
    pos = [0] * B
    for counts in steps:
        n_max = max(max(counts), 1)
        kn = np.zeros((B, Hkv, n_max, D), np.float32)
        vn = np.zeros((B, Hkv, n_max, D), np.float32)
        for b in range(B):
            n = counts[b]
            kn[b, :, :n] = K[b, :, pos[b]:pos[b] + n]
            vn[b, :, :n] = V[b, :, pos[b]:pos[b] + n]
            if n:
                ocs[b].append(K[b:b + 1, :, pos[b]:pos[b] + n], V[b:b + 1, :, pos[b]:pos[b] + n])
            pos[b] += n
        kvq.kvq_quantize_append_ragged(gc, dev(kn), dev(vn), counts)
    torch.cuda.synchronize()
    return gc, ocs


def _selected(ocs, Hkv, k, g):
    """Per-sequence selected indices below each sequence's own Lq (-1 pads)."""
    B = len(ocs)
    sel = np.full((B, Hkv, k), -1, np.int32)
    for b, oc in enumerate(ocs):
        for h in range(Hkv):
            m = min(k - 1, oc.Lq)
            if m:
                sel[b, h, :m] = g.choice(oc.Lq, m, replace=False)
    return sel


@pytest.mark.parametrize("fmt,modes,D,G", [("int2", ("int2",), 128, 32), ("hier8", ("int8", "int4", "int4mid"), 128, 64),
                                           ("int1", ("int1", "int1c"), 64, 32)])
def test_ragged_append_attend_topk_match_oracle_per_sequence(fmt, modes, D, G):
    B, Hkv, Hq, gamma, P, k = 5, 2, 8, 2, 2, 9
    steps = [[700, 130, 2 * G + 5, 33, 0],          # bulk prefill: flushes, residual only, nothing
             [1, 0, 2 * G - 7, 5, 2 * G],           # mixed: one sequence fills exactly 2G and flushes
             [G + 3, 1, 1, 0, 3]]
    gc, ocs = _build_ragged(fmt, B, Hkv, D, G, steps, seed=41)
    for b in range(B):
        _compare_sequence(gc, b, ocs[b])
    assert gc.quantized_len == max(oc.Lq for oc in ocs) and gc.residual_len == max(oc.r for oc in ocs)
    q = ki.queries(41, B, gamma, Hq, D)
    pk, pv = ki.pending(41, B, Hkv, P, D)
    g = ki.rng(41, 3)
    sel = _selected(ocs, Hkv, k, g)
    sk, sv = ki.normal_bf16(g, (B, Hkv, k, D)), ki.normal_bf16(g, (B, Hkv, k, D))
    for mode in modes:
        out, lse = kvq.kvq_attend(gc, mode, dev(q), dev(pk), dev(pv), torch.from_numpy(sel).cuda(), dev(sk), dev(sv))
        torch.cuda.synchronize()
        for b in range(B):
            ref, ref_lse = oracle.attend(ocs[b], mode, q[b:b + 1], pk[b:b + 1], pv[b:b + 1], sel[b:b + 1],
                                         sk[b:b + 1], sv[b:b + 1])
            assert_attention_close(out[b:b + 1], lse[b:b + 1], ref, ref_lse, what=f"{mode} sequence {b}")
        if mode != "int8":
            idx, sc = kvq.kvq_topk(gc, mode, dev(q[:, 1]), k)
            # the fused call: attention plus the next step's top-k from one key read
            out2, _, idx2, sc2 = kvq.kvq_attend_topk(gc, mode, dev(q), k, 1, dev(pk), dev(pv),
                                                     torch.from_numpy(sel).cuda(), dev(sk), dev(sv))
            torch.cuda.synchronize()
            np.testing.assert_array_equal(idx2.cpu().numpy(), idx.cpu().numpy())
            np.testing.assert_array_equal(sc2.cpu().numpy().view(np.uint32), sc.cpu().numpy().view(np.uint32))
            for b in range(B):
                ridx, rsc = oracle.topk(ocs[b], mode, q[b:b + 1, 1], k)
                np.testing.assert_array_equal(idx[b:b + 1].cpu().numpy(), ridx, err_msg=f"{mode} top-k seq {b}")
                np.testing.assert_array_equal(sc[b:b + 1].cpu().numpy().view(np.uint32), rsc.view(np.uint32))
                ref, ref_lse = oracle.attend(ocs[b], mode, q[b:b + 1], pk[b:b + 1], pv[b:b + 1], sel[b:b + 1],
                                             sk[b:b + 1], sv[b:b + 1])
                assert_attention_close(out2[b:b + 1], None, ref, ref_lse, what=f"fused {mode} sequence {b}")


def test_ragged_specache_batch_36():
    """The SpeCache batch shape with unequal lengths in one call: 36
    sequences, 32 query / 8 KV heads, D = 128, G = 32, INT2, two query tokens,
    64 selected tokens; lengths drawn between 300 and 6000 tokens.  Codes of
    every sequence, attention and top-k of six of them are checked."""
    B, Hkv, Hq, D, G, gamma, k = 36, 8, 32, 128, 32, 2, 64
    g = ki.rng(77, 1)
    lengths = g.integers(300, 6000, size=B)
    steps = [[int(x) - 3 for x in lengths], [1, 2, 3] * (B // 3)]
    gc, ocs = _build_ragged("int2", B, Hkv, D, G, steps, seed=77)
    check = [0, 7, 13, 21, 30, 35]
    for b in check:
        _compare_sequence(gc, b, ocs[b])
    q = ki.queries(77, B, gamma, Hq, D)
    pk, pv = ki.pending(77, B, Hkv, gamma, D)
    sel = _selected(ocs, Hkv, k, g)
    sk, sv = ki.normal_bf16(g, (B, Hkv, k, D)), ki.normal_bf16(g, (B, Hkv, k, D))
    out, lse = kvq.kvq_attend(gc, "int2", dev(q), dev(pk), dev(pv), torch.from_numpy(sel).cuda(), dev(sk), dev(sv))
    idx, sc = kvq.kvq_topk(gc, "int2", dev(q[:, 1]), k)
    torch.cuda.synchronize()
    for b in check:
        ref, ref_lse = oracle.attend(ocs[b], "int2", q[b:b + 1], pk[b:b + 1], pv[b:b + 1], sel[b:b + 1],
                                     sk[b:b + 1], sv[b:b + 1])
        assert_attention_close(out[b:b + 1], lse[b:b + 1], ref, ref_lse, what=f"sequence {b}")
        ridx, rsc = oracle.topk(ocs[b], "int2", q[b:b + 1, 1], k)
        np.testing.assert_array_equal(idx[b:b + 1].cpu().numpy(), ridx)
        np.testing.assert_array_equal(sc[b:b + 1].cpu().numpy().view(np.uint32), rsc.view(np.uint32))
