"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses.  Where the oracle cannot redo a whole workload in seconds, the
device computes everything and the oracle recomputes sampled KV heads from the
same inputs.  Codes, scales, top-k indices and scores must match bit for bit;
attention must be within 2e-3*max|ref| + 1e-3 over the sampled heads."""
import numpy as np
import pytest
import torch

import kvq_inputs as ki
import oracle
import quantized_kv_speculative_gb300 as kvq
from quantized_kv_speculative_gb300 import _build

from kvq_testlib import assert_attention_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kvq.load_library()


def _sampled_oracle(K_dev, V_dev, units, fmt, G, cap, n_tokens):
    """Oracle cache for the sampled (b, kv head) units, built from the device
    inputs (downloaded bf16): one oracle 'batch' row with the units as heads."""
    ks = np.stack([ki.bf16_tensor_to_f32(K_dev[b, h, :n_tokens]) for (b, h) in units])[None]
    vs = np.stack([ki.bf16_tensor_to_f32(V_dev[b, h, :n_tokens]) for (b, h) in units])[None]
    oc = oracle.OracleCache(1, len(units), K_dev.shape[-1], G, fmt, cap)
    oc.append(ks, vs)
    return oc


def _compare_units(gc, oc, units):
    L, G = oc.Lq, oc.G
    Hkv = gc.desc.num_kv_heads
    for j, (b, h) in enumerate(units):
        u = b * Hkv + h
        for i, plane in enumerate(oc.packed_k_planes()):
            np.testing.assert_array_equal(gc.k_plane(i)[u, :L].cpu().numpy(), plane[0, j])
        for i, plane in enumerate(oc.packed_v_planes()):
            np.testing.assert_array_equal(gc.v_plane(i)[u, :L // 32].cpu().numpy(), plane[0, j])
        ksz = gc.k_scale_zero()[u, :L // G].cpu().numpy()
        np.testing.assert_array_equal(ksz[:, 0].view(np.uint32), oc.k_scale[0, j, :L // G].view(np.uint32))
        np.testing.assert_array_equal(ksz[:, 1].view(np.uint32), oc.k_zero[0, j, :L // G].view(np.uint32))
        vsz = gc.v_scale_zero()[u, :L].cpu().numpy()
        np.testing.assert_array_equal(vsz[:, 0].view(np.uint32), oc.v_scale[0, j, :L].view(np.uint32))
        np.testing.assert_array_equal(vsz[:, 1].view(np.uint32), oc.v_zero[0, j, :L].view(np.uint32))


def _attend_units(out_dev, lse_dev, oc, mode, q, units, hg, pk=None, pv=None, sel=None, sk=None, sv=None):
    """Oracle attention for the sampled units vs the device output's rows."""
    qh = [x for (b, h) in units for x in range(h * hg, (h + 1) * hg)]
    bsel = [b for (b, h) in units for _ in range(hg)]
    qs = np.stack([q[b, :, x] for b, x in zip(bsel, qh)], axis=1)[None]     # [1, gamma, U*hg, D]
    take = lambda a: None if a is None else np.stack([a[b, h] for (b, h) in units])[None]
    ref, ref_lse = oracle.attend(oc, mode, qs, take(pk), take(pv), take(sel), take(sk), take(sv))
    got = torch.stack([out_dev[b, :, x] for b, x in zip(bsel, qh)], dim=1)[None]
    gl = torch.stack([lse_dev[b, :, x] for b, x in zip(bsel, qh)], dim=1)[None]
    assert_attention_close(got, gl, ref, ref_lse, what="sampled units")


def test_llama7b_layer_verify_8k_all_heads():
    """One Llama-2-7B-shaped layer: 32 heads, D = 128, G = 128, 8192 quantized
    + 252 residual tokens, INT8 verify with gamma = 8 causal pending tokens,
    INT4 top-64, then an 8-token append with a flush: every head checked."""
    B, Hkv, Hq, D, G, gamma, P = 1, 32, 32, 128, 128, 8, 8
    N = 8192 + 252
    K, V = ki.kv_stream(0, B, Hkv, N + 8, D)
    q = ki.queries(0, B, gamma, Hq, D)
    pk, pv = ki.pending(0, B, Hkv, P, D)
    up = lambda x: ki.f32_to_bf16_tensor(x, "cuda")
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, "hier8", 8192 + 2 * G)
    kvq.kvq_quantize_append(gc, up(K[:, :, :N]), up(V[:, :, :N]))
    oc = oracle.OracleCache(B, Hkv, D, G, "hier8", 8192 + 2 * G)
    oc.append(K[:, :, :N], V[:, :, :N])
    out, lse = kvq.kvq_attend(gc, "int8", up(q), up(pk), up(pv))
    ref, ref_lse = oracle.attend(oc, "int8", q, pk, pv)
    assert_attention_close(out, lse, ref, ref_lse, what="llama7b layer verify 8k")
    idx, sc = kvq.kvq_topk(gc, "int4", up(q[:, -1]), 64)
    ridx, rsc = oracle.topk(oc, "int4", q[:, -1], 64)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), rsc.view(np.uint32))
    kvq.kvq_quantize_append(gc, up(K[:, :, N:]), up(V[:, :, N:]))
    oc.append(K[:, :, N:], V[:, :, N:])
    torch.cuda.synchronize()
    from kvq_testlib import compare_cache
    compare_cache(gc, oc)


@pytest.mark.parametrize("fmt", ["int2", "int1"])
def test_specache_b36_32k_sampled(fmt):
    """SpeCache shape: batch 36, 32 query / 8 KV heads, D = 128, G = 32, 32768
    quantized + 32 residual tokens, gamma = 2, top-64 from the speculative
    token, then attention with those tokens at 16 bits.  The device runs the
    full batch; the oracle checks 4 sampled (b, kv head) units."""
    B, Hkv, Hq, D, G, gamma, P, k = 36, 8, 32, 128, 32, 2, 2, 64
    N = 32768 + 32
    K_dev, V_dev = ki.kv_stream_torch(41, B, Hkv, N, D)
    q = ki.queries(41, B, gamma, Hq, D)
    pk, pv = ki.pending(41, B, Hkv, P, D)
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, fmt, 32768 + 2 * G)
    kvq.kvq_quantize_append(gc, K_dev, V_dev)
    up = lambda x: ki.f32_to_bf16_tensor(x, "cuda")
    idx, sc = kvq.kvq_topk(gc, fmt, up(q[:, 1]), k)
    idx_np = idx.cpu().numpy()
    sel_k = torch.gather(K_dev, 2, idx.long().clamp_min(0)[..., None].expand(-1, -1, -1, D)).contiguous()
    sel_v = torch.gather(V_dev, 2, idx.long().clamp_min(0)[..., None].expand(-1, -1, -1, D)).contiguous()
    out, lse = kvq.kvq_attend(gc, fmt, up(q), up(pk), up(pv), idx, sel_k, sel_v)
    torch.cuda.synchronize()
    units = [(0, 0), (17, 3), (35, 7), (8, 5)]
    oc = _sampled_oracle(K_dev, V_dev, units, fmt, G, 32768 + 2 * G, N)
    _compare_units(gc, oc, units)
    hg = Hq // Hkv
    qh = [x for (b, h) in units for x in range(h * hg, (h + 1) * hg)]
    qspec = np.stack([q[b, 1, x] for (b, h) in units for x in range(h * hg, (h + 1) * hg)])[None]
    ridx, rsc = oracle.topk(oc, fmt, qspec, k)
    for j, (b, h) in enumerate(units):
        np.testing.assert_array_equal(idx_np[b, h], ridx[0, j])
        np.testing.assert_array_equal(sc[b, h].cpu().numpy().view(np.uint32), rsc[0, j].view(np.uint32))
    sk = ki.bf16_tensor_to_f32(sel_k)
    sv = ki.bf16_tensor_to_f32(sel_v)
    _attend_units(out, lse, oc, fmt, q, units, hg, pk, pv, idx_np, sk, sv)


@pytest.mark.parametrize("mode,gamma,P", [("int8", 6, 6), ("int4", 1, 3)])
def test_long_context_128k_sampled(mode, gamma, P):
    """One layer of the 128K stress case: 131072 quantized + 253 residual
    tokens, 32 heads, G = 128.  INT8 verify (gamma = 6) and an INT4 draft step.
    The oracle checks 2 sampled heads."""
    B, Hkv, Hq, D, G = 1, 32, 32, 128, 128
    N = 131072 + 253
    K_dev, V_dev = ki.kv_stream_torch(51, B, Hkv, N, D)
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, "hier8", 131072 + 2 * G)
    kvq.kvq_quantize_append(gc, K_dev, V_dev)
    q = ki.queries(51, B, gamma, Hq, D)
    pk, pv = ki.pending(51, B, Hkv, P, D)
    up = lambda x: ki.f32_to_bf16_tensor(x, "cuda")
    out, lse = kvq.kvq_attend(gc, mode, up(q), up(pk), up(pv))
    torch.cuda.synchronize()
    units = [(0, 0), (0, 31)]
    oc = _sampled_oracle(K_dev, V_dev, units, "hier8", G, 131072 + 2 * G, N)
    _compare_units(gc, oc, units)
    _attend_units(out, lse, oc, mode, q, units, 1, pk, pv)


def test_sweep_256k_int4_sampled():
    """The longest sweep point: 262144 quantized + 128 residual tokens, INT4
    draft attention (gamma = 1), one sampled head checked."""
    B, Hkv, Hq, D, G = 1, 32, 32, 128, 128
    N = 262144 + 128                 # closed form: Lq = 128*(floor(N/128) - 1) = 262144, r = 128
    K_dev, V_dev = ki.kv_stream_torch(61, B, Hkv, N, D)
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, "hier8", 262144 + 2 * G)
    kvq.kvq_quantize_append(gc, K_dev, V_dev)
    assert gc.quantized_len == 262144
    q = ki.queries(61, B, 1, Hq, D)
    up = lambda x: ki.f32_to_bf16_tensor(x, "cuda")
    out, lse = kvq.kvq_attend(gc, "int4", up(q))
    torch.cuda.synchronize()
    units = [(0, 13)]
    oc = _sampled_oracle(K_dev, V_dev, units, "hier8", G, 262144 + 2 * G, N)
    _attend_units(out, lse, oc, "int4", q, units, 1)
