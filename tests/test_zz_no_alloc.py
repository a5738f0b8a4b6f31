"""The allocation-free attention entry point, kvq_attend_static_scratch.

It serves callers that cannot allocate device memory (for example a decode
loop that must not allocate after start-up).  Its workspace is a fixed array
inside the library.  Through the C ABI, its output must equal kvq_attend's
with a caller workspace on two calls in a row: the second call reuses the
array the first one left behind.  Both run the same deterministic kernel with
the same launch plan, so the outputs and LSEs must be identical bytes, which
is stricter than the attention tolerance the other tests use.  A call with a
bad argument between the two must be refused with kvq_attend's status code
and leave the next call's result unchanged.  This file is collected last, so
a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import kvq_inputs as ki
import quantized_kv_speculative_gb300 as kvq
from quantized_kv_speculative_gb300 import _build


pytestmark = pytest.mark.gpu


def _call_static(lib, cache, mode, q, pk, pv, sel, sk, sv, out, lse):
    ptr = lambda t: None if t is None else t.data_ptr()
    top_k = 0 if sel is None else sel.shape[2]
    n_pend = 0 if pk is None else pk.shape[2]
    return lib.kvq_attend_static_scratch(ctypes.byref(cache.struct), kvq.MODES[mode], ptr(q), q.shape[2],
                                         q.shape[1], ptr(pk), ptr(pv), n_pend, ptr(sel), ptr(sk), ptr(sv),
                                         top_k, 0.0, ptr(out), ptr(lse),
                                         torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("mode,B,Hkv,Hq,D,G,N,gamma,P,top_k", [
    ("int8", 1, 32, 32, 128, 128, 8192 + 252, 8, 8, 0),      # Llama-2-7B layer verify shape
    ("int4", 1, 4, 4, 64, 32, 544, 1, 1, 0),                # tiny case
    ("int2", 3, 2, 8, 128, 32, 2100, 2, 2, 16),             # GQA, selected 16-bit tokens
])
def test_static_scratch_matches_workspace_version(mode, B, Hkv, Hq, D, G, N, gamma, P, top_k):
    _build.build()
    lib = kvq.load_library()
    fmt = kvq.MODE_FORMAT[mode]
    K, V = ki.kv_stream(31, B, Hkv, N, D)
    up = lambda x: ki.f32_to_bf16_tensor(x, "cuda")
    cache = kvq.QuantizedKVCache(B, Hkv, D, G, fmt, (N // G + 1) * G)
    kvq.kvq_quantize_append(cache, up(K), up(V))
    pk, pv = (up(x) for x in ki.pending(31, B, Hkv, P, D))
    sel = sk = sv = None
    if top_k:
        g = ki.rng(31, 3)
        s = np.stack([np.stack([g.choice(cache.quantized_len, top_k, replace=False) for _ in range(Hkv)])
                      for _ in range(B)]).astype(np.int32)
        sel = torch.from_numpy(s).cuda()
        sk, sv = up(ki.normal_bf16(g, (B, Hkv, top_k, D))), up(ki.normal_bf16(g, (B, Hkv, top_k, D)))
    q = up(ki.queries(31, B, gamma, Hq, D))
    ref_out, ref_lse = kvq.kvq_attend(cache, mode, q, pk, pv, sel, sk, sv)
    torch.cuda.synchronize()
    ref = ref_out.view(torch.int16).cpu().numpy()
    ref_l = ref_lse.view(torch.int32).cpu().numpy()
    for call in range(2):
        out = torch.empty_like(q)
        lse = torch.empty((B, gamma, Hq), dtype=torch.float32, device="cuda")
        assert _call_static(lib, cache, mode, q, pk, pv, sel, sk, sv, out, lse) == 0, f"call {call}"
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy(), ref, err_msg=f"call {call}: out")
        np.testing.assert_array_equal(lse.view(torch.int32).cpu().numpy(), ref_l, err_msg=f"call {call}: lse")
        if call == 0:
            # a refused call (null query) between the two must change nothing
            bad = lib.kvq_attend_static_scratch(ctypes.byref(cache.struct), kvq.MODES[mode], None, Hq, gamma,
                                                None, None, 0, None, None, None, 0, 0.0, out.data_ptr(), None,
                                                torch.cuda.current_stream().cuda_stream)
            assert bad == 1, "a null query must be refused with KVQ_ERR_INVALID_ARG"


def test_static_scratch_rejects_oversized_workspace():
    """A cache whose attention workspace exceeds the fixed 16 MiB array gets
    KVQ_ERR_WORKSPACE, and nothing is enqueued."""
    lib = kvq.load_library()
    big = kvq.QuantizedKVCache(64, 32, 128, 128, "hier8", 1024)   # 2048 heads: workspace > 16 MiB
    assert kvq.kvq_workspace_bytes(big, 32, 8, 0) > (16 << 20)
    q = torch.zeros((64, 8, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((64, 8, 32), dtype=torch.float32, device="cuda")
    assert _call_static(lib, big, "int8", q, None, None, None, None, None, out, lse) == kvq.KVQError(4).status
