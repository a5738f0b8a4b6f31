"""Host-side checks of the C ABI (no GPU needed).

The library loads.  It exports every function declared in include/kvq.h.  The
ctypes structs match the C layout (checked against a small program compiled
with gcc).  And argument errors come back before any CUDA call is made.
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import quantized_kv_speculative_gb300 as kvq
from quantized_kv_speculative_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_build.LIB) and shutil.which(_build.nvcc()) is None and not os.path.exists(_build.nvcc()):
        pytest.skip("nvcc not available to build the library")
    _build.build()
    return kvq.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_what_the_binding_lists():
    assert _declared_functions() == sorted(kvq.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)", out))
    for name in _declared_functions():
        assert name in exported, f"{name} not exported"
        assert getattr(lib, name) is not None


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "kvq.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(kvq_cache_desc), sizeof(kvq_cache),
         offsetof(kvq_cache, base), offsetof(kvq_cache, off_k_plane), offsetof(kvq_cache, quantized_len),
         offsetof(kvq_cache, residual_start), offsetof(kvq_cache, magic), sizeof(kvq_attend_plan_info),
         offsetof(kvq_attend_plan_info, chunk_tokens), offsetof(kvq_attend_plan_info, cluster),
         offsetof(kvq_cache, seqs), sizeof(kvq_seq_state), offsetof(kvq_seq_state, residual_start));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    C = kvq.KvqCache
    P = kvq.KvqAttendPlanInfo
    S = kvq.KvqSeqState
    assert vals == [ctypes.sizeof(kvq.KvqCacheDesc), ctypes.sizeof(C), C.base.offset, C.off_k_plane.offset,
                    C.quantized_len.offset, C.residual_start.offset, C.magic.offset, ctypes.sizeof(P),
                    P.chunk_tokens.offset, P.cluster.offset, C.seqs.offset, ctypes.sizeof(S),
                    S.residual_start.offset]


def _desc(**kw):
    d = dict(batch=1, num_kv_heads=4, head_dim=64, group_size=32, format=8, reserved0=0, capacity_tokens=512)
    d.update(kw)
    return kvq.KvqCacheDesc(**d)


def test_cache_bytes_and_validation(lib):
    good = _desc()
    n = lib.kvq_cache_bytes(ctypes.byref(good))
    # 2 key + 2 value nibble planes, key/value scale+zero, 2 residual buffers, the
    # per-head flush counters (each region 256-aligned)
    U, C, D, G = 4, 512, 64, 32
    expect = (4 * U * C * D // 2 + U * (C // G) * 2 * D * 4 + U * C * 2 * (D // G) * 4 + 2 * U * 2 * G * D * 2
              + 256)
    assert n == expect
    for bad in [_desc(head_dim=96), _desc(group_size=16), _desc(group_size=128), _desc(format=4),
                _desc(capacity_tokens=100), _desc(batch=0), _desc(reserved0=1)]:
        assert lib.kvq_cache_bytes(ctypes.byref(bad)) == 0


def _host_cache(lib, **kw):
    """A cache struct laid out over a fake, never-dereferenced device address."""
    d = _desc(**kw)
    c = kvq.KvqCache()
    n = lib.kvq_cache_bytes(ctypes.byref(d))
    assert lib.kvq_cache_init(ctypes.byref(c), ctypes.byref(d), 1 << 40, n) == 0
    return c, n


def test_cache_init_layout_and_alignment(lib):
    c, n = _host_cache(lib)
    offs = [c.off_k_plane[0], c.off_k_plane[1], c.off_v_plane[0], c.off_v_plane[1], c.off_k_sz, c.off_v_sz,
            c.off_res_k, c.off_res_v]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs) and offs[-1] < n
    assert (c.quantized_len, c.residual_len, c.residual_start) == (0, 0, 0)
    d = _desc()
    c2 = kvq.KvqCache()
    assert lib.kvq_cache_init(ctypes.byref(c2), ctypes.byref(d), (1 << 40) + 16, n) == 1   # misaligned
    assert lib.kvq_cache_init(ctypes.byref(c2), ctypes.byref(d), 1 << 40, n - 1) == 1      # too small


def test_argument_errors_return_before_any_launch(lib):
    c, _ = _host_cache(lib)
    fake = ctypes.c_void_p(1 << 41)
    # append: negative count, misaligned input, capacity exceeded (checked before any write)
    assert lib.kvq_quantize_append(ctypes.byref(c), fake, fake, -1, None) == 1
    assert lib.kvq_quantize_append(ctypes.byref(c), ctypes.c_void_p((1 << 41) + 2), fake, 4, None) == 1
    assert lib.kvq_quantize_append(ctypes.byref(c), fake, fake, 512 + 64, None) == 3
    assert (c.quantized_len, c.residual_len) == (0, 0)
    assert lib.kvq_quantize_append(ctypes.byref(c), fake, fake, 0, None) == 0
    uninit = kvq.KvqCache()
    assert lib.kvq_quantize_append(ctypes.byref(uninit), fake, fake, 1, None) == 7
    ws_n = lib.kvq_workspace_bytes(ctypes.byref(c), 4, 1, 0)
    assert ws_n > 0
    assert lib.kvq_workspace_bytes(ctypes.byref(c), 4, 9, 0) == 0           # 9 rows per KV head
    assert lib.kvq_workspace_bytes(ctypes.byref(c), 6, 1, 0) == 0           # Hq % Hkv != 0
    # attend: mode/format mismatch, too many rows, missing workspace, pending < gamma
    args = dict(q=fake, pk=None, pv=None, P=0, si=None, sk=None, sv=None, k=0, out=fake, lse=None, ws=fake, wsn=ws_n)

    def attend(mode, Hq=4, gamma=1, **over):
        a = dict(args, **over)
        return lib.kvq_attend(ctypes.byref(c), mode, a["q"], Hq, gamma, a["pk"], a["pv"], a["P"], a["si"], a["sk"],
                              a["sv"], a["k"], 0.0, a["out"], a["lse"], a["ws"], a["wsn"], None)
    assert attend(2) == 2 and attend(3) == 2
    assert attend(0, Hq=36, gamma=1) == 2                                     # 9 rows per KV head
    assert attend(0, wsn=16) == 4 and attend(0, ws=None) == 4
    assert attend(0, gamma=2, P=1, pk=fake, pv=fake) == 1
    assert attend(0, k=3) == 1                                                # sel pointers missing
    assert attend(0, q=ctypes.c_void_p((1 << 41) + 8)) == 1
    # top-k: INT8 has no low-bit keys; k out of range
    assert lib.kvq_topk(ctypes.byref(c), 0, fake, 4, 8, fake, None, fake, ws_n, None) == 2
    assert lib.kvq_topk(ctypes.byref(c), 1, fake, 4, 0, fake, None, fake, ws_n, None) == 1
    assert lib.kvq_topk(ctypes.byref(c), 1, fake, 4, 2000, fake, None, fake, ws_n, None) == 1
    assert lib.kvq_selftest_bounded_wait(None, 0, 100, None) == 4
    assert lib.kvq_status_string(6) == b"device wait timed out"


def test_host_state_machine_without_launch(lib):
    """The closed form of the 2G buffer, checked on the host counters alone:
    an append that flushes nothing launches only the residual copy, so it is
    checked through the capacity errors that precede any launch.  After N
    tokens, Lq = G*(floor(N/G) - 1) must fit the capacity; one token more than
    that closed form allows fails with KVQ_ERR_CAPACITY and leaves the state
    unchanged."""
    G, C = 32, 128
    c, _ = _host_cache(lib, capacity_tokens=C)
    fake = ctypes.c_void_p(1 << 41)
    # the largest N whose closed-form Lq fits the capacity: Lq = C when floor(N/G) - 1 = C/G
    n_max = (C // G + 2) * G - 1
    assert lib.kvq_quantize_append(ctypes.byref(c), fake, fake, n_max + 1, None) == 3
    assert (c.quantized_len, c.residual_len) == (0, 0)


def test_gather_and_plan_argument_errors_need_no_gpu(lib):
    """The fetch and the plan query refuse bad arguments before touching the
    device: null pointers, head_dim outside {64, 128}, top_k outside
    [1, 1024], misaligned rows, and an uninitialized cache."""
    fake = ctypes.c_void_p(1 << 41)
    odd = ctypes.c_void_p((1 << 41) + 8)

    def gather(fk=fake, fv=fake, n=64, B=1, H=2, D=128, si=fake, k=4, sk=fake, sv=fake):
        return lib.kvq_gather_selected(fk, fv, n, B, H, D, si, k, sk, sv, None)
    assert gather(fk=None) == 1 and gather(si=None) == 1 and gather(sv=None) == 1
    assert gather(D=96) == 1 and gather(k=0) == 1 and gather(k=1025) == 1
    assert gather(B=0) == 1 and gather(n=0) == 1
    assert gather(fk=odd) == 1 and gather(sk=odd) == 1
    info = kvq.KvqAttendPlanInfo()
    uninit = kvq.KvqCache()
    assert lib.kvq_attend_plan(ctypes.byref(uninit), 0, 4, 1, 0, 0, ctypes.byref(info)) == 7
    c, _ = _host_cache(lib)
    assert lib.kvq_attend_plan(ctypes.byref(c), 0, 4, 1, 0, 0, None) == 1
    assert lib.kvq_attend_plan(ctypes.byref(c), 2, 4, 1, 0, 0, ctypes.byref(info)) == 2    # INT2 on hier8
    assert lib.kvq_attend_plan(ctypes.byref(c), 0, 36, 1, 0, 0, ctypes.byref(info)) == 2   # 9 rows per KV head
    assert lib.kvq_attend_plan(ctypes.byref(c), 0, 6, 1, 0, 0, ctypes.byref(info)) == 1    # Hq % Hkv != 0


def test_static_scratch_argument_errors_need_no_gpu(lib):
    """The allocation-free attention entry point checks every argument with
    kvq_attend's own status codes before it touches the shared array: an
    uninitialized cache (7), mode vs format (2), more than 8 rows per KV head
    (2), a null or misaligned query and too few pending tokens (1).  None of
    these needs a GPU, because nothing is enqueued."""
    c, _ = _host_cache(lib)
    fake = ctypes.c_void_p(1 << 41)

    def static(cache, mode, q=fake, Hq=4, gamma=1, pk=None, pv=None, P=0, out=fake):
        return lib.kvq_attend_static_scratch(ctypes.byref(cache), mode, q, Hq, gamma, pk, pv, P, None, None, None,
                                             0, 0.0, out, None, None)
    assert static(kvq.KvqCache(), 0) == 7
    assert static(c, 2) == 2
    assert static(c, 0, Hq=36) == 2
    assert static(c, 0, q=None) == 1
    assert static(c, 0, q=ctypes.c_void_p((1 << 41) + 8)) == 1
    assert static(c, 0, out=None) == 1
    assert static(c, 0, gamma=2, pk=fake, pv=fake, P=1) == 1


def test_ragged_state_machine_without_launch(lib):
    """A ragged cache: set-up refuses a wrong count or a non-empty cache; the
    per-sequence appends check every sequence's capacity before anything is
    enqueued and leave all states unchanged on refusal; counts outside
    [0, n_max] are refused.  Appends of zero tokens change nothing and need
    no GPU."""
    c, _ = _host_cache(lib, batch=3, capacity_tokens=128)
    seqs = (kvq.KvqSeqState * 3)()
    assert lib.kvq_cache_set_ragged(ctypes.byref(c), seqs, 2) == 1
    assert lib.kvq_cache_set_ragged(ctypes.byref(kvq.KvqCache()), seqs, 3) == 7
    assert lib.kvq_cache_set_ragged(ctypes.byref(c), seqs, 3) == 0
    assert ctypes.cast(c.seqs, ctypes.c_void_p).value == ctypes.cast(seqs, ctypes.c_void_p).value
    fake = ctypes.c_void_p(1 << 41)
    counts = (ctypes.c_int32 * 3)(5, 0, (128 // 32 + 2) * 32)      # the last one overflows its capacity
    assert lib.kvq_quantize_append_ragged(ctypes.byref(c), fake, fake, 192, counts, None) == 3
    assert [(s.quantized_len, s.residual_len) for s in seqs] == [(0, 0)] * 3
    counts = (ctypes.c_int32 * 3)(5, 7, 3)
    assert lib.kvq_quantize_append_ragged(ctypes.byref(c), fake, fake, 6, counts, None) == 1   # 7 > n_max
    assert lib.kvq_quantize_append_ragged(ctypes.byref(c), fake, fake, 8, None, None) == 1
    zeros = (ctypes.c_int32 * 3)(0, 0, 0)
    assert lib.kvq_quantize_append_ragged(ctypes.byref(c), fake, fake, 8, zeros, None) == 0
    u, _ = _host_cache(lib, batch=3)
    assert lib.kvq_quantize_append_ragged(ctypes.byref(u), fake, fake, 8, zeros, None) == 1   # not ragged
    big, _ = _host_cache(lib, batch=65)
    many = (kvq.KvqSeqState * 65)()
    assert lib.kvq_cache_set_ragged(ctypes.byref(big), many, 65) == 2


def test_attend_topk_argument_errors_need_no_gpu(lib):
    """The fused attention + top-k call refuses, before any launch: an
    uninitialized cache (7), a mode without low-bit keys to rank (INT8: 2), a
    score row outside [0, gamma) or a top-k count outside [1, 1024] or a null
    index buffer (1), and a workspace without room for the per-token scores
    (4)."""
    c, _ = _host_cache(lib)
    fake = ctypes.c_void_p(1 << 41)
    ws_n = lib.kvq_workspace_bytes(ctypes.byref(c), 4, 2, 16)
    ws_att = lib.kvq_workspace_bytes(ctypes.byref(c), 4, 2, 0)
    assert ws_n > ws_att > 0

    def call(cache, mode, gamma=2, row=1, k=16, idx=fake, wsn=ws_n, P=2):
        return lib.kvq_attend_topk(ctypes.byref(cache), mode, fake, 4, gamma, fake, fake, P, None, None, None, 0,
                                   0.0, fake, None, row, k, idx, None, fake, wsn, None)
    assert call(kvq.KvqCache(), 1) == 7
    assert call(c, 0) == 2
    assert call(c, 1, row=2) == 1 and call(c, 1, row=-1) == 1
    assert call(c, 1, k=0) == 1 and call(c, 1, k=1025) == 1
    assert call(c, 1, idx=None) == 1
    assert call(c, 1, wsn=ws_att) == 4
