"""GB300 quantized-KV speculative decode attention.

A thin ctypes binding of the CUDA library ``libkvq.so`` (C ABI in
``include/kvq.h``).  The functions keep the C names.  They only marshal
arguments: PyTorch supplies device memory and streams, and every step of the
path runs in the library's kernels.  No CPU fallback exists.  If the library
is missing, importing the binding raises.

Methods (see the header for the full contract):
  * QuantSpec (hierarchical INT8/INT4 KV cache + 2G full-precision buffer):
    ``kvq_quantize_append``, ``kvq_attend`` with modes "int8" / "int4";
  * SpeCache (1/2-bit KV copy, speculative top-k, 16-bit overrides):
    ``kvq_attend`` with modes "int2" / "int1" and ``sel_*``, ``kvq_topk``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

FORMATS = {"hier8": 8, "int2": 2, "int1": 1}
MODES = {"int8": 0, "int4": 1, "int2": 2, "int1": 3, "int4mid": 4, "int1c": 5}
MODE_FORMAT = {"int8": "hier8", "int4": "hier8", "int2": "int2", "int1": "int1", "int4mid": "hier8", "int1c": "int1"}
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_CAPACITY",
          4: "KVQ_ERR_WORKSPACE", 5: "KVQ_ERR_CUDA", 6: "KVQ_ERR_DEVICE_TIMEOUT",
          7: "KVQ_ERR_NOT_INITIALIZED"}

# Every symbol the header declares.
EXPORTED = (
    "kvq_status_string", "kvq_cache_bytes", "kvq_cache_init", "kvq_quantize_append",
    "kvq_workspace_bytes", "kvq_attend", "kvq_topk", "kvq_workspace_status",
    "kvq_selftest_bounded_wait", "kvq_attend_static_scratch", "kvq_attend_plan", "kvq_gather_selected",
    "kvq_cache_set_ragged", "kvq_quantize_append_ragged", "kvq_attend_topk",
)


class KvqCacheDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("format", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("capacity_tokens", ctypes.c_int64)]


class KvqSeqState(ctypes.Structure):
    _fields_ = [("quantized_len", ctypes.c_int64), ("residual_len", ctypes.c_int32),
                ("residual_start", ctypes.c_int32)]


class KvqCache(ctypes.Structure):
    _fields_ = [("desc", KvqCacheDesc), ("base", ctypes.c_void_p), ("bytes", ctypes.c_uint64),
                ("off_k_plane", ctypes.c_uint64 * 2), ("off_v_plane", ctypes.c_uint64 * 2),
                ("off_k_sz", ctypes.c_uint64), ("off_v_sz", ctypes.c_uint64),
                ("off_res_k", ctypes.c_uint64), ("off_res_v", ctypes.c_uint64),
                ("quantized_len", ctypes.c_int64), ("residual_len", ctypes.c_int32),
                ("residual_start", ctypes.c_int32), ("magic", ctypes.c_uint32),
                ("flags", ctypes.c_uint32), ("seqs", ctypes.POINTER(KvqSeqState))]


class KvqAttendPlanInfo(ctypes.Structure):
    _fields_ = [("quant_splits", ctypes.c_int32), ("tail_splits", ctypes.c_int32),
                ("chunk_tokens", ctypes.c_int64), ("cluster", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class KVQError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libkvq.so (built by ``_build.build()``).  Raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libkvq.so not built ({p}); run quantized_kv_speculative_gb300._build.build()")
    lib = ctypes.CDLL(p)
    vp, sz, i32, i64, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    cache_p = ctypes.POINTER(KvqCache)
    lib.kvq_status_string.argtypes = [ctypes.c_int]
    lib.kvq_status_string.restype = ctypes.c_char_p
    lib.kvq_cache_bytes.argtypes = [ctypes.POINTER(KvqCacheDesc)]
    lib.kvq_cache_bytes.restype = sz
    lib.kvq_cache_init.argtypes = [cache_p, ctypes.POINTER(KvqCacheDesc), vp, sz]
    lib.kvq_cache_init.restype = ctypes.c_int
    lib.kvq_quantize_append.argtypes = [cache_p, vp, vp, i32, vp]
    lib.kvq_quantize_append.restype = ctypes.c_int
    lib.kvq_cache_set_ragged.argtypes = [cache_p, ctypes.POINTER(KvqSeqState), i32]
    lib.kvq_cache_set_ragged.restype = ctypes.c_int
    lib.kvq_quantize_append_ragged.argtypes = [cache_p, vp, vp, i32, ctypes.POINTER(ctypes.c_int32), vp]
    lib.kvq_quantize_append_ragged.restype = ctypes.c_int
    lib.kvq_workspace_bytes.argtypes = [cache_p, i32, i32, i32]
    lib.kvq_workspace_bytes.restype = sz
    lib.kvq_attend.argtypes = [cache_p, ctypes.c_int, vp, i32, i32, vp, vp, i32, vp, vp, vp, i32, f32,
                               vp, vp, vp, sz, vp]
    lib.kvq_attend.restype = ctypes.c_int
    lib.kvq_attend_topk.argtypes = [cache_p, ctypes.c_int, vp, i32, i32, vp, vp, i32, vp, vp, vp, i32, f32,
                                    vp, vp, i32, i32, vp, vp, vp, sz, vp]
    lib.kvq_attend_topk.restype = ctypes.c_int
    lib.kvq_attend_static_scratch.argtypes = [cache_p, ctypes.c_int, vp, i32, i32, vp, vp, i32, vp, vp, vp,
                                              i32, f32, vp, vp, vp]
    lib.kvq_attend_static_scratch.restype = ctypes.c_int
    lib.kvq_attend_plan.argtypes = [cache_p, ctypes.c_int, i32, i32, i32, i32, ctypes.POINTER(KvqAttendPlanInfo)]
    lib.kvq_attend_plan.restype = ctypes.c_int
    lib.kvq_gather_selected.argtypes = [vp, vp, i64, i32, i32, i32, vp, i32, vp, vp, vp]
    lib.kvq_gather_selected.restype = ctypes.c_int
    lib.kvq_topk.argtypes = [cache_p, ctypes.c_int, vp, i32, i32, vp, vp, vp, sz, vp]
    lib.kvq_topk.restype = ctypes.c_int
    lib.kvq_workspace_status.argtypes = [vp, sz, vp]
    lib.kvq_workspace_status.restype = ctypes.c_int
    lib.kvq_selftest_bounded_wait.argtypes = [vp, sz, i64, vp]
    lib.kvq_selftest_bounded_wait.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise KVQError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


class QuantizedKVCache:
    """One layer's quantized KV cache in a caller-owned (torch) device buffer."""

    def __init__(self, batch: int, num_kv_heads: int, head_dim: int, group_size: int, fmt: str,
                 capacity_tokens: int, device="cuda", ragged: bool = False):
        lib = load_library()
        self.desc = KvqCacheDesc(batch, num_kv_heads, head_dim, group_size, FORMATS[fmt], 0,
                                 capacity_tokens)
        self.nbytes = lib.kvq_cache_bytes(ctypes.byref(self.desc))
        if self.nbytes == 0:
            raise KVQError(1, "kvq_cache_bytes")
        self.storage = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        self._pad = (-self.storage.data_ptr()) % 256
        self.struct = KvqCache()
        _check(lib.kvq_cache_init(ctypes.byref(self.struct), ctypes.byref(self.desc),
                                  self.storage.data_ptr() + self._pad, self.nbytes), "kvq_cache_init")
        self.fmt = fmt
        self.seq_states = None
        if ragged:
            # per-sequence state: host memory the cache struct points at, kept alive here
            self.seq_states = (KvqSeqState * batch)()
            _check(lib.kvq_cache_set_ragged(ctypes.byref(self.struct), self.seq_states, batch),
                   "kvq_cache_set_ragged")

    # host-side state
    @property
    def quantized_len(self) -> int:
        return int(self.struct.quantized_len)

    @property
    def residual_len(self) -> int:
        return int(self.struct.residual_len)

    @property
    def residual_start(self) -> int:
        return int(self.struct.residual_start)

    def state(self):
        st = (self.quantized_len, self.residual_len, self.residual_start)
        if self.seq_states is not None:
            st = st + (tuple(self.seq_state(b) for b in range(self.desc.batch)),)
        return st

    def set_state(self, st):
        """Restore host counters saved by ``state()`` (device data is not touched)."""
        self.struct.quantized_len, self.struct.residual_len, self.struct.residual_start = st[:3]
        if self.seq_states is not None:
            for b, (lq, r, start) in enumerate(st[3]):
                self.seq_states[b].quantized_len, self.seq_states[b].residual_len = lq, r
                self.seq_states[b].residual_start = start

    def seq_state(self, b: int):
        """(Lq, r, residual_start) of sequence b of a ragged cache."""
        x = self.seq_states[b]
        return (int(x.quantized_len), int(x.residual_len), int(x.residual_start))

    # raw region views (uint8 / float32 / bf16), for inspection and tests
    def _region(self, off: int, nbytes: int) -> torch.Tensor:
        o = self._pad + off
        return self.storage[o:o + nbytes]

    def k_plane(self, i: int) -> torch.Tensor:
        d = self.desc
        pb = 4 if self.fmt == "hier8" else FORMATS[self.fmt]
        row = d.head_dim * pb // 8
        n = d.batch * d.num_kv_heads * d.capacity_tokens * row
        return self._region(self.struct.off_k_plane[i], n).view(d.batch * d.num_kv_heads, d.capacity_tokens, row)

    def v_plane(self, i: int) -> torch.Tensor:
        d = self.desc
        pb = 4 if self.fmt == "hier8" else FORMATS[self.fmt]
        row = 32 * pb // 8
        n = d.batch * d.num_kv_heads * d.capacity_tokens * d.head_dim * pb // 8
        return self._region(self.struct.off_v_plane[i], n).view(
            d.batch * d.num_kv_heads, d.capacity_tokens // 32, d.head_dim, row)

    def k_scale_zero(self) -> torch.Tensor:
        d = self.desc
        U, C, D, G = d.batch * d.num_kv_heads, d.capacity_tokens, d.head_dim, d.group_size
        return self._region(self.struct.off_k_sz, U * (C // G) * 2 * D * 4).view(torch.float32).view(U, C // G, 2, D)

    def v_scale_zero(self) -> torch.Tensor:
        d = self.desc
        U, C, D, G = d.batch * d.num_kv_heads, d.capacity_tokens, d.head_dim, d.group_size
        return self._region(self.struct.off_v_sz, U * C * 2 * (D // G) * 4).view(torch.float32).view(U, C, 2, D // G)

    def residual(self):
        """Residual buffers as stored: bf16 ``[U, 2G, D]`` keys and values."""
        d = self.desc
        U, D, G = d.batch * d.num_kv_heads, d.head_dim, d.group_size
        n = U * 2 * G * D * 2
        rk = self._region(self.struct.off_res_k, n).view(torch.bfloat16).view(U, 2 * G, D)
        rv = self._region(self.struct.off_res_v, n).view(torch.bfloat16).view(U, 2 * G, D)
        return rk, rv


def kvq_quantize_append(cache: QuantizedKVCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
    """Append tokens ``[B, Hkv, n, D]`` (bf16); see ``kvq_quantize_append`` in kvq.h."""
    d = cache.desc
    shape = (d.batch, d.num_kv_heads, k_new.shape[2] if k_new.dim() == 4 else -1, d.head_dim)
    if k_new.shape != v_new.shape or tuple(k_new.shape) != shape:
        raise ValueError(f"k_new/v_new must be [B, Hkv, n, D] = {shape}")
    lib = load_library()
    _check(lib.kvq_quantize_append(ctypes.byref(cache.struct), _ptr(k_new, torch.bfloat16, "k_new"),
                                   _ptr(v_new, torch.bfloat16, "v_new"), k_new.shape[2], _stream(stream)),
           "kvq_quantize_append")


def kvq_quantize_append_ragged(cache: QuantizedKVCache, k_new: torch.Tensor, v_new: torch.Tensor, n_new,
                               stream=None):
    """Append ``n_new[b]`` tokens to sequence b of a ragged cache: the first
    ``n_new[b]`` rows of ``k_new, v_new [B, Hkv, n_max, D]`` (bf16)."""
    d = cache.desc
    if k_new.dim() != 4 or k_new.shape != v_new.shape or k_new.shape[0] != d.batch or \
            k_new.shape[1] != d.num_kv_heads or k_new.shape[3] != d.head_dim:
        raise ValueError("k_new/v_new must be [B, Hkv, n_max, D]")
    counts = (ctypes.c_int32 * d.batch)(*[int(x) for x in n_new])
    _check(load_library().kvq_quantize_append_ragged(ctypes.byref(cache.struct), _ptr(k_new, torch.bfloat16, "k_new"),
                                                     _ptr(v_new, torch.bfloat16, "v_new"), k_new.shape[2], counts,
                                                     _stream(stream)),
           "kvq_quantize_append_ragged")


def kvq_workspace_bytes(cache: QuantizedKVCache, num_q_heads: int, gamma: int, top_k: int = 0) -> int:
    return int(load_library().kvq_workspace_bytes(ctypes.byref(cache.struct), num_q_heads, gamma, top_k))


def make_workspace(cache: QuantizedKVCache, num_q_heads: int, gamma: int, top_k: int = 0) -> torch.Tensor:
    """Zero-filled workspace for ``kvq_attend`` / ``kvq_topk`` on this cache."""
    n = kvq_workspace_bytes(cache, num_q_heads, gamma, top_k)
    if n == 0:
        raise KVQError(1, "kvq_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=cache.storage.device)


def kvq_attend(cache: QuantizedKVCache, mode: str, q: torch.Tensor, pend_k=None, pend_v=None,
               sel_idx=None, sel_k=None, sel_v=None, sm_scale: float = 0.0, out=None, lse=None,
               workspace: Optional[torch.Tensor] = None, want_lse: bool = True, stream=None):
    """Decode attention; ``q [B, gamma, Hq, D]`` bf16.  Returns (out, lse)."""
    B, gamma, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, gamma, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = make_workspace(cache, Hq, gamma, 0 if sel_idx is None else sel_idx.shape[-1])
    n_pend = 0 if pend_k is None else pend_k.shape[2]
    top_k = 0 if sel_idx is None else sel_idx.shape[2]
    lib = load_library()
    _check(lib.kvq_attend(ctypes.byref(cache.struct), MODES[mode], _ptr(q, torch.bfloat16, "q"), Hq, gamma,
                          _ptr(pend_k, torch.bfloat16, "pend_k"), _ptr(pend_v, torch.bfloat16, "pend_v"),
                          n_pend, _ptr(sel_idx, torch.int32, "sel_idx"),
                          _ptr(sel_k, torch.bfloat16, "sel_k"), _ptr(sel_v, torch.bfloat16, "sel_v"),
                          top_k, float(sm_scale), _ptr(out, torch.bfloat16, "out"),
                          _ptr(lse, torch.float32, "lse"), _ptr(workspace, torch.uint8, "workspace"),
                          workspace.numel(), _stream(stream)),
           "kvq_attend")
    return out, lse


def kvq_attend_topk(cache: QuantizedKVCache, mode: str, q: torch.Tensor, next_k: int, score_row: int = 1,
                    pend_k=None, pend_v=None, sel_idx=None, sel_k=None, sel_v=None, sm_scale: float = 0.0,
                    out=None, lse=None, next_idx=None, next_score=None, workspace: Optional[torch.Tensor] = None,
                    want_lse: bool = True, stream=None):
    """Attention plus the next step's top-k from one read of the low-bit keys;
    ``score_row`` picks the query token whose summed heads score the tokens
    (1: the speculative token, 0: the output token).  Returns
    (out, lse, next_idx, next_score)."""
    B, gamma, Hq, D = q.shape
    Hkv = cache.desc.num_kv_heads
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, gamma, Hq), dtype=torch.float32, device=q.device)
    if next_idx is None:
        next_idx = torch.empty((B, Hkv, next_k), dtype=torch.int32, device=q.device)
    if next_score is None:
        next_score = torch.empty((B, Hkv, next_k), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = make_workspace(cache, Hq, gamma, next_k)
    n_pend = 0 if pend_k is None else pend_k.shape[2]
    top_k = 0 if sel_idx is None else sel_idx.shape[2]
    lib = load_library()
    _check(lib.kvq_attend_topk(ctypes.byref(cache.struct), MODES[mode], _ptr(q, torch.bfloat16, "q"), Hq, gamma,
                               _ptr(pend_k, torch.bfloat16, "pend_k"), _ptr(pend_v, torch.bfloat16, "pend_v"), n_pend,
                               _ptr(sel_idx, torch.int32, "sel_idx"), _ptr(sel_k, torch.bfloat16, "sel_k"),
                               _ptr(sel_v, torch.bfloat16, "sel_v"), top_k, float(sm_scale),
                               _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"), int(score_row),
                               int(next_k), _ptr(next_idx, torch.int32, "next_idx"),
                               _ptr(next_score, torch.float32, "next_score"), _ptr(workspace, torch.uint8, "workspace"),
                               workspace.numel(), _stream(stream)),
           "kvq_attend_topk")
    return out, lse, next_idx, next_score


def kvq_attend_plan(cache: QuantizedKVCache, mode: str, num_q_heads: int, gamma: int, n_pend: int = 0,
                    top_k: int = 0) -> dict:
    """How ``kvq_attend`` would split such a call on the current device:
    quantized splits, tail splits, chunk tokens and whether each (b, kv head)
    runs as one thread-block cluster."""
    info = KvqAttendPlanInfo()
    lib = load_library()
    _check(lib.kvq_attend_plan(ctypes.byref(cache.struct), MODES[mode], num_q_heads, gamma, n_pend, top_k,
                               ctypes.byref(info)), "kvq_attend_plan")
    return {"quant_splits": info.quant_splits, "tail_splits": info.tail_splits,
            "chunk_tokens": info.chunk_tokens, "cluster": bool(info.cluster)}


def kvq_gather_selected(full_k: torch.Tensor, full_v: torch.Tensor, sel_idx: torch.Tensor, sel_k=None, sel_v=None,
                        stream=None):
    """The selected tokens' 16-bit K/V, ``sel_idx [B, Hkv, k]`` int32 on the
    device, from the full store ``full_k, full_v [B, Hkv, N, D]`` bf16 in
    pinned host memory (or on the device).  Returns ``(sel_k, sel_v)``
    ``[B, Hkv, k, D]`` bf16 on the device; entries outside [0, N) are zero."""
    B, Hkv, N, D = full_k.shape
    if full_v.shape != full_k.shape or full_k.dtype != torch.bfloat16 or full_v.dtype != torch.bfloat16:
        raise ValueError("full_k and full_v must be bf16 tensors of one shape")
    if not (full_k.is_contiguous() and full_v.is_contiguous()):
        raise ValueError("full_k and full_v must be contiguous")
    if full_k.device.type == "cpu" and not (full_k.is_pinned() and full_v.is_pinned()):
        raise ValueError("a host store must be in pinned memory")
    k = sel_idx.shape[2]
    if sel_k is None:
        sel_k = torch.empty((B, Hkv, k, D), dtype=torch.bfloat16, device=sel_idx.device)
    if sel_v is None:
        sel_v = torch.empty_like(sel_k)
    lib = load_library()
    _check(lib.kvq_gather_selected(full_k.data_ptr(), full_v.data_ptr(), N, B, Hkv, D,
                                   _ptr(sel_idx, torch.int32, "sel_idx"), k, _ptr(sel_k, torch.bfloat16, "sel_k"),
                                   _ptr(sel_v, torch.bfloat16, "sel_v"), _stream(stream)),
           "kvq_gather_selected")
    return sel_k, sel_v


def kvq_attend_static_scratch(cache: QuantizedKVCache, mode: str, q: torch.Tensor, pend_k=None, pend_v=None,
                              sel_idx=None, sel_k=None, sel_v=None, sm_scale: float = 0.0, out=None, lse=None,
                              stream=None):
    """``kvq_attend`` for callers that cannot allocate device memory: the
    workspace is a fixed 16 MiB array inside the library (see kvq.h).  The output
    and LSE buffers must still be passed in; nothing is allocated here either."""
    B, gamma, Hq, D = q.shape
    if out is None or lse is None:
        raise ValueError("pass preallocated out and lse")
    n_pend = 0 if pend_k is None else pend_k.shape[2]
    top_k = 0 if sel_idx is None else sel_idx.shape[2]
    lib = load_library()
    _check(lib.kvq_attend_static_scratch(ctypes.byref(cache.struct), MODES[mode], _ptr(q, torch.bfloat16, "q"),
                                         Hq, gamma, _ptr(pend_k, torch.bfloat16, "pend_k"),
                                         _ptr(pend_v, torch.bfloat16, "pend_v"), n_pend,
                                         _ptr(sel_idx, torch.int32, "sel_idx"), _ptr(sel_k, torch.bfloat16, "sel_k"),
                                         _ptr(sel_v, torch.bfloat16, "sel_v"), top_k, float(sm_scale),
                                         _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
                                         _stream(stream)),
           "kvq_attend_static_scratch")
    return out, lse


def kvq_topk(cache: QuantizedKVCache, mode: str, q_spec: torch.Tensor, k: int, idx_out=None,
             score_out=None, workspace: Optional[torch.Tensor] = None, want_scores: bool = True,
             stream=None):
    """Top-k token indices per KV head; ``q_spec [B, Hq, D]`` bf16.  Returns (idx, score)."""
    B, Hq, D = q_spec.shape
    Hkv = cache.desc.num_kv_heads
    if idx_out is None:
        idx_out = torch.empty((B, Hkv, k), dtype=torch.int32, device=q_spec.device)
    if score_out is None and want_scores:
        score_out = torch.empty((B, Hkv, k), dtype=torch.float32, device=q_spec.device)
    if workspace is None:
        workspace = make_workspace(cache, Hq, 1, k)
    lib = load_library()
    _check(lib.kvq_topk(ctypes.byref(cache.struct), MODES[mode], _ptr(q_spec, torch.bfloat16, "q_spec"), Hq, k,
                        _ptr(idx_out, torch.int32, "idx_out"), _ptr(score_out, torch.float32, "score_out"),
                        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)),
           "kvq_topk")
    return idx_out, score_out


def kvq_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Read and clear the workspace's device status word (synchronizes the stream)."""
    return int(load_library().kvq_workspace_status(_ptr(workspace, torch.uint8, "workspace"),
                                                   workspace.numel(), _stream(stream)))


def kvq_selftest_bounded_wait(workspace: torch.Tensor, limit_cycles: int, stream=None):
    _check(load_library().kvq_selftest_bounded_wait(_ptr(workspace, torch.uint8, "workspace"),
                                                    workspace.numel(), int(limit_cycles), _stream(stream)),
           "kvq_selftest_bounded_wait")


def kvq_status_string(status: int) -> str:
    return load_library().kvq_status_string(status).decode()
