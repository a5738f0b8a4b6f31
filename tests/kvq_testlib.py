"""Helpers for the GPU parity tests: build the same cache with the CUDA library
and with the CPU oracle from the same seeded inputs, then compare."""
from __future__ import annotations

import numpy as np
import torch

import kvq_inputs as ki
import oracle
import quantized_kv_speculative_gb300 as kvq

TOL_REL = 2e-3   # |err| <= 2e-3 * max|ref| + 1e-3 over the whole output of a call
TOL_ABS = 1e-3


def dev(x: np.ndarray) -> torch.Tensor:
    return ki.f32_to_bf16_tensor(x, "cuda")


def build_pair(fmt, B, Hkv, D, G, cap, K, V, chunks):
    """Append K/V ``[B, Hkv, N, D]`` in the given chunk sizes to a device cache
    and to an oracle cache (which appends token by token)."""
    gc = kvq.QuantizedKVCache(B, Hkv, D, G, fmt, cap)
    oc = oracle.OracleCache(B, Hkv, D, G, fmt, cap)
    pos = 0
    for n in chunks:
        kvq.kvq_quantize_append(gc, dev(K[:, :, pos:pos + n]), dev(V[:, :, pos:pos + n]))
        oc.append(K[:, :, pos:pos + n], V[:, :, pos:pos + n])
        pos += n
    torch.cuda.synchronize()
    assert (gc.quantized_len, gc.residual_len) == (oc.Lq, oc.r)
    return gc, oc


def compare_cache(gc: kvq.QuantizedKVCache, oc: oracle.OracleCache):
    """Bit-exact comparison of codes, scales, zeros and the residual buffer."""
    L, G = oc.Lq, oc.G
    U = oc.B * oc.H
    if L > 0:
        _compare_quantized(gc, oc, L, G, U)
    rk, rv = gc.residual()
    slots = [(gc.residual_start + i) % (2 * G) for i in range(gc.residual_len)]
    ork, orv = oc.residual()
    got_k = ki.bf16_tensor_to_f32(rk[:, slots]) if slots else np.zeros((U, 0, oc.D), np.float32)
    got_v = ki.bf16_tensor_to_f32(rv[:, slots]) if slots else np.zeros((U, 0, oc.D), np.float32)
    np.testing.assert_array_equal(got_k, ork.reshape(U, -1, oc.D))
    np.testing.assert_array_equal(got_v, orv.reshape(U, -1, oc.D))


def _compare_quantized(gc, oc, L, G, U):
    """The L quantized tokens: code planes, key scale/zero, value scale/zero."""
    for i, plane in enumerate(oc.packed_k_planes()):
        got = gc.k_plane(i)[:, :L].cpu().numpy()
        np.testing.assert_array_equal(got, plane.reshape(U, L, -1), err_msg=f"key plane {i}")
    for i, plane in enumerate(oc.packed_v_planes()):
        got = gc.v_plane(i)[:, :L // 32].cpu().numpy()
        np.testing.assert_array_equal(got, plane.reshape(U, L // 32, oc.D, -1), err_msg=f"value plane {i}")
    ksz = gc.k_scale_zero()[:, :L // G].cpu().numpy()
    np.testing.assert_array_equal(ksz[:, :, 0].view(np.uint32), oc.k_scale[:, :, :L // G].reshape(U, L // G, -1).view(np.uint32))
    np.testing.assert_array_equal(ksz[:, :, 1].view(np.uint32), oc.k_zero[:, :, :L // G].reshape(U, L // G, -1).view(np.uint32))
    vsz = gc.v_scale_zero()[:, :L].cpu().numpy()
    np.testing.assert_array_equal(vsz[:, :, 0].view(np.uint32), oc.v_scale[:, :, :L].reshape(U, L, -1).view(np.uint32))
    np.testing.assert_array_equal(vsz[:, :, 1].view(np.uint32), oc.v_zero[:, :, :L].reshape(U, L, -1).view(np.uint32))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits): 2^(floor(log2|x|) - 7)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def assert_attention_close(out_dev: torch.Tensor, lse_dev, ref_out: np.ndarray, ref_lse: np.ndarray, what=""):
    """Attention parity for bf16 outputs.

    The stated bound is |err| <= 2e-3*max|ref| + 1e-3 over the call's output.
    A bf16 output cannot do better than its own rounding, which alone reaches
    2^-8*|ref_i| (about 7.8e-3 just above 2.0).  So each element also gets one
    bf16 ulp of its reference value as an output-rounding allowance.  The
    accuracy before rounding is checked separately, and ten times more
    tightly: every output must be within half a bf16 ulp of its reference
    plus 2e-4*max|ref|.
    """
    got = ki.bf16_tensor_to_f32(out_dev).astype(np.float64)
    if got.size == 0:
        return 0.0
    err = np.abs(got - ref_out)
    tol = TOL_REL * np.abs(ref_out).max() + TOL_ABS + bf16_ulp(ref_out)
    worst = np.argmax(err - tol)
    assert np.all(err <= tol), (f"{what}: |err| {err.flat[worst]:.3e} > tol {tol.flat[worst]:.3e} "
                                f"at ref {ref_out.flat[worst]:.4f}")
    tight = 0.5 * bf16_ulp(ref_out) + 2e-4 * np.abs(ref_out).max()
    worst = np.argmax(err - tight)
    assert np.all(err <= tight), (f"{what}: |err| {err.flat[worst]:.3e} beyond half an ulp + 2e-4*max "
                                  f"({tight.flat[worst]:.3e}) at ref {ref_out.flat[worst]:.4f}")
    if lse_dev is not None:
        gl = lse_dev.cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin), f"{what}: lse finiteness differs"
        if fin.any():
            dl = np.abs(gl[fin] - ref_lse[fin]).max()
            assert dl <= 1e-3 + 1e-4 * np.abs(ref_lse[fin]).max(), f"{what}: max |dlse| {dl:.3e}"
    return float(err.max())


def mode_fmt(mode):
    return kvq.MODE_FORMAT[mode]
