"""Per-element tolerance of the fused projection (tensor-core GEMM + rotate /
quantise epilogue) against the oracle.

The GPU accumulates x . W^T in fp32 on the tensor cores, 16 products per MMA
step along K in ascending order; the oracle accumulates in fp64 and rounds
once.  Every later step (RMSNorm, RoPE, the rotation, the quantiser) is the
same arithmetic on both sides, so the results may differ only where the
accumulator's error moves a value across a rounding boundary.  This module
bounds that error per head vector and checks every difference against it:

  accumulator  |acc_gpu - acc| <= 2^-23 sum_b |S_b| + 2^-22 sum_k |x_k w_k|
               S_b = the running sum after MMA step b: each step may commit up to
               one fp32 ulp of the running sum (rounding or truncation) and two
               of its own 16 products' absolute sum;
  RMSNorm      n_j = a_j r w_j, r = (mean a^2 + eps)^-1/2:
               |dn_j| <= |w_j| r |da_j| + |n_j| (sum_i |a_i da_i| / sum_i a_i^2 + 2^-16)
               (the second term is r's change; 2^-16 covers its fp32 evaluation);
  RoPE         each output mixes two inputs with |cos|, |sin| <= 1: the L1 error
               at most doubles, plus 2^-22 of the values for the fp32 products;
  rotation     y = (FWHT v) c: every |dy_i| <= c sum_j |dv_j| (each y_i is a
               signed sum of all v_j), plus each side's fp32 butterfly rounding,
               7 stages x 2^-24 x c sum_j |v_j|.

A scale may differ only by one fp16 step, and only where the oracle's
amax / Q lies within the amax bound (/Q) of the fp16 midpoint between the
two.  A code may differ only by one, and only where the oracle's y / s (s the
GPU's scale, so a legitimately different scale is followed through) lies
within the y bound (/s) of the half-integer between the two codes.  Q (BF16)
must lie within half a BF16 ulp plus the y bound of the oracle's fp32 value.
"""
from __future__ import annotations

import numpy as np

HD = 128
U32 = 2.0 ** -24  # fp32 unit roundoff
C_ROT = float(np.float32(2.0 ** -3.5))


def _bf16(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def accumulator_bound(x_bits, w_bits, k_step: int = 16, out_block: int = 2048):
    """(acc fp64 [rows, O], bound fp64 [rows, O]) for x [rows, C] and W [O, C] (BF16 bits)."""
    x = _bf16(x_bits)
    w_all = np.asarray(w_bits, np.uint16)
    rows, C = x.shape
    O = w_all.shape[0]
    assert C % k_step == 0
    nb = C // k_step
    xb = np.ascontiguousarray(x.reshape(rows, nb, k_step).transpose(1, 0, 2))  # [nb, rows, k]
    acc = np.empty((rows, O))
    bound = np.empty((rows, O))
    for o0 in range(0, O, out_block):
        w = _bf16(w_all[o0:o0 + out_block])
        wb = np.ascontiguousarray(w.reshape(w.shape[0], nb, k_step).transpose(1, 2, 0))  # [nb, k, o]
        run = np.zeros((rows, w.shape[0]))
        sum_abs = np.zeros_like(run)
        for b in range(nb):
            run += xb[b] @ wb[b]
            sum_abs += np.abs(run)
        acc[:, o0:o0 + w.shape[0]] = run
        bound[:, o0:o0 + w.shape[0]] = 2.0 * U32 * sum_abs + 4.0 * U32 * (np.abs(x) @ np.abs(w).T)
    return acc, bound


def _norm_bound(a, da, wgt, eps):
    """Propagates the per-element bound da [.., 128] of a [.., 128] through the
    RMSNorm with weight wgt [128] (None: no norm).  Returns (v, dv)."""
    if wgt is None:
        return a, da
    ss = np.sum(a * a, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(ss / HD + eps)
    n = a * r * wgt
    rel_r = np.sum(np.abs(a) * da, axis=-1, keepdims=True) / np.maximum(ss, 1e-300) + 2.0 ** -16
    return n, np.abs(wgt) * r * da + np.abs(n) * rel_r


def _rope_bound(v, dv, rot_dim):
    if not rot_dim:
        return v, dv
    l1 = np.sum(dv, axis=-1, keepdims=True)
    # the L1 error at most doubles; spread it as a per-element bound that sums to that
    return v, np.broadcast_to(2.0 * l1 / HD, dv.shape) + 4.0 * U32 * np.abs(v)


def head_bounds(x_bits, w_bits, q_norm_w=None, k_norm_w=None, eps: float = 1e-6, rot_dim: int = 0):
    """Bounds on |y_gpu - y_oracle| of the rotated Q, K and V head vectors:
    dict q, k, v -> fp64 [rows, heads] (one bound per head vector, valid for
    each of its 128 elements)."""
    acc, dacc = accumulator_bound(x_bits, w_bits)
    rows, O = acc.shape
    C = O // 3
    heads = C // HD
    qn = None if q_norm_w is None else np.asarray(q_norm_w, np.float64)
    kn = None if k_norm_w is None else np.asarray(k_norm_w, np.float64)
    out = {}
    for name, blk, wgt in (("q", 0, qn), ("k", 1, kn), ("v", 2, None)):
        a = acc[:, blk * C:(blk + 1) * C].reshape(rows, heads, HD)
        da = dacc[:, blk * C:(blk + 1) * C].reshape(rows, heads, HD)
        v, dv = _norm_bound(a, da, wgt, eps)
        if name != "v":
            v, dv = _rope_bound(v, dv, rot_dim)
        l1v = np.sum(np.abs(v), axis=-1)
        out[name] = C_ROT * np.sum(dv, axis=-1) + 2.0 * 7.0 * U32 * C_ROT * l1v * (1 + 1e-3)
    return out


def _codes_int(codes, bits):
    codes = np.asarray(codes, np.uint8)
    if bits == 8:
        return codes.view(np.int8).astype(np.int32)
    lo = (codes & 0x0F).astype(np.int32)
    hi = (codes >> 4).astype(np.int32)
    v = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], -1)
    return np.where(v >= 8, v - 16, v)


def check_kv(gpu_codes, gpu_scales, ref_codes, ref_scales, y_ref, bound, bits: int, group: int,
             what: str = "") -> dict:
    """gpu_codes / ref_codes [rows, heads, 128*bits/8] uint8, gpu_scales /
    ref_scales [rows, heads, 128/group] fp16 bits, y_ref [rows, heads*128] the
    oracle's rotated values (fp32), bound [rows, heads].  Asserts that every
    difference from the oracle's codes and scales is justified; returns the counts."""
    Q = 7.0 if bits == 4 else 127.0
    rows, heads = bound.shape
    y = np.asarray(y_ref, np.float64).reshape(rows, heads, HD)
    g_codes = _codes_int(gpu_codes, bits)
    expect = _codes_int(ref_codes, bits)
    g_bits = np.asarray(gpu_scales, np.uint16).reshape(rows, heads, -1)
    r_bits = np.asarray(ref_scales, np.uint16).reshape(rows, heads, -1)
    s_gpu, s_ref = _f16(g_bits), _f16(r_bits)
    ng = HD // group
    amax = np.max(np.abs(y.reshape(rows, heads, ng, group)), axis=-1)
    exact = amax / Q
    # scales
    diff = g_bits != r_bits
    n_scale = int(diff.sum())
    if n_scale:
        steps = np.abs(g_bits[diff].astype(np.int64) - r_bits[diff].astype(np.int64))
        assert steps.max() <= 1, f"{what}: a scale differs by more than one fp16 step"
        mid = 0.5 * (s_gpu[diff] + s_ref[diff])
        slack = np.broadcast_to(bound[:, :, None], diff.shape)[diff] / Q + 2.0 * U32 * exact[diff]
        dist = np.abs(exact[diff] - mid)
        assert np.all(dist <= slack), (f"{what}: {int((dist > slack).sum())} of {n_scale} differing scales are not "
                                       f"within the accumulator bound of an fp16 midpoint "
                                       f"(worst {float((dist / slack).max()):.2f}x the bound)")
    # codes: the oracle's, or, in a group whose scale legitimately differs, the
    # oracle's values quantised with the GPU's scale
    s_el = np.repeat(s_gpu, group, axis=-1).reshape(rows, heads, HD)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(s_el > 0, y / s_el, 0.0)
    dgrp = np.repeat(diff, group, axis=-1).reshape(rows, heads, HD)
    expect = np.where(dgrp, np.clip(np.rint(t), -Q, Q).astype(np.int32), expect)
    cd = g_codes != expect
    n_code = int(cd.sum())
    if n_code:
        dc = np.abs(g_codes[cd] - expect[cd])
        assert dc.max() <= 1, f"{what}: a code differs by more than one"
        half = 0.5 * (g_codes[cd] + expect[cd])
        slack = np.broadcast_to(bound[:, :, None], cd.shape)[cd] / s_el[cd] + 2.0 * U32 * np.abs(t[cd])
        dist = np.abs(t[cd] - half)
        assert np.all(dist <= slack), (f"{what}: {int((dist > slack).sum())} of {n_code} differing codes are not "
                                       f"within the accumulator bound of a rounding boundary "
                                       f"(worst {float((dist / slack).max()):.2f}x the bound)")
    return {"scales": int(diff.size), "scales_differing": n_scale, "codes": int(cd.size), "codes_differing": n_code}


def check_q(q_gpu_bits, q_ref_f32, q_ref_bits, bound, what: str = "q") -> dict:
    """Q BF16 [rows, C] against the oracle's fp32 value: within half a BF16 ulp
    (at the value plus its bound) plus the y bound."""
    got = _bf16(q_gpu_bits)
    ref = np.asarray(q_ref_f32, np.float64)
    rows, C = ref.shape
    b = np.repeat(bound, HD, axis=1).reshape(rows, C)
    mag = np.maximum(np.abs(ref) + b, 2.0 ** -126)
    half_ulp = 2.0 ** (np.floor(np.log2(mag)) - 8)
    err = np.abs(got - ref)
    ok = err <= half_ulp + b
    assert np.all(ok), f"{what}: {int((~ok).sum())} values beyond half a BF16 ulp + the bound"
    differ = np.asarray(q_gpu_bits, np.uint16) != np.asarray(q_ref_bits, np.uint16)
    return {"q": int(err.size), "q_differing": int(differ.sum())}
