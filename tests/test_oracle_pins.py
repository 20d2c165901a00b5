"""Pins for the CPU oracle: each test checks it against something other than
itself -- a library routine for a special case, a closed form, an invariant,
a hand-worked value, a bound the method guarantees, or brute force on tiny
inputs -- chosen so that a dropped term, a wrong sign or index or a
transposed operand in the oracle fails at least one of them.

Sources: the comfy-kitchen feature request "Streamed QKV Projection and Packed
Low-Bit K/V Support for Extreme Long-Sequence Attention" and vram_lab.py
("VRAM Lab"): `_hadamard`, `_fq_int4`, `_Int8KV`, `_online_combine`, the kvi8r
docstring's rotated-basis identities.
"""
import numpy as np
import pytest
import scipy.linalg
import scipy.special
import torch

import oracle

HD = 128
H_UNNORM = scipy.linalg.hadamard(HD).astype(np.float64)  # Sylvester construction (library)
H = H_UNNORM / np.sqrt(HD)


def _rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ number formats
def test_f16_conversion_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7C00) != 0x7C00
    ref = bits.view(np.float16).astype(np.float32)
    got = oracle.f16_to_f32(bits[finite])
    assert np.array_equal(got.view(np.uint32), ref[finite].view(np.uint32))


def test_f32_to_f16_round_to_nearest_even_matches_numpy():
    r = _rng(1)
    vals = np.concatenate([
        r.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** r.integers(-9, 5, 20000).astype(np.float32),
        # exact ties between adjacent fp16 values, in the normal and subnormal ranges
        (np.arange(1, 2000, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -10),
        (np.arange(1, 2000, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24),
        np.array([65504, 65519.99, 65520, 65536, 1e9, 2.0 ** -25, 2.0 ** -25 * 1.0001, 2.0 ** -26, 0.0, -0.0],
                 np.float32),
    ]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16(vals)
    assert np.array_equal(got, ref)


def test_f32_to_bf16_round_to_nearest_even_matches_torch():
    r = _rng(2)
    vals = (r.standard_normal(50000) * 10.0 ** r.integers(-20, 20, 50000)).astype(np.float32)
    ties = (np.arange(1, 500, dtype=np.uint32) << 16 | 0x8000).view(np.float32) + np.float32(0)
    vals = np.concatenate([vals, ties, -ties])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16(vals), ref)


# ------------------------------------------------------------------ rotation
def test_rotation_scale_is_fp32_of_inverse_sqrt_128():
    c = oracle.rot_scale()
    assert np.float32(c).view(np.uint32) == 0x3DB504F3
    assert np.float32(c) == np.float32(2.0 ** -3.5)


def test_rotation_of_unit_vectors_is_scaled_sylvester_column():
    # e_i . H = row i of H: the Sylvester matrix built by doubling [[h, h], [h, -h]]
    eye = np.eye(HD, dtype=np.float32)
    got = oracle.rotate(eye)
    c = np.float32(oracle.rot_scale())
    assert np.array_equal(got, (H_UNNORM.astype(np.float32) * c))


def test_rotation_matches_matrix_form_exactly_on_small_integers():
    # integer inputs make every butterfly exact, so the fast transform equals
    # the dense product with the library's Sylvester matrix, times c rounded once
    r = _rng(3)
    x = r.integers(-50, 51, size=(64, HD)).astype(np.float32)
    got = oracle.rotate(x)
    ref = (x.astype(np.float64) @ H_UNNORM).astype(np.float32) * np.float32(oracle.rot_scale())
    assert np.array_equal(got, ref)


def test_rotation_is_orthonormal():
    r = _rng(4)
    x = r.standard_normal((256, HD)).astype(np.float32)
    y = oracle.rotate(x)
    assert np.allclose(y, x.astype(np.float64) @ H, rtol=0, atol=2e-6 * np.abs(x).max())
    # H H^T = I: rotating twice returns the input (H is symmetric)
    z = oracle.rotate(y)
    assert np.max(np.abs(z - x)) < 1e-5
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)
    assert np.allclose(H @ H.T, np.eye(HD), atol=1e-12)


def test_rotation_spreads_a_spike_evenly():
    # the outlier-suppression property: a single spike becomes a flat vector
    x = np.zeros(HD, np.float32)
    x[17] = 20.0
    y = oracle.rotate(x)
    assert np.allclose(np.abs(y), 20.0 / np.sqrt(HD), rtol=1e-6)


# ------------------------------------------------------------------ quantiser
def _unpack_nibbles(codes):
    lo = (codes & 0x0F).astype(np.int16)
    hi = (codes >> 4).astype(np.int16)
    v = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], -1)
    return np.where(v >= 8, v - 16, v)


def test_quantiser_hand_cases_ties_round_to_even():
    # group max 7 gives a scale of exactly 1, so codes are rint(y) with ties to even
    y = np.zeros(HD, np.float32)
    y[:8] = [7.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5]
    codes, scales = oracle.quant_head(y, 32, 4)
    assert scales[0] == np.float16(1.0).view(np.uint16)
    q = _unpack_nibbles(codes)
    assert list(q[:8]) == [7, 2, 4, -2, -4, 0, 2, 0]
    # packing: element 2i low nibble, 2i+1 high nibble, two's complement
    assert codes[0] == 0x27  # (7, 2)
    assert codes[1] == 0xE4  # (4, -2)


def test_packing_bytes():
    y = np.zeros(HD, np.float32)
    y[0:4] = [-1.0, 7.0, 3.0, -7.0]
    codes, scales = oracle.quant_head(y, 32, 4)
    assert scales[0] == np.float16(1.0).view(np.uint16)
    assert codes[0] == 0x7F and codes[1] == 0x93
    assert np.all(codes[2:] == 0)


def test_quantiser_zero_group_and_subnormal_scale():
    y = np.zeros(HD, np.float32)
    y[32] = 7.0 * 2.0 ** -20  # scale 2^-20 is an fp16 subnormal, represented exactly
    y[64] = 1.4 * 2.0 ** -24  # amax/7 = 0.2 * 2^-24 rounds to 0 -> code 0
    y[96] = 9.8 * 2.0 ** -24  # amax/7 = 1.4 * 2^-24 rounds to 2^-24 -> 9.8 clamps to 7
    codes, scales = oracle.quant_head(y, 32, 4)
    q = _unpack_nibbles(codes)
    assert scales[0] == 0 and np.all(q[:32] == 0)
    assert oracle.f16_to_f32(scales[1:2])[0] == np.float32(2.0 ** -20) and q[32] == 7
    assert scales[2] == 0 and q[64] == 0
    assert scales[3] == 1 and q[96] == 7


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("bits", [4, 8])
def test_quantiser_error_bound_and_full_range(group, bits):
    qmax = 7 if bits == 4 else 127
    r = _rng(5 + group + bits)
    for _ in range(200):
        y = (r.standard_normal(HD) * r.choice([1e-3, 1.0, 30.0])).astype(np.float32)
        y[r.integers(0, HD)] *= 20.0
        codes, scales = oracle.quant_head(y, group, bits)
        assert codes.shape == (HD * bits // 8,) and scales.shape == (HD // group,)
        q = _unpack_nibbles(codes) if bits == 4 else codes.view(np.int8).astype(np.int16)
        s = scales.view(np.float16).astype(np.float64)
        s_el = np.repeat(s, group)
        # scale: fp16 round-to-nearest of group absmax / qmax
        amax = np.abs(y.reshape(-1, group)).max(axis=1)
        assert np.array_equal(scales, (amax / np.float32(qmax)).astype(np.float32).astype(np.float16).view(np.uint16))
        assert np.all(np.abs(q) <= qmax)
        # every group with a normal, non-zero scale reaches the end of the code range
        assert np.all(np.abs(q.reshape(-1, group)).max(axis=1) == qmax)
        # |y - code * s| <= s / 2
        err = np.abs(y.astype(np.float64) - q * s_el)
        assert np.all(err <= s_el / 2 * (1 + 1e-6))
        # dequantisation is code * scale
        assert np.array_equal(oracle.dequant_head(codes, scales, group, bits), (q * s_el).astype(np.float32))


def test_int8_codes_are_plain_bytes():
    y = np.zeros(HD, np.float32)
    y[0], y[1], y[2] = 127.0, -127.0, 63.5
    codes, scales = oracle.quant_head(y, 32, 8)
    assert scales[0] == np.float16(1.0).view(np.uint16)
    assert list(codes[:3].view(np.int8)) == [127, -127, 64]


# ------------------------------------------------------------------ a1 / a1b on token rows
def _bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_kv_pack_spike_row_is_all_sevens():
    # a K head that is a single spike a.e_0 rotates to the constant a.c: every
    # code is 7 and every scale is fp16(a.c / 7)
    hidden = 256
    kv = torch.zeros((1, 2 * hidden), dtype=torch.bfloat16)
    kv[0, 0] = 3.0
    kv[0, hidden + 128 + 5] = -2.0
    kc, vc, ks, vs = oracle.kv_rotate_quant_pack(_bf16_bits(kv), hidden=hidden)
    c = np.float32(oracle.rot_scale())
    q = _unpack_nibbles(kc[0, 0])
    assert np.all(q == 7)
    assert np.all(ks[0, 0] == np.float16(np.float32(3.0) * c / np.float32(7.0)).view(np.uint16))
    assert np.all(kc[0, 1] == 0) and np.all(ks[0, 1] == 0)
    qv = _unpack_nibbles(vc[0, 1])
    assert np.all(np.abs(qv) == 7)
    assert np.array_equal(np.sign(qv), -np.sign(H_UNNORM[5]).astype(np.int16))


def test_kv_pack_unpack_roundtrip_bound_and_row_independence():
    hidden = 512
    kv = (torch.randn((40, 2 * hidden), generator=torch.Generator().manual_seed(7)) * 3).to(torch.bfloat16)
    bits = _bf16_bits(kv)
    kc, vc, ks, vs = oracle.kv_rotate_quant_pack(bits, hidden=hidden)
    out = oracle.kv_unpack(kc, vc, ks, vs)
    x = kv.float().numpy()
    y = oracle.bf16_to_f32(out)
    heads = hidden // HD
    s = np.concatenate([ks, vs], axis=1).view(np.float16).astype(np.float64)  # [n, 2*heads, 4]
    # the un-rotation is orthonormal: the per-head L2 error is at most the
    # rotated-basis error, sqrt(sum over elements (s/2)^2), plus BF16 rounding
    err = (y - x).reshape(40, 2 * heads, HD)
    bound = np.sqrt(np.sum((s / 2) ** 2 * 32, axis=-1)) + np.linalg.norm(x.reshape(40, 2 * heads, HD), axis=-1) * 2 ** -8
    assert np.all(np.linalg.norm(err, axis=-1) <= bound)
    # rows are independent: any subset gives the same codes (row-chunk exactness)
    sub = np.array([39, 3, 17], np.int64)
    kc2, vc2, ks2, vs2 = oracle.kv_rotate_quant_pack(bits, sub, hidden=hidden)
    assert np.array_equal(kc2, kc[sub]) and np.array_equal(vs2, vs[sub])


# ------------------------------------------------------------------ a2 projection
def _small_block(n=24, C=256, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, C), generator=g).to(torch.bfloat16)
    w = (torch.randn((3 * C, C), generator=g) * C ** -0.5).to(torch.bfloat16)
    return x, w


def test_qkv_projection_q_is_rotated_matmul():
    x, w = _small_block()
    C = x.shape[1]
    out = oracle.qkv_proj(_bf16_bits(x), _bf16_bits(w))
    acc = x.double().numpy() @ w.double().numpy().T  # library matmul
    q_ref = (acc[:, :C].reshape(-1, C // HD, HD) @ H).reshape(-1, C)
    assert np.max(np.abs(out["q_f32"] - q_ref)) < 1e-5
    assert np.array_equal(out["q_bf16"], oracle.f32_to_bf16(out["q_f32"]))


def test_qkv_projection_sections_k_and_v():
    # K columns [C, 2C) and V columns [2C, 3C): zero the K block of W and the
    # K codes and scales vanish while V stays non-zero; the V codes dequantise
    # and un-rotate to x . W_V^T within the quantiser bound
    x, w = _small_block()
    C = x.shape[1]
    w = w.clone()
    w[C:2 * C] = 0
    out = oracle.qkv_proj(_bf16_bits(x), _bf16_bits(w))
    assert np.all(out["k_codes"] == 0) and np.all(out["k_scales"] == 0)
    assert np.any(out["v_codes"] != 0)
    acc_v = x.double().numpy() @ w.double().numpy()[2 * C:].T
    n, heads = out["v_codes"].shape[:2]
    for t in range(n):
        for h in range(heads):
            yv = oracle.dequant_head(out["v_codes"][t, h], out["v_scales"][t, h], 32, 4).astype(np.float64)
            s = np.repeat(out["v_scales"][t, h].view(np.float16).astype(np.float64), 32)
            assert np.all(np.abs(yv - acc_v[t, h * HD:(h + 1) * HD] @ H) <= s / 2 + 1e-6)


def test_qkv_projection_rmsnorm_properties():
    x, w = _small_block(n=16)
    C = x.shape[1]
    ones = np.ones(HD, np.float32)
    out = oracle.qkv_proj(_bf16_bits(x), _bf16_bits(w), q_norm_w=ones, k_norm_w=ones, eps=1e-6)
    q = out["q_f32"].reshape(16, C // HD, HD).astype(np.float64)
    # unit weight: each normalised head has RMS 1, and the rotation keeps norms
    assert np.allclose(np.sqrt(np.mean(q ** 2, axis=-1)), 1.0, atol=1e-5)
    # scale invariance: doubling x (exact in BF16) leaves normalised Q unchanged
    out2 = oracle.qkv_proj(_bf16_bits(x * 2), _bf16_bits(w), q_norm_w=ones, k_norm_w=ones, eps=1e-6)
    assert np.max(np.abs(out2["q_f32"] - out["q_f32"])) < 1e-5
    # the weight multiplies elementwise before the rotation
    wv = (1.0 + 0.5 * np.arange(HD) / HD).astype(np.float32)
    out3 = oracle.qkv_proj(_bf16_bits(x), _bf16_bits(w), q_norm_w=wv, k_norm_w=ones, eps=1e-6)
    unrot = out3["q_f32"].reshape(16, C // HD, HD).astype(np.float64) @ H
    unrot1 = q @ H
    assert np.allclose(unrot, unrot1 * wv, atol=1e-5)
    # K normalisation: the K codes dequantise to a unit-RMS head (within quantiser error)
    kq = oracle.dequant_head(out["k_codes"][0, 0], out["k_scales"][0, 0], 32, 4)
    assert abs(np.sqrt(np.mean(kq.astype(np.float64) ** 2)) - 1.0) < 0.1


# ------------------------------------------------------------------ split-half RoPE in the projection (next row f2)
def _rope_table(n, rot_dim, base=10000.0, pos=None):
    """Standard rotary table: angle pos * base^(-2i/rot_dim) for frequency i."""
    pos = np.arange(n, dtype=np.float64) if pos is None else np.asarray(pos, np.float64)
    freq = base ** (-2.0 * np.arange(rot_dim // 2) / rot_dim)
    ang = pos[:, None] * freq[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)


def _proj_inputs(n=6, C=256, seed=31):
    r = _rng(seed)
    x = _bf16_bits(torch.from_numpy(r.standard_normal((n, C)).astype(np.float32)).to(torch.bfloat16))
    w = _bf16_bits(torch.from_numpy((r.standard_normal((3 * C, C)) * C ** -0.5).astype(np.float32)).to(torch.bfloat16))
    return x, w


def test_rope_identity_table_changes_nothing():
    x, w = _proj_inputs()
    cs = np.zeros((x.shape[0], 64, 2), np.float32)
    cs[..., 0] = 1.0
    a = oracle.qkv_proj(x, w)
    b = oracle.qkv_proj(x, w, rope_cs=cs)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("rot_dim", [128, 64])
def test_rope_quarter_turn_moves_the_second_half_with_a_minus_sign(rot_dim):
    # cos 0, sin 1: y_i = -x_{i+h}, y_{i+h} = x_i for i < h = rot_dim/2; dims past rot_dim unchanged
    x, w = _proj_inputs()
    n, C = x.shape
    cs = np.zeros((n, rot_dim // 2, 2), np.float32)
    cs[..., 1] = 1.0
    u0 = oracle.qkv_proj(x, w)["q_f32"].reshape(n, C // HD, HD).astype(np.float64) @ H
    u1 = oracle.qkv_proj(x, w, rope_cs=cs)["q_f32"].reshape(n, C // HD, HD).astype(np.float64) @ H
    h = rot_dim // 2
    exp = u0.copy()
    exp[..., :h] = -u0[..., h:rot_dim]
    exp[..., h:rot_dim] = u0[..., :h]
    assert np.allclose(u1, exp, atol=1e-5)


def test_rope_keeps_norms_and_dot_products_depend_on_position_difference():
    # the same token at every position: |q| unchanged, and q_m . q_n depends on m - n only
    x, w = _proj_inputs(n=1)
    n = 12
    xs = np.repeat(x, n, axis=0)
    cs = _rope_table(n, 128)
    q0 = oracle.qkv_proj(xs, w)["q_f32"].astype(np.float64)
    q1 = oracle.qkv_proj(xs, w, rope_cs=cs)["q_f32"].astype(np.float64)
    heads = x.shape[1] // HD
    q0 = q0.reshape(n, heads, HD)
    q1 = q1.reshape(n, heads, HD)
    assert np.allclose(np.linalg.norm(q1, axis=-1), np.linalg.norm(q0, axis=-1), rtol=1e-5)
    for d in (1, 3, 5):
        dots = np.array([np.sum(q1[m] * q1[m + d], axis=-1) for m in range(n - d)])
        assert np.allclose(dots, dots[0], rtol=1e-4, atol=1e-4)
    # and it is not the identity: neighbouring positions differ
    assert not np.allclose(q1[1], q1[0], atol=1e-3)


# ------------------------------------------------------------------ a4 attention
def _head_major(kc, vc, ks, vs, n_pad):
    """compact token-major [n, heads, ...] -> head-major [heads, n_pad, ...] with zero pad rows."""
    def hm(a):
        n = a.shape[0]
        out = np.zeros((a.shape[1], n_pad, a.shape[2]), a.dtype)
        out[:, :n] = a.transpose(1, 0, 2)
        return out
    return hm(kc), hm(vc), hm(ks), hm(vs)


def _brute_attention(q_bits, kc, vc, ks, vs, n_kv, group, bits, sm_scale):
    """Independent brute force: numpy unpacking, scipy softmax, float64 matmuls,
    un-rotation by the library Sylvester matrix."""
    heads = kc.shape[0]
    q = oracle.bf16_to_f32(q_bits).astype(np.float64).reshape(q_bits.shape[0], heads, HD)

    def deq(codes, scales):
        if bits == 4:
            v = _unpack_nibbles(codes)
        else:
            v = codes.view(np.int8).astype(np.int16)
        return v.astype(np.float64) * np.repeat(scales.view(np.float16).astype(np.float64), group, axis=-1)

    out = np.empty_like(q)
    for h in range(heads):
        K = deq(kc[h, :n_kv], ks[h, :n_kv])
        V = deq(vc[h, :n_kv], vs[h, :n_kv])
        P = scipy.special.softmax(q[:, h] @ K.T * sm_scale, axis=-1)
        out[:, h] = (P @ V) @ H.T
    return out.reshape(q_bits.shape[0], -1)


@pytest.mark.parametrize("bits", [4, 8])
def test_attention_matches_brute_force(bits):
    from serving_tcgen05_streamed_gb300 import inputs
    heads, n, n_pad, nq = 2, 200, 256, 37
    kc, vc, ks, vs = [t.numpy() for t in inputs.random_packed_kv(heads, n, n_pad, 32, bits, seed=3)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    q = _bf16_bits(inputs.random_q(nq, heads * HD, seed=4, std=2.0))
    got = oracle.attention(q, kc, vc, ks, vs, n_kv=n, group=32, bits=bits)
    ref = _brute_attention(q, kc, vc, ks, vs, n, 32, bits, HD ** -0.5)
    assert np.max(np.abs(got - ref)) < 1e-5 * max(1.0, np.abs(ref).max())


def _brute_attention_causal(q_bits, kc, vc, ks, vs, n_kv, q_pos0, group, bits, sm_scale):
    """Independent brute force of the prefix (causal) mask: the full score
    matrix plus -inf above the shifted diagonal, scipy softmax, float64."""
    heads = kc.shape[0]
    nq = q_bits.shape[0]
    q = oracle.bf16_to_f32(q_bits).astype(np.float64).reshape(nq, heads, HD)

    def deq(codes, scales):
        v = _unpack_nibbles(codes) if bits == 4 else codes.view(np.int8).astype(np.int16)
        return v.astype(np.float64) * np.repeat(scales.view(np.float16).astype(np.float64), group, axis=-1)

    mask = np.where(np.arange(n_kv)[None, :] > (q_pos0 + np.arange(nq))[:, None], -np.inf, 0.0)
    out = np.empty_like(q)
    for h in range(heads):
        K = deq(kc[h, :n_kv], ks[h, :n_kv])
        V = deq(vc[h, :n_kv], vs[h, :n_kv])
        P = scipy.special.softmax(q[:, h] @ K.T * sm_scale + mask, axis=-1)
        out[:, h] = (P @ V) @ H.T
    return out.reshape(nq, -1)


@pytest.mark.parametrize("bits,q_pos0", [(4, 0), (4, 5), (8, 150), (4, 180)])
def test_attention_causal_matches_masked_brute_force(bits, q_pos0):
    from serving_tcgen05_streamed_gb300 import inputs
    heads, n, n_pad, nq = 2, 200, 256, 37
    kc, vc, ks, vs = [t.numpy() for t in inputs.random_packed_kv(heads, n, n_pad, 32, bits, seed=21)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    q = _bf16_bits(inputs.random_q(nq, heads * HD, seed=22, std=2.0))
    got = oracle.attention_causal(q, kc, vc, ks, vs, n_kv=n, q_pos0=q_pos0, group=32, bits=bits)
    ref = _brute_attention_causal(q, kc, vc, ks, vs, n, q_pos0, 32, bits, HD ** -0.5)
    assert np.max(np.abs(got - ref)) < 1e-5 * max(1.0, np.abs(ref).max())


def test_attention_causal_closed_forms_and_limits():
    from serving_tcgen05_streamed_gb300 import inputs
    heads, n, nq = 1, 64, 8
    kc, vc, ks, vs = [t.numpy() for t in inputs.random_packed_kv(heads, n, n, 32, 4, seed=23)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    q = _bf16_bits(inputs.random_q(nq, HD, seed=24, std=2.0))
    # position 0 sees key 0 alone: its value, un-rotated
    out = oracle.attention_causal(q, kc, vc, ks, vs, n_kv=n, q_pos0=0)
    v0 = oracle.dequant_head(vc[0, 0], vs[0, 0], 32, 4).astype(np.float64) @ H
    assert np.allclose(out[0], v0, atol=1e-6)
    # positions past the last key see every key: the unmasked attention, bit for bit
    full = oracle.attention(q, kc, vc, ks, vs, n_kv=n)
    assert np.array_equal(oracle.attention_causal(q, kc, vc, ks, vs, n_kv=n, q_pos0=n - 1), full)
    # a mask on key j changes nothing for rows that cannot see it: perturbing the
    # last key leaves every row at a position before it unchanged
    kc2 = kc.copy()
    kc2[0, n - 1] ^= 0x77
    a = oracle.attention_causal(q, kc, vc, ks, vs, n_kv=n, q_pos0=20)
    b = oracle.attention_causal(q, kc2, vc, ks, vs, n_kv=n, q_pos0=20)
    assert np.array_equal(a, b)
    # row sampling returns the same rows
    rows = np.array([7, 0, 3], np.int64)
    assert np.array_equal(oracle.attention_causal(q, kc, vc, ks, vs, n_kv=n, q_pos0=20, rows=rows), a[rows])


def test_attention_closed_forms():
    heads, C = 1, 128
    r = _rng(8)
    # n_kv = 1: the output is that key's value, un-rotated
    y = r.standard_normal((1, HD)).astype(np.float32)
    kc, vc, ks, vs = [np.ascontiguousarray(a.transpose(1, 0, 2)) for a in oracle.kv_rotate_quant_pack(
        oracle.f32_to_bf16(np.concatenate([y, y], axis=1)), hidden=C)]
    q = oracle.f32_to_bf16(r.standard_normal((3, C)).astype(np.float32))
    out = oracle.attention(q, kc, vc, ks, vs, n_kv=1)
    vhat = oracle.dequant_head(vc[0, 0], vs[0, 0], 32, 4).astype(np.float64) @ H
    assert np.allclose(out, np.broadcast_to(vhat, out.shape), atol=1e-6)
    # all keys equal: uniform weights, output = mean of the values, un-rotated
    from serving_tcgen05_streamed_gb300 import inputs
    n = 50
    kc, vc, ks, vs = [t.numpy() for t in inputs.random_packed_kv(1, n, n, 32, 4, seed=9)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    kc[:] = kc[:, :1]
    ks[:] = ks[:, :1]
    out = oracle.attention(q, kc, vc, ks, vs, n_kv=n)
    vmean = np.mean([oracle.dequant_head(vc[0, j], vs[0, j], 32, 4) for j in range(n)], axis=0) @ H
    assert np.allclose(out, np.broadcast_to(vmean, out.shape), atol=1e-5)
    # one dominant key: the output tends to its value
    q1 = np.zeros((1, C), np.float32)
    k1 = oracle.dequant_head(kc[0, 0], ks[0, 0], 32, 4)
    kc2 = kc.copy()
    kc2[0, 7] = kc[0, 0] ^ 0xFF  # a different key
    q1[0] = k1 * 40.0
    out = oracle.attention(oracle.f32_to_bf16(q1), kc2, vc, ks, vs, n_kv=n)
    # keys equal to k1 share the weight equally; key 7 gets none
    v_rest = np.mean([oracle.dequant_head(vc[0, j], vs[0, j], 32, 4) for j in range(n) if j != 7], axis=0) @ H
    assert np.allclose(out[0], v_rest, atol=1e-4)


def test_attention_rotated_basis_identity():
    # q.k = (qH).(kH) and P.V = (P.(VH)).H^T: attention in the rotated basis
    # then one un-rotation equals plain softmax attention on un-rotated vectors
    from serving_tcgen05_streamed_gb300 import inputs
    heads, n, nq = 2, 64, 9
    kc, vc, ks, vs = [t.numpy() for t in inputs.random_packed_kv(heads, n, n, 64, 4, seed=11)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    q = _bf16_bits(inputs.random_q(nq, heads * HD, seed=12, std=3.0))
    got = oracle.attention(q, kc, vc, ks, vs, n_kv=n, group=64)
    qf = oracle.bf16_to_f32(q).astype(np.float64).reshape(nq, heads, HD)
    for h in range(heads):
        K = np.stack([oracle.dequant_head(kc[h, j], ks[h, j], 64, 4) for j in range(n)]).astype(np.float64) @ H.T
        V = np.stack([oracle.dequant_head(vc[h, j], vs[h, j], 64, 4) for j in range(n)]).astype(np.float64) @ H.T
        qm = qf[:, h] @ H.T
        P = scipy.special.softmax(qm @ K.T / np.sqrt(HD), axis=-1)
        assert np.allclose(got[:, h * HD:(h + 1) * HD], P @ V, atol=1e-5)


def test_attention_key_permutation_invariance_and_row_sampling():
    from serving_tcgen05_streamed_gb300 import inputs
    heads, n, nq = 1, 96, 12
    kc, vc, ks, vs = [t.numpy() for t in inputs.random_packed_kv(heads, n, n, 32, 4, seed=13)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    q = _bf16_bits(inputs.random_q(nq, HD, seed=14, std=2.0))
    out = oracle.attention(q, kc, vc, ks, vs, n_kv=n)
    perm = _rng(15).permutation(n)
    out_p = oracle.attention(q, kc[:, perm], vc[:, perm], ks[:, perm], vs[:, perm], n_kv=n)
    assert np.allclose(out, out_p, atol=1e-6)
    rows = np.array([11, 0, 5], np.int64)
    assert np.array_equal(oracle.attention(q, kc, vc, ks, vs, n_kv=n, rows=rows), out[rows])


def test_attention_mixed_equals_concatenated_store():
    from serving_tcgen05_streamed_gb300 import inputs
    heads, nq = 2, 5
    a = [t.numpy() for t in inputs.random_packed_kv(heads, 40, 64, 32, 8, seed=16)]
    b = [t.numpy() for t in inputs.random_packed_kv(heads, 70, 128, 32, 4, seed=17)]
    q = _bf16_bits(inputs.random_q(nq, heads * HD, seed=18, std=2.0))
    ranges = [dict(start=0, len=40, bits=8, k_codes=a[0], v_codes=a[1], k_scales=a[2].view(np.uint16),
                   v_scales=a[3].view(np.uint16)),
              dict(start=40, len=70, bits=4, k_codes=b[0], v_codes=b[1], k_scales=b[2].view(np.uint16),
                   v_scales=b[3].view(np.uint16))]
    got = oracle.attention_mixed(q, ranges)
    # reference: brute force over the two stores' dequantised keys, concatenated
    qf = oracle.bf16_to_f32(q).astype(np.float64).reshape(nq, heads, HD)
    for h in range(heads):
        K = np.concatenate([
            np.stack([oracle.dequant_head(a[0][h, j], a[2].view(np.uint16)[h, j], 32, 8) for j in range(40)]),
            np.stack([oracle.dequant_head(b[0][h, j], b[2].view(np.uint16)[h, j], 32, 4) for j in range(70)])])
        V = np.concatenate([
            np.stack([oracle.dequant_head(a[1][h, j], a[3].view(np.uint16)[h, j], 32, 8) for j in range(40)]),
            np.stack([oracle.dequant_head(b[1][h, j], b[3].view(np.uint16)[h, j], 32, 4) for j in range(70)])])
        P = scipy.special.softmax(qf[:, h] @ K.astype(np.float64).T / np.sqrt(HD), axis=-1)
        assert np.allclose(got[:, h * HD:(h + 1) * HD], (P @ V) @ H.T, atol=1e-5)


# ------------------------------------------------------------------ next row f3: attention over key chunks
def _deq_np(codes, scales, group, bits):
    v = _unpack_nibbles(codes) if bits == 4 else codes.view(np.int8).astype(np.int16)
    return v.astype(np.float64) * np.repeat(scales.view(np.float16).astype(np.float64), group, axis=-1)


def _chunk_ranges(stores, lens):
    """Range table of one key chunk: consecutive ranges over the given stores
    (each a head-major (kc, vc, ks, vs, bits) tuple) with the given lengths."""
    out, start = [], 0
    for (kc, vc, ks, vs, bits), ln in zip(stores, lens):
        out.append(dict(start=start, len=ln, bits=bits, k_codes=kc, v_codes=vc, k_scales=ks.view(np.uint16),
                        v_scales=vs.view(np.uint16)))
        start += ln
    return out


def _store_np(heads, n, cap, group, bits, seed):
    from serving_tcgen05_streamed_gb300 import inputs
    kc, vc, ks, vs = [t.numpy() for t in inputs.random_packed_kv(heads, n, cap, group, bits, seed=seed)]
    return kc, vc, ks.view(np.uint16), vs.view(np.uint16), bits


@pytest.mark.parametrize("bits", [4, 8])
def test_attention_partial_matches_brute_force_logsumexp(bits):
    # o = softmax-weighted dequantised V in the rotated basis, lse = log sum exp(s):
    # against numpy unpacking, scipy.special.softmax and scipy.special.logsumexp
    from serving_tcgen05_streamed_gb300 import inputs
    heads, n, nq = 2, 150, 11
    st = _store_np(heads, n, 256, 32, bits, seed=31)
    q = _bf16_bits(inputs.random_q(nq, heads * HD, seed=32, std=2.0))
    o, lse = oracle.attention_partial(q, _chunk_ranges([st], [n]))
    qf = oracle.bf16_to_f32(q).astype(np.float64).reshape(nq, heads, HD)
    for h in range(heads):
        K = _deq_np(st[0][h, :n], st[2][h, :n], 32, bits)
        V = _deq_np(st[1][h, :n], st[3][h, :n], 32, bits)
        s = qf[:, h] @ K.T * float(np.float32(HD ** -0.5))  # the scale crosses the C boundary as fp32
        assert np.allclose(lse[:, h], scipy.special.logsumexp(s, axis=-1), rtol=0, atol=1e-10)
        assert np.allclose(o[:, h], scipy.special.softmax(s, axis=-1) @ V, rtol=0, atol=1e-10)


def test_lse_merge_of_disjoint_chunks_is_the_partial_of_their_union():
    # _online_combine: merging the partials of two disjoint key sets gives the
    # partial of the union; a wrong weight sign or a missing term fails this
    from serving_tcgen05_streamed_gb300 import inputs
    heads, nq = 2, 7
    a = _store_np(heads, 60, 128, 32, 8, seed=33)
    b = _store_np(heads, 90, 128, 32, 4, seed=34)
    q = _bf16_bits(inputs.random_q(nq, heads * HD, seed=35, std=3.0))
    oa, la = oracle.attention_partial(q, _chunk_ranges([a], [60]))
    ob, lb = oracle.attention_partial(q, _chunk_ranges([b], [90]))
    ou, lu = oracle.attention_partial(q, _chunk_ranges([a, b], [60, 90]))
    om, lm = oracle.lse_merge(oa, la, ob, lb)
    assert np.allclose(lm, lu, rtol=0, atol=1e-12)
    assert np.allclose(om, ou, rtol=0, atol=1e-12)
    # the merge is symmetric and leaves its inputs untouched
    om2, lm2 = oracle.lse_merge(ob, lb, oa, la)
    assert np.allclose(om2, om, rtol=0, atol=1e-14) and np.allclose(lm2, lm, rtol=0, atol=1e-14)
    assert np.array_equal(oa, oracle.attention_partial(q, _chunk_ranges([a], [60]))[0])
    # the log-sum-exp of the union: log(e^la + e^lb), from numpy's own logaddexp
    assert np.allclose(lm, np.logaddexp(la, lb), rtol=0, atol=1e-12)


def test_lse_merge_limits():
    # a chunk whose log-sum-exp is far below the other's contributes nothing;
    # two equal partials merge to the same output with lse + log 2
    r = _rng(36)
    o = r.standard_normal((3, 2, HD))
    lse = r.standard_normal((3, 2))
    o2 = r.standard_normal((3, 2, HD))
    om, lm = oracle.lse_merge(o, lse, o2, lse - 800.0)
    assert np.array_equal(om, o) and np.array_equal(lm, lse)
    om, lm = oracle.lse_merge(o, lse, o, lse)
    assert np.allclose(om, o, rtol=0, atol=1e-14) and np.allclose(lm, lse + np.log(2.0), rtol=0, atol=1e-14)


@pytest.mark.parametrize("splits", [[200], [1, 199], [128, 72], [50, 50, 50, 50], [127, 1, 72]])
def test_blockwise_attention_equals_one_call_attention(splits):
    # any key chunking, merged in order and un-rotated once, is the attention
    # over all keys (exact in exact arithmetic; fp32 output rounding here).  A
    # single chunk gives the one-call oracle's bits: same sums, one rounding.
    from serving_tcgen05_streamed_gb300 import inputs
    heads, n, nq = 2, 200, 9
    kc, vc, ks, vs, _ = _store_np(heads, n, 256, 32, 4, seed=37)
    q = _bf16_bits(inputs.random_q(nq, heads * HD, seed=38, std=2.0))
    full = oracle.attention(q, kc, vc, ks, vs, n_kv=n)
    chunks, a = [], 0
    for ln in splits:  # each chunk a window of rows [a, a+ln) of the one store
        chunks.append(_chunk_ranges([(kc[:, a:], vc[:, a:], ks[:, a:], vs[:, a:], 4)], [ln]))
        a += ln
    got = oracle.attention_blockwise(q, chunks)
    if len(splits) == 1:
        assert np.array_equal(got, full)
    else:
        assert np.max(np.abs(got - full)) < 2e-6 * max(1.0, np.abs(full).max())


def test_qkv_projection_rotated_kv_outputs():
    # k_rot / v_rot are what the quantiser sees: re-quantising them gives the
    # stored codes and scales, and v_rot is x . W_V^T . H (library matmul)
    r = _rng(39)
    n, C = 5, 256
    x = oracle.f32_to_bf16(r.standard_normal((n, C)).astype(np.float32))
    w = oracle.f32_to_bf16((r.standard_normal((3 * C, C)) / np.sqrt(C)).astype(np.float32))
    qn = (1.0 + 0.1 * r.standard_normal(HD)).astype(np.float32)
    ref = oracle.qkv_proj(x, w, q_norm_w=qn, k_norm_w=qn)
    for t in range(n):
        for h in range(C // HD):
            for rot, cn, sn in (("k_rot", "k_codes", "k_scales"), ("v_rot", "v_codes", "v_scales")):
                codes, scales = oracle.quant_head(ref[rot][t, h * HD:(h + 1) * HD], 32, 4)
                assert np.array_equal(codes, ref[cn][t, h]) and np.array_equal(scales, ref[sn][t, h])
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    wf = oracle.bf16_to_f32(w).astype(np.float64)
    v = (xf @ wf[2 * C:].T).reshape(n, C // HD, HD) @ H
    assert np.allclose(ref["v_rot"].reshape(n, C // HD, HD), v, rtol=0, atol=1e-5 * np.abs(v).max())
