"""Parity of the packed-K/V attention kernel with the CPU oracle.

Tolerance (fp32 output, oracle fed the same packed K/V and the same BF16 Q):
max-abs <= 1e-2 and relative L2 <= 5e-3.  The BF16 output must equal the
fp32 output rounded to BF16 within one BF16 ulp."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bf16_ulp, bits16

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 5e-3


def _store(heads, n, group=32, bits=4, seed=0, device="cuda", **kw):
    cap = kvq.padded_rows(n)
    kc, vc, ks, vs = inputs.random_packed_kv(heads, n, cap, group, bits, seed=seed, device=device, **kw)
    return kvq.PackedKV(kc.to("cuda"), vc.to("cuda"), ks.to("cuda"), vs.to("cuda"), n, bits, group)


def _oracle(q, st, rows=None):
    return oracle.attention(bits16(q), st.k_codes.cpu().numpy(), st.v_codes.cpu().numpy(),
                            bits16(st.k_scales), bits16(st.v_scales), n_kv=st.n, group=st.group, bits=st.bits,
                            rows=rows)


def _assert_close(got, ref):
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= MAX_ABS, float(err.max())
    assert rel <= REL_L2, float(rel)
    return float(err.max()), float(rel)


@pytest.mark.parametrize("n_q,n_kv,heads", [(77, 1, 2), (1, 300, 2), (1, 1, 1), (128, 128, 2), (256, 256, 1), (300, 129, 2),
                                         (129, 1000, 3), (513, 2000, 2)])
def test_random_store_fp32(n_q, n_kv, heads):
    st = _store(heads, n_kv, seed=n_kv)
    q = inputs.random_q(n_q, heads * 128, seed=n_q, std=2.0).cuda()
    out = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    _assert_close(out.cpu().numpy(), _oracle(q, st))


@pytest.mark.parametrize("group", [64, 128])
def test_groups(group):
    st = _store(2, 700, group=group, seed=group)
    q = inputs.random_q(200, 256, seed=1, std=2.0).cuda()
    out = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    _assert_close(out.cpu().numpy(), _oracle(q, st))


def test_growing_scores_exercise_rescaling():
    # key scales grow 20x along the sequence, so the running max of each row
    # jumps several times (the lazy-rescale path); scores stay within what
    # RMS-normalised Q and K produce (|s| <~ 12 nats)
    heads, n = 2, 1500
    st = _store(heads, n, seed=3)
    ramp = torch.linspace(0.03, 0.6, st.cap, device="cuda").view(1, -1, 1)
    g = torch.Generator(device="cuda").manual_seed(3)
    st.k_scales.copy_((torch.rand(st.k_scales.shape, device="cuda", generator=g) * 0.2 + 0.9) * ramp)
    st.k_scales[:, n:] = 0
    q = inputs.random_q(256, heads * 128, seed=3, std=1.5).cuda()
    out = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    ref = _oracle(q, st)
    _assert_close(out.cpu().numpy(), ref)


def test_bf16_output_and_in_place():
    st = _store(2, 900, seed=4)
    q = inputs.random_q(333, 256, seed=4, std=2.0).cuda()
    f32 = kvq.packed_kv_attention(q, st, out_fp32=True)
    b16 = kvq.packed_kv_attention(q, st, out_fp32=False)
    q2 = q.clone()
    kvq.packed_kv_attention(q2, st, out_fp32=False, out=q2)  # output written over Q
    torch.cuda.synchronize()
    ref = f32.cpu().double().numpy()
    got = b16.cpu().double().numpy()
    assert np.all(np.abs(got - ref) <= bf16_ulp(ref) * 0.5 + 1e-12)
    assert torch.equal(q2, b16)


def test_query_tiling_invariance():
    # each output row depends only on its own query row: any sub-range of the
    # queries, aligned to the 128-row tiles or not, gives identical rows
    st = _store(2, 1000, seed=5)
    q = inputs.random_q(500, 256, seed=5, std=2.0).cuda()
    full = kvq.packed_kv_attention(q, st, out_fp32=True)
    for a, b in ((128, 256), (5, 133), (300, 301), (499, 500)):
        part = kvq.packed_kv_attention(q[a:b].contiguous(), st, out_fp32=True)
        torch.cuda.synchronize()
        assert torch.equal(part, full[a:b]), (a, b)


def test_tiny_block_chain_from_oracle_store():
    # the packed store and rotated Q of the tiny block, as produced by the
    # oracle's projection, attended by the kernel and by the oracle
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    ref_p = oracle.qkv_proj(bits16(x), bits16(w))
    n, heads = x.shape[0], inputs.TINY.heads
    cap = kvq.padded_rows(n)

    def hm(a, dt):
        out = np.zeros((heads, cap, a.shape[2]), a.dtype)
        out[:, :n] = a.transpose(1, 0, 2)
        return torch.from_numpy(out.view(dt) if dt is not None else out).cuda()

    st = kvq.PackedKV(hm(ref_p["k_codes"], None), hm(ref_p["v_codes"], None), hm(ref_p["k_scales"], np.float16),
                      hm(ref_p["v_scales"], np.float16), n, 4, 32)
    q = torch.from_numpy(ref_p["q_bf16"].view(np.int16)).view(torch.bfloat16).cuda()
    out = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    _assert_close(out.cpu().numpy(), _oracle(q, st))


@pytest.mark.slow
def test_h3_ref2va_full_size_sampled_rows():
    # N = 152,263 keys and queries, 56 heads, as the benchmark runs it; the
    # oracle computes a sample of query rows (exact per row)
    n, C = inputs.H3_REF2VA.n, inputs.H3_REF2VA.hidden
    st = _store(C // 128, n, seed=11, device="cuda")
    q = inputs.random_q(n, C, seed=12, std=2.0, device="cuda")
    out = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    rows = inputs.sample_rows(n, 8, seed=13).numpy()
    qs = q[torch.as_tensor(rows, device="cuda")]
    ref = _oracle(qs, st)
    _assert_close(out[torch.as_tensor(rows, device="cuda")].cpu().numpy(), ref)


# Score range.  The MMA operands are FP16: K^ = code x scale rounded to 11
# significant bits moves a score s = tau q.k^ by about |s| 2^-12 (random
# rounding over 128 terms), which shifts the softmax weights by that much
# relative, so the output error grows with the size of the scores.  Q and K
# RMS-normalised per head (the H3 block) keep |s| <= |q||k| tau ~ 11.3 (x the
# norm weights, ~14).  Q drawn with std sigma against the random store gives
# row maxima of |s| of about 9 sigma.  Measured on a GB300: sigma 2, 4, 8, 16
# reach max |s| 17, 35, 70, 139 with max-abs 2.8e-3, 7.5e-3, 1.15e-2, ... and
# relative L2 about 1e-3.  The bar is asserted up to sigma = 4 (max |s| ~ 35,
# more than twice the normalised range); beyond it the errors are recorded.
@pytest.mark.parametrize("std", [2.0, 4.0, 8.0, 16.0, 32.0])
def test_score_range_sweep(std):
    heads, n, nq = 2, 2000, 256
    st = _store(heads, n, seed=71)
    q = inputs.random_q(nq, heads * 128, seed=72, std=std).cuda()
    out = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    ref = _oracle(q, st)
    got = out.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    qf = q.float().cpu().numpy().reshape(nq, heads, 128)
    kd = (st.k_codes.cpu().numpy(), bits16(st.k_scales))
    smax = 0.0
    for h in range(heads):  # the row maxima of the scores, from the dequantised keys
        lo = (kd[0][h, :n] & 0x0F).astype(np.int16)
        hi = (kd[0][h, :n] >> 4).astype(np.int16)
        c = np.stack([lo, hi], -1).reshape(n, 128)
        c = np.where(c >= 8, c - 16, c).astype(np.float64)
        k = c * np.repeat(kd[1][h, :n].view(np.float16).astype(np.float64), 32, axis=-1)
        smax = max(smax, float(np.abs(qf[:, h] @ k.T).max()) / np.sqrt(128))
    print(f"q std {std}: max |score| {smax:.1f}, max-abs {err:.3e}, rel-L2 {rel:.3e}")
    if std <= 4.0:
        assert err <= 1e-2 and rel <= 5e-3, (err, rel)
