"""The projection's sections and the two-phase block built from them.

Phase 1 projects K/V only, by token chunks, into row windows of one store;
phase 2 recomputes Q only, by query chunks, and attends each chunk against
the whole store (vram_lab.py's phases: K/V kept per token chunk with Q
discarded, then Q recomputed per chunk).  Every byte equals the one-call
path: projection rows are independent, the sections write the full call's
bytes, and the attention does not depend on query tiling.  The two-phase
result is also compared with the oracle on sampled rows: the phase-1 store
against the oracle's projection, the phase-2 output against the oracle's
attention over that store."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bf16_ulp, bits16
from tests.test_qkv_proj_gpu import _compare

pytestmark = pytest.mark.gpu


def _inputs(n, C, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, C), generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn((3 * C, C), generator=g) * C ** -0.5).to(torch.bfloat16).cuda()
    return x, w


@pytest.mark.parametrize("n,C", [(1000, 1024), (200, 384)])  # 384: a 256-column tile straddles Q and K
def test_sections_write_the_full_call_bytes(n, C):
    x, w = _inputs(n, C, seed=C)
    q0, s0 = kvq.streamed_qkv_proj(x, w)
    store = kvq.PackedKV.empty(n, C, 32, 4, "cuda")
    store.k_codes.fill_(0x5A)  # rows past n stay whatever they were, rows below n must all be written
    assert kvq.streamed_qkv_proj_ex(x, w, [store], sections=kvq.SECTION_KV) is None
    q1 = kvq.streamed_qkv_proj_ex(x, w, sections=kvq.SECTION_Q)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    assert torch.equal(q0, q1)
    for a, b in ((s0.k_codes, store.k_codes), (s0.v_codes, store.v_codes), (s0.k_scales, store.k_scales),
                 (s0.v_scales, store.v_scales)):
        assert torch.equal(a[:, :n], b[:, :n])


def test_two_phase_block_equals_one_call():
    wl = inputs.MID
    x, w, qn, kn = inputs.block_inputs(wl, device="cuda")
    n, C = x.shape
    # one call
    q_ref, st_ref = kvq.streamed_qkv_proj(x, w, chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn)
    out_ref = kvq.packed_kv_attention(q_ref, st_ref)
    # phase 1: K/V by token chunks into row windows; phase 2: Q by query chunks, then attention
    store = kvq.PackedKV.empty(n, C, 32, 4, "cuda")
    for s in range(0, n, 5000):
        ln = min(5000, n - s)
        kvq.streamed_qkv_proj_ex(x[s:s + ln], w, [store.rows(s, ln)], sections=kvq.SECTION_KV,
                                 chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn)
    out = torch.empty_like(out_ref)
    qbuf = torch.empty((6144, C), dtype=torch.bfloat16, device="cuda")
    for s in range(0, n, 6144):
        ln = min(6144, n - s)
        qc = kvq.streamed_qkv_proj_ex(x[s:s + ln], w, sections=kvq.SECTION_Q, chunk_tokens=wl.chunk_tokens,
                                      q_norm_w=qn, k_norm_w=kn, q_out=qbuf[:ln])
        kvq.packed_kv_attention(qc, store, out=out[s:s + ln])
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    assert torch.equal(store.k_codes[:, :n], st_ref.k_codes[:, :n])
    assert torch.equal(store.v_scales[:, :n], st_ref.v_scales[:, :n])
    assert torch.equal(out, out_ref)
    # against the oracle: phase 1's store and phase 2's Q on sampled token rows,
    # phase 2's output on the same rows
    rows = inputs.sample_rows(n, 24, seed=61).numpy()
    idx = torch.as_tensor(rows, device="cuda")
    xs = x[idx]
    ref = oracle.qkv_proj(bits16(xs), bits16(w), q_norm_w=qn.cpu().numpy(), k_norm_w=kn.cpu().numpy())
    q2 = torch.zeros_like(q_ref)
    q2[idx] = kvq.streamed_qkv_proj_ex(xs, w, sections=kvq.SECTION_Q, chunk_tokens=wl.chunk_tokens, q_norm_w=qn,
                                       k_norm_w=kn)
    _compare(q2, store, ref, rows, xs, w, qn, kn, what="two-phase block")
    att = oracle.attention(ref["q_bf16"], store.k_codes.cpu().numpy(), store.v_codes.cpu().numpy(),
                           bits16(store.k_scales), bits16(store.v_scales), n_kv=n)
    # the oracle's attention takes the oracle's Q; the GPU's differs from it only
    # within the projection tolerance, so compare with the GPU's own Q as well
    att_gpu_q = oracle.attention(bits16(q_ref[idx]), store.k_codes.cpu().numpy(), store.v_codes.cpu().numpy(),
                                 bits16(store.k_scales), bits16(store.v_scales), n_kv=n)
    got = out[idx].float().cpu().numpy().astype(np.float64)
    for r_ in (att_gpu_q, att):
        err = np.abs(got - r_)
        assert np.all(err <= 1e-2 + 0.5 * bf16_ulp(r_)), float(err.max())
        assert np.linalg.norm(got - r_) / np.linalg.norm(r_) <= 5e-3
