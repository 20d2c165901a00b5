"""Parity of the projection with split-half RoPE of Q and K (after the
RMSNorm, before the Hadamard rotation) with the CPU oracle.  Tolerance as for
the plain projection (tests/_fused_tol.py: every differing code, scale or Q
value within the accumulator's error bound of the rounding boundary it
crossed), with the bound carried through the RoPE (its fp32 products and the
mixing of two elements)."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bits16
from tests.test_qkv_proj_gpu import _compare

pytestmark = pytest.mark.gpu


def _table(n, rot_dim, base=10000.0, offset=0):
    pos = np.arange(offset, offset + n, dtype=np.float64)
    freq = base ** (-2.0 * np.arange(rot_dim // 2) / rot_dim)
    ang = pos[:, None] * freq[None, :]
    return np.ascontiguousarray(np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32))


def _run(x, w, cs, qn=None, kn=None, chunk=0):
    n, C = x.shape
    store = kvq.PackedKV.empty(n, C, 32, 4, "cuda")
    q = kvq.streamed_qkv_proj_ex(x.cuda(), w.cuda(), [store], torch.from_numpy(cs).cuda(), chunk_tokens=chunk,
                                   q_norm_w=None if qn is None else qn.cuda(),
                                   k_norm_w=None if kn is None else kn.cuda())
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    return q, store


@pytest.mark.parametrize("rot_dim", [128, 64])
def test_tiny_block_with_rope(rot_dim):
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    cs = _table(x.shape[0], rot_dim)
    q, store = _run(x, w, cs)
    ref = oracle.qkv_proj(bits16(x), bits16(w), rope_cs=cs)
    _compare(q, store, ref, np.arange(x.shape[0]), x, w, rot_dim=rot_dim, what=f"tiny block RoPE {rot_dim}")


def test_identity_table_gives_the_plain_bits():
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    cs = np.zeros((x.shape[0], 64, 2), np.float32)
    cs[..., 0] = 1.0
    q1, s1 = _run(x, w, cs)
    q0, s0 = kvq.streamed_qkv_proj(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert torch.equal(q0, q1)
    for a, b in ((s0.k_codes, s1.k_codes), (s0.v_codes, s1.v_codes), (s0.k_scales, s1.k_scales),
                 (s0.v_scales, s1.v_scales)):
        assert torch.equal(a, b)


def test_rope_results_do_not_depend_on_chunk_size():
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    cs = _table(x.shape[0], 128)
    q0, s0 = _run(x, w, cs)
    q1, s1 = _run(x, w, cs, chunk=384)
    assert torch.equal(q0, q1)
    assert torch.equal(s0.k_codes, s1.k_codes) and torch.equal(s0.k_scales, s1.k_scales)


def test_h3_block_with_rmsnorm_and_rope_sampled_rows():
    wl = inputs.MID
    x, w, qn, kn = inputs.block_inputs(wl)
    cs = _table(wl.n, 128)
    q, store = _run(x, w, cs, qn, kn, chunk=wl.chunk_tokens)
    rows = inputs.sample_rows(wl.n, 40, seed=5).numpy()
    ref = oracle.qkv_proj(bits16(x), bits16(w), rows, q_norm_w=qn.numpy(), k_norm_w=kn.numpy(), eps=1e-6,
                          rope_cs=cs)
    _compare(q, store, ref, rows, x[torch.as_tensor(rows)], w, qn, kn, rot_dim=128, what="H3 mid RoPE 128")
