"""Parity of the causal packed-K/V attention with the CPU oracle.

Query row i sits at key position q_pos0 + i and attends keys j <= q_pos0 + i.
Tolerance as for the unmasked attention (fp32 output, oracle fed the same
packed K/V and BF16 Q): max-abs <= 1e-2 and relative L2 <= 5e-3.  Tiles past
a row's position contribute exact zeros, so splitting the queries into
chunks, or a position past the last key, gives the same bits."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bits16

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 5e-3


def _store(heads, n, group=32, seed=0):
    cap = kvq.padded_rows(n)
    kc, vc, ks, vs = inputs.random_packed_kv(heads, n, cap, group, 4, seed=seed, device="cuda")
    return kvq.PackedKV(kc, vc, ks, vs, n, 4, group)


def _oracle(q, st, q_pos0, rows=None):
    return oracle.attention_causal(bits16(q), st.k_codes.cpu().numpy(), st.v_codes.cpu().numpy(),
                                   bits16(st.k_scales), bits16(st.v_scales), n_kv=st.n, q_pos0=q_pos0,
                                   group=st.group, bits=4, rows=rows)


def _assert_close(got, ref):
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= MAX_ABS, float(err.max())
    assert rel <= REL_L2, float(rel)


@pytest.mark.parametrize("n_q,n_kv,q_pos0,heads", [
    (300, 300, 0, 2),      # square, ragged
    (129, 129, 0, 1),      # one row past a tile
    (77, 1000, 500, 2),    # a query chunk in the middle of the sequence
    (513, 2000, 1487, 2),  # the last chunk: its last row sees every key
    (600, 700, 0, 2),      # fewer queries than keys
    (1100, 300, 0, 1),     # more queries than keys: rows past 299 see them all
    (1, 1, 0, 1),          # one query, one key
    (1, 700, 699, 2),      # one query at the last position: sees every key
    (1, 700, 200, 2),      # one query in the middle
])
def test_causal_matches_oracle(n_q, n_kv, q_pos0, heads):
    st = _store(heads, n_kv, seed=n_kv + q_pos0)
    q = inputs.random_q(n_q, heads * 128, seed=n_q, std=2.0).cuda()
    out = kvq.packed_kv_attention_causal(q, st, q_pos0=q_pos0, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    _assert_close(out.cpu().numpy(), _oracle(q, st, q_pos0))


@pytest.mark.parametrize("group", [64, 128])
def test_causal_groups(group):
    st = _store(2, 700, group=group, seed=group)
    q = inputs.random_q(700, 256, seed=3, std=2.0).cuda()
    out = kvq.packed_kv_attention_causal(q, st, out_fp32=True)
    torch.cuda.synchronize()
    _assert_close(out.cpu().numpy(), _oracle(q, st, 0))


def test_query_chunks_give_the_one_call_bits():
    n = 1500
    st = _store(2, n, seed=5)
    q = inputs.random_q(n, 256, seed=6, std=2.0).cuda()
    whole = kvq.packed_kv_attention_causal(q, st, out_fp32=True)
    parts = torch.empty_like(whole)
    for a, b in ((0, 512), (512, 1100), (1100, 1500)):
        kvq.packed_kv_attention_causal(q[a:b], st, q_pos0=a, out_fp32=True, out=parts[a:b])
    torch.cuda.synchronize()
    assert torch.equal(whole, parts)


def test_position_past_the_last_key_is_the_unmasked_attention():
    st = _store(2, 400, seed=7)
    q = inputs.random_q(200, 256, seed=8, std=2.0).cuda()
    causal = kvq.packed_kv_attention_causal(q, st, q_pos0=399, out_fp32=True)
    full = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    assert torch.equal(causal, full)


def test_bf16_output_in_place():
    st = _store(2, 640, seed=9)
    q = inputs.random_q(640, 256, seed=10, std=2.0).cuda()
    ref = kvq.packed_kv_attention_causal(q, st, out_fp32=True)
    q2 = q.clone()
    kvq.packed_kv_attention_causal(q2, st, out=q2)
    torch.cuda.synchronize()
    assert torch.equal(q2, ref.to(torch.bfloat16))


@pytest.mark.slow
def test_h3_ref2va_full_size_sampled_rows():
    # N = 152,263 keys and queries, 56 heads, causal; the oracle computes sampled rows,
    # each at its own position
    n, C = inputs.H3_REF2VA.n, inputs.H3_REF2VA.hidden
    st = _store(C // 128, n, seed=11)
    q = inputs.random_q(n, C, seed=12, std=2.0, device="cuda")
    out = kvq.packed_kv_attention_causal(q, st, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    rows = np.concatenate([[0, 1, 127, 128, n - 1], inputs.sample_rows(n, 3, seed=13).numpy()])
    for r in rows:
        ref = _oracle(q[int(r):int(r) + 1], st, int(r))
        _assert_close(out[int(r):int(r) + 1].cpu().numpy(), ref)
