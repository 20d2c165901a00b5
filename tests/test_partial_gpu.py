"""Attention over key chunks with a carried state (vram_lab.py ("VRAM Lab"):
`_blockwise_attention_q` attends K/V blocks and `_online_combine` merges each
block's normalised output and log-sum-exp; the module notes plan K/V staged
in host memory and streamed to the device block by block).

Parity: the chunked result against the oracle's blockwise attention over the
same chunks, and against the one-call oracle, with the attention's bar
(max-abs <= 1e-2, relative L2 <= 5e-3 on fp32 output).  The carried state
itself (normalised output in the rotated basis, log-sum-exp) is compared with
the oracle's partial results.  Query rows are independent: any query
chunking gives the same bits for the same key chunking."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bf16_ulp, bits16

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 5e-3
LSE_ABS = 5e-3  # score error from the FP16 K^ operand: about |s| 2^-12, a few 1e-3 at |s| ~ 10


def _store(heads, n, group=32, bits=4, seed=0, device="cuda"):
    cap = kvq.padded_rows(n)
    kc, vc, ks, vs = inputs.random_packed_kv(heads, n, cap, group, bits, seed=seed, device=device)
    if bits == 8:  # INT8 codes are about 18x finer: keep K.q scores and V of the INT4 stores' size
        ks, vs = (ks.float() / 18).half(), (vs.float() / 18).half()
    return kvq.PackedKV(kc.to("cuda"), vc.to("cuda"), ks.to("cuda"), vs.to("cuda"), n, bits, group)


def _windows(store, sizes):
    """Consecutive key chunks of one store, each a one-range table (a row window)."""
    out, a = [], 0
    for ln in sizes:
        out.append([store.rows(a, ln)])
        a += ln
    assert a == store.n
    return out


def _oracle_ranges(chunk):
    rs, start = [], 0
    for st in chunk:
        rs.append(dict(start=start, len=st.n, bits=st.bits, k_codes=st.k_codes.cpu().numpy(),
                       v_codes=st.v_codes.cpu().numpy(), k_scales=bits16(st.k_scales), v_scales=bits16(st.v_scales)))
        start += st.n
    return rs


def _run(q, chunks, out_fp32=True, out=None):
    state = None
    for i, ch in enumerate(chunks):
        last = i == len(chunks) - 1
        r = kvq.packed_kv_attention_partial(q, ch, state=state, merge=i > 0, final=last, out_fp32=out_fp32, out=out)
        if not last:
            state = r
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    return r


def _assert_close(got, ref, max_abs=MAX_ABS, rel_l2=REL_L2):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= max_abs, float(err.max())
    assert rel <= rel_l2, float(rel)


@pytest.mark.parametrize("sizes", [[700], [128, 572], [1, 699], [300, 300, 100], [129, 255, 316], [699, 1]])
def test_key_chunks_match_oracle_blockwise_and_one_call(sizes):
    heads, n, nq = 2, 700, 300
    st = _store(heads, n, seed=len(sizes) + sizes[0])
    q = inputs.random_q(nq, heads * 128, seed=sizes[-1], std=2.0).cuda()
    chunks = _windows(st, sizes)
    got = _run(q, chunks).cpu().numpy()
    qb = bits16(q)
    ref_blockwise = oracle.attention_blockwise(qb, [_oracle_ranges(c) for c in chunks])
    _assert_close(got, ref_blockwise)
    ref_one = oracle.attention(qb, st.k_codes.cpu().numpy(), st.v_codes.cpu().numpy(), bits16(st.k_scales),
                               bits16(st.v_scales), n_kv=n)
    _assert_close(got, ref_one)


def test_carried_state_matches_oracle_partials():
    # after the first chunk: the chunk's own (o, lse); after the second: the merge
    heads, n, nq = 3, 900, 257
    st = _store(heads, n, seed=41)
    q = inputs.random_q(nq, heads * 128, seed=42, std=2.5).cuda()
    c0, c1, c2 = _windows(st, [384, 300, 216])
    qb = bits16(q)
    o_acc, lse_acc = kvq.packed_kv_attention_partial(q, c0)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention_partial(qb, _oracle_ranges(c0))
    _assert_close(o_acc.cpu().numpy().reshape(nq, heads, 128), o_ref)
    assert np.abs(lse_acc.cpu().numpy() - l_ref).max() <= LSE_ABS
    kvq.packed_kv_attention_partial(q, c1, state=(o_acc, lse_acc), merge=True)
    torch.cuda.synchronize()
    o1, l1 = oracle.attention_partial(qb, _oracle_ranges(c1))
    o_ref, l_ref = oracle.lse_merge(o_ref, l_ref, o1, l1)
    _assert_close(o_acc.cpu().numpy().reshape(nq, heads, 128), o_ref)
    assert np.abs(lse_acc.cpu().numpy() - l_ref).max() <= LSE_ABS
    # the union's log-sum-exp from the oracle's one-chunk partial over both chunks
    _, l_union = oracle.attention_partial(qb, _oracle_ranges([st.rows(0, 684)]))
    assert np.abs(lse_acc.cpu().numpy() - l_union).max() <= LSE_ABS
    out = kvq.packed_kv_attention_partial(q, c2, state=(o_acc, lse_acc), merge=True, final=True, out_fp32=True)
    torch.cuda.synchronize()
    _assert_close(out.cpu().numpy(), oracle.attention_blockwise(qb, [_oracle_ranges(c) for c in (c0, c1, c2)]))


def test_mixed_precision_chunks():
    # a chunk made of an INT8 range and an INT4 range, then an INT4 chunk
    heads, nq = 2, 200
    a = _store(heads, 300, bits=8, seed=43)
    b = _store(heads, 500, bits=4, seed=44)
    q = inputs.random_q(nq, heads * 128, seed=45, std=2.0).cuda()
    chunks = [[a, b.rows(0, 200)], [b.rows(200, 300)]]
    got = _run(q, chunks).cpu().numpy()
    ref = oracle.attention_blockwise(bits16(q), [_oracle_ranges(c) for c in chunks])
    _assert_close(got, ref)
    one = kvq.packed_kv_attention_mixed(q, [a, b], out_fp32=True)
    torch.cuda.synchronize()
    _assert_close(got, one.cpu().numpy())


def test_query_chunking_does_not_change_the_bits():
    heads, n, nq = 2, 1000, 600
    st = _store(heads, n, seed=46)
    q = inputs.random_q(nq, heads * 128, seed=47, std=2.0).cuda()
    chunks = _windows(st, [256, 500, 244])
    full = _run(q, chunks)
    for a, b in ((0, 128), (128, 333), (333, 600), (599, 600)):
        part = _run(q[a:b].contiguous(), chunks)
        assert torch.equal(part, full[a:b]), (a, b)


def test_single_final_chunk_is_the_one_call_attention():
    heads, n, nq = 2, 777, 130
    st = _store(heads, n, seed=48)
    q = inputs.random_q(nq, heads * 128, seed=49, std=2.0).cuda()
    got = kvq.packed_kv_attention_partial(q, [st], final=True, out_fp32=True)
    one = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    assert torch.equal(got, one)


def test_bf16_final_output_in_place():
    heads, n, nq = 2, 640, 333
    st = _store(heads, n, seed=50)
    q = inputs.random_q(nq, heads * 128, seed=51, std=2.0).cuda()
    chunks = _windows(st, [200, 440])
    f32 = _run(q, chunks, out_fp32=True).cpu().double().numpy()
    q2 = q.clone()
    _run(q2, chunks, out_fp32=False, out=q2)  # the output written over Q
    got = q2.cpu().double().numpy()
    assert np.all(np.abs(got - f32) <= bf16_ulp(f32) * 0.5 + 1e-12)


def test_host_staged_store_streamed_by_chunks():
    # the packed store lives in pinned host memory as one contiguous buffer per key
    # chunk; each chunk is copied whole into a device chunk buffer and attended from
    # there: the bits of the device-resident run
    heads, n, nq, chunk = 2, 1100, 257, 384
    st = _store(heads, n, seed=52)
    q = inputs.random_q(nq, heads * 128, seed=53, std=2.0).cuda()
    sizes = [chunk, chunk, n - 2 * chunk]
    ref = _run(q, _windows(st, sizes))
    host, a = [], 0
    for ln in sizes:
        hc = kvq.PackedKV(*(torch.zeros_like(t[:, :chunk], device="cpu").pin_memory()
                            for t in (st.k_codes, st.v_codes, st.k_scales, st.v_scales)), chunk, 4, 32)
        for d, s_ in ((hc.k_codes, st.k_codes), (hc.v_codes, st.v_codes), (hc.k_scales, st.k_scales),
                      (hc.v_scales, st.v_scales)):
            d[:, :ln] = s_[:, a:a + ln].cpu()
        host.append(hc)
        a += ln
    buf = kvq.PackedKV.empty(chunk, heads * 128, 32, 4, "cuda")
    state, out = None, None
    for i, (ln, hc) in enumerate(zip(sizes, host)):
        for d, s_ in ((buf.k_codes, hc.k_codes), (buf.v_codes, hc.v_codes), (buf.k_scales, hc.k_scales),
                      (buf.v_scales, hc.v_scales)):
            d.copy_(s_, non_blocking=True)
        last = i == len(sizes) - 1
        r = kvq.packed_kv_attention_partial(q, [buf.rows(0, ln)], state=state, merge=i > 0, final=last, out_fp32=True)
        if last:
            out = r
        else:
            state = r
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.slow
def test_h3_width_key_chunks_sampled_rows():
    # 56 heads x 128, N = 16,384 keys in four chunks (one ragged), 2,000 queries;
    # the oracle checks sampled rows against all keys
    C, n, nq = 7168, 16384, 2000
    st = _store(C // 128, n, seed=54, device="cuda")
    q = inputs.random_q(nq, C, seed=55, std=2.0, device="cuda")
    chunks = _windows(st, [4096, 4096, 5000, 3192])
    got = _run(q, chunks)
    one = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    _assert_close(got.cpu().numpy(), one.cpu().numpy())
    rows = inputs.sample_rows(nq, 12, seed=56).numpy()
    idx = torch.as_tensor(rows, device="cuda")
    ref = oracle.attention(bits16(q[idx]), st.k_codes.cpu().numpy(), st.v_codes.cpu().numpy(), bits16(st.k_scales),
                           bits16(st.v_scales), n_kv=n)
    _assert_close(got[idx].cpu().numpy(), ref)
