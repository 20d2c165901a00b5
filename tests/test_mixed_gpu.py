"""Mixed precision by token range: chosen ranges stored at INT8 (per-32
absmax scales), the rest at rotated INT4, in one projection call and one
attention call."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._fused_tol import check_q, head_bounds
from tests._util import bits16
from tests.test_qkv_proj_gpu import _compare

pytestmark = pytest.mark.gpu


def _np_store(st):
    return dict(k_codes=st.k_codes.cpu().numpy(), v_codes=st.v_codes.cpu().numpy(),
                k_scales=bits16(st.k_scales), v_scales=bits16(st.v_scales), bits=st.bits, len=st.n)


def test_mixed_projection_writes_each_range_at_its_precision():
    # segments like the H3 layout, scaled down: text, reference, audio at INT8, video at INT4
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    C = x.shape[1]
    segs = [(100, 8), (300, 8), (60, 8), (564, 4)]
    stores = [kvq.PackedKV.empty(n, C, 32, b) for n, b in segs]
    for s in stores:  # poison, so that unwritten rows would show
        for t in (s.k_codes, s.v_codes):
            t.fill_(0x77)
    q = kvq.streamed_qkv_proj_mixed(x.cuda(), w.cuda(), stores, group=32, chunk_tokens=256)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    q_ref, _ = kvq.streamed_qkv_proj(x.cuda(), w.cuda(), group=32)
    torch.cuda.synchronize()
    assert torch.equal(q, q_ref)  # Q does not depend on the K/V precision
    start = 0
    for (n, bits), st in zip(segs, stores):
        rows = np.arange(start, start + n)
        ref = oracle.qkv_proj(bits16(x), bits16(w), rows, bits=bits)
        _compare(None, st, ref, np.arange(n), x[start:start + n], w, bits=bits, what=f"range of {n} at INT{bits}")
        start += n


@pytest.mark.parametrize("lens", [[(40, 8), (700, 4)], [(128, 8), (256, 8), (129, 4), (1, 8)]])
def test_mixed_attention_matches_oracle(lens):
    heads, C = 2, 256
    stores = []
    for i, (n, bits) in enumerate(lens):
        cap = kvq.padded_rows(n)
        kc, vc, ks, vs = inputs.random_packed_kv(heads, n, cap, 32, bits, seed=20 + i)
        if bits == 8:  # INT8 codes are about 18x finer: keep K.q scores of the same size
            ks, vs = (ks.float() / 18).half(), (vs.float() / 18).half()
        stores.append(kvq.PackedKV(kc.cuda(), vc.cuda(), ks.cuda(), vs.cuda(), n, bits, 32))
    q = inputs.random_q(300, C, seed=30, std=2.0).cuda()
    out = kvq.packed_kv_attention_mixed(q, stores, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    ranges, start = [], 0
    for st in stores:
        d = _np_store(st)
        ranges.append(dict(start=start, **{k: d[k] for k in ("k_codes", "v_codes", "k_scales", "v_scales", "bits",
                                                               "len")}))
        start += st.n
    ref = oracle.attention_mixed(bits16(q), ranges)
    got = out.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-2
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3


@pytest.mark.slow
def test_mixed_block_full_size_sampled_rows():
    # The mixed-precision block at full size (N = 217,088: text, reference and audio
    # at INT8, generated video at INT4), projected and attended as the benchmark runs
    # it.  The oracle checks sampled token rows of the projection in every segment and
    # sampled query rows of the attention, each exact per row.
    wl = inputs.MIXED
    x, w, qn, kn = inputs.block_inputs(wl, device="cuda")
    n, C = x.shape
    segs = inputs.MIXED_SEGMENTS
    assert sum(sn for _, sn, _ in segs) == n
    stores = [kvq.PackedKV.empty(sn, C, 32, bits, "cuda") for _, sn, bits in segs]
    q = kvq.streamed_qkv_proj_mixed(x, w, stores, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn)
    out = kvq.packed_kv_attention_mixed(q, stores, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    rng = np.random.default_rng(17)
    wb, qn_np, kn_np = bits16(w), qn.cpu().numpy(), kn.cpu().numpy()
    picks, start = [], 0
    for (name, sn, bits), st in zip(segs, stores):
        local = np.unique(np.concatenate([[0, sn - 1], rng.integers(0, sn, 2)]))
        rows = start + local
        picks.append(rows)
        ref = oracle.qkv_proj(bits16(x[torch.as_tensor(rows, device="cuda")]), wb, bits=bits, q_norm_w=qn_np,
                              k_norm_w=kn_np, eps=1e-6)
        xs = x[torch.as_tensor(rows, device="cuda")]
        c = _compare(None, st, ref, local, xs, w, qn, kn, bits=bits, what=name)
        b = head_bounds(bits16(xs), wb, qn_np, kn_np)
        got_q = bits16(q[torch.as_tensor(rows, device="cuda")]).view(np.uint16)
        c.update(check_q(got_q, ref["q_f32"], ref["q_bf16"], b["q"], f"{name} q"))
        print(name, c)
        start += sn
    # attention: the sampled query rows against every key of the four stores
    rows = np.concatenate(picks)
    ranges, start = [], 0
    for st in stores:
        d = _np_store(st)
        ranges.append(dict(start=start, **{k: d[k] for k in ("k_codes", "v_codes", "k_scales", "v_scales", "bits",
                                                               "len")}))
        start += st.n
    ref = oracle.attention_mixed(bits16(q[torch.as_tensor(rows, device="cuda")]), ranges)
    got = out[torch.as_tensor(rows, device="cuda")].cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-2
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3
