"""Routing chosen query rows to a finer store (next row f4).

vram_lab.py's `_exact_av_rows` re-runs the text and audio query rows against a
finer K/V while the video rows stay on the coarse store: audio is a small
part of the sequence and more sensitive, not quantised worse.  Here the finer
path is the INT8 store of every key (the projection's K/V section run once
more into it), and the routed rows attend it with the same kernel.  Checked:
each row equals the oracle on the store it was routed to, and on routed rows
the error against an unquantised fp64 attention drops well below that of the
coarse store."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bits16

pytestmark = pytest.mark.gpu

HD = 128
# (name, tokens, key bits, routed): text and audio query rows take the fine path
SEGS = [("text", 128, 8, True), ("reference", 256, 8, False), ("audio", 64, 8, True), ("video", 576, 4, False)]


def _np(st, start):
    return dict(start=start, len=st.n, bits=st.bits, k_codes=st.k_codes.cpu().numpy(),
                v_codes=st.v_codes.cpu().numpy(), k_scales=bits16(st.k_scales), v_scales=bits16(st.v_scales))


def _run():
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    x, w = x.cuda(), w.cuda()
    n, C = x.shape
    assert sum(s[1] for s in SEGS) == n
    coarse = [kvq.PackedKV.empty(ln, C, 32, b, "cuda") for _, ln, b, _ in SEGS]
    fine = kvq.PackedKV.empty(n, C, 32, 8, "cuda")
    q = kvq.streamed_qkv_proj_mixed(x, w, coarse)
    kvq.streamed_qkv_proj_ex(x, w, [fine], sections=kvq.SECTION_KV)
    out = torch.empty((n, C), dtype=torch.float32, device="cuda")
    start = 0
    for _, ln, _, routed in SEGS:
        qs = q[start:start + ln]
        if routed:
            kvq.packed_kv_attention_mixed(qs, [fine], out_fp32=True, out=out[start:start + ln])
        else:
            kvq.packed_kv_attention_mixed(qs, coarse, out_fp32=True, out=out[start:start + ln])
        start += ln
    coarse_all = kvq.packed_kv_attention_mixed(q, coarse, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    return x, w, q, coarse, fine, out, coarse_all


def test_routed_rows_match_the_oracle_on_their_store():
    x, w, q, coarse, fine, out, _ = _run()
    starts = np.cumsum([0] + [s[1] for s in SEGS])
    coarse_np = [_np(st, int(s0)) for st, s0 in zip(coarse, starts)]
    fine_np = [_np(fine, 0)]
    qb = bits16(q)
    for (name, ln, _, routed), s0 in zip(SEGS, starts):
        rows = np.arange(s0, s0 + ln)
        ref = oracle.attention_mixed(qb, fine_np if routed else coarse_np, rows=rows)
        got = out[int(s0):int(s0) + ln].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(got - ref)) <= 1e-2, name
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3, name


def test_routing_lowers_the_error_of_the_routed_rows():
    x, w, q, coarse, fine, out, coarse_all = _run()
    n, C = x.shape
    # unquantised attention in fp64 from the BF16 inputs (the rotation cancels)
    acc = bits16(x).astype(np.uint32) << 16
    xf = acc.view(np.float32).astype(np.float64)
    wf = (bits16(w).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qkv = xf @ wf.T
    ref = np.empty((n, C))
    for h in range(C // HD):
        Q, K, V = (qkv[:, s * C + h * HD:s * C + (h + 1) * HD] for s in range(3))
        S = Q @ K.T / np.sqrt(HD)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        ref[:, h * HD:(h + 1) * HD] = (P / P.sum(axis=1, keepdims=True)) @ V
    routed = np.concatenate([np.arange(s0, s0 + ln) for (_, ln, _, r), s0 in
                             zip(SEGS, np.cumsum([0] + [s[1] for s in SEGS])) if r])
    e_fine = np.linalg.norm(out.cpu().numpy()[routed] - ref[routed]) / np.linalg.norm(ref[routed])
    e_coarse = np.linalg.norm(coarse_all.cpu().numpy()[routed] - ref[routed]) / np.linalg.norm(ref[routed])
    assert e_fine < 0.5 * e_coarse, (e_fine, e_coarse)
