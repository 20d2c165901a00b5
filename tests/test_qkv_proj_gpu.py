"""Parity of the streamed fused QKV projection (tcgen05 GEMM + rotate /
quantise epilogue) with the CPU oracle.

The GEMM accumulates in a different order from the oracle, so results may
differ where the accumulator's error moves a value across a rounding
boundary; tests/_fused_tol.py bounds that error per head vector (the fp32
tensor-core accumulation, then the RMSNorm, RoPE and rotation) and accepts
a differing scale, code or Q value only where the oracle's value lies within
the bound of the boundary it crossed.  The counts of differing values are
printed.  With inputs whose products and sums are exact (one-hot rows),
everything is bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._fused_tol import check_kv, check_q, head_bounds
from tests._util import bits16, to_token_major

pytestmark = pytest.mark.gpu


def _compare(q_gpu, store, ref, rows, x_rows, w, qn=None, kn=None, rot_dim=0, bits=4, group=32, exact=False,
             what=""):
    """Checks the GPU's Q rows `rows` (None: no Q) and store rows against the
    oracle's results `ref` for the same token rows; x_rows: those rows of x."""
    counts = {}
    if exact:
        if q_gpu is not None:
            q = bits16(q_gpu[torch.as_tensor(rows, device=q_gpu.device)]).view(np.uint16)
            assert np.array_equal(q, ref["q_bf16"])
        for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
            got = to_token_major(getattr(store, name), rows)
            assert np.array_equal(got.view(np.uint16) if "scales" in name else got, ref[name]), name
        return counts
    tonp = lambda t: None if t is None else (t.cpu().numpy() if torch.is_tensor(t) else np.asarray(t))  # noqa: E731
    b = head_bounds(bits16(x_rows), bits16(w), tonp(qn), tonp(kn), rot_dim=rot_dim)
    if q_gpu is not None:
        q = bits16(q_gpu[torch.as_tensor(rows, device=q_gpu.device)]).view(np.uint16)
        counts.update(check_q(q, ref["q_f32"], ref["q_bf16"], b["q"], what + " q"))
    for n in ("k", "v"):
        gc = to_token_major(getattr(store, f"{n}_codes"), rows)
        gs = to_token_major(getattr(store, f"{n}_scales"), rows).view(np.uint16)
        c = check_kv(gc, gs, ref[f"{n}_codes"], ref[f"{n}_scales"], ref[f"{n}_rot"], b[n], bits, group,
                     f"{what} {n}")
        counts.update({f"{n}_{k}": v for k, v in c.items()})
    print(f"{what}: {counts}")
    return counts


def _run(x, w, qn=None, kn=None, group=32, chunk=0):
    q, store = kvq.streamed_qkv_proj(x.cuda(), w.cuda(), group=group, chunk_tokens=chunk,
                                     q_norm_w=None if qn is None else qn.cuda(),
                                     k_norm_w=None if kn is None else kn.cuda())
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    return q, store


def test_tiny_block_full():
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    q, store = _run(x, w)
    ref = oracle.qkv_proj(bits16(x), bits16(w))
    _compare(q, store, ref, np.arange(x.shape[0]), x, w, what="tiny block")
    for t in (store.k_codes, store.v_codes):
        assert int(t[:, x.shape[0]:].count_nonzero()) == 0


@pytest.mark.parametrize("group", [32, 64, 128])
def test_one_hot_rows_are_bit_exact(group):
    # x rows = +-2^e * e_k: every accumulator is one exact product, so Q, the
    # codes and the scales must match the oracle bit for bit
    n, C = 700, 768
    g = torch.Generator().manual_seed(group)
    x = torch.zeros((n, C))
    k = torch.randint(0, C, (n,), generator=g)
    sgn = torch.randint(0, 2, (n,), generator=g) * 2 - 1
    e = torch.randint(-3, 4, (n,), generator=g).float()
    x[torch.arange(n), k] = sgn * 2.0 ** e
    x = x.to(torch.bfloat16)
    w = (torch.randn((3 * C, C), generator=g) * 0.1).to(torch.bfloat16)
    q, store = _run(x, w, group=group)
    ref = oracle.qkv_proj(bits16(x), bits16(w), group=group)
    _compare(q, store, ref, np.arange(n), x, w, exact=True)


@pytest.mark.parametrize("n,C", [(1, 256), (129, 384), (1000, 1024)])
def test_ragged_sizes_and_odd_head_counts(n, C):
    g = torch.Generator().manual_seed(n)
    x = torch.randn((n, C), generator=g).to(torch.bfloat16)
    w = (torch.randn((3 * C, C), generator=g) * C ** -0.5).to(torch.bfloat16)
    q, store = _run(x, w)
    ref = oracle.qkv_proj(bits16(x), bits16(w))
    _compare(q, store, ref, np.arange(n), x, w, what=f"n={n} C={C}")


def test_results_do_not_depend_on_chunk_size():
    x, w, _, _ = inputs.block_inputs(inputs.TINY)
    q0, s0 = _run(x, w, chunk=0)
    for chunk in (128, 384, 1000):
        q1, s1 = _run(x, w, chunk=chunk)
        assert torch.equal(q0, q1)
        for a, b in ((s0.k_codes, s1.k_codes), (s0.v_codes, s1.v_codes), (s0.k_scales, s1.k_scales),
                     (s0.v_scales, s1.v_scales)):
            assert torch.equal(a, b)


def test_token_chunks_through_store_windows_match_one_call():
    # the end-to-end path projects token chunks into row windows of one store;
    # rows are independent, so every byte equals the one-call result (ragged last chunk)
    x, w, qn, kn = inputs.block_inputs(inputs.TINY)
    x = x.cuda()
    w = w.cuda()
    n, C = x.shape
    n = n - 37  # a ragged tail
    x = x[:n]
    q0, s0 = kvq.streamed_qkv_proj(x, w)
    store = kvq.PackedKV.empty(n, C, 32, 4, "cuda")
    q1 = torch.empty_like(q0)
    for s in range(0, n, 256):
        ln = min(256, n - s)
        win = store.rows(s, ln)
        assert win.cap == store.cap
        kvq.streamed_qkv_proj_mixed(x[s:s + ln], w, [win], q_out=q1[s:s + ln])
    torch.cuda.synchronize()
    assert torch.equal(q0, q1)
    for a, b in ((s0.k_codes, store.k_codes), (s0.v_codes, store.v_codes), (s0.k_scales, store.k_scales),
                 (s0.v_scales, store.v_scales)):
        assert torch.equal(a[:, :n], b[:, :n])


def test_h3_block_with_rmsnorm_sampled_rows():
    # H3 width (7168, 56 heads), Q/K RMSNorm, chunk 4096; the oracle checks sampled rows
    wl = inputs.MID
    x, w, qn, kn = inputs.block_inputs(wl)
    q, store = _run(x, w, qn, kn, chunk=wl.chunk_tokens)
    rows = inputs.sample_rows(wl.n, 40, seed=4).numpy()
    ref = oracle.qkv_proj(bits16(x), bits16(w), rows, q_norm_w=qn.numpy(), k_norm_w=kn.numpy(), eps=1e-6)
    _compare(q, store, ref, rows, x[torch.as_tensor(rows)], w, qn, kn, what="H3 mid")


@pytest.mark.slow
def test_h3_ref2va_full_size_sampled_rows():
    # the headline size, N = 152,263 (ragged tail of 71 rows), as the benchmark runs it
    wl = inputs.H3_REF2VA
    x, w, qn, kn = inputs.block_inputs(wl, device="cuda")
    q, store = kvq.streamed_qkv_proj(x, w, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    rows = inputs.sample_rows(wl.n, 24, seed=5).numpy()
    xs = x[torch.as_tensor(rows, device="cuda")]  # rows are independent: the oracle sees only the samples
    ref = oracle.qkv_proj(bits16(xs), bits16(w), q_norm_w=qn.cpu().numpy(), k_norm_w=kn.cpu().numpy())
    _compare(q, store, ref, rows, xs, w, qn, kn, what="H3 Ref2VA")
    # pad rows of the last tile are zero
    assert int(store.k_codes[:, wl.n:].count_nonzero()) == 0
