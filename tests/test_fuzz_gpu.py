"""Randomised parity sweeps with fixed seeds.  Each case draws its shapes and
options (token and key counts, head counts, groups, precisions, input strides,
range tables, query positions, key chunkings, projection chunk sizes) from a
seeded generator and compares the CUDA path with the oracle under the bars of
the dedicated tests: bit-exact codes and scales for the standalone pack,
max-abs 1e-2 and relative L2 5e-3 for the attention's fp32 output, and the
accumulator-error bound of tests/_fused_tol.py for the fused projection."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bits16, to_token_major
from tests.test_qkv_proj_gpu import _compare

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 5e-3


def _rng(kind, seed):
    return np.random.default_rng([zlib.crc32(kind.encode()), seed])


def _assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    print(f"{what}: max-abs {err:.2e} rel-L2 {rel:.2e}")
    assert err <= MAX_ABS, (what, err)
    assert rel <= REL_L2, (what, rel)


def _store(heads, n, group, bits, seed):
    cap = kvq.padded_rows(n)
    kc, vc, ks, vs = inputs.random_packed_kv(heads, n, cap, group, bits, seed=seed, device="cuda")
    if bits == 8:  # INT8 codes are about 18x finer: keep K.q scores and V of the INT4 stores' size
        ks, vs = (ks.float() / 18).half(), (vs.float() / 18).half()
    return kvq.PackedKV(kc, vc, ks, vs, n, bits, group)


def _ranges(stores):
    rs, start = [], 0
    for st in stores:
        rs.append(dict(start=start, len=st.n, bits=st.bits, k_codes=st.k_codes.cpu().numpy(),
                       v_codes=st.v_codes.cpu().numpy(), k_scales=bits16(st.k_scales), v_scales=bits16(st.v_scales)))
        start += st.n
    return rs


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_pack(seed):
    r = _rng("pack", seed)
    n = int(r.integers(1, 900))
    heads = int(r.integers(1, 7))
    C = 128 * heads
    group = int(r.choice([32, 64, 128]))
    bits = int(r.choice([4, 8]))
    pad = int(r.choice([0, 8, 64, 136]))  # extra columns: the K/V rows have a stride of 2C + pad
    kv = inputs.sweep_kv(n, C, seed=1000 + seed)
    wide = torch.zeros((n, 2 * C + pad), dtype=torch.bfloat16)
    wide[:, :2 * C] = kv
    store = kvq.kv_rotate_quant_pack(wide.cuda()[:, :2 * C], C, group, bits)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    kc, vc, ks, vs = oracle.kv_rotate_quant_pack(bits16(kv), hidden=C, group=group, bits=bits)
    rows = np.arange(n)
    assert np.array_equal(to_token_major(store.k_codes, rows), kc)
    assert np.array_equal(to_token_major(store.v_codes, rows), vc)
    assert np.array_equal(to_token_major(store.k_scales, rows).view(np.uint16), ks)
    assert np.array_equal(to_token_major(store.v_scales, rows).view(np.uint16), vs)
    for t in (store.k_codes, store.v_codes, store.k_scales, store.v_scales):
        assert int(t[:, n:].view(torch.uint8).count_nonzero()) == 0
    # the output with the same padded row stride: 32-byte aligned rows take the 32-byte stores,
    # others the interleaved 16-byte form
    wide_out = torch.empty((n, 2 * C + pad), dtype=torch.bfloat16, device="cuda")
    out = kvq.kv_unpack(store, C, out=wide_out[:, :2 * C])
    torch.cuda.synchronize()
    assert np.array_equal(bits16(out), oracle.kv_unpack(kc, vc, ks, vs, group=group, bits=bits))


@pytest.mark.parametrize("seed", range(10))
def test_fuzz_attention(seed):
    r = _rng("attention", seed)
    heads = int(r.integers(1, 4))
    n_kv = int(r.integers(1, 1500))
    n_q = int(r.integers(1, 700))
    group = int(r.choice([32, 64, 128]))
    st = _store(heads, n_kv, group, 4, seed=2000 + seed)
    q = inputs.random_q(n_q, heads * 128, seed=3000 + seed, std=float(r.uniform(0.5, 3.0))).cuda()
    out = kvq.packed_kv_attention(q, st, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    ref = oracle.attention(bits16(q), st.k_codes.cpu().numpy(), st.v_codes.cpu().numpy(), bits16(st.k_scales),
                           bits16(st.v_scales), n_kv=n_kv, group=group, bits=4)
    _assert_close(out.cpu().numpy(), ref, f"heads={heads} n_q={n_q} n_kv={n_kv} G={group}")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_mixed_ranges(seed):
    r = _rng("mixed", seed)
    heads = int(r.integers(1, 3))
    stores = [_store(heads, int(r.integers(1, 500)), 32, int(r.choice([4, 8])), seed=4000 + 10 * seed + i)
              for i in range(int(r.integers(2, 5)))]
    q = inputs.random_q(int(r.integers(1, 400)), heads * 128, seed=5000 + seed, std=2.0).cuda()
    out = kvq.packed_kv_attention_mixed(q, stores, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    ref = oracle.attention_mixed(bits16(q), _ranges(stores))
    _assert_close(out.cpu().numpy(), ref, f"ranges {[(s.n, s.bits) for s in stores]}")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_causal(seed):
    r = _rng("causal", seed)
    heads = int(r.integers(1, 3))
    n_kv = int(r.integers(1, 1200))
    n_q = int(r.integers(1, 600))
    q_pos0 = int(r.integers(0, n_kv + 1))
    st = _store(heads, n_kv, 32, 4, seed=6000 + seed)
    q = inputs.random_q(n_q, heads * 128, seed=7000 + seed, std=2.0).cuda()
    out = kvq.packed_kv_attention_causal(q, st, q_pos0=q_pos0, out_fp32=True)
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    ref = oracle.attention_causal(bits16(q), st.k_codes.cpu().numpy(), st.v_codes.cpu().numpy(),
                                  bits16(st.k_scales), bits16(st.v_scales), n_kv=n_kv, q_pos0=q_pos0, group=32, bits=4)
    _assert_close(out.cpu().numpy(), ref, f"n_q={n_q} n_kv={n_kv} q_pos0={q_pos0}")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_key_chunks(seed):
    r = _rng("chunks", seed)
    heads = int(r.integers(1, 3))
    n_chunks = int(r.integers(2, 5))
    sizes = [int(x) for x in r.integers(1, 400, size=n_chunks)]
    bits = [int(b) for b in r.choice([4, 8], size=n_chunks)]
    chunks = [[_store(heads, n, 32, b, seed=8000 + 10 * seed + i)] for i, (n, b) in enumerate(zip(sizes, bits))]
    q = inputs.random_q(int(r.integers(1, 400)), heads * 128, seed=9000 + seed, std=2.0).cuda()
    state = None
    for i, ch in enumerate(chunks):
        last = i == n_chunks - 1
        res = kvq.packed_kv_attention_partial(q, ch, state=state, merge=i > 0, final=last, out_fp32=True)
        if not last:
            state = res
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    got = res.cpu().numpy()
    what = f"chunks {list(zip(sizes, bits))}"
    _assert_close(got, oracle.attention_blockwise(bits16(q), [_ranges(ch) for ch in chunks]), what + " blockwise")
    _assert_close(got, oracle.attention_mixed(bits16(q), _ranges([c[0] for c in chunks])), what + " one call")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_projection(seed):
    r = _rng("projection", seed)
    n = int(r.integers(1, 600))
    heads = int(r.integers(1, 4))
    C = 128 * heads
    group = int(r.choice([32, 64, 128]))
    chunk = int(r.choice([0, 128, 256, 384]))
    norm = bool(r.integers(0, 2))
    g = torch.Generator().manual_seed(10000 + seed)
    x = torch.randn((n, C), generator=g).to(torch.bfloat16)
    w = (torch.randn((3 * C, C), generator=g) * C ** -0.5).to(torch.bfloat16)
    qn = (1.0 + 0.1 * torch.randn((128,), generator=g)) if norm else None
    kn = (1.0 + 0.1 * torch.randn((128,), generator=g)) if norm else None
    q, store = kvq.streamed_qkv_proj(x.cuda(), w.cuda(), group=group, chunk_tokens=chunk,
                                     q_norm_w=None if qn is None else qn.cuda(),
                                     k_norm_w=None if kn is None else kn.cuda())
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK
    ref = oracle.qkv_proj(bits16(x), bits16(w), group=group, q_norm_w=None if qn is None else qn.numpy(),
                          k_norm_w=None if kn is None else kn.numpy())
    _compare(q, store, ref, np.arange(n), x, w, qn, kn, group=group,
             what=f"n={n} C={C} G={group} chunk={chunk} norm={norm}")
