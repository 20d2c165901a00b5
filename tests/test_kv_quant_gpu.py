"""Parity of the standalone rotate + quantise + pack kernel (and its inverse)
with the CPU oracle: codes and scales must be bit-exact, pad rows zero."""
import numpy as np
import pytest
import torch

import oracle
import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import inputs
from tests._util import bits16, to_token_major

pytestmark = pytest.mark.gpu


def _check_store(store, kv_cpu, hidden, group, bits, rows=None):
    n = kv_cpu.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    kc, vc, ks, vs = oracle.kv_rotate_quant_pack(bits16(kv_cpu[rows]), hidden=hidden, group=group, bits=bits)
    assert np.array_equal(to_token_major(store.k_codes, rows), kc)
    assert np.array_equal(to_token_major(store.v_codes, rows), vc)
    assert np.array_equal(to_token_major(store.k_scales, rows).view(np.uint16), ks)
    assert np.array_equal(to_token_major(store.v_scales, rows).view(np.uint16), vs)
    # rows n .. cap-1 are zero
    for t in (store.k_codes, store.v_codes, store.k_scales, store.v_scales):
        assert int(t[:, n:].view(torch.uint8).count_nonzero()) == 0
    return kc, vc, ks, vs


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("n,hidden", [(1000, 1024), (1, 256), (129, 384), (7, 256), (127, 256), (128, 256),
                                      (255, 256)])
def test_pack_bit_exact(n, hidden, group, bits):
    # a block of the kernel covers 128 tokens in 16 passes of 8 and prefetches the next
    # pass's rows: sizes below, at and past one block and one pass, with ragged tails
    kv = inputs.sweep_kv(n, hidden, seed=n + group + bits)
    store = kvq.kv_rotate_quant_pack(kv.cuda(), hidden, group, bits)
    torch.cuda.synchronize()
    assert store.cap == kvq.padded_rows(n)
    _check_store(store, kv, hidden, group, bits)


def test_pack_strided_input_and_extreme_values():
    # K/V as a column slice of a wider [n, 3C] buffer (ld = 3C), with zero
    # rows, spikes, tiny and large values: zero groups, subnormal scales
    n, C = 300, 512
    qkv = torch.randn((n, 3 * C), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    qkv[0] = 0
    qkv[1, C:] = 0
    qkv[1, C + 7] = 3.0
    qkv[2, C:] *= 1e-6
    qkv[3, C:] *= 2.0 ** -30
    qkv[4, C:] *= 3e3
    g = qkv.cuda()
    store = kvq.kv_rotate_quant_pack(g[:, C:], C, 32, 4)
    torch.cuda.synchronize()
    _check_store(store, qkv[:, C:].contiguous(), C, 32, 4)


def test_pack_h3_width_full():
    # the H3 width (2 x 7168) with heavy-tailed channels, every row
    n, C = 4096, 7168
    kv = inputs.sweep_kv(n, C, seed=1)
    store = kvq.kv_rotate_quant_pack(kv.cuda(), C, 32, 4)
    torch.cuda.synchronize()
    _check_store(store, kv, C, 32, 4)


@pytest.mark.parametrize("group,bits", [(32, 4), (128, 4), (64, 8), (128, 8)])
def test_pack_sweep_max_size_sampled(group, bits):
    # the largest sweep size, N = 262,144, sampled rows (rows are independent)
    n, C = 262144, 7168
    kv = inputs.sweep_kv(n, C, seed=2, device="cuda")
    store = kvq.kv_rotate_quant_pack(kv, C, group, bits)
    torch.cuda.synchronize()
    rows = inputs.sample_rows(n, 256, seed=3).numpy()
    kc, vc, ks, vs = oracle.kv_rotate_quant_pack(bits16(kv[torch.as_tensor(rows, device="cuda")]), hidden=C,
                                                 group=group, bits=bits)
    assert np.array_equal(to_token_major(store.k_codes, rows), kc)
    assert np.array_equal(to_token_major(store.v_codes, rows), vc)
    assert np.array_equal(to_token_major(store.k_scales, rows).view(np.uint16), ks)
    assert np.array_equal(to_token_major(store.v_scales, rows).view(np.uint16), vs)
    # and back: the unpack of the whole store, the same sampled rows
    del kv
    out = kvq.kv_unpack(store, C)
    torch.cuda.synchronize()
    got = bits16(out[torch.as_tensor(rows, device="cuda")])
    assert np.array_equal(got, oracle.kv_unpack(kc, vc, ks, vs, group=group, bits=bits))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("n", [333, 9, 128])
def test_unpack_bit_exact(group, bits, n):
    C = 768
    kv = inputs.sweep_kv(n, C, seed=7)
    store = kvq.kv_rotate_quant_pack(kv.cuda(), C, group, bits)
    out = kvq.kv_unpack(store, C)
    torch.cuda.synchronize()
    kc, vc, ks, vs = oracle.kv_rotate_quant_pack(bits16(kv), hidden=C, group=group, bits=bits)
    ref = oracle.kv_unpack(kc, vc, ks, vs, group=group, bits=bits)
    assert np.array_equal(bits16(out), ref)


@pytest.mark.parametrize("pad", [0, 8, 16])
def test_pack_and_unpack_strided_rows(pad):
    # rows of 2C + pad BF16: pad 0 and 16 keep them 32-byte aligned (32-byte loads and
    # stores), pad 8 does not (16-byte forms); all give the same bits
    n, C = 300, 512
    kv = inputs.sweep_kv(n, C, seed=11)
    wide_in = torch.zeros((n, 2 * C + pad), dtype=torch.bfloat16)
    wide_in[:, :2 * C] = kv
    store = kvq.kv_rotate_quant_pack(wide_in.cuda()[:, :2 * C], C, 32, 8)
    wide_out = torch.empty((n, 2 * C + pad), dtype=torch.bfloat16, device="cuda")
    out = kvq.kv_unpack(store, C, out=wide_out[:, :2 * C])
    torch.cuda.synchronize()
    kc, vc, ks, vs = _check_store(store, kv, C, 32, 8)
    assert np.array_equal(bits16(out), oracle.kv_unpack(kc, vc, ks, vs, group=32, bits=8))


def test_pack_is_deterministic_and_stream_ordered():
    n, C = 2048, 1024
    kv = inputs.sweep_kv(n, C, seed=9).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = kvq.kv_rotate_quant_pack(kv, C, 32, 4, stream=s)
        b = kvq.kv_rotate_quant_pack(kv, C, 32, 4, stream=s)
    s.synchronize()
    assert torch.equal(a.k_codes, b.k_codes) and torch.equal(a.v_scales, b.v_scales)
    assert kvq.device_status() == kvq.KVQ_OK
