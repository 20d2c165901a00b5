"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/kvq.h declares, its size helpers reproduce the pages'
memory arithmetic, and argument errors are reported before any launch."""
import ctypes
import os
import re

import pytest

import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GiB = 2.0 ** 30


def _declared():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))


def test_library_exports_every_declared_symbol():
    lib = kvq.load()
    declared = _declared()
    assert declared == set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert "sm_103a" in kvq.version()


def _golden():
    vals = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "pages_memory_arithmetic.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            name, v, tol = line.split()
            vals[name] = (float(v), float(tol))
    return vals


def test_store_sizes_reproduce_the_pages_memory_arithmetic():
    g = _golden()
    n, C = int(g["tokens"][0]), int(g["hidden"][0])
    cap = kvq.padded_rows(n)
    assert cap == 152320 and cap % 128 == 0 and cap - n < 128
    bf16_qkv = n * 3 * C * 2 / GiB
    q = n * C * 2 / GiB
    k = kvq.codes_bytes(cap, C, 4) / GiB
    v = kvq.codes_bytes(cap, C, 4) / GiB
    for name, val in (("bf16_qkv", bf16_qkv), ("q_bf16", q), ("k_4bit", k), ("v_4bit", v),
                      ("qkv_packed_total", q + k + v)):
        ref, tol = g[name]
        assert abs(val - ref) <= tol, (name, val, ref)
    # metadata: one fp16 scale per 32 elements per K and V
    assert kvq.scales_bytes(cap, C, 32) == 56 * cap * 4 * 2
    assert kvq.scales_bytes(cap, C, 128) == 56 * cap * 2
    assert kvq.codes_bytes(cap, C, 8) == 2 * kvq.codes_bytes(cap, C, 4)
    # invalid arguments give 0
    assert kvq.codes_bytes(cap, 100, 4) == 0 and kvq.scales_bytes(cap, C, 48) == 0


def test_status_strings():
    assert kvq.status_str(kvq.KVQ_OK) == "ok"
    assert "timed out" in kvq.status_str(kvq.KVQ_ERR_TIMEOUT)
    assert kvq.status_str(99) == "unknown status"


def test_argument_errors_are_reported_before_any_launch():
    lib = kvq.load()
    a16 = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation first
    odd = ctypes.c_void_p((1 << 20) + 8)
    S = None
    # null pointers / bad sizes
    assert lib.kv_rotate_quant_pack(None, 10, 1024, 2048, 32, 4, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.kv_rotate_quant_pack(a16, 0, 1024, 2048, 32, 4, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.kv_rotate_quant_pack(a16, 10, 1000, 2048, 32, 4, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.kv_rotate_quant_pack(a16, 10, 1024, 2048, 48, 4, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.kv_rotate_quant_pack(a16, 10, 1024, 2048, 32, 2, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.kv_rotate_quant_pack(a16, 10, 1024, 2000, 32, 4, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ARG
    # alignment
    assert lib.kv_rotate_quant_pack(odd, 10, 1024, 2048, 32, 4, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ALIGN
    assert lib.kv_rotate_quant_pack(a16, 10, 1024, 2052, 32, 4, a16, a16, a16, a16, S) == kvq.KVQ_ERR_ALIGN
    assert lib.kv_unpack(a16, a16, a16, None, 10, 1024, 32, 4, a16, 2048, S) == kvq.KVQ_ERR_ARG
    # projection
    P = ctypes.c_void_p
    assert lib.streamed_qkv_proj(a16, a16, 0, 1024, 32, 0, None, None, 1e-6, P(2 << 20), a16, a16, a16, a16, S) \
        == kvq.KVQ_ERR_ARG
    assert lib.streamed_qkv_proj(a16, a16, 10, 1024, 32, -1, None, None, 1e-6, P(2 << 20), a16, a16, a16, a16, S) \
        == kvq.KVQ_ERR_ARG
    assert lib.streamed_qkv_proj(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, a16, a16, a16, a16, a16, S) \
        == kvq.KVQ_ERR_ARG  # q_out aliases x
    assert lib.streamed_qkv_proj(a16, odd, 10, 1024, 32, 0, None, None, 1e-6, P(2 << 20), a16, a16, a16, a16, S) \
        == kvq.KVQ_ERR_ALIGN
    # attention
    assert lib.packed_kv_attention(a16, 10, a16, a16, a16, a16, 0, 1024, 32, 0.0, 0, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.packed_kv_attention(a16, 10, a16, a16, a16, a16, 5, 1024, 32, 0.0, 2, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.packed_kv_attention(a16, 10, a16, a16, a16, a16, 5, 1024, 32, 0.0, 1, a16, S) == kvq.KVQ_ERR_ARG
    assert lib.packed_kv_attention(a16, 10, a16, odd, a16, a16, 5, 1024, 32, 0.0, 0, a16, S) == kvq.KVQ_ERR_ALIGN
    # RoPE: rot_dim 64 or 128 only, 16-byte aligned table
    R1 = (_lib._Range * 1)(_lib._Range(0, 10, 128, 4, 0, a16.value, a16.value, a16.value, a16.value))
    assert lib.streamed_qkv_proj_ex(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, a16, 32, 3, P(2 << 20), R1, 1, S) \
        == kvq.KVQ_ERR_UNSUPPORTED
    assert lib.streamed_qkv_proj_ex(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, odd, 128, 3, P(2 << 20), R1, 1, S) \
        == kvq.KVQ_ERR_ALIGN
    assert lib.streamed_qkv_proj_ex(None, a16, 10, 1024, 32, 0, None, None, 1e-6, a16, 128, 3, P(2 << 20), R1, 1, S) \
        == kvq.KVQ_ERR_ARG
    # sections: 1..3 only; Q-only needs no ranges, K/V-only no q_out
    assert lib.streamed_qkv_proj_ex(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, None, 0, 0, P(2 << 20), R1, 1, S) \
        == kvq.KVQ_ERR_ARG
    assert lib.streamed_qkv_proj_ex(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, None, 0, 4, P(2 << 20), R1, 1, S) \
        == kvq.KVQ_ERR_ARG
    assert lib.streamed_qkv_proj_ex(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, None, 0, 1, None, R1, 1, S) \
        == kvq.KVQ_ERR_ARG  # Q asked for, no q_out
    assert lib.streamed_qkv_proj_ex(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, None, 0, 2, None, None, 0, S) \
        == kvq.KVQ_ERR_ARG  # K/V asked for, no ranges
    # causal: a negative query position, and the checks it shares
    assert lib.packed_kv_attention_causal(a16, 10, -1, a16, a16, a16, a16, 5, 1024, 32, 0.0, 0, a16, S) \
        == kvq.KVQ_ERR_ARG
    assert lib.packed_kv_attention_causal(a16, 10, 0, a16, a16, a16, a16, 0, 1024, 32, 0.0, 0, a16, S) \
        == kvq.KVQ_ERR_ARG
    assert lib.packed_kv_attention_causal(a16, 10, 0, a16, odd, a16, a16, 5, 1024, 32, 0.0, 0, a16, S) \
        == kvq.KVQ_ERR_ALIGN
    # mixed range tables: gaps, bad bits, capacity
    R = _lib._Range
    bad_gap = (R * 2)(R(0, 100, 128, 4, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20),
                      R(101, 50, 128, 8, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20))
    assert lib.packed_kv_attention_mixed(a16, 10, bad_gap, 2, 1024, 32, 0.0, 0, P(2 << 20), S) == kvq.KVQ_ERR_ARG
    bad_bits = (R * 1)(R(0, 100, 128, 6, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20))
    assert lib.packed_kv_attention_mixed(a16, 10, bad_bits, 1, 1024, 32, 0.0, 0, P(2 << 20), S) == kvq.KVQ_ERR_ARG
    bad_cap = (R * 1)(R(0, 100, 100, 4, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20))
    assert lib.packed_kv_attention_mixed(a16, 10, bad_cap, 1, 1024, 32, 0.0, 0, P(2 << 20), S) == kvq.KVQ_ERR_ARG
    too_many = (R * 17)()
    assert lib.packed_kv_attention_mixed(a16, 10, too_many, 17, 1024, 32, 0.0, 0, P(2 << 20), S) == kvq.KVQ_ERR_ARG
    gap_proj = (R * 2)(R(0, 5, 128, 4, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20),
                       R(5, 4, 128, 8, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20))
    assert lib.streamed_qkv_proj_mixed(a16, a16, 10, 1024, 32, 0, None, None, 1e-6, P(2 << 20), gap_proj, 2, S) \
        == kvq.KVQ_ERR_ARG
    assert lib.kvq_selftest_wait_timeout(0, S) == kvq.KVQ_ERR_ARG
    # attention over a key chunk with a carried state
    ok1 = (R * 1)(R(0, 100, 128, 4, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20))
    acc, lse, out = P(4 << 20), P(6 << 20), P(8 << 20)
    part = lib.packed_kv_attention_partial
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 4, acc, lse, 0, out, S) == kvq.KVQ_ERR_ARG  # flags
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, -1, acc, lse, 0, out, S) == kvq.KVQ_ERR_ARG
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 0, None, lse, 0, None, S) == kvq.KVQ_ERR_ARG  # no state to start
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 1, acc, None, 0, None, S) == kvq.KVQ_ERR_ARG  # no state to merge
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 3, acc, lse, 0, None, S) == kvq.KVQ_ERR_ARG  # final, no out
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 0, a16, lse, 0, None, S) == kvq.KVQ_ERR_ARG  # state aliases q
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 3, acc, lse, 0, acc, S) == kvq.KVQ_ERR_ARG  # state aliases out
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 3, acc, lse, 1, a16, S) == kvq.KVQ_ERR_ARG  # fp32 over q
    assert part(a16, 10, ok1, 1, 1024, 32, 0.0, 0, P((4 << 20) + 4), lse, 0, None, S) == kvq.KVQ_ERR_ALIGN
    assert part(a16, 10, bad_gap, 2, 1024, 32, 0.0, 0, acc, lse, 0, None, S) == kvq.KVQ_ERR_ARG
    assert part(a16, 0, ok1, 1, 1024, 32, 0.0, 0, acc, lse, 0, None, S) == kvq.KVQ_ERR_ARG


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kvq.kv_rotate_quant_pack(x, 128)


def test_store_row_window_keeps_the_head_stride():
    # a row window shares the store's memory and reports the whole store's rows per
    # head, which the range-table calls take as the head stride
    st = kvq.PackedKV.empty(1000, 512, 32, 4, "cpu")
    assert st.cap == kvq.padded_rows(1000) == 1024
    win = st.rows(256, 300)
    assert win.n == 300 and win.cap == 1024 and win.heads == 4
    assert win.k_codes.data_ptr() - st.k_codes.data_ptr() == 256 * 64
    assert win.k_scales.data_ptr() - st.k_scales.data_ptr() == 256 * 4 * 2
    win.v_codes[1, 0, 0] = 7
    assert st.v_codes[1, 256, 0] == 7


def test_range_scales_need_only_row_alignment():
    # a window may start at any row: scales pointers are checked against one
    # scales row (2 * 128 / group bytes), codes pointers against 16 bytes
    lib = kvq.load()
    R, P = _lib._Range, ctypes.c_void_p
    base = 1 << 20
    # (acceptance of row-aligned windows needs a launch: the GPU tests attend windows at odd rows)
    for group, row in ((32, 8), (64, 4), (128, 2)):
        bad = (R * 1)(R(0, 100, 128, 4, 0, base, base, base + row // 2, base))
        badc = (R * 1)(R(0, 100, 128, 4, 0, base + 8, base, base, base))
        assert lib.packed_kv_attention_partial(P(4 << 20), 10, bad, 1, 1024, group, 0.0, 0, P(6 << 20),
                                               P(8 << 20), 0, None, None) == kvq.KVQ_ERR_ALIGN
        assert lib.packed_kv_attention_partial(P(4 << 20), 10, badc, 1, 1024, group, 0.0, 0, P(6 << 20),
                                               P(8 << 20), 0, None, None) == kvq.KVQ_ERR_ALIGN
