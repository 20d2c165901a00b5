"""The key-chunk attention for callers that cannot allocate device memory
(packed_kv_attention_partial_static): its carried state lives in the
library's fixed device area instead of caller buffers.

 - CPU: requests larger than the area are refused with KVQ_ERR_TOO_LARGE
   before anything touches the device (the boundary at hidden 7168 is 580
   query rows).
 - GPU, through the C ABI: two sequences of calls in a row (start, merge,
   final), each on its own queries, give the output of the same sequence
   through packed_kv_attention_partial with caller-owned state, within the
   attention's tolerance (max-abs 1e-2, relative L2 5e-3); the second
   sequence shows that the first one's leftovers in the shared area do not
   leak into it.  The first call of the process on the device looks up the
   area's address, so the test passes alone in a fresh process as well as
   after the other tests.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import serving_tcgen05_streamed_gb300 as kvq
from serving_tcgen05_streamed_gb300 import _lib, inputs

MAX_ABS, REL_L2 = 1e-2, 5e-3


def test_requests_beyond_the_area_are_refused():
    lib = kvq.load()
    R, P = _lib._Range, ctypes.c_void_p
    r1 = (R * 1)(R(0, 100, 128, 4, 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20))
    rows_max = kvq.STATIC_STATE_BYTES // ((7168 + 56) * 4)
    assert rows_max == 580
    st = lib.packed_kv_attention_partial_static(P(1 << 20), rows_max + 1, r1, 1, 7168, 32, 0.0, 0, 0, None, None)
    assert st == kvq.KVQ_ERR_TOO_LARGE
    assert "fixed state area" in kvq.status_str(st)
    assert lib.packed_kv_attention_partial_static(P(1 << 20), 0, r1, 1, 7168, 32, 0.0, 0, 0, None, None) \
        == kvq.KVQ_ERR_ARG


def _store(heads, n, seed):
    cap = kvq.padded_rows(n)
    kc, vc, ks, vs = inputs.random_packed_kv(heads, n, cap, 32, 4, seed=seed, device="cuda")
    return kvq.PackedKV(kc, vc, ks, vs, n, 4, 32)


def _static_sequence(lib, q, chunks, out):
    """start, merges, final through the C ABI of the no-allocation entry point"""
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    n_q, C = q.shape
    for i, ch in enumerate(chunks):
        last = i == len(chunks) - 1
        flags = (kvq.PARTIAL_MERGE if i > 0 else 0) | (kvq.PARTIAL_FINAL if last else 0)
        arr = _lib._ranges(ch)
        st = lib.packed_kv_attention_partial_static(ctypes.c_void_p(q.data_ptr()), n_q, arr, len(ch), C, 32, 0.0,
                                                    flags, 1, ctypes.c_void_p(out.data_ptr()) if last else None,
                                                    stream)
        assert st == kvq.KVQ_OK, kvq.status_str(st)


def _caller_state_sequence(q, chunks):
    state = None
    for i, ch in enumerate(chunks):
        last = i == len(chunks) - 1
        r = kvq.packed_kv_attention_partial(q, ch, state=state, merge=i > 0, final=last, out_fp32=True)
        if not last:
            state = r
    return r


def _close(got, ref):
    got, ref = got.double().cpu().numpy(), ref.double().cpu().numpy()
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, (err, rel)
    return err, rel


@pytest.mark.gpu
@pytest.mark.parametrize("heads,n,nq,sizes", [(2, 900, 300, [400, 500]), (56, 3000, 512, [1024, 1024, 952])])
def test_no_alloc_entry_matches_the_caller_state_entry_twice(heads, n, nq, sizes):
    lib = kvq.load()
    st = _store(heads, n, seed=81)
    chunks, a = [], 0
    for ln in sizes:
        chunks.append([st.rows(a, ln)])
        a += ln
    for rep in range(2):  # two sequences in a row, on different queries
        q = inputs.random_q(nq, heads * 128, seed=82 + rep, std=2.0).cuda()
        ref = _caller_state_sequence(q, chunks)
        out = torch.empty((nq, heads * 128), dtype=torch.float32, device="cuda")
        _static_sequence(lib, q, chunks, out)
        torch.cuda.synchronize()
        assert kvq.device_status() == kvq.KVQ_OK
        err, rel = _close(out, ref)
        print(f"sequence {rep}: max-abs {err:.2e}, rel-L2 {rel:.2e} against the caller-state entry point")
