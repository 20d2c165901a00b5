"""ctypes binding of libkvq.so (include/kvq.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch is used for device memory and streams.  There is no CPU
fallback: if the library is missing or cannot be loaded, calls raise.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import torch

from . import build as _build

HEAD_DIM = 128
ROW_TILE = 128
MAX_RANGES = 16

KVQ_OK, KVQ_ERR_ARG, KVQ_ERR_ALIGN, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CUDA, KVQ_ERR_TIMEOUT, KVQ_ERR_TOO_LARGE = range(7)
STATIC_STATE_BYTES = 16 << 20

#: Every function the header declares.
EXPORTS = (
    "kvq_status_str", "kvq_version", "kvq_padded_rows", "kvq_codes_bytes", "kvq_scales_bytes",
    "kv_rotate_quant_pack", "kv_unpack", "streamed_qkv_proj", "packed_kv_attention",
    "packed_kv_attention_causal", "streamed_qkv_proj_mixed", "streamed_qkv_proj_ex", "packed_kv_attention_mixed",
    "packed_kv_attention_partial", "packed_kv_attention_partial_static", "kvq_device_status",
    "kvq_selftest_wait_timeout",
)


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})")


class _Range(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int64), ("len", ctypes.c_int64), ("cap", ctypes.c_int64),
                ("bits", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads libkvq.so (building it with nvcc first if it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; run serving_tcgen05_streamed_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, I64, I, F, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.kvq_status_str.restype = ctypes.c_char_p
        lib.kvq_status_str.argtypes = [I]
        lib.kvq_version.restype = ctypes.c_char_p
        lib.kvq_version.argtypes = []
        lib.kvq_padded_rows.restype = I64
        lib.kvq_padded_rows.argtypes = [I64]
        lib.kvq_codes_bytes.restype = S
        lib.kvq_codes_bytes.argtypes = [I64, I, I]
        lib.kvq_scales_bytes.restype = S
        lib.kvq_scales_bytes.argtypes = [I64, I, I]
        lib.kv_rotate_quant_pack.restype = I
        lib.kv_rotate_quant_pack.argtypes = [P, I64, I, I64, I, I, P, P, P, P, P]
        lib.kv_unpack.restype = I
        lib.kv_unpack.argtypes = [P, P, P, P, I64, I, I, I, P, I64, P]
        lib.streamed_qkv_proj.restype = I
        lib.streamed_qkv_proj.argtypes = [P, P, I64, I, I, I64, P, P, F, P, P, P, P, P, P]
        lib.packed_kv_attention.restype = I
        lib.packed_kv_attention.argtypes = [P, I64, P, P, P, P, I64, I, I, F, I, P, P]
        lib.packed_kv_attention_causal.restype = I
        lib.packed_kv_attention_causal.argtypes = [P, I64, I64, P, P, P, P, I64, I, I, F, I, P, P]
        lib.streamed_qkv_proj_mixed.restype = I
        lib.streamed_qkv_proj_mixed.argtypes = [P, P, I64, I, I, I64, P, P, F, P, ctypes.POINTER(_Range), I, P]
        lib.streamed_qkv_proj_ex.restype = I
        lib.streamed_qkv_proj_ex.argtypes = [P, P, I64, I, I, I64, P, P, F, P, I, I, P, ctypes.POINTER(_Range), I, P]
        lib.packed_kv_attention_mixed.restype = I
        lib.packed_kv_attention_mixed.argtypes = [P, I64, ctypes.POINTER(_Range), I, I, I, F, I, P, P]
        lib.packed_kv_attention_partial.restype = I
        lib.packed_kv_attention_partial.argtypes = [P, I64, ctypes.POINTER(_Range), I, I, I, F, I, P, P, I, P, P]
        lib.packed_kv_attention_partial_static.restype = I
        lib.packed_kv_attention_partial_static.argtypes = [P, I64, ctypes.POINTER(_Range), I, I, I, F, I, I, P, P]
        lib.kvq_device_status.restype = I
        lib.kvq_device_status.argtypes = [P]
        lib.kvq_selftest_wait_timeout.restype = I
        lib.kvq_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P]
        _lib = lib
        return lib


def status_str(status: int) -> str:
    return load().kvq_status_str(int(status)).decode()


def version() -> str:
    return load().kvq_version().decode()


def padded_rows(n: int) -> int:
    return int(load().kvq_padded_rows(int(n)))


def codes_bytes(cap: int, hidden: int, bits: int = 4) -> int:
    return int(load().kvq_codes_bytes(int(cap), int(hidden), int(bits)))


def scales_bytes(cap: int, hidden: int, group: int = 32) -> int:
    return int(load().kvq_scales_bytes(int(cap), int(hidden), int(group)))


def _check(status: int, what: str):
    if status != KVQ_OK:
        raise KvqError(status, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _whole_store(store: "PackedKV", what: str):
    # the single-store calls take the head stride from n; a row window (PackedKV.rows)
    # goes through the range-table calls, which take it explicitly
    if store.cap != padded_rows(store.n):
        raise ValueError(f"{what}: store rows per head {store.cap} != padded_rows(n) {padded_rows(store.n)}; "
                         "pass row windows to the *_mixed calls")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (the library has no CPU path)")


@dataclasses.dataclass
class PackedKV:
    """K and V packed stores of one token range (head-major; see kvq.h)."""
    k_codes: torch.Tensor   # uint8 [heads, cap, 128*bits/8]
    v_codes: torch.Tensor
    k_scales: torch.Tensor  # float16 [heads, cap, 128/group]
    v_scales: torch.Tensor
    n: int
    bits: int = 4
    group: int = 32

    @property
    def cap(self) -> int:
        """Rows per head in memory (the head stride), also for a row window."""
        return self.k_codes.stride(0) // self.k_codes.stride(1)

    def rows(self, start: int, length: int) -> "PackedKV":
        """Window of `length` token rows starting at `start` of every head, sharing
        this store's memory (a projection over a token chunk writes into it)."""
        assert 0 <= start and start + length <= self.n
        sl = lambda t: t[:, start:start + length]  # noqa: E731
        return PackedKV(sl(self.k_codes), sl(self.v_codes), sl(self.k_scales), sl(self.v_scales), length, self.bits,
                        self.group)

    @property
    def heads(self) -> int:
        return self.k_codes.shape[0]

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.k_codes, self.v_codes, self.k_scales, self.v_scales))

    @staticmethod
    def empty(n: int, hidden: int, group: int = 32, bits: int = 4, device="cuda", cap: int | None = None):
        heads = hidden // HEAD_DIM
        cap = padded_rows(n) if cap is None else cap
        cb = HEAD_DIM * bits // 8
        mk = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        return PackedKV(mk((heads, cap, cb), torch.uint8), mk((heads, cap, cb), torch.uint8),
                        mk((heads, cap, HEAD_DIM // group), torch.float16),
                        mk((heads, cap, HEAD_DIM // group), torch.float16), n, bits, group)


# ---------------------------------------------------------------------- calls (names follow the C ABI)
def kv_rotate_quant_pack(kv: torch.Tensor, hidden: int, group: int = 32, bits: int = 4,
                         out: PackedKV | None = None, stream=None) -> PackedKV:
    """BF16 K/V [n, >= 2*hidden] (row stride kv.stride(0)) -> packed store."""
    _need_cuda(kv)
    assert kv.dtype == torch.bfloat16 and kv.dim() == 2 and kv.stride(1) == 1
    n = kv.shape[0]
    out = PackedKV.empty(n, hidden, group, bits, kv.device) if out is None else out
    _whole_store(out, "kv_rotate_quant_pack")
    st = load().kv_rotate_quant_pack(_ptr(kv), n, hidden, kv.stride(0), group, bits, _ptr(out.k_codes),
                                     _ptr(out.v_codes), _ptr(out.k_scales), _ptr(out.v_scales), _stream(stream))
    _check(st, "kv_rotate_quant_pack")
    return out


def kv_unpack(store: PackedKV, hidden: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Packed store -> BF16 K/V [n, 2*hidden] (diagnostic; materialises K/V)."""
    _need_cuda(store.k_codes)
    _whole_store(store, "kv_unpack")
    n = store.n
    out = torch.empty((n, 2 * hidden), dtype=torch.bfloat16, device=store.k_codes.device) if out is None else out
    st = load().kv_unpack(_ptr(store.k_codes), _ptr(store.v_codes), _ptr(store.k_scales), _ptr(store.v_scales), n,
                          hidden, store.group, store.bits, _ptr(out), out.stride(0), _stream(stream))
    _check(st, "kv_unpack")
    return out


def streamed_qkv_proj(x: torch.Tensor, w_qkv: torch.Tensor, group: int = 32, chunk_tokens: int = 0,
                      q_norm_w: torch.Tensor | None = None, k_norm_w: torch.Tensor | None = None,
                      eps: float = 1e-6, q_out: torch.Tensor | None = None, store: PackedKV | None = None,
                      stream=None):
    """x BF16 [n, C], w_qkv BF16 [3C, C] -> (q_rot BF16 [n, C], PackedKV INT4)."""
    _need_cuda(x, w_qkv, q_norm_w, k_norm_w)
    n, C = x.shape
    q_out = torch.empty((n, C), dtype=torch.bfloat16, device=x.device) if q_out is None else q_out
    store = PackedKV.empty(n, C, group, 4, x.device) if store is None else store
    _whole_store(store, "streamed_qkv_proj")
    st = load().streamed_qkv_proj(_ptr(x), _ptr(w_qkv), n, C, group, chunk_tokens, _ptr(q_norm_w), _ptr(k_norm_w),
                                  eps, _ptr(q_out), _ptr(store.k_codes), _ptr(store.v_codes), _ptr(store.k_scales),
                                  _ptr(store.v_scales), _stream(stream))
    _check(st, "streamed_qkv_proj")
    return q_out, store


def packed_kv_attention(q: torch.Tensor, store: PackedKV, sm_scale: float = 0.0, out_fp32: bool = False,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q BF16 [n_q, C] (rotated) against an INT4 store -> out [n_q, C] (BF16 or fp32).
    `out` may be `q` itself for BF16 output."""
    _need_cuda(q, store.k_codes)
    _whole_store(store, "packed_kv_attention")
    n_q, C = q.shape
    if out is None:
        out = torch.empty((n_q, C), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=q.device)
    st = load().packed_kv_attention(_ptr(q), n_q, _ptr(store.k_codes), _ptr(store.v_codes), _ptr(store.k_scales),
                                    _ptr(store.v_scales), store.n, C, store.group, sm_scale, int(out_fp32),
                                    _ptr(out), _stream(stream))
    _check(st, "packed_kv_attention")
    return out


def packed_kv_attention_causal(q: torch.Tensor, store: PackedKV, q_pos0: int = 0, sm_scale: float = 0.0,
                               out_fp32: bool = False, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal form: query row i sits at key position q_pos0 + i and attends keys
    j <= q_pos0 + i.  A query chunk starting at row a of a sequence passes
    q = rows a.. and q_pos0 = a."""
    _need_cuda(q, store.k_codes)
    _whole_store(store, "packed_kv_attention_causal")
    n_q, C = q.shape
    if out is None:
        out = torch.empty((n_q, C), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=q.device)
    st = load().packed_kv_attention_causal(_ptr(q), n_q, int(q_pos0), _ptr(store.k_codes), _ptr(store.v_codes),
                                           _ptr(store.k_scales), _ptr(store.v_scales), store.n, C, store.group,
                                           sm_scale, int(out_fp32), _ptr(out), _stream(stream))
    _check(st, "packed_kv_attention_causal")
    return out


def _ranges(stores: list[PackedKV]):
    arr = (_Range * len(stores))()
    start = 0
    for i, s in enumerate(stores):
        arr[i] = _Range(start, s.n, s.cap, s.bits, 0, s.k_codes.data_ptr(), s.v_codes.data_ptr(),
                        s.k_scales.data_ptr(), s.v_scales.data_ptr())
        start += s.n
    return arr


def streamed_qkv_proj_mixed(x: torch.Tensor, w_qkv: torch.Tensor, stores: list[PackedKV], group: int = 32,
                            chunk_tokens: int = 0, q_norm_w=None, k_norm_w=None, eps: float = 1e-6,
                            q_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Like streamed_qkv_proj, with consecutive token ranges each going to its
    own store (bits 4 or 8).  Returns q_rot."""
    _need_cuda(x, w_qkv, q_norm_w, k_norm_w)
    n, C = x.shape
    q_out = torch.empty((n, C), dtype=torch.bfloat16, device=x.device) if q_out is None else q_out
    arr = _ranges(stores)
    st = load().streamed_qkv_proj_mixed(_ptr(x), _ptr(w_qkv), n, C, group, chunk_tokens, _ptr(q_norm_w),
                                        _ptr(k_norm_w), eps, _ptr(q_out), arr, len(stores), _stream(stream))
    _check(st, "streamed_qkv_proj_mixed")
    return q_out


SECTION_Q, SECTION_KV = 1, 2


def streamed_qkv_proj_ex(x: torch.Tensor, w_qkv: torch.Tensor, stores: list[PackedKV] | None = None,
                         rope_cs: torch.Tensor | None = None, sections: int = SECTION_Q | SECTION_KV, group: int = 32,
                         chunk_tokens: int = 0, q_norm_w=None, k_norm_w=None, eps: float = 1e-6,
                         q_out: torch.Tensor | None = None, stream=None) -> torch.Tensor | None:
    """streamed_qkv_proj_mixed with optional split-half RoPE of Q and K after the
    RMSNorm (rope_cs: fp32 [n, rot_dim/2, 2] (cos, sin) per token row of x,
    rot_dim 64 or 128) and a section mask: SECTION_Q writes Q only, SECTION_KV
    the stores only.  Returns q_rot (None without SECTION_Q)."""
    _need_cuda(x, w_qkv, q_norm_w, k_norm_w, rope_cs)
    n, C = x.shape
    want_q, want_kv = bool(sections & SECTION_Q), bool(sections & SECTION_KV)
    if rope_cs is not None:
        assert rope_cs.dtype == torch.float32 and rope_cs.is_contiguous() and rope_cs.shape[0] == n
        assert rope_cs.dim() == 3 and rope_cs.shape[2] == 2
    if want_q and q_out is None:
        q_out = torch.empty((n, C), dtype=torch.bfloat16, device=x.device)
    if want_kv:
        arr, nr = _ranges(stores), len(stores)
    else:
        arr, nr = None, 0
    st = load().streamed_qkv_proj_ex(_ptr(x), _ptr(w_qkv), n, C, group, chunk_tokens, _ptr(q_norm_w), _ptr(k_norm_w),
                                     eps, _ptr(rope_cs), 0 if rope_cs is None else 2 * rope_cs.shape[1], sections,
                                     _ptr(q_out) if want_q else None, arr, nr, _stream(stream))
    _check(st, "streamed_qkv_proj_ex")
    return q_out if want_q else None


def packed_kv_attention_mixed(q: torch.Tensor, stores: list[PackedKV], sm_scale: float = 0.0,
                              out_fp32: bool = False, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need_cuda(q)
    n_q, C = q.shape
    if out is None:
        out = torch.empty((n_q, C), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=q.device)
    arr = _ranges(stores)
    st = load().packed_kv_attention_mixed(_ptr(q), n_q, arr, len(stores), C, stores[0].group, sm_scale,
                                          int(out_fp32), _ptr(out), _stream(stream))
    _check(st, "packed_kv_attention_mixed")
    return out


PARTIAL_MERGE, PARTIAL_FINAL = 1, 2


def partial_state(n_q: int, hidden: int, device="cuda"):
    """Carried state of packed_kv_attention_partial: (o_acc fp32 [n_q, hidden],
    lse_acc fp32 [n_q, heads])."""
    return (torch.empty((n_q, hidden), dtype=torch.float32, device=device),
            torch.empty((n_q, hidden // HEAD_DIM), dtype=torch.float32, device=device))


def packed_kv_attention_partial(q: torch.Tensor, stores: list[PackedKV], state=None, merge: bool = False,
                                final: bool = False, sm_scale: float = 0.0, out_fp32: bool = False,
                                out: torch.Tensor | None = None, stream=None):
    """Attention of q against ONE key chunk (`stores`: its ranges, e.g. row
    windows of a larger store) with a carried state (o_acc, lse_acc):
    merge=False starts the state, merge=True merges this chunk into it;
    final=True writes the un-rotated result to `out` and returns it, otherwise
    the state is updated and returned.  Chunks merge in call order."""
    _need_cuda(q)
    n_q, C = q.shape
    if state is None:
        state = partial_state(n_q, C, q.device) if (merge or not final) else (None, None)
    o_acc, lse_acc = state
    if final and out is None:
        out = torch.empty((n_q, C), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=q.device)
    arr = _ranges(stores)
    flags = (PARTIAL_MERGE if merge else 0) | (PARTIAL_FINAL if final else 0)
    st = load().packed_kv_attention_partial(_ptr(q), n_q, arr, len(stores), C, stores[0].group, sm_scale, flags,
                                            _ptr(o_acc), _ptr(lse_acc), int(out_fp32), _ptr(out) if final else None,
                                            _stream(stream))
    _check(st, "packed_kv_attention_partial")
    return out if final else state


def packed_kv_attention_partial_static(q: torch.Tensor, stores: list[PackedKV], merge: bool = False,
                                       final: bool = False, sm_scale: float = 0.0, out_fp32: bool = False,
                                       out: torch.Tensor | None = None, stream=None):
    """packed_kv_attention_partial with the carried state in the library's fixed
    device area (for callers that cannot allocate device memory; at most
    STATIC_STATE_BYTES of state, one sequence of calls at a time per device).
    Returns `out` with final=True, else None."""
    _need_cuda(q)
    n_q, C = q.shape
    if final and out is None:
        out = torch.empty((n_q, C), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=q.device)
    arr = _ranges(stores)
    flags = (PARTIAL_MERGE if merge else 0) | (PARTIAL_FINAL if final else 0)
    st = load().packed_kv_attention_partial_static(_ptr(q), n_q, arr, len(stores), C, stores[0].group, sm_scale,
                                                   flags, int(out_fp32), _ptr(out) if final else None,
                                                   _stream(stream))
    _check(st, "packed_kv_attention_partial_static")
    return out if final else None


def device_status(stream=None) -> int:
    """Synchronises `stream` and returns KVQ_OK or KVQ_ERR_TIMEOUT (and clears it)."""
    return int(load().kvq_device_status(_stream(stream)))


def selftest_wait_timeout(ns: int, stream=None) -> None:
    _check(load().kvq_selftest_wait_timeout(int(ns), _stream(stream)), "kvq_selftest_wait_timeout")
