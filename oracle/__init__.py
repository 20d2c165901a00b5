"""CPU oracle for the streamed QKV projection and packed rotated low-bit K/V
attention -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline use this package.  The library never imports it, and it imports
nothing from the library.  The arithmetic lives in ``kvq_oracle.c`` (plain C,
built here with gcc); this module builds it and marshals numpy arrays.

Arrays of BF16 or FP16 values are passed as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

HD = 128


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into libkvq_oracle.so (gcc, -O2, no fast-math,
    no FMA contraction, OpenMP when the compiler has it)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            lib.kvqo_bf16_to_f32.restype = F
            lib.kvqo_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.kvqo_f32_to_bf16.restype = ctypes.c_uint16
            lib.kvqo_f32_to_bf16.argtypes = [F]
            lib.kvqo_f16_to_f32.restype = F
            lib.kvqo_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.kvqo_f32_to_f16.restype = ctypes.c_uint16
            lib.kvqo_f32_to_f16.argtypes = [F]
            lib.kvqo_rot_scale.restype = F
            lib.kvqo_rot_scale.argtypes = []
            lib.kvqo_rotate.restype = None
            lib.kvqo_rotate.argtypes = [P, I64, P]
            lib.kvqo_quant_head.restype = None
            lib.kvqo_quant_head.argtypes = [P, I, I, P, P]
            lib.kvqo_dequant_head.restype = None
            lib.kvqo_dequant_head.argtypes = [P, P, I, I, P]
            lib.kvqo_kv_rotate_quant_pack.restype = I
            lib.kvqo_kv_rotate_quant_pack.argtypes = [P, I64, I, P, I64, I, I, P, P, P, P]
            lib.kvqo_kv_unpack.restype = I
            lib.kvqo_kv_unpack.argtypes = [P, P, P, P, I64, I, I, I, P]
            lib.kvqo_qkv_proj.restype = I
            lib.kvqo_qkv_proj.argtypes = [P, P, I, P, I64, I, I, P, P, F, P, I, P, P, P, P, P, P, P, P]
            lib.kvqo_attention.restype = I
            lib.kvqo_attention.argtypes = [P, I64, I, P, P, P, P, I64, I64, I, I, F, P, I64, P]
            lib.kvqo_attention_causal.restype = I
            lib.kvqo_attention_causal.argtypes = [P, I64, I, P, P, P, P, I64, I64, I, I, F, I64, P, I64, P]
            lib.kvqo_attention_mixed.restype = I
            lib.kvqo_attention_mixed.argtypes = [P, I64, I, I, P, P, P, P, P, P, P, P, I, F, P, I64, P]
            lib.kvqo_attention_partial.restype = I
            lib.kvqo_attention_partial.argtypes = [P, I64, I, I, P, P, P, P, P, P, P, P, I, F, P, I64, P, P]
            lib.kvqo_lse_merge.restype = None
            lib.kvqo_lse_merge.argtypes = [P, P, P, P, I64]
            lib.kvqo_partial_finish.restype = None
            lib.kvqo_partial_finish.argtypes = [P, I64, P]
            lib.kvqo_threads.restype = I
            lib.kvqo_threads.argtypes = []
            lib.kvqo_set_threads.restype = None
            lib.kvqo_set_threads.argtypes = [I]
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().kvqo_threads())


def set_threads(n: int) -> None:
    """OpenMP threads for later oracle calls."""
    _load().kvqo_set_threads(int(n))


# ----------------------------------------------------------------- number formats
def bf16_to_f32(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float32, exactly."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32)
    return np.array([lib.kvqo_f32_to_bf16(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def f32_to_f16(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32)
    return np.array([lib.kvqo_f32_to_f16(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def f16_to_f32(h) -> np.ndarray:
    lib = _load()
    h = _c(h, np.uint16)
    return np.array([lib.kvqo_f16_to_f32(int(v)) for v in h.ravel()], dtype=np.float32).reshape(h.shape)


def rot_scale() -> float:
    return float(_load().kvqo_rot_scale())


# ----------------------------------------------------------------- rotation and quantiser
def rotate(x) -> np.ndarray:
    """x[..., 128] -> x . H (fp32, the FWHT order the format fixes)."""
    x = _c(x, np.float32)
    assert x.shape[-1] == HD
    y = np.empty_like(x)
    _load().kvqo_rotate(_p(x), x.size // HD, _p(y))
    return y


def quant_head(y, group: int, bits: int):
    """One rotated head vector y[128] -> (codes bytes, fp16 scale bits)."""
    y = _c(y, np.float32)
    assert y.shape == (HD,)
    codes = np.empty(HD * bits // 8, np.uint8)
    scales = np.empty(HD // group, np.uint16)
    _load().kvqo_quant_head(_p(y), group, bits, _p(codes), _p(scales))
    return codes, scales


def dequant_head(codes, scales, group: int, bits: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    y = np.empty(HD, np.float32)
    _load().kvqo_dequant_head(_p(codes), _p(scales), group, bits, _p(y))
    return y


# ----------------------------------------------------------------- a1 / a1b
def kv_rotate_quant_pack(kv, rows=None, *, hidden: int, group: int = 32, bits: int = 4):
    """kv: uint16 BF16 bits [n, >= 2*hidden] (K then V).  Returns compact
    token-major (k_codes, v_codes, k_scales, v_scales) for `rows`:
    codes [n_rows, heads, 128*bits/8] uint8, scales [n_rows, heads, 128/group] uint16."""
    kv = _c(kv, np.uint16)
    n, ld = kv.shape
    rows = np.arange(n, dtype=np.int64) if rows is None else _c(rows, np.int64)
    heads = hidden // HD
    kc = np.empty((len(rows), heads, HD * bits // 8), np.uint8)
    vc = np.empty_like(kc)
    ks = np.empty((len(rows), heads, HD // group), np.uint16)
    vs = np.empty_like(ks)
    rc = _load().kvqo_kv_rotate_quant_pack(_p(kv), ld, hidden, _p(rows), len(rows), group, bits,
                                           _p(kc), _p(vc), _p(ks), _p(vs))
    if rc:
        raise ValueError("oracle kv_rotate_quant_pack: bad arguments")
    return kc, vc, ks, vs


def kv_unpack(kc, vc, ks, vs, *, group: int = 32, bits: int = 4) -> np.ndarray:
    kc, vc = _c(kc, np.uint8), _c(vc, np.uint8)
    ks, vs = _c(ks, np.uint16), _c(vs, np.uint16)
    n_rows, heads = kc.shape[:2]
    out = np.empty((n_rows, 2 * heads * HD), np.uint16)
    rc = _load().kvqo_kv_unpack(_p(kc), _p(vc), _p(ks), _p(vs), n_rows, heads * HD, group, bits, _p(out))
    if rc:
        raise ValueError("oracle kv_unpack: bad arguments")
    return out


# ----------------------------------------------------------------- a2
def qkv_proj(x, w, rows=None, *, group: int = 32, bits: int = 4, q_norm_w=None, k_norm_w=None, eps: float = 1e-6,
             rope_cs=None):
    """x: uint16 BF16 bits [n, C]; w: uint16 BF16 bits [3C, C].  Returns a dict
    with q_f32 [n_rows, C], q_bf16 [n_rows, C] (uint16), compact token-major
    k_codes, v_codes, k_scales, v_scales for `rows`, and k_rot / v_rot
    [n_rows, C] fp32: the rotated K and V vectors the quantiser was given.
    rope_cs: optional fp32 [n, rot_dim/2, 2] (cos, sin) per token row for the
    split-half RoPE of Q and K after the RMSNorm."""
    x, w = _c(x, np.uint16), _c(w, np.uint16)
    n, C = x.shape
    assert w.shape == (3 * C, C)
    rows = np.arange(n, dtype=np.int64) if rows is None else _c(rows, np.int64)
    heads = C // HD
    qn = None if q_norm_w is None else _c(q_norm_w, np.float32)
    kn = None if k_norm_w is None else _c(k_norm_w, np.float32)
    rc_ = None if rope_cs is None else _c(rope_cs, np.float32)
    rot = 0 if rc_ is None else 2 * rc_.shape[1]
    assert rc_ is None or (rc_.shape[0] == n and rc_.shape[2] == 2)
    out = dict(
        q_f32=np.empty((len(rows), C), np.float32),
        q_bf16=np.empty((len(rows), C), np.uint16),
        k_codes=np.empty((len(rows), heads, HD * bits // 8), np.uint8),
        v_codes=np.empty((len(rows), heads, HD * bits // 8), np.uint8),
        k_scales=np.empty((len(rows), heads, HD // group), np.uint16),
        v_scales=np.empty((len(rows), heads, HD // group), np.uint16),
        k_rot=np.empty((len(rows), C), np.float32),
        v_rot=np.empty((len(rows), C), np.float32),
    )
    rc = _load().kvqo_qkv_proj(_p(x), _p(w), C, _p(rows), len(rows), group, bits, _p(qn), _p(kn), eps, _p(rc_), rot,
                               _p(out["q_f32"]), _p(out["q_bf16"]), _p(out["k_codes"]), _p(out["v_codes"]),
                               _p(out["k_scales"]), _p(out["v_scales"]), _p(out["k_rot"]), _p(out["v_rot"]))
    if rc:
        raise ValueError("oracle qkv_proj: bad arguments")
    return out


# ----------------------------------------------------------------- a4
def attention(q, k_codes, v_codes, k_scales, v_scales, *, n_kv: int, group: int = 32, bits: int = 4,
              sm_scale: float | None = None, rows=None) -> np.ndarray:
    """q: uint16 BF16 bits [n_q, C] (rotated basis).  K/V store in the
    library's head-major layout: codes [heads, n_pad, 128*bits/8] uint8,
    scales [heads, n_pad, 128/group] uint16.  Returns fp32 [n_rows, C]."""
    q = _c(q, np.uint16)
    n_q, C = q.shape
    heads = C // HD
    kc, vc = _c(k_codes, np.uint8), _c(v_codes, np.uint8)
    ks, vs = _c(k_scales, np.uint16), _c(v_scales, np.uint16)
    n_pad = kc.shape[1]
    assert kc.shape[0] == heads and ks.shape[:2] == (heads, n_pad)
    rows = np.arange(n_q, dtype=np.int64) if rows is None else _c(rows, np.int64)
    sm = HD ** -0.5 if sm_scale is None else sm_scale
    out = np.empty((len(rows), C), np.float32)
    rc = _load().kvqo_attention(_p(q), C, heads, _p(kc), _p(vc), _p(ks), _p(vs), n_kv, n_pad, group, bits, sm,
                                _p(rows), len(rows), _p(out))
    if rc:
        raise ValueError("oracle attention: bad arguments")
    return out


def attention_causal(q, k_codes, v_codes, k_scales, v_scales, *, n_kv: int, q_pos0: int = 0, group: int = 32,
                     bits: int = 4, sm_scale: float | None = None, rows=None) -> np.ndarray:
    """As attention(), with query row i at key position q_pos0 + i attending
    keys j <= q_pos0 + i only."""
    q = _c(q, np.uint16)
    n_q, C = q.shape
    heads = C // HD
    kc, vc = _c(k_codes, np.uint8), _c(v_codes, np.uint8)
    ks, vs = _c(k_scales, np.uint16), _c(v_scales, np.uint16)
    n_pad = kc.shape[1]
    assert kc.shape[0] == heads and ks.shape[:2] == (heads, n_pad)
    rows = np.arange(n_q, dtype=np.int64) if rows is None else _c(rows, np.int64)
    sm = HD ** -0.5 if sm_scale is None else sm_scale
    out = np.empty((len(rows), C), np.float32)
    rc = _load().kvqo_attention_causal(_p(q), C, heads, _p(kc), _p(vc), _p(ks), _p(vs), n_kv, n_pad, group, bits, sm,
                                       int(q_pos0), _p(rows), len(rows), _p(out))
    if rc:
        raise ValueError("oracle causal attention: bad arguments")
    return out


class _RangeArgs:
    """A range table marshalled for the C oracle (keeps the arrays alive)."""

    def __init__(self, ranges):
        self.keep = []
        self.arrs = {}
        for key, dt in (("k_codes", np.uint8), ("v_codes", np.uint8), ("k_scales", np.uint16),
                        ("v_scales", np.uint16)):
            lst = [_c(r[key], dt) for r in ranges]
            ptrs = (ctypes.c_void_p * len(lst))(*[a.ctypes.data for a in lst])
            self.keep += lst + [ptrs]
            self.arrs[key] = ctypes.cast(ptrs, ctypes.c_void_p)
        self.n = len(ranges)
        self.starts = np.array([r["start"] for r in ranges], np.int64)
        self.lens = np.array([r["len"] for r in ranges], np.int64)
        self.bitss = np.array([r["bits"] for r in ranges], np.int32)
        self.caps = np.array([_c(r["k_codes"], np.uint8).shape[1] for r in ranges], np.int64)

    def args(self):
        a = self.arrs
        return (self.n, _p(self.starts), _p(self.lens), _p(self.bitss), _p(self.caps), a["k_codes"], a["v_codes"],
                a["k_scales"], a["v_scales"])


def attention_mixed(q, ranges, *, group: int = 32, sm_scale: float | None = None, rows=None) -> np.ndarray:
    """ranges: list of dicts with start, len, bits and the range's own
    head-major store (k_codes, v_codes, k_scales, v_scales; capacity = their
    second dimension).  Ranges must tile [0, n_kv) in order."""
    q = _c(q, np.uint16)
    n_q, C = q.shape
    heads = C // HD
    rows = np.arange(n_q, dtype=np.int64) if rows is None else _c(rows, np.int64)
    sm = HD ** -0.5 if sm_scale is None else sm_scale
    ra = _RangeArgs(ranges)
    out = np.empty((len(rows), C), np.float32)
    rc = _load().kvqo_attention_mixed(_p(q), C, heads, *ra.args(), group, sm, _p(rows), len(rows), _p(out))
    if rc:
        raise ValueError("oracle attention_mixed: bad arguments")
    return out


# ----------------------------------------------------------------- next row f3: attention over key chunks
def attention_partial(q, ranges, *, group: int = 32, sm_scale: float | None = None, rows=None):
    """Partial attention of query rows against one key chunk (vram_lab.py's
    blockwise attention: each K/V block's normalised output and its
    log-sum-exp).  `ranges` as attention_mixed, tiling the chunk's keys.
    Returns (o, lse): o fp64 [n_rows, heads, 128] in the ROTATED basis, lse fp64
    [n_rows, heads] = log sum_j exp(s_j) over the chunk's keys."""
    q = _c(q, np.uint16)
    n_q, C = q.shape
    heads = C // HD
    rows = np.arange(n_q, dtype=np.int64) if rows is None else _c(rows, np.int64)
    sm = HD ** -0.5 if sm_scale is None else sm_scale
    ra = _RangeArgs(ranges)
    o = np.empty((len(rows), heads, HD), np.float64)
    lse = np.empty((len(rows), heads), np.float64)
    rc = _load().kvqo_attention_partial(_p(q), C, heads, *ra.args(), group, sm, _p(rows), len(rows), _p(o), _p(lse))
    if rc:
        raise ValueError("oracle attention_partial: bad arguments")
    return o, lse


def lse_merge(o_a, lse_a, o_b, lse_b):
    """vram_lab.py `_online_combine` of two partials over disjoint key sets;
    returns the merged (o, lse) as new arrays."""
    o = _c(o_a, np.float64).copy()
    lse = _c(lse_a, np.float64).copy()
    ob, lb = _c(o_b, np.float64), _c(lse_b, np.float64)
    assert o.shape == ob.shape and lse.shape == lb.shape and o.shape[:-1] == lse.shape and o.shape[-1] == HD
    _load().kvqo_lse_merge(_p(o), _p(lse), _p(ob), _p(lb), lse.size)
    return o, lse


def partial_finish(o) -> np.ndarray:
    """Merged o [n_rows, heads, 128] (rotated) -> fp32 output [n_rows, heads*128],
    rounded to fp32 and un-rotated."""
    o = _c(o, np.float64)
    out = np.empty(o.shape, np.float32)
    _load().kvqo_partial_finish(_p(o), o.size // HD, _p(out))
    return out.reshape(o.shape[0], -1)


def attention_blockwise(q, chunks, *, group: int = 32, sm_scale: float | None = None, rows=None) -> np.ndarray:
    """Attention over a sequence of key chunks (each a range table, as
    attention_partial), merged in the given order and un-rotated once at the
    end: vram_lab.py's `_blockwise_attention_q` on the packed store."""
    o = lse = None
    for ch in chunks:
        ob, lb = attention_partial(q, ch, group=group, sm_scale=sm_scale, rows=rows)
        o, lse = (ob, lb) if o is None else lse_merge(o, lse, ob, lb)
    return partial_finish(o)
