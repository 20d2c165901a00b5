"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method itself (no rotation, no
quantisation, no projection, no attention): only random draws with the
shapes and value distributions of the workloads, so that the CUDA path and
the CPU oracle can be fed identical inputs.

Workloads (MiniMax-H3-shaped blocks; hidden 7168 = 56 heads x 128):
  * TINY     N=1024,    hidden 1024, 8 heads, 4 outlier channels x20, no RMSNorm
  * MID      N=16,384,  hidden 7168, 1% outlier channels x20, Q/K RMSNorm, chunk 4096
  * H3_REF2VA N=152,263 packed tokens, as MID (the Ref2VA size that ran out of memory)
  * MIXED    N=217,088: text 512 + reference 16,384 + audio 2,048 at INT8, 198,144 video at INT4
  * SWEEP    K/V BF16 [N, 2*7168], N(0,1) with 1% heavy-tailed (Student-t, nu=3) channels
"""
from __future__ import annotations

import dataclasses

import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n: int
    hidden: int
    outlier_channels: int
    outlier_scale: float = 20.0
    rmsnorm: bool = False
    chunk_tokens: int = 0
    group: int = 32
    seed: int = 0

    @property
    def heads(self) -> int:
        return self.hidden // HEAD_DIM


TINY = Workload("tiny N=1024 hidden=1024 8x128", 1024, 1024, 4)
MID = Workload("H3 block N=16384 hidden=7168 56x128", 16384, 7168, 72, rmsnorm=True, chunk_tokens=4096)
H3_REF2VA = Workload("H3 Ref2VA block N=152263 hidden=7168 56x128", 152263, 7168, 72, rmsnorm=True,
                     chunk_tokens=4096)

# Mixed precision by token range: (name, tokens, bits)
MIXED_SEGMENTS = (("text", 512, 8), ("reference image/video", 16384, 8), ("audio", 2048, 8),
                  ("generated video", 198144, 4))
MIXED = Workload("H3 mixed N=217088 hidden=7168 56x128", 217088, 7168, 72, rmsnorm=True, chunk_tokens=4096)

SWEEP_N = tuple(4096 << i for i in range(7))  # 4,096 ... 262,144
SWEEP_GROUPS = (32, 64, 128)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def block_inputs(w: Workload, device="cpu", n: int | None = None):
    """(x [n, C] bf16, W_qkv [3C, C] bf16, q_norm_w [128] fp32 | None,
    k_norm_w [128] fp32 | None).

    x ~ N(0, 1) with `outlier_channels` channels (a seeded random choice)
    multiplied by `outlier_scale`; W ~ N(0, 1/C); RMSNorm weights
    1 + 0.1 N(0, 1) when the workload normalises Q and K."""
    n = w.n if n is None else n
    C = w.hidden
    g = _gen(w.seed, device)
    x = torch.randn((n, C), generator=g, device=device, dtype=torch.float32)
    chans = torch.randperm(C, generator=g, device=device)[: w.outlier_channels]
    x[:, chans] *= w.outlier_scale
    x = x.to(torch.bfloat16)
    W = (torch.randn((3 * C, C), generator=g, device=device, dtype=torch.float32) * C ** -0.5).to(torch.bfloat16)
    qn = kn = None
    if w.rmsnorm:
        qn = 1.0 + 0.1 * torch.randn((HEAD_DIM,), generator=g, device=device, dtype=torch.float32)
        kn = 1.0 + 0.1 * torch.randn((HEAD_DIM,), generator=g, device=device, dtype=torch.float32)
    return x, W, qn, kn


def sweep_kv(n: int, hidden: int = 7168, seed: int = 0, device="cpu") -> torch.Tensor:
    """K/V BF16 [n, 2*hidden]: N(0, 1) with 1% of the channels of K and of V
    (a seeded choice) drawn from Student-t with nu = 3 instead."""
    g = _gen(seed, device)
    kv = torch.randn((n, 2 * hidden), generator=g, device=device, dtype=torch.float32)
    n_heavy = max(1, hidden // 100)
    for half in range(2):
        chans = torch.randperm(hidden, generator=g, device=device)[:n_heavy] + half * hidden
        z = torch.randn((n, n_heavy), generator=g, device=device, dtype=torch.float32)
        chi2 = sum(torch.randn((n, n_heavy), generator=g, device=device, dtype=torch.float32) ** 2
                   for _ in range(3))
        kv[:, chans] = z / torch.sqrt(chi2 / 3.0)
    return kv.to(torch.bfloat16)


def random_packed_kv(heads: int, n: int, n_pad: int, group: int = 32, bits: int = 4, seed: int = 0,
                     device="cpu", scale_lo: float = 0.05, scale_hi: float = 0.5):
    """A random packed K/V store in the library's head-major layout:
    codes uint8 [heads, n_pad, 128*bits/8] (INT4: two nibbles per byte, each
    a uniform code in [-7, 7]; INT8: uniform in [-127, 127]); scales fp16
    [heads, n_pad, 128/group] uniform in [scale_lo, scale_hi].  Rows n..n_pad-1
    are zero.  Returns (k_codes, v_codes, k_scales, v_scales)."""
    g = _gen(seed, device)
    out = []
    qmax = 7 if bits == 4 else 127
    for _ in range(2):
        c = torch.randint(-qmax, qmax + 1, (heads, n_pad, HEAD_DIM), generator=g, device=device, dtype=torch.int32)
        c[:, n:] = 0
        if bits == 4:
            c = c & 0xF
            c = (c[..., 0::2] | (c[..., 1::2] << 4)).to(torch.uint8)
        else:
            c = (c & 0xFF).to(torch.uint8)
        out.append(c)
    sc = []
    for _ in range(2):
        s = torch.empty((heads, n_pad, HEAD_DIM // group), device=device, dtype=torch.float32)
        s.uniform_(scale_lo, scale_hi, generator=g)
        s[:, n:] = 0
        sc.append(s.to(torch.float16))
    return out[0], out[1], sc[0], sc[1]


def random_q(n: int, hidden: int, seed: int = 0, std: float = 1.0, device="cpu") -> torch.Tensor:
    """A rotated-basis query matrix stand-in: BF16 [n, hidden] ~ N(0, std^2)."""
    g = _gen(seed, device)
    return (torch.randn((n, hidden), generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def sample_rows(n: int, k: int, seed: int = 0, include_edges: bool = True) -> torch.Tensor:
    """k distinct sorted token rows of [0, n), always including the first and
    the last row (the ragged tail) when include_edges is set."""
    g = _gen(seed, "cpu")
    k = min(k, n)
    r = torch.randperm(n, generator=g)[:k]
    if include_edges and k >= 2:
        r[0], r[1] = 0, n - 1
        r = torch.unique(r)
    return torch.sort(r).values.to(torch.int64)
