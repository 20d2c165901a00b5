"""Small helpers shared by the tests (conversions between torch tensors and
the uint16 bit patterns the oracle takes)."""
import numpy as np
import torch


def bits16(t: torch.Tensor) -> np.ndarray:
    """BF16 / FP16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f16_np(bits: np.ndarray) -> np.ndarray:
    return bits.view(np.float16).astype(np.float64)


def to_token_major(a: torch.Tensor, rows, n=None) -> np.ndarray:
    """Head-major store array [heads, cap, x] -> numpy [len(rows), heads, x] for the given rows."""
    idx = torch.as_tensor(np.asarray(rows), dtype=torch.long, device=a.device)
    return a.index_select(1, idx).permute(1, 0, 2).contiguous().cpu().numpy()


def unpack_int4(codes: np.ndarray) -> np.ndarray:
    lo = (codes & 0x0F).astype(np.int16)
    hi = (codes >> 4).astype(np.int16)
    v = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], -1)
    return np.where(v >= 8, v - 16, v)


def codes_as_int(codes: np.ndarray, bits: int) -> np.ndarray:
    return unpack_int4(codes) if bits == 4 else codes.view(np.int8).astype(np.int16)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x.astype(np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)
