"""Test-side helpers: layout conversions written from the library header's
documented layouts (independent of the kernels), and tensor transfers."""
import numpy as np
import torch

from oracle.formats import unpack_nibbles


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def codes_np(t: torch.Tensor, cols: int) -> np.ndarray:
    """Packed device codes [rows, >= cols/2] -> one code per element [rows, cols]."""
    return unpack_nibbles(t.cpu().numpy()[:, : cols // 2])


def unswizzle(sf: torch.Tensor, rows: int, cols: int) -> np.ndarray:
    """Tensor-core scale layout -> linear [rows, cols/16]: byte of (r, c) at
    ((r/128)*(n16/4) + c/4)*512 + (r%32)*16 + ((r/32)%4)*4 + c%4."""
    b = sf.cpu().numpy().reshape(-1)
    n16 = cols // 16
    r = np.arange(rows)[:, None]
    c = np.arange(n16)[None, :]
    off = ((r // 128) * (n16 // 4) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    return b[off]


def linear_scales(q, rows=None, cols=None) -> np.ndarray:
    rows = q.rows if rows is None else rows
    cols = q.cols if cols is None else cols
    if q.layout == 1:
        return unswizzle(q.scales, rows, cols)
    return q.scales.cpu().numpy().reshape(-1)[: rows * (cols // 16)].reshape(rows, cols // 16)


def swizzle_np(lin: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Linear [rows, cols/16] -> tensor-core layout bytes (padding rows 0)."""
    n16 = cols // 16
    rp = (rows + 127) // 128 * 128
    out = np.zeros(rp * n16, np.uint8)
    r = np.arange(rows)[:, None]
    c = np.arange(n16)[None, :]
    off = ((r // 128) * (n16 // 4) + c // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + c % 4
    out[off] = lin
    return out


def check_combine(out, idx, gates, y_slots):
    """The GPU's combined output against the oracle's combine on the same gates
    and expert outputs.  Both sides round to bf16, the GPU after a float32 sum,
    the oracle after a float64 one, so an element may land one bf16 step away
    (2^-7 of its magnitude) where the float32 sum crosses a rounding boundary;
    such flips must be rare."""
    from oracle import moe as M
    ref = M.combine(idx, gates, y_slots)
    out = np.asarray(out, np.float64)
    mag = np.abs(y_slots.astype(np.float64)).sum(1)
    assert np.all(np.abs(out - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-5 * mag + 1e-30)
    assert np.mean(out == ref) >= 0.999
