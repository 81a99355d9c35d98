"""Shifted 3D window partition of a latent grid into packed segments -- test infrastructure only.

Source: [H3-fast] "Breaking the memory wall: window attention across GPUs".  The 3D token grid
is cut into equal local windows; alternate layers shift the window grid by half a window so
that neighbouring windows' boundary tokens meet; windows at the grid edge are incomplete
("cropped", of unequal size); after attention the scattered tokens are put back in their
original order.

Readings of the pages taken here:
  * Along an axis of length L with window w and shift s, token x belongs to axis window
    floor((x + s) / w); there are ceil((L + s) / w) axis windows; when s > 0 the first is
    w - s wide and the last is cropped by the grid edge.  Edge windows are cropped, not rolled
    cyclically.
  * Window id = lexicographic (i_t, i_h, i_w).  Packed order: windows ascending by id; inside a
    window, tokens ascending by their original row-major index t*H*W + h*W + w.
  * cu_seqlens = exclusive prefix of window sizes.

The oracle builds the permutation by a STABLE SORT of all tokens by window id.
"""
from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np


def axis_window_count(L: int, w: int, s: int) -> int:
    return (L + s + w - 1) // w


def window_count(grid: Sequence[int], win: Sequence[int], shift: Sequence[int]) -> int:
    n = 1
    for L, w, s in zip(grid, win, shift):
        n *= axis_window_count(L, w, s)
    return n


def window_ids(grid: Sequence[int], win: Sequence[int], shift: Sequence[int]) -> np.ndarray:
    """Window id of every token in row-major order, int64 [T*H*W]."""
    T, H, W = grid
    t, h, w = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    it = (t + shift[0]) // win[0]
    ih = (h + shift[1]) // win[1]
    iw = (w + shift[2]) // win[2]
    nh = axis_window_count(H, win[1], shift[1])
    nw = axis_window_count(W, win[2], shift[2])
    return ((it * nh + ih) * nw + iw).reshape(-1).astype(np.int64)


def window_partition(grid: Sequence[int], win: Sequence[int], shift: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """Return (perm int32 [N], cu_seqlens int32 [nwin+1]); perm[j] = original index of packed row j."""
    ids = window_ids(grid, win, shift)
    perm = np.argsort(ids, kind="stable").astype(np.int32)
    nwin = window_count(grid, win, shift)
    sizes = np.bincount(ids, minlength=nwin)
    cu = np.zeros(nwin + 1, dtype=np.int64)
    cu[1:] = np.cumsum(sizes)
    return perm, cu.astype(np.int32)


def window_pack(x, perm: np.ndarray):
    """Packed row j = original row perm[j]."""
    idx = np.asarray(perm, dtype=np.int64)
    if isinstance(x, np.ndarray):
        return x[idx]
    import torch
    return x[torch.from_numpy(idx)]


def window_unpack(y, perm: np.ndarray):
    """Inverse of window_pack: original row perm[j] = packed row j."""
    idx = np.asarray(perm, dtype=np.int64)
    if isinstance(y, np.ndarray):
        out = np.empty_like(y)
        out[idx] = y
        return out
    import torch  # torch tensors (e.g. bf16 rows) are permuted the same way
    out = torch.empty_like(y)
    out[torch.from_numpy(idx)] = y
    return out
