"""Block-sparse video attention (VSA) in fp64 -- test infrastructure only, never product code.

Source: [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section
"VSA: block-sparse attention -- select first, then compute" and its table of the three steps
(blocking: 4x4x4 = 64-token blocks; gated scoring and coarse selection at block level: keep the
top-k blocks; fine attention at token level between the selected blocks only).  The pages do not
give the top-k ratio.

Readings where the pages leave a step open:
  * Blocks: the (T, H, W) latent grid is cut into (bt, bh, bw) = (4, 4, 4) cubes along each axis
    starting at 0, without shift; a token at (t, h, w) is in block (t // bt, h // bh, w // bw);
    edge blocks are cropped by the grid.  Block id is lexicographic (i_t, i_h, i_w).
  * Query side: queries are grouped in the same blocks; every query of block a uses block a's
    selection ("relevance of the block to the current query" read per query block).
  * Gate score: with no learned gate given, the score of key block b for query block a (per head)
    is the scaled dot product of the block means, scale * <mean_a(q), mean_b(k)>, the means taken
    over the block's tokens inside the grid.
  * Selection: the k highest scores per (head, query block); equal scores are taken in ascending
    block id.  The list is reported in ascending block id.
  * Fine attention: query i of block a attends, with an ordinary softmax, to every key token of
    the selected blocks of a (and to nothing else), scale = 1/sqrt(D).  The pages mention no
    second (coarse) output branch, so the output is the fine attention alone.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().float().numpy()
    return np.asarray(x, dtype=np.float64)


def vsa_block_counts(grid: Sequence[int], block: Sequence[int]):
    """Blocks per axis: ceil(L / b)."""
    return tuple((int(L) + int(b) - 1) // int(b) for L, b in zip(grid, block))


def vsa_block_count(grid: Sequence[int], block: Sequence[int]) -> int:
    nt, nh, nw = vsa_block_counts(grid, block)
    return nt * nh * nw


def vsa_block_ids(grid: Sequence[int], block: Sequence[int]) -> np.ndarray:
    """Block id of every token of the row-major (t, h, w) grid, int64 [T*H*W]."""
    T, H, W = grid
    _, nh, nw = vsa_block_counts(grid, block)
    t, h, w = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    ids = ((t // block[0]) * nh + (h // block[1])) * nw + (w // block[2])
    return ids.reshape(-1).astype(np.int64)


def vsa_block_means(x, grid: Sequence[int], block: Sequence[int]) -> np.ndarray:
    """Mean of the rows of each block: x [N, H, D] -> fp64 [H, nblk, D]."""
    xa = _as_f64(x)
    N, H, D = xa.shape
    ids = vsa_block_ids(grid, block)
    nblk = vsa_block_count(grid, block)
    order = np.argsort(ids, kind="stable")                 # rows grouped by block
    counts = np.bincount(ids, minlength=nblk)              # every block holds >= 1 row
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    sums = np.add.reduceat(xa[order], starts, axis=0)      # [nblk, H, D]
    return np.transpose(sums / counts[:, None, None].astype(np.float64), (1, 0, 2))


def vsa_block_scores(q, k, grid: Sequence[int], block: Sequence[int],
                     scale: Optional[float] = None) -> np.ndarray:
    """Gate scores fp64 [H, nblk(query), nblk(key)] = scale * <mean q, mean k>."""
    qm = vsa_block_means(q, grid, block)
    km = vsa_block_means(k, grid, block)
    D = qm.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return scale * np.matmul(qm, np.transpose(km, (0, 2, 1)))


def vsa_select(scores: np.ndarray, topk: int) -> np.ndarray:
    """Top-k key blocks per (head, query block), reported ascending: int32 [H, nblk, topk].

    Order of preference: higher score first, then lower block id (a stable sort of -score).
    """
    H, A, B = scores.shape
    if not 1 <= topk <= B:
        raise ValueError("topk must be in [1, number of blocks]")
    out = np.empty((H, A, topk), dtype=np.int32)
    for h in range(H):
        for a in range(A):
            order = np.argsort(-scores[h, a], kind="stable")
            out[h, a] = np.sort(order[:topk])
    return out


def vsa_attention(q, k, v, grid: Sequence[int], block: Sequence[int], selection,
                  scale: Optional[float] = None, rows: Optional[np.ndarray] = None,
                  heads: Optional[Sequence[int]] = None):
    """Fine attention over the selected blocks.  Returns (o fp64 [N,H,D], lse fp64 [H,N]).

    selection: int [H, nblk, k] key-block ids per (head, query block) in any order.
    rows / heads restrict the evaluated queries (others stay NaN).
    """
    qa, ka, va = _as_f64(q), _as_f64(k), _as_f64(v)
    N, H, D = qa.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    sel = np.asarray(selection, dtype=np.int64)
    ids = vsa_block_ids(grid, block)
    nblk = vsa_block_count(grid, block)
    members = [np.nonzero(ids == b)[0] for b in range(nblk)]  # rows of each block, ascending
    want = np.ones(N, dtype=bool)
    if rows is not None:
        want[:] = False
        want[np.asarray(rows, dtype=np.int64)] = True
    head_list = list(range(H)) if heads is None else list(heads)
    o = np.full((N, H, D), np.nan)
    lse = np.full((H, N), np.nan)
    for h in head_list:
        for a in range(nblk):
            qi = members[a][want[members[a]]]
            if qi.size == 0:
                continue
            kj = np.concatenate([members[b] for b in sel[h, a]])
            s = scale * (qa[qi, h, :] @ ka[kj, h, :].T)
            m = np.max(s, axis=1, keepdims=True)
            e = np.exp(s - m)
            l = np.sum(e, axis=1, keepdims=True)
            o[qi, h, :] = (e / l) @ va[kj, h, :]
            lse[h, qi] = (m + np.log(l))[:, 0]
    return o, lse
