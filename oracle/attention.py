"""fp64 block-diagonal (packed varlen) softmax attention -- test infrastructure, never product code.

Definition followed ([H3-vLLM] §3 "Packed sequence and modality identity", causal chain item 2
and the minimal example): cu_seqlens lists the start/end offsets of the sub-sequences of one
packed sequence; a query of sub-sequence g takes its dot products only with the keys of g and
softmax-normalises over them, so every key outside g gets weight exactly zero.  The example's
token 15 (video, rows 10..29) dots with keys 10..29 -- including keys after it, so there is no
causal mask.  [H3-vLLM] §6 "Boundary trim": rows at or beyond cu_seqlens[-1] (alignment padding)
never take part.

Per segment g, head h and query i in [cu_g, cu_{g+1}):
    S_ij  = scale * <q_i, k_j>                for j in [cu_g, cu_{g+1})
    m_i   = max_j S_ij
    P_ij  = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)
    o_i   = sum_j P_ij v_j
    LSE_i = m_i + log sum_j exp(S_ij - m_i)
scale defaults to 1/sqrt(D) (the pages do not state it; the standard choice).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor (bf16 upcasts exactly through fp32)
        x = x.detach().float().numpy()
    return np.asarray(x, dtype=np.float64)


def varlen_attention(q, k, v, cu_seqlens: Sequence[int], scale: Optional[float] = None,
                     rows: Optional[np.ndarray] = None, heads: Optional[Sequence[int]] = None):
    """Return (o, lse) for the packed sequence.

    q, k, v: [C, H, D] (any float type; upcast to fp64).  cu_seqlens: [S+1].
    rows: optional sorted array of query rows to evaluate (others are left NaN); heads likewise.
    Output o: fp64 [C, H, D] (NaN where not evaluated, including rows >= cu_seqlens[-1]);
    lse: fp64 [H, C] (NaN likewise).
    """
    C, H, D = q.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    head_list = list(range(H)) if heads is None else list(heads)
    o = np.full((C, H, D), np.nan, dtype=np.float64)
    lse = np.full((H, C), np.nan, dtype=np.float64)
    row_mask = None
    if rows is not None:
        row_mask = np.zeros(C, dtype=bool)
        row_mask[np.asarray(rows, dtype=np.int64)] = True
    for g in range(len(cu) - 1):
        a, b = int(cu[g]), int(cu[g + 1])
        if b <= a:
            continue  # empty segment: nothing to compute
        qi = np.arange(a, b) if row_mask is None else np.nonzero(row_mask[a:b])[0] + a
        if qi.size == 0:
            continue
        for h in head_list:
            qh = _as_f64(q[qi, h, :])
            kh = _as_f64(k[a:b, h, :])
            vh = _as_f64(v[a:b, h, :])
            s = scale * (qh @ kh.T)                      # [nq, n]
            m = np.max(s, axis=1, keepdims=True)
            e = np.exp(s - m)
            l = np.sum(e, axis=1, keepdims=True)
            o[qi, h, :] = (e / l) @ vh
            lse[h, qi] = (m + np.log(l))[:, 0]
    return o, lse


def attention_weights(q, k, cu_seqlens: Sequence[int], row: int, head: int,
                      scale: Optional[float] = None) -> np.ndarray:
    """Softmax weights of query ``row`` over ALL C key rows (zero outside its own segment)."""
    C, H, D = q.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    w = np.zeros(C, dtype=np.float64)
    g = int(np.searchsorted(cu, row, side="right")) - 1
    a, b = int(cu[g]), int(cu[g + 1])
    s = scale * (_as_f64(k[a:b, head, :]) @ _as_f64(q[row, head, :]))
    e = np.exp(s - np.max(s))
    w[a:b] = e / np.sum(e)
    return w


def dense_masked_attention_bruteforce(q, k, v, segment_of_row: Sequence[int],
                                      scale: Optional[float] = None):
    """Tiny-input brute force in pure Python: full N x N scores, -inf where segments differ.

    segment_of_row[i] is the segment id of row i (or -1 for a row that takes no part).
    Written with explicit loops and math.exp so that it shares nothing with varlen_attention.
    Returns (o [N,H,D], lse [H,N]) as nested Python-float numpy arrays (NaN for rows with id -1).
    """
    qa, ka, va = _as_f64(q), _as_f64(k), _as_f64(v)
    N, H, D = qa.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = np.full((N, H, D), np.nan)
    lse = np.full((H, N), np.nan)
    for h in range(H):
        for i in range(N):
            if segment_of_row[i] < 0:
                continue
            scores = []
            for j in range(N):
                if segment_of_row[j] == segment_of_row[i]:
                    acc = 0.0
                    for d in range(D):
                        acc += qa[i, h, d] * ka[j, h, d]
                    scores.append(scale * acc)
                else:
                    scores.append(-math.inf)
            mx = max(scores)
            ex = [math.exp(s - mx) if s != -math.inf else 0.0 for s in scores]
            tot = math.fsum(ex)
            for d in range(D):
                # masked keys take no part at all (not even as 0 * v_j, which is NaN for a NaN row)
                o[i, h, d] = math.fsum(ex[j] * va[j, h, d] for j in range(N)
                                       if segment_of_row[j] == segment_of_row[i]) / tot
            lse[h, i] = mx + math.log(tot)
    return o, lse
