"""Three-pass fp64 definitions: the oracle proper.  TEST INFRASTRUCTURE ONLY.

Readings of points the pages leave open (each is also listed with its reason in
the repository's design notes):

* Layout: every attention tensor is a contiguous [B, H, N, d] array; K and V have
  the same N as Q (self-attention).  The pages give no layout.
* Scale: the scores are s_ij = scale * q_i . k_j, scale applied before the softmax.
  "为什么 Flash Attention 算出来的结果和标准注意力有微小差异？有损但值得" writes
  softmax(QK^T/sqrt(d)) V; "Softmax 数值稳定性与 IO-Aware Attention" §七 writes
  S = QK^T with no factor.  ``scale`` is a parameter, 1/sqrt(d) in the workloads.
* Causal: top-left aligned, key j is visible to query i iff j <= i.
* LSE: LSE_i = m_i + ln l_i, natural log, in units of the scaled scores.  The pages
  only say that fewer statistics are kept for the backward pass
  ("Softmax 数值稳定性与 IO-Aware Attention" §7.2).
"""

from __future__ import annotations

import numpy as np


def visible_mask(query_rows: np.ndarray, n_keys: int, causal: bool) -> np.ndarray:
    """Boolean [len(query_rows), n_keys]: True where key j is visible to query i.

    Without a mask every key is visible.  With the causal mask (named, not defined,
    in "Softmax 数值稳定性与 IO-Aware Attention" §八 and §9.2) key j is visible to
    query i iff j <= i.
    """
    rows = np.asarray(query_rows, dtype=np.int64).reshape(-1, 1)
    keys = np.arange(n_keys, dtype=np.int64).reshape(1, -1)
    if causal:
        return keys <= rows
    return np.ones((rows.shape[0], n_keys), dtype=bool)


def row_state(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-row softmax state (m, l) of a [rows, len] array, in float64.

    "Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention", §二 2.1
    (subtract the maximum) and §三 (three passes): pass one takes m = max_t x_t, pass
    two takes l = sum_t exp(x_t - m).  Pass three (the normalised outputs) is not
    part of the state.  The inputs are converted to float64 exactly as stored.
    """
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 2 or x.shape[1] < 1:
        raise ValueError("row_state expects a [rows, len] array with len >= 1")
    m = x.max(axis=1)                                   # pass 1
    l = np.exp(x - m[:, None]).sum(axis=1)              # pass 2
    return m, l


def softmax_rows(x: np.ndarray) -> np.ndarray:
    """Row-wise softmax of a [rows, len] array, in float64.

    "Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention", §三: pass one
    m = max_t x_t, pass two l = sum_t exp(x_t - m), pass three y_t = exp(x_t - m) / l.
    """
    m, l = row_state(x)
    x = np.asarray(x, dtype=np.float64)
    return np.exp(x - m[:, None]) / l[:, None]          # pass 3


def attention_forward(q, k, v, scale: float, causal: bool, rows=None):
    """Standard attention in float64; returns (O, LSE).

    "Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention", §七
    ("标准 Attention 可以写成 ..."): S = Q K^T, P = softmax(S), O = P V, with the
    softmax taken in the three passes of §三 on each score row.  One score row (or
    one block of requested rows) of one head is materialised at a time.

    q, k, v: arrays [B, H, N, d] (any float dtype; converted exactly to float64).
    rows:    optional 1-D array of query indices; default all N rows.
    Returns O [B, H, len(rows), d] and LSE [B, H, len(rows)], both float64, where
    LSE_i = m_i + ln l_i with m_i = max_j s_ij and l_i = sum_j exp(s_ij - m_i) over
    the visible keys j.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B, H, N, d] of one shape")
    B, H, N, d = q.shape
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    visible = visible_mask(rows, N, causal)
    out = np.empty((B, H, rows.size, d), dtype=np.float64)
    lse = np.empty((B, H, rows.size), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h, rows, :] @ k[b, h].T)          # S = scale * Q K^T
            s = np.where(visible, s, -np.inf)                    # masked keys drop out
            m = s.max(axis=1)                                    # pass 1: row max
            e = np.exp(s - m[:, None])                           # exp(s - m); 0 where masked
            l = e.sum(axis=1)                                    # pass 2: denominator
            p = e / l[:, None]                                   # pass 3: P = softmax(S)
            out[b, h] = p @ v[b, h]                              # O = P V
            lse[b, h] = m + np.log(l)
    return out, lse
