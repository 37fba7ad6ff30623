"""Gradients of standard attention in float64.  TEST INFRASTRUCTURE ONLY.

"Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention" §7.2 says that the
backward pass keeps only a few statistics of the forward (here LSE) and recomputes the
local scores instead of storing the probability matrix; §九 9.1 asks for gradients to be
checked against a high-precision CPU reference.  The pages print no gradient formula,
so the reading taken here is the plainest one: the gradients are those of the exact
attention function of the forward,

    S = scale * Q K^T (masked keys -> -inf),  P = softmax_rows(S),  O = P V,

with respect to Q, K and V, for an upstream gradient dO = dL/dO.  By the chain rule:

    dV = P^T dO
    dP = dO V^T
    dS = P * (dP - D),   D_i = sum_j P_ij dP_ij  (= sum_c dO_ic O_ic)
    dQ = scale * dS K
    dK = scale * dS^T Q

The dS line is the softmax Jacobian, dP_ij/dS_ik = P_ij (delta_jk - P_ik), applied to
a row; masked entries have P = 0 and so dS = 0.  These lines are pinned to the
derivative's own definition by central finite differences of sum(O * dO) (the forward
oracle, itself pinned) in ``tests/test_oracle_bwd_pins.py``, and to invariants that
follow from softmax rows summing to one.
"""

from __future__ import annotations

import numpy as np

from .reference import attention_forward, visible_mask


def _f64(*arrays):
    return [np.asarray(a, dtype=np.float64) for a in arrays]


def _check_shapes(q, k, v, do):
    if q.ndim != 4 or any(t.shape != q.shape for t in (k, v, do)):
        raise ValueError("q, k, v, dO must all be [B, H, N, d] of one shape")


def attention_backward(q, k, v, do, scale: float, causal: bool, block: int = 512):
    """(dQ, dK, dV) of standard attention, float64, all rows.

    q, k, v, do: [B, H, N, d] (any float dtype; converted exactly to float64).
    Query rows are taken ``block`` at a time so that one block of the score matrix
    is held at once; every row of P is complete (all N keys), so the blocking only
    bounds memory and changes no formula.
    """
    q, k, v, do = _f64(q, k, v, do)
    _check_shapes(q, k, v, do)
    B, H, N, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, block):
                rows = np.arange(r0, min(N, r0 + block))
                s = scale * (q[b, h, rows] @ k[b, h].T)              # S rows
                s = np.where(visible_mask(rows, N, causal), s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                p = e / e.sum(axis=1, keepdims=True)                 # P rows
                dp = do[b, h, rows] @ v[b, h].T                      # dP = dO V^T
                dd = (p * dp).sum(axis=1, keepdims=True)             # D_i
                ds = p * (dp - dd)                                   # dS
                dv[b, h] += p.T @ do[b, h, rows]                     # dV = P^T dO
                dq[b, h, rows] = scale * (ds @ k[b, h])              # dQ = scale dS K
                dk[b, h] += scale * (ds.T @ q[b, h, rows])           # dK = scale dS^T Q
    return dq, dk, dv


def attention_backward_rows(q, k, v, do, scale: float, causal: bool, bh, q_rows, k_rows,
                            block: int = 512):
    """The same gradients at a sample: dQ at query rows ``q_rows`` and dK, dV at key
    rows ``k_rows`` of head ``bh = (b, h)``.  float64.

    dK_j and dV_j need P_ij for every query i, so the per-row statistics (m, l via the
    forward oracle's LSE, and D_i = sum_c dO_ic O_ic) are first computed for all queries
    of the head; then only the requested rows and columns of dS are formed.
    Returns (dq [len(q_rows), d], dk [len(k_rows), d], dv [len(k_rows), d]).
    """
    q, k, v, do = _f64(q, k, v, do)
    _check_shapes(q, k, v, do)
    b, h = bh
    N = q.shape[2]
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    qh, kh, vh, doh = q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], do[b:b + 1, h:h + 1]
    o_all = np.empty((N, q.shape[3]))
    lse_all = np.empty(N)
    for r0 in range(0, N, block):
        rows = np.arange(r0, min(N, r0 + block))
        o_blk, lse_blk = attention_forward(qh, kh, vh, scale, causal, rows=rows)
        o_all[rows] = o_blk[0, 0]
        lse_all[rows] = lse_blk[0, 0]
    d_all = (doh[0, 0] * o_all).sum(axis=1)                       # D_i = sum_c dO_ic O_ic

    # dQ rows: complete score rows of the sampled queries.
    s = scale * (qh[0, 0, q_rows] @ kh[0, 0].T)
    vis = visible_mask(q_rows, N, causal)
    p = np.where(vis, np.exp(np.where(vis, s, 0.0) - lse_all[q_rows, None]), 0.0)
    dp = doh[0, 0, q_rows] @ vh[0, 0].T
    ds = p * (dp - d_all[q_rows, None])
    dq = scale * (ds @ kh[0, 0])

    # dK, dV rows: complete score columns of the sampled keys.
    all_q = np.arange(N)
    s_t = scale * (qh[0, 0] @ kh[0, 0, k_rows].T)                  # [N, len(k_rows)]
    vis_t = visible_mask(all_q, N, causal)[:, k_rows]
    p_t = np.where(vis_t, np.exp(np.where(vis_t, s_t, 0.0) - lse_all[:, None]), 0.0)
    dp_t = doh[0, 0] @ vh[0, 0, k_rows].T
    ds_t = p_t * (dp_t - d_all[:, None])
    dk = scale * (ds_t.T @ qh[0, 0])
    dv = p_t.T @ doh[0, 0]
    return dq, dk, dv
