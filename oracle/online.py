"""Online (streaming) forms of the same quantities.  TEST INFRASTRUCTURE ONLY.

These restate the pages' recurrences so that the three-pass oracle in
``oracle.reference`` can be checked against a second, differently ordered route to
the same numbers.  They are never compared with the CUDA path directly.
"""

from __future__ import annotations

import math

import numpy as np

from .reference import visible_mask


def online_weighted_sum(scores, values) -> float:
    """Scalar online weighted sum (m, l, u) of the lihaoran.work FlashAttention note,
    section "为什么不能平均各块的softmax".

    For each new score a with value v: m' = max(m, a); the old totals are multiplied
    by exp(m - m'), the new term has weight exp(a - m'):
        l' = exp(m - m') l + exp(a - m'),   u' = exp(m - m') u + exp(a - m') v,
    and the result is u / l.  Starts from m = -inf, l = u = 0.
    """
    m, l, u = -math.inf, 0.0, 0.0
    for a, val in zip(scores, values):
        m_new = max(m, a)
        old = math.exp(m - m_new)   # exp(-inf) = 0 on the first term
        w = math.exp(a - m_new)
        l = old * l + w
        u = old * u + w * val
        m = m_new
    return u / l


def online_state(xs) -> tuple[float, float]:
    """Element-by-element (m, l) state.

    "Softmax 数值稳定性与 IO-Aware Attention：从在线归一化到 FlashAttention", §四:
    m_{k+1} = max(m_k, x_{k+1}),  l_{k+1} = l_k exp(m_k - m_{k+1}) + exp(x_{k+1} - m_{k+1}),
    from m = -inf, l = 0.
    """
    m, l = -math.inf, 0.0
    for x in xs:
        m_new = max(m, float(x))
        l = l * math.exp(m - m_new) + math.exp(float(x) - m_new)
        m = m_new
    return m, l


def merge_state(a, b) -> tuple[float, float]:
    """Merge of two local states, same page §4.1:
    m = max(m_a, m_b),  l = l_a exp(m_a - m) + l_b exp(m_b - m).

    The page does not treat the empty state (m = -inf, l = 0).  Reading taken: an
    empty side contributes nothing, so that two empty states merge to (-inf, 0)
    instead of evaluating exp(-inf - (-inf)).
    """
    ma, la = a
    mb, lb = b
    if ma == -math.inf:
        return mb, lb
    if mb == -math.inf:
        return ma, la
    m = max(ma, mb)
    return m, la * math.exp(ma - m) + lb * math.exp(mb - m)


def tiled_attention_forward(q, k, v, scale: float, causal: bool, block: int):
    """The per-Q-tile loop of "Softmax 数值稳定性与 IO-Aware Attention" §七, in float64.

    For each query row (a Q tile of height one): m = -inf, l = 0, O = 0; for each K/V
    tile of ``block`` keys: S = scale Q K_j^T, m_new = max(m, rowmax S),
    P = exp(S - m_new), alpha = exp(m - m_new), l = alpha l + rowsum P,
    O = alpha O + P V_j; finally O = O / l and LSE = m + ln l.  Masked keys carry
    s = -inf (P = 0).  A tile in which every key of the row is masked leaves the
    state unchanged (the empty-state reading of ``merge_state``).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    out = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    visible = visible_mask(np.arange(N), N, causal)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                m, l, o = -np.inf, 0.0, np.zeros(d)
                for j0 in range(0, N, block):
                    j1 = min(j0 + block, N)
                    s = scale * (k[b, h, j0:j1] @ q[b, h, i])
                    s = np.where(visible[i, j0:j1], s, -np.inf)
                    m_new = max(m, s.max())
                    if m_new == -np.inf:
                        continue
                    p = np.exp(s - m_new)
                    alpha = math.exp(m - m_new)
                    l = alpha * l + p.sum()
                    o = alpha * o + p @ v[b, h, j0:j1]
                    m = m_new
                out[b, h, i] = o / l
                lse[b, h, i] = m + math.log(l)
    return out, lse


def combine_partials(o_parts, lse_parts):
    """Merge attention results computed over disjoint key subsets.

    lihaoran.work FlashAttention note, section "为什么不能平均各块的softmax": results of
    blocks normalised separately cannot be averaged; they must be brought to the same
    reference maximum.  With each part s given as its normalised output O_s and its
    LSE_s = m_s + ln l_s, the common reference is M = max_s LSE_s, the weights are
    w_s = exp(LSE_s - M), and O = sum_s w_s O_s / sum_s w_s, LSE = M + ln sum_s w_s
    ("Softmax 数值稳定性与 IO-Aware Attention", §4.1 merge rule applied to (O, l) pairs).
    A part with LSE_s = -inf (no visible key) has weight 0.

    o_parts: [S, ..., d]; lse_parts: [S, ...].  Returns (O [..., d], LSE [...]).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = lse_parts.max(axis=0)
    w = np.where(np.isneginf(lse_parts), 0.0, np.exp(lse_parts - M))
    wsum = w.sum(axis=0)
    o = (w[..., None] * o_parts).sum(axis=0) / wsum[..., None]
    return o, M + np.log(wsum)
