"""Pins of the fp64 backward oracle to facts other than its own formulas (CPU only).

The main pin is the definition of the derivative: central finite differences of the
scalar L = sum(O * dO), with O from the forward oracle (itself pinned in
test_oracle_pins.py), must match every entry of dQ, dK and dV.  The others follow from
softmax rows summing to one (rows of dS sum to zero, so the dK rows of a head sum to
zero, dV rows sum to the dO rows, and identical keys give dQ = 0) and from cases with
a closed form.  The mutation tests plant plausible mistakes in copies of the backward
oracle and check that some pin rejects each.
"""

import numpy as np
import pytest

import oracle


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def _loss(q, k, v, do, scale, causal):
    o, _ = oracle.attention_forward(q, k, v, scale, causal)
    return float((o * do).sum())


def _finite_differences(q, k, v, do, scale, causal, h=1e-5):
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(args[which])
        it = np.nditer(g, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = args[which][idx]
            args[which][idx] = x0 + h
            up = _loss(*args, do, scale, causal)
            args[which][idx] = x0 - h
            dn = _loss(*args, do, scale, causal)
            args[which][idx] = x0
            g[idx] = (up - dn) / (2 * h)
        grads.append(g)
    return grads  # dQ, dK, dV


# ----------------------------------------------------------------------------
# Pin functions: each takes a backward function bwd(q, k, v, do, scale, causal)
# returning (dq, dk, dv), and raises AssertionError when the pin fails.
# ----------------------------------------------------------------------------

def pin_finite_differences(bwd):
    for causal, shape, seed in ((False, (1, 2, 5, 3), 11), (True, (1, 1, 6, 4), 12)):
        q, k, v, do = (_rand(shape, seed + 100 * i) for i in range(4))
        scale = 0.7
        ref = _finite_differences(q, k, v, do, scale, causal)
        got = bwd(q, k, v, do, scale, causal)
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            err = np.abs(np.asarray(a) - b).max()
            assert err < 1e-7, (name, causal, err)


def pin_invariants(bwd):
    """Rows of dS sum to zero, so sum_j dK_j = 0; rows of P sum to one, so
    sum_j dV_j = sum_i dO_i; identical keys make every score row constant, so dQ = 0."""
    shape = (2, 2, 37, 8)
    for causal in (False, True):
        q, k, v, do = (_rand(shape, 21 + i) for i in range(4))
        dq, dk, dv = bwd(q, k, v, do, 0.35, causal)
        assert np.abs(dk.sum(axis=2)).max() < 1e-12 * np.abs(dk).sum(), causal
        assert np.allclose(dv.sum(axis=2), do.sum(axis=2), rtol=0, atol=1e-12), causal
        k_same = np.broadcast_to(k[:, :, :1], k.shape).copy()
        dq_same, _, _ = bwd(q, k_same, v, do, 0.35, causal)
        assert np.abs(dq_same).max() < 1e-12, causal


def pin_closed_forms(bwd):
    # One key: P = 1, so dV = dO and dQ = dK = 0.
    q, k, v, do = (_rand((1, 1, 1, 5), 31 + i) for i in range(4))
    dq, dk, dv = bwd(q, k, v, do, 0.5, False)
    assert np.array_equal(dv, do)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
    # Causal row 0 sees only key 0: dQ_0 = 0.
    q, k, v, do = (_rand((1, 1, 7, 4), 41 + i) for i in range(4))
    dq, _, _ = bwd(q, k, v, do, 0.5, True)
    assert np.abs(dq[0, 0, 0]).max() == 0
    # One query that matters, two keys, d = 1, non-causal.  Row 1 of dO is zero, so only
    # query 0 enters L.  With P_0 = (p, 1-p), p = sigmoid(s0 - s1):
    # dL/ds0 = -dL/ds1 = p (1 - p) (dO_0 v0 - dO_0 v1), dQ_0 = scale (dL/ds0 k0 + dL/ds1 k1),
    # and dV_0 = P_00 dO_0 = p dO_0.
    q = np.array([[[[0.3], [0.0]]]])
    k = np.array([[[[1.2], [-0.4]]]])
    v = np.array([[[[2.0], [-1.0]]]])
    do = np.array([[[[0.5], [0.0]]]])
    scale = 1.5
    dq, dk, dv = bwd(q, k, v, do, scale, False)
    s0, s1 = scale * 0.3 * 1.2, scale * 0.3 * -0.4
    p = 1.0 / (1.0 + np.exp(s1 - s0))
    g0 = p * (1 - p) * (0.5 * 2.0 - 0.5 * -1.0)
    assert abs(dq[0, 0, 0, 0] - scale * (g0 * 1.2 - g0 * -0.4)) < 1e-14
    assert abs(dv[0, 0, 0, 0] - (p * 0.5 + 0.5 * 0.0)) < 1e-14


BWD_PINS = [pin_finite_differences, pin_invariants, pin_closed_forms]


def test_finite_differences():
    pin_finite_differences(oracle.attention_backward)


def test_invariants():
    pin_invariants(oracle.attention_backward)


def test_closed_forms():
    pin_closed_forms(oracle.attention_backward)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_full(causal):
    shape = (2, 3, 45, 8)
    q, k, v, do = (_rand(shape, 51 + i) for i in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.4, causal, block=16)
    q_rows = np.array([0, 7, 44, 16])
    k_rows = np.array([44, 0, 3, 31])
    for bh in ((0, 0), (1, 2)):
        sq, sk, sv = oracle.attention_backward_rows(q, k, v, do, 0.4, causal, bh, q_rows, k_rows,
                                                    block=16)
        b, h = bh
        assert np.allclose(sq, dq[b, h, q_rows], rtol=1e-12, atol=1e-13)
        assert np.allclose(sk, dk[b, h, k_rows], rtol=1e-12, atol=1e-13)
        assert np.allclose(sv, dv[b, h, k_rows], rtol=1e-12, atol=1e-13)


def test_block_size_changes_nothing():
    shape = (1, 2, 50, 6)
    q, k, v, do = (_rand(shape, 61 + i) for i in range(4))
    a = oracle.attention_backward(q, k, v, do, 0.3, True, block=7)
    b = oracle.attention_backward(q, k, v, do, 0.3, True, block=512)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------------
# Mutation tests: plausible mistakes must fail at least one pin.
# ----------------------------------------------------------------------------

def _mutant(kind):
    def bwd(q, k, v, do, scale, causal):
        q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
        B, H, N, d = q.shape
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        keys = np.arange(N)[None, :]
        rows = np.arange(N)[:, None]
        vis = keys <= rows if causal else np.ones((N, N), bool)
        if kind == "causal_flipped" and causal:
            vis = keys >= rows
        for b in range(B):
            for h in range(H):
                s = scale * (q[b, h] @ k[b, h].T)
                s = np.where(vis, s, -np.inf)
                e = np.exp(s - s.max(axis=1, keepdims=True))
                p = e / e.sum(axis=1, keepdims=True)
                dp = do[b, h] @ v[b, h].T
                if kind == "dp_transposed":
                    dp = dp.T
                dd = (p * dp).sum(axis=1, keepdims=True)
                ds = p * dp if kind == "no_d_term" else p * (dp - dd)
                if kind == "ds_sign":
                    ds = -ds
                dv[b, h] = (p @ do[b, h]) if kind == "dv_not_transposed" else p.T @ do[b, h]
                sq = 1.0 if kind == "dq_no_scale" else scale
                dq[b, h] = sq * (ds @ k[b, h])
                dk[b, h] = scale * (ds.T @ q[b, h]) if kind != "dk_uses_k" else scale * (ds.T @ k[b, h])
        return dq, dk, dv
    return bwd


def _fails_some_pin(bwd):
    for pin in BWD_PINS:
        try:
            pin(bwd)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            return True
    return False


def test_unmutated_copy_passes():
    with np.errstate(all="ignore"):
        assert not _fails_some_pin(_mutant("none"))


@pytest.mark.parametrize("kind", ["no_d_term", "ds_sign", "dv_not_transposed", "dq_no_scale",
                                  "dk_uses_k", "dp_transposed", "causal_flipped"])
def test_mutants_are_caught(kind):
    with np.errstate(all="ignore"):
        assert _fails_some_pin(_mutant(kind))
