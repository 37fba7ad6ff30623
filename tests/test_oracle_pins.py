"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each pin comes from the pages or from mathematics, never from the oracle's own
formula retyped: the worked example the lihaoran.work note prints, the +1000 shift
it checks, its 390-row randomised recipe, the chunk-merge check of
"Softmax 数值稳定性与 IO-Aware Attention" §4.1, brute force with a different route
(plain exponentials, no max subtraction, compensated sums), and closed forms.
The mutation tests at the end plant plausible mistakes in copies of the oracle and
check that at least one pin rejects each of them.
"""

import math
import os
import random

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _scores_as_attention(scores, values):
    """Express one score row as attention with d = 1: q = 1, k_j = s_j, scale = 1.

    Then s_j = q k_j exactly, so the attention output is the weighted sum of the
    values.  The value row is padded into the same N (one value per key)."""
    n = len(scores)
    q = np.zeros((1, 1, n, 1))
    q[0, 0, 0, 0] = 1.0
    k = np.asarray(scores, dtype=np.float64).reshape(1, 1, n, 1)
    v = np.asarray(values, dtype=np.float64).reshape(1, 1, n, 1)
    return q, k, v


# ----------------------------------------------------------------------------
# Pin functions (shared by the tests and by the mutation tests).  Each raises
# AssertionError on a mismatch.
# ----------------------------------------------------------------------------

def pin_worked_example(attn):
    g = _golden()
    q, k, v = _scores_as_attention(g["scores"], g["values"])
    o, lse = attn(q, k, v, 1.0, False, rows=np.array([0]))
    assert round(float(o[0, 0, 0, 0]), 6) == g["result_6dp"][0]
    # LSE of [0, 1, 2] has the closed form ln(1 + e + e^2).
    assert abs(float(lse[0, 0, 0]) - math.log(1 + math.e + math.e ** 2)) < 1e-13


def pin_shift(attn):
    """Adding c to every score leaves O unchanged and moves LSE by exactly c.
    The shift is injected through an extra head dimension: q' = [q, 1], k' = [k, c]."""
    g = _golden()
    c = g["shift"][0]
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 2, 5, 3))
    k = rng.standard_normal((1, 2, 5, 3))
    v = rng.standard_normal((1, 2, 5, 3))
    o, lse = attn(q, k, v, 0.5, False)
    q2 = np.concatenate([q, np.full((1, 2, 5, 1), 2.0)], axis=-1)   # 0.5 * 2 = 1
    k2 = np.concatenate([k, np.full((1, 2, 5, 1), c)], axis=-1)
    v2 = np.concatenate([v, np.zeros((1, 2, 5, 1))], axis=-1)
    o2, lse2 = attn(q2, k2, v2, 0.5, False)
    assert np.allclose(o2[..., :3], o, rtol=g["shift_rel_tol"][0], atol=1e-12)
    assert np.allclose(lse2 - c, lse, rtol=0, atol=1e-9)


def pin_brute_force(attn, causal):
    """Tiny attention by enumeration: plain exponentials (no max subtraction, the
    values are small), Python loops and math.fsum -- another route to the same sums."""
    rng = random.Random(11 + int(causal))
    for N in range(1, 5):
        for d in range(1, 5):
            for H in (1, 2):
                q = np.array([[[[rng.uniform(-2, 2) for _ in range(d)] for _ in range(N)] for _ in range(H)]])
                k = np.array([[[[rng.uniform(-2, 2) for _ in range(d)] for _ in range(N)] for _ in range(H)]])
                v = np.array([[[[rng.uniform(-2, 2) for _ in range(d)] for _ in range(N)] for _ in range(H)]])
                scale = rng.uniform(0.2, 1.5)
                o, lse = attn(q, k, v, scale, causal)
                for h in range(H):
                    for i in range(N):
                        keys = [j for j in range(N) if (not causal or j <= i)]
                        w = {j: math.exp(scale * math.fsum(q[0, h, i, t] * k[0, h, j, t] for t in range(d)))
                             for j in keys}
                        z = math.fsum(w.values())
                        assert abs(lse[0, h, i] - math.log(z)) < 1e-12
                        for t in range(d):
                            ref = math.fsum(w[j] * v[0, h, j, t] for j in keys) / z
                            assert abs(o[0, h, i, t] - ref) < 1e-12


def pin_closed_forms(attn):
    rng = np.random.default_rng(3)
    # Uniform V rows: every output row equals that row exactly (weights sum to one).
    q = rng.standard_normal((1, 1, 7, 4))
    k = rng.standard_normal((1, 1, 7, 4))
    vrow = rng.standard_normal(4)
    v = np.broadcast_to(vrow, (1, 1, 7, 4)).copy()
    for causal in (False, True):
        o, _ = attn(q, k, v, 0.7, causal)
        assert np.allclose(o[0, 0], vrow, rtol=0, atol=1e-14)
    # Causal row 0 sees only key 0: O_0 = v_0 and LSE_0 = s_00.
    v = rng.standard_normal((1, 1, 7, 4))
    o, lse = attn(q, k, v, 0.7, True)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-14)
    assert abs(lse[0, 0, 0] - 0.7 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-13
    # Two keys: softmax reduces to the logistic function.
    q2 = rng.standard_normal((1, 1, 2, 3))
    k2 = rng.standard_normal((1, 1, 2, 3))
    v2 = rng.standard_normal((1, 1, 2, 3))
    o2, lse2 = attn(q2, k2, v2, 1.3, False)
    for i in range(2):
        s0 = 1.3 * float(q2[0, 0, i] @ k2[0, 0, 0])
        s1 = 1.3 * float(q2[0, 0, i] @ k2[0, 0, 1])
        sig = 1.0 / (1.0 + math.exp(s0 - s1))
        assert np.allclose(o2[0, 0, i], v2[0, 0, 0] + sig * (v2[0, 0, 1] - v2[0, 0, 0]), atol=1e-14)
        assert abs(lse2[0, 0, i] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-13
    # One dominant logit: the output is the value at the argmax (weights of the
    # others are below exp(-700)).
    q3 = np.zeros((1, 1, 4, 1))
    q3[..., 0] = 1.0
    k3 = np.array([0.0, 800.0, 1.0, -3.0]).reshape(1, 1, 4, 1)
    v3 = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 4, 1)
    o3, lse3 = attn(q3, k3, v3, 1.0, False)
    assert np.all(o3[0, 0, :, 0] == 2.0)
    assert np.all(lse3 == 800.0)


def pin_structure(attn):
    """Permuting keys together with values leaves a non-causal output unchanged;
    the output is linear in V; rows of Q are independent (a row subset equals the
    matching rows of the full result)."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 3, 9, 5))
    k = rng.standard_normal((2, 3, 9, 5))
    v = rng.standard_normal((2, 3, 9, 5))
    w = rng.standard_normal((2, 3, 9, 5))
    o, lse = attn(q, k, v, 0.4, False)
    perm = rng.permutation(9)
    op, lsep = attn(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    assert np.allclose(op, o, atol=1e-13) and np.allclose(lsep, lse, atol=1e-13)
    ow, _ = attn(q, k, w, 0.4, False)
    olin, _ = attn(q, k, 2.0 * v - 3.0 * w, 0.4, False)
    assert np.allclose(olin, 2.0 * o - 3.0 * ow, atol=1e-12)
    for causal in (False, True):
        full, lfull = attn(q, k, v, 0.4, causal)
        sub = np.array([8, 0, 4])
        part, lpart = attn(q, k, v, 0.4, causal, rows=sub)
        assert np.allclose(part, full[:, :, sub], atol=1e-14)
        assert np.allclose(lpart, lfull[:, :, sub], atol=1e-14)


ATTENTION_PINS = [
    pin_worked_example,
    pin_shift,
    lambda a: pin_brute_force(a, False),
    lambda a: pin_brute_force(a, True),
    pin_closed_forms,
    pin_structure,
]


# ----------------------------------------------------------------------------
# Tests of the attention oracle
# ----------------------------------------------------------------------------

def test_worked_example_three_pass():
    pin_worked_example(oracle.attention_forward)


def test_worked_example_online_and_shift():
    g = _golden()
    a = oracle.online_weighted_sum(g["scores"], g["values"])
    assert round(a, 6) == g["result_6dp"][0]
    shifted = oracle.online_weighted_sum([s + g["shift"][0] for s in g["scores"]], g["values"])
    assert math.isclose(shifted, a, rel_tol=g["shift_rel_tol"][0])


def test_shift_invariance():
    pin_shift(oracle.attention_forward)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    pin_brute_force(oracle.attention_forward, causal)


def test_closed_forms():
    pin_closed_forms(oracle.attention_forward)


def test_structure():
    pin_structure(oracle.attention_forward)


def test_390_random_rows_online_vs_three_pass():
    """The note's randomised recipe: 390 rows of lengths 1 to 39, online vs
    full-weight, unmasked, scalar values."""
    rng = random.Random(390)
    count = 0
    for n in range(1, 40):
        for _ in range(10):
            scores = [rng.uniform(-30, 30) for _ in range(n)]
            values = [rng.uniform(-100, 100) for _ in range(n)]
            a = oracle.online_weighted_sum(scores, values)
            q, k, v = _scores_as_attention(scores, values)
            o, lse = oracle.attention_forward(q, k, v, 1.0, False, rows=np.array([0]))
            assert math.isclose(a, float(o[0, 0, 0, 0]), rel_tol=1e-12, abs_tol=1e-12)
            m, l = oracle.online_state(scores)
            rm, rl = oracle.row_state(np.array([scores]))
            assert m == rm[0] and math.isclose(l, rl[0], rel_tol=1e-12)
            assert math.isclose(m + math.log(l), float(lse[0, 0, 0]), rel_tol=1e-12, abs_tol=1e-12)
            count += 1
    assert count == 390


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 3, 4, 16])
def test_tiled_loop_equals_three_pass(causal, block):
    rng = np.random.default_rng(block)
    q = rng.standard_normal((1, 2, 13, 6)) * 3.0
    k = rng.standard_normal((1, 2, 13, 6))
    v = rng.standard_normal((1, 2, 13, 6))
    o, lse = oracle.attention_forward(q, k, v, 0.5, causal)
    ot, lset = oracle.tiled_attention_forward(q, k, v, 0.5, causal, block)
    assert np.allclose(ot, o, rtol=1e-12, atol=1e-13)
    assert np.allclose(lset, lse, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# Tests of the row-state oracle
# ----------------------------------------------------------------------------

def test_row_state_closed_forms():
    # All-equal row: m = c and l = len exactly (every term is exp(0) = 1).
    m, l = oracle.row_state(np.full((3, 37), 3.0))
    assert np.all(m == 3.0) and np.all(l == 37.0)
    # Length one: l = 1.
    m, l = oracle.row_state(np.array([[-5.5], [1e4], [0.0]]))
    assert np.all(l == 1.0) and list(m) == [-5.5, 1e4, 0.0]
    # Rows near -1e4: the plain exponential sum underflows to 0 in float64, the
    # max-subtracted one does not (the overflow/underflow point of §二).
    x = -1e4 + np.random.default_rng(1).standard_normal((2, 50))
    assert np.all(np.exp(x).sum(axis=1) == 0.0)
    m, l = oracle.row_state(x)
    assert np.all(l >= 1.0) and np.all(np.isfinite(l))
    # Two values: l = 1 + exp(-|a - b|).
    m, l = oracle.row_state(np.array([[2.0, -1.5]]))
    assert m[0] == 2.0 and abs(l[0] - (1 + math.exp(-3.5))) < 1e-15


def test_row_state_shift():
    """Shifting a row by an exactly representable offset: m moves by it, l stays.
    Values are multiples of 2^-10 so that x + 1000 is exact in float64."""
    rng = np.random.default_rng(9)
    x = np.round(rng.standard_normal((4, 100)) * 3 * 1024) / 1024
    m, l = oracle.row_state(x)
    m2, l2 = oracle.row_state(x + 1000.0)
    assert np.all(m2 - m == 1000.0)
    assert np.allclose(l2, l, rtol=1e-12)


def test_chunk_merge_equals_whole_row():
    """§4.1 check: split a row into random chunks, take the state of each chunk,
    merge them in a random order; the denominator must equal the whole row's."""
    rng = random.Random(41)
    for _ in range(200):
        n = rng.randint(1, 60)
        xs = [rng.uniform(-20, 20) for _ in range(n)]
        cuts = sorted(rng.sample(range(1, n), rng.randint(0, n - 1))) if n > 1 else []
        chunks = [xs[a:b] for a, b in zip([0] + cuts, cuts + [n])]
        states = [oracle.online_state(c) for c in chunks]
        while len(states) > 1:   # random merge tree
            i = rng.randrange(len(states) - 1)
            states[i:i + 2] = [oracle.merge_state(states[i], states[i + 1])]
        m, l = states[0]
        rm, rl = oracle.row_state(np.array([xs]))
        assert m == rm[0] and math.isclose(l, rl[0], rel_tol=1e-12)


def test_merge_empty_state():
    e = (-math.inf, 0.0)
    assert oracle.merge_state(e, e) == e
    assert oracle.merge_state(e, (1.5, 2.0)) == (1.5, 2.0)
    assert oracle.merge_state((1.5, 2.0), e) == (1.5, 2.0)
    assert oracle.online_state([]) == e


# ----------------------------------------------------------------------------
# Mutation tests: plausible mistakes must fail at least one pin.
# ----------------------------------------------------------------------------

def _mutant(kind):
    def attn(q, k, v, scale, causal, rows=None):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        B, H, N, d = q.shape
        rows = np.arange(N) if rows is None else np.asarray(rows)
        out = np.empty((B, H, rows.size, d))
        lse = np.empty((B, H, rows.size))
        keys = np.arange(N)[None, :]
        if kind == "causal_strict":
            vis = keys < rows[:, None] if causal else np.ones((rows.size, N), bool)
            vis[:, 0] |= True                      # keep row 0 non-empty
        elif kind == "causal_flipped":
            vis = keys >= rows[:, None] if causal else np.ones((rows.size, N), bool)
        else:
            vis = keys <= rows[:, None] if causal else np.ones((rows.size, N), bool)
        for b in range(B):
            for h in range(H):
                sc = 1.0 if kind == "no_scale" else scale
                s = sc * (q[b, h, rows] @ k[b, h].T)
                if kind == "transposed":
                    s = sc * (k[b, h, rows] @ q[b, h].T)
                s = np.where(vis, s, -np.inf)
                m = s.max(axis=1)
                e = np.exp(s - m[:, None])
                l = e.sum(axis=1)
                vv = k[b, h] if kind == "k_as_v" else v[b, h]
                p = e / l[:, None] if kind != "no_normalise" else e
                out[b, h] = p @ vv
                lse[b, h] = (m + np.log2(l)) if kind == "log2_lse" else (
                    np.log(l) if kind == "lse_no_max" else m + np.log(l))
        return out, lse
    return attn


def _tiled_mutant_alpha_on_l_only(q, k, v, scale, causal, rows=None):
    """The mistake §七 warns about: alpha rescales l but not the O accumulator."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    rows = np.arange(N) if rows is None else np.asarray(rows)
    out = np.empty((B, H, rows.size, d))
    lse = np.empty((B, H, rows.size))
    for b in range(B):
        for h in range(H):
            for r, i in enumerate(rows):
                m, l, o = -np.inf, 0.0, np.zeros(d)
                for j in range(N):
                    if causal and j > i:
                        continue
                    s = scale * float(q[b, h, i] @ k[b, h, j])
                    m_new = max(m, s)
                    alpha = math.exp(m - m_new)
                    l = alpha * l + math.exp(s - m_new)
                    o = o + math.exp(s - m_new) * v[b, h, j]   # missing alpha * o
                    m = m_new
                out[b, h, r] = o / l
                lse[b, h, r] = m + math.log(l)
    return out, lse


def _fails_some_pin(attn):
    for pin in ATTENTION_PINS:
        try:
            pin(attn)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            return True
    return False


@pytest.mark.parametrize("kind", ["no_scale", "transposed", "k_as_v", "no_normalise",
                                  "log2_lse", "lse_no_max", "causal_strict", "causal_flipped"])
def test_mutants_are_caught(kind):
    with np.errstate(all="ignore"):
        assert _fails_some_pin(_mutant(kind))


def test_unmutated_copy_passes_and_alpha_mutant_caught():
    with np.errstate(all="ignore"):
        assert not _fails_some_pin(_mutant("none"))
        assert _fails_some_pin(_tiled_mutant_alpha_on_l_only)


# ----------------------------------------------------------------------------
# Tests of the row softmax output (pass three)
# ----------------------------------------------------------------------------

def test_softmax_rows_worked_example_weights():
    """The weights behind the worked example: e^s / (1 + e + e^2) for s = 0, 1, 2, and
    their weighted sum of the values reproduces the printed 25.752104."""
    g = _golden()
    y = oracle.softmax_rows(np.array([g["scores"]]))[0]
    z = 1 + math.e + math.e ** 2
    assert np.allclose(y, [1 / z, math.e / z, math.e ** 2 / z], rtol=1e-15, atol=0)
    assert round(float(y @ np.array(g["values"])), 6) == g["result_6dp"][0]


def test_softmax_rows_properties():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((6, 41)) * 3
    y = oracle.softmax_rows(x)
    assert np.allclose(y.sum(axis=1), 1.0, atol=1e-14)          # rows sum to one
    assert np.all(y > 0)
    assert np.all(np.argsort(y, axis=1) == np.argsort(x, axis=1))  # monotone in x
    y2 = oracle.softmax_rows(x + 1000.0)                           # shift invariance
    assert np.allclose(y2, y, rtol=1e-11, atol=0)
    # naive softmax where it does not overflow
    xs = rng.uniform(-5, 5, (3, 9))
    naive = np.exp(xs) / np.exp(xs).sum(axis=1, keepdims=True)
    assert np.allclose(oracle.softmax_rows(xs), naive, rtol=1e-14)
    # all-equal rows are uniform, length-1 rows are 1
    assert np.all(oracle.softmax_rows(np.full((2, 8), -7.0)) == 0.125)
    assert np.all(oracle.softmax_rows(np.array([[1e4], [-3.0]])) == 1.0)


# ----------------------------------------------------------------------------
# Merging results over key subsets (split-KV combine)
# ----------------------------------------------------------------------------

def _attention_on_keys(q, k, v, scale, causal, key_lo, key_hi):
    """Attention restricted to keys [key_lo, key_hi), by enumeration (plain exponentials
    and math.fsum, as in the brute-force pin).  Rows with no visible key in the range
    give LSE = -inf and O = 0 (the empty part)."""
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d))
    lse = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = [j for j in range(key_lo, key_hi) if (not causal or j <= i)]
                if not keys:
                    continue
                w = [math.exp(scale * float(q[b, h, i] @ k[b, h, j])) for j in keys]
                z = math.fsum(w)
                lse[b, h, i] = math.log(z)
                for t in range(d):
                    o[b, h, i, t] = math.fsum(wj * v[b, h, j, t] for wj, j in zip(w, keys)) / z
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_combine_of_key_splits_equals_whole(causal):
    rng = np.random.default_rng(21)
    q = rng.standard_normal((1, 2, 11, 4)) * 2
    k = rng.standard_normal((1, 2, 11, 4))
    v = rng.standard_normal((1, 2, 11, 4))
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.6, causal)
    for cuts in ([0, 11], [0, 4, 11], [0, 1, 2, 7, 11], [0, 3, 6, 9, 11]):
        parts = [_attention_on_keys(q, k, v, 0.6, causal, a, b) for a, b in zip(cuts, cuts[1:])]
        o, lse = oracle.combine_partials([p[0] for p in parts], [p[1] for p in parts])
        assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        assert np.allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)


def test_combine_rejects_averaging():
    """The note's point: averaging per-block softmax results is wrong; the combine is
    not the mean of the parts (unless their denominators agree)."""
    o_parts = np.array([[1.0], [3.0]])
    lse_parts = np.array([0.0, np.log(3.0)])
    o, lse = oracle.combine_partials(o_parts[:, None, :], lse_parts[:, None])
    assert abs(o[0, 0] - (1 * 1 + 3 * 3) / 4) < 1e-15 and abs(o[0, 0] - 2.0) > 0.4
    assert abs(lse[0] - np.log(4.0)) < 1e-15
