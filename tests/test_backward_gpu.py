"""Parity of the attention backward (fa_bwd, through the C ABI) with the fp64 oracle.

O and LSE come from the library's own forward (fa_fwd_dt), as in use; the oracle's
gradients are the exact ones of the inputs as rounded to the kernel's dtype.

Tolerance, from the arithmetic: the backward rounds three things to the 16-bit type,
each with relative error <= 2^-9 (bf16): P before dV = P^T dO, dS before dK and dQ,
and the outputs.  Over many terms the errors are independent, so the relative RMS
error of each gradient tensor should be a few times 2^-9 / sqrt(1) ~ 2e-3..4e-3;
the gate is 1e-2 on ||g - g_ref|| / ||g_ref|| and 2e-2 * max|g_ref| on the largest
element error (the forward's 2e-2 on O, taken relative to the gradient's scale).
fp16 rounds with 2^-11 and gets the same gates.  fp32 (CUDA cores, no 16-bit rounding):
unit roundoff 6e-8, dot products of <= 128 terms and sums over <= a few hundred keys keep
the relative error near 1e-6; gates 1e-5 relative RMS and 1e-4 * max|g_ref|.
"""

import numpy as np
import pytest

import oracle
from online_softmax_07_gb300 import abi, synth

from gpu_helpers import sample_rows, to_device

pytestmark = pytest.mark.gpu

REL_RMS = 1e-2
MAX_REL = 2e-2


def _run_bwd(q, k, v, do, scale, causal, dtype="bf16"):
    """fa_fwd_dt then fa_bwd through the C ABI; returns numpy fp32 dq, dk, dv."""
    import torch
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
    code = {"bf16": abi.FA_BF16, "f16": abi.FA_F16, "f32": abi.FA_F32}[dtype]
    B, H, N, d = q.shape
    tq, tk, tv, tdo = (to_device(x, tdt) for x in (q, k, v, do))
    o = torch.empty_like(tq)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    abi.fa_fwd_dt(tq, tk, tv, o, lse, B, H, N, d, scale, int(causal), code)
    ws_bytes = abi.fa_bwd_workspace_bytes(B, H, N)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    outs = [torch.full_like(tq, float("nan")) for _ in range(3)]
    abi.fa_bwd(tq, tk, tv, o, lse, tdo, *outs, B, H, N, d, scale, int(causal), ws, ws_bytes, code)
    assert abi.fa_last_device_error() == abi.FA_OK
    return [t.float().cpu().numpy() for t in outs]


def _inputs(B, H, N, d, seed, dtype="bf16"):
    q, k, v = synth.attention_inputs(B, H, N, d, seed, dtype=dtype)
    do = synth.attention_inputs(B, H, N, d, seed + 7, dtype=dtype)[0]
    return q, k, v, do


def _check(name, got, ref, rel_rms_gate=None, max_rel_gate=None):
    rel_rms_gate = REL_RMS if rel_rms_gate is None else rel_rms_gate
    max_rel_gate = MAX_REL if max_rel_gate is None else max_rel_gate
    got = got.astype(np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = got - ref
    scale = np.abs(ref).max()
    rel_rms = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    assert rel_rms <= rel_rms_gate, f"{name}: relative RMS error {rel_rms:.3e}"
    assert np.abs(err).max() <= max_rel_gate * scale, (
        f"{name}: max error {np.abs(err).max():.3e} vs max |ref| {scale:.3e}")
    return rel_rms


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 300, 64, True),
    (1, 2, 300, 128, False),
    (2, 1, 129, 128, True),
    (1, 1, 64, 64, False),
    (1, 2, 256, 128, True),
    (1, 1, 383, 64, False),
    (2, 3, 1000, 64, True),    # d = 64: up to 8 query tiles per key tile (dQ buffers reused)
    (1, 2, 1000, 64, False),
])
def test_backward_all_rows(B, H, N, d, causal):
    q, k, v, do = _inputs(B, H, N, d, seed=900 + N + d)
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv = _run_bwd(q, k, v, do, scale, causal)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, causal)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        _check(name, g, r)


def test_backward_single_key():
    """N = 1: P = 1, so dV = dO and dQ = dK = 0 (up to rounding of LSE)."""
    q, k, v, do = _inputs(1, 2, 1, 64, seed=950)
    dq, dk, dv = _run_bwd(q, k, v, do, 0.125, False)
    assert np.abs(dv - do).max() <= 2 ** -8 * np.abs(do).max()
    assert np.abs(dq).max() < 1e-3 and np.abs(dk).max() < 1e-3


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_f16(d, causal):
    q, k, v, do = _inputs(1, 2, 200, d, seed=960 + d, dtype="f16")
    dq, dk, dv = _run_bwd(q, k, v, do, 1.0 / np.sqrt(d), causal, dtype="f16")
    rq, rk, rv = oracle.attention_backward(q, k, v, do, 1.0 / np.sqrt(d), causal)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        _check(name, g, r)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_large_logits(d):
    """Q with standard deviation 4: peaky probability rows (few keys carry the weight)."""
    q, k, v = synth.attention_inputs(1, 2, 700, d, seed=965 + d, q_std=4.0)
    do = synth.attention_inputs(1, 2, 700, d, seed=966 + d)[0]
    dq, dk, dv = _run_bwd(q, k, v, do, 1.0 / np.sqrt(d), True)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, 1.0 / np.sqrt(d), True)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        _check(name, g, r)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_backward_large_score_offset(d, dtype):
    """Q and K share a constant 45 in dimension 0, so every score carries +2025: the
    softmax (and every gradient but the shifted dimension's) is that of the problem
    without it, while LSE/scale is ~2025.  The key-outer kernels add -LSE/scale through
    the tensor core as a high and a low bf16 term; the high term alone would be off by up
    to 4 there (a factor 1.65 in P at scale 1/8), the pair is within about 0.01.
    Dimension 0 of dQ is 45·scale·(row sum of dS) = 0 exactly, so there only the rounding
    of dS shows (times 45), and that of dK is 45× the others: both gradients are compared
    on dimensions 1 .. d-1, dV in full (a wrong P shows in all three)."""
    q, k, v, do = _inputs(1, 2, 500, d, seed=2600 + d, dtype=dtype)
    q[..., 0] = 45.0
    k[..., 0] = 45.0
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv = _run_bwd(q, k, v, do, scale, True, dtype=dtype)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, True)
    _check("dQ", dq[..., 1:], rq[..., 1:])
    _check("dK", dk[..., 1:], rk[..., 1:])
    _check("dV", dv, rv)


def _dq_close(got, ref):
    """dQ at d = 64 is summed in fp32 by several blocks in a varying order: two runs may
    differ by the rounding of those sums, at most about one 16-bit ulp per element."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = 2.0 ** -7 * np.abs(ref) + 1e-5 * np.abs(ref).max()
    return bool(np.all(np.abs(got - ref) <= tol))


@pytest.mark.parametrize("d", [64, 128])
def test_backward_deterministic(d):
    """dK and dV elements are written once by one block: two runs agree bitwise; dQ too
    at d = 128, and within the rounding of its fp32 sums at d = 64."""
    q, k, v, do = _inputs(1, 4, 1000, d, seed=970 + d)
    a = _run_bwd(q, k, v, do, 0.09, True)
    b = _run_bwd(q, k, v, do, 0.09, True)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    if d == 128:
        assert np.array_equal(a[0], b[0])
    else:
        assert _dq_close(a[0], b[0])


@pytest.mark.parametrize("B,H,N,d,causal,n_sample", [
    (2, 16, 8192, 128, True, 48),
    (2, 16, 8191, 128, True, 32),
    (4, 16, 4096, 64, False, 48),
])
def test_backward_workload_sampled(B, H, N, d, causal, n_sample):
    """Workload sizes: sampled query rows (dQ) and key rows (dK, dV) of two heads against
    the oracle, plus the sum invariants over every head."""
    q, k, v, do = _inputs(B, H, N, d, seed=980 + d)
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv = _run_bwd(q, k, v, do, scale, causal)
    rows = sample_rows(N, n_sample, seed=N + d)
    for bh in ((0, 0), (B - 1, H - 1)):
        rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, scale, causal, bh, rows, rows)
        b, h = bh
        _check("dQ", dq[b, h, rows], rq)
        _check("dK", dk[b, h, rows], rk)
        _check("dV", dv[b, h, rows], rv)
    # Rows of P sum to one: sum_j dV_j = sum_i dO_i; rows of dS sum to zero: sum_j dK_j = 0.
    dv_sum = dv.astype(np.float64).sum(axis=2)
    do_sum = do.astype(np.float64).sum(axis=2)
    assert np.abs(dv_sum - do_sum).max() <= 1e-2 * np.abs(dv).sum(axis=2).max()
    dk_sum = np.abs(dk.astype(np.float64).sum(axis=2))
    assert (dk_sum <= 1e-2 * np.abs(dk.astype(np.float64)).sum(axis=2)).all()


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 1, 128, 64, False),   # the fp32 configuration
    (1, 1, 128, 64, True),
    (2, 2, 100, 17, True),
    (1, 2, 257, 128, False),
    (1, 1, 1, 1, False),
    (1, 3, 70, 1, True),
])
def test_backward_f32(B, H, N, d, causal):
    q, k, v, do = _inputs(B, H, N, d, seed=1900 + N + d, dtype="f32")
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv = _run_bwd(q, k, v, do, scale, causal, dtype="f32")
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, causal)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        if np.abs(r).max() == 0:          # N = 1: dQ = dK = 0 exactly
            assert np.abs(g).max() < 1e-6
            continue
        _check(name, g, r, rel_rms_gate=1e-5, max_rel_gate=1e-4)


def test_backward_noncausal_d128_sampled():
    B, H, N, d = 1, 4, 4096, 128
    q, k, v, do = _inputs(B, H, N, d, seed=2100)
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv = _run_bwd(q, k, v, do, scale, False)
    rows = sample_rows(N, 40, seed=2101)
    for bh in ((0, 1), (0, 3)):
        rq, rk, rv = oracle.attention_backward_rows(q, k, v, do, scale, False, bh, rows, rows)
        b, h = bh
        _check("dQ", dq[b, h, rows], rq)
        _check("dK", dk[b, h, rows], rk)
        _check("dV", dv[b, h, rows], rv)


def test_backward_from_splitkv_forward():
    """fa_bwd takes O and LSE from the split-KV forward as well (same LSE convention):
    the gradients agree with those from the plain forward's O and LSE."""
    import torch
    B, H, N, d = 1, 2, 3000, 128
    q, k, v, do = _inputs(B, H, N, d, seed=2200)
    scale = 1.0 / np.sqrt(d)
    tq, tk, tv, tdo = (to_device(x, torch.bfloat16) for x in (q, k, v, do))
    grads = []
    for splits in (1, 4):
        o = torch.empty_like(tq)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        if splits == 1:
            abi.fa_fwd(tq, tk, tv, o, lse, B, H, N, d, scale, 1)
        else:
            nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits)
            ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            abi.fa_fwd_splitkv(tq, tk, tv, o, lse, B, H, N, d, scale, 1, splits, ws, nbytes,
                               abi.FA_BF16)
        nb = abi.fa_bwd_workspace_bytes(B, H, N)
        wsb = torch.empty(nb, dtype=torch.uint8, device="cuda")
        outs = [torch.empty_like(tq) for _ in range(3)]
        abi.fa_bwd(tq, tk, tv, o, lse, tdo, *outs, B, H, N, d, scale, 1, wsb, nb, abi.FA_BF16)
        assert abi.fa_last_device_error() == abi.FA_OK
        grads.append([t.float().cpu().numpy() for t in outs])
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale, True)
    for (name, r), g1, g4 in zip((("dQ", rq), ("dK", rk), ("dV", rv)), grads[0], grads[1]):
        _check(name, g1, r)
        _check(name, g4, r)
        # the two differ only through the rounding of O and LSE
        assert np.linalg.norm(g1 - g4) <= 5e-3 * np.linalg.norm(r), name


def _bwd_job(B, H, N, d, causal, seed):
    """Device inputs, forward outputs, workspace and NaN-filled gradient buffers."""
    import torch
    q, k, v, do = (to_device(x, torch.bfloat16) for x in _inputs(B, H, N, d, seed))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    abi.fa_fwd_dt(q, k, v, o, lse, B, H, N, d, 1 / np.sqrt(d), int(causal), abi.FA_BF16)
    nb = abi.fa_bwd_workspace_bytes(B, H, N)
    return dict(q=q, k=k, v=v, do=do, o=o, lse=lse, B=B, H=H, N=N, d=d, causal=int(causal),
                nb=nb, ws=torch.empty(nb, dtype=torch.uint8, device="cuda"),
                g=[torch.full_like(q, float("nan")) for _ in range(3)])


def _bwd_call(j, stream):
    abi.fa_bwd(j["q"], j["k"], j["v"], j["o"], j["lse"], j["do"], *j["g"], j["B"], j["H"], j["N"],
               j["d"], 1 / np.sqrt(j["d"]), j["causal"], j["ws"], j["nb"], abi.FA_BF16, stream)


def test_backward_concurrent_threads():
    """Three host threads, each with its own stream and inputs, call fa_bwd at the same
    time: at d = 128 the dQ pass runs on a stream of the library that all calls share,
    forked from and joined to each caller's stream; at d = 64 the dQ accumulator sits in
    each call's own workspace.  Every result must equal the sequential one (dQ at d = 64
    within the rounding of its fp32 sums)."""
    import threading

    import torch
    jobs = [_bwd_job(1, 3, 700 + 130 * t, (64, 128, 64)[t], t % 2, 2300 + t) for t in range(3)]
    refs = []
    for j in jobs:
        _bwd_call(j, torch.cuda.current_stream())
        torch.cuda.synchronize()
        refs.append([g.clone() for g in j["g"]])
    ok = [True] * len(jobs)

    def worker(t):
        j = jobs[t]
        s = torch.cuda.Stream()
        for _ in range(8):
            for g in j["g"]:
                with torch.cuda.stream(s):
                    g.fill_(float("nan"))
            _bwd_call(j, s)
            s.synchronize()
            same = [torch.equal(g, r) for g, r in zip(j["g"], refs[t])]
            if j["d"] == 64:
                same[0] = _dq_close(j["g"][0].float().cpu().numpy(),
                                    refs[t][0].float().cpu().numpy())
            if not all(same):
                ok[t] = False

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(len(jobs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert abi.fa_last_device_error() == abi.FA_OK
    assert all(ok)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_in_cuda_graph(d):
    """A captured fa_bwd (at d = 128 the fork to the library's dQ stream and the join back
    are part of the capture; at d = 64 the zeroing of the dQ accumulator) replays to the
    same gradients as the eager call (dQ at d = 64 within the rounding of its sums)."""
    import torch
    j = _bwd_job(2, 2, 900, d, True, 2400 + d)
    _bwd_call(j, torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = [g.clone() for g in j["g"]]
    for g in j["g"]:
        g.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=s):
        _bwd_call(j, s)
    for _ in range(3):
        for g in j["g"]:
            g.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(j["g"][1], ref[1]) and torch.equal(j["g"][2], ref[2])
        if d == 128:
            assert torch.equal(j["g"][0], ref[0])
        else:
            assert _dq_close(j["g"][0].float().cpu().numpy(), ref[0].float().cpu().numpy())
    assert abi.fa_last_device_error() == abi.FA_OK
