"""Tensors of more than 2^31 elements: B=1 N=4096 bf16, H=4100 at d=128 and H=8196 at
d=64, 4.3 GB per tensor.  The last four heads start at or beyond element 2^31, so every
index into Q, K, V, O, LSE, dO, the gradients and (d = 64) the backward's dQ accumulator
and statistics terms must be 64-bit.  Sampled rows of heads on both sides of that
boundary, forward and backward, against the fp64 oracle."""

import numpy as np
import pytest

import oracle
from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

from gpu_helpers import check_attention, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    abi.load()


@pytest.mark.parametrize("d", [128, 64])
def test_forward_and_backward_beyond_2_31_elements(d):
    import torch

    B, N = 1, 4096
    hb = 2 ** 31 // (N * d)   # the first head at element 2^31
    H = hb + 4
    assert B * H * N * d > 2 ** 31 and hb * N * d == 2 ** 31
    scale = 1.0 / np.sqrt(d)
    q, k, v, do = (synth.device_normal((B, H, N, d), seed=5_000_000 + i, dtype=torch.bfloat16)
                   for i in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda")
    abi.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, 1)
    assert abi.fa_last_device_error() == abi.FA_OK
    nbytes = abi.fa_bwd_workspace_bytes_dt(B, H, N, d, abi.FA_BF16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    abi.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, 1, ws, nbytes, abi.FA_BF16)
    assert abi.fa_last_device_error() == abi.FA_OK
    torch.cuda.synchronize()

    def head(t, h):
        return t[0, h].float().cpu().numpy()[None, None]

    for h in (0, hb - 1, hb, H - 1):
        rows = sample_rows(N, 24, seed=h)
        qh, kh, vh, doh = (head(t, h) for t in (q, k, v, do))
        o_ref, lse_ref = oracle.attention_forward(qh, kh, vh, scale, True, rows=rows)
        check_attention(head(o, h)[:, :, rows], lse[0, h].cpu().numpy()[None, None, rows],
                        o_ref, lse_ref)
        refs = oracle.attention_backward_rows(qh, kh, vh, doh, scale, True, (0, 0), rows, rows)
        for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
            got = head(g, h)[0, 0, rows]
            rel = np.linalg.norm(got - r) / np.linalg.norm(r)
            assert rel <= 1e-2, f"{name} head {h}: rel RMS {rel:.3e}"
            assert np.abs(got - r).max() <= 2e-2 * np.abs(r).max(), f"{name} head {h}"


@pytest.mark.parametrize("d,q_std", [(128, 1.0), (64, 4.0)])
def test_forward_sequence_of_131072(d, q_std):
    """One head of N = 131072, causal: the last query block runs over 1024 K/V tiles
    (with Q std 4 the row maximum keeps moving).  Sampled rows, including the last,
    against the oracle; the API's default split count agrees as well."""
    import torch

    import online_softmax_07_gb300 as osf

    B, H, N = 1, 1, 131072
    scale = 1.0 / np.sqrt(d)
    q = synth.device_normal((B, H, N, d), seed=6_000_000 + d, std=q_std, dtype=torch.bfloat16)
    k, v = (synth.device_normal((B, H, N, d), seed=6_000_010 + d + i, dtype=torch.bfloat16)
            for i in range(2))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda")
    abi.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, 1)
    assert abi.fa_last_device_error() == abi.FA_OK
    o2, lse2 = osf.attention_forward(q, k, v, causal=True, splits=4)
    torch.cuda.synchronize()
    rows = sample_rows(N, 32, seed=7 + d)
    qh, kh, vh = (t[0, 0].float().cpu().numpy()[None, None] for t in (q, k, v))
    o_ref, lse_ref = oracle.attention_forward(qh, kh, vh, scale, True, rows=rows)
    for oo, ll in ((o, lse), (o2, lse2)):
        check_attention(oo[0, 0].float().cpu().numpy()[None, None, rows],
                        ll[0, 0].cpu().numpy()[None, None, rows], o_ref, lse_ref)
