"""Parity of the split-KV forward (partials + combine) against the oracle."""

import math

import numpy as np
import pytest

import oracle
from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

from gpu_helpers import check_attention, sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    abi.load()


def run_splitkv(q, k, v, scale, causal, splits, dtype="bf16"):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    code = abi.FA_BF16 if dtype == "bf16" else abi.FA_F16
    B, H, N, d = q.shape
    dq, dk, dv = (to_device(t, tdt) for t in (q, k, v))
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits)
    ws = torch.full((max(1, nbytes // 4),), float("nan"), device="cuda")   # garbage is fine
    abi.fa_fwd_splitkv(dq, dk, dv, o, lse, B, H, N, d, scale, int(causal), splits, ws, nbytes,
                       code)
    assert abi.fa_last_device_error() == abi.FA_OK
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,splits", [(2000, 2), (2000, 3), (777, 7), (300, 8), (129, 2)])
def test_splitkv_all_rows(N, splits, d, causal):
    """Every output element; (300, 8) and (129, 2) leave some splits without any K/V
    tile (empty partials)."""
    q, k, v = synth.attention_inputs(1, 2, N, d, seed=90000 + N + splits + d + int(causal),
                                     q_std=2.0)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_splitkv(q, k, v, scale, causal, splits)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
    check_attention(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_more_blocks_than_sms(d, causal):
    """64 heads x 2 query blocks x 3 splits = 384 blocks, more than the SMs; some
    partials are empty (causal early blocks)."""
    q, k, v = synth.attention_inputs(1, 64, 500, d, seed=90500 + d + int(causal), q_std=2.0)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_splitkv(q, k, v, scale, causal, 3)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
    check_attention(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def test_splitkv_f16():
    q, k, v = synth.attention_inputs(1, 1, 1500, 128, seed=91000, dtype="f16")
    o, lse = run_splitkv(q, k, v, 1 / math.sqrt(128), True, 4, dtype="f16")
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 1 / math.sqrt(128), True)
    check_attention(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, dtype="f16")


def test_splitkv_long_sequence_default_splits():
    """B=1 H=1 N=32768 d=128 causal, Q std 4: 128 query blocks, fewer than the SMs, and
    the last one is 256 K/V tiles long; the default splits it."""
    import torch
    B, H, N, d = 1, 1, 32768, 128
    q, k, v = synth.attention_inputs(B, H, N, d, seed=92000, q_std=4.0)
    splits = abi.fa_fwd_splitkv_default_splits(B, H, N, True)
    assert splits >= 2
    o, lse = run_splitkv(q, k, v, 1 / math.sqrt(d), True, splits)
    for h in range(H):
        rows = sample_rows(N, 128, seed=92100 + h)
        o_ref, lse_ref = oracle.attention_forward(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1],
                                                  1 / math.sqrt(d), True, rows=rows)
        idx = torch.from_numpy(rows).cuda()
        check_attention(o[0, h].index_select(0, idx).float().cpu().numpy()[None, None],
                        lse[0, h].index_select(0, idx).cpu().numpy()[None, None], o_ref, lse_ref)
