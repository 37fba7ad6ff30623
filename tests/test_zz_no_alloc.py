"""fa_fwd_splitkv_static: the split-KV forward for callers that cannot allocate device
memory (memory pools that own the device, plugin interfaces without an allocator, paths
where cudaMalloc would synchronise).  Its partials live in the library's static device
scratch; the results must match fa_fwd_splitkv with a caller workspace.

This file is collected last so that a run stopping at the first failure has run every
other test; it also passes on its own in a fresh process."""

import math

import numpy as np
import pytest

from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

from gpu_helpers import check_attention, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    abi.load()


def _inputs(B, H, N, d, seed):
    import torch
    q, k, v = synth.attention_inputs(B, H, N, d, seed=seed, q_std=2.0)
    return tuple(to_device(t, torch.bfloat16) for t in (q, k, v))


def _with_workspace(q, k, v, causal, splits):
    import torch
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda")
    nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits)
    ws = torch.empty(nbytes // 4, device="cuda")
    abi.fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, 1 / math.sqrt(d), causal, splits, ws, nbytes,
                       abi.FA_BF16)
    return o, lse


def _static(q, k, v, causal, splits):
    import torch
    B, H, N, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    abi.fa_fwd_splitkv_static(q, k, v, o, lse, B, H, N, d, 1 / math.sqrt(d), causal, splits,
                              abi.FA_BF16)
    return o, lse


def test_static_scratch_matches_workspace_two_calls_in_a_row():
    # Two calls with different shapes and split counts: the second runs over what the
    # first left in the shared scratch.
    for (B, H, N, d, causal, splits, seed) in [(1, 2, 8192, 128, 1, 4, 95000),
                                              (2, 1, 3000, 64, 0, 3, 95001)]:
        q, k, v = _inputs(B, H, N, d, seed)
        o_ref, lse_ref = _with_workspace(q, k, v, causal, splits)
        o, lse = _static(q, k, v, causal, splits)
        assert abi.fa_last_device_error() == abi.FA_OK
        check_attention(o.float().cpu().numpy(), lse.cpu().numpy(),
                        o_ref.float().cpu().numpy().astype(np.float64),
                        lse_ref.cpu().numpy().astype(np.float64))


def test_static_scratch_rejects_problems_beyond_its_size():
    import torch
    B, H, N, d, splits = 1, 8, 32768, 128, 8        # partials need about 1.1 GB
    assert abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits) > (64 << 20)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = abi.load().fa_fwd_splitkv_static(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                          dummy.data_ptr(), None, B, H, N, d, 0.1, 1, splits,
                                          abi.FA_BF16, None)
    assert st == abi.FA_ERR_TOO_LARGE
