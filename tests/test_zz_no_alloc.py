"""fa_fwd_splitkv_static: the split-KV forward for callers that cannot allocate device
memory (memory pools that own the device, plugin interfaces without an allocator, paths
where cudaMalloc would synchronise).  Its partials live in the library's static device
scratch; the results must equal fa_fwd_splitkv's with a caller workspace bit for bit (the
same kernels and split count), and meet the oracle's gates.

This file is collected last so that a run stopping at the first failure has run every
other test; it also passes on its own in a fresh process."""

import math

import pytest

from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

from gpu_helpers import check_attention, sample_rows, to_device

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
    # first left in the shared scratch.  The same kernels run with the same split count,
    # so O and LSE must equal the caller-workspace results bit for bit; the first call is
    # also held to the oracle's gates on sampled rows of each head.
    import torch

    import oracle
    for i, (B, H, N, d, causal, splits, seed) in enumerate([(1, 2, 8192, 128, 1, 4, 95000),
                                                           (2, 1, 3000, 64, 0, 3, 95001)]):
        qn, kn, vn = synth.attention_inputs(B, H, N, d, seed=seed, q_std=2.0)
        q, k, v = (to_device(t, torch.bfloat16) for t in (qn, kn, vn))
        o_ref, lse_ref = _with_workspace(q, k, v, causal, splits)
        o, lse = _static(q, k, v, causal, splits)
        assert abi.fa_last_device_error() == abi.FA_OK
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), "O differs"
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), "LSE differs"
        if i == 0:
            rows = sample_rows(N, 96, seed=seed + 1)
            idx = torch.from_numpy(rows).cuda()
            for h in range(H):
                exp_o, exp_lse = oracle.attention_forward(qn[:, h:h + 1], kn[:, h:h + 1],
                                                          vn[:, h:h + 1], 1 / math.sqrt(d),
                                                          bool(causal), rows=rows)
                got_o = o[:, h].index_select(1, idx).float().cpu().numpy()[:, None]
                got_lse = lse[:, h].index_select(1, idx).cpu().numpy()[:, None]
                check_attention(got_o, got_lse, exp_o, exp_lse)


def test_static_scratch_one_split_is_the_plain_forward():
    import torch
    B, H, N, d = 1, 3, 1000, 64
    q, k, v = _inputs(B, H, N, d, 95002)
    o_plain = torch.empty_like(q)
    lse_plain = torch.empty((B, H, N), device="cuda")
    abi.fa_fwd_dt(q, k, v, o_plain, lse_plain, B, H, N, d, 1 / math.sqrt(d), 1, abi.FA_BF16)
    o, lse = _static(q, k, v, 1, 1)
    assert abi.fa_last_device_error() == abi.FA_OK
    assert torch.equal(o.view(torch.int16), o_plain.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_plain.view(torch.int32))


def test_static_scratch_empty_and_invalid_calls_touch_nothing():
    """An empty problem returns OK and writes nothing; invalid arguments are reported
    (without a workspace size to check, the call is decided by fa_fwd_splitkv)."""
    import torch
    out = torch.full((4, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    lib = abi.load()
    p = out.data_ptr()
    assert lib.fa_fwd_splitkv_static(p, p, p, p, None, 0, 4, 64, 64, 0.1, 1, 2, abi.FA_BF16,
                                     None) == abi.FA_OK
    assert lib.fa_fwd_splitkv_static(p, p, p, p, None, 1, 1, 0, 64, 0.1, 1, 2, abi.FA_BF16,
                                     None) == abi.FA_OK
    assert lib.fa_fwd_splitkv_static(p, p, p, p, None, 1, 1, 64, 96, 0.1, 1, 2, abi.FA_BF16,
                                     None) == abi.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_splitkv_static(p, p, p, p, None, 1, 1, 64, 64, 0.1, 1, 0, abi.FA_BF16,
                                     None) == abi.FA_ERR_INVALID
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def test_static_scratch_rejects_problems_beyond_its_size():
    import torch
    B, H, N, d, splits = 1, 8, 32768, 128, 8        # partials need about 1.1 GB
    assert abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits) > (64 << 20)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = abi.load().fa_fwd_splitkv_static(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                          dummy.data_ptr(), None, B, H, N, d, 0.1, 1, splits,
                                          abi.FA_BF16, None)
    assert st == abi.FA_ERR_TOO_LARGE
