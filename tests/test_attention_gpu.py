"""Parity of the attention forward (C ABI, CUDA kernels) against the fp64 oracle."""

import math

import numpy as np
import pytest

import oracle
from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

from gpu_helpers import check_attention, run_attention, sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    abi.load()


SMALL_N = [1, 2, 100, 127, 128, 129, 255, 256, 257, 300, 511, 640, 1000]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", SMALL_N)
def test_bf16_small_all_rows(N, d, causal):
    """Several tiles and a ragged tail, every output element compared."""
    q, k, v = synth.attention_inputs(1, 2, N, d, seed=70000 + N * 4 + d + int(causal))
    scale = 1.0 / math.sqrt(d)
    o, lse = run_attention(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
    check_attention(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_large_logits_rescales(d, causal):
    """Q with standard deviation 4: large logits that move the row max often."""
    q, k, v = synth.attention_inputs(2, 3, 777, d, seed=71000 + d, q_std=4.0)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_attention(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
    check_attention(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_growing_logits_force_every_rescale(d, dtype):
    """Keys whose scores grow along the sequence: every 128-key tile raises the row max
    by 48 (natural log units), far more than the kernel's lazy-rescale threshold (8 log2
    units = 5.5), so the O rescale runs on every tile."""
    N = 1024
    rnd = synth.round_to_bf16 if dtype == "bf16" else synth.round_to_f16
    q, k, v = synth.attention_inputs(1, 1, N, d, seed=72000 + d, dtype=dtype)
    q[...] = rnd(np.abs(q) * 0 + 1.0)                            # q = (1, ..., 1)
    ramp = (np.arange(N, dtype=np.float32) / 128.0) * 6.0        # +6 per 128 keys
    k = rnd(k * 0.1 + ramp[None, None, :, None] / math.sqrt(d))
    scale = 1.0 / math.sqrt(d) * 8.0
    for causal in (False, True):
        o, lse = run_attention(q, k, v, scale, causal, dtype=dtype)
        o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
        check_attention(o, lse, o_ref, lse_ref, dtype=dtype)


@pytest.mark.parametrize("d", [64, 128])
def test_f16_large_logits_rescales(d):
    """fp16 with Q standard deviation 4 (the lazy-rescale reference moves often) against
    the oracle."""
    q, k, v = synth.attention_inputs(1, 2, 900, d, seed=71500 + d, dtype="f16", q_std=4.0)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse = run_attention(q, k, v, scale, causal, dtype="f16")
        o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
        check_attention(o, lse, o_ref, lse_ref, dtype="f16")


def test_bf16_scale_and_batch_layout():
    """Several batches and heads with distinct contents (catches a wrong head stride)
    and a non-default scale."""
    q, k, v = synth.attention_inputs(3, 5, 200, 64, seed=73000)
    o, lse = run_attention(q, k, v, 0.37, False)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.37, False)
    check_attention(o, lse, o_ref, lse_ref)


def test_bf16_without_lse():
    q, k, v = synth.attention_inputs(1, 2, 300, 128, seed=74000)
    o, _ = run_attention(q, k, v, 1 / math.sqrt(128), True, with_lse=False)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 1 / math.sqrt(128), True)
    check_attention(o, None, o_ref, lse_ref)


def test_bf16_uniform_keys_give_mean_of_values():
    """All keys equal: the softmax is uniform, O_i = mean of the visible values
    (a property that needs no oracle)."""
    N, d = 300, 64
    q, k, v = synth.attention_inputs(1, 1, N, d, seed=75000)
    k[...] = k[:, :, :1, :]
    o, lse = run_attention(q, k, v, 0.125, True)
    csum = np.cumsum(v[0, 0].astype(np.float64), axis=0) / np.arange(1, N + 1)[:, None]
    assert np.abs(o[0, 0] - csum).max() <= 2e-2
    s = 0.125 * (q[0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64))
    assert np.abs(lse[0, 0] - (s + np.log(np.arange(1, N + 1)))).max() <= 1e-3


def test_empty_problem_writes_nothing():
    import torch
    o = torch.full((1, 1, 4, 64), 7.0, device="cuda", dtype=torch.bfloat16)
    abi.fa_fwd(o, o, o, o, None, 0, 1, 4, 64, 0.125, 0)
    abi.fa_fwd(o, o, o, o, None, 1, 1, 0, 64, 0.125, 0)
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())


@pytest.mark.parametrize("d", [1, 17, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_path(d, causal):
    q, k, v = synth.attention_inputs(2, 2, 77, d, seed=76000 + d, dtype="f32")
    scale = 1.0 / math.sqrt(d)
    o, lse = run_attention(q, k, v, scale, causal, dtype="f32")
    o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
    check_attention(o, lse, o_ref, lse_ref, dtype="f32")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", [(2, 160, 300), (1, 48, 1000)])
def test_bf16_more_blocks_than_sms(B, H, N, d, causal):
    """More blocks (256-row query blocks x heads) than SMs, so the launch runs in
    several waves and each SM runs blocks back to back; (1, 48, 1000) mixes block
    lengths (causal) and ragged last blocks.  Q std 2 makes the O rescale run.  Every
    element compared; two launches must agree bit for bit."""
    q, k, v = synth.attention_inputs(B, H, N, d, seed=73000 + H + N + d + int(causal),
                                     q_std=2.0)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_attention(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
    check_attention(o, lse, o_ref, lse_ref)
    o2, lse2 = run_attention(q, k, v, scale, causal)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_f16_more_blocks_than_sms():
    q, k, v = synth.attention_inputs(1, 200, 256, 64, seed=73900, dtype="f16", q_std=2.0)
    o, lse = run_attention(q, k, v, 0.125, False, dtype="f16")
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.125, False)
    check_attention(o, lse, o_ref, lse_ref, dtype="f16")


def test_workload_f32_b1h1n128d64():
    """fp32, B1 H1 N128 d64, scale 1/8, no mask: every element against the oracle;
    also the same inputs rounded to bf16 through the tensor-core kernel."""
    q, k, v = synth.workload_attention_inputs("attn_f32_b1h1n128d64")
    o, lse = run_attention(q, k, v, 0.125, False, dtype="f32")
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.125, False)
    check_attention(o, lse, o_ref, lse_ref, dtype="f32")
    qb, kb, vb = (synth.round_to_bf16(t) for t in (q, k, v))
    o, lse = run_attention(qb, kb, vb, 0.125, False)
    o_ref, lse_ref = oracle.attention_forward(qb, kb, vb, 0.125, False)
    check_attention(o, lse, o_ref, lse_ref)


def _full_size(name, rows_per_head):
    import torch
    w = synth.WORKLOADS[name]
    q, k, v = synth.workload_attention_inputs(name)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = (to_device(t, torch.bfloat16) for t in (q, k, v))
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    abi.fa_fwd(dq, dk, dv, o, lse, B, H, N, d, scale, int(w["causal"]))
    assert abi.fa_last_device_error() == abi.FA_OK
    assert bool(torch.isfinite(lse).all()) and bool(torch.isfinite(o.float()).all())
    worst = 0.0
    for b in range(B):
        for h in range(H):
            rows = sample_rows(N, rows_per_head, seed=w["seed"] + 100 * b + h)
            o_ref, lse_ref = oracle.attention_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                                      v[b:b + 1, h:h + 1], scale, w["causal"],
                                                      rows=rows)
            idx = torch.from_numpy(rows).cuda()
            o_s = o[b, h].index_select(0, idx).float().cpu().numpy()[None, None]
            lse_s = lse[b, h].index_select(0, idx).cpu().numpy()[None, None]
            mx, _ = check_attention(o_s, lse_s, o_ref, lse_ref)
            worst = max(worst, mx)
    return worst


def test_workload_b4h16n4096d64_sampled():
    _full_size("attn_bf16_b4h16n4096d64", 128)


def test_workload_b2h16n8192d128_causal_sampled():
    _full_size("attn_bf16_b2h16n8192d128_causal", 128)


def test_workload_b2h16n8191d128_causal_sampled():
    _full_size("attn_bf16_b2h16n8191d128_causal", 128)


def test_workload_b1h8n32768d128_causal_qstd4_sampled():
    _full_size("attn_bf16_b1h8n32768d128_causal_qstd4", 256)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300, 640])
def test_f16_small_all_rows(N, d, causal):
    """fp16 inputs through the same tensor-core kernel (operand format F16)."""
    q, k, v = synth.attention_inputs(2, 2, N, d, seed=77000 + N + d + int(causal), dtype="f16")
    scale = 1.0 / math.sqrt(d)
    o, lse = run_attention(q, k, v, scale, causal, dtype="f16")
    o_ref, lse_ref = oracle.attention_forward(q, k, v, scale, causal)
    check_attention(o, lse, o_ref, lse_ref, dtype="f16")


def test_f16_large_logits():
    q, k, v = synth.attention_inputs(1, 4, 1000, 128, seed=78000, dtype="f16", q_std=4.0)
    o, lse = run_attention(q, k, v, 1 / math.sqrt(128), True, dtype="f16")
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 1 / math.sqrt(128), True)
    check_attention(o, lse, o_ref, lse_ref, dtype="f16")
