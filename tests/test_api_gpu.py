"""The public Python API (online_softmax_07_gb300.attention_forward / attention_backward /
row_state / softmax): host tensors in and out, with the copies pipelined against the
kernels in chunks of heads, must give exactly what the device path gives (the kernels
compute every head independently, so chunking changes no arithmetic)."""

import numpy as np
import pytest
import torch

import online_softmax_07_gb300 as osf
from online_softmax_07_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,causal,pin", [
    (1, 3, 300, 128, True, True),     # 3 chunks of one head
    (2, 5, 257, 64, False, False),    # 10 heads in 5 chunks of 2, inputs not pinned
    (1, 1, 129, 128, True, True),     # a single chunk
    (4, 16, 1024, 128, True, True),   # 64 heads: four chunks of 13 and a last one of 12
])
def test_host_path_equals_device_path(B, H, N, d, causal, pin):
    q, k, v = (torch.from_numpy(t).to(torch.bfloat16)
               for t in synth.attention_inputs(B, H, N, d, seed=991 + N))
    if pin:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_h, lse_h = osf.attention_forward(q, k, v, causal=causal)
    assert not o_h.is_cuda and o_h.is_pinned()
    o_d, lse_d = osf.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(lse_h, lse_d.cpu())


def test_host_path_into_given_buffers_and_without_lse():
    B, H, N, d = 2, 4, 200, 64
    q, k, v = (torch.from_numpy(t).to(torch.bfloat16).pin_memory()
               for t in synth.attention_inputs(B, H, N, d, seed=995))
    out = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16, pin_memory=True)
    lse_out = torch.full((B, H, N), float("nan"), pin_memory=True)
    o1, l1 = osf.attention_forward(q, k, v, scale=0.2, out=out, lse_out=lse_out)
    assert o1.data_ptr() == out.data_ptr() and l1.data_ptr() == lse_out.data_ptr()
    o2, l2 = osf.attention_forward(q, k, v, scale=0.2, with_lse=False)
    assert l2 is None
    assert torch.equal(o1, o2)
    o_d, _ = osf.attention_forward(q.cuda(), k.cuda(), v.cuda(), scale=0.2)
    assert torch.equal(o1, o_d.cpu())
    # Device tensors without LSE (the kernels skip the LSE writes): the same O.
    o_d2, l_d2 = osf.attention_forward(q.cuda(), k.cuda(), v.cuda(), scale=0.2, with_lse=False)
    assert l_d2 is None
    assert torch.equal(o1, o_d2.cpu())


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 1, 4096, 128, True),     # 16 query blocks: the default splits
    (1, 2, 2048, 64, False),     # 16 blocks, not causal: the default splits
])
def test_forward_api_splits(B, H, N, d, causal):
    """attention_forward takes the library's default split count for small grids: the
    result is within the gates of the oracle on sampled rows, splits=1 is exactly the
    plain kernel, and the host path gives exactly what the device path gives."""
    import oracle
    from online_softmax_07_gb300 import abi

    from gpu_helpers import check_attention, sample_rows

    assert abi.fa_fwd_splitkv_default_splits(B, H, N, causal) > 1
    qn, kn, vn = synth.attention_inputs(B, H, N, d, seed=998 + N, q_std=2.0)
    q, k, v = (torch.from_numpy(t).to("cuda", torch.bfloat16) for t in (qn, kn, vn))
    o, lse = osf.attention_forward(q, k, v, causal=causal)
    scale = 1.0 / np.sqrt(d)
    for h in range(H):
        rows = sample_rows(N, 96, seed=999 + h)
        o_ref, lse_ref = oracle.attention_forward(qn[:, h:h + 1], kn[:, h:h + 1], vn[:, h:h + 1],
                                                  scale, causal, rows=rows)
        idx = torch.from_numpy(rows).cuda()
        check_attention(o[0, h].index_select(0, idx).float().cpu().numpy()[None, None],
                        lse[0, h].index_select(0, idx).cpu().numpy()[None, None], o_ref, lse_ref)
    o1, lse1 = osf.attention_forward(q, k, v, causal=causal, splits=1)
    o_plain = torch.empty_like(q)
    lse_plain = torch.empty_like(lse)
    abi.fa_fwd(q, k, v, o_plain, lse_plain, B, H, N, d, scale, int(causal))
    torch.cuda.synchronize()
    assert torch.equal(o1, o_plain) and torch.equal(lse1, lse_plain)
    o_h, lse_h = osf.attention_forward(q.cpu(), k.cpu(), v.cpu(), causal=causal)
    assert torch.equal(o_h, o.cpu()) and torch.equal(lse_h, lse.cpu())


@pytest.mark.parametrize("dtype,d,causal,chunks", [
    ("bf16", 128, True, 1), ("bf16", 64, False, 3), ("f16", 128, True, 7),
    ("bf16", 128, False, 100),   # more chunks than heads
    ("f32", 40, True, 4),        # the fp32 kernel, d not a multiple of 16
])
@pytest.mark.parametrize("with_lse,pin", [(True, True), (False, False)])
def test_fwd_host_equals_device(dtype, d, causal, chunks, with_lse, pin):
    """fa_fwd_host (host tensors, copies and kernels overlapped in groups of heads) gives
    exactly what fa_fwd_dt gives on device copies of the same tensors; from pageable
    memory as well (the copies are then synchronous)."""
    from online_softmax_07_gb300 import abi

    B, H, N = 2, 5, 333
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
    code = {"bf16": abi.FA_BF16, "f16": abi.FA_F16, "f32": abi.FA_F32}[dtype]
    q, k, v = (torch.from_numpy(t).to(tdt)
               for t in synth.attention_inputs(B, H, N, d, seed=1200 + d + chunks, dtype="f32"))
    if pin:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    scale = 1.0 / np.sqrt(d)
    o_h = torch.full((B, H, N, d), float("nan"), dtype=tdt, pin_memory=pin)
    lse_h = torch.full((B, H, N), float("nan"), pin_memory=pin) if with_lse else None
    nbytes = abi.fa_fwd_host_workspace_bytes(B, H, N, d, code, chunks)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    abi.fa_fwd_host(q, k, v, o_h, lse_h, B, H, N, d, scale, int(causal), code, chunks, ws, nbytes)
    torch.cuda.current_stream().synchronize()
    assert abi.fa_last_device_error() == abi.FA_OK
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_d = torch.empty_like(qd)
    lse_d = torch.empty((B, H, N), device="cuda")
    abi.fa_fwd_dt(qd, kd, vd, o_d, lse_d, B, H, N, d, scale, int(causal), code)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    if with_lse:
        assert torch.equal(lse_h, lse_d.cpu())


def test_fwd_host_concurrent_threads():
    """Four host threads, each on its own stream with its own inputs, workspace and group
    count, call fa_fwd_host repeatedly at the same time: the library's copy streams and
    slot events are shared, and every result must still equal the device path's."""
    import threading

    from online_softmax_07_gb300 import abi

    B, H, N, d = 1, 6, 400, 64
    scale = 1.0 / np.sqrt(d)
    jobs = []
    for t in range(4):
        q, k, v = (torch.from_numpy(x).to(torch.bfloat16).pin_memory()
                   for x in synth.attention_inputs(B, H, N, d, seed=1300 + t))
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o_ref = torch.empty_like(qd)
        lse_ref = torch.empty((B, H, N), device="cuda")
        abi.fa_fwd_dt(qd, kd, vd, o_ref, lse_ref, B, H, N, d, scale, t % 2, abi.FA_BF16)
        chunks = 1 + t
        nbytes = abi.fa_fwd_host_workspace_bytes(B, H, N, d, abi.FA_BF16, chunks)
        jobs.append(dict(q=q, k=k, v=v, causal=t % 2, chunks=chunks, nbytes=nbytes,
                         ws=torch.empty(nbytes, dtype=torch.uint8, device="cuda"),
                         stream=torch.cuda.Stream(), o_ref=o_ref, lse_ref=lse_ref,
                         ok=True))
    torch.cuda.synchronize()

    def worker(j):
        for _ in range(10):
            o = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16, pin_memory=True)
            lse = torch.full((B, H, N), float("nan"), pin_memory=True)
            abi.fa_fwd_host(j["q"], j["k"], j["v"], o, lse, B, H, N, d, scale, j["causal"],
                            abi.FA_BF16, j["chunks"], j["ws"], j["nbytes"], j["stream"])
            j["stream"].synchronize()
            if not (torch.equal(o, j["o_ref"].cpu()) and torch.equal(lse, j["lse_ref"].cpu())):
                j["ok"] = False

    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert abi.fa_last_device_error() == abi.FA_OK
    assert all(j["ok"] for j in jobs)


def test_backward_api_matches_abi():
    B, H, N, d = 1, 2, 300, 128
    q, k, v = (torch.from_numpy(t).to("cuda", torch.bfloat16)
               for t in synth.attention_inputs(B, H, N, d, seed=996))
    do = torch.from_numpy(synth.attention_inputs(B, H, N, d, seed=997)[0]).to("cuda", torch.bfloat16)
    o, lse = osf.attention_forward(q, k, v, causal=True)
    g1 = osf.attention_backward(q, k, v, o, lse, do, causal=True)
    g2 = osf.attention_backward(q, k, v, o, lse, do, causal=True)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
        assert torch.isfinite(a.float()).all()


def test_row_state_and_softmax_host_and_device():
    x = torch.from_numpy(synth.row_inputs(37, 3001, seed=998))
    m_h, l_h = osf.row_state(x)
    m_d, l_d = osf.row_state(x.cuda())
    assert torch.equal(m_h, m_d.cpu()) and torch.equal(l_h, l_d.cpu())
    y, m, l = osf.softmax(x.cuda())
    assert torch.equal(m.cpu(), m_h)
    rows_sum = y.double().sum(dim=1).cpu().numpy()
    assert np.abs(rows_sum - 1).max() < 1e-5


def test_forward_paths_in_cuda_graph():
    """The forward (plain and split-KV with its combine) and the row kernels captured in
    one CUDA graph replay to the eager results, bitwise: every launch of the library is
    stream-ordered and capturable (the first calls, which look up the library's device
    addresses, are made eagerly before the capture)."""
    from online_softmax_07_gb300 import abi

    B, H, N, d = 1, 2, 3000, 128
    q, k, v = (torch.from_numpy(t).to(torch.bfloat16).cuda()
               for t in synth.attention_inputs(B, H, N, d, seed=2500))
    x = torch.from_numpy(synth.row_inputs(64, 5000, 2501, 3.0)).cuda()
    scale = 1.0 / np.sqrt(d)
    splits = 3
    nb = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    outs = dict(o=torch.empty_like(q), lse=torch.empty((B, H, N), device="cuda"),
                o_s=torch.empty_like(q), lse_s=torch.empty((B, H, N), device="cuda"),
                m=torch.empty(64, device="cuda"), l=torch.empty(64, device="cuda"))

    def calls(s):
        abi.fa_fwd_dt(q, k, v, outs["o"], outs["lse"], B, H, N, d, scale, 1, abi.FA_BF16, s)
        abi.fa_fwd_splitkv(q, k, v, outs["o_s"], outs["lse_s"], B, H, N, d, scale, 1, splits,
                           ws, nb, abi.FA_BF16, s)
        abi.online_softmax_rows(x, outs["m"], outs["l"], 64, 5000, s)

    calls(torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = {key: t.clone() for key, t in outs.items()}
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=s):
        calls(s)
    for _ in range(3):
        for t in outs.values():
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for key, t in outs.items():
            assert torch.equal(t, ref[key]), key
    assert abi.fa_last_device_error() == abi.FA_OK
