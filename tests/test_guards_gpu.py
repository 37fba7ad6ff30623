"""Guard words around every buffer the kernels write, and their inputs checked unchanged.

Each output, workspace and host buffer is allocated with 4 KB of a sentinel byte pattern
on both sides; after the call the sentinels must be bit-for-bit intact (a write past
either end of a buffer shows up here even when the values inside are right), and every
input must be unchanged.  The shapes are the edge cases of the tile loop ("Softmax
数值稳定性与 IO-Aware Attention" §9.2: unaligned lengths and tail blocks, mask
boundaries): ragged N around the 128-row tiles and 256-row query blocks, rows of length
1, 3 and 32767 (unaligned row starts), split-KV with empty chunks, in-place and
misaligned softmax outputs, the backward's prep rows, and the host pipeline's slot
copies.
"""

import math

import numpy as np
import pytest

from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

pytestmark = pytest.mark.gpu

GUARD = 4096      # bytes of sentinel on each side
PATTERN = 0xA7    # sentinel byte (not a byte of 0, 1.0, NaN or inf encodings)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    abi.load()


class Guarded:
    """A tensor of `shape` and `dtype` inside a byte buffer with GUARD sentinel bytes on
    each side; `offset` shifts the tensor's start by that many bytes (misaligned views).
    On the device unless `host` (then page-locked host memory)."""

    def __init__(self, shape, dtype, offset=0, host=False, fill=None):
        import torch
        self.shape, self.dtype, self.offset = tuple(shape), dtype, offset
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(self.shape, dtype=np.int64)) * itemsize
        total = GUARD + offset + self.nbytes + GUARD
        if host:
            self.buf = torch.full((total,), PATTERN, dtype=torch.uint8).pin_memory()
        else:
            self.buf = torch.full((total,), PATTERN, dtype=torch.uint8, device="cuda")
        lo = GUARD + offset
        self.t = self.buf[lo:lo + self.nbytes].view(dtype).view(self.shape)
        if fill is not None:
            self.t.copy_(fill.to(dtype).reshape(self.shape))

    def guards_intact(self):
        lo = GUARD + self.offset
        head = self.buf[:lo].cpu()
        tail = self.buf[lo + self.nbytes:].cpu()
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _check(*bufs):
    import torch
    torch.cuda.synchronize()
    assert abi.fa_last_device_error() == abi.FA_OK
    for i, g in enumerate(bufs):
        assert g.guards_intact(), f"guard words of buffer {i} were overwritten"


def _inputs(B, H, N, d, seed, dtype):
    import torch
    q, k, v = synth.attention_inputs(B, H, N, d, seed=seed, q_std=2.0)
    out = []
    for t in (q, k, v):
        src = torch.from_numpy(t)
        out.append(Guarded(t.shape, dtype, fill=src.cuda()))
    return out


def _unchanged(guarded_inputs, copies):
    import torch
    for g, c in zip(guarded_inputs, copies):
        assert torch.equal(g.t.view(torch.uint8), c.view(torch.uint8)), "an input was written"


@pytest.mark.parametrize("N", [1, 127, 129, 255, 257, 8191])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [0, 1])
def test_forward_output_guards(N, d, causal):
    import torch
    B, H = 1, 2
    ins = _inputs(B, H, N, d, 101000 + N + d + causal, torch.bfloat16)
    copies = [g.t.clone() for g in ins]
    o = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    abi.fa_fwd(ins[0].t, ins[1].t, ins[2].t, o.t, lse.t, B, H, N, d, 1 / math.sqrt(d), causal)
    _check(o, lse, *ins)
    _unchanged(ins, copies)
    assert bool(torch.isfinite(o.t.float()).all()) and bool(torch.isfinite(lse.t).all())


@pytest.mark.parametrize("N", [1, 65, 257, 1000, 8191])
@pytest.mark.parametrize("d,block_n", [(64, 64), (64, 256), (128, 64)])
@pytest.mark.parametrize("causal", [0, 1])
def test_block_size_output_guards(N, d, block_n, causal):
    """The 64- and 256-key tile kernels (rings of 16, 6 and 10 slots) keep the guards of
    O and LSE and leave the inputs alone."""
    import torch
    B, H = 1, 2
    ins = _inputs(B, H, N, d, 101500 + N + d + block_n, torch.bfloat16)
    copies = [g.t.clone() for g in ins]
    o = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    abi.fa_fwd_block(ins[0].t, ins[1].t, ins[2].t, o.t, lse.t, B, H, N, d, 1 / math.sqrt(d),
                     causal, abi.FA_BF16, block_n)
    _check(o, lse, *ins)
    _unchanged(ins, copies)
    assert bool(torch.isfinite(o.t.float()).all()) and bool(torch.isfinite(lse.t).all())


@pytest.mark.parametrize("N", [1, 100, 257])
def test_forward_f32_guards(N):
    import torch
    B, H, d = 1, 2, 17
    ins = _inputs(B, H, N, d, 102000 + N, torch.float32)
    copies = [g.t.clone() for g in ins]
    o = Guarded((B, H, N, d), torch.float32)
    lse = Guarded((B, H, N), torch.float32)
    abi.fa_fwd_dt(ins[0].t, ins[1].t, ins[2].t, o.t, lse.t, B, H, N, d, 0.25, 1, abi.FA_F32)
    _check(o, lse, *ins)
    _unchanged(ins, copies)


@pytest.mark.parametrize("N,splits,causal", [(300, 4, 1), (1000, 7, 1), (257, 3, 0),
                                              (8191, 5, 1)])
@pytest.mark.parametrize("d", [64, 128])
def test_splitkv_guards_with_empty_chunks(N, splits, causal, d):
    """More splits than a query block has K/V tiles leaves chunks empty (their partial is
    written as LSE = -inf, O = 0 into rows padded to 256): the workspace, O and LSE keep
    their guards."""
    import torch
    B, H = 1, 2
    ins = _inputs(B, H, N, d, 103000 + N + d, torch.bfloat16)
    copies = [g.t.clone() for g in ins]
    o = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits)
    ws = Guarded((nbytes,), torch.uint8)
    abi.fa_fwd_splitkv(ins[0].t, ins[1].t, ins[2].t, o.t, lse.t, B, H, N, d, 1 / math.sqrt(d),
                       causal, splits, ws.t, nbytes, abi.FA_BF16)
    _check(o, lse, ws, *ins)
    _unchanged(ins, copies)
    # the static-scratch entry writes only O and LSE
    o2 = Guarded((B, H, N, d), torch.bfloat16)
    lse2 = Guarded((B, H, N), torch.float32)
    abi.fa_fwd_splitkv_static(ins[0].t, ins[1].t, ins[2].t, o2.t, lse2.t, B, H, N, d,
                              1 / math.sqrt(d), causal, splits, abi.FA_BF16)
    _check(o2, lse2)
    assert torch.equal(o2.t.view(torch.int16), o.t.view(torch.int16))


@pytest.mark.parametrize("rows,length", [(64, 1), (33, 3), (7, 32767), (3, 65539)])
def test_row_state_guards(rows, length):
    import torch
    x = synth.row_inputs(rows, length, seed=104000 + length)
    xg = Guarded((rows, length), torch.float32, fill=torch.from_numpy(x).cuda())
    xc = xg.t.clone()
    m = Guarded((rows,), torch.float32)
    l = Guarded((rows,), torch.float32)
    abi.online_softmax_rows(xg.t, m.t, l.t, rows, length)
    _check(m, l, xg)
    assert torch.equal(xg.t, xc)


@pytest.mark.parametrize("rows,length", [(64, 1), (33, 3), (7, 32767), (3, 65539)])
@pytest.mark.parametrize("mode", ["separate", "misaligned", "in_place"])
def test_softmax_output_guards(rows, length, mode):
    """y written separately, at a 4-byte (not 16-byte) aligned address, or over x."""
    import torch
    x = synth.row_inputs(rows, length, seed=105000 + length)
    xg = Guarded((rows, length), torch.float32, fill=torch.from_numpy(x).cuda())
    xc = xg.t.clone()
    m = Guarded((rows,), torch.float32)
    l = Guarded((rows,), torch.float32)
    if mode == "in_place":
        y = xg
    else:
        y = Guarded((rows, length), torch.float32, offset=4 if mode == "misaligned" else 0)
    abi.online_softmax_forward(xg.t, y.t.data_ptr(), m.t, l.t, rows, length)
    _check(m, l, y, xg)
    if mode != "in_place":
        assert torch.equal(xg.t, xc)
    assert bool(torch.isfinite(y.t).all())


@pytest.mark.parametrize("N,d,causal", [(129, 64, 1), (300, 128, 0), (257, 128, 1),
                                        (1, 64, 0)])
def test_backward_guards(N, d, causal):
    """dQ, dK, dV and the backward's workspace, sized exactly for this d (rows padded to
    128; the prep kernel writes four query rows per warp; at d = 64 the dQ accumulator
    takes the TMA reduce-adds) keep their guards; Q, K, V, O, LSE and dO are not
    written."""
    import torch
    B, H = 1, 2
    ins = _inputs(B, H, N, d, 106000 + N + d, torch.bfloat16)
    scale = 1 / math.sqrt(d)
    o = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    abi.fa_fwd(ins[0].t, ins[1].t, ins[2].t, o.t, lse.t, B, H, N, d, scale, causal)
    do_host = synth.attention_inputs(B, H, N, d, seed=106500 + N)[0]
    dout = Guarded((B, H, N, d), torch.bfloat16, fill=torch.from_numpy(do_host).cuda())
    fixed = ins + [o, lse, dout]
    copies = [g.t.clone() for g in fixed]
    grads = [Guarded((B, H, N, d), torch.bfloat16) for _ in range(3)]
    nbytes = abi.fa_bwd_workspace_bytes_dt(B, H, N, d, abi.FA_BF16)
    ws = Guarded((nbytes,), torch.uint8)
    abi.fa_bwd(ins[0].t, ins[1].t, ins[2].t, o.t, lse.t, dout.t, grads[0].t, grads[1].t,
               grads[2].t, B, H, N, d, scale, causal, ws.t, nbytes, abi.FA_BF16)
    _check(*grads, ws, *fixed)
    _unchanged(fixed, copies)
    for g in grads:
        assert bool(torch.isfinite(g.t.float()).all())


@pytest.mark.parametrize("chunks", [1, 3, 4])
def test_host_pipeline_guards(chunks):
    """fa_fwd_host copies groups of heads through three rotating slots of the device
    workspace: the host O and LSE buffers and the workspace keep their guards, and the
    host inputs are not written."""
    import torch
    B, H, N, d, causal = 1, 5, 300, 64, 1
    q, k, v = synth.attention_inputs(B, H, N, d, seed=107000 + chunks)
    hq, hk, hv = (Guarded(t.shape, torch.bfloat16, host=True, fill=torch.from_numpy(t))
                  for t in (q, k, v))
    copies = [g.t.clone() for g in (hq, hk, hv)]
    ho = Guarded((B, H, N, d), torch.bfloat16, host=True)
    hl = Guarded((B, H, N), torch.float32, host=True)
    nbytes = abi.fa_fwd_host_workspace_bytes(B, H, N, d, abi.FA_BF16, chunks)
    ws = Guarded((nbytes,), torch.uint8)
    abi.fa_fwd_host(hq.t, hk.t, hv.t, ho.t, hl.t, B, H, N, d, 1 / math.sqrt(d), causal,
                    abi.FA_BF16, chunks, ws.t, nbytes)
    _check(ho, hl, ws, hq, hk, hv)
    for g, c in zip((hq, hk, hv), copies):
        assert torch.equal(g.t.view(torch.int16), c.view(torch.int16))
    # same result as the device forward
    dq, dk, dv = (g.t.cuda() for g in (hq, hk, hv))
    o_dev = torch.empty_like(dq)
    l_dev = torch.empty((B, H, N), device="cuda")
    abi.fa_fwd(dq, dk, dv, o_dev, l_dev, B, H, N, d, 1 / math.sqrt(d), causal)
    torch.cuda.synchronize()
    assert torch.equal(ho.t.view(torch.int16), o_dev.cpu().view(torch.int16))
