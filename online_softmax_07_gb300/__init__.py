"""GB300 (sm_103a) online-softmax attention forward and backward, and row softmax state.

The compute lives in ``lib/libosfa.so`` (hand-written CUDA, C ABI in include/fa.h);
this package only binds it.  ``abi`` exposes the C calls by their C names; the two
helpers below allocate outputs with torch and call them.  CPU tensors are copied
to the GPU and the results copied back (the end-to-end path); the computation itself
always runs in the library's kernels.
"""

from __future__ import annotations

import math

from . import abi
from .abi import (FAError, fa_fwd, fa_fwd_dt, fa_bwd, online_softmax_rows,
                  online_softmax_forward, fa_last_device_error)

__all__ = ["attention_forward", "attention_backward", "row_state", "softmax", "abi", "FAError",
           "fa_fwd", "fa_fwd_dt", "fa_bwd", "online_softmax_rows", "online_softmax_forward",
           "fa_last_device_error"]


def _one_device(ts, what):
    """Raises unless every tensor in ts lives on the same device."""
    if any(t.device != ts[0].device for t in ts):
        raise ValueError(f"{what} must all be on one device")


def _check_host_out(t, shape, dtype, name):
    """A caller-supplied host result buffer must match exactly: the copies out write
    shape's bytes into it."""
    if (t.is_cuda or tuple(t.shape) != tuple(shape) or t.dtype != dtype
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous host tensor of shape {tuple(shape)} "
                         f"and dtype {dtype}")


def attention_forward(q, k, v, scale=None, causal=False, stream=None, with_lse=True,
                      out=None, lse_out=None, splits=None):
    """O = softmax(scale * Q K^T) V and LSE for [B, H, N, d] tensors (bf16, fp16 or fp32).

    Returns (O, LSE) with O of q's dtype and LSE fp32 [B, H, N] (None without
    ``with_lse``), on q's device.  For CPU inputs the copies to and from the current
    CUDA device are part of the call: pinned inputs are copied asynchronously (others
    are pinned first), and the results land in ``out`` / ``lse_out`` when given
    (pinned host tensors of the right shape), else in new pinned tensors.  Everything
    is ordered on ``stream`` (a torch.cuda.Stream; default: torch's current stream).

    ``splits``: split-KV count for bf16 / fp16 with d in {64, 128} (fa_fwd_splitkv, its
    workspace allocated here): None takes the library's default for the shape
    (fa_fwd_splitkv_default_splits; 1 when a split does not pay), 1 never splits.
    """
    import torch

    if stream is not None:
        with torch.cuda.stream(stream):
            return attention_forward(q, k, v, scale, causal, None, with_lse, out, lse_out,
                                     splits)
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must be [B, H, N, d] of one shape")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float16,
                                                               torch.float32):
        raise ValueError("q, k, v must all be bf16, all fp16 or all fp32")
    _one_device((q, k, v), "q, k, v")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dtype = {torch.bfloat16: abi.FA_BF16, torch.float16: abi.FA_F16,
             torch.float32: abi.FA_F32}[q.dtype]
    if splits is not None and int(splits) < 1:
        raise ValueError("splits must be None or >= 1")
    # One split count for the whole problem (the host path's chunks use it too, so that
    # both paths compute the same arithmetic).
    s = 1
    if dtype in (abi.FA_BF16, abi.FA_F16) and d in (64, 128) and B * H * N > 0:
        s = int(splits) if splits is not None else \
            abi.fa_fwd_splitkv_default_splits(B, H, N, int(bool(causal)))
    if q.is_cuda:
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if with_lse else None
        with torch.cuda.device(q.device):
            _forward_on_device(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, s)
        return o, lse
    if out is not None:
        _check_host_out(out, (B, H, N, d), q.dtype, "out")
    if with_lse and lse_out is not None:
        _check_host_out(lse_out, (B, H, N), torch.float32, "lse_out")
    return _attention_forward_host(q, k, v, scale, causal, with_lse, out, lse_out, dtype, s)


def _forward_on_device(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, s):
    """fa_fwd_dt, or with s > 1 split-KV fa_fwd_splitkv with a torch-allocated workspace."""
    import torch

    if s <= 1:
        fa_fwd_dt(q, k, v, o, lse, B, H, N, d, scale, int(bool(causal)), dtype)
        return
    nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, s)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    abi.fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, int(bool(causal)), s, ws, nbytes,
                       dtype)


_COPY_STREAMS = {}


def _copy_streams(dev):
    """The copy-in and copy-out streams of a device, created once."""
    import torch

    if dev.index not in _COPY_STREAMS:
        _COPY_STREAMS[dev.index] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    return _COPY_STREAMS[dev.index]


# Groups of (batch, head) slabs of the host path: the copies of one group overlap the
# kernels of its neighbours, so more groups shorten the exposed first copy in and last
# copy out, until a group's kernel is held up by its longest query block and the fixed
# cost of each copy adds up.  Measured on B2 H16 N8192 d128 causal (attention_forward,
# median wall time per call, two boxes): 4 groups 1.300 / 1.306 ms, 5 (7, 7, 7, 7 and 4
# heads) 1.265 / 1.271, 6 1.281 / 1.285, 8 1.315 / 1.319; earlier 2 groups 1.405, 16 1.689.
_HOST_CHUNKS = 5


def _attention_forward_host(q, k, v, scale, causal, with_lse, out, lse_out, dtype, s):
    """Host tensors in, host tensors out, with the copies overlapped with the kernels:
    the (batch, head) slabs are split into chunks; chunk c is copied in on one stream,
    computed on the caller's stream and copied out on a third, so the copy of chunk c+1
    runs while chunk c computes and the copy out of chunk c overlaps both.  Without
    split-KV the library does this itself (fa_fwd_host); with it, the chunks are
    enqueued from here."""
    import torch

    B, H, N, d = q.shape
    BH = B * H
    dev = torch.device("cuda", torch.cuda.current_device())

    def pinned(t):
        t = t.contiguous()
        return t if t.is_pinned() else t.pin_memory()

    o_h = out if out is not None else torch.empty((B, H, N, d), dtype=q.dtype, pin_memory=True)
    lse_h = None
    if with_lse:
        lse_h = lse_out if lse_out is not None else torch.empty((B, H, N), dtype=torch.float32,
                                                                pin_memory=True)
    if s <= 1:
        qp, kp, vp = (pinned(t) for t in (q, k, v))
        nbytes = abi.fa_fwd_host_workspace_bytes(B, H, N, d, dtype, _HOST_CHUNKS)
        ws = torch.empty(max(1, nbytes), dtype=torch.uint8, device=dev)
        abi.fa_fwd_host(qp, kp, vp, o_h, lse_h, B, H, N, d, scale, int(bool(causal)), dtype,
                        _HOST_CHUNKS, ws, nbytes)
        # The caller's stream waits for the last copy out: after this, the results are in
        # o_h / lse_h and the workspace is no longer in use.
        torch.cuda.current_stream().synchronize()
        return o_h, lse_h
    qh, kh, vh = (pinned(t).view(BH, N, d) for t in (q, k, v))
    o_hv = o_h.view(BH, N, d)
    lse_hv = lse_h.view(BH, N) if lse_h is not None else None
    qd, kd, vd = (torch.empty((BH, N, d), dtype=q.dtype, device=dev) for _ in range(3))
    od = torch.empty((BH, N, d), dtype=q.dtype, device=dev)
    lsed = torch.empty((BH, N), dtype=torch.float32, device=dev) if with_lse else None
    compute = torch.cuda.current_stream()
    s_in, s_out = _copy_streams(dev)
    s_in.wait_stream(compute)      # device buffers are ordered after earlier work
    n_chunks = max(1, min(BH, _HOST_CHUNKS))
    bounds = [BH * c // n_chunks for c in range(n_chunks + 1)]
    for c in range(n_chunks):
        h0, h1 = bounds[c], bounds[c + 1]
        if h1 == h0:
            continue
        with torch.cuda.stream(s_in):
            for dst, src in ((qd, qh), (kd, kh), (vd, vh)):
                dst[h0:h1].copy_(src[h0:h1], non_blocking=True)
        compute.wait_stream(s_in)
        _forward_on_device(qd[h0:h1], kd[h0:h1], vd[h0:h1], od[h0:h1],
                           lsed[h0:h1] if lsed is not None else None, 1, h1 - h0, N, d,
                           scale, causal, dtype, s)
        s_out.wait_stream(compute)
        with torch.cuda.stream(s_out):
            o_hv[h0:h1].copy_(od[h0:h1], non_blocking=True)
            if lsed is not None:
                lse_hv[h0:h1].copy_(lsed[h0:h1], non_blocking=True)
    s_out.synchronize()
    compute.synchronize()
    return o_h, lse_h


def attention_backward(q, k, v, o, lse, dout, scale=None, causal=False, stream=None):
    """(dQ, dK, dV) of attention_forward for the upstream gradient ``dout``.

    q, k, v, o, dout: CUDA [B, H, N, d] tensors, all bf16 or all fp16, d in {64, 128};
    o and lse (fp32 [B, H, N]) as attention_forward returned them for the same scale and
    causal flag.  The outputs and the library's workspace are allocated here with torch;
    the computation runs in the library's kernels (fa_bwd).
    """
    import torch

    if stream is not None:
        with torch.cuda.stream(stream):
            return attention_backward(q, k, v, o, lse, dout, scale, causal, None)
    ts = (q, k, v, o, dout)
    if q.dim() != 4 or any(t.shape != q.shape for t in ts):
        raise ValueError("q, k, v, o, dout must be [B, H, N, d] of one shape")
    if any(t.dtype != q.dtype for t in ts) or q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v, o, dout must all be bf16 or all fp16")
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be fp32 [B, H, N]")
    if not all(t.is_cuda for t in ts) or not lse.is_cuda:
        raise ValueError("attention_backward takes CUDA tensors")
    _one_device(ts + (lse,), "q, k, v, o, lse, dout")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    q, k, v, o, dout = (t.contiguous() for t in ts)
    lse = lse.contiguous()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dtype = abi.FA_BF16 if q.dtype == torch.bfloat16 else abi.FA_F16
    ws_bytes = abi.fa_bwd_workspace_bytes_dt(B, H, N, d, dtype)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, int(bool(causal)), ws,
               ws_bytes, dtype)
    return dq, dk, dv


def row_state(x, stream=None):
    """Per-row (m, l) of an fp32 [rows, len] tensor: m = max, l = sum exp(x - m)."""
    import torch

    if stream is not None:
        with torch.cuda.stream(stream):
            return row_state(x, None)
    if x.dim() != 2 or x.dtype != torch.float32:
        raise ValueError("x must be an fp32 [rows, len] tensor")
    host = not x.is_cuda
    if host:
        x = x.contiguous()
        if not x.is_pinned():
            x = x.pin_memory()
        x = x.to(torch.device("cuda", torch.cuda.current_device()), non_blocking=True)
    else:
        x = x.contiguous()
    rows, length = x.shape
    m = torch.empty(rows, dtype=torch.float32, device=x.device)
    l = torch.empty(rows, dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        online_softmax_rows(x, m, l, rows, length)
    if host:
        return m.cpu(), l.cpu()
    return m, l


def softmax(x, stream=None):
    """Row softmax of an fp32 [rows, len] CUDA tensor; returns (y, m, l)."""
    import torch

    if stream is not None:
        with torch.cuda.stream(stream):
            return softmax(x, None)
    if x.dim() != 2 or x.dtype != torch.float32 or not x.is_cuda:
        raise ValueError("x must be an fp32 [rows, len] CUDA tensor")
    x = x.contiguous()
    rows, length = x.shape
    y = torch.empty_like(x)
    m = torch.empty(rows, dtype=torch.float32, device=x.device)
    l = torch.empty(rows, dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        online_softmax_forward(x, y, m, l, rows, length)
    return y, m, l
