"""Helpers for the GPU parity tests: run the C ABI on seeded inputs and compare with
the fp64 oracle element by element."""

from __future__ import annotations

import numpy as np

from online_softmax_07_gb300 import abi

# Tolerances.  bf16 attention: O max abs <= 2e-2, O mean abs <= 2e-3, LSE abs <= 1e-3
# (the stated gates).  Row state: (m, l) within 1e-5 relative.  fp32 attention: 1e-5
# absolute on O and LSE (no gate is stated; fp32 rounding of 64-128 term dot products
# and of the exponentials keeps the error near 1e-6 for these unit-variance inputs).
BF16_O_MAX_ABS = 2e-2
BF16_O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
ROW_REL = 1e-5
F32_O_MAX_ABS = 1e-5
F32_LSE_ABS = 1e-5


def to_device(x, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(device="cuda", dtype=dtype).contiguous()


def run_attention(q, k, v, scale, causal, dtype="bf16", with_lse=True):
    """Calls fa_fwd_dt through the C ABI; returns O (fp32 numpy) and LSE."""
    import torch
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
    B, H, N, d = q.shape
    dq, dk, dv = to_device(q, tdt), to_device(k, tdt), to_device(v, tdt)
    o = torch.full_like(dq, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda") if with_lse else None
    code = {"bf16": abi.FA_BF16, "f16": abi.FA_F16, "f32": abi.FA_F32}[dtype]
    abi.fa_fwd_dt(dq, dk, dv, o, lse, B, H, N, d, scale, int(causal), code)
    assert abi.fa_last_device_error() == abi.FA_OK
    o_h = o.float().cpu().numpy()
    lse_h = lse.cpu().numpy() if with_lse else None
    return o_h, lse_h


def run_rows(x):
    import torch
    rows, length = x.shape
    dx = to_device(x, torch.float32)
    m = torch.full((rows,), float("nan"), device="cuda")
    l = torch.full((rows,), float("nan"), device="cuda")
    abi.online_softmax_rows(dx, m, l, rows, length)
    assert abi.fa_last_device_error() == abi.FA_OK
    return m.cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64)


def check_attention(o, lse, o_ref, lse_ref, dtype="bf16"):
    err = np.abs(o.astype(np.float64) - o_ref)
    assert np.all(np.isfinite(o)), "non-finite output"
    if dtype in ("bf16", "f16"):
        assert err.max() <= BF16_O_MAX_ABS, f"O max abs err {err.max():.3e}"
        assert err.mean() <= BF16_O_MEAN_ABS, f"O mean abs err {err.mean():.3e}"
        lse_tol = LSE_ABS
    else:
        assert err.max() <= F32_O_MAX_ABS, f"O max abs err {err.max():.3e}"
        lse_tol = F32_LSE_ABS
    if lse is not None:
        lerr = np.abs(lse.astype(np.float64) - lse_ref)
        assert np.all(np.isfinite(lse)), "non-finite LSE"
        assert lerr.max() <= lse_tol, f"LSE max abs err {lerr.max():.3e}"
    return float(err.max()), float(err.mean())


def block_edge_rows(N: int) -> list:
    """Rows at the edges of the forward kernel's work: 128-row Q tiles inside 256-row
    query blocks.  The first tile, the tile edge inside the first block (127 / 128), the
    first block edge (255 / 256) and the second (511 / 512), the last block's first row
    and its first tile-1 row, and the last rows (where the most rescales have
    happened)."""
    last_block = ((N - 1) // 256) * 256
    cand = (0, 127, 128, 255, 256, 511, 512, last_block, last_block + 127, last_block + 128,
            N - 129, N - 1)
    return sorted({r for r in cand if 0 <= r < N})


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    """Seeded rows without replacement plus the block-edge rows above."""
    forced = block_edge_rows(N)
    rest = np.setdiff1d(np.arange(N), forced)
    g = np.random.Generator(np.random.PCG64(seed))
    pick = g.choice(rest, size=min(count - len(forced), rest.size), replace=False)
    return np.sort(np.concatenate([np.array(forced, dtype=np.int64), pick.astype(np.int64)]))
