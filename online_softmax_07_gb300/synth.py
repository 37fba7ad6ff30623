"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds none of the method's arithmetic: it only draws numbers
(numpy PCG64, standard normal) and rounds them to the storage type.  Both the
CUDA path and the oracle receive the same arrays from here.

Workloads (sizes, distributions and special rows follow the five stated
configurations; names say what each one is):
"""

from __future__ import annotations

import numpy as np

# name -> description; seeds are 1000 * workload id + tensor index (q 0, k 1, v 2, x 3).
WORKLOADS = {
    "attn_f32_b1h1n128d64": dict(kind="attn", B=1, H=1, N=128, d=64, dtype="f32",
                                 causal=False, q_std=1.0, kv_std=1.0, seed=1000),
    "rows_4096x32768": dict(kind="rows", rows=4096, length=32768, std=3.0, seed=2000),
    "attn_bf16_b4h16n4096d64": dict(kind="attn", B=4, H=16, N=4096, d=64, dtype="bf16",
                                    causal=False, q_std=1.0, kv_std=1.0, seed=3000),
    "attn_bf16_b2h16n8192d128_causal": dict(kind="attn", B=2, H=16, N=8192, d=128,
                                            dtype="bf16", causal=True, q_std=1.0,
                                            kv_std=1.0, seed=4000),
    "attn_bf16_b2h16n8191d128_causal": dict(kind="attn", B=2, H=16, N=8191, d=128,
                                            dtype="bf16", causal=True, q_std=1.0,
                                            kv_std=1.0, seed=4100),
    "attn_bf16_b1h8n32768d128_causal_qstd4": dict(kind="attn", B=1, H=8, N=32768, d=128,
                                                  dtype="bf16", causal=True, q_std=4.0,
                                                  kv_std=1.0, seed=5000),
}


def _normal(seed: int, shape, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32 holding bf16 values."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).to(torch.float32).numpy()


def round_to_f16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest fp16 (ties to even), returned as fp32 holding fp16 values."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def attention_inputs(B, H, N, d, seed, dtype="bf16", q_std=1.0, kv_std=1.0):
    """q, k, v as fp32 numpy [B, H, N, d], i.i.d. normal; bf16- (or fp16-) representable
    when dtype == 'bf16' ('f16'): the values the GPU path receives, exactly."""
    q = _normal(seed + 0, (B, H, N, d), q_std)
    k = _normal(seed + 1, (B, H, N, d), kv_std)
    v = _normal(seed + 2, (B, H, N, d), kv_std)
    if dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    elif dtype == "f16":
        q, k, v = round_to_f16(q), round_to_f16(k), round_to_f16(v)
    elif dtype != "f32":
        raise ValueError(dtype)
    return q, k, v


def device_normal(shape, seed: int, std: float = 1.0, dtype=None, device="cuda"):
    """i.i.d. N(0, std^2) drawn on a CUDA device by torch's seeded generator, for inputs
    too large to draw on the host (tensors of several GB); cast to ``dtype`` (a torch
    dtype; default fp32).  Tests copy the rows they check back to the host, so the
    oracle sees exactly the values the kernels saw."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x if dtype is None else x.to(dtype)


def workload_attention_inputs(name: str):
    w = WORKLOADS[name]
    return attention_inputs(w["B"], w["H"], w["N"], w["d"], w["seed"], w["dtype"],
                            w["q_std"], w["kv_std"])


# Special rows of the row-state workload (first and last rows of the main array).
SPECIAL_ROWS = {
    0: "all equal (3.0)",
    1: "+1000 shift of a N(0, 9) draw (stored fp32)",
    2: "all about -1e4 (-1e4 + N(0, 1))",
}


def row_inputs(rows: int, length: int, seed: int, std: float = 3.0, specials: bool = False):
    """fp32 [rows, length] i.i.d. N(0, std^2).  With ``specials`` the rows listed in
    SPECIAL_ROWS, and the same three again as the last three rows, are replaced."""
    x = _normal(seed + 3, (rows, length), std)
    if specials and rows >= 6:
        for base in (0, rows - 3):
            x[base + 0, :] = np.float32(3.0)
            x[base + 1, :] = x[base + 1, :] + np.float32(1000.0)
            x[base + 2, :] = np.float32(-1e4) + x[base + 2, :] / np.float32(std)
    return x


def workload_row_inputs():
    """The three calls of the row-state workload: the main 4096 x 32768 array with
    special rows, 64 rows of length 1, and 1024 rows of length 32767 (rows start at
    float offsets that are not 16-byte aligned)."""
    w = WORKLOADS["rows_4096x32768"]
    main = row_inputs(w["rows"], w["length"], w["seed"], w["std"], specials=True)
    single = row_inputs(64, 1, w["seed"] + 10, w["std"])
    ragged = row_inputs(1024, 32767, w["seed"] + 20, w["std"])
    return main, single, ragged
