"""The C-ABI library on the host (no GPU): it builds, loads, exports every symbol
include/fa.h declares, and rejects bad arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

from online_softmax_07_gb300 import abi
from online_softmax_07_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_library()
    return abi.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(names) == set(abi._SIGNATURES), names
    for name in names:
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    for code in range(7):
        assert abi.status_str(code) != "unknown status"
    assert abi.status_str(99) == "unknown status"


FAKE = 0x10000  # an aligned address that is never dereferenced (checks fail first)


@pytest.mark.parametrize("args,expect", [
    (dict(d=96), abi.FA_ERR_UNSUPPORTED),
    (dict(d=32), abi.FA_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), abi.FA_ERR_INVALID),
    (dict(scale=float("inf")), abi.FA_ERR_INVALID),
    (dict(scale=0.0), abi.FA_ERR_INVALID),
    (dict(scale=-0.125), abi.FA_ERR_INVALID),
    (dict(causal=2), abi.FA_ERR_INVALID),
    (dict(N=-1), abi.FA_ERR_INVALID),
    (dict(B=-2), abi.FA_ERR_INVALID),
    (dict(q=None), abi.FA_ERR_INVALID),
    (dict(o=None), abi.FA_ERR_INVALID),
    (dict(q=FAKE + 8), abi.FA_ERR_ALIGN),
    (dict(v=FAKE + 2), abi.FA_ERR_ALIGN),
    (dict(lse=FAKE + 2), abi.FA_ERR_ALIGN),
    (dict(B=0), abi.FA_OK),          # empty problems launch nothing
    (dict(H=0), abi.FA_OK),
    (dict(N=0), abi.FA_OK),
    (dict(B=65536, H=65536), abi.FA_ERR_INVALID),
])
def test_fa_fwd_argument_checks(lib, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125,
             causal=0)
    a.update(args)
    st = lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                    a["scale"], a["causal"], None)
    assert st == expect, abi.status_str(st)


@pytest.mark.parametrize("d,align,dtype,expect", [
    (200, 4, abi.FA_F32, abi.FA_ERR_UNSUPPORTED),
    (0, 4, abi.FA_F32, abi.FA_ERR_UNSUPPORTED),
    (17, 2, abi.FA_F32, abi.FA_ERR_ALIGN),
    (64, 16, 7, abi.FA_ERR_UNSUPPORTED),
])
def test_fa_fwd_dt_argument_checks(lib, d, align, dtype, expect):
    p = FAKE + (align if align < 4 else 0)
    st = lib.fa_fwd_dt(p, p, p, p, None, 1, 1, 16, d, 0.5, 0, dtype, None)
    assert st == expect


@pytest.mark.parametrize("x,m,l,rows,length,expect", [
    (FAKE, FAKE, FAKE, 0, 0, abi.FA_OK),          # nothing to do
    (None, None, None, 0, 5, abi.FA_OK),
    (FAKE, FAKE, FAKE, 3, 0, abi.FA_ERR_INVALID),  # the max of an empty row is undefined
    (FAKE, FAKE, FAKE, -1, 5, abi.FA_ERR_INVALID),
    (None, FAKE, FAKE, 3, 5, abi.FA_ERR_INVALID),
    (FAKE, None, FAKE, 3, 5, abi.FA_ERR_INVALID),
    (FAKE + 1, FAKE, FAKE, 3, 5, abi.FA_ERR_ALIGN),
    (FAKE, FAKE, FAKE + 2, 3, 5, abi.FA_ERR_ALIGN),
])
def test_row_state_argument_checks(lib, x, m, l, rows, length, expect):
    assert lib.online_softmax_rows(x, m, l, rows, length, None) == expect


def test_selftest_limit_checked(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == abi.FA_ERR_INVALID
    assert lib.fa_selftest_wait_timeout(3_000_000_000, None) == abi.FA_ERR_INVALID


def test_binding_has_no_fallback(tmp_path):
    saved = abi._lib
    try:
        abi._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            abi.load(str(tmp_path / "libosfa.so"))
    finally:
        abi._lib = saved


def test_splitkv_workspace_size(lib):
    # splits * B * H * ceil(N/256)*256 * (d + 1) * 4
    assert abi.fa_fwd_splitkv_workspace_bytes(1, 2, 300, 128, 3) == 3 * 2 * 512 * 129 * 4
    assert abi.fa_fwd_splitkv_workspace_bytes(2, 1, 256, 64, 1) == 1 * 2 * 256 * 65 * 4
    assert abi.fa_fwd_splitkv_workspace_bytes(1, 1, 100, 96, 2) == 0      # unsupported d
    assert abi.fa_fwd_splitkv_workspace_bytes(1, 1, 100, 64, 0) == 0      # no splits


@pytest.mark.parametrize("sms", [148, 152])
def test_splitkv_split_rule(lib, sms):
    """The split-count rule (the same answers with 148 or 152 SMs).  Query blocks =
    B * H * ceil(N / 256)."""
    f = lambda B, H, N, c: abi.fa_fwd_splitkv_splits_for(B, H, N, c, sms)
    assert f(1, 1, 16384, True) == 4        # causal, 64 blocks: floor(2 * SMs / 64 + 0.2)
    assert f(1, 1, 32768, True) == 2        # causal, 128 blocks
    assert f(1, 5, 8192, True) == 2         # causal, 160 blocks
    assert f(1, 2, 32768, True) == 1        # causal, 256 blocks: no split
    assert f(1, 1, 8192, False) == 4        # not causal, 32 blocks: 128 pieces, one wave
    assert f(1, 2, 16384, False) == 1       # not causal, 128 blocks
    assert f(1, 1, 512, True) == 2          # 2 blocks, but 4 K/V tiles: two per split
    assert f(1, 1, 100, False) == 1         # a single K/V tile
    assert f(1, 1, 100000, True) <= 64
    assert f(0, 1, 1024, True) == 1 and f(1, 1, 1024, 2) == 1
    assert abi.fa_fwd_splitkv_splits_for(1, 1, 16384, 1, 0) == 1     # no SMs: no split


def test_splitkv_default_splits_without_a_device(lib):
    """With no device to read the SM count from, the default is one split."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert abi.fa_fwd_splitkv_default_splits(1, 1, 16384, True) == 1


@pytest.mark.parametrize("splits,ws,ws_bytes,expect", [
    (0, FAKE, 1 << 30, abi.FA_ERR_INVALID),
    (65, FAKE, 1 << 30, abi.FA_ERR_INVALID),
    (2, None, 1 << 30, abi.FA_ERR_INVALID),
    (2, FAKE, 100, abi.FA_ERR_INVALID),        # workspace too small
    (2, FAKE + 8, 1 << 30, abi.FA_ERR_ALIGN),
])
def test_splitkv_argument_checks(lib, splits, ws, ws_bytes, expect):
    st = lib.fa_fwd_splitkv(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1000, 128, 0.1, 1, splits, ws,
                            ws_bytes, abi.FA_BF16, None)
    assert st == expect, abi.status_str(st)


@pytest.mark.parametrize("args,expect", [
    (dict(splits=0), abi.FA_ERR_INVALID),          # out of range: rejected before any CUDA call
    (dict(splits=65), abi.FA_ERR_INVALID),
    (dict(splits=65, B=1, H=64, N=32768), abi.FA_ERR_INVALID),   # not "too large"
    (dict(d=96), abi.FA_ERR_UNSUPPORTED),          # no workspace size: fa_fwd_splitkv decides
    (dict(scale=-1.0), abi.FA_ERR_INVALID),
    (dict(B=0), abi.FA_OK),                        # empty problem: nothing launched
    (dict(N=0), abi.FA_OK),
    (dict(H=64, N=32768), abi.FA_ERR_TOO_LARGE),   # 2 splits need ~1.1 GB of partials
    (dict(H=64, N=32768, scale=float("nan")), abi.FA_ERR_INVALID),   # argument errors first
    (dict(H=64, N=32768, q=None), abi.FA_ERR_INVALID),
    (dict(H=64, N=32768, k=FAKE + 8), abi.FA_ERR_ALIGN),
])
def test_splitkv_static_argument_checks(lib, args, expect):
    """The scratch-memory split-KV entry checks its arguments on the host; none of these
    cases touches the device."""
    a = dict(q=FAKE, k=FAKE, v=FAKE, B=1, H=1, N=1000, d=128, scale=0.1, splits=2)
    a.update(args)
    st = lib.fa_fwd_splitkv_static(a["q"], a["k"], a["v"], FAKE, None, a["B"], a["H"], a["N"],
                                   a["d"], a["scale"], 1, a["splits"], abi.FA_BF16, None)
    assert st == expect, abi.status_str(st)


@pytest.mark.parametrize("block_n,d,dtype,expect", [
    (32, 64, abi.FA_BF16, abi.FA_ERR_INVALID),
    (160, 64, abi.FA_BF16, abi.FA_ERR_INVALID),
    (192, 128, abi.FA_BF16, abi.FA_ERR_UNSUPPORTED),    # 192-key tiles only at d = 64
    (256, 128, abi.FA_BF16, abi.FA_ERR_UNSUPPORTED),    # 256-key tiles only at d = 64
    (64, 64, abi.FA_F16, abi.FA_ERR_UNSUPPORTED),       # study kernels are bf16 only
    (64, 64, abi.FA_F32, abi.FA_ERR_UNSUPPORTED),
    (64, 96, abi.FA_BF16, abi.FA_ERR_UNSUPPORTED),
])
def test_fa_fwd_block_argument_checks(lib, block_n, d, dtype, expect):
    st = lib.fa_fwd_block(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 256, d, 0.1, 1, dtype, block_n, None)
    assert st == expect, abi.status_str(st)


def test_fa_fwd_block_empty_and_bad_scale(lib):
    # checked on the host before any CUDA call, whatever the block size
    for block_n in (64, 192, 256):
        assert lib.fa_fwd_block(FAKE, FAKE, FAKE, FAKE, None, 0, 1, 256, 64, 0.1, 1, abi.FA_BF16,
                                block_n, None) == abi.FA_OK
        assert lib.fa_fwd_block(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 256, 64, -1.0, 1, abi.FA_BF16,
                                block_n, None) == abi.FA_ERR_INVALID


def test_splitkv_rejects_f32(lib):
    st = lib.fa_fwd_splitkv(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 100, 64, 0.1, 0, 2, FAKE, 1 << 30,
                            abi.FA_F32, None)
    assert st == abi.FA_ERR_UNSUPPORTED


def test_bwd_workspace_size(lib):
    # Per (head, query row), rows padded to a multiple of 128: bf16/fp16 at d = 128 2 fp32
    # statistics and 16 bf16 statistics terms; at d = 64 the terms and a 64-float dQ
    # accumulator row; fp32 2 fp32 statistics.
    dt = abi.fa_bwd_workspace_bytes_dt
    assert dt(2, 3, 300, 128, abi.FA_BF16) == (2 * 4 + 16 * 2) * 6 * 384
    assert dt(2, 3, 300, 128, abi.FA_F16) == (2 * 4 + 16 * 2) * 6 * 384
    assert dt(2, 3, 300, 64, abi.FA_BF16) == (16 * 2 + 64 * 4) * 6 * 384
    assert dt(1, 1, 128, 64, abi.FA_F16) == (16 * 2 + 64 * 4) * 128
    assert dt(1, 1, 128, 64, abi.FA_F32) == 2 * 128 * 4
    assert dt(1, 1, 100, 17, abi.FA_F32) == 2 * 128 * 4
    assert dt(1, 1, 100, 96, abi.FA_BF16) == 0       # unsupported d
    assert dt(1, 1, 100, 129, abi.FA_F32) == 0
    assert dt(1, 1, 100, 64, 7) == 0                 # unsupported dtype
    assert dt(-1, 1, 100, 64, abi.FA_BF16) == 0
    assert dt(0, 4, 100, 64, abi.FA_BF16) == 0
    # The dtype-free size serves every case: the d = 64 one.
    assert abi.fa_bwd_workspace_bytes(2, 3, 300) == (16 * 2 + 64 * 4) * 6 * 384
    assert abi.fa_bwd_workspace_bytes(1, 1, 128) == (16 * 2 + 64 * 4) * 128
    assert abi.fa_bwd_workspace_bytes(0, 4, 100) == 0
    assert abi.fa_bwd_workspace_bytes(-1, 4, 100) == 0


def test_bwd_d64_workspace_must_hold_the_dq_accumulator(lib):
    """A workspace that serves d = 128 is too small at d = 64 (rejected before any launch)."""
    small = abi.fa_bwd_workspace_bytes_dt(1, 2, 300, 128, abi.FA_BF16)
    st = lib.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 300, 64, 0.1, 0,
                    FAKE, small, abi.FA_BF16, None)
    assert st == abi.FA_ERR_INVALID


@pytest.mark.parametrize("args,expect", [
    (dict(B=0), abi.FA_OK),                       # empty problems launch nothing
    (dict(N=0, q=None), abi.FA_OK),
    (dict(d=96), abi.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), abi.FA_ERR_UNSUPPORTED),
    (dict(dtype=abi.FA_F32, d=129), abi.FA_ERR_UNSUPPORTED),
    (dict(dtype=abi.FA_F32, d=0), abi.FA_ERR_UNSUPPORTED),
    (dict(dtype=abi.FA_F32, d=17, dq=FAKE + 2), abi.FA_ERR_ALIGN),
    (dict(dtype=abi.FA_F32, d=17, ws=FAKE + 4), abi.FA_ERR_ALIGN),
    (dict(scale=0.0), abi.FA_ERR_INVALID),
    (dict(causal=3), abi.FA_ERR_INVALID),
    (dict(lse=None), abi.FA_ERR_INVALID),         # the backward needs the forward's LSE
    (dict(dout=None), abi.FA_ERR_INVALID),
    (dict(ws=None), abi.FA_ERR_INVALID),
    (dict(ws_bytes=100), abi.FA_ERR_INVALID),     # workspace too small
    (dict(dq=FAKE + 8), abi.FA_ERR_ALIGN),
    (dict(ws=FAKE + 4), abi.FA_ERR_ALIGN),
    (dict(lse=FAKE + 2), abi.FA_ERR_ALIGN),
])
def test_fa_bwd_argument_checks(lib, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1,
             H=2, N=300, d=128, scale=0.1, causal=1, ws=FAKE, ws_bytes=1 << 20, dtype=abi.FA_BF16)
    a.update(args)
    st = lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dout"], a["dq"], a["dk"], a["dv"],
                    a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"], a["ws"], a["ws_bytes"],
                    a["dtype"], None)
    assert st == expect, abi.status_str(st)

def test_fwd_host_workspace_size(lib):
    """Three groups' Q, K, V, O (256-byte aligned) and LSE at most; heads per group =
    ceil(B * H / chunks)."""
    f = abi.fa_fwd_host_workspace_bytes
    # B*H = 8 in 3 groups of 3 heads: 3 slots of 4 * 115200 + 3840 bytes
    assert f(2, 4, 300, 64, abi.FA_BF16, 3) == 3 * (4 * 115200 + 3840)
    # one head, fp32 d = 64: one slot; 100 * 4 LSE bytes rounded up to 512
    assert f(1, 1, 100, 64, abi.FA_F32, 5) == 4 * 25600 + 512
    # 16 heads in 8 groups of 2: still three slots
    assert f(1, 16, 128, 128, abi.FA_F16, 8) == 3 * (4 * 65536 + 1024)
    assert f(1, 1, 100, 64, abi.FA_BF16, 0) == 0          # no chunks
    assert f(1, 1, 100, 96, abi.FA_BF16, 2) == 0          # unsupported d
    assert f(0, 4, 100, 64, abi.FA_BF16, 2) == 0          # empty


@pytest.mark.parametrize("args,expect", [
    (dict(chunks=0), abi.FA_ERR_INVALID),
    (dict(d=96), abi.FA_ERR_UNSUPPORTED),
    (dict(causal=2), abi.FA_ERR_INVALID),
    (dict(ws=None), abi.FA_ERR_INVALID),
    (dict(ws_bytes=16), abi.FA_ERR_INVALID),
    (dict(ws=8), abi.FA_ERR_ALIGN),
    (dict(q=None), abi.FA_ERR_INVALID),
    (dict(B=0), abi.FA_OK),                               # empty: nothing to do
])
def test_fwd_host_argument_checks(lib, args, expect):
    """Rejected (or, for an empty problem, accepted) before any CUDA call."""
    a = dict(q=4096, B=1, H=2, N=100, d=64, causal=0, chunks=2, ws=1 << 20, ws_bytes=1 << 30)
    a.update(args)
    st = lib.fa_fwd_host(a["q"], 8192, 12288, 16384, None, a["B"], a["H"], a["N"], a["d"],
                         0.125, a["causal"], abi.FA_BF16, a["chunks"], a["ws"], a["ws_bytes"],
                         None)
    assert st == expect
