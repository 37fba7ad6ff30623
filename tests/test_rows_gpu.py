"""Parity of the row online-softmax state (C ABI, CUDA kernels) against the oracle."""

import numpy as np
import pytest

import oracle
from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

from gpu_helpers import ROW_REL, run_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    abi.load()


def check_rows(x, m, l):
    m_ref, l_ref = oracle.row_state(x)
    assert np.all(m == m_ref), "m is a max of stored fp32 values: it must be exact"
    rel = np.abs(l - l_ref) / l_ref
    assert rel.max() <= ROW_REL, f"l max rel err {rel.max():.3e}"
    return float(rel.max())


def test_workload_main_with_special_rows():
    """4096 x 32768 N(0, 9) with all-equal, +1000-shifted and ~-1e4 rows."""
    main, _, _ = synth.workload_row_inputs()
    m, l = run_rows(main)
    check_rows(main, m, l)
    # the special rows against closed forms as well
    assert m[0] == 3.0 and l[0] == 32768.0 and m[-3] == 3.0 and l[-3] == 32768.0


def test_workload_length_one_and_ragged():
    _, single, ragged = synth.workload_row_inputs()
    m, l = run_rows(single)
    check_rows(single, m, l)
    assert np.all(l == 1.0)
    m, l = run_rows(ragged)           # 32767 floats per row: rows start unaligned
    check_rows(ragged, m, l)


@pytest.mark.parametrize("length", [1, 2, 3, 5, 31, 32, 33, 255, 1023, 1024, 1025, 1027,
                                    2048, 4099, 65536 + 3])
def test_lengths(length):
    x = synth.row_inputs(37, length, seed=80000 + length)
    m, l = run_rows(x)
    check_rows(x, m, l)


@pytest.mark.parametrize("rows,length,sigma", [(2, 4_000_003, 3.0), (1, 16_000_001, 3.0),
                                               (1, 16_000_001, 0.01)])
def test_very_long_rows(rows, length, sigma):
    """Rows of 4 M and 16 M floats (each thread folds hundreds of batches into its l);
    sigma 0.01 makes every term of l close to 1, so l is a sum of 16 M similar terms."""
    x = synth.row_inputs(rows, length, seed=84000 + int(sigma * 100), std=sigma)
    m, l = run_rows(x)
    check_rows(x, m, l)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_base_pointer(offset):
    """The array itself starts 4, 8 or 12 bytes past a 16-byte boundary."""
    import torch
    rows, length = 9, 5000
    x = synth.row_inputs(rows, length, seed=81000 + offset)
    buf = torch.zeros(rows * length + 4, device="cuda")
    buf[offset:offset + rows * length] = to_device(x.reshape(-1), torch.float32)
    view = buf[offset:offset + rows * length]
    m = torch.empty(rows, device="cuda")
    l = torch.empty(rows, device="cuda")
    abi.online_softmax_rows(view.data_ptr(), m, l, rows, length)
    assert abi.fa_last_device_error() == abi.FA_OK
    check_rows(x, m.cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64))


def test_zero_rows_is_noop():
    import torch
    m = torch.full((2,), 5.0, device="cuda")
    abi.online_softmax_rows(m, m, m, 0, 7)
    torch.cuda.synchronize()
    assert bool((m == 5.0).all())


def test_wait_timeout_reports_and_context_survives():
    """The bounded-wait path: a wait on a barrier that never completes gives up after
    its limit, the host reads FA_ERR_TIMEOUT, and later work runs normally."""
    abi.fa_selftest_wait_timeout(50_000_000)
    assert abi.fa_last_device_error() == abi.FA_ERR_TIMEOUT
    assert abi.fa_last_device_error() == abi.FA_OK      # the word was cleared
    x = synth.row_inputs(5, 3000, seed=82000)
    m, l = run_rows(x)
    check_rows(x, m, l)
