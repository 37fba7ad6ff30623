"""Parity of the row softmax output y = exp(x - m) / l (C ABI) against the oracle."""

import numpy as np
import pytest

import oracle
from online_softmax_07_gb300 import abi, synth
from online_softmax_07_gb300.build import build_library

from gpu_helpers import ROW_REL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    abi.load()


def run_softmax(x, with_state=True, in_place=False, y_offset=0):
    import torch
    rows, length = x.shape
    dx = to_device(x, torch.float32)
    if in_place:
        y = dx
    elif y_offset:
        buf = torch.full((rows * length + 4,), float("nan"), device="cuda")
        y = buf[y_offset:y_offset + rows * length]
    else:
        y = torch.full_like(dx, float("nan"))
    m = torch.full((rows,), float("nan"), device="cuda") if with_state else None
    l = torch.full((rows,), float("nan"), device="cuda") if with_state else None
    abi.online_softmax_forward(dx, y.data_ptr(), m, l, rows, length)
    assert abi.fa_last_device_error() == abi.FA_OK
    out = y.reshape(rows, length).cpu().numpy().astype(np.float64)
    if with_state:
        return out, m.cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64)
    return out, None, None


def check(x, y, m, l):
    ref = oracle.softmax_rows(x)
    assert np.all(np.isfinite(y))
    err = np.abs(y - ref)
    assert np.all(err <= ROW_REL * ref + 1e-37), f"max rel err {np.max(err / np.maximum(ref, 1e-30)):.3e}"
    if m is not None:
        m_ref, l_ref = oracle.row_state(x)
        assert np.all(m == m_ref)
        assert np.max(np.abs(l - l_ref) / l_ref) <= ROW_REL


def test_workload_main_array():
    main, _, _ = synth.workload_row_inputs()
    y, m, l = run_softmax(main)
    check(main, y, m, l)
    assert np.all(y[0] == np.float32(1.0 / 32768))      # all-equal row: uniform


@pytest.mark.parametrize("length", [1, 2, 3, 31, 33, 1000, 1024, 1025, 4099, 32767, 32768,
                                    32769, 70001])
def test_lengths(length):
    x = synth.row_inputs(5, length, seed=83000 + length)
    y, m, l = run_softmax(x)
    check(x, y, m, l)


def test_in_place_and_no_state():
    x = synth.row_inputs(7, 5000, seed=84000)
    y, _, _ = run_softmax(x, with_state=False, in_place=True)
    check(x, y, None, None)
    x = synth.row_inputs(9, 600, seed=84001)
    y, _, _ = run_softmax(x, with_state=False, in_place=True)
    check(x, y, None, None)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_output_misaligned_from_input(offset):
    x = synth.row_inputs(6, 6000, seed=85000 + offset)
    y, m, l = run_softmax(x, y_offset=offset)
    check(x, y, m, l)
