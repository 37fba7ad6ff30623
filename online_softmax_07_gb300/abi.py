"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

The functions here carry the C names and signatures: ``fa_fwd``, ``fa_fwd_dt``,
``fa_fwd_block``,
``fa_fwd_splitkv``, ``fa_fwd_splitkv_workspace_bytes``, ``fa_fwd_splitkv_default_splits``,
``fa_fwd_splitkv_splits_for``, ``fa_fwd_splitkv_static``, ``fa_bwd``, ``fa_bwd_workspace_bytes``,
``fa_bwd_workspace_bytes_dt``,
``fa_fwd_host``, ``fa_fwd_host_workspace_bytes``,
``online_softmax_rows``, ``online_softmax_forward``, ``fa_status_str``,
``fa_last_device_error`` and ``fa_selftest_wait_timeout``.  Pointer arguments accept a CUDA ``torch.Tensor``
(its data pointer is passed), an ``int`` address, or ``None`` (NULL).  A non-OK
status raises :class:`FAError`.  Every computation runs in the library's CUDA
kernels; there is no other implementation to fall back to, and loading fails
loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes
import os

(FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_ALIGN, FA_ERR_CUDA, FA_ERR_TIMEOUT,
 FA_ERR_TOO_LARGE) = range(7)
FA_BF16, FA_F32, FA_F16 = 0, 1, 2

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libosfa.so")

# Every exported symbol of include/fa.h with its ctypes signature.
_SIGNATURES = {
    "fa_fwd": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 4
               + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_dt": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 4
                  + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_block": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 4
                     + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_splitkv": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 4
                       + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                          ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_splitkv_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 5),
    "fa_fwd_splitkv_static": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p]
                              + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_splitkv_default_splits": (ctypes.c_int, [ctypes.c_int] * 4),
    "fa_fwd_splitkv_splits_for": (ctypes.c_int, [ctypes.c_int] * 5),
    "fa_fwd_host": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 4
                    + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                       ctypes.c_size_t, ctypes.c_void_p]),
    "fa_fwd_host_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 6),
    "fa_bwd": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 4
               + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                  ctypes.c_void_p]),
    "fa_bwd_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 3),
    "fa_bwd_workspace_bytes_dt": (ctypes.c_size_t, [ctypes.c_int] * 5),
    "online_softmax_rows": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2
                            + [ctypes.c_void_p]),
    "online_softmax_forward": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int] * 2
                               + [ctypes.c_void_p]),
    "fa_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_last_device_error": (ctypes.c_int, [ctypes.c_void_p]),
    "fa_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_longlong, ctypes.c_void_p]),
}


class FAError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {status_str(status)} (status {status})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libosfa.so (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -m online_softmax_07_gb300.build); "
                "the attention and row-state operations exist only as CUDA kernels")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("device pointer expected: pass a CUDA tensor")
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x).__name__} as a pointer")


def _host_ptr(x):
    """Address of a host buffer: a contiguous CPU torch.Tensor, an int, or None."""
    if x is None or isinstance(x, int):
        return x
    if x.is_cuda:
        raise ValueError("host pointer expected: pass a CPU tensor")
    if not x.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, call: str) -> None:
    if status != FA_OK:
        raise FAError(status, call)


def status_str(status: int) -> str:
    return load().fa_status_str(status).decode()


fa_status_str = status_str


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream=None) -> None:
    _check(load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                         float(scale), int(causal), _stream(stream)), "fa_fwd")


def fa_fwd_dt(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream=None) -> None:
    _check(load().fa_fwd_dt(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                            float(scale), int(causal), int(dtype), _stream(stream)), "fa_fwd_dt")


def fa_fwd_block(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, block_n, stream=None) -> None:
    """fa_fwd_dt with the keys per K/V tile chosen (block-size study: 64, 128 or 256)."""
    _check(load().fa_fwd_block(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                               float(scale), int(causal), int(dtype), int(block_n),
                               _stream(stream)), "fa_fwd_block")


def fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, num_splits, workspace,
                   workspace_bytes, dtype, stream=None) -> None:
    _check(load().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                 float(scale), int(causal), int(num_splits), _ptr(workspace),
                                 int(workspace_bytes), int(dtype), _stream(stream)),
           "fa_fwd_splitkv")


def fa_fwd_splitkv_static(q, k, v, o, lse, B, H, N, d, scale, causal, num_splits, dtype,
                          stream=None) -> None:
    """fa_fwd_splitkv with the partials in the library's static scratch: no workspace
    argument and no allocation (for callers that cannot allocate device memory)."""
    _check(load().fa_fwd_splitkv_static(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                        float(scale), int(causal), int(num_splits), int(dtype),
                                        _stream(stream)), "fa_fwd_splitkv_static")


def fa_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits) -> int:
    return int(load().fa_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits))


def fa_fwd_host(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, chunks, workspace,
                workspace_bytes, stream=None) -> None:
    """q, k, v, o, lse are host tensors (page-locked for overlapped copies); workspace is a
    device buffer of fa_fwd_host_workspace_bytes bytes."""
    _check(load().fa_fwd_host(_host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(o),
                              _host_ptr(lse), B, H, N, d, float(scale), int(causal), int(dtype),
                              int(chunks), _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "fa_fwd_host")


def fa_fwd_host_workspace_bytes(B, H, N, d, dtype, chunks) -> int:
    return int(load().fa_fwd_host_workspace_bytes(B, H, N, d, int(dtype), int(chunks)))


def fa_fwd_splitkv_default_splits(B, H, N, causal) -> int:
    return int(load().fa_fwd_splitkv_default_splits(B, H, N, int(causal)))


def fa_fwd_splitkv_splits_for(B, H, N, causal, sms) -> int:
    return int(load().fa_fwd_splitkv_splits_for(B, H, N, int(causal), int(sms)))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace,
           workspace_bytes, dtype, stream=None) -> None:
    _check(load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(causal),
                         _ptr(workspace), int(workspace_bytes), int(dtype), _stream(stream)),
           "fa_bwd")


def fa_bwd_workspace_bytes(B, H, N) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N))


def fa_bwd_workspace_bytes_dt(B, H, N, d, dtype) -> int:
    return int(load().fa_bwd_workspace_bytes_dt(B, H, N, d, dtype))


def online_softmax_rows(x, m_out, l_out, rows, length, stream=None) -> None:
    _check(load().online_softmax_rows(_ptr(x), _ptr(m_out), _ptr(l_out), rows, length,
                                      _stream(stream)), "online_softmax_rows")


def online_softmax_forward(x, y, m_out, l_out, rows, length, stream=None) -> None:
    _check(load().online_softmax_forward(_ptr(x), _ptr(y), _ptr(m_out), _ptr(l_out), rows, length,
                                         _stream(stream)), "online_softmax_forward")


def fa_last_device_error(stream=None) -> int:
    """Returns the status code (does not raise)."""
    return load().fa_last_device_error(_stream(stream))


def fa_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load().fa_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "fa_selftest_wait_timeout")
