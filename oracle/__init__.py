"""CPU oracle for the deterministic W-way bf16 reduce and its slot protocol.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product path (the C-ABI library and its Python binding) never imports, loads
or calls it, and this package never imports the product.  The two share only
the seeded input generator module, which holds none of the method's
arithmetic.

Contents
--------
* ``reduce`` / ``reduce_rows``: the rank-order fp32 sum rounded once to bf16,
  in plain C (``arx_oracle.c``), following arx.cu, ``arx_kernel``'s reduce
  loop.  Pinned by the ``-m "not gpu"`` tests against exhaustive rounding of
  all 2**32 binary32 patterns by torch, exact rational brute force, exact
  integer sums, the W=1 identity, zeros and signed zeros, and hand-derived
  fixtures under ``tests/golden/``.
* ``round_bf16`` / ``widen_bf16``: the two conversions, exposed for the pins.
* ``protocol``: a sequential model of the seq/parity slot protocol with its
  Semaphore epochs, signal pad and last-block counters.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib() -> ctypes.CDLL:
    """The oracle's shared library, built on first use."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        L.oracle_reduce.argtypes = [ctypes.POINTER(u16p), ctypes.c_int, u16p, ctypes.c_size_t]
        L.oracle_reduce.restype = ctypes.c_int
        L.oracle_reduce_mt.argtypes = [ctypes.POINTER(u16p), ctypes.c_int, u16p,
                                       ctypes.c_size_t, ctypes.c_int]
        L.oracle_reduce_mt.restype = ctypes.c_int
        L.oracle_reduce_rows.argtypes = [u16p, ctypes.c_int, u16p, ctypes.c_size_t, ctypes.c_int]
        L.oracle_reduce_rows.restype = ctypes.c_int
        L.oracle_round_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
        L.oracle_round_bf16_array.restype = None
        L.oracle_round_bf16_patterns.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t]
        L.oracle_round_bf16_patterns.restype = None
        L.oracle_widen_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
        L.oracle_widen_bf16_array.restype = None
        L.oracle_add_f32.argtypes = [ctypes.c_float, ctypes.c_float]
        L.oracle_add_f32.restype = ctypes.c_float
        L.oracle_fp_env_ok.argtypes = []
        L.oracle_fp_env_ok.restype = ctypes.c_int
        if L.oracle_fp_env_ok() != 1:
            raise RuntimeError("oracle: host floating point is not round-to-nearest with "
                               "subnormals kept; the oracle's sums would be wrong")
        _lib = L
    return _lib


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        if a.dtype == np.int16:
            a = a.view(np.uint16)
        else:
            raise TypeError(f"expected uint16 bf16 patterns, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr16(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def reduce(slots, out: np.ndarray | None = None, threads: int = 1) -> np.ndarray:
    """out[i] = bf16_rne(sum_{r=0}^{W-1} widen(slots[r][i])), accumulated in fp32 from +0.

    ``slots`` is a sequence of W uint16 arrays of equal length (or a [W, n]
    array).  ``out`` may be one of the slot arrays (the in-place form).
    """
    arrs = [_u16(s).reshape(-1) for s in slots]
    W = len(arrs)
    if W < 1:
        raise ValueError("W must be >= 1")
    n = arrs[0].size
    if any(a.size != n for a in arrs):
        raise ValueError("all slots must have the same length")
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    if out.dtype != np.uint16 or not out.flags.c_contiguous or out.size != n:
        raise ValueError("out must be a contiguous uint16 array of length n")
    ptrs = (ctypes.POINTER(ctypes.c_uint16) * W)(*[_ptr16(a) for a in arrs])
    rc = lib().oracle_reduce_mt(ptrs, W, _ptr16(out), n, int(threads))
    if rc != 0:
        raise ValueError("oracle_reduce rejected its arguments")
    return out


def reduce_rows(block: np.ndarray, threads: int = 1) -> np.ndarray:
    """Reduce a contiguous [W, n] uint16 block (slot r is row r)."""
    block = _u16(block)
    if block.ndim != 2:
        raise ValueError("expected a [W, n] block")
    W, n = block.shape
    out = np.empty(n, dtype=np.uint16)
    rc = lib().oracle_reduce_rows(_ptr16(block), W, _ptr16(out), n, int(threads))
    if rc != 0:
        raise ValueError("oracle_reduce_rows rejected its arguments")
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 patterns, round to nearest, ties to even."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_round_bf16_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def round_bf16_patterns(first: int, count: int) -> np.ndarray:
    """bf16 patterns of the binary32 patterns first .. first+count-1."""
    out = np.empty(count, dtype=np.uint16)
    lib().oracle_round_bf16_patterns(first, out.ctypes.data, count)
    return out


def widen_bf16(b: np.ndarray) -> np.ndarray:
    """bf16 patterns -> binary32 values (exact)."""
    b = _u16(b)
    out = np.empty(b.shape, dtype=np.float32)
    lib().oracle_widen_bf16_array(b.ctypes.data, out.ctypes.data, b.size)
    return out


def add_f32(a: float, b: float) -> float:
    """One host binary32 addition (round to nearest, ties to even)."""
    return lib().oracle_add_f32(a, b)


def is_nan_bf16(b: np.ndarray) -> np.ndarray:
    b = _u16(b)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


from . import protocol  # noqa: E402  (the protocol model needs reduce())
