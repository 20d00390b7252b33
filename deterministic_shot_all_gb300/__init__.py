"""Deterministic W-way bf16 reduce for one GB300 (sm_103a): Python binding.

This module only marshals arguments to the C ABI of ``libarx.so`` (declared
in ``include/arx.h``): tensors become device pointers, the current torch
stream becomes a ``cudaStream_t``.  Every step of the computation runs in the
library's CUDA kernels.  Importing fails loudly when the library has not been
built (``python -c "import __graft_entry__ as g; g.build()"``); there is no
CPU fallback.

Functions keep the C names:

* ``arx_reduce(slots, out)``: out = bf16(rank-order fp32 sum of slots), out
  may be one of the slots.
* ``arx_reduce_host(host_slots, host_out, staging)``: the same from and to
  host buffers, copies included.
* ``arx_ctx_workspace_bytes / arx_ctx_init / arx_step / arx_ctx_query /
  arx_ctx_reset / arx_ctx_set_timeout / arx_ctx_set_fault / arx_ctx_set_sync``:
  the seq/parity protocol step with Semaphore epochs and a zero-resetting
  signal pad, in five barrier variants.
* ``arx_ext_*``: the external-writer form -- a host thread writes each
  rank's partial into page-locked slots and raises its flag, the GPU waits
  for the flags and reduces.
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libarx.so")

ARX_OK, ARX_EINVAL, ARX_EOVERLAP, ARX_ECUDA, ARX_ETIMEOUT, ARX_ESTATE = range(6)
ARX_MAX_W = 8
ARX_STEP_MAX_BLOCKS = 256
ARX_DEFAULT_TIMEOUT_NS = 1_000_000_000
ARX_NOALLOC_MAX_N = 131072
ARX_SYNC_SEMAPHORE, ARX_SYNC_PAD, ARX_SYNC_PAD_FENCED, ARX_SYNC_CLUSTER, ARX_SYNC_SEMAPHORE_GLOBAL = range(5)
ARX_SLOTS_DEVICE, ARX_SLOTS_HOST = range(2)


class ArxError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{arx_status_string(status)}: {detail}" if detail else arx_status_string(status))
        self.status = status


class arx_watch_report(ctypes.Structure):
    """Mirror of ``struct arx_watch_report`` in include/arx.h."""
    _fields_ = [
        ("seq", ctypes.c_uint32),
        ("published", ctypes.c_uint32),
        ("dev_err", ctypes.c_uint32),
        ("polls", ctypes.c_uint32),
        ("stalled_ns", ctypes.c_uint64),
        ("waited_ns", ctypes.c_uint64),
    ]


class arx_ctx(ctypes.Structure):
    """Mirror of ``struct arx_ctx`` in include/arx.h."""
    _fields_ = [
        ("magic", ctypes.c_uint32),
        ("W", ctypes.c_int32),
        ("nblocks", ctypes.c_int32),
        ("fault_rank", ctypes.c_int32),
        ("sync_mode", ctypes.c_int32),
        ("slots_where", ctypes.c_int32),
        ("max_n", ctypes.c_uint64),
        ("slot_stride", ctypes.c_uint64),
        ("timeout_ns", ctypes.c_uint64),
        ("ws", ctypes.c_void_p),
        ("ws_bytes", ctypes.c_uint64),
        ("off_epoch", ctypes.c_uint64),
        ("off_sem", ctypes.c_uint64),
        ("off_pad", ctypes.c_uint64),
        ("off_slots", ctypes.c_uint64),
        ("ctrl_bytes", ctypes.c_uint64),
        ("slots", ctypes.c_void_p),
        ("slots_bytes", ctypes.c_uint64),
        ("failed_err", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
    ]


class arx_ext(ctypes.Structure):
    """Mirror of ``struct arx_ext`` in include/arx.h."""
    _fields_ = [
        ("magic", ctypes.c_uint32),
        ("W", ctypes.c_int32),
        ("nblocks", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("max_n", ctypes.c_uint64),
        ("slot_stride", ctypes.c_uint64),
        ("timeout_ns", ctypes.c_uint64),
        ("words", ctypes.c_void_p),
        ("host_region", ctypes.c_void_p),
        ("dev_region", ctypes.c_void_p),
        ("region_bytes", ctypes.c_uint64),
        ("failed_err", ctypes.c_uint32),
        ("reserved1", ctypes.c_uint32),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()'); there is no CPU fallback")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, u32p, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_uint32), ctypes.c_uint64
    ptrs = ctypes.POINTER(ctypes.c_void_p)
    ctxp = ctypes.POINTER(arx_ctx)
    extp = ctypes.POINTER(arx_ext)
    u32 = ctypes.c_uint32
    sigs = {
        "arx_status_string": ([i32], ctypes.c_char_p),
        "arx_last_error": ([], ctypes.c_char_p),
        "arx_reduce": ([ptrs, i32, vp, sz, vp], i32),
        "arx_reduce_host_staging_bytes": ([i32, sz], sz),
        "arx_reduce_host": ([ptrs, i32, vp, sz, vp, sz, vp], i32),
        "arx_ctx_workspace_bytes": ([i32, sz, i32], sz),
        "arx_ctx_init": ([ctxp, vp, sz, i32, sz, i32], i32),
        "arx_ctx_words_bytes": ([i32, i32], sz),
        "arx_ctx_slots_bytes": ([i32, sz], sz),
        "arx_ctx_init_split": ([ctxp, vp, sz, vp, sz, i32, i32, sz, i32], i32),
        "arx_ctx_set_timeout": ([ctxp, u64], i32),
        "arx_ctx_set_fault": ([ctxp, i32], i32),
        "arx_ctx_set_sync": ([ctxp, i32], i32),
        "arx_ctx_reset": ([ctxp, vp], i32),
        "arx_step": ([ctxp, ptrs, vp, sz, vp], i32),
        "arx_ctx_query": ([ctxp, u32p, u32p, vp], i32),
        "arx_step_noalloc": ([ptrs, i32, vp, sz, vp, vp], i32),
        "arx_watch_step": ([ctxp, ctypes.c_uint32, u64, u64, u64, u32p, vp, ctypes.POINTER(arx_watch_report)], i32),
        "arx_ext_region_bytes": ([i32, sz], sz),
        "arx_ext_words_bytes": ([], sz),
        "arx_ext_init": ([extp, vp, sz, vp, sz, i32, sz, i32], i32),
        "arx_ext_set_timeout": ([extp, u64], i32),
        "arx_ext_wait_free": ([extp, u32, u64], i32),
        "arx_ext_slot": ([extp, u32, i32], vp),
        "arx_ext_publish": ([extp, i32, u32], i32),
        "arx_ext_post": ([extp, i32, u32, vp, sz, u64], i32),
        "arx_ext_publish_all": ([extp, u32, u64], i32),
        "arx_ext_step": ([extp, vp, sz, vp], i32),
        "arx_ext_query": ([extp, u32p, u32p, vp], i32),
        "arx_ext_reset": ([extp, vp], i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


lib = _load()


def arx_status_string(status: int) -> str:
    return lib.arx_status_string(int(status)).decode()


def arx_last_error() -> str:
    return lib.arx_last_error().decode()


def _check(status: int) -> None:
    if status != ARX_OK:
        raise ArxError(status, arx_last_error())


def _ptr(x) -> int:
    """Address of a tensor's first element, or an int address as given."""
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an integer address, got {type(x).__name__}")


def _check_bf16(xs: Sequence, n: int | None, where: str, what: str) -> None:
    """Marshalling checks of tensor arguments (integer addresses pass unchecked):
    bf16, contiguous, at least n elements, and on the side the call expects --
    ``where`` is "cuda" (the current device) or "cpu".  Catches a host tensor
    handed to a device entry point, or a wrong dtype, before any kernel sees
    the pointer."""
    import torch
    current = None
    for i, x in enumerate(xs):
        if isinstance(x, int) or not hasattr(x, "dtype"):
            continue
        ok = (x.dtype == torch.bfloat16 and x.is_contiguous() and (n is None or x.numel() >= n)
              and x.is_cuda == (where == "cuda"))
        if ok and where == "cuda":
            if current is None:
                current = torch.cuda.current_device()
            ok = x.device.index == current
        if ok:
            continue
        name = f"{what}[{i}]" if len(xs) > 1 else what
        if x.dtype != torch.bfloat16:
            raise TypeError(f"{name}: expected torch.bfloat16, got {x.dtype}")
        if not x.is_contiguous():
            raise ValueError(f"{name}: must be contiguous")
        if n is not None and x.numel() < n:
            raise ValueError(f"{name}: {x.numel()} elements, the call needs {n}")
        if where == "cuda" and not x.is_cuda:
            raise ValueError(f"{name}: expected a CUDA tensor, got one on {x.device}")
        if where != "cuda" and x.is_cuda:
            raise ValueError(f"{name}: expected a host (CPU) tensor, got one on {x.device}")
        raise ValueError(f"{name}: on {x.device}, but the current device is cuda:{current}")


def _ptr_array(xs: Sequence) -> ctypes.Array:
    return _ptr_array_type(len(xs))(*[_ptr(x) for x in xs])


_ARRAY_TYPES: dict = {}
_BF16 = None


def _ptr_array_type(k: int):
    t = _ARRAY_TYPES.get(k)
    if t is None:
        t = _ARRAY_TYPES[k] = ctypes.c_void_p * k
    return t


def _marshal(xs: Sequence, out, n: int, where: str, what: str, what_out: str):
    """Checks ``xs`` and ``out`` as _check_bf16 does and returns (array of the
    xs' addresses, out's address).  One pass over the tensors with one call
    per property; on any failure the per-tensor checks run again to raise
    their message."""
    global _BF16
    if _BF16 is None:
        import torch
        _BF16 = torch.bfloat16
    cuda = where == "cuda"
    want = None  # the current device, looked up once a tensor is on a GPU
    addrs = []
    for x in (*xs, out):
        if isinstance(x, int):
            addrs.append(x)
            continue
        try:
            if x.dtype is _BF16 and x.is_contiguous() and x.numel() >= n:
                d = x.get_device()
                if cuda and d >= 0:
                    if want is None:
                        import torch
                        want = torch.cuda.current_device()
                    if d == want:
                        addrs.append(x.data_ptr())
                        continue
                elif not cuda and d < 0:
                    addrs.append(x.data_ptr())
                    continue
        except AttributeError:
            pass
        _check_bf16(xs, n, where, what)
        _check_bf16([out], n, where, what_out)
        addrs = [_ptr(y) for y in (*xs, out)]
        break
    return _ptr_array_type(len(xs))(*addrs[:-1]), addrs[-1]


def _stream(stream) -> int:
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _numel(n, out) -> int:
    if n is not None:
        return int(n)
    if hasattr(out, "numel"):
        return int(out.numel())
    raise ValueError("n is required when out is an address")


def arx_reduce(slots: Sequence, out, n: int | None = None, stream=None, check: bool = True) -> int:
    """Enqueue out = bf16(sum over slots in rank order, fp32) on ``stream``.

    ``slots``: W (1..8) bf16 device tensors or addresses; ``out``: bf16 device
    tensor or address, may be one of the slots.  Returns the arx_status (and
    raises ArxError on failure when ``check``).
    """
    n = _numel(n, out)
    arr, optr = _marshal(slots, out, n, "cuda", "slots", "out")
    st = lib.arx_reduce(arr, len(arr), optr, n, _stream(stream))
    if check:
        _check(st)
    return st


class arx_reduce_plan:
    """A prepared ``arx_reduce``: the arguments are checked and marshalled once,
    and every call of the plan is one C call with the stored pointers, for
    eager callers that repeat the same reduce (graph replays need no plan).
    The plan keeps the tensors alive; their contents may change between calls,
    their storage must not."""

    def __init__(self, slots: Sequence, out, n: int | None = None, stream=None):
        n = _numel(n, out)
        self._arr, self._out = _marshal(slots, out, n, "cuda", "slots", "out")
        self._refs = (list(slots), out)
        self._W = len(slots)
        self._n = n
        self._stream = _stream(stream)
        self._fn = lib.arx_reduce

    def __call__(self) -> None:
        st = self._fn(self._arr, self._W, self._out, self._n, self._stream)
        if st != ARX_OK:
            _check(st)


def arx_reduce_host_staging_bytes(W: int, n: int) -> int:
    return int(lib.arx_reduce_host_staging_bytes(W, n))


def arx_reduce_host(host_slots: Sequence, host_out, staging=None, n: int | None = None,
                    stream=None, check: bool = True) -> int:
    """Enqueue the reduce of host partials into a host output.

    Page-locked buffers are read and written by the kernel directly; pageable
    ones go through ``staging`` (a device tensor of
    ``arx_reduce_host_staging_bytes(W, n)`` bytes).
    """
    if staging is None:
        sptr, nb = None, 0
    elif hasattr(staging, "numel"):
        if not staging.is_cuda:
            raise ValueError("staging must be a CUDA tensor")
        sptr, nb = (staging.data_ptr() or None), staging.numel() * staging.element_size()
    else:
        raise TypeError("staging must be a device tensor or None")
    n = _numel(n, host_out)
    arr, optr = _marshal(host_slots, host_out, n, "cpu", "host_slots", "host_out")
    st = lib.arx_reduce_host(arr, len(arr), optr, n, sptr, nb, _stream(stream))
    if check:
        _check(st)
    return st


def arx_ctx_workspace_bytes(W: int, max_n: int, nblocks: int = 0) -> int:
    return int(lib.arx_ctx_workspace_bytes(W, max_n, nblocks))


def arx_ctx_init(ws, W: int, max_n: int, nblocks: int = 0, ws_bytes: int | None = None) -> arx_ctx:
    """Context for the protocol step over a zero-filled device workspace ``ws``."""
    if hasattr(ws, "is_cuda") and not ws.is_cuda:
        raise ValueError("the workspace must be a CUDA tensor")
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    ctx = arx_ctx()
    _check(lib.arx_ctx_init(ctypes.byref(ctx), _ptr(ws), ws_bytes, W, max_n, nblocks))
    ctx._ws_ref = ws  # keep the workspace alive as long as the context
    return ctx


def arx_ctx_words_bytes(W: int, nblocks: int = 0) -> int:
    return int(lib.arx_ctx_words_bytes(W, nblocks))


def arx_ctx_slots_bytes(W: int, max_n: int) -> int:
    return int(lib.arx_ctx_slots_bytes(W, max_n))


def arx_ctx_init_split(words, slots, W: int, max_n: int, nblocks: int = 0) -> arx_ctx:
    """Context with the protocol words in ``words`` (a zero-filled device tensor) and
    the slot banks in ``slots``: a device tensor, or a page-locked host tensor
    (``pin_memory()``), which the kernel then writes and reads over the CPU-GPU link."""
    if not getattr(words, "is_cuda", True):
        raise ValueError("the protocol words must be a CUDA tensor")
    where = ARX_SLOTS_DEVICE if getattr(slots, "is_cuda", True) else ARX_SLOTS_HOST
    ctx = arx_ctx()
    _check(lib.arx_ctx_init_split(ctypes.byref(ctx), _ptr(words), words.numel() * words.element_size(),
                                  _ptr(slots), slots.numel() * slots.element_size(), where, W, max_n,
                                  nblocks))
    ctx._ws_ref = (words, slots)  # keep both buffers alive as long as the context
    return ctx


def arx_ctx_set_timeout(ctx: arx_ctx, ns: int) -> None:
    _check(lib.arx_ctx_set_timeout(ctypes.byref(ctx), int(ns)))


def arx_ctx_set_sync(ctx: arx_ctx, mode: int) -> None:
    """Barrier variant of later steps: ARX_SYNC_SEMAPHORE, ARX_SYNC_PAD,
    ARX_SYNC_PAD_FENCED, ARX_SYNC_CLUSTER or ARX_SYNC_SEMAPHORE_GLOBAL."""
    _check(lib.arx_ctx_set_sync(ctypes.byref(ctx), int(mode)))


def arx_ctx_set_fault(ctx: arx_ctx, rank: int) -> None:
    _check(lib.arx_ctx_set_fault(ctypes.byref(ctx), int(rank)))


def arx_ctx_reset(ctx: arx_ctx, stream=None) -> None:
    _check(lib.arx_ctx_reset(ctypes.byref(ctx), _stream(stream)))


def arx_step(ctx: arx_ctx, inputs: Sequence, out, n: int | None = None, stream=None,
             check: bool = True) -> int:
    """Enqueue one protocol step: out = rank-order reduce of ``inputs``."""
    n = _numel(n, out)
    arr, optr = _marshal(inputs, out, n, "cuda", "inputs", "out")
    st = lib.arx_step(ctypes.byref(ctx), arr, optr, n, _stream(stream))
    if check:
        _check(st)
    return st


class arx_step_plan:
    """A prepared ``arx_step`` on one context (see ``arx_reduce_plan``): checked
    and marshalled once, one C call per step.  The context's later settings
    (sync mode, timeout, fault) apply to later calls, as it is passed by
    reference."""

    def __init__(self, ctx: arx_ctx, inputs: Sequence, out, n: int | None = None, stream=None):
        n = _numel(n, out)
        self._arr, self._out = _marshal(inputs, out, n, "cuda", "inputs", "out")
        self._refs = (ctx, list(inputs), out)
        self._ctx = ctypes.byref(ctx)
        self._n = n
        self._stream = _stream(stream)
        self._fn = lib.arx_step

    def __call__(self) -> None:
        st = self._fn(self._ctx, self._arr, self._out, self._n, self._stream)
        if st != ARX_OK:
            _check(st)


def arx_ctx_query(ctx: arx_ctx, stream=None) -> tuple[int, int, int]:
    """Synchronise ``stream``; return (status, completed seq, device error word).

    A nonzero error word is also kept in ``ctx.failed_err``: later
    ``arx_step`` calls on the context return ARX_ESTATE without launching
    until ``arx_ctx_reset``."""
    seq = ctypes.c_uint32(0)
    err = ctypes.c_uint32(0)
    st = lib.arx_ctx_query(ctypes.byref(ctx), ctypes.byref(seq), ctypes.byref(err), _stream(stream))
    return st, seq.value, err.value


def arx_watch_step(ctx: arx_ctx, target_seq: int, stall_s: float, poll_s: float = 1e-3,
                   max_wait_s: float = 10.0, host_words=None, stream=None) -> tuple[int, arx_watch_report]:
    """Block until the context's completed seq reaches ``target_seq``, a staged
    step stays not done for ``stall_s`` (a stall), or the device reports an
    error.  Polls on ``stream`` (default: a fresh non-blocking side stream),
    never on the steps' stream; ctypes releases the GIL for the call, so run
    it on a thread of your own.  Returns (status, report)."""
    import torch
    if host_words is None:
        host_words = torch.zeros(8, dtype=torch.int32).pin_memory()
    if stream is None:
        stream = torch.cuda.Stream()
    rep = arx_watch_report()
    st = lib.arx_watch_step(ctypes.byref(ctx), int(target_seq) & 0xFFFFFFFF, int(stall_s * 1e9),
                            int(poll_s * 1e9), int(max_wait_s * 1e9),
                            ctypes.cast(_ptr(host_words), ctypes.POINTER(ctypes.c_uint32)),
                            _stream(stream), ctypes.byref(rep))
    return st, rep


def arx_step_noalloc(inputs: Sequence, out, n: int | None = None, dev_status=None, stream=None,
                     check: bool = True) -> int:
    """Enqueue one protocol step whose workspace is the library's static array (no allocation).

    ``dev_status``: optional device int32/uint32 tensor (or address) that
    receives the step's device error word.  n is limited to ARX_NOALLOC_MAX_N.
    """
    n = _numel(n, out)
    arr, optr = _marshal(inputs, out, n, "cuda", "inputs", "out")
    st = lib.arx_step_noalloc(arr, len(arr), optr, n,
                              _ptr(dev_status) if dev_status is not None else None, _stream(stream))
    if check:
        _check(st)
    return st


# ---- external-writer form: a host thread writes the slots, the GPU reduces ----------

def arx_ext_region_bytes(W: int, max_n: int) -> int:
    return int(lib.arx_ext_region_bytes(W, max_n))


def arx_ext_words_bytes() -> int:
    return int(lib.arx_ext_words_bytes())


def arx_ext_init(words, region, W: int, max_n: int, nblocks: int = 0) -> arx_ext:
    """External-writer context: ``words`` a zero-filled device tensor of
    ``arx_ext_words_bytes()`` bytes, ``region`` a zero-filled page-locked host
    tensor (``pin_memory()``) of ``arx_ext_region_bytes(W, max_n)`` bytes."""
    if not getattr(words, "is_cuda", True):
        raise ValueError("the device words must be a CUDA tensor")
    if getattr(region, "is_cuda", False):
        raise ValueError("the region must be page-locked host memory")
    x = arx_ext()
    _check(lib.arx_ext_init(ctypes.byref(x), _ptr(words), words.numel() * words.element_size(),
                            _ptr(region), region.numel() * region.element_size(), W, max_n, nblocks))
    x._refs = (words, region)  # keep both buffers alive as long as the context
    return x


def arx_ext_set_timeout(x: arx_ext, ns: int) -> None:
    _check(lib.arx_ext_set_timeout(ctypes.byref(x), int(ns)))


def arx_ext_wait_free(x: arx_ext, seq: int, wait_s: float = 10.0, check: bool = True) -> int:
    st = lib.arx_ext_wait_free(ctypes.byref(x), int(seq) & 0xFFFFFFFF, int(wait_s * 1e9))
    if check:
        _check(st)
    return st


def arx_ext_slot(x: arx_ext, seq: int, rank: int) -> int:
    """Host address of recv[seq & 1][rank] (raises for bad arguments)."""
    p = lib.arx_ext_slot(ctypes.byref(x), int(seq) & 0xFFFFFFFF, int(rank))
    if not p:
        raise ArxError(ARX_EINVAL, f"no slot for rank {rank}")
    return int(p)


def arx_ext_publish(x: arx_ext, rank: int, seq: int) -> None:
    _check(lib.arx_ext_publish(ctypes.byref(x), int(rank), int(seq) & 0xFFFFFFFF))


def arx_ext_post(x: arx_ext, rank: int, seq: int, src, n: int | None = None, wait_s: float = 10.0,
                 check: bool = True) -> int:
    """Producer: wait until bank ``seq & 1`` is free, copy ``src`` (a host bf16
    tensor or address of n elements) into recv[seq & 1][rank], raise flag[rank]."""
    if n is None:
        n = int(src.numel())
    if not isinstance(src, int):
        _check_bf16([src], n, "cpu", "src")
    st = lib.arx_ext_post(ctypes.byref(x), int(rank), int(seq) & 0xFFFFFFFF, _ptr(src), n, int(wait_s * 1e9))
    if check:
        _check(st)
    return st


def arx_ext_publish_all(x: arx_ext, seq: int, wait_s: float = 10.0, check: bool = True) -> int:
    st = lib.arx_ext_publish_all(ctypes.byref(x), int(seq) & 0xFFFFFFFF, int(wait_s * 1e9))
    if check:
        _check(st)
    return st


def arx_ext_step(x: arx_ext, out, n: int | None = None, stream=None, check: bool = True) -> int:
    """Consumer: enqueue the next step, out = rank-order reduce of the posted slots."""
    n = _numel(n, out)
    if not isinstance(out, int):
        _check_bf16([out], n, "cuda", "out")
    st = lib.arx_ext_step(ctypes.byref(x), _ptr(out), n, _stream(stream))
    if check:
        _check(st)
    return st


def arx_ext_query(x: arx_ext, stream=None) -> tuple[int, int, int]:
    seq = ctypes.c_uint32(0)
    err = ctypes.c_uint32(0)
    st = lib.arx_ext_query(ctypes.byref(x), ctypes.byref(seq), ctypes.byref(err), _stream(stream))
    return st, seq.value, err.value


def arx_ext_reset(x: arx_ext, stream=None) -> None:
    _check(lib.arx_ext_reset(ctypes.byref(x), _stream(stream)))


__all__ = [
    "ArxError", "arx_ctx", "lib", "arx_status_string", "arx_last_error", "arx_reduce", "arx_reduce_plan",
    "arx_step_plan",
    "arx_reduce_host_staging_bytes", "arx_reduce_host", "arx_ctx_workspace_bytes", "arx_ctx_init",
    "arx_ctx_words_bytes", "arx_ctx_slots_bytes", "arx_ctx_init_split",
    "arx_ctx_set_timeout", "arx_ctx_set_fault", "arx_ctx_set_sync", "arx_ctx_reset", "arx_step", "arx_ctx_query",
    "arx_step_noalloc", "arx_watch_step", "arx_watch_report",
    "arx_ext", "arx_ext_region_bytes", "arx_ext_words_bytes", "arx_ext_init", "arx_ext_set_timeout",
    "arx_ext_wait_free", "arx_ext_slot", "arx_ext_publish", "arx_ext_post", "arx_ext_publish_all",
    "arx_ext_step", "arx_ext_query", "arx_ext_reset",
]
