"""Random cases through the bounds-checking build of the library.

``libarx_boundscheck.so`` is the same library built with ``ARX_BOUNDS_CHECK``:
every data access of the reduce, step and external-writer kernels (partials,
slots, output) is first checked against the buffer it belongs to; a failed check is counted
and the access skipped.  With compute-sanitizer unavailable, this stands in
for an out-of-bounds detector: random shapes, offsets, aliasing, block counts
and barrier variants must give the oracle's bits with a counter of zero.  A
probe shows the counter moves on an out-of-range address (which it never
accesses).
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic_partials as sp
from test_gpu_reduce import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked(arx):
    import importlib.util
    import os
    from conftest import ROOT
    spec = importlib.util.spec_from_file_location(
        "arx_build_check", os.path.join(ROOT, "deterministic_shot_all_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    L = ctypes.CDLL(b.build(bounds_check=True))
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    ptrs = ctypes.POINTER(ctypes.c_void_p)
    ctxp = ctypes.POINTER(arx.arx_ctx)
    for name, args, res in (
            ("arx_reduce", [ptrs, i32, vp, sz, vp], i32),
            ("arx_ctx_workspace_bytes", [i32, sz, i32], sz),
            ("arx_ctx_init", [ctxp, vp, sz, i32, sz, i32], i32),
            ("arx_ctx_words_bytes", [i32, i32], sz),
            ("arx_ctx_slots_bytes", [i32, sz], sz),
            ("arx_ctx_init_split", [ctxp, vp, sz, vp, sz, i32, i32, sz, i32], i32),
            ("arx_ctx_set_sync", [ctxp, i32], i32),
            ("arx_step", [ctxp, ptrs, vp, sz, vp], i32),
            ("arx_bounds_violations", [ctypes.POINTER(ctypes.c_uint32), i32], i32),
            ("arx_bounds_probe", [vp], i32),
            ("arx_ext_region_bytes", [i32, sz], sz),
            ("arx_ext_words_bytes", [], sz),
            ("arx_ext_init", [ctypes.POINTER(arx.arx_ext), vp, sz, vp, sz, i32, sz, i32], i32),
            ("arx_ext_post", [ctypes.POINTER(arx.arx_ext), i32, ctypes.c_uint32, vp, sz, ctypes.c_uint64], i32),
            ("arx_ext_step", [ctypes.POINTER(arx.arx_ext), vp, sz, vp], i32),
            ("arx_ext_query", [ctypes.POINTER(arx.arx_ext), ctypes.POINTER(ctypes.c_uint32),
                               ctypes.POINTER(ctypes.c_uint32), vp], i32),
            ("arx_last_error", [], ctypes.c_char_p)):
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


def _violations(L, reset=True) -> int:
    c = ctypes.c_uint32(0)
    assert L.arx_bounds_violations(ctypes.byref(c), 1 if reset else 0) == 0, L.arx_last_error()
    return c.value


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_release_build_has_no_checks(arx):
    c = ctypes.c_uint32(0)
    assert arx.lib.arx_bounds_violations(ctypes.byref(c), 0) == arx.ARX_EINVAL


def test_counter_counts_an_out_of_range_address(checked):
    dev = torch.device("cuda:0")
    _violations(checked)
    buf = torch.zeros(16, dtype=torch.uint8, device=dev)
    assert checked.arx_bounds_probe(buf.data_ptr()) == 0
    assert _violations(checked) == 1
    assert _violations(checked) == 0


def test_random_reduces_stay_in_bounds(checked):
    dev = torch.device("cuda:0")
    _violations(checked)
    rng = np.random.default_rng(5150)
    sizes = [(1 << 22) - 3, (1 << 22) + 9, (1 << 23) + 5, (1 << 21) + 5, 1_400_003]
    for case in range(120):
        W = int(rng.integers(1, 9))
        if case % 10 == 0:
            n = sizes[(case // 10) % 5]
            W = 1 + (case // 10) % 4 if n == (1 << 21) + 5 else W  # the batched 8-byte form
            W = 8 if n == 1_400_003 else W  # the pipelined 16-byte form past one 8-byte pass
        else:
            n = int(rng.integers(0, 5000))
        same = bool(rng.integers(0, 2))
        offs = [int(rng.integers(0, 8))] * (W + 1) if same else [int(v) for v in rng.integers(0, 8, W + 1)]
        alias = int(rng.integers(-1, W)) if n else -1
        x = sp.partials(W, n, "special" if n < 10000 else "normal", seed=30_000 + case)
        buf = torch.zeros(W + 1, n + 16, dtype=torch.int16, device=dev)
        for r in range(W):
            buf[r, offs[r]:offs[r] + n] = x[r].view(torch.int16).to(dev)
        slots = [buf[r, offs[r]:offs[r] + n] for r in range(W)]
        out = slots[alias] if alias >= 0 else buf[W, offs[W]:offs[W] + n]
        arr = (ctypes.c_void_p * W)(*[t.data_ptr() for t in slots])
        assert checked.arx_reduce(arr, W, out.data_ptr(), n, _stream()) == 0, checked.arx_last_error()
        torch.cuda.synchronize()
        if n:
            want = oracle.reduce(list(sp.to_u16_numpy(x)), threads=oracle.default_threads())
            assert_bits_equal(out.cpu().numpy().view(np.uint16), want,
                              f"case {case}: W={W} n={n} offs={offs} alias={alias}")
    assert _violations(checked) == 0


def test_random_steps_stay_in_bounds(checked, arx):
    dev = torch.device("cuda:0")
    _violations(checked)
    rng = np.random.default_rng(6160)
    for case in range(30):
        W = int(rng.integers(1, 9))
        n = int(rng.integers(1, 40000)) if case % 6 else 1 << 20
        B = int(rng.integers(0, 8))
        mode = int(rng.integers(0, 5))   # every barrier variant, the cluster ones included
        in_off, out_off = int(rng.integers(0, 8)), int(rng.integers(0, 8))
        ctx = arx.arx_ctx()
        if case % 12 == 0:
            # Slots in page-locked host memory, 2 MiB partials: the steps stage
            # in turn (the staggered kernels), in the default mode, the
            # cluster mode and a random one.
            mode = {0: 0, 12: 3}.get(case, mode)
            B = max(B, 2)
            ws = torch.zeros(checked.arx_ctx_words_bytes(W, B), dtype=torch.uint8, device=dev)
            slots = torch.empty(checked.arx_ctx_slots_bytes(W, n), dtype=torch.uint8).pin_memory()
            assert checked.arx_ctx_init_split(ctypes.byref(ctx), ws.data_ptr(), ws.numel(), slots.data_ptr(),
                                              slots.numel(), arx.ARX_SLOTS_HOST, W, n, B) == 0, \
                checked.arx_last_error()
        else:
            ws = torch.zeros(checked.arx_ctx_workspace_bytes(W, n, B), dtype=torch.uint8, device=dev)
            assert checked.arx_ctx_init(ctypes.byref(ctx), ws.data_ptr(), ws.numel(), W, n, B) == 0
        assert checked.arx_ctx_set_sync(ctypes.byref(ctx), mode) == 0
        for s in range(2):
            x = sp.partials(W, n, "normal", seed=40_000 + 2 * case + s)
            buf = torch.zeros(W, n + 16, dtype=torch.int16, device=dev)
            buf[:, in_off:in_off + n] = x.view(torch.int16).to(dev)
            ins = (ctypes.c_void_p * W)(*[buf[r, in_off:in_off + n].data_ptr() for r in range(W)])
            ob = torch.zeros(n + 16, dtype=torch.int16, device=dev)
            out = ob[out_off:out_off + n]
            assert checked.arx_step(ctypes.byref(ctx), ins, out.data_ptr(), n, _stream()) == 0
            torch.cuda.synchronize()
            want = oracle.reduce(list(sp.to_u16_numpy(x)), threads=oracle.default_threads())
            assert_bits_equal(out.cpu().numpy().view(np.uint16), want,
                              f"case {case} step {s}: W={W} n={n} B={ctx.nblocks} mode={mode}")
        words = ws[:8].cpu().numpy().view(np.uint32)
        assert words[0] == 2 and words[1] == 0, f"case {case}: seq {words[0]} err {words[1]:#x}"
    assert _violations(checked) == 0


def test_random_external_writer_steps_stay_in_bounds(checked, arx):
    # The external-writer kernel through the checking build: random W, ragged
    # n (slots of a larger max_n) and output offsets, two steps each (both
    # banks), outputs against the oracle and no access outside its buffer.
    dev = torch.device("cuda:0")
    _violations(checked)
    rng = np.random.default_rng(7171)
    for case in range(20):
        W = int(rng.integers(1, 9))
        max_n = int(rng.integers(1, 70000))
        n = int(rng.integers(1, max_n + 1))
        off = int(rng.integers(0, 8))
        words = torch.zeros(checked.arx_ext_words_bytes(), dtype=torch.uint8, device=dev)
        region = torch.zeros(checked.arx_ext_region_bytes(W, max_n), dtype=torch.uint8).pin_memory()
        x = arx.arx_ext()
        assert checked.arx_ext_init(ctypes.byref(x), words.data_ptr(), words.numel(), region.data_ptr(),
                                    region.numel(), W, max_n, 0) == 0, checked.arx_last_error()
        ob = torch.zeros(n + 16, dtype=torch.int16, device=dev)
        out = ob[off:off + n]
        for s in (1, 2):
            p = sp.partials(W, n, "special", seed=71_000 + 2 * case + s)
            for r in range(W):
                assert checked.arx_ext_post(ctypes.byref(x), r, s, p[r].data_ptr(), n, 10**9) == 0
            assert checked.arx_ext_step(ctypes.byref(x), out.data_ptr(), n, _stream()) == 0
            seq, err = ctypes.c_uint32(0), ctypes.c_uint32(0)
            assert checked.arx_ext_query(ctypes.byref(x), ctypes.byref(seq), ctypes.byref(err), _stream()) == 0
            assert (seq.value, err.value) == (s, 0)
            assert_bits_equal(out.cpu().numpy().view(np.uint16), oracle.reduce(list(sp.to_u16_numpy(p))),
                              f"case {case} step {s}: W={W} n={n} max_n={max_n} off={off}")
    assert _violations(checked) == 0
