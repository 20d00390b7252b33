"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* the library loads and exports every function ``include/arx.h`` declares;
* argument validation returns the documented status before touching CUDA;
* the protocol context's workspace layout is consistent.

Addresses used here are fabricated integers: every call below is rejected (or
needs no device) before anything could dereference them.
"""

import ctypes
import os
import re

import pytest

from conftest import ROOT, gpu_available

HEADER = os.path.join(ROOT, "include", "arx.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(arx_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for must in ("arx_reduce", "arx_step", "arx_ctx_init", "arx_ctx_query",
                 "arx_ctx_workspace_bytes", "arx_status_string", "arx_ext_step", "arx_ext_post",
                 "arx_step_noalloc"):
        assert must in names


def test_library_exports_every_declared_symbol(product_lib_path):
    lib = ctypes.CDLL(product_lib_path)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in arx.h but not exported: {missing}"


def test_status_strings(arx):
    for code in range(6):
        assert arx.arx_status_string(code).startswith("ARX_")
    assert "unknown" in arx.arx_status_string(99)


FAKE = 1 << 40  # 16-byte aligned fabricated address


def _reduce(arx, slots, W, out, n):
    arr = (ctypes.c_void_p * max(1, len(slots)))(*slots) if slots else None
    return arx.lib.arx_reduce(arr, W, out, n, None)


def test_reduce_n0_is_a_no_op_even_with_null_pointers(arx):
    assert arx.lib.arx_reduce(None, 0, None, 0, None) == arx.ARX_OK


@pytest.mark.parametrize("W", [0, -1, 9, 100])
def test_reduce_rejects_w_out_of_range(arx, W):
    slots = [FAKE + 4096 * i for i in range(max(W, 1))][:8]
    assert _reduce(arx, slots, W, FAKE + (1 << 30), 16) == arx.ARX_EINVAL


def test_reduce_rejects_null_and_misaligned_pointers(arx):
    out = FAKE + (1 << 30)
    assert _reduce(arx, [FAKE, 0], 2, out, 16) == arx.ARX_EINVAL
    assert _reduce(arx, [FAKE, FAKE + 4096], 2, 0, 16) == arx.ARX_EINVAL
    assert _reduce(arx, [FAKE + 1, FAKE + 4096], 2, out, 16) == arx.ARX_EINVAL
    assert _reduce(arx, [FAKE, FAKE + 4096], 2, out + 1, 16) == arx.ARX_EINVAL
    assert "aligned" in arx.arx_last_error()


def test_reduce_rejects_partial_overlap(arx):
    n = 1024
    a, b = FAKE, FAKE + 4 * n
    assert _reduce(arx, [a, b], 2, a + 2, n) == arx.ARX_EOVERLAP   # shifted by one element
    assert _reduce(arx, [a, b], 2, b - 2 * n + 2, n) == arx.ARX_EOVERLAP
    assert "overlap" in arx.arx_last_error()


@pytest.mark.skipif(gpu_available(), reason="checks the no-device error path")
def test_reduce_without_a_device_reports_cuda_error(arx):
    n = 1024
    st = _reduce(arx, [FAKE, FAKE + 4 * n], 2, FAKE, n)  # exact alias: valid arguments
    assert st == arx.ARX_ECUDA
    assert arx.arx_last_error()


def test_staging_bytes(arx):
    assert arx.arx_reduce_host_staging_bytes(8, 131072) == 8 * 262144
    assert arx.arx_reduce_host_staging_bytes(3, 5) == 3 * 256
    assert arx.arx_reduce_host_staging_bytes(0, 5) == 0
    assert arx.arx_reduce_host_staging_bytes(9, 5) == 0


def test_workspace_layout(arx):
    W, n, B = 8, 131072, 19
    nbytes = arx.arx_ctx_workspace_bytes(W, n, B)
    assert nbytes > 2 * W * n * 2
    assert arx.arx_ctx_workspace_bytes(W, n, 0) >= nbytes  # sized for the block maximum
    assert arx.arx_ctx_workspace_bytes(0, n, B) == 0
    assert arx.arx_ctx_workspace_bytes(W, n, arx.ARX_STEP_MAX_BLOCKS + 1) == 0
    ctx = arx.arx_ctx()
    st = arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, nbytes, W, n, B)
    assert st == arx.ARX_OK
    assert ctx.W == W and ctx.nblocks == B and ctx.fault_rank == -1
    assert ctx.timeout_ns == arx.ARX_DEFAULT_TIMEOUT_NS
    assert ctx.off_epoch >= 20                                 # after the header words
    assert ctx.off_sem >= ctx.off_epoch + W * B * 4 and ctx.off_sem % 128 == 0
    assert ctx.off_pad >= ctx.off_sem + W * B * 128
    assert ctx.off_slots >= ctx.off_pad + W * B * W * 4 and ctx.off_slots % 256 == 0
    assert ctx.slot_stride >= n and ctx.slot_stride % 128 == 0
    assert ctx.ctrl_bytes == ctx.off_slots
    assert ctx.off_slots + 2 * W * ctx.slot_stride * 2 == nbytes


def test_ctx_init_rejections(arx):
    ctx = arx.arx_ctx()
    nbytes = arx.arx_ctx_workspace_bytes(4, 1000, 4)
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE + 16, nbytes, 4, 1000, 4) == arx.ARX_EINVAL
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, nbytes - 1, 4, 1000, 4) == arx.ARX_EINVAL
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), 0, nbytes, 4, 1000, 4) == arx.ARX_EINVAL
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, nbytes, 9, 1000, 4) == arx.ARX_EINVAL
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, nbytes, 4, 1000, -1) == arx.ARX_EINVAL


def test_ctx_knobs_and_step_validation(arx):
    W, n, B = 4, 4096, 2
    nbytes = arx.arx_ctx_workspace_bytes(W, n, B)
    ctx = arx.arx_ctx()
    # An uninitialised context is refused.
    assert arx.lib.arx_step(ctypes.byref(ctx), None, FAKE, 16, None) == arx.ARX_ESTATE
    assert arx.lib.arx_ctx_set_timeout(ctypes.byref(ctx), 5) == arx.ARX_ESTATE
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, nbytes, W, n, B) == arx.ARX_OK
    assert arx.lib.arx_ctx_set_timeout(ctypes.byref(ctx), 0) == arx.ARX_EINVAL
    assert arx.lib.arx_ctx_set_timeout(ctypes.byref(ctx), 12345) == arx.ARX_OK
    assert ctx.timeout_ns == 12345
    assert arx.lib.arx_ctx_set_fault(ctypes.byref(ctx), W) == arx.ARX_EINVAL
    assert arx.lib.arx_ctx_set_fault(ctypes.byref(ctx), -2) == arx.ARX_EINVAL
    assert arx.lib.arx_ctx_set_fault(ctypes.byref(ctx), 1) == arx.ARX_OK and ctx.fault_rank == 1
    assert arx.lib.arx_ctx_set_fault(ctypes.byref(ctx), -1) == arx.ARX_OK
    ins = (ctypes.c_void_p * W)(*[FAKE + (1 << 32) + i * (1 << 20) for i in range(W)])
    # n == 0: nothing to do.
    assert arx.lib.arx_step(ctypes.byref(ctx), ins, FAKE + (1 << 34), 0, None) == arx.ARX_OK
    # n beyond the slot capacity.
    assert arx.lib.arx_step(ctypes.byref(ctx), ins, FAKE + (1 << 34), n + 1, None) == arx.ARX_EINVAL
    # Output inside the workspace.
    assert arx.lib.arx_step(ctypes.byref(ctx), ins, FAKE + 256, n, None) == arx.ARX_EOVERLAP
    # Output partially overlapping an input.
    assert arx.lib.arx_step(ctypes.byref(ctx), ins, ins[1] + 2, n, None) == arx.ARX_EOVERLAP
    # Null input.
    bad = (ctypes.c_void_p * W)(*([0] + list(ins[1:])))
    assert arx.lib.arx_step(ctypes.byref(ctx), bad, FAKE + (1 << 34), n, None) == arx.ARX_EINVAL


def test_failed_context_refuses_to_launch(arx):
    # The pages check an error flag before every launch; here the flag is the
    # device error word arx_ctx_query last read, kept in the host struct.
    # arx_step must refuse before any CUDA call (none can run on this host).
    W, n, B = 4, 4096, 2
    ctx = arx.arx_ctx()
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, arx.arx_ctx_workspace_bytes(W, n, B), W, n, B) == 0
    assert ctx.failed_err == 0
    ins = (ctypes.c_void_p * W)(*[FAKE + (1 << 32) + i * (1 << 20) for i in range(W)])
    ctx.failed_err = 0x00120204  # ETIMEOUT at the end wait, rank 2, block 18
    assert arx.lib.arx_step(ctypes.byref(ctx), ins, FAKE + (1 << 34), n, None) == arx.ARX_ESTATE
    assert "0x00120204" in arx.arx_last_error() and "arx_ctx_reset" in arx.arx_last_error()
    with pytest.raises(arx.ArxError):
        arx.arx_step(ctx, [FAKE + (1 << 32) + i * (1 << 20) for i in range(W)], FAKE + (1 << 34), n, stream=0)
    # Even an empty step is refused, and re-initialising clears the flag.
    assert arx.lib.arx_step(ctypes.byref(ctx), ins, FAKE + (1 << 34), 0, None) == arx.ARX_ESTATE
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, arx.arx_ctx_workspace_bytes(W, n, B), W, n, B) == 0
    assert ctx.failed_err == 0


def test_split_layout_and_rejections(arx):
    W, n, B = 8, 131072, 19
    words = arx.arx_ctx_words_bytes(W, B)
    slots = arx.arx_ctx_slots_bytes(W, n)
    assert words + slots == arx.arx_ctx_workspace_bytes(W, n, B)
    assert arx.arx_ctx_words_bytes(W, 0) >= words and arx.arx_ctx_words_bytes(0, B) == 0
    assert arx.arx_ctx_slots_bytes(9, n) == 0
    ctx = arx.arx_ctx()
    S = FAKE + (1 << 32)
    init = arx.lib.arx_ctx_init_split
    assert init(ctypes.byref(ctx), FAKE, words, S, slots, arx.ARX_SLOTS_DEVICE, W, n, B) == arx.ARX_OK
    assert ctx.slots == S and ctx.slots_bytes == slots and ctx.ctrl_bytes == words
    assert ctx.slots_where == arx.ARX_SLOTS_DEVICE and ctx.ws == FAKE
    assert init(ctypes.byref(ctx), FAKE, words - 1, S, slots, 0, W, n, B) == arx.ARX_EINVAL
    assert init(ctypes.byref(ctx), FAKE, words, S, slots - 1, 0, W, n, B) == arx.ARX_EINVAL
    assert init(ctypes.byref(ctx), FAKE, words, S + 16, slots, 0, W, n, B) == arx.ARX_EINVAL
    assert init(ctypes.byref(ctx), FAKE, words, 0, slots, 0, W, n, B) == arx.ARX_EINVAL
    assert init(ctypes.byref(ctx), FAKE, words, FAKE + 256, slots, 0, W, n, B) == arx.ARX_EOVERLAP
    assert init(ctypes.byref(ctx), FAKE, words, S, slots, 2, W, n, B) == arx.ARX_EINVAL
    # The single-buffer form places the slots right after the words.
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, words + slots, W, n, B) == arx.ARX_OK
    assert ctx.slots == FAKE + ctx.off_slots and ctx.slots_bytes == slots


def test_step_rejects_inputs_overlapping_the_slots(arx):
    W, n, B = 2, 4096, 2
    words, slots = arx.arx_ctx_words_bytes(W, B), arx.arx_ctx_slots_bytes(W, n)
    ctx = arx.arx_ctx()
    S = FAKE + (1 << 32)
    assert arx.lib.arx_ctx_init_split(ctypes.byref(ctx), FAKE, words, S, slots, 0, W, n, B) == arx.ARX_OK
    out = FAKE + (1 << 34)
    ok_in = (ctypes.c_void_p * W)(FAKE + (1 << 35), FAKE + (1 << 35) + (1 << 20))
    in_slots = (ctypes.c_void_p * W)(S + 512, FAKE + (1 << 35))
    assert arx.lib.arx_step(ctypes.byref(ctx), in_slots, out, n, None) == arx.ARX_EOVERLAP
    assert arx.lib.arx_step(ctypes.byref(ctx), ok_in, S, n, None) == arx.ARX_EOVERLAP
    assert "slots" in arx.arx_last_error()


def test_binding_rejects_tensors_of_the_wrong_kind(arx):
    # Checked in the binding before any pointer reaches the library.
    import torch
    x = torch.zeros(2, 64, dtype=torch.bfloat16)              # host tensors
    with pytest.raises(ValueError, match="CUDA tensor"):
        arx.arx_reduce([x[0], x[1]], x[0])
    f = torch.zeros(2, 64, dtype=torch.float32)
    with pytest.raises(TypeError, match="bfloat16"):
        arx.arx_reduce([f[0], f[1]], f[0])
    t = torch.zeros(64, 2, dtype=torch.bfloat16).t()          # non-contiguous rows
    with pytest.raises(ValueError, match="contiguous"):
        arx.arx_reduce([t[0], t[1]], x[0])
    with pytest.raises(ValueError, match="elements"):
        arx.arx_reduce([x[0][:10], x[1]], x[0])
    ws = torch.zeros(arx.arx_ctx_workspace_bytes(2, 64, 1), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        arx.arx_ctx_init(ws, 2, 64, 1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        arx.arx_step_noalloc([x[0], x[1]], x[0])
    with pytest.raises(TypeError, match="bfloat16"):
        arx.arx_reduce_host([f[0], f[1]], f[0])


def test_watchdog_argument_checks(arx):
    ctx = arx.arx_ctx()
    words = (ctypes.c_uint32 * 8)()
    rep = arx.arx_watch_report()
    w = arx.lib.arx_watch_step
    assert w(ctypes.byref(ctx), 1, 10**6, 10**5, 10**9, words, None, ctypes.byref(rep)) == arx.ARX_ESTATE
    n = arx.arx_ctx_workspace_bytes(2, 64, 1)
    assert arx.lib.arx_ctx_init(ctypes.byref(ctx), FAKE, n, 2, 64, 1) == arx.ARX_OK
    assert w(ctypes.byref(ctx), 1, 10**6, 10**5, 10**9, None, None, ctypes.byref(rep)) == arx.ARX_EINVAL
    assert w(ctypes.byref(ctx), 1, 0, 10**5, 10**9, words, None, ctypes.byref(rep)) == arx.ARX_EINVAL
    assert w(ctypes.byref(ctx), 1, 10**6, 0, 10**9, words, None, ctypes.byref(rep)) == arx.ARX_EINVAL
    assert w(ctypes.byref(ctx), 1, 10**6, 10**5, 0, words, None, None) == arx.ARX_EINVAL


def test_plan_checks_its_arguments_once(arx):
    import torch
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        arx.arx_reduce_plan([x[0], x[1]], x[0])


def test_external_writer_layout_and_rejections(arx):
    # Sizes: 1 KiB of control words, then two banks of W slots of max_n
    # elements rounded up to 128 (the header's layout).
    W, n = 8, 131072
    assert arx.arx_ext_region_bytes(W, n) == 1024 + 2 * W * n * 2
    assert arx.arx_ext_region_bytes(3, 100) == 1024 + 2 * 3 * 128 * 2
    assert arx.arx_ext_region_bytes(0, n) == 0 and arx.arx_ext_region_bytes(9, n) == 0
    assert arx.arx_ext_words_bytes() == 256
    x = arx.arx_ext()
    init = arx.lib.arx_ext_init
    region = (ctypes.c_uint8 * (arx.arx_ext_region_bytes(2, 64) + 256))()
    R = (ctypes.addressof(region) + 255) // 256 * 256
    rb = arx.arx_ext_region_bytes(2, 64)
    assert init(ctypes.byref(x), FAKE, 256, R, rb, 0, 64, 1) == arx.ARX_EINVAL           # W
    assert init(ctypes.byref(x), FAKE + 16, 256, R, rb, 2, 64, 1) == arx.ARX_EINVAL      # alignment
    assert init(ctypes.byref(x), FAKE, 255, R, rb, 2, 64, 1) == arx.ARX_EINVAL           # words too small
    assert init(ctypes.byref(x), FAKE, 256, R, rb - 1, 2, 64, 1) == arx.ARX_EINVAL       # region too small
    assert init(ctypes.byref(x), FAKE, 256, 0, rb, 2, 64, 1) == arx.ARX_EINVAL           # no region
    # Ordinary (pageable) host memory is not a region the GPU can read.
    assert init(ctypes.byref(x), FAKE, 256, R, rb, 2, 64, 1) == arx.ARX_EINVAL
    assert "page-locked" in arx.arx_last_error()
    # An uninitialised context is refused by every call.
    y = arx.arx_ext()
    assert arx.lib.arx_ext_step(ctypes.byref(y), FAKE, 64, None) == arx.ARX_ESTATE
    assert arx.lib.arx_ext_post(ctypes.byref(y), 0, 1, R, 64, 10**6) == arx.ARX_ESTATE
    assert arx.lib.arx_ext_publish(ctypes.byref(y), 0, 1) == arx.ARX_ESTATE
    assert arx.lib.arx_ext_publish_all(ctypes.byref(y), 1, 10**6) == arx.ARX_ESTATE
    assert arx.lib.arx_ext_wait_free(ctypes.byref(y), 1, 10**6) == arx.ARX_ESTATE
    assert arx.lib.arx_ext_slot(ctypes.byref(y), 1, 0) is None
    assert arx.lib.arx_ext_set_timeout(ctypes.byref(y), 5) == arx.ARX_ESTATE
