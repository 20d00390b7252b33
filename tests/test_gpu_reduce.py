"""GPU parity of the stateless reduce (``arx_reduce``) against the CPU oracle.

Bar: bit-exact (integer comparison of the bf16 patterns) on every element;
NaN outputs compare by NaN-ness only (the payload is unpinned, as the oracle
header states).  Every call goes through the C ABI via the binding.

Covers the workloads the one-shot all-reduce targets -- W = 2, 4, 8 partials
of bf16 [32, 4096] and [1024, 8192] (arx.cu, ``kMaxBytes`` comment, widened),
the in-place form (arx.cu: "in and out may alias"), the power-of-two size
sweep from 1 KiB to 256 MiB per partial -- plus ragged sizes, every W,
misaligned pointers, hard floating-point patterns and guard bytes.
"""

import numpy as np
import pytest
import torch

import oracle
import synthetic_partials as sp

pytestmark = pytest.mark.gpu

GUARD = 64
SENTINEL = 0x7E57


def _is_nan16(b):
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = got.view(np.uint16)
    want = want.view(np.uint16)
    assert got.shape == want.shape
    nan_w = _is_nan16(want)
    same = (got == want) | (nan_w & _is_nan16(got))
    if not same.all():
        bad = np.flatnonzero(~same)
        i = int(bad[0])
        pytest.fail(f"{what}: {bad.size} of {got.size} elements differ; first at {i}: "
                    f"gpu {int(got[i]):#06x} oracle {int(want[i]):#06x}")


@pytest.fixture(scope="module")
def dev(arx):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return torch.device("cuda:0")


def _run(arx, dev, x: torch.Tensor, alias: bool = False) -> np.ndarray:
    """Reduce the [W, n] CPU bf16 partials on the GPU; returns the output patterns."""
    W, n = x.shape
    xd = x.to(dev)
    slots = [xd[r] for r in range(W)]
    if alias:
        out = slots[0]
    else:
        buf = torch.full((n + 2 * GUARD,), 0, dtype=torch.int16, device=dev)
        buf.fill_(SENTINEL)
        out = buf[GUARD:GUARD + n].view(torch.bfloat16)
    arx.arx_reduce(slots, out)
    torch.cuda.synchronize()
    if not alias:
        g = buf.cpu().numpy().view(np.uint16)
        assert (g[:GUARD] == SENTINEL).all() and (g[GUARD + n:] == SENTINEL).all(), "guard bytes written"
    for r in range(1 if alias else 0, W):  # inputs other than the aliased slot are untouched
        assert torch.equal(xd[r].cpu().view(torch.int16), x[r].view(torch.int16))
    return out.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["w2_32x4096_uniform", "w8_32x4096_normal"])
def test_decode_sized_workloads(arx, dev, name):
    x, alias = sp.workload(name)
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    assert_bits_equal(_run(arx, dev, x, alias), want, name)


def test_in_place_1024x8192_w4(arx, dev):
    x, alias = sp.workload("w4_1024x8192_alias")
    assert alias
    want = oracle.reduce(list(sp.to_u16_numpy(x)), threads=oracle.default_threads())
    got = _run(arx, dev, x, alias=True)   # first call on a pristine copy
    assert_bits_equal(got, want, "w4 [1024,8192] in place")


@pytest.mark.parametrize("k", list(sp.SWEEP_LOG2))
def test_size_sweep_integer_partials(arx, dev, k):
    n = 1 << k
    x, _ = sp.workload("w8_sweep_int", n=n)
    want = oracle.reduce(list(sp.to_u16_numpy(x)), threads=oracle.default_threads())
    got = _run(arx, dev, x)
    assert_bits_equal(got, want, f"sweep n=2^{k}")
    # Integer partials in [-8, 8]: the sum is exact, check it against integers too.
    if k <= 20:
        exact = x.to(torch.int64).sum(0).to(torch.float32).to(torch.bfloat16)
        assert_bits_equal(got, sp.to_u16_numpy(exact), "exact integer sum")


@pytest.mark.parametrize("W", range(1, 9))
def test_every_w_with_hard_patterns(arx, dev, W):
    # Random bit patterns: subnormals, infinities, NaN, signed zeros, ties.
    for n in (1, 7, 8, 9, 255, 4099, 70001):
        x = sp.partials(W, n, "special", seed=1000 * W + n)
        want = oracle.reduce(list(sp.to_u16_numpy(x)))
        assert_bits_equal(_run(arx, dev, x), want, f"W={W} n={n}")


@pytest.mark.parametrize("W", [1, 2, 3, 8])
def test_in_place_small_and_ragged(arx, dev, W):
    for n in (1, 5, 8, 13, 1000, 65537):
        x = sp.partials(W, n, "normal", seed=77 + n)
        want = oracle.reduce(list(sp.to_u16_numpy(x)))
        assert_bits_equal(_run(arx, dev, x, alias=True), want, f"alias W={W} n={n}")


@pytest.mark.parametrize("W", [1, 3, 8])
@pytest.mark.parametrize("n", [(1 << 22) - 3, (1 << 22) + 9])
def test_both_vector_forms_ragged_misaligned_in_place(arx, dev, W, n):
    # Sizes just below and above the switch from 8-byte to 16-byte vectors,
    # with a scalar head (every pointer 2 bytes past a 16-byte boundary), a
    # ragged tail, and the output aliasing the last slot.
    x = sp.partials(W, n, "normal", seed=n % 1000 + W)
    want = oracle.reduce(list(sp.to_u16_numpy(x)), threads=oracle.default_threads())
    buf = torch.zeros(W, n + 16, dtype=torch.bfloat16, device=dev)
    buf[:, 1:1 + n] = x.to(dev)
    slots = [buf[r, 1:1 + n] for r in range(W)]
    arx.arx_reduce(slots, slots[W - 1])
    torch.cuda.synchronize()
    assert_bits_equal(slots[W - 1].cpu().view(torch.int16).numpy(), want, f"W={W} n={n} in place")
    assert not buf[W - 1, 0].view(torch.int16).item() and not buf[W - 1, 1 + n:].view(torch.int16).any()


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("n", [1_250_003, (1 << 21) + 5, 3_000_017, (1 << 22) - 1])
@pytest.mark.parametrize("alias", [False, True])
def test_batched_8_byte_form(arx, dev, W, n, alias):
    # For W <= 4, sizes one pass of the one-vector grid does not cover take
    # the batched 8-byte form (8 / W vectors per slot per thread, then twice
    # that for W = 2, 3) while one pass of it does, else the 16-byte form.
    # On 152 SMs: 1,250,003 elements sit just above one one-vector pass;
    # 3,000,017 take the deeper tier at W = 3; 2^22 - 1 takes it at W = 2
    # and the 16-byte form at W = 3, 4.  Scalar head (pointers 2 bytes past
    # a 16-byte boundary), ragged tail, in place or not; guard elements intact.
    x = sp.partials(W, n, "normal", seed=n % 997 + 10 * W + alias)
    want = oracle.reduce(list(sp.to_u16_numpy(x)), threads=oracle.default_threads())
    buf = torch.zeros(W + 1, n + 16, dtype=torch.bfloat16, device=dev)
    buf[:W, 1:1 + n] = x.to(dev)
    slots = [buf[r, 1:1 + n] for r in range(W)]
    row = 0 if alias else W
    arx.arx_reduce(slots, buf[row, 1:1 + n])
    torch.cuda.synchronize()
    assert_bits_equal(buf[row, 1:1 + n].cpu().view(torch.int16).numpy(), want, f"W={W} n={n} alias={alias}")
    assert not buf[row, 0].view(torch.int16).item() and not buf[row, 1 + n:].view(torch.int16).any()


@pytest.mark.parametrize("W", [5, 7, 8])
@pytest.mark.parametrize("n", [1_250_003, 1_400_003, (1 << 21) + 5, (1 << 22) - 1, (1 << 22) + 9, 9_000_011])
@pytest.mark.parametrize("alias", [False, True])
def test_pipelined_16_byte_form(arx, dev, W, n, alias):
    # W = 8 takes the pipelined 16-byte form (one group per slot per thread,
    # the next group's loads in flight while the current one is summed) once
    # one pass of the one-vector 8-byte grid no longer covers the body (with
    # 1/16 slack: on 152 SMs 1,250,003 elements stay in the 8-byte form,
    # 1,400,003 leave it); W = 5-7 keep the 8-byte form, with a second pass,
    # up to 2^22; above 2^22 every W >= 5 takes the pipelined form, several
    # passes of it at 9,000,011.  Scalar head (pointers 2 bytes past a
    # 16-byte boundary), ragged tail, in place or not; guard elements intact.
    x = sp.partials(W, n, "normal", seed=n % 991 + 10 * W + alias)
    want = oracle.reduce(list(sp.to_u16_numpy(x)), threads=oracle.default_threads())
    buf = torch.zeros(W + 1, n + 16, dtype=torch.bfloat16, device=dev)
    buf[:W, 1:1 + n] = x.to(dev)
    slots = [buf[r, 1:1 + n] for r in range(W)]
    row = W - 1 if alias else W
    arx.arx_reduce(slots, buf[row, 1:1 + n])
    torch.cuda.synchronize()
    assert_bits_equal(buf[row, 1:1 + n].cpu().view(torch.int16).numpy(), want, f"W={W} n={n} alias={alias}")
    assert not buf[row, 0].view(torch.int16).item() and not buf[row, 1 + n:].view(torch.int16).any()


def test_alias_to_last_slot(arx, dev):
    x = sp.partials(5, 40000, "normal", seed=9)
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    xd = x.to(dev)
    slots = [xd[r] for r in range(5)]
    arx.arx_reduce(slots, slots[4])
    torch.cuda.synchronize()
    assert_bits_equal(xd[4].cpu().view(torch.int16).numpy(), want, "alias slot 4")


@pytest.mark.parametrize("offsets", [
    (1, 1, 1),          # same misalignment: vector path with a scalar head
    (3, 3, 3),
    (7, 7, 7),
    (0, 1, 0),          # mixed: scalar path
    (2, 5, 1),
    (0, 0, 4),          # output misaligned only
])
def test_misaligned_pointers(arx, dev, offsets):
    W, n = 2, 10007
    x = sp.partials(W, n, "uniform", seed=sum(offsets))
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    bufs = []
    slots = []
    for r in range(W):
        b = torch.zeros(n + 16, dtype=torch.bfloat16, device=dev)
        b[offsets[r]:offsets[r] + n] = x[r].to(dev)
        bufs.append(b)
        slots.append(b[offsets[r]:offsets[r] + n])
    ob = torch.full((n + 16 + 2 * GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    o0 = GUARD + offsets[2]
    out = ob[o0:o0 + n].view(torch.bfloat16)
    arx.arx_reduce(slots, out)
    torch.cuda.synchronize()
    g = ob.cpu().numpy().view(np.uint16)
    assert (g[:o0] == SENTINEL).all() and (g[o0 + n:] == SENTINEL).all()
    assert_bits_equal(g[o0:o0 + n], want, f"offsets {offsets}")


def test_w1_identity_and_negative_zero(arx, dev):
    x = sp.partials(1, 100003, "special", seed=4)
    got = _run(arx, dev, x)
    u = sp.to_u16_numpy(x)[0]
    nan = _is_nan16(u)
    want = np.where(u == 0x8000, np.uint16(0), u)
    assert np.array_equal(_is_nan16(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    nz = torch.full((3, 4096), -0.0, dtype=torch.bfloat16)
    assert not _run(arx, dev, nz).any(), "(-0) + (-0) + (-0) from +0 must be +0"


def test_subnormals_are_not_flushed(arx, dev):
    tiny = torch.from_numpy(np.array([0x0001, 0x0003, 0x007F, 0x8001], dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    x = torch.stack([tiny, tiny])
    got = _run(arx, dev, x)
    assert list(got) == [0x0002, 0x0006, 0x00FE, 0x8002]


def test_repeated_slot_pointer(arx, dev):
    x = sp.partials(1, 5000, "normal", seed=3)
    xd = x.to(dev)
    out = torch.empty(5000, dtype=torch.bfloat16, device=dev)
    arx.arx_reduce([xd[0]] * 3, out)
    torch.cuda.synchronize()
    u = sp.to_u16_numpy(x)[0]
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce([u, u, u]), "slot repeated")


def test_partial_overlap_is_rejected_on_device_buffers(arx, dev):
    x = torch.zeros(2, 1024, dtype=torch.bfloat16, device=dev)
    st = arx.arx_reduce([x[0], x[1]], x.view(-1)[1:1025], check=False)
    assert st == arx.ARX_EOVERLAP


def test_zero_length_launches_nothing(arx, dev):
    x = torch.zeros(2, 0, dtype=torch.bfloat16, device=dev)
    assert arx.arx_reduce([x[0], x[1]], x[0], n=0, check=False) == arx.ARX_OK


def test_nondefault_stream_and_graph_capture(arx, dev):
    x, _ = sp.workload("w8_32x4096_normal")
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    xd = x.to(dev)
    slots = [xd[r] for r in range(8)]
    outs = torch.zeros(16, x.shape[1], dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        arx.arx_reduce(slots, outs[0], stream=s)       # warm the launch caches off-capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        for i in range(16):
            arx.arx_reduce(slots, outs[i], stream=s)
    outs.zero_()
    g.replay()
    torch.cuda.synchronize()
    for i in range(16):
        assert_bits_equal(outs[i].cpu().view(torch.int16).numpy(), want, f"graph call {i}")


def test_host_buffer_form_pinned_direct(arx, dev):
    # Page-locked buffers: the kernel reads and writes host memory directly.
    W, n = 8, 131072 + 3
    x = sp.partials(W, n, "normal", seed=21)
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    host = [x[r].clone().pin_memory() for r in range(W)]
    hout = torch.empty(n, dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        hout.zero_()
        lib_rc = arx.lib.arx_reduce_host(arx._ptr_array(host), W, hout.data_ptr(), n, None, 0,
                                         torch.cuda.current_stream().cuda_stream)
        assert lib_rc == arx.ARX_OK, arx.arx_last_error()   # no staging needed
        torch.cuda.current_stream().synchronize()
        assert_bits_equal(hout.view(torch.int16).numpy(), want, "pinned direct")
    for r in range(W):
        assert torch.equal(host[r].view(torch.int16), x[r].view(torch.int16))


def test_host_buffer_form_pinned_in_place(arx, dev):
    W, n = 4, 50001
    x = sp.partials(W, n, "normal0.02", seed=22)
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    host = [x[r].clone().pin_memory() for r in range(W)]
    arx.arx_reduce_host(host, host[0], torch.empty(0, dtype=torch.uint8, device=dev))
    torch.cuda.current_stream().synchronize()
    assert_bits_equal(host[0].view(torch.int16).numpy(), want, "pinned in place")


def test_host_buffer_form_pageable_staged(arx, dev):
    W, n = 3, 70001
    x = sp.partials(W, n, "special", seed=23)
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    host = [x[r].clone() for r in range(W)]                  # pageable
    hout = torch.zeros(n, dtype=torch.bfloat16)
    staging = torch.empty(arx.arx_reduce_host_staging_bytes(W, n), dtype=torch.uint8, device=dev)
    arx.arx_reduce_host(host, hout, staging)
    torch.cuda.current_stream().synchronize()
    assert_bits_equal(hout.view(torch.int16).numpy(), want, "pageable staged")
    small = torch.empty(arx.arx_reduce_host_staging_bytes(W, n) - 2, dtype=torch.uint8, device=dev)
    assert arx.arx_reduce_host(host, hout, small, check=False) == arx.ARX_EINVAL
    rc = arx.lib.arx_reduce_host(arx._ptr_array(host), W, hout.data_ptr(), n, None, 0,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == arx.ARX_EINVAL and "staging" in arx.arx_last_error()


def test_random_small_cases(arx, dev):
    # Seeded fuzz over the shapes the vector paths split into: W = 1..8,
    # n in [0, 64] and a few larger ragged sizes, every pointer at its own
    # 2-byte offset within a 16-byte line (same offset for all -> vector path
    # with a scalar head; different -> scalar path), output separate or equal
    # to one slot.  Every element is compared with the oracle, guards checked.
    rng = np.random.default_rng(20261202)
    for case in range(300):
        W = int(rng.integers(1, 9))
        n = int(rng.integers(0, 65)) if case % 4 else int(rng.integers(65, 5000))
        same = bool(rng.integers(0, 2))
        base_off = int(rng.integers(0, 8))
        offs = [base_off] * (W + 1) if same else [int(v) for v in rng.integers(0, 8, W + 1)]
        alias = int(rng.integers(-1, W)) if n else -1       # -1: separate output
        x = sp.partials(W, n, "special", seed=10_000 + case)
        want = oracle.reduce(list(sp.to_u16_numpy(x))) if n else np.empty(0, np.uint16)
        stride = n + 16 + 2 * GUARD
        buf = torch.full((W + 1, stride), SENTINEL, dtype=torch.int16, device=dev)
        for r in range(W):
            buf[r, GUARD + offs[r]:GUARD + offs[r] + n] = x[r].view(torch.int16).to(dev)
        slots = [buf[r, GUARD + offs[r]:GUARD + offs[r] + n].view(torch.bfloat16) for r in range(W)]
        if alias >= 0:
            out, orow, ooff = slots[alias], alias, offs[alias]
        else:
            out, orow, ooff = buf[W, GUARD + offs[W]:GUARD + offs[W] + n].view(torch.bfloat16), W, offs[W]
        arx.arx_reduce(slots, out, n=n)
        torch.cuda.synchronize()
        host = buf.cpu().numpy().view(np.uint16)
        what = f"case {case}: W={W} n={n} offs={offs} alias={alias}"
        if n:
            assert_bits_equal(host[orow, GUARD + ooff:GUARD + ooff + n], want, what)
        for r in range(W + 1):                     # nothing outside the n elements moved
            o = offs[r]
            assert (host[r, :GUARD + o] == SENTINEL).all(), what
            assert (host[r, GUARD + o + n:] == SENTINEL).all(), what
            if r < W and r != orow:
                assert np.array_equal(host[r, GUARD + o:GUARD + o + n], sp.to_u16_numpy(x[r])), what


def test_more_than_2_to_31_elements(arx, dev):
    # W = 2 partials of 2^31 + 13 elements (4 GiB each, 12 GiB with the
    # output): any 32-bit element or byte index in the launch would wrap.
    # The partials are hashed from the element index on the device, and the
    # oracle recomputes sampled outputs one by one from the same patterns:
    # random indices plus both sides of 2^31 and 2^32 bytes and the tail.
    W, n = 2, (1 << 31) + 13
    free, _ = torch.cuda.mem_get_info(dev)
    if free < 14 * 2**30:
        pytest.skip("needs 14 GiB of free device memory")
    x = torch.empty(W, n, dtype=torch.int16, device=dev)
    chunk = 1 << 28
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        i = torch.arange(lo, hi, dtype=torch.int64, device=dev)
        for r in range(W):
            h = (i * 2654435761 + (r + 1) * 40503) & 0xFFFF
            h = torch.where((h & 0x7F80) == 0x7F80, h & 0xBFFF, h)    # finite patterns only
            x[r, lo:hi] = (h - ((h >= 0x8000).long() << 16)).to(torch.int16)
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    arx.arx_reduce([x[0].view(torch.bfloat16), x[1].view(torch.bfloat16)], out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(31)
    idx = np.concatenate([rng.integers(0, n, 200_000),
                          np.arange((1 << 31) - 64, (1 << 31) + 13), np.arange(n - 64, n),
                          np.arange(0, 64)])
    ti = torch.from_numpy(idx).to(dev)
    got = out.view(torch.int16)[ti].cpu().numpy().view(np.uint16)
    parts = [x[r][ti].cpu().numpy().view(np.uint16).copy() for r in range(W)]
    want = oracle.reduce(parts)
    assert_bits_equal(got, want, f"sampled outputs of a 2^31 + 13 element reduce")
    del x, out
    torch.cuda.empty_cache()


def test_prepared_plan_matches_and_rereads_contents(arx, dev):
    x, _ = sp.workload("w8_32x4096_normal")
    xd = x.to(dev)
    out = torch.empty(x.shape[1], dtype=torch.bfloat16, device=dev)
    plan = arx.arx_reduce_plan([xd[r] for r in range(8)], out)
    plan()
    torch.cuda.synchronize()
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))), "plan")
    y = sp.partials(8, x.shape[1], "normal", seed=77)
    xd.copy_(y.to(dev))                     # same storage, new contents
    plan()
    torch.cuda.synchronize()
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(y))), "plan again")
