"""GPU tests of the protocol step (``arx_step``) against the oracle and its model.

* Output: bit-exact against the oracle's rank-order reduce (and therefore
  against ``arx_reduce``) for every W, ragged n and misaligned buffers.
* Protocol words after k steps equal the oracle's sequential model
  (oracle/protocol.py): seq, per-block epochs, Semaphore flag == counter
  (common.cuh, ``PullController::sync``), the signal pad all zero
  (triton_barrier.py, ``barrier_test``'s assertion), both block counters
  back at zero (arx.cu), and the two slot banks holding the last two steps'
  inputs (arx.cu: two buffers by parity).
* Unsigned wrap of seq and flags.
* 10,000 steps captured in one CUDA graph with fresh partials per step.
* Failure detection without any GPU fault: a missing end-barrier signal
  makes the bounded waits expire (ARX_ETIMEOUT read by the host, context
  usable after a reset); a corrupted epoch reports ARX_ESTATE.
* All of the above in each barrier variant (``ARX_SYNC_SEMAPHORE`` with the
  flags in the cluster's shared memory, ``ARX_SYNC_SEMAPHORE_GLOBAL`` with
  them in global memory: common.cuh's Semaphore barriers;
  ``ARX_SYNC_PAD``, ``ARX_SYNC_PAD_FENCED``: triton_barrier.py's pad barrier
  in its Patterns 0/1/2, relaxed or acq_rel; ``ARX_SYNC_CLUSTER``), and
  switching variants between steps of one context.
* The slot banks in a separate buffer (``arx_ctx_init_split``), in device
  memory or in page-locked host memory (arx.cu's GB10 layout: pinned host
  slots the GPU writes and reads over the CPU-GPU link): single steps, the
  words against the model, the fault test and the 10,000-step graph.
"""

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from oracle import protocol as model
import synthetic_partials as sp
from test_gpu_reduce import assert_bits_equal

pytestmark = pytest.mark.gpu

M32 = 0xFFFFFFFF
SYNCS = ["semaphore", "pad", "pad_fenced", "cluster", "semaphore_global"]
FLAG_SYNCS = ["semaphore", "pad", "pad_fenced", "semaphore_global"]   # with in-protocol fault injection
SEM_SYNCS = ("semaphore", "semaphore_global")     # the variants that advance the Semaphore words


@pytest.fixture(scope="module")
def dev(arx):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return torch.device("cuda:0")


class Ctx:
    """A context plus typed views of its workspace words."""

    def __init__(self, arx, dev, W, max_n, nblocks=0, sync="semaphore", slots="one"):
        """slots: "one" (words and slots in one device buffer), "device" or "host"
        (separate slot buffer in device memory or in page-locked host memory)."""
        self.arx = arx
        self.where = slots
        if slots == "one":
            nbytes = arx.arx_ctx_workspace_bytes(W, max_n, nblocks)
            self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
            self.ctx = arx.arx_ctx_init(self.ws, W, max_n, nblocks)
        else:
            self.ws = torch.zeros(arx.arx_ctx_words_bytes(W, nblocks), dtype=torch.uint8, device=dev)
            sb = arx.arx_ctx_slots_bytes(W, max_n)
            # Fill the slots with garbage: their contents must not matter.
            self.slots = torch.full((sb,), 0xA5, dtype=torch.uint8)
            self.slots = self.slots.pin_memory() if slots == "host" else self.slots.to(dev)
            self.ctx = arx.arx_ctx_init_split(self.ws, self.slots, W, max_n, nblocks)
            assert self.ctx.slots_where == (arx.ARX_SLOTS_HOST if slots == "host" else arx.ARX_SLOTS_DEVICE)
        self.W, self.B = W, self.ctx.nblocks
        self.set_sync(sync)

    def set_sync(self, sync):
        self.arx.arx_ctx_set_sync(self.ctx, SYNCS.index(sync))
        self.sync = sync

    def words(self):
        c, W, B = self.ctx, self.W, self.B
        host = self.ws[: c.ctrl_bytes].cpu().numpy()
        u32 = lambda off, cnt: host[off: off + 4 * cnt].view(np.uint32).astype(np.int64)
        hdr = u32(0, 5)
        sem = host[c.off_sem: c.off_sem + 128 * W * B].reshape(W * B, 128)[:, :8].copy().view(np.uint32)
        return dict(seq=int(hdr[0]), err=int(hdr[1]), blocks=[int(hdr[2]), int(hdr[3])],
                    published=int(hdr[4]), stagger=u32(128, 32),
                    epoch=u32(c.off_epoch, W * B).reshape(W, B),
                    flag=sem[:, 0].astype(np.int64).reshape(W, B),
                    counter=sem[:, 1].astype(np.int64).reshape(W, B),
                    pad=u32(c.off_pad, W * B * W).reshape(W, B, W))

    def slot(self, par, r, n):
        c = self.ctx
        off = (par * self.W + r) * c.slot_stride * 2
        if self.where == "one":
            off += c.off_slots
            return self.ws[off: off + 2 * n].cpu().numpy().view(np.uint16)
        torch.cuda.synchronize()
        return self.slots[off: off + 2 * n].cpu().numpy().view(np.uint16)

    def poke(self, off, value):
        self.ws[off: off + 4] = torch.tensor([value], dtype=torch.int64).view(torch.uint8)[:4].to(self.ws.device)


def _assert_stagger_word(words, last_staggered_seq):
    """Staggered staging's start word (header bytes 128-135): the seq of the
    context's last staggered step in its high half (the low half is that
    step's global-timer start), zero before the first; the rest of the
    header's upper half zero."""
    w = words["stagger"]
    if last_staggered_seq:
        assert w[1] == last_staggered_seq, (int(w[1]), last_staggered_seq)
    else:
        assert not w[:2].any()
    assert not w[2:].any()


def _stagger_groups(W, n, B):
    """Block groups of a host-slot step: about 128 KiB of staged data each, at
    most B; none below two (as include/arx.h describes)."""
    K = min((W * n * 2 + (64 << 10)) >> 17, B)
    return K if K >= 2 else 0


def _compare_to_model(words, st: model.State):
    assert words["seq"] == st.seq and words["published"] == st.published
    assert words["blocks"] == st.blocks
    assert (words["err"] & 0xFF) == st.err
    assert np.array_equal(words["epoch"], st.epoch)
    assert np.array_equal(words["flag"], st.flag)
    assert np.array_equal(words["counter"], st.counter)
    assert np.array_equal(words["pad"], st.pad)


def _step(arx, c: Ctx, x: torch.Tensor, dev, out_offset=0, in_offset=0):
    W, n = x.shape
    if in_offset:
        buf = torch.zeros(W, n + 8, dtype=torch.bfloat16, device=dev)
        buf[:, in_offset:in_offset + n] = x.to(dev)
        ins = [buf[r, in_offset:in_offset + n] for r in range(W)]
    else:
        xd = x.to(dev)
        ins = [xd[r] for r in range(W)]
    ob = torch.zeros(n + 16, dtype=torch.bfloat16, device=dev)
    out = ob[out_offset:out_offset + n]
    arx.arx_step(c.ctx, ins, out)
    return out


@pytest.mark.parametrize("sync", SYNCS)
@pytest.mark.parametrize("W", range(1, 9))
def test_single_step_every_w(arx, dev, W, sync):
    for n, nblocks in ((131072, 0), (1000003, 0), (13, 1), (4096 + 5, 3)):
        c = Ctx(arx, dev, W, n, nblocks, sync)
        x = sp.partials(W, n, "special" if n < 5000 else "normal", seed=W * 7 + n)
        out = _step(arx, c, x, dev)
        st, seq, err = arx.arx_ctx_query(c.ctx)
        assert (st, seq, err) == (arx.ARX_OK, 1, 0)
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))),
                          f"step W={W} n={n} B={c.B}")


@pytest.mark.parametrize("W", [1, 2, 5, 8])
def test_single_step_host_slots(arx, dev, W):
    # The slot banks in page-locked host memory: staged partials go out over
    # the CPU-GPU link and are read back from there.
    for n, nblocks in ((131072, 0), (1000003, 0), (13, 1), (4096 + 5, 3)):
        c = Ctx(arx, dev, W, n, nblocks, "semaphore", "host")
        x = sp.partials(W, n, "special" if n < 5000 else "normal", seed=W * 11 + n)
        out = _step(arx, c, x, dev)
        st, seq, err = arx.arx_ctx_query(c.ctx)
        assert (st, seq, err) == (arx.ARX_OK, 1, 0)
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))),
                          f"host slots W={W} n={n} B={c.B}")
        assert np.array_equal(c.slot(1, W - 1, n), sp.to_u16_numpy(x)[W - 1])


def test_host_slot_steps_of_varying_size(arx, dev):
    # Slots in host memory: steps of 192 KiB of partials or more stage in
    # turn, in a number of block groups that follows each step's size; smaller
    # ones all at once.  Mixing them on one context must not matter: every
    # output bit-exact, the start word tagged with the last staggered step.
    W, max_n = 8, 131072
    c = Ctx(arx, dev, W, max_n, 0, "semaphore", "host")
    staggered = last = 0
    for s, n in enumerate((131072, 4096, 70001, 131072, 11, 65536)):
        for sync in SYNCS:
            arx.arx_ctx_set_sync(c.ctx, SYNCS.index(sync))
            x = sp.partials(W, n, "normal", seed=700 + 10 * s + SYNCS.index(sync))
            out = _step(arx, c, x, dev)
            st, seq, err = arx.arx_ctx_query(c.ctx)
            assert (st, err) == (arx.ARX_OK, 0)
            assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))),
                              f"n={n} {sync}")
            if _stagger_groups(W, n, c.B):
                staggered += 1
                last = seq
            _assert_stagger_word(c.words(), last)
    assert staggered > 0


def test_random_small_steps(arx, dev):
    # Seeded fuzz of the step: W = 1..8, small and ragged n, B from 1 to the
    # automatic choice, every barrier variant, slots in one buffer or in host
    # memory; each step's output against the oracle and its words against the
    # model.
    rng = np.random.default_rng(4242)
    for case in range(40):
        W = int(rng.integers(1, 9))
        n = int(rng.integers(1, 3000))
        B = int(rng.integers(0, 6))
        sync = SYNCS[int(rng.integers(0, len(SYNCS)))]
        slots = "host" if case % 5 == 0 else "one"
        c = Ctx(arx, dev, W, n, B, sync, slots)
        st = model.State(W=W, B=c.B)
        for s in range(2):
            x = sp.partials(W, n, "special", seed=20_000 + 2 * case + s)
            out = _step(arx, c, x, dev)
            want = model.step(st, list(sp.to_u16_numpy(x)), sync=sync)
            assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK
            assert_bits_equal(out.cpu().view(torch.int16).numpy(), want,
                              f"case {case} step {s}: W={W} n={n} B={c.B} {sync} {slots}")
            _compare_to_model(c.words(), st)


def test_contexts_step_concurrently_on_separate_streams(arx, dev):
    # Independent contexts share no state: four of them (different W and
    # barrier variants) run 200 steps each on four streams at once -- two
    # cooperative grids and two of clusters resident together, each waiting
    # only on its own blocks -- and every output of all four is checked.
    steps = 200
    cfg = [(8, 65536, "semaphore"), (3, 40000, "pad"), (5, 30000, "cluster"), (6, 20000, "semaphore_global")]
    ctxs, ins, outs, wants = [], [], [], []
    for W, n, sync in cfg:
        c = Ctx(arx, dev, W, n, 0, sync)
        k = 4
        xs = [sp.partials(W, n, "normal", seed=900 + 10 * W + j) for j in range(k)]
        ins.append([x.to(dev) for x in xs])
        wants.append([oracle.reduce(list(sp.to_u16_numpy(x))) for x in xs])
        outs.append(torch.zeros(steps, n, dtype=torch.bfloat16, device=dev))
        ctxs.append(c)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in cfg]
    for t in range(steps):
        for j, (W, n, sync) in enumerate(cfg):
            xd = ins[j][t % 4]
            arx.arx_step(ctxs[j].ctx, [xd[r] for r in range(W)], outs[j][t], stream=streams[j])
    torch.cuda.synchronize()
    for j, (W, n, sync) in enumerate(cfg):
        st, seq, err = arx.arx_ctx_query(ctxs[j].ctx)
        assert (st, seq, err) == (arx.ARX_OK, steps, 0), sync
        got = outs[j].cpu().view(torch.int16).numpy().view(np.uint16)
        for t in range(steps):
            assert_bits_equal(got[t], wants[j][t % 4], f"context {j} step {t}")
        w = ctxs[j].words()
        assert not w["pad"].any() and (w["epoch"] == steps % 2).all()


@pytest.mark.parametrize("sync", ["pad", "pad_fenced"])
def test_barrier_test_pattern_pad_all_zero(arx, dev, sync):
    # triton_barrier.py's barrier_test: the blockwise barrier on a launch of
    # 32 blocks, then assert the signal pad is all zero.  Here 32 blocks per
    # virtual rank run three pad barriers per step (Patterns 0, 1, 2); the pad
    # must be all zero after every step.
    W, n, B = 8, 32 * 8 * 64, 32
    c = Ctx(arx, dev, W, n, B, sync)
    assert c.B == B
    for s in range(5):
        x = sp.partials(W, n, "normal", seed=700 + s)
        out = _step(arx, c, x, dev)
        assert arx.arx_ctx_query(c.ctx)[:3] == (arx.ARX_OK, s + 1, 0)
        assert not c.words()["pad"].any(), f"pad not zero after step {s + 1}"
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))),
                          f"step {s + 1}")


def test_step_plan(arx, dev):
    W, n = 4, 30000
    c = Ctx(arx, dev, W, n, 0, "pad")
    x = sp.partials(W, n, "normal", seed=61)
    xd = x.to(dev)
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    plan = arx.arx_step_plan(c.ctx, [xd[r] for r in range(W)], out)
    st = model.State(W=W, B=c.B)
    for s in range(3):
        plan()
        want = model.step(st, list(sp.to_u16_numpy(x)), sync="pad")
        assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), want, f"plan step {s}")
    _compare_to_model(c.words(), st)


def test_step_equals_stateless_reduce(arx, dev):
    x, _ = sp.workload("w8_32x4096_normal")
    xd = x.to(dev)
    c = Ctx(arx, dev, 8, x.shape[1])
    a = torch.empty(x.shape[1], dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    arx.arx_reduce([xd[r] for r in range(8)], a)
    arx.arx_step(c.ctx, [xd[r] for r in range(8)], b)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("in_off,out_off", [(1, 0), (0, 3), (5, 5)])
def test_step_misaligned_buffers(arx, dev, in_off, out_off):
    W, n = 4, 20011
    c = Ctx(arx, dev, W, n)
    x = sp.partials(W, n, "normal", seed=in_off * 10 + out_off)
    out = _step(arx, c, x, dev, out_offset=out_off, in_offset=in_off)
    assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))),
                      f"offsets in={in_off} out={out_off}")


def test_step_output_aliases_an_input(arx, dev):
    W, n = 3, 50000
    c = Ctx(arx, dev, W, n)
    x = sp.partials(W, n, "normal", seed=31)
    xd = x.to(dev)
    ins = [xd[r] for r in range(W)]
    arx.arx_step(c.ctx, ins, ins[1])
    assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK
    assert_bits_equal(xd[1].cpu().view(torch.int16).numpy(),
                      oracle.reduce(list(sp.to_u16_numpy(x))), "step in place")


@pytest.mark.parametrize("slots", ["one", "device", "host"])
@pytest.mark.parametrize("sync", SYNCS)
@pytest.mark.parametrize("W,n,B,k", [(8, 131072, 0, 5), (3, 777, 2, 4), (5, 65536 + 7, 7, 3), (1, 100, 1, 2)])
def test_protocol_words_follow_the_model(arx, dev, W, n, B, k, sync, slots):
    c = Ctx(arx, dev, W, n, B, sync, slots)
    st = model.State(W=W, B=c.B)
    hist = []
    for s in range(k):
        x = sp.partials(W, n, "normal", seed=4 + s)
        u = list(sp.to_u16_numpy(x))
        hist.append(u)
        out = _step(arx, c, x, dev)
        want = model.step(st, u, sync=sync)
        assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), want, f"step {s}")
        _compare_to_model(c.words(), st)
    assert (c.words()["flag"] == (2 * W * k if sync in SEM_SYNCS else 0)).all()
    # Staggered staging's start word: tagged with the last step when the
    # steps staged in turn (host slots), else never written.
    _assert_stagger_word(c.words(), k if slots == "host" and _stagger_groups(W, n, c.B) else 0)
    for r in range(W):
        assert np.array_equal(c.slot(k & 1, r, n), hist[k - 1][r])
        if k >= 2:
            assert np.array_equal(c.slot((k - 1) & 1, r, n), hist[k - 2][r])


def test_unsigned_wrap_of_seq_and_flags(arx, dev):
    W, n, B = 8, 4096, 4
    c = Ctx(arx, dev, W, n, B)
    seq0, flag0 = M32 - 1, M32 - 5
    c.poke(0, seq0)
    ctx = c.ctx
    for i in range(W * B):
        c.poke(ctx.off_sem + 128 * i, flag0)
        c.poke(ctx.off_sem + 128 * i + 4, flag0)
        c.poke(ctx.off_epoch + 4 * i, seq0 % 2)
    st = model.State(W=W, B=B, seq=seq0)
    st.epoch[:] = seq0 % 2
    st.flag[:] = flag0
    st.counter[:] = flag0
    st.published = 0
    for s in range(3):
        x = sp.partials(W, n, "normal", seed=50 + s)
        out = _step(arx, c, x, dev)
        want = model.step(st, list(sp.to_u16_numpy(x)))
        assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), want, f"wrap step {s}")
    w = c.words()
    _compare_to_model(w, st)
    assert w["seq"] == 1


def test_unsigned_wrap_with_staggered_host_slots(arx, dev):
    # The same wrap on a host-slot context whose steps stage in turn.  The
    # step numbered 0 finds the never-written start word's tag (0) equal to
    # its seq and takes that stale start, so its groups start at once; the
    # steps numbered 1 and 2 install their own.  Every output bit-exact, the
    # words as the model says, the start word tagged with the last step.
    W, n = 8, 131072
    c = Ctx(arx, dev, W, n, 0, "semaphore", "host")
    B = c.B
    assert _stagger_groups(W, n, B)
    seq0, flag0 = M32, M32 - 5      # 2^32 - 1 steps done: the next is numbered 0
    c.poke(0, seq0)
    ctx = c.ctx
    for i in range(W * B):
        c.poke(ctx.off_sem + 128 * i, flag0)
        c.poke(ctx.off_sem + 128 * i + 4, flag0)
        c.poke(ctx.off_epoch + 4 * i, seq0 % 2)
    st = model.State(W=W, B=B, seq=seq0)
    st.epoch[:] = seq0 % 2
    st.flag[:] = flag0
    st.counter[:] = flag0
    st.published = 0
    for s in range(3):
        x = sp.partials(W, n, "normal", seed=60 + s)
        out = _step(arx, c, x, dev)
        want = model.step(st, list(sp.to_u16_numpy(x)))
        assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), want, f"host-slot wrap step {s}")
    w = c.words()
    _compare_to_model(w, st)
    assert w["seq"] == 2
    _assert_stagger_word(w, 2)


@pytest.mark.parametrize("sync,slots,n", [(m, "one", 8192) for m in FLAG_SYNCS]
                         + [("semaphore", "host", 8192), ("semaphore", "host", 65536)])
def test_timeout_is_reported_and_context_recovers(arx, dev, sync, slots, n):
    # n = 65536 on host slots: 512 KiB of partials, so the step stages in turn
    # (two block groups at B = 2) and the staggered kernel's end wait expires.
    W = 4
    c = Ctx(arx, dev, W, n, 2, sync, slots)
    assert bool(_stagger_groups(W, n, c.B)) == (slots == "host" and n == 65536)
    x = sp.partials(W, n, "normal", seed=8)
    _step(arx, c, x, dev)
    assert arx.arx_ctx_query(c.ctx)[:2] == (arx.ARX_OK, 1)
    arx.arx_ctx_set_timeout(c.ctx, 20_000_000)      # 20 ms bound on every wait
    arx.arx_ctx_set_fault(c.ctx, 2)                 # virtual rank 2 never sends its end signal
    _step(arx, c, x, dev)
    st, seq, err = arx.arx_ctx_query(c.ctx)
    assert st == arx.ARX_ETIMEOUT
    # stage: the end-barrier wait (2 on the Semaphores, 9 on the pad)
    assert err & 0xFF == arx.ARX_ETIMEOUT and (err >> 8) & 15 == (2 if sync in SEM_SYNCS else 9)
    assert seq == 2                                  # the kernel still finished
    w = c.words()
    assert w["blocks"] == [0, 0]
    if sync in SEM_SYNCS:
        assert not w["pad"].any()
    # The context remembers the failure: the next step is refused on the host,
    # with nothing launched (output and protocol words untouched).
    assert c.ctx.failed_err == err
    arx.arx_ctx_set_fault(c.ctx, -1)
    sentinel = torch.full((n,), 7.0, dtype=torch.bfloat16, device=dev)
    xd = x.to(dev)
    words_before = c.ws[:c.ctx.ctrl_bytes].clone()
    assert arx.arx_step(c.ctx, [xd[r] for r in range(W)], sentinel, check=False) == arx.ARX_ESTATE
    torch.cuda.synchronize()
    assert bool((sentinel == 7.0).all())
    assert torch.equal(c.ws[:c.ctx.ctrl_bytes], words_before)
    # Recovery: zero the protocol words, step again.
    arx.arx_ctx_reset(c.ctx)
    assert c.ctx.failed_err == 0
    out = _step(arx, c, x, dev)
    assert arx.arx_ctx_query(c.ctx)[:3] == (arx.ARX_OK, 1, 0)
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))),
                      "after reset")


def test_host_watchdog_reports_a_stall_before_the_device_bound(arx, dev):
    # arx.cu's proxy watchdog, on the host: a step published but not done for
    # longer than the stall threshold is reported while the kernel is still
    # inside its own bounded wait.  The stall comes from the in-protocol fault
    # (a virtual rank skips its end signal); no GPU fault is involved.
    import threading
    W, n = 4, 8192
    c = Ctx(arx, dev, W, n, 2)
    x = sp.partials(W, n, "normal", seed=8)
    res = {}

    def watch(key, target):
        res[key] = arx.arx_watch_step(c.ctx, target, stall_s=0.05, poll_s=0.001, max_wait_s=5.0)

    th = threading.Thread(target=watch, args=("ok", 1))
    th.start()
    _step(arx, c, x, dev)
    th.join()
    st, rep = res["ok"]
    assert st == arx.ARX_OK and rep.seq == 1 and rep.dev_err == 0 and rep.polls >= 1

    arx.arx_ctx_set_timeout(c.ctx, 600_000_000)     # device bound: 600 ms
    arx.arx_ctx_set_fault(c.ctx, 1)
    th = threading.Thread(target=watch, args=("stall", 2))
    th.start()
    _step(arx, c, x, dev)
    th.join()
    st, rep = res["stall"]
    assert st == arx.ARX_ETIMEOUT
    assert rep.published == 2 and rep.seq == 1 and rep.dev_err == 0
    assert rep.stalled_ns >= 50_000_000 and rep.waited_ns < 600_000_000
    # The device then reports its own expired wait, and the context recovers.
    st, seq, err = arx.arx_ctx_query(c.ctx)
    assert st == arx.ARX_ETIMEOUT and seq == 2
    arx.arx_ctx_set_fault(c.ctx, -1)
    arx.arx_ctx_reset(c.ctx)
    out = _step(arx, c, x, dev)
    assert arx.arx_ctx_query(c.ctx)[:3] == (arx.ARX_OK, 1, 0)
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))),
                      "after the stall")


def test_epoch_mismatch_reports_state_error(arx, dev):
    W, n = 2, 1024
    c = Ctx(arx, dev, W, n, 2)
    c.poke(c.ctx.off_epoch + 4 * 3, 1)   # epoch[1][1] claims an odd step count
    x = sp.partials(W, n, "normal", seed=2)
    out = _step(arx, c, x, dev)
    st, seq, err = arx.arx_ctx_query(c.ctx)
    assert st == arx.ARX_ESTATE and (err >> 8) & 15 == 5 and (err >> 12) & 15 == 1
    # The data path is unaffected.
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))), "data")


def test_switching_sync_modes_between_steps(arx, dev):
    W, n = 6, 30011
    c = Ctx(arx, dev, W, n, 3)
    st = model.State(W=W, B=c.B)
    for s, sync in enumerate(["semaphore", "pad", "cluster", "pad_fenced", "semaphore_global", "semaphore",
                              "cluster", "pad_fenced", "semaphore_global", "pad", "cluster", "semaphore"]):
        c.set_sync(sync)
        x = sp.partials(W, n, "normal", seed=300 + s)
        out = _step(arx, c, x, dev)
        want = model.step(st, list(sp.to_u16_numpy(x)), sync=sync)
        assert arx.arx_ctx_query(c.ctx)[0] == arx.ARX_OK, sync
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), want, f"step {s} ({sync})")
        _compare_to_model(c.words(), st)


def test_mixed_variants_in_one_graph(arx, dev):
    # 999 steps captured in one graph, the barrier variant changing every
    # step (Semaphore, pad, pad all acq_rel, ...): back-to-back dependent
    # launches of different kernels on one context.  Every output is checked,
    # and the final words against the model run with the same sequence.
    W, n, steps = 5, 20000, 999
    c = Ctx(arx, dev, W, n, 0)
    xs = [sp.partials(W, n, "normal", seed=1500 + j) for j in range(3)]
    xd = [x.to(dev) for x in xs]
    wants = [oracle.reduce(list(sp.to_u16_numpy(x))) for x in xs]
    outs = torch.zeros(steps, n, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(steps):
            c.set_sync(SYNCS[t % len(SYNCS)])
            arx.arx_step(c.ctx, [xd[t % 3][r] for r in range(W)], outs[t], stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert arx.arx_ctx_query(c.ctx)[:3] == (arx.ARX_OK, steps, 0)
    got = outs.cpu().view(torch.int16).numpy().view(np.uint16)
    for t in range(steps):
        assert_bits_equal(got[t], wants[t % 3], f"step {t} ({SYNCS[t % len(SYNCS)]})")
    st = model.State(W=W, B=c.B)
    for t in range(steps):
        model.step(st, list(sp.to_u16_numpy(xs[t % 3])), sync=SYNCS[t % len(SYNCS)])
    _compare_to_model(c.words(), st)


def test_unknown_sync_mode_is_rejected(arx, dev):
    c = Ctx(arx, dev, 2, 64, 1)
    with pytest.raises(arx.ArxError):
        arx.arx_ctx_set_sync(c.ctx, len(SYNCS))
    assert c.ctx.sync_mode == arx.ARX_SYNC_SEMAPHORE


def test_cluster_variant_refuses_fault_injection(arx, dev):
    # The cluster barrier has no flag signal a rank could skip (a block that
    # never arrived would hold the hardware barrier forever), so the knob is
    # refused on the host before anything is launched.
    W, n = 4, 4096
    c = Ctx(arx, dev, W, n, 2, "cluster")
    arx.arx_ctx_set_fault(c.ctx, 1)
    x = sp.partials(W, n, "normal", seed=5)
    xd = x.to(dev)
    out = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    assert arx.arx_step(c.ctx, [xd[r] for r in range(W)], out, check=False) == arx.ARX_EINVAL
    arx.arx_ctx_set_fault(c.ctx, -1)
    arx.arx_step(c.ctx, [xd[r] for r in range(W)], out)
    assert arx.arx_ctx_query(c.ctx)[:3] == (arx.ARX_OK, 1, 0)
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(x))), "cluster")


# ---- 10,000 steps in one CUDA graph --------------------------------------------------------

GRAPH_STEPS = sp.GRAPH_STEPS
W8, N8 = 8, sp.N_32x4096


@pytest.fixture(scope="module")
def graph_workload(dev):
    """10,000 steps of fresh normal(0, 1) partials (seed 4 + step) on the device, with
    the oracle's output of every step and the last two steps' inputs."""
    steps, chunk = GRAPH_STEPS, 500
    inputs = torch.empty(steps, W8, N8, dtype=torch.bfloat16, device=dev)
    want = np.empty((steps, N8), dtype=np.uint16)
    last_two = {}
    host = torch.empty(chunk, W8, N8, dtype=torch.int16).pin_memory()
    host_np = host.numpy().view(np.uint16)

    # Torch's RNG and the oracle's C code release the GIL, so threads generate
    # in parallel.
    def fill(s, base):
        u = sp.to_u16_numpy(sp.graph_step_partials(s))
        host_np[s - base] = u
        want[s] = oracle.reduce_rows(u)
        if s >= steps - 2:
            last_two[s] = u.copy()

    with ThreadPoolExecutor(max_workers=min(16, oracle.default_threads())) as ex:
        for base in range(0, steps, chunk):
            hi = min(steps, base + chunk)
            list(ex.map(lambda s: fill(s, base), range(base, hi)))
            inputs[base:hi].view(torch.int16).copy_(host[: hi - base])
    torch.cuda.synchronize()
    yield inputs, want, last_two
    del inputs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("sync,slots", [(m, "one") for m in SYNCS] + [("semaphore", "host")])
def test_ten_thousand_steps_in_one_graph(arx, dev, graph_workload, sync, slots):
    inputs, want, last_two = graph_workload
    steps = inputs.shape[0]
    c = Ctx(arx, dev, W8, N8, 0, sync, slots)
    outputs = torch.zeros(steps, N8, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for t in range(steps):
            arx.arx_step(c.ctx, [inputs[t, r] for r in range(W8)], outputs[t], stream=s)
    g.replay()
    torch.cuda.synchronize()
    st, seq, err = arx.arx_ctx_query(c.ctx)
    assert (st, seq, err) == (arx.ARX_OK, steps, 0)
    got = outputs.cpu().view(torch.int16).numpy().view(np.uint16)
    bad = np.flatnonzero((got != want).any(axis=1))
    assert bad.size == 0, f"{bad.size} of {steps} steps differ; first step {int(bad[0])}"
    w = c.words()
    assert not w["pad"].any(), "signal pad must be all zero after the last step"
    flags = 2 * W8 * steps if sync in SEM_SYNCS else 0   # the pad variants leave the Semaphores alone
    assert (w["flag"] == flags).all() and (w["counter"] == w["flag"]).all()
    assert (w["epoch"] == steps % 2).all() and w["blocks"] == [0, 0]
    assert w["published"] == steps
    _assert_stagger_word(w, steps if slots == "host" and _stagger_groups(W8, N8, c.B) else 0)
    for r in range(W8):
        assert np.array_equal(c.slot(steps & 1, r, N8), last_two[steps - 1][r])
        assert np.array_equal(c.slot((steps - 1) & 1, r, N8), last_two[steps - 2][r])
