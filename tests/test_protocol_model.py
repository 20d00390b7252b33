"""Pins for the oracle's sequential protocol model.

The model (oracle/protocol.py) runs the seq/parity slot protocol: Semaphore
start/end barriers (common.cuh, ``PullController::sync``), the per-block
parity epoch (common.cuh, ``PushController``), the zero-resetting signal pad
(triton_barrier.py, ``blockwise_barrier``) and the last-block counters
(arx.cu, ``arx_kernel``).  It is checked here against closed forms derived by
hand from those definitions, and against the stated invariants of the pages:
the pad is all zero after every completed barrier, ``counter == flag`` after
an end stage, the epoch is the step count mod 2, and two slot banks hold the
last two steps' inputs.
"""

import numpy as np
import pytest

import oracle
from oracle import protocol as P
import synthetic_partials as sp

M32 = 0xFFFFFFFF


def _inputs(W, n, step):
    return list(sp.to_u16_numpy(sp.partials(W, n, "normal", 4 + step)))


@pytest.mark.parametrize("W,B,k", [(1, 1, 1), (2, 3, 2), (4, 2, 5), (8, 4, 7)])
def test_closed_form_after_k_steps(W, B, k):
    st = P.State(W=W, B=B)
    hist = []
    for s in range(k):
        x = _inputs(W, 64, s)
        hist.append(x)
        out = P.step(st, x)
        # Output is the rank-order reduce of this step's inputs.
        assert np.array_equal(out, oracle.reduce(x))
    # Each step adds W (start) + W (end) to every flag; the end stage moves the
    # counter by 2W; so flag == counter == 2Wk.
    assert (st.flag == 2 * W * k).all() and (st.counter == 2 * W * k).all()
    assert (st.epoch == k % 2).all()
    assert not st.pad.any()
    assert st.blocks == [0, 0]
    assert st.seq == k and st.published == k and st.err == 0
    # Bank k & 1 holds step k's inputs, the other bank step k-1's.
    for r in range(W):
        assert np.array_equal(st.slots[k & 1][r], hist[k - 1][r])
        if k >= 2:
            assert np.array_equal(st.slots[(k - 1) & 1][r], hist[k - 2][r])


def test_unsigned_wrap_of_seq_and_flags():
    W, B = 8, 2
    seq0 = M32 - 1          # two steps before seq wraps
    flag0 = M32 - 5         # flags wrap during the first step
    st = P.State(W=W, B=B, seq=seq0)
    st.epoch[:] = seq0 % 2
    st.flag[:] = flag0
    st.counter[:] = flag0
    for s in range(3):
        P.step(st, _inputs(W, 16, s))
    assert st.err == 0
    assert st.seq == (seq0 + 3) & M32 == 1
    assert (st.flag == (flag0 + 6 * W) & M32).all()
    assert (st.counter == st.flag).all()
    assert (st.epoch == (seq0 + 3) % 2).all()


def test_missing_end_signal_reports_timeout():
    st = P.State(W=4, B=2)
    P.step(st, _inputs(4, 16, 0))
    assert st.err == 0
    P.step(st, _inputs(4, 16, 1), skip_end_signal_rank=2)
    assert st.err == P.ETIMEOUT


def test_epoch_mismatch_reports_state_error():
    st = P.State(W=2, B=3)
    st.epoch[1, 2] = 1
    P.step(st, _inputs(2, 16, 0))
    assert st.err == P.ESTATE


def test_parity_alternates_banks():
    st = P.State(W=2, B=1)
    a, b, c = _inputs(2, 8, 0), _inputs(2, 8, 1), _inputs(2, 8, 2)
    P.step(st, a)          # seq 1 -> bank 1
    P.step(st, b)          # seq 2 -> bank 0
    assert np.array_equal(st.slots[1][0], a[0]) and np.array_equal(st.slots[0][0], b[0])
    P.step(st, c)          # seq 3 -> bank 1 again, bank 0 untouched
    assert np.array_equal(st.slots[1][1], c[1]) and np.array_equal(st.slots[0][1], b[1])


# ---- barrier variants (triton_barrier.py Patterns 0/1/2 on the signal pad) ----------------

@pytest.mark.parametrize("sync", ["pad", "pad_fenced"])
@pytest.mark.parametrize("W,B,k", [(1, 1, 1), (3, 2, 4), (8, 3, 5)])
def test_pad_modes_closed_form(sync, W, B, k):
    st = P.State(W=W, B=B)
    for s in range(k):
        x = _inputs(W, 32, s)
        assert np.array_equal(P.step(st, x, sync=sync), oracle.reduce(x))
    # Three pad barriers per step, each pairing every send with one wait, so
    # the pad is zero after every step; the Semaphores are never touched.
    assert not st.pad.any()
    assert not st.flag.any() and not st.counter.any()
    assert (st.epoch == k % 2).all() and st.blocks == [0, 0]
    assert st.seq == k and st.published == k and st.err == 0


def test_switching_modes_between_steps():
    W, B = 4, 2
    st = P.State(W=W, B=B)
    modes = ["semaphore", "pad", "pad_fenced", "semaphore", "pad", "semaphore"]
    for s, m in enumerate(modes):
        P.step(st, _inputs(W, 16, s), sync=m)
    # Only the Semaphore steps move the flags, by 2W each.
    assert st.err == 0
    assert (st.flag == 2 * W * modes.count("semaphore")).all() and (st.counter == st.flag).all()
    assert not st.pad.any() and (st.epoch == len(modes) % 2).all()


@pytest.mark.parametrize("sync", ["pad", "pad_fenced"])
def test_pad_mode_missing_end_signal_reports_timeout(sync):
    st = P.State(W=3, B=2)
    P.step(st, _inputs(3, 16, 0), sync=sync)
    assert st.err == 0
    P.step(st, _inputs(3, 16, 1), skip_end_signal_rank=1, sync=sync)
    assert st.err == P.ETIMEOUT


@pytest.mark.parametrize("W,B,k", [(1, 1, 1), (3, 2, 4), (8, 3, 5)])
def test_cluster_mode_closed_form(W, B, k):
    # The single-GPU reading with the W blocks of a chunk in one cluster: the
    # barriers are the cluster's own, so pad and Semaphores stay untouched
    # while seq, published, epochs and the slot banks advance as in the others.
    st = P.State(W=W, B=B)
    for s in range(k):
        x = _inputs(W, 32, s)
        assert np.array_equal(P.step(st, x, sync="cluster"), oracle.reduce(x))
    assert not st.pad.any() and not st.flag.any() and not st.counter.any()
    assert (st.epoch == k % 2).all() and st.blocks == [0, 0]
    assert st.seq == k and st.published == k and st.err == 0
    assert np.array_equal(st.slots[k & 1][W - 1], _inputs(W, 32, k - 1)[W - 1])


def test_cluster_mode_has_no_signal_to_skip():
    with pytest.raises(ValueError):
        P.step(P.State(W=2, B=1), _inputs(2, 8, 0), skip_end_signal_rank=0, sync="cluster")


def test_unknown_mode_is_rejected():
    with pytest.raises(ValueError):
        P.step(P.State(W=1, B=1), _inputs(1, 8, 0), sync="fenced")


@pytest.mark.parametrize("W,B,k", [(1, 1, 2), (3, 2, 3), (8, 4, 5)])
def test_semaphore_global_mode_closed_form(W, B, k):
    # Where the GPU holds a Semaphore flag during the step (global memory, or
    # the shared memory of a thread-block cluster) does not change
    # PullController::sync's arithmetic: after k steps flag == counter == 2Wk,
    # the pad is all zero, the epoch is k mod 2 -- as in the default mode.
    st = P.State(W=W, B=B)
    for s in range(k):
        x = _inputs(W, 64, s)
        assert np.array_equal(P.step(st, x, sync="semaphore_global"), oracle.reduce(x))
    assert (st.flag == 2 * W * k).all() and (st.counter == 2 * W * k).all()
    assert not st.pad.any() and (st.epoch == k % 2).all() and st.seq == k and st.err == 0


def test_semaphore_global_missing_end_signal_reports_timeout():
    # One rank skips its end signal: every flag gets 2W - 1 adds, no counter
    # advances, and the error word reports ETIMEOUT -- the same words as the
    # default mode's.
    W, B = 4, 2
    st = P.State(W=W, B=B)
    P.step(st, _inputs(W, 32, 0), skip_end_signal_rank=1, sync="semaphore_global")
    assert st.err == P.ETIMEOUT
    assert (st.flag == 2 * W - 1).all() and (st.counter == 0).all()
