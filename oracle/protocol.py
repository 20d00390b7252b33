"""Sequential model of the one-GPU slot protocol (one step = one all-reduce call).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages synchronise ranks on different GPUs.  On one GPU the W ranks become
W *virtual ranks*: the step runs as one grid of B x W thread blocks, where
block (b, r) plays rank r's block b.  This model executes the step's phases
for every block in lock-step, which is one valid serialisation of the
concurrent kernel (every barrier is satisfied when all of its participants
have arrived), and returns the output together with every protocol word.

Phases of one step, with the passage each follows:

1. seq/parity -- arx.cu, ``arx_kernel``: ``seq`` is the last completed
   sequence number plus one and the slot bank is ``seq & 1`` (header comment:
   two buffers by parity are enough).
   The per-block ``PushController`` epoch (common.cuh, ``PushController``,
   ``kNumStages = 2``) must equal the parity of the completed steps, i.e.
   ``(seq - 1) & 1``; a mismatch is a state error.
2. start barrier -- common.cuh, ``PullController::sync`` with the start stage
   (unfenced): every virtual rank adds 1 to the Semaphore flag of block b of
   every rank; rank r waits until ``flag - counter >= W``.
3. stage -- arx.cu, ``arx_kernel`` stage copy: rank r's input goes to
   ``slots[par][r]`` (standing in for the RDMA write into every peer's
   ``recv[seq & 1][rank]``).  The last block past the copy resets the first
   block counter and publishes ``seq`` (arx.cu, the "last block publishes"
   step).
4. end barrier -- common.cuh, ``PullController::sync`` with the end stage
   (fenced): again one add per rank; rank r waits until
   ``flag - counter >= 2W`` and then sets ``counter = base + 2W``.
5. reduce -- arx.cu, ``arx_kernel`` reduce loop over ``slots[par][0..W-1]``
   in rank order (this model calls the oracle's ``reduce``).
6. exit -- triton_barrier.py, ``blockwise_barrier`` in Pattern 2 (relaxed):
   rank r sends to ``pad[t][b][r]`` by a 0 -> 1 compare-and-swap and waits on
   ``pad[r][b][t]`` by a 1 -> 0 compare-and-swap, for every t, so the pad is
   all zero again afterwards ("CUDA graph friendliness" in its docstring).
   Then ``PushController::exit`` flips ``epoch[r][b]`` and the last block out
   resets the second block counter and records ``seq`` as completed
   (arx.cu, "last block out").

Barrier variants (``sync``), with the same data path:

* ``"semaphore"`` -- the phases above.
* ``"pad"`` -- every barrier is triton_barrier.py's ``blockwise_barrier`` on
  the signal pad, in its three patterns: Pattern 0 for the start barrier,
  Pattern 1 (acq_rel) for the end barrier, Pattern 2 at exit.  The
  Semaphore flags and counters are not touched.
* ``"pad_fenced"`` -- as ``"pad"``; only the memory ordering of the start and
  exit barriers differs (acq_rel), which a sequential model does not see, so
  the words after a step are the same as for ``"pad"``.
* ``"semaphore_global"`` -- the same words as ``"semaphore"``: the two differ
  only in where a GPU holds the Semaphore flag during the step (global memory,
  or the shared memory of a thread-block cluster, loaded at entry and written
  back at exit) and in how the exit waits (the pad barrier above, or the
  cluster's hardware barrier, which leaves the pad at zero as well).
  common.cuh's ``PullController::sync`` fixes the arithmetic, not the place.
* ``"cluster"`` -- the single-GPU reading in which every barrier is a
  thread-block cluster's hardware barrier: no protocol word takes part.

All protocol words are unsigned 32-bit and wrap modulo 2**32, as the pages'
``uint32_t`` flags do (``flag - base`` in ``PullController::sync`` is an
unsigned difference).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import reduce as _reduce

MASK32 = 0xFFFFFFFF

# Status codes carried in the low 8 bits of the device error word.
ETIMEOUT = 4
ESTATE = 5


@dataclass
class State:
    W: int
    B: int
    seq: int = 0                      # last completed step
    published: int = 0                # last step whose slots were all staged
    err: int = 0                      # first error code (0 = none)
    blocks: list = field(default_factory=lambda: [0, 0])
    epoch: np.ndarray = None          # [W][B]  PushController parity
    flag: np.ndarray = None           # [W][B]  Semaphore flag
    counter: np.ndarray = None        # [W][B]  Semaphore counter
    pad: np.ndarray = None            # [W][B][W] signal pad: pad[owner][b][sender]
    slots: list = None                # slots[parity][r] -> uint16 array or None

    def __post_init__(self):
        if not (1 <= self.W <= 8) or self.B < 1:
            raise ValueError("need 1 <= W <= 8 and B >= 1")
        if self.epoch is None:
            self.epoch = np.zeros((self.W, self.B), dtype=np.int64)
        if self.flag is None:
            self.flag = np.zeros((self.W, self.B), dtype=np.int64)
        if self.counter is None:
            self.counter = np.zeros((self.W, self.B), dtype=np.int64)
        if self.pad is None:
            self.pad = np.zeros((self.W, self.B, self.W), dtype=np.int64)
        if self.slots is None:
            self.slots = [[None] * self.W for _ in range(2)]


def _set_err(st: State, code: int) -> None:
    if st.err == 0:
        st.err = code


SYNC_MODES = ("semaphore", "pad", "pad_fenced", "cluster", "semaphore_global")


def _pad_barrier(st: State, skip_rank: int | None = None) -> None:
    """triton_barrier.py ``blockwise_barrier`` for every block: rank r sends to
    ``pad[t][b][r]`` (0 -> 1) for every t, then waits on ``pad[r][b][t]``
    (1 -> 0) for every t.  A rank in ``skip_rank`` sends nothing, so the waits
    on its words expire (ETIMEOUT) and leave them at 0."""
    W, B = st.W, st.B
    for b in range(B):
        for r in range(W):          # sends: 0 -> 1
            if r == skip_rank:
                continue
            for t in range(W):
                if st.pad[t, b, r] != 0:
                    _set_err(st, ETIMEOUT)
                st.pad[t, b, r] = 1
        for r in range(W):          # waits: 1 -> 0
            for t in range(W):
                if st.pad[r, b, t] != 1:
                    _set_err(st, ETIMEOUT)
                st.pad[r, b, t] = 0


def step(st: State, inputs, skip_end_signal_rank: int | None = None,
         sync: str = "semaphore") -> np.ndarray:
    """Run one protocol step on ``st`` in place; return the bf16 output patterns.

    ``inputs`` is a sequence of W uint16 arrays of equal length.
    ``skip_end_signal_rank`` models a virtual rank that never sends its
    end-barrier signal (the host-side fault injection): every wait of that
    barrier then expires and the error word reports ETIMEOUT.  ``sync`` is
    the barrier variant (``SYNC_MODES``).
    """
    W, B = st.W, st.B
    if len(inputs) != W:
        raise ValueError("need one input per virtual rank")
    if sync not in SYNC_MODES:
        raise ValueError(f"unknown sync mode {sync!r}")
    # "cluster": the single-GPU reading in which the W blocks of a chunk form
    # one thread-block cluster and every barrier is its hardware barrier --
    # no protocol word takes part, and there is no signal to skip.
    cluster = sync == "cluster"
    if cluster and skip_end_signal_rank is not None:
        raise ValueError("the cluster barrier has no signal to skip")
    pad_mode = sync in ("pad", "pad_fenced")
    inputs = [np.ascontiguousarray(np.asarray(x, dtype=np.uint16)).reshape(-1) for x in inputs]

    # 1. seq / parity, and the per-block epoch check.
    seq = (st.seq + 1) & MASK32
    par = seq & 1
    expect_epoch = (seq - 1) & 1
    if np.any(st.epoch != expect_epoch):
        _set_err(st, ESTATE)

    # 2. start barrier: Semaphore start stage (unfenced): one add per rank,
    # wait for W -- or Pattern 0 of the pad barrier.
    if cluster:
        pass
    elif pad_mode:
        _pad_barrier(st)
    else:
        st.flag = (st.flag + W) & MASK32
        ok = ((st.flag - st.counter) & MASK32) >= W
        if not ok.all():
            _set_err(st, ETIMEOUT)

    # 3. stage rank r's input into slots[par][r]; last block publishes seq.
    for r in range(W):
        st.slots[par][r] = inputs[r].copy()
    st.blocks[0] = 0
    st.published = seq

    # 4. end barrier (fenced): Semaphore end stage -- one add per sending rank,
    # wait for 2W, advance counter -- or Pattern 1 of the pad barrier.
    if cluster:
        pass
    elif pad_mode:
        _pad_barrier(st, skip_end_signal_rank)
    else:
        senders = W - (1 if skip_end_signal_rank is not None else 0)
        st.flag = (st.flag + senders) & MASK32
        reached = ((st.flag - st.counter) & MASK32) >= 2 * W
        if not reached.all():
            _set_err(st, ETIMEOUT)
        st.counter = np.where(reached, (st.counter + 2 * W) & MASK32, st.counter)

    # 5. rank-order reduce of the staged slots.
    out = _reduce([st.slots[par][r] for r in range(W)])

    # 6. exit: zero-resetting pad barrier (Pattern 2; the cluster barrier in
    # the cluster reading), epoch flip, last block out.
    if not cluster:
        _pad_barrier(st)
    st.epoch = (st.epoch + 1) % 2
    st.blocks[1] = 0
    st.seq = seq
    return out

