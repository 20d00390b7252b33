"""Host buffers the CPU rewrites between GPU calls (NVLink-C2C coherence).

arx.cu reads buffers that another agent writes (there the NIC, through the
CPU proxy) with cache-bypassing loads, because a cached copy of an earlier
step's data would be summed again.  On GB300 the direct host-buffer form of
the reduce reads page-locked host memory over NVLink-C2C, and the GPU may
keep lines of host memory it read in its caches.  These tests rewrite the
same page-locked buffers from the CPU between calls -- eager calls and
replays of one captured graph -- and check every output bit for bit against
the oracle, so a stale line from the previous call would show:

* ``arx_reduce_host`` (direct form) with a separate host output, and in place
  (the output one of the partials);
* ``arx_step`` whose inputs are page-locked host buffers rewritten by the
  CPU, with the slot banks in device memory and in page-locked host memory;
* chained calls, each reading the previous call's output, on device and on
  page-locked host buffers (the L2 prefetch issued before the dependency
  wait touches the buffer the predecessor is still writing).
"""

import pytest
import torch

import oracle
import synthetic_partials as sp
from test_gpu_reduce import assert_bits_equal

pytestmark = pytest.mark.gpu

CALLS = 100


@pytest.fixture(scope="module")
def dev(arx):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return torch.device("cuda:0")


def _fresh(W, n, k, seed0):
    """k rounds of partials (alternating distributions) and their oracle sums."""
    xs, wants = [], []
    for i in range(k):
        x = sp.partials(W, n, "special" if i % 2 else "normal", seed=seed0 + i)
        xs.append(x)
        wants.append(oracle.reduce(list(sp.to_u16_numpy(x)), threads=4))
    return xs, wants


@pytest.mark.parametrize("in_place", [False, True])
def test_reduce_host_rereads_rewritten_partials(arx, dev, in_place):
    W, n = 8, 131072 + 3
    xs, wants = _fresh(W, n, 8, 31_000 + 100 * in_place)
    host = torch.empty(W, n, dtype=torch.bfloat16).pin_memory()
    hout = host[0] if in_place else torch.empty(n, dtype=torch.bfloat16).pin_memory()
    slots = [host[r] for r in range(W)]
    s = torch.cuda.Stream()
    # Eager calls, the CPU rewriting the same page-locked partials between them.
    for i in range(CALLS):
        host.copy_(xs[i % len(xs)])
        if not in_place:
            hout.fill_(0)
        arx.arx_reduce_host(slots, hout, stream=s)
        s.synchronize()
        assert_bits_equal(hout.view(torch.int16).numpy(), wants[i % len(xs)], f"eager call {i}")
    # One captured call replayed, the partials rewritten between replays.
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        arx.arx_reduce_host(slots, hout, stream=s)
    for i in range(CALLS):
        host.copy_(xs[(i + 3) % len(xs)])
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert_bits_equal(hout.view(torch.int16).numpy(), wants[(i + 3) % len(xs)], f"replay {i}")


@pytest.mark.parametrize("slots_where", ["device", "host"])
def test_step_rereads_rewritten_host_inputs(arx, dev, slots_where):
    # The step's inputs are page-locked host buffers (passed by their device
    # addresses), rewritten by the CPU between steps; the slot banks in device
    # memory or in page-locked host memory.  The partials total just over
    # 4 MiB, above the size up to which the step asks L2 to prefetch its
    # inputs (that hint is meant for device memory).
    W, n = 8, (1 << 18) + 5
    xs, wants = _fresh(W, n, 6, 32_000 + 100 * (slots_where == "host"))
    words = torch.zeros(arx.arx_ctx_words_bytes(W), dtype=torch.uint8, device=dev)
    sb = arx.arx_ctx_slots_bytes(W, n)
    slot_buf = torch.empty(sb, dtype=torch.uint8).pin_memory() if slots_where == "host" else \
        torch.empty(sb, dtype=torch.uint8, device=dev)
    ctx = arx.arx_ctx_init_split(words, slot_buf, W, n)
    host = torch.empty(W, n, dtype=torch.bfloat16).pin_memory()
    ins = [host[r].data_ptr() for r in range(W)]      # page-locked: same address on the device
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    for i in range(CALLS):
        host.copy_(xs[i % len(xs)])
        arx.arx_step(ctx, ins, out, n=n, stream=s)
        s.synchronize()
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), wants[i % len(xs)], f"step {i}")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        arx.arx_step(ctx, ins, out, n=n, stream=s)
    for i in range(CALLS):
        host.copy_(xs[(i + 1) % len(xs)])
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), wants[(i + 1) % len(xs)], f"replayed step {i}")
    st, seq, err = arx.arx_ctx_query(ctx, stream=s)
    assert (st, seq, err) == (arx.ARX_OK, 2 * CALLS, 0)


@pytest.mark.parametrize("where", ["device", "host"])
def test_chained_calls_read_their_predecessors_output(arx, dev, where):
    # Each call's output is the next call's first partial, enqueued back to
    # back on one stream (and replayed from one captured graph).  The reduce
    # prefetches its partials into L2 before it waits for its predecessor,
    # so here the prefetch touches a buffer the predecessor is still
    # writing; the loads after the wait must see the finished sum.  Device
    # buffers through arx_reduce, page-locked host buffers through
    # arx_reduce_host.
    W, n, steps = 4, 131072 + 3, 24
    x = sp.partials(W, n, "normal", seed=33_000 + (where == "host"))
    u = list(sp.to_u16_numpy(x))
    wants, first = [], u[0]
    for _ in range(steps):
        first = oracle.reduce([first] + u[1:], threads=4)
        wants.append(first)
    if where == "device":
        parts = x.to(dev)
        outs = torch.zeros(steps, n, dtype=torch.bfloat16, device=dev)
    else:
        parts = x.clone().pin_memory()
        outs = torch.zeros(steps, n, dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.Stream()

    def run():
        for k in range(steps):
            slots = [outs[k - 1] if k else parts[0]] + [parts[r] for r in range(1, W)]
            if where == "device":
                arx.arx_reduce(slots, outs[k], stream=s)
            else:
                arx.arx_reduce_host(slots, outs[k], stream=s)

    run()
    s.synchronize()
    for k in range(steps):
        assert_bits_equal(outs[k].cpu().view(torch.int16).numpy(), wants[k], f"{where} eager call {k}")
    g = torch.cuda.CUDAGraph()
    outs.zero_() if where == "device" else outs.fill_(0)
    with torch.cuda.graph(g, stream=s):
        run()
    for rep in range(3):
        outs.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        for k in range(steps):
            assert_bits_equal(outs[k].cpu().view(torch.int16).numpy(), wants[k], f"{where} replay {rep} call {k}")
