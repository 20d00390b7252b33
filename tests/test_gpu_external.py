"""GPU tests of the external-writer form (``arx_ext_*``): a host thread writes
the partials, the GPU waits for its flags and reduces.

arx.cu's GB10 design (header comment, steps 1-3; ``arx_kernel``'s wait
phase and reduce loop): another agent writes every rank's partial into pinned
``recv[seq & 1][rank]`` and then raises ``flag[rank]``; the kernel waits for
the flags with system-scope acquires and reads the slots with
cache-bypassing loads.  Here a Python thread is that agent (the proxy and the
NIC), writing page-locked host memory while the GPU's steps run:

* 1,000 steps with fresh partials for every step, each output bit-exact
  against the oracle, the producer and the GPU running concurrently (the
  producer up to two steps ahead, as the two banks allow), then steps
  captured in a CUDA graph and replayed against the same producer;
* every W with ragged n and a misaligned output;
* a producer that withholds one rank's flag: the GPU's bounded wait
  expires, the host reads ARX_ETIMEOUT (stage 11, that rank), the next step
  is refused on the host, and the context recovers after ``arx_ext_reset``.
No GPU fault is involved: the failure is a flag the host never raises.
"""

import threading

import numpy as np
import pytest
import torch

import oracle
import synthetic_partials as sp
from test_gpu_reduce import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(arx):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return torch.device("cuda:0")


def _ext(arx, dev, W, max_n, nblocks=0):
    words = torch.zeros(arx.arx_ext_words_bytes(), dtype=torch.uint8, device=dev)
    region = torch.zeros(arx.arx_ext_region_bytes(W, max_n), dtype=torch.uint8).pin_memory()
    return arx.arx_ext_init(words, region, W, max_n, nblocks)


def _producer(arx, x, steps, first, parts, errors):
    """Posts steps first .. first + steps - 1: rank r of step s gets parts[s - first][r]."""
    try:
        W = parts.shape[1]
        n = parts.shape[2]
        for i in range(steps):
            for r in range(W):
                arx.arx_ext_post(x, r, first + i, parts[i, r].data_ptr(), n=n, wait_s=20.0)
    except Exception as e:  # surfaced by the test
        errors.append(e)


def test_thousand_steps_with_a_concurrent_host_producer(arx, dev):
    W, n, steps = 8, 8192 + 3, 1000
    parts = torch.empty(steps, W, n, dtype=torch.bfloat16)
    want = np.empty((steps, n), dtype=np.uint16)
    for s in range(steps):
        x = sp.partials(W, n, "normal", seed=50_000 + s)
        parts[s] = x
        want[s] = oracle.reduce(list(sp.to_u16_numpy(x)))
    x = _ext(arx, dev, W, n)
    arx.arx_ext_set_timeout(x, 100_000_000)     # a failed producer costs 0.1 s per step, not 1 s
    out = torch.zeros(steps, n, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream()
    errors = []
    th = threading.Thread(target=_producer, args=(arx, x, steps, 1, parts, errors))
    th.start()
    for s in range(steps):
        arx.arx_ext_step(x, out[s], stream=stream)
    th.join()
    assert not errors, errors
    st, seq, err = arx.arx_ext_query(x, stream=stream)
    assert (st, seq, err) == (arx.ARX_OK, steps, 0)
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    bad = np.flatnonzero((got != want).any(axis=1))
    assert bad.size == 0, f"{bad.size} of {steps} steps differ; first step {int(bad[0]) + 1}"

    # The same context, steps 1001..1300 replayed from a captured graph of 100.
    k, reps = 100, 3
    gout = torch.zeros(k, n, dtype=torch.bfloat16, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(k):
            arx.arx_ext_step(x, gout[i], stream=stream)
    for rep in range(reps):
        first = steps + 1 + rep * k
        th = threading.Thread(target=_producer, args=(arx, x, k, first, parts[rep * k:(rep + 1) * k], errors))
        th.start()
        with torch.cuda.stream(stream):
            g.replay()
        th.join()
        assert not errors, errors
        stream.synchronize()
        gg = gout.cpu().view(torch.int16).numpy().view(np.uint16)
        for i in range(k):
            assert_bits_equal(gg[i], want[rep * k + i], f"graph replay {rep} step {first + i}")
    assert arx.arx_ext_query(x, stream=stream)[:3] == (arx.ARX_OK, steps + reps * k, 0)


@pytest.mark.parametrize("W", range(1, 9))
def test_every_w_ragged_and_misaligned(arx, dev, W):
    for n, out_off in ((1, 0), (13, 1), (4096 + 5, 3), (131072, 0)):
        x = _ext(arx, dev, W, n)
        parts = sp.partials(W, n, "special", seed=60_000 + 10 * W + out_off)
        for r in range(W):
            arx.arx_ext_post(x, r, 1, parts[r])
        ob = torch.zeros(n + 8, dtype=torch.bfloat16, device=dev)
        out = ob[out_off:out_off + n]
        arx.arx_ext_step(x, out)
        assert arx.arx_ext_query(x)[:3] == (arx.ARX_OK, 1, 0)
        assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(parts))),
                          f"W={W} n={n} offset {out_off}")


def test_withheld_flag_times_out_and_the_context_recovers(arx, dev):
    W, n = 4, 4096
    x = _ext(arx, dev, W, n)
    arx.arx_ext_set_timeout(x, 20_000_000)        # 20 ms bound on the flag waits
    a = sp.partials(W, n, "normal", seed=7)
    out = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    for r in range(W):
        arx.arx_ext_post(x, r, 1, a[r])
    arx.arx_ext_step(x, out)
    assert arx.arx_ext_query(x)[:3] == (arx.ARX_OK, 1, 0)
    # Step 2: rank 2's writer never raises its flag.
    b = sp.partials(W, n, "normal", seed=8)
    for r in (0, 1, 3):
        arx.arx_ext_post(x, r, 2, b[r])
    arx.arx_ext_step(x, out)
    st, seq, err = arx.arx_ext_query(x)
    assert st == arx.ARX_ETIMEOUT and seq == 2
    assert err & 0xFF == arx.ARX_ETIMEOUT and (err >> 8) & 15 == 11 and (err >> 12) & 15 == 2
    # Refused on the host until reset: nothing is launched.
    sentinel = torch.full((n,), 3.0, dtype=torch.bfloat16, device=dev)
    assert arx.arx_ext_step(x, sentinel, check=False) == arx.ARX_ESTATE
    torch.cuda.synchronize()
    assert bool((sentinel == 3.0).all())
    arx.arx_ext_reset(x)
    assert x.failed_err == 0
    c = sp.partials(W, n, "normal", seed=9)
    for r in range(W):
        arx.arx_ext_post(x, r, 1, c[r])
    arx.arx_ext_step(x, out)
    assert arx.arx_ext_query(x)[:3] == (arx.ARX_OK, 1, 0)
    assert_bits_equal(out.cpu().view(torch.int16).numpy(), oracle.reduce(list(sp.to_u16_numpy(c))), "after reset")


def test_producer_waits_for_the_bank_to_be_consumed(arx, dev):
    # The producer may run two steps ahead; the third must wait until the GPU
    # has consumed the step whose bank it reuses (here: never, so it times out).
    W, n = 2, 1024
    x = _ext(arx, dev, W, n)
    p = sp.partials(W, n, "normal", seed=11)
    for s in (1, 2):
        for r in range(W):
            assert arx.arx_ext_post(x, r, s, p[r], wait_s=0.5) == arx.ARX_OK
    assert arx.arx_ext_post(x, 0, 3, p[0], wait_s=0.05, check=False) == arx.ARX_ETIMEOUT
    out = torch.zeros(2, n, dtype=torch.bfloat16, device=dev)
    arx.arx_ext_step(x, out[0])
    arx.arx_ext_step(x, out[1])
    assert arx.arx_ext_query(x)[:3] == (arx.ARX_OK, 2, 0)
    assert arx.arx_ext_wait_free(x, 3, wait_s=1.0) == arx.ARX_OK
    assert arx.arx_ext_wait_free(x, 4, wait_s=1.0) == arx.ARX_OK
    assert arx.arx_ext_wait_free(x, 5, wait_s=0.05, check=False) == arx.ARX_ETIMEOUT
