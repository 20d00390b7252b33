"""GPU test of ``arx_step_noalloc``, the protocol step whose workspace is a
static device array inside the library.

That entry point serves callers that cannot allocate device memory when they
call it (an engine that reserved nearly all HBM for its own pool, a plug-in
whose framework owns every allocation, a serving loop that forbids allocating
after start-up).  Here it is called through the C ABI and checked bit for bit --
the tolerance every parity test in this suite uses -- against the existing
``arx_step`` on two calls in a row with different inputs, so a call that
leaked the previous call's state from the shared array would show.

This file is named to be collected last; it passes alone in a fresh process
and after the rest of the suite.
"""

import ctypes

import pytest
import torch

import synthetic_partials as sp

pytestmark = pytest.mark.gpu


def _noalloc(arx, inputs, out, n, status):
    ptrs = (ctypes.c_void_p * len(inputs))(*[t.data_ptr() for t in inputs])
    stream = torch.cuda.current_stream().cuda_stream
    return arx.lib.arx_step_noalloc(ptrs, len(inputs), out.data_ptr(), n,
                                    status.data_ptr() if status is not None else None, stream)


@pytest.mark.parametrize("W,n", [(8, 131072), (3, 4099)])
def test_noalloc_step_matches_arx_step_on_two_calls(arx, W, n):
    assert torch.cuda.is_available(), "this test needs a GPU"
    dev = torch.device("cuda:0")
    ws = torch.zeros(arx.arx_ctx_workspace_bytes(W, n), dtype=torch.uint8, device=dev)
    ctx = arx.arx_ctx_init(ws, W, n)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for call in range(2):
        x = sp.partials(W, n, "normal", seed=4 + call).to(dev)
        inputs = [x[r] for r in range(W)]
        want = torch.empty(n, dtype=torch.bfloat16, device=dev)
        arx.arx_step(ctx, inputs, want)
        got = torch.full((n,), float("nan"), dtype=torch.bfloat16, device=dev)
        status.fill_(-1)
        assert _noalloc(arx, inputs, got, n, status) == arx.ARX_OK, arx.arx_last_error()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"call {call} differs"
        assert int(status.item()) == 0, f"device error word {int(status.item()):#x}"
    st, seq, err = arx.arx_ctx_query(ctx)
    assert (st, seq, err) == (arx.ARX_OK, 2, 0)


def test_noalloc_rejects_sizes_beyond_its_limit(arx):
    dev = torch.device("cuda:0")
    n = arx.ARX_NOALLOC_MAX_N + 1
    x = torch.zeros(2, n, dtype=torch.bfloat16, device=dev)
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    assert _noalloc(arx, [x[0], x[1]], out, n, None) == arx.ARX_EINVAL
    assert "static scratch limit" in arx.arx_last_error()
