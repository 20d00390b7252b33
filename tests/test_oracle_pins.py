"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

* rounding fp32 -> bf16 over all 2**32 binary32 patterns against torch's
  library conversion (round to nearest even; NaN compared by NaN-ness);
* widening over all 2**16 bf16 patterns against torch's conversion;
* the rank-order reduce against an exact rational model of IEEE arithmetic
  (``exact_ieee``) on random and adversarial tiny inputs;
* integer-valued inputs whose sums are exact, against an int64 sum;
* the W = 1 identity, all-zero and signed-zero inputs;
* hand-derived single-element fixtures in ``tests/golden/reduce_cases.txt``.

The definition being pinned is arx.cu, ``arx_kernel``'s reduce loop: an fp32
accumulator from +0, rank-order adds, one rounding to bf16.
"""

import os

import numpy as np
import pytest
import torch

import oracle
import synthetic_partials as sp
from exact_ieee import rank_order_sum_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "reduce_cases.txt")


def _torch_round_bf16(f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _is_nan16(b: np.ndarray) -> np.ndarray:
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def test_fp_env_round_to_nearest_and_subnormals():
    assert oracle.lib().oracle_fp_env_ok() == 1


def test_round_bf16_all_binary32_patterns():
    chunk = 1 << 26
    for first in range(0, 1 << 32, chunk):
        got = oracle.round_bf16_patterns(first, chunk)
        f = np.arange(first, first + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        want = _torch_round_bf16(f)
        nan_g, nan_w = _is_nan16(got), _is_nan16(want)
        assert np.array_equal(nan_g, nan_w), f"NaN-ness differs in chunk {first:#x}"
        ok = nan_g | (got == want)
        if not ok.all():
            i = int(np.flatnonzero(~ok)[0])
            pytest.fail(f"pattern {first + i:#010x}: oracle {got[i]:#06x} torch {want[i]:#06x}")


def test_round_bf16_nan_encoding_keeps_sign():
    f = np.array([0x7FC00001, 0xFFC00001, 0x7F800001, 0xFF800001], dtype=np.uint32).view(np.float32)
    got = oracle.round_bf16(f)
    assert list(got) == [0x7FC0, 0xFFC0, 0x7FC0, 0xFFC0]


def test_widen_all_bf16_patterns():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen_bf16(b)
    want = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got.view(np.uint32)[~nan], want.view(np.uint32)[~nan])


def test_host_add_matches_numpy_binary32():
    rng = np.random.default_rng(7)
    a = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    b = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    with np.errstate(all="ignore"):
        want = (a + b).astype(np.float32)
    for x, y, w in zip(a[:4000], b[:4000], want[:4000]):
        g = np.float32(oracle.add_f32(float(x), float(y)))
        if np.isnan(w):
            assert np.isnan(g)
        else:
            assert g.view(np.uint32) == w.view(np.uint32)


def _load_golden():
    cases = []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split(";")[0].strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            toks = lhs.split()
            W = int(toks[0])
            vals = [int(t, 16) for t in toks[1:]]
            assert len(vals) == W, line
            cases.append((vals, int(rhs.strip(), 16)))
    return cases


GOLDEN_CASES = _load_golden()


@pytest.mark.parametrize("vals,want", GOLDEN_CASES, ids=[f"g{i}" for i in range(len(GOLDEN_CASES))])
def test_golden_fixture(vals, want):
    slots = [np.array([v], dtype=np.uint16) for v in vals]
    got = int(oracle.reduce(slots)[0])
    assert got == want, f"{[hex(v) for v in vals]}: oracle {got:#06x}, fixture {want:#06x}"


def test_golden_fixtures_agree_with_exact_model():
    # The hand derivations and the exact rational model must agree too.
    for vals, want in GOLDEN_CASES:
        assert rank_order_sum_bits(vals) == want, [hex(v) for v in vals]


@pytest.mark.parametrize("W", [1, 2, 3, 5, 8])
def test_reduce_matches_exact_rational_model(W):
    x = sp.partials(W, 300, "special", seed=100 + W)
    u = sp.to_u16_numpy(x)
    got = oracle.reduce(list(u))
    for i in range(u.shape[1]):
        want = rank_order_sum_bits([int(u[r, i]) for r in range(W)])
        if want is None:
            assert _is_nan16(got[i:i + 1])[0], f"element {i}: expected NaN"
        else:
            assert int(got[i]) == want, (
                f"element {i} inputs {[hex(int(u[r, i])) for r in range(W)]}: "
                f"oracle {int(got[i]):#06x} exact model {want:#06x}")


@pytest.mark.parametrize("W", [1, 2, 4, 8])
def test_integer_inputs_sum_exactly(W):
    x = sp.partials(W, 1 << 16, "int8", seed=3)
    u = sp.to_u16_numpy(x)
    ints = x.to(torch.int64).sum(dim=0)                 # exact integer sum
    want = ints.to(torch.float32).to(torch.bfloat16)    # |sum| <= 64 is exact in bf16
    got = oracle.reduce(list(u))
    assert np.array_equal(got, sp.to_u16_numpy(want))


def test_wider_integer_sums_round_once():
    # Integers in [-128, 128]: every partial sum is exact in fp32 (< 2**24), so
    # the only rounding is the final one to bf16, done here by torch.
    g = torch.Generator().manual_seed(11)
    ints = torch.randint(-128, 129, (8, 50000), generator=g)
    x = ints.to(torch.bfloat16)
    assert torch.equal(x.to(torch.int64), ints)
    want = ints.sum(dim=0).to(torch.float32).to(torch.bfloat16)
    got = oracle.reduce(list(sp.to_u16_numpy(x)))
    assert np.array_equal(got, sp.to_u16_numpy(want))


def test_w1_identity_except_negative_zero():
    x = sp.partials(1, 1 << 16, "special", seed=5)
    u = sp.to_u16_numpy(x)[0]
    got = oracle.reduce([u])
    nan = _is_nan16(u)
    assert np.array_equal(_is_nan16(got), nan)
    want = np.where(u == 0x8000, np.uint16(0), u)
    assert np.array_equal(got[~nan], want[~nan])


def test_all_zero_and_negative_zero_inputs_give_positive_zero():
    for W in (1, 2, 8):
        z = np.zeros((W, 1000), dtype=np.uint16)
        assert not oracle.reduce(list(z)).any()
        nz = np.full((W, 1000), 0x8000, dtype=np.uint16)
        assert not oracle.reduce(list(nz)).any()


def test_in_place_output_aliasing_slot0():
    x = sp.to_u16_numpy(sp.partials(4, 4096, "normal0.02", seed=2))
    want = oracle.reduce(list(x))
    slots = [x[r].copy() for r in range(4)]
    oracle.reduce(slots, out=slots[0])
    assert np.array_equal(slots[0], want)


def test_multithreaded_reduce_is_identical():
    x = sp.to_u16_numpy(sp.partials(8, 300001, "normal", seed=1))
    a = oracle.reduce(list(x), threads=1)
    b = oracle.reduce(list(x), threads=7)
    c = oracle.reduce_rows(x, threads=3)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_reduce_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.reduce([])
    with pytest.raises(ValueError):
        oracle.reduce([np.zeros(3, np.uint16), np.zeros(4, np.uint16)])
    with pytest.raises(TypeError):
        oracle.reduce([np.zeros(3, np.float32)])
