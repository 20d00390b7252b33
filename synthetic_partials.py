"""Seeded synthetic bf16 partials for the W-way deterministic reduce workloads.

This module only draws numbers and rounds them to bf16 with torch's own
float32 -> bfloat16 conversion.  It holds none of the reduce's arithmetic.  It
is the one piece of code that both sides of every parity check use: the CPU
oracle and the CUDA path consume exactly the 16-bit patterns returned here.

Every generator is a CPU ``torch.Generator`` seeded explicitly, so the bits
are a pure function of (workload, seed).  The shapes and value distributions
are those of the workloads the one-shot all-reduce is meant for
(arx.cu, header comment and ``kMaxBytes``: a decode-sized bf16 [32, 4096]
message per rank, at most 8 ranks), widened to large bandwidth-bound sizes.

Workloads (name -> recipe):

* ``w2_32x4096_uniform``   W=2, bf16 [32,4096], uniform [-1, 1), seed 0.
* ``w8_32x4096_normal``    W=8, bf16 [32,4096], normal(0, 1), seed 1.
* ``w4_1024x8192_alias``   W=4, bf16 [1024,8192], normal(0, 0.02), seed 2;
                           the output aliases slot 0.
* ``w8_sweep_int``         W=8, n = 2**k for k in 9..27, integers uniform in
                           {-8..8}, seed 3 (sums are exact in fp32 and bf16).
* ``w8_32x4096_graph``     W=8, bf16 [32,4096], normal(0, 1), step s drawn
                           from seed 4 + s (10,000 steps in one CUDA graph).

``partials(...)`` returns a CPU ``torch.bfloat16`` tensor of shape [W, n].
``bits(t)`` views any bf16 tensor as int16 so that comparisons are bitwise.
"""

from __future__ import annotations

import torch

N_32x4096 = 32 * 4096
N_1024x8192 = 1024 * 8192
SWEEP_LOG2 = tuple(range(9, 28))
GRAPH_STEPS = 10_000

# Integer draws are produced in fixed chunks so that the sequence consumed from
# the generator does not depend on how large the request is.
_INT_CHUNK = 1 << 24

WORKLOADS = {
    "w2_32x4096_uniform": dict(W=2, n=N_32x4096, dist="uniform", seed=0, alias=False),
    "w8_32x4096_normal": dict(W=8, n=N_32x4096, dist="normal", seed=1, alias=False),
    "w4_1024x8192_alias": dict(W=4, n=N_1024x8192, dist="normal0.02", seed=2, alias=True),
    "w8_sweep_int": dict(W=8, n=None, dist="int8", seed=3, alias=False),
    "w8_32x4096_graph": dict(W=8, n=N_32x4096, dist="normal", seed=4, alias=False),
}

DISTS = ("uniform", "normal", "normal0.02", "int8", "special")


def _draw_float(shape, dist: str, g: torch.Generator) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "normal0.02":
        return torch.randn(shape, generator=g, dtype=torch.float32) * 0.02
    raise ValueError(f"unknown float distribution {dist!r}")


def _draw_int8(W: int, n: int, g: torch.Generator) -> torch.Tensor:
    flat = torch.empty(W * n, dtype=torch.int8)
    for lo in range(0, W * n, _INT_CHUNK):
        hi = min(lo + _INT_CHUNK, W * n)
        flat[lo:hi].random_(-8, 9, generator=g)
    # Small integers are exactly representable in bf16; torch's conversion is exact here.
    return flat.view(W, n).to(torch.bfloat16)


def _draw_special(W: int, n: int, g: torch.Generator) -> torch.Tensor:
    """Random bf16 bit patterns biased toward the hard cases of the sum.

    Mixes uniformly random 16-bit patterns (every exponent, subnormals, +-inf,
    NaN) with +-0, +-1, values one ulp apart and large exponent gaps.
    """
    raw = torch.randint(0, 1 << 16, (W, n), generator=g, dtype=torch.int32)
    pick = torch.randint(0, 8, (W, n), generator=g, dtype=torch.int32)
    specials = torch.tensor(
        [0x0000, 0x8000, 0x3F80, 0xBF80, 0x3F81, 0x4B00, 0x0001, 0x7F7F],
        dtype=torch.int32)
    sidx = torch.randint(0, len(specials), (W, n), generator=g, dtype=torch.int32)
    out = torch.where(pick < 5, raw, specials[sidx.long()])
    return (out - ((out >= 0x8000).int() << 16)).to(torch.int16).view(torch.bfloat16)


def partials(W: int, n: int, dist: str, seed: int) -> torch.Tensor:
    """[W, n] bf16 partials on the CPU, a pure function of the arguments."""
    if W < 0 or n < 0:
        raise ValueError("W and n must be non-negative")
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    if dist == "int8":
        return _draw_int8(W, n, g)
    if dist == "special":
        return _draw_special(W, n, g)
    return _draw_float((W, n), dist, g).to(torch.bfloat16)


def workload(name: str, n: int | None = None, step: int = 0) -> tuple[torch.Tensor, bool]:
    """(partials [W, n] bf16 CPU, out_aliases_slot0) for a named workload.

    ``n`` is required for the size sweep; ``step`` picks the per-step seed of
    the graph workload (seed 4 + step).
    """
    spec = WORKLOADS[name]
    size = spec["n"] if n is None else n
    if size is None:
        raise ValueError(f"workload {name} needs an explicit n")
    seed = spec["seed"] + (step if name == "w8_32x4096_graph" else 0)
    return partials(spec["W"], size, spec["dist"], seed), spec["alias"]


def graph_step_partials(step: int, W: int = 8, n: int = N_32x4096) -> torch.Tensor:
    """Fresh normal(0, 1) partials of one protocol step, drawn from seed 4 + step."""
    return partials(W, n, "normal", 4 + step)


def bits(t: torch.Tensor) -> torch.Tensor:
    """The raw 16-bit patterns of a bf16 tensor, as int16 (no copy)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return t.view(torch.int16)


def to_u16_numpy(t: torch.Tensor):
    """The bit patterns of a CPU bf16 tensor as a contiguous numpy uint16 array."""
    return bits(t.contiguous()).numpy().view("uint16")
