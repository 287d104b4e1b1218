"""Seeded synthetic inputs for the AllReduce workloads.

This module draws random numbers and nothing else: it holds none of the
reduction's arithmetic, so both the GPU path and the CPU oracle can take their
inputs from it.

Recipe (the same for every workload): call ``c`` of a workload with seed ``s``
draws its ``[R, n]`` block from its own CPU generator,
``torch.Generator().manual_seed(s * 2**32 + c)``; ``uniform`` is
``rand * 2 - 1`` (uniform on [-1, 1)), ``normal`` is ``randn * sigma``,
``int`` is a uniform integer in [-sigma, sigma] (sigma <= 256 keeps every
value exact in bf16); the binary32 draw is then rounded to nearest-even into
bf16, or kept as fp32.
Because every call has its own generator, any single call can be redrawn on
its own (the sampled parity checks at full size rely on this).  Values are
finite, so they never equal the sentinel bit patterns (all ones).

The large-message (bandwidth) workloads, 4-256 MB per rank, draw the same
distributions with the device's generator instead (:func:`draw_device`);
their bits reach the oracle by a copy to the host.
"""
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    R: int              # simulated ranks
    n: int              # elements per rank
    dtype: str          # "bf16" or "fp32"
    dist: str           # "uniform" (on [-1, 1)) or "normal"
    sigma: float        # standard deviation for "normal"
    seed: int
    calls: int          # calls in the workload

    @property
    def bytes_per_rank(self) -> int:
        return self.n * (2 if self.dtype == "bf16" else 4)


# The workloads of the tensor-parallel decode study.  Sizes follow the decode
# shape of "vLLM distributed inference core" (TP = 8, hidden 8192, 80 layers,
# two AllReduces per layer, i.e. 160 per token) and the message classes of
# "Every Microsecond Counts" (one-shot below 64 KB, two-shot from 64 KB to 1 MB).
WORKLOADS = {
    "small-r4-8k": Workload("small-r4-8k", 4, 4096, "bf16", "uniform", 1.0, 0, 100),
    "tp-decode-r8-16k": Workload("tp-decode-r8-16k", 8, 8192, "bf16", "normal", 1.0, 1, 160 * 64),
    "batched-decode-r8-896k": Workload("batched-decode-r8-896k", 8, 64 * 7168, "bf16", "normal", 0.5, 3, 64),
}

SWEEP_BYTES = [1 << 10, 4 << 10, 16 << 10, 64 << 10, 256 << 10, 1 << 20]   # per rank, seed 2
BANDWIDTH_BYTES = [4 << 20, 8 << 20, 16 << 20, 32 << 20, 64 << 20, 128 << 20, 256 << 20]  # seed 4


def call_generator(seed: int, call: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed) * (1 << 32) + int(call))


def draw(seed: int, call: int, R: int, n: int, dist: str = "uniform", sigma: float = 1.0,
         dtype: str = "bf16") -> torch.Tensor:
    """One call's inputs as a CPU tensor of shape [R, n] (bf16 or fp32)."""
    g = call_generator(seed, call)
    if dist == "uniform":
        x = torch.rand(R, n, generator=g) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(R, n, generator=g) * sigma
    elif dist == "int":
        k = int(sigma)
        x = torch.randint(-k, k + 1, (R, n), generator=g).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def draw_workload_call(w: Workload, call: int) -> torch.Tensor:
    return draw(w.seed, call, w.R, w.n, w.dist, w.sigma, w.dtype)


def draw_device(seed: int, call: int, R: int, n: int, dist: str = "normal", sigma: float = 1.0,
                dtype: str = "bf16", device="cuda") -> list:
    """Inputs of the large-message workloads (hundreds of MB per rank, too slow
    to draw on the host): R separate device buffers of n elements, drawn by
    the device's own generator seeded with ``seed * 2**32 + call``, one rank
    after another, with the same distributions and rounding as :func:`draw`.
    The bit patterns differ from :func:`draw`'s; both sides of a comparison
    read the same buffers (the oracle after a copy to the host)."""
    g = torch.Generator(device=device).manual_seed(int(seed) * (1 << 32) + int(call))
    out = []
    for _ in range(R):
        if dist == "uniform":
            x = torch.rand(n, generator=g, device=device) * 2.0 - 1.0
        elif dist == "normal":
            x = torch.randn(n, generator=g, device=device) * sigma
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        out.append(x.to(torch.bfloat16) if dtype == "bf16" else x)
    return out


def to_bits(x: torch.Tensor) -> np.ndarray:
    """A CPU tensor as the numpy array the oracle takes: uint16 bit patterns for
    bf16, float32 for fp32."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    if x.dtype == torch.float32:
        return x.numpy()
    raise TypeError(f"unsupported dtype {x.dtype}")


def from_bits(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    if a.dtype == np.float32:
        return torch.from_numpy(a.copy())
    raise TypeError(f"unsupported dtype {a.dtype}")
