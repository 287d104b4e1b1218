"""The large-message two-shot TMA path at the bandwidth workload's sizes,
every element of every rank against the oracle.

Workload: R in {2, 4, 8, 16}, bf16 and fp32, 4, 16 and 64 MB per rank, and
256 MB per rank at R = 8; values normal(0, 1), seed 4, drawn on the device
(``inputs.draw_device``).  Each n is 3 elements short of the round size, so
the chunks, the per-CTA ranges and the tiles all end ragged, and the last
element run (shorter than 16 bytes) takes the element-by-element tail.  At
these sizes every CTA streams many tiles, so the stage ring and the
output-buffer ring wrap many times.

The oracle runs on the host (its multithreaded variant, the same bits as
one thread) on a copy of the device inputs; the comparison runs on the
device.  Sources: "SiFAR" (page 3), "Limits of existing algorithms" (two-shot
reduce-scatter / all-gather); "Every Microsecond Counts" (page 1), "Tensor
parallelism and AllReduce" (large messages are bandwidth-bound).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import ensure_built, status_ok

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
ES = {"bf16": 2, "fp32": 4}
POOL_MB = 64
RAGGED = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _int(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.fixture(scope="module")
def pools():
    """Per dtype: 16 ranks x 64 MB of inputs on the device and their host bits."""
    out = {}
    for dtype in ("bf16", "fp32"):
        n = (POOL_MB << 20) // ES[dtype]
        x = torch.stack(inputs.draw_device(4, 0 if dtype == "bf16" else 1, 16, n, "normal", 1.0, dtype))
        out[dtype] = (x, inputs.to_bits(x.cpu()))
    return out


def check_call(h, xs_dev, x_bits, R, n, dtype, ctx):
    """One twoshot_tma call on rank buffers xs_dev[r][:n] (host bits x_bits,
    [R, >= n]); every output element of every rank against the oracle's row."""
    ins = [xs_dev[r][:n] for r in range(R)]
    outs = [torch.empty_like(t) for t in ins]
    for o in outs:
        _int(o).fill_(-1)
    h.allreduce(ins, outs, "twoshot_tma")
    torch.cuda.synchronize()
    status_ok(h.h, ctx)
    want = oracle.allreduce(np.ascontiguousarray(x_bits[:R, :n]), threads=THREADS)[0]
    exp = torch.from_numpy(want.view(np.int16) if dtype == "bf16" else want.view(np.int32)).cuda()
    for r in range(R):
        eq = _int(outs[r]) == exp
        if not bool(eq.all()):
            bad = torch.nonzero(~eq).flatten()
            raise AssertionError(f"{ctx}: rank {r}: {bad.numel()} of {n} elements differ, first at {int(bad[0])}")
    return outs


@pytest.mark.parametrize("mb", [4, 16, 64])
@pytest.mark.parametrize("R", [2, 4, 8, 16])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_bandwidth_sizes_every_element(pools, dtype, R, mb):
    x, xb = pools[dtype]
    n = (mb << 20) // ES[dtype] - RAGGED
    h = sfar.Sfar(R, mb << 20, dtype)
    try:
        k, t = h.launch(n, "twoshot_tma")
        assert k >= 1 and t > 0
        check_call(h, [x[r] for r in range(R)], xb, R, n, dtype, f"R={R} {mb} MB {dtype}")
        # a second call on the same handle: the epochs and flags carry over
        rot = [(r + 1) % 16 for r in range(R)]
        check_call(h, [x[q] for q in rot], xb[rot, :n], R, n, dtype, f"R={R} {mb} MB {dtype} call 2")
    finally:
        h.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_256_mb_per_rank_r8(dtype):
    R, mb = 8, 256
    n = (mb << 20) // ES[dtype] - RAGGED
    xs = inputs.draw_device(4, 2 if dtype == "bf16" else 3, R, n, "normal", 1.0, dtype)
    xb = np.stack([inputs.to_bits(t.cpu()) for t in xs])
    h = sfar.Sfar(R, mb << 20, dtype)
    try:
        check_call(h, xs, xb, R, n, dtype, f"R=8 256 MB {dtype}")
    finally:
        h.close()
        del xs, xb
        torch.cuda.empty_cache()
