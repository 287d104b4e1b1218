"""The atomic-accumulation protocol (ll128_atomic) against the oracle.

Its binary32 adds run in the order of the hardware atomics, so most results
are compared against the oracle's admissible interval (``oracle.atomic``)
rather than bit for bit; what is unique is still compared exactly:
* every rank receives the same bits;
* sums whose partial sums are all exact (small integers, all-ones) equal the
  fixed-order fold bit for bit, in every order -- this catches a lost or
  doubled contribution anywhere;
* non-finite inputs give the class (NaN, +inf, -inf) every order gives.
The chains reuse accumulator lines thousands of times (cleared by their
owner after each use), under both launch modes and with a straggler.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import atomic
from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import assert_bits_equal, device_io, ensure_built, expected_bits, run_once, status_ok

pytestmark = pytest.mark.gpu
P = "ll128_atomic"
SIZES = [1, 3, 30, 31, 32, 62, 255, 1000, 4099, 7937, 65536 + 7]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def bits(t):
    b = inputs.to_bits(t.cpu())
    return b.view(np.uint32) if b.dtype == np.float32 else b


def assert_same_on_every_rank(outs, ctx):
    b0 = bits(outs[0])
    for r in range(1, len(outs)):
        assert np.array_equal(bits(outs[r]), b0), f"{ctx}: rank {r} differs from rank 0"


def assert_admissible(x_cpu, outs, ctx):
    x = inputs.to_bits(x_cpu)
    assert_same_on_every_rank(outs, ctx)
    ok = atomic.check(x, inputs.to_bits(outs[0].cpu()))
    if not ok.all():
        i = int(np.nonzero(~ok)[0][0])
        lo, hi = atomic.interval(x[:, i:i + 1])
        raise AssertionError(f"{ctx}: {int((~ok).sum())} of {ok.size} elements outside the interval; first at "
                             f"{i}: got {float(outs[0][i])} interval [{lo[0]}, {hi[0]}]")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [2, 3, 8, 16])
def test_within_bound_ragged_sizes(R, dtype):
    h = sfar.Sfar(R, 1 << 20, dtype)
    try:
        for n in SIZES:
            x = inputs.draw(300 + R, n, R, n, "normal", 1.0, dtype)
            assert_admissible(x, run_once(h, x, P), f"R={R} n={n} {dtype}")
    finally:
        h.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [2, 5, 8, 16])
def test_small_integers_bit_exact(R, dtype):
    h = sfar.Sfar(R, 1 << 20, dtype)
    try:
        for n in SIZES:
            x = inputs.draw(400 + R, n, R, n, "int", 16.0, dtype)
            assert_bits_equal(run_once(h, x, P), expected_bits(x), f"integers R={R} n={n} {dtype}")
    finally:
        h.close()


def test_all_ones_closed_form():
    for R in (2, 7, 16):
        h = sfar.Sfar(R, 1 << 16, "bf16")
        try:
            outs = run_once(h, torch.ones(R, 4097, dtype=torch.bfloat16), P)
            for o in outs:
                assert torch.all(o.float() == float(R))
        finally:
            h.close()


def test_wide_dynamic_range_and_subnormals():
    R, n = 8, 5000
    g = torch.Generator().manual_seed(17)
    mant = torch.randn(R, n, generator=g)
    expo = torch.randint(-140, 20, (R, n), generator=g).to(torch.float32)
    x = (mant * torch.pow(2.0, expo)).to(torch.float32)
    h = sfar.Sfar(R, 1 << 16, "fp32")
    try:
        assert_admissible(x, run_once(h, x, P), "wide range fp32")
        xb = x.to(torch.bfloat16)
    finally:
        h.close()
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        assert_admissible(xb, run_once(h, xb, P), "wide range bf16")
    finally:
        h.close()


def test_non_finite_inputs():
    R, n = 4, 999
    x = inputs.draw(18, 0, R, n, "normal", 1.0, "fp32")
    x[1, 10] = float("nan")
    x[0, 20], x[3, 20] = float("inf"), float("-inf")
    x[2, 30] = float("inf")
    x[3, 40] = float("-inf")
    h = sfar.Sfar(R, 1 << 16, "fp32")
    try:
        assert_admissible(x, run_once(h, x, P), "non-finite")
    finally:
        h.close()


def test_empty_and_geometry():
    h = sfar.Sfar(8, 1 << 20, "bf16")
    try:
        x = torch.zeros(8, 16, dtype=torch.bfloat16)
        ins, outs = device_io(x)
        before = [o.clone() for o in outs]
        assert sfar.sfar_allreduce(h.h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], 0,
                                   P) == sfar.SFAR_OK
        torch.cuda.synchronize()
        assert all(torch.equal(o, b) for o, b in zip(outs, before))
        for n in (1, 8192, 458752):
            k, t = h.launch(n, P)
            assert 1 <= k <= 128 and t in (64, 128, 256)
        for t in (64, 128, 256):
            assert sfar.sfar_test_set_geometry(h.h, 3, t) == sfar.SFAR_OK
            xi = inputs.draw(19, t, 8, 20000, "int", 8.0, "bf16")
            assert_bits_equal(run_once(h, xi, P), expected_bits(xi), f"geometry 3 x {t}")
        assert sfar.sfar_test_set_geometry(h.h, 0, 0) == sfar.SFAR_OK
        status_ok(h.h)
    finally:
        h.close()


# ------------------------------------------------------------ chained calls
def capture(h, x_dev, out_dev, calls):
    g = torch.cuda.CUDAGraph()
    R, n = x_dev.shape[1], x_dev.shape[2]
    with torch.cuda.graph(g):
        for c in range(calls):
            code = sfar.sfar_allreduce(h.h, [x_dev[c, r].data_ptr() for r in range(R)],
                                       [out_dev[c, r].data_ptr() for r in range(R)], n, P)
            assert code == sfar.SFAR_OK
    return g


def warm(h, R, n, dtype):
    x = torch.zeros(R, n, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)
    run_once(h, x, P)


@pytest.fixture(scope="module")
def int_chain():
    """The decode workload's shape (R = 8, 8192 bf16, 10,240 calls) with
    integer values, whose sum is unique in every order."""
    w = inputs.WORKLOADS["tp-decode-r8-16k"]
    x = torch.stack([inputs.draw(w.seed + 1000, c, w.R, w.n, "int", 16.0, w.dtype) for c in range(w.calls)])
    flat = inputs.to_bits(x.transpose(0, 1).reshape(w.R, w.calls * w.n))
    exp = oracle.allreduce(flat, threads=8)[0].reshape(w.calls, w.n)
    x_dev = x.cuda()
    del x
    return w, x_dev, torch.empty_like(x_dev), torch.from_numpy(exp.view(np.int16)).cuda()


def compare_rows(out, exp, ctx):
    got = out.view(torch.int16)
    for r in range(out.shape[1]):
        eq = got[:, r, :] == exp
        if not bool(eq.all()):
            bad = torch.nonzero(~eq.all(dim=1)).flatten()
            raise AssertionError(f"{ctx}: rank {r} differs in {bad.numel()} calls (first {int(bad[0])})")


@pytest.mark.parametrize("mode", ["serial", "overlap"])
def test_integer_chain_10240_calls(int_chain, mode):
    w, x_dev, out, exp = int_chain
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        h.set_mode(mode)
        warm(h, w.R, w.n, w.dtype)
        out.view(torch.int16).fill_(-1)
        g = capture(h, x_dev, out, w.calls)
        for rep in range(2):
            out.view(torch.int16).fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            status_ok(h.h, f"{mode} replay {rep}")
            compare_rows(out, exp, f"integer chain {mode} replay {rep}")
    finally:
        h.close()


@pytest.mark.parametrize("phase", [0, 1])
def test_integer_chain_overlap_with_straggler(int_chain, phase):
    w, x_dev, out, exp = int_chain
    calls = 2048
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        h.set_mode("overlap")
        warm(h, w.R, w.n, w.dtype)
        gen = torch.Generator().manual_seed(23)
        delays = torch.randint(0, 20001, (calls,), generator=gen).to(torch.int32).cuda()
        assert sfar.sfar_test_set_straggler(h.h, delays.data_ptr(), calls, -1, phase) == sfar.SFAR_OK
        out.view(torch.int16).fill_(-1)
        g = capture(h, x_dev[:calls], out[:calls], calls)
        g.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"straggler phase {phase}")
        compare_rows(out[:calls], exp[:calls], f"straggler phase {phase}")
    finally:
        h.close()


def test_decode_workload_chain_within_bound():
    """The decode workload itself (normal values) for 1,024 chained calls:
    ranks agree everywhere, and every element of 64 sampled calls is
    admissible."""
    w = inputs.WORKLOADS["tp-decode-r8-16k"]
    calls = 1024
    x = torch.stack([inputs.draw_workload_call(w, c) for c in range(calls)])
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        warm(h, w.R, w.n, w.dtype)
        x_dev = x.cuda()
        out = torch.empty_like(x_dev)
        g = capture(h, x_dev, out, calls)
        g.replay()
        torch.cuda.synchronize()
        status_ok(h.h)
        o16 = out.view(torch.int16)
        assert bool((o16 == o16[:, :1, :]).all()), "ranks disagree"
        for c in range(0, calls, calls // 64):
            ok = atomic.check(inputs.to_bits(x[c]), inputs.to_bits(out[c, 0].cpu()))
            assert ok.all(), f"call {c}: {int((~ok).sum())} elements outside the interval"
    finally:
        h.close()


def test_alternating_sizes_reuse_lines():
    R = 8
    h = sfar.Sfar(R, 1 << 20, "bf16")
    try:
        for i, n in enumerate([8192, 37, 65536 + 7, 31, 8192, 4099, 1, 131072, 62] * 3):
            x = inputs.draw(24, i, R, n, "int", 16.0, "bf16")
            assert_bits_equal(run_once(h, x, P), expected_bits(x), f"call {i} n={n}")
    finally:
        h.close()


def test_interleaved_with_exact_protocols():
    R, n = 8, 8192
    h = sfar.Sfar(R, 1 << 20, "bf16")
    try:
        for i in range(24):
            proto = [P, "ll", "twoshot", "ll128"][i % 4]
            x = inputs.draw(25, i, R, n, "int", 16.0, "bf16")
            assert_bits_equal(run_once(h, x, proto), expected_bits(x), f"{proto} call {i}")
    finally:
        h.close()


def test_dropped_rank_times_out_and_reset_recovers():
    R, n = 4, 6000
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        x = inputs.draw(26, 0, R, n, "int", 16.0, "bf16")
        run_once(h, x, P)
        ins, outs = device_io(x)
        assert sfar.sfar_test_set_timeout(h.h, 2_000_000) == sfar.SFAR_OK
        assert sfar.sfar_test_drop_rank(h.h, 2) == sfar.SFAR_OK
        h.allreduce(ins, outs, P)
        torch.cuda.synchronize()
        code, f = sfar.sfar_status_get(h.h)
        assert code == sfar.SFAR_ERR_TIMEOUT
        assert sfar.WAIT_NAMES[f.where] in ("counter", "ag") and 0 <= f.rank < R
        h.reset()
        assert sfar.sfar_test_drop_rank(h.h, -1) == sfar.SFAR_OK
        torch.cuda.synchronize()
        assert_bits_equal(run_once(h, x, P), expected_bits(x), "after reset")
    finally:
        h.close()
