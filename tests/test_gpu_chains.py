"""Graph-chained calls at the workloads' full sizes: bit-exact over 10,240
calls, under both launch modes, with a straggler, and the failure paths
(a dropped rank, the sentinel precondition, a single-buffered overlap)."""
import os

import numpy as np
import pytest
import torch

import oracle
from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import (ALL_PROTOS, DOUBLE_BUFFERED, ONESHOT, assert_bits_equal, device_io, ensure_built,
                         expected_bits, status_ok)

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def draw_calls(w, calls):
    return torch.stack([inputs.draw_workload_call(w, c) for c in range(calls)])   # [calls, R, n] CPU


def expected_rows(x):
    """Oracle result of every call: [calls, n] bits (all ranks get the same row)."""
    calls, R, n = x.shape
    flat = inputs.to_bits(x.transpose(0, 1).reshape(R, calls * n))
    return oracle.allreduce(flat, threads=THREADS)[0].reshape(calls, n)


def compare_chain(out_dev, exp_rows, ctx):
    """out_dev [calls, R, n] on the device vs exp_rows [calls, n] (host bits)."""
    calls, R, n = out_dev.shape
    exp = torch.from_numpy(exp_rows.view(np.int16) if exp_rows.dtype == np.uint16 else exp_rows.view(np.int32))
    exp = exp.cuda()
    got = out_dev.view(torch.int16) if out_dev.dtype == torch.bfloat16 else out_dev.view(torch.int32)
    for r in range(R):
        eq = got[:, r, :] == exp
        if not bool(eq.all()):
            bad_calls = torch.nonzero(~eq.all(dim=1)).flatten()
            raise AssertionError(f"{ctx}: rank {r} differs in {bad_calls.numel()} of {calls} calls "
                                 f"(first call {int(bad_calls[0])})")


def capture_chain(h, x_dev, out_dev, proto, calls):
    g = torch.cuda.CUDAGraph()
    R, n = x_dev.shape[1], x_dev.shape[2]
    with torch.cuda.graph(g):
        for c in range(calls):
            code = sfar.sfar_allreduce(h.h, [x_dev[c, r].data_ptr() for r in range(R)],
                                       [out_dev[c, r].data_ptr() for r in range(R)], n, proto)
            assert code == sfar.SFAR_OK
    return g


def warm(h, proto, R, n, dtype):
    x = torch.zeros(R, n, dtype=inputs_dtype(dtype))
    ins, outs = device_io(x)
    h.allreduce(ins, outs, proto)
    torch.cuda.synchronize()
    status_ok(h.h, "warm-up " + proto)


def inputs_dtype(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


# ------------------------------------------------------------ small workload
def test_small_r4_100_calls_ll():
    w = inputs.WORKLOADS["small-r4-8k"]
    x = draw_calls(w, w.calls)
    exp = expected_rows(x)
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        warm(h, "ll", w.R, w.n, w.dtype)
        x_dev = x.cuda()
        out = torch.full_like(x_dev, float("nan"))
        g = capture_chain(h, x_dev, out, "ll", w.calls)
        g.replay()
        torch.cuda.synchronize()
        status_ok(h.h)
        compare_chain(out, exp, "small-r4-8k ll")
    finally:
        h.close()


# -------------------------------------------------- decode chain, 10,240 calls
@pytest.fixture(scope="module")
def decode_chain():
    w = inputs.WORKLOADS["tp-decode-r8-16k"]
    x = draw_calls(w, w.calls)
    exp = expected_rows(x)
    x_dev = x.cuda()
    del x
    out = torch.empty_like(x_dev)
    return w, x_dev, out, exp


@pytest.mark.parametrize("mode", ["serial", "overlap", "cooperative"])
@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_decode_chain_10240_calls(decode_chain, proto, mode):
    w, x_dev, out, exp = decode_chain
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        h.set_mode(mode)
        warm(h, proto, w.R, w.n, w.dtype)
        out.view(torch.int16).fill_(-1)
        g = capture_chain(h, x_dev, out, proto, w.calls)
        g.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"{proto} {mode}")
        compare_chain(out, exp, f"decode chain {proto} {mode}")
        # replay again: the epochs keep counting on the device
        out.view(torch.int16).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"{proto} {mode} replay 2")
        compare_chain(out, exp, f"decode chain {proto} {mode} replay 2")
    finally:
        h.close()


@pytest.fixture(scope="module")
def fused_decode_chain(decode_chain):
    """The fused AllReduce + residual add + RMSNorm over the decode chain: call
    c reduces the decode workload's call c (one row of 8192 bf16 per rank)
    with call (c + 1) mod 10,240 as its residual; weight normal(0, 1) seed 8.
    Returns the device buffers and the oracle's y and z, [R, calls, n] each
    (computed on the host in blocks of rows, one thread per block)."""
    import concurrent.futures as cf
    w, x_dev, _, _ = decode_chain
    calls, R, n = x_dev.shape
    eps = 1e-5
    wt = inputs.draw(8, 0, 1, n, "normal", 1.0, "bf16")[0]
    xb = inputs.to_bits(x_dev.cpu())                              # [calls, R, n]
    X = np.ascontiguousarray(xb.transpose(1, 0, 2))               # [R, calls, n]
    RES = np.roll(X, -1, axis=1)
    wb = inputs.to_bits(wt[None, :])[0]
    ys, zs = np.empty_like(X), np.empty_like(X)
    step = -(-calls // THREADS)

    def block(b0):
        b1 = min(calls, b0 + step)
        y, z = oracle.add_rmsnorm(X[:, b0:b1].reshape(R, -1), RES[:, b0:b1].reshape(R, -1), wb, eps, n)
        ys[:, b0:b1] = y.reshape(R, b1 - b0, n)
        zs[:, b0:b1] = z.reshape(R, b1 - b0, n)

    with cf.ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(block, range(0, calls, step)))
    del X, RES, xb
    return wt.cuda(), eps, ys, zs


@pytest.mark.parametrize("mode", ["serial", "overlap", "cooperative"])
def test_fused_decode_chain_10240_calls(decode_chain, fused_decode_chain, mode):
    """10,240 fused calls (R = 8, one row of 8192 bf16) in one graph, replayed
    twice, every rank of every call bit for bit against the oracle."""
    w, x_dev, _, _ = decode_chain
    wd, eps, ys, zs = fused_decode_chain
    calls, R, n = x_dev.shape
    y = torch.empty_like(x_dev)
    z = torch.empty_like(x_dev)
    h = sfar.Sfar(R, 2 * n, "bf16")
    try:
        h.set_mode(mode)
        P = lambda t, c: [t[c, r].data_ptr() for r in range(R)]
        assert sfar.sfar_allreduce_add_rmsnorm(h.h, P(x_dev, 0), P(x_dev, 1), wd.data_ptr(), P(y, 0), P(z, 0), 1, n,
                                               eps) == sfar.SFAR_OK
        torch.cuda.synchronize()
        status_ok(h.h, "fused warm-up")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in range(calls):
                code = sfar.sfar_allreduce_add_rmsnorm(h.h, P(x_dev, c), P(x_dev, (c + 1) % calls), wd.data_ptr(),
                                                       P(y, c), P(z, c), 1, n, eps)
                assert code == sfar.SFAR_OK
        ey = torch.from_numpy(ys.view(np.int16)).cuda()
        ez = torch.from_numpy(zs.view(np.int16)).cuda()
        for rep in range(2):
            y.view(torch.int16).fill_(-1)
            z.view(torch.int16).fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            status_ok(h.h, f"fused {mode} replay {rep}")
            for name, got, want in (("y", y, ey), ("z", z, ez)):
                eq = (got.view(torch.int16).transpose(0, 1) == want).all(dim=2)      # [R, calls]
                if not bool(eq.all()):
                    r, c = (int(v) for v in torch.nonzero(~eq)[0])
                    raise AssertionError(f"fused {mode} replay {rep}: {name} differs in "
                                         f"{int((~eq).sum())} (rank, call) pairs, first rank {r} call {c}")
        del g
    finally:
        h.close()


def straggler_delays(calls, seed=3, hi_ns=20000):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, hi_ns + 1, (calls,), generator=g, dtype=torch.int64).to(torch.int32).cuda()


@pytest.mark.parametrize("phase", [0, 1])
@pytest.mark.parametrize("proto", DOUBLE_BUFFERED + ["twoshot_tma"])
def test_decode_chain_overlap_with_straggler(decode_chain, proto, phase):
    """All 10,240 calls of the decode chain in one graph, in overlap mode, with
    a straggler rank (call mod R) delayed 0-20 us per call: calls overtake one
    another across ranks, and double buffering (the arrival and completion
    flags for the TMA path, which has no receive buffers) keeps every call
    exact."""
    w, x_dev, out, exp = decode_chain
    calls = w.calls
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        h.set_mode("overlap")
        delays = straggler_delays(calls)
        assert sfar.sfar_test_set_straggler(h.h, delays.data_ptr(), calls, -1, phase) == sfar.SFAR_OK
        warm(h, proto, w.R, w.n, w.dtype)
        out.view(torch.int16).fill_(-1)
        g = capture_chain(h, x_dev, out, proto, calls)
        g.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"{proto} straggler phase {phase}")
        compare_chain(out[:calls], exp[:calls], f"{proto} overlap straggler phase {phase}")
    finally:
        h.close()


@pytest.mark.parametrize("proto", ["db", "ll"])
def test_single_buffer_overlap_fails_detectably(decode_chain, proto):
    """Negative test of double buffering: with one buffer, a slow reader and
    overlapping calls, a fast peer overwrites data before it is read.  The
    result must be a detected timeout or a detected mismatch, never a hang."""
    w, x_dev, out, exp = decode_chain
    calls = 640
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        h.set_mode("overlap")
        assert sfar.sfar_test_set_timeout(h.h, 5_000_000) == sfar.SFAR_OK      # 5 ms
        assert sfar.sfar_test_force_single_buffer(h.h, True) == sfar.SFAR_OK
        delays = torch.full((calls,), 30000, dtype=torch.int32, device="cuda")
        assert sfar.sfar_test_set_straggler(h.h, delays.data_ptr(), calls, -1, 1) == sfar.SFAR_OK
        warm(h, proto, w.R, w.n, w.dtype)
        out.view(torch.int16).fill_(-1)
        g = capture_chain(h, x_dev, out, proto, calls)
        g.replay()
        torch.cuda.synchronize()
        code, fault = sfar.sfar_status_get(h.h)
        if code == sfar.SFAR_OK:
            with pytest.raises(AssertionError):
                compare_chain(out[:calls], exp[:calls], "single buffer")
        else:
            assert code == sfar.SFAR_ERR_TIMEOUT
    finally:
        h.close()


# ------------------------------------------------ batched decode, two-shot
@pytest.mark.parametrize("mode", ["serial", "overlap"])
@pytest.mark.parametrize("phase", [0, 1])
def test_batched_decode_twoshot_straggler(mode, phase):
    w = inputs.WORKLOADS["batched-decode-r8-896k"]
    x = draw_calls(w, w.calls)
    exp = expected_rows(x)
    h = sfar.Sfar(w.R, w.bytes_per_rank, w.dtype)
    try:
        h.set_mode(mode)
        delays = straggler_delays(w.calls)
        assert sfar.sfar_test_set_straggler(h.h, delays.data_ptr(), w.calls, -1, phase) == sfar.SFAR_OK
        warm(h, "twoshot", w.R, w.n, w.dtype)
        x_dev = x.cuda()
        out = torch.empty_like(x_dev)
        out.view(torch.int16).fill_(-1)
        g = capture_chain(h, x_dev, out, "twoshot", w.calls)
        g.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"twoshot {mode}")
        compare_chain(out, exp, f"batched decode twoshot {mode} phase {phase}")
    finally:
        h.close()


# ------------------------------------------------------------ message sweep
@pytest.mark.parametrize("R", [4, 8])
@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_message_sweep(R, proto):
    h = sfar.Sfar(R, 1 << 20, "bf16")
    try:
        warm(h, proto, R, 512, "bf16")
        for b in inputs.SWEEP_BYTES:
            n = b // 2
            calls = 8
            x = torch.stack([inputs.draw(2, c, R, n, "uniform", 1.0, "bf16") for c in range(calls)])
            exp = expected_rows(x)
            x_dev = x.cuda()
            out = torch.empty_like(x_dev)
            out.view(torch.int16).fill_(-1)
            g = capture_chain(h, x_dev, out, proto, calls)
            g.replay()
            torch.cuda.synchronize()
            status_ok(h.h, f"{proto} {b}")
            compare_chain(out, exp, f"sweep {proto} R={R} {b} B")
    finally:
        h.close()


# ------------------------------------------------- mixed sizes on one handle
@pytest.mark.parametrize("mode", ["serial", "overlap"])
@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_alternating_sizes_on_one_handle(proto, mode):
    """Sizes whose launch geometries differ (16 KB: 16 CTAs x 64 threads per
    rank, 20 KB: 10 x 128, ...) alternate on one handle inside one graph.  A
    receive-buffer address then belongs to different CTAs from call to call,
    so a flag left by one call must never pass for the next call's."""
    R = 8
    sizes = [8192, 10240, 8192 + 3000, 2000, 10240, 8192]
    calls = 240
    h = sfar.Sfar(R, 1 << 20, "bf16")
    try:
        h.set_mode(mode)
        xs, outs, exps = [], [], []
        for c in range(calls):
            n = sizes[c % len(sizes)]
            x = inputs.draw(21, c, R, n, "normal", 1.0, "bf16")
            xs.append(x.cuda())
            outs.append(torch.empty_like(xs[-1]))
            exps.append(expected_bits(x))
        for n in set(sizes):
            warm(h, proto, R, n, "bf16")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in range(calls):
                code = sfar.sfar_allreduce(h.h, [xs[c][r].data_ptr() for r in range(R)],
                                           [outs[c][r].data_ptr() for r in range(R)], xs[c].shape[1], proto)
                assert code == sfar.SFAR_OK
        for rep in range(2):
            for o in outs:
                o.view(torch.int16).fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            status_ok(h.h, f"{proto} {mode} replay {rep}")
            for c in range(calls):
                assert_bits_equal(list(outs[c]), exps[c], f"{proto} {mode} call {c} n={xs[c].shape[1]}")
    finally:
        h.close()


# ------------------------------------------------------------ failure paths
@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_dropped_rank_times_out_and_reset_recovers(proto):
    R, n = 4, 6000
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        x = inputs.draw(9, 0, R, n, "normal", 1.0, "bf16")
        ins, outs = device_io(x)
        h.allreduce(ins, outs, proto)
        torch.cuda.synchronize()
        status_ok(h.h)
        assert sfar.sfar_test_set_timeout(h.h, 2_000_000) == sfar.SFAR_OK       # 2 ms
        assert sfar.sfar_test_drop_rank(h.h, 2) == sfar.SFAR_OK
        h.allreduce(ins, outs, proto)
        h.allreduce(ins, outs, proto)                                          # exits at once: sticky status
        torch.cuda.synchronize()
        code, f = sfar.sfar_status_get(h.h)
        assert code == sfar.SFAR_ERR_TIMEOUT
        assert f.peer in (2, -1) and 0 <= f.rank < R and f.where > 0
        assert sfar.sfar_allreduce(h.h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], n,
                                   proto) == sfar.SFAR_ERR_POISONED
        h.reset()
        assert sfar.sfar_test_drop_rank(h.h, -1) == sfar.SFAR_OK
        torch.cuda.synchronize()
        h.allreduce(ins, outs, proto)
        torch.cuda.synchronize()
        status_ok(h.h, "after reset")
        assert_bits_equal(outs, expected_bits(x), f"{proto} after reset")
    finally:
        h.close()


def test_sentinel_pattern_in_the_data_is_reported():
    R, n = 4, 1024
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        assert sfar.sfar_test_set_timeout(h.h, 2_000_000) == sfar.SFAR_OK
        bits = inputs.to_bits(inputs.draw(10, 0, R, n, "normal", 1.0, "bf16")).copy()
        bits[1, 77] = 0xFFFF
        x = inputs.from_bits(bits)
        ins, outs = device_io(x)
        h.allreduce(ins, outs, "sentinel")
        torch.cuda.synchronize()
        code, f = sfar.sfar_status_get(h.h)
        assert code == sfar.SFAR_ERR_TIMEOUT and f.where == 3 and f.peer == 1
        h.reset()
        x2 = inputs.draw(10, 1, R, n, "normal", 1.0, "bf16")
        ins2, outs2 = device_io(x2)
        h.allreduce(ins2, outs2, "sentinel")
        torch.cuda.synchronize()
        status_ok(h.h)
        assert_bits_equal(outs2, expected_bits(x2), "sentinel after reset")
    finally:
        h.close()


def test_protocols_interleaved_on_one_handle():
    R, n = 8, 8192
    h = sfar.Sfar(R, 1 << 20, "bf16")
    try:
        for i in range(40):
            proto = ALL_PROTOS[i % len(ALL_PROTOS)]
            x = inputs.draw(11, i, R, n, "normal", 1.0, "bf16")
            ins, outs = device_io(x)
            h.allreduce(ins, outs, proto)
            torch.cuda.synchronize()
            status_ok(h.h, proto)
            assert_bits_equal(outs, expected_bits(x), f"interleaved {proto}")
    finally:
        h.close()
