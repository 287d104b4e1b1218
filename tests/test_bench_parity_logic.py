"""The benchmark's parity bookkeeping, on the CPU: which token graphs the
replays run, the oracle rows of a set of calls, and the device-side
comparison (run here on CPU tensors).  A check that looks at calls the
replays never computed, or that misses a wrong element, fails here."""
import sys

import numpy as np
import torch

import oracle
from barrier_free_message_gb300 import inputs


def _bench():
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        import bench
    finally:
        sys.argv = argv
    return bench


def test_replayed_tokens_are_the_ones_the_timing_loop_runs():
    bench = _bench()
    # the driver's run: 5 warm-up + 20 timed replays of 64 token graphs
    assert bench.replayed_tokens(64, 5, 20) == list(range(25))
    # the default run wraps around every token
    assert bench.replayed_tokens(64, 8, 640) == list(range(64))
    # replay i runs token i mod tokens
    assert bench.replayed_tokens(4, 3, 2) == [0, 1, 2, 3]
    assert bench.replayed_tokens(10, 3, 3) == [0, 1, 2, 3, 4, 5]


def test_oracle_rows_match_the_oracle_call_by_call():
    bench = _bench()
    calls, R, n = 7, 3, 50
    x = torch.stack([inputs.draw(5, c, R, n, "normal", 1.0, "bf16") for c in range(calls)])
    ids = [0, 3, 6]
    rows = bench.oracle_rows(x, ids, threads=2)
    for i, c in enumerate(ids):
        want = oracle.allreduce(inputs.to_bits(x[c]))
        assert all(np.array_equal(rows[i], want[r]) for r in range(R))


def test_device_mismatches_counts_every_wrong_call():
    bench = _bench()
    calls, R, n = 6, 4, 33
    for dtype in ("bf16", "fp32"):
        x = torch.stack([inputs.draw(6, c, R, n, "normal", 1.0, dtype) for c in range(calls)])
        out = torch.empty_like(x)
        for c in range(calls):
            out[c] = inputs.from_bits(oracle.allreduce(inputs.to_bits(x[c])))
        ids = [1, 2, 5]
        exp = bench.oracle_rows(x, ids, threads=1)
        exp_t = torch.from_numpy(exp.view(np.int16) if dtype == "bf16" else exp.view(np.int32))
        assert bench.device_mismatches(out, ids, exp_t) == 0
        out[5, 3, 32] = 1e9                                         # one element of the last rank
        assert bench.device_mismatches(out, ids, exp_t) == 1
        out[0, 0, 0] = 1e9                                          # a call outside the checked set
        assert bench.device_mismatches(out, ids, exp_t) == 1
        out[2, 1, 7] = -out[2, 1, 7] - 1.0
        assert bench.device_mismatches(out, ids, exp_t, block=1) == 2
        # an output never written (the NaN pattern the bench fills in first) is a mismatch
        bench._as_int(out[1]).fill_(-1)
        assert bench.device_mismatches(out, ids, exp_t) == 3
