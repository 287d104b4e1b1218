"""The allocation-free entry point (sfar_allreduce_noalloc) against the
regular one.

sfar_allreduce_noalloc exists for callers that cannot allocate device memory
when they need an AllReduce (under stream capture, inside a framework whose
allocator owns all device memory, or on a path that cannot afford
cudaMalloc's implicit synchronisation); it takes its working memory from a
fixed array compiled into the library.  This file is named so that pytest
collects it last.  It must pass on its own in a fresh process and after the
other tests.
"""
import numpy as np
import pytest
import torch

from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import as_uint, device_io, ensure_built, expected_bits, status_ok

pytestmark = pytest.mark.gpu

MAX_RANKS = 8
MAX_BYTES = 16384


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _bits(t):
    return as_uint(inputs.to_bits(t.cpu()))


@pytest.mark.parametrize("dtype,R,n", [("bf16", 8, 8192), ("bf16", 4, 4099), ("fp32", 8, 4096), ("fp32", 3, 37)])
def test_noalloc_matches_the_handle_path_on_two_calls(dtype, R, n):
    h = sfar.Sfar(R, MAX_BYTES, dtype)
    try:
        for call in range(2):      # two calls in a row: the second reuses the shared array
            x = inputs.draw(31, call, R, n, "normal", 1.0, dtype)
            ins, outs_ref = device_io(x)
            outs_na = [torch.empty_like(t) for t in ins]
            for o in outs_na:
                o.view(torch.uint8).fill_(0x5A)
            h.allreduce(ins, outs_ref, "ll")
            code = sfar.sfar_allreduce_noalloc([t.data_ptr() for t in ins], [t.data_ptr() for t in outs_na],
                                               R, n, dtype)
            assert code == sfar.SFAR_OK, sfar.strerror(code)
            torch.cuda.synchronize()
            status_ok(h.h)
            assert sfar.sfar_noalloc_status()[0] == sfar.SFAR_OK
            want = expected_bits(x)
            for r in range(R):
                # bit-exact: the same fixed-order reduction on both paths
                assert np.array_equal(_bits(outs_na[r]), _bits(outs_ref[r])), (call, r)
                assert np.array_equal(_bits(outs_na[r]), as_uint(want[r])), (call, r)
    finally:
        h.close()


def test_noalloc_in_a_graph_after_setup():
    R, n = 8, 8192
    xs = [inputs.draw(32, c, R, n, "normal", 1.0, "bf16") for c in range(4)]
    io = [device_io(x) for x in xs]
    # the first call sets the array up (not under capture)
    ins, outs = io[0]
    assert sfar.sfar_allreduce_noalloc([t.data_ptr() for t in ins], [t.data_ptr() for t in outs], R, n) == 0
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for ins, outs in io:
            assert sfar.sfar_allreduce_noalloc([t.data_ptr() for t in ins], [t.data_ptr() for t in outs], R,
                                               n) == 0
    for _ in range(2):
        for _, outs in io:
            for o in outs:
                o.view(torch.int16).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        for x, (_, outs) in zip(xs, io):
            want = expected_bits(x)
            for r in range(R):
                assert np.array_equal(_bits(outs[r]), as_uint(want[r]))


def _noalloc_call(x, dtype):
    R, n = x.shape
    ins, outs = device_io(x)
    code = sfar.sfar_allreduce_noalloc([t.data_ptr() for t in ins], [t.data_ptr() for t in outs], R, n, dtype)
    return code, outs


def test_noalloc_chain_of_mixed_sizes_and_types():
    """R = 8 calls of different sizes (so different grids: 8192 elements, 37,
    4099) and both element types in a row on the shared array, each compared
    bit for bit with the oracle; the array's status stays clear."""
    R = 8
    plan = [("bf16", 8192), ("bf16", 37), ("fp32", 4093), ("bf16", 4099), ("fp32", 37), ("fp32", 4096),
            ("bf16", 8192), ("fp32", 1)]
    for i, (dtype, n) in enumerate(plan * 2):
        x = inputs.draw(33, i, R, n, "normal", 1.0, dtype)
        code, outs = _noalloc_call(x, dtype)
        assert code == sfar.SFAR_OK, sfar.strerror(code)
        torch.cuda.synchronize()
        want = expected_bits(x)
        for r in range(R):
            assert np.array_equal(_bits(outs[r]), as_uint(want[r])), (i, dtype, n, r)
    code, f = sfar.sfar_noalloc_status()
    assert code == sfar.SFAR_OK, (code, f.where)


def test_noalloc_failure_is_reported_then_cleared():
    """A failed device wait (recorded on the host, as a wait that ran out
    would record it): the next kernel writes nothing, the status call reports
    the failure, later calls are refused until the record is cleared, and
    calls after the clear compute the right sums again."""
    R, n = 4, 1000
    try:
        assert sfar.sfar_test_noalloc_record_failure(2, 1, 2) == sfar.SFAR_OK
        x = inputs.draw(34, 0, R, n, "normal", 1.0, "bf16")
        code, outs = _noalloc_call(x, "bf16")
        assert code == sfar.SFAR_OK                  # enqueued: the host has not read the record yet
        torch.cuda.synchronize()
        for o in outs:                               # the kernel saw the record and wrote nothing
            assert (o.view(torch.uint8) == 0xA5).all()
        code, f = sfar.sfar_noalloc_status()
        assert code == sfar.SFAR_ERR_TIMEOUT and (f.rank, f.peer, f.where) == (2, 1, 2)
        code, _ = _noalloc_call(x, "bf16")
        assert code == sfar.SFAR_ERR_POISONED        # reported, so refused on the host
        code, f = sfar.sfar_noalloc_status(clear=True)
        assert code == sfar.SFAR_ERR_TIMEOUT         # the clearing read still returns what it cleared
    finally:
        sfar.sfar_noalloc_status(clear=True)
    assert sfar.sfar_noalloc_status()[0] == sfar.SFAR_OK
    for c in range(3):
        x = inputs.draw(34, 1 + c, R, n, "normal", 1.0, "bf16")
        code, outs = _noalloc_call(x, "bf16")
        assert code == sfar.SFAR_OK
        torch.cuda.synchronize()
        want = expected_bits(x)
        for r in range(R):
            assert np.array_equal(_bits(outs[r]), as_uint(want[r])), (c, r)


def test_noalloc_rejects_what_does_not_fit():
    R, n = 8, MAX_BYTES // 2
    x = torch.zeros(R, n + 8, dtype=torch.bfloat16)
    ins, outs = device_io(x)
    ip, op = [t.data_ptr() for t in ins], [t.data_ptr() for t in outs]
    assert sfar.sfar_allreduce_noalloc(ip, op, R, n + 1, "bf16") == sfar.SFAR_ERR_INVALID          # too many bytes
    assert sfar.sfar_allreduce_noalloc(ip * 2, op * 2, 9, 64, "bf16") == sfar.SFAR_ERR_INVALID     # too many ranks
    assert sfar.sfar_allreduce_noalloc(ip, op, 1, 64, "bf16") == sfar.SFAR_ERR_INVALID             # too few ranks
    assert sfar.sfar_allreduce_noalloc(ip, [op[0] + 2] + op[1:], R, 64, "bf16") == sfar.SFAR_ERR_INVALID
    assert sfar.sfar_allreduce_noalloc(ip, [ip[0]] + op[1:], R, 64, "bf16") == sfar.SFAR_ERR_INVALID
    assert sfar.sfar_allreduce_noalloc(ip, op, R, 0, "bf16") == sfar.SFAR_OK                       # empty: no-op
    torch.cuda.synchronize()
