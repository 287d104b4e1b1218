"""Every protocol against the CPU oracle, bit for bit on every rank, through
the C ABI (small and ragged sizes, hand-derived cases, the brute-force value
set, argument checks)."""
import numpy as np
import pytest
import torch

import oracle_pins
from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import (ALL_PROTOS, assert_bits_equal, device_io, ensure_built, expected_bits, run_once,
                         status_ok)

pytestmark = pytest.mark.gpu

SIZES = [1, 3, 8, 37, 248, 255, 1000, 4099, 7937, 65536 + 7]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [2, 3, 8, 16])
@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_parity_ragged_sizes(proto, R, dtype):
    h = sfar.Sfar(R, 1 << 20, dtype)
    try:
        for n in SIZES:
            x = inputs.draw(100 + R, n, R, n, "normal", 1.0, dtype)
            outs = run_once(h, x, proto)
            assert_bits_equal(outs, expected_bits(x), f"{proto} R={R} n={n} {dtype}")
    finally:
        h.close()


@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_hand_derived_cases(proto):
    cases = oracle_pins.load_golden()
    by_key = {}
    for dtype, ins, want in cases:
        by_key.setdefault((dtype, len(ins)), []).append((ins, want))
    for (dtype, R), group in by_key.items():
        h = sfar.Sfar(R, 1 << 16, dtype)
        try:
            npdt = np.uint16 if dtype == "bf16" else np.uint32
            bits = np.array([g[0] for g in group], dtype=npdt).T.copy()      # [R, cases]
            x = inputs.from_bits(bits if dtype == "bf16" else bits.view(np.float32))
            outs = run_once(h, x, proto)
            want = np.array([g[1] for g in group], dtype=npdt)
            for r in range(R):
                got = inputs.to_bits(outs[r].cpu())
                got = got.view(np.uint32) if dtype == "fp32" else got
                assert np.array_equal(got, want), (proto, dtype, R, [hex(v) for v in got], [hex(v) for v in want])
        finally:
            h.close()


@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_brute_force_value_set(proto):
    # every 4-tuple of the 16 awkward bf16 values, one call of n = 65536
    cols = np.concatenate(oracle_pins.brute_force_cases(4), axis=1)
    x = inputs.from_bits(cols)
    h = sfar.Sfar(4, 1 << 20, "bf16")
    try:
        outs = run_once(h, x, proto)
        assert_bits_equal(outs, expected_bits(x), proto)
    finally:
        h.close()


@pytest.mark.parametrize("proto", ALL_PROTOS)
def test_all_ones_closed_form(proto):
    for R in (2, 5, 16):
        h = sfar.Sfar(R, 1 << 16, "bf16")
        try:
            x = torch.ones(R, 4097, dtype=torch.bfloat16)
            outs = run_once(h, x, proto)
            for o in outs:
                assert torch.all(o.float() == float(R))
        finally:
            h.close()


def test_empty_call_is_a_noop():
    h = sfar.Sfar(4, 1 << 16, "bf16")
    try:
        x = torch.zeros(4, 16, dtype=torch.bfloat16)
        ins, outs = device_io(x)
        before = [o.clone() for o in outs]
        for proto in ALL_PROTOS:
            assert sfar.sfar_allreduce(h.h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], 0,
                                       proto) == sfar.SFAR_OK
        torch.cuda.synchronize()
        for o, b in zip(outs, before):
            assert torch.equal(o, b)
        status_ok(h.h)
    finally:
        h.close()


def test_argument_checks():
    R = 4
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        x = torch.zeros(R, 1024, dtype=torch.bfloat16)
        ins, outs = device_io(x)
        ip = [t.data_ptr() for t in ins]
        op = [t.data_ptr() for t in outs]
        call = lambda i, o, n, p="ll": sfar.sfar_allreduce(h.h, i, o, n, p)
        assert call(ip, op, 1024) == sfar.SFAR_OK
        assert call([ip[0] + 2] + ip[1:], op, 1000) == sfar.SFAR_ERR_INVALID          # misaligned input
        assert call(ip, [op[0] + 8] + op[1:], 1000) == sfar.SFAR_ERR_INVALID          # misaligned output
        assert call(ip, [ip[0]] + op[1:], 1024) == sfar.SFAR_ERR_INVALID              # output overlaps input
        assert call(ip, [op[1]] + op[1:], 1024) == sfar.SFAR_ERR_INVALID              # two outputs alias
        assert call(ip, op, (1 << 16) // 2 + 1) == sfar.SFAR_ERR_INVALID              # over max_bytes
        assert call(ip, op, 1024, len(sfar.PROTOS)) == sfar.SFAR_ERR_INVALID          # unknown protocol
        assert call([0] + ip[1:], op, 1024) == sfar.SFAR_ERR_INVALID                  # null pointer
        torch.cuda.synchronize()
        status_ok(h.h)
    finally:
        h.close()


def test_inputs_may_alias_each_other():
    R = 4
    h = sfar.Sfar(R, 1 << 16, "fp32")
    try:
        x = inputs.draw(7, 0, 1, 3000, "uniform", 1.0, "fp32").repeat(R, 1)
        shared = x[0].cuda()
        outs = [torch.empty_like(shared) for _ in range(R)]
        for proto in ALL_PROTOS:
            h.allreduce([shared] * R, outs, proto)
            torch.cuda.synchronize()
            status_ok(h.h, proto)
            assert_bits_equal(outs, expected_bits(x), proto)
    finally:
        h.close()


def test_query_launch_geometry():
    h = sfar.Sfar(8, 1 << 20, "bf16")
    try:
        for proto in ALL_PROTOS:
            k, t = h.launch(8192, proto)
            assert 1 <= k <= 128 and t in (64, 128, 256, 320)
            assert 8 * k <= torch.cuda.get_device_properties(0).multi_processor_count * 8
        assert sfar.sfar_test_set_geometry(h.h, 3, 128) == sfar.SFAR_OK
        assert h.launch(8192, "ll") == (3, 128)
        assert sfar.sfar_test_set_geometry(h.h, 3, 96) == sfar.SFAR_ERR_INVALID
        assert sfar.sfar_test_set_geometry(h.h, 0, 0) == sfar.SFAR_OK
        assert sfar.sfar_max_bytes(h.h, "ll") == 1 << 20
    finally:
        h.close()
