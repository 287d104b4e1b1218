"""The checks that pin the CPU oracle to something other than itself.

Each ``check_*`` takes the oracle variant to test (0 = the oracle, other
numbers = a copy with one planted mistake) and raises AssertionError when the
variant disagrees with what the pin fixes:

* closed form: all-ones inputs reduce to exactly R;
* invariants: every rank gets the same bits; scaling every input by 2**k
  scales the result by 2**k bit for bit; on small integers the result is the
  exact integer sum and the reduction is additive;
* hand-derived cases (``golden/oracle_cases.txt``): an order witness, ties in
  the final rounding, signed zeros, subnormals, overflow;
* brute force: every R-tuple (R <= 4) from a 16-value set of awkward bf16
  values against an exact big-integer evaluation (``exact_ref``);
* a library cross-check: the bf16 narrowing against torch's conversion.
"""
import itertools
import os

import numpy as np
import torch

import oracle
import exact_ref
from barrier_free_message_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_cases.txt")

# 16 awkward bf16 values: signed zeros, 1, the smallest normal, the smallest
# subnormal, 1 + 2^-7, 2^24, 3*2^20, a quarter of the largest finite value.
BRUTE_SET = [0x0000, 0x8000, 0x3F80, 0xBF80, 0x0080, 0x8080, 0x0001, 0x8001,
             0x3F81, 0xBF81, 0x4B80, 0xCB80, 0x4A40, 0xCA40, 0x7E7F, 0xFE7F]


def _bf16(values):
    return inputs.to_bits(torch.tensor(values, dtype=torch.float32).to(torch.bfloat16))


def load_golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("->")
            toks = lhs.split()
            dtype, ins = toks[0], [int(t, 16) for t in toks[1:]]
            cases.append((dtype, ins, int(rhs.strip(), 16)))
    return cases


def check_all_ones(mutant=0):
    for dtype in ("bf16", "fp32"):
        for R in (2, 3, 4, 8, 16):
            n = 37
            x = np.ones((R, n), np.float32)
            x = _bf16(x) if dtype == "bf16" else x
            out = oracle.allreduce(x, mutant=mutant)
            got = inputs.from_bits(out).float().numpy()
            assert np.all(got == float(R)), (dtype, R)


def check_identical_ranks(mutant=0):
    x = inputs.to_bits(inputs.draw(11, 0, 8, 1000, "normal", 1.0, "bf16"))
    out = oracle.allreduce(x, mutant=mutant)
    for r in range(1, 8):
        assert np.array_equal(out[r], out[0]), r


def check_power_of_two_scaling(mutant=0):
    base = inputs.draw(12, 0, 8, 4096, "normal", 1.0, "bf16")
    y = inputs.from_bits(oracle.allreduce(inputs.to_bits(base), mutant=mutant))
    for k in (-3, 1, 6):
        s = 2.0 ** k
        xs = (base.float() * s).to(torch.bfloat16)            # exact: no over/underflow here
        ys = inputs.from_bits(oracle.allreduce(inputs.to_bits(xs), mutant=mutant))
        want = (y.float() * s).to(torch.bfloat16)
        assert torch.equal(ys.view(torch.int16), want.view(torch.int16)), k


def check_small_integers(mutant=0):
    g = torch.Generator().manual_seed(13)
    R, n = 16, 512
    a = torch.randint(-8, 9, (R, n), generator=g).float()
    b = torch.randint(-8, 9, (R, n), generator=g).float()
    fa = inputs.from_bits(oracle.allreduce(_bf16(a.numpy()), mutant=mutant)).float()
    fb = inputs.from_bits(oracle.allreduce(_bf16(b.numpy()), mutant=mutant)).float()
    fab = inputs.from_bits(oracle.allreduce(_bf16((a + b).numpy()), mutant=mutant)).float()
    # every partial sum is an integer below 2^8 in magnitude, hence exact in bf16
    assert torch.equal(fa[0], a.sum(0)), "integer sum"
    assert torch.equal(fab, fa + fb), "additivity"


def check_golden(mutant=0):
    for dtype, ins, want in load_golden():
        if dtype == "bf16":
            x = np.array([[b] for b in ins], dtype=np.uint16)
        else:
            x = np.array([[b] for b in ins], dtype=np.uint32).view(np.float32)
        out = oracle.allreduce(x, mutant=mutant)
        got = [int(v) for v in (out[:, 0] if dtype == "bf16" else out[:, 0].view(np.uint32))]
        assert all(g == want for g in got), (dtype, [hex(v) for v in ins], hex(want), [hex(g) for g in got])


def brute_force_cases(R):
    """Every R-tuple from BRUTE_SET, packed 64 tuples per call: list of [R, 64] arrays."""
    tuples = list(itertools.product(BRUTE_SET, repeat=R))
    calls = []
    for i in range(0, len(tuples), 64):
        blk = tuples[i:i + 64]
        calls.append(np.array(blk, dtype=np.uint16).T.copy())
    return calls


def check_brute_force(mutant=0, ranks=(2, 3, 4)):
    for R in ranks:
        for x in brute_force_cases(R):
            out = oracle.allreduce(x, mutant=mutant)
            for j in range(x.shape[1]):
                want = exact_ref.fold_bf16([int(v) for v in x[:, j]])
                got = out[:, j]
                assert np.all(got == want), (R, [hex(int(v)) for v in x[:, j]], hex(want), hex(int(got[0])))


def check_narrowing_vs_torch(mutant=0):
    g = torch.Generator().manual_seed(14)
    bits = torch.randint(0, 2**31 - 1, (20000,), generator=g, dtype=torch.int64)
    sign = torch.randint(0, 2, (20000,), generator=g, dtype=torch.int64) << 31
    u = (bits | sign).to(torch.int64)
    f = torch.from_numpy((u.numpy() & 0xFFFFFFFF).astype(np.uint32).view(np.float32))
    finite = torch.isfinite(f)
    f = f[finite]
    want = inputs.to_bits(f.to(torch.bfloat16))
    got = np.array([oracle.narrow_bf16(float(v), mutant=mutant) for v in f.numpy()], dtype=np.uint16)
    assert np.array_equal(got, want)


ALL_CHECKS = [check_all_ones, check_identical_ranks, check_power_of_two_scaling,
              check_small_integers, check_golden, check_brute_force, check_narrowing_vs_torch]
