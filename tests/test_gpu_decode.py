"""The row-parallel projection (the AllReduce's producer in a decode layer)
and the projection -> AllReduce chain, bit for bit against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import ensure_built, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def draw_gemv(seed, R, k, h, w_sigma=0.05):
    x = inputs.draw(seed, 0, R, k, "normal", 1.0, "bf16")
    W = inputs.draw(seed, 1, R, k * h, "normal", w_sigma, "bf16").reshape(R, k, h)
    return x, W


def run_gemv(hd, x, W, prefetch=0):
    R, k, h = W.shape
    xs = [x[r].contiguous().cuda() for r in range(R)]
    ws = [W[r].contiguous().cuda() for r in range(R)]
    ys = [torch.empty(h, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    for y in ys:
        y.view(torch.int16).fill_(-1)
    hd.rowpar_gemv(xs, ws, ys, prefetch)
    torch.cuda.synchronize()
    return torch.stack([y.cpu() for y in ys])


@pytest.mark.parametrize("mode", ["serial", "plain"])
@pytest.mark.parametrize("R", [2, 8])
def test_gemv_parity(R, mode):
    hd = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        hd.set_mode(mode)
        for k, h in ((1, 8), (7, 264), (24, 40), (33, 8), (257, 512), (1024, 8192), (3584, 1024), (1000, 2056)):
            x, W = draw_gemv(70 + k, R, k, h)
            want = oracle.gemv(inputs.to_bits(x), inputs.to_bits(W))
            for prefetch in (0, 16, 10 ** 6):
                got = inputs.to_bits(run_gemv(hd, x, W, prefetch))
                assert np.array_equal(got, want), f"R={R} k={k} h={h} prefetch={prefetch} {mode}"
        status_ok(hd.h)
    finally:
        hd.close()


def test_gemv_sixteen_ranks_and_unaligned_input():
    """R = 16 (a weight tensor map per rank in the kernel's parameters), and
    inputs x that start 2 bytes past an aligned address (the API asks for
    2-byte alignment of x only)."""
    for R, k, h, shift in ((16, 300, 520, 0), (16, 64, 256, 1), (3, 129, 1032, 1)):
        x, W = draw_gemv(90 + R + k, R, k, h)
        want = oracle.gemv(inputs.to_bits(x), inputs.to_bits(W))
        hd = sfar.Sfar(R, 1 << 16, "bf16")
        try:
            xb = [torch.zeros(k + 8, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
            xs = [b[shift:shift + k] for b in xb]
            for r in range(R):
                xs[r].copy_(x[r].cuda())
            ws = [W[r].contiguous().cuda() for r in range(R)]
            ys = [torch.empty(h, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
            for y in ys:
                y.view(torch.int16).fill_(-1)
            assert all((t.data_ptr() & 15) == (2 * shift) for t in xs)
            hd.rowpar_gemv(xs, ws, ys, 64)
            torch.cuda.synchronize()
            got = inputs.to_bits(torch.stack([y.cpu() for y in ys]))
            assert np.array_equal(got, want), f"R={R} k={k} h={h} x shifted by {shift}"
            status_ok(hd.h)
        finally:
            hd.close()


def test_gemv_products_that_underflow_or_overflow():
    R, k, h = 2, 64, 64
    g = torch.Generator().manual_seed(71)
    x = (torch.randn(R, k, generator=g) * torch.pow(2.0, torch.randint(-70, 70, (R, k), generator=g).float()))
    W = (torch.randn(R, k, h, generator=g) * torch.pow(2.0, torch.randint(-70, 70, (R, k, h), generator=g).float()))
    x, W = x.to(torch.bfloat16), W.to(torch.bfloat16)
    hd = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        want = oracle.gemv(inputs.to_bits(x), inputs.to_bits(W))
        got = inputs.to_bits(run_gemv(hd, x, W))
        same = (got == want) | (((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0) &
                                ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0))
        assert same.all(), f"{int((~same).sum())} outputs differ"
    finally:
        hd.close()


def test_gemv_argument_checks():
    R, k, h = 2, 16, 64
    hd = sfar.Sfar(R, 1 << 16, "bf16")
    hf = sfar.Sfar(R, 1 << 16, "fp32")
    try:
        xs = [torch.zeros(k, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        ws = [torch.zeros(k, h, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        ys = [torch.zeros(h, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        P = lambda ts: [t.data_ptr() for t in ts]
        call = lambda hh=hd.h, x=P(xs), w=P(ws), y=P(ys), kk=k, hh2=h: sfar.sfar_rowpar_gemv(hh, x, w, y, kk, hh2)
        assert call() == sfar.SFAR_OK
        assert call(hh=hf.h) == sfar.SFAR_ERR_INVALID                        # bf16 only
        assert call(hh2=60) == sfar.SFAR_ERR_INVALID                         # hidden not a multiple of 8
        assert call(kk=0) == sfar.SFAR_ERR_INVALID
        assert call(w=[P(ws)[0] + 2] + P(ws)[1:]) == sfar.SFAR_ERR_INVALID   # misaligned weights
        assert call(y=[P(ws)[1]] + P(ys)[1:]) == sfar.SFAR_ERR_INVALID       # output over another rank's weights
        assert call(y=[P(ys)[1]] + P(ys)[1:]) == sfar.SFAR_ERR_INVALID       # two outputs alias
        torch.cuda.synchronize()
    finally:
        hd.close()
        hf.close()


@pytest.mark.parametrize("ar", ["fused", "ll"])
@pytest.mark.parametrize("mode,prefetch", [("serial", 32), ("serial", 0), ("plain", 0)])
def test_projection_allreduce_chain(ar, mode, prefetch):
    """Eight decode calls (attention output and MLP down projections
    alternating, R = 8, hidden 8192), each a projection into the partial
    sums and the AllReduce of them (fused with the residual add and RMSNorm,
    residual updated in place), captured in one graph and replayed twice."""
    R, h, calls, eps = 8, 8192, 8, 1e-5
    ks = [1024, 3584]
    Ws = [inputs.draw(80, i, R, k * h, "normal", 0.02, "bf16").reshape(R, k, h) for i, k in enumerate(ks)]
    xs = [inputs.draw(81, c, R, ks[c % 2], "normal", 1.0, "bf16") for c in range(calls)]
    res0 = inputs.draw(82, 0, R, h, "normal", 1.0, "bf16")
    wn = inputs.draw(83, 0, 1, h, "normal", 1.0, "bf16")[0]
    # oracle: projections, then the AllReduce (+ residual add + RMSNorm) call by call
    want_out, want_res = [], []
    res = inputs.to_bits(res0)
    for c in range(calls):
        part = oracle.gemv(inputs.to_bits(xs[c]), inputs.to_bits(Ws[c % 2]))
        if ar == "fused":
            y, res = oracle.add_rmsnorm(part, res, inputs.to_bits(wn[None, :])[0], eps, h)
            want_out.append(y)
        else:
            want_out.append(oracle.allreduce(part))
    want_res = res
    hd = sfar.Sfar(R, 2 * h, "bf16")
    try:
        hd.set_mode(mode)
        Wd = [[W[r].contiguous().cuda() for r in range(R)] for W in Ws]
        xd = [[x[r].contiguous().cuda() for r in range(R)] for x in xs]
        part_d = [[torch.empty(h, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(calls)]
        out_d = [[torch.empty(h, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(calls)]
        res_d = [res0[r].contiguous().cuda() for r in range(R)]
        wnd = wn.cuda()
        P = lambda ts: [t.data_ptr() for t in ts]

        def step(c):
            assert sfar.sfar_rowpar_gemv(hd.h, P(xd[c]), P(Wd[c % 2]), P(part_d[c]), ks[c % 2], h,
                                         prefetch) == sfar.SFAR_OK
            if ar == "fused":
                assert sfar.sfar_allreduce_add_rmsnorm(hd.h, P(part_d[c]), P(res_d), wnd.data_ptr(), P(out_d[c]),
                                                       P(res_d), 1, h, eps) == sfar.SFAR_OK
            else:
                assert sfar.sfar_allreduce(hd.h, P(part_d[c]), P(out_d[c]), h, "ll") == sfar.SFAR_OK

        res_start = [t.clone() for t in res_d]
        step(0)                                  # shapes warmed outside the graph
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in range(calls):
                step(c)
        for rep in range(2):
            for t, t0 in zip(res_d, res_start):
                t.copy_(t0)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            status_ok(hd.h, f"{ar} {mode} replay {rep}")
            for c in range(calls):
                got = np.stack([inputs.to_bits(t.cpu()) for t in out_d[c]])
                assert np.array_equal(got, want_out[c]), f"{ar} {mode} call {c} replay {rep}"
            if ar == "fused":
                got_res = np.stack([inputs.to_bits(t.cpu()) for t in res_d])
                assert np.array_equal(got_res, want_res), f"{ar} {mode} residual after the chain"
    finally:
        hd.close()
