"""The fused AllReduce + residual add + RMS normalisation (and the
normalisation on its own) against the oracle, bit for bit on every rank.

NaN results are compared as NaN (the oracle's NaN payloads follow the host
CPU, the GPU's are canonical); every other element is compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import ensure_built, status_ok

pytestmark = pytest.mark.gpu
TDT = {"bf16": torch.bfloat16, "fp32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def draw_case(seed, R, rows, h, dtype, sigma=1.0):
    x = inputs.draw(seed, 0, R, rows * h, "normal", sigma, dtype)
    res = inputs.draw(seed, 1, R, rows * h, "normal", 2.0, dtype)
    w = inputs.draw(seed, 2, 1, h, "normal", 1.0, dtype)[0]
    return x, res, w


def bits(t):
    b = inputs.to_bits(t.detach().cpu())
    return b.view(np.uint32) if b.dtype == np.float32 else b


def assert_equal_nan_aware(got_t, want, ctx):
    got = bits(got_t)
    want = want.view(np.uint32) if want.dtype == np.float32 else want
    if want.dtype == np.uint16:
        gn = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
        wn = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
    else:
        gn = ((got & 0x7F800000) == 0x7F800000) & ((got & 0x7FFFFF) != 0)
        wn = ((want & 0x7F800000) == 0x7F800000) & ((want & 0x7FFFFF) != 0)
    bad = (got != want) & ~(gn & wn)
    if bad.any():
        i = int(np.nonzero(bad)[0][0])
        raise AssertionError(f"{ctx}: {int(bad.sum())} of {bad.size} elements differ; first at {i}: "
                             f"got {int(got[i]):#x} want {int(want[i]):#x}")


def run_fused(h, x, res, w, hidden, eps, allreduce=True, in_place=False):
    R = x.shape[0]
    ins = [x[r].contiguous().cuda() for r in range(R)]
    rs = [res[r].contiguous().cuda() for r in range(R)]
    wd = w.contiguous().cuda()
    outs = [torch.empty_like(t) for t in ins]
    for o in outs:
        o.view(torch.uint8).fill_(0xA5)
    routs = rs if in_place else [torch.empty_like(t) for t in rs]
    if allreduce:
        h.allreduce_add_rmsnorm(ins, rs, wd, outs, routs, hidden, eps)
    else:
        h.add_rmsnorm(ins, rs, wd, outs, routs, hidden, eps)
    torch.cuda.synchronize()
    status_ok(h.h, "fused")
    return outs, routs


def check(h, x, res, w, hidden, eps, ctx, allreduce=True, in_place=False):
    want_y, want_z = oracle.add_rmsnorm(inputs.to_bits(x), inputs.to_bits(res), inputs.to_bits(w[None, :])[0],
                                        eps, hidden, allreduce_first=allreduce)
    outs, routs = run_fused(h, x, res, w, hidden, eps, allreduce, in_place)
    for r in range(x.shape[0]):
        assert_equal_nan_aware(routs[r], want_z[r], f"{ctx} z rank {r}")
        assert_equal_nan_aware(outs[r], want_y[r], f"{ctx} y rank {r}")


SHAPES = {"bf16": [(1, 8192), (3, 7168), (5, 64), (2, 8), (1, 24), (4, 1000), (2, 32768), (1, 65536), (64, 7168)],
          "fp32": [(1, 8192), (3, 7168), (5, 64), (2, 4), (1, 20), (4, 1000), (1, 32768), (32, 4096)]}


@pytest.mark.parametrize("path", ["auto", "oneshot"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [2, 3, 8, 16])
def test_fused_parity(R, dtype, path):
    h = sfar.Sfar(R, 1 << 20, dtype)
    es = 2 if dtype == "bf16" else 4
    try:
        assert sfar.sfar_test_set_fused_path(h.h, path) == sfar.SFAR_OK
        for rows, hidden in SHAPES[dtype]:
            code, k, cl, t = sfar.sfar_test_query_norm_launch(h.h, rows, hidden)
            if R > 8 and hidden * es > 65536:
                assert code == sfar.SFAR_ERR_INVALID          # rows above 64 KiB need R <= 8
                continue
            assert code == sfar.SFAR_OK and k % cl == 0 and 1 <= cl <= 8 and t in (32, 64, 128, 256)
            x, res, w = draw_case(500 + R + rows, R, rows, hidden, dtype)
            check(h, x, res, w, hidden, 1e-5,
                  f"{path} R={R} {rows}x{hidden} {dtype} ({k} CTAs/rank, cluster {cl}, {t})")
    finally:
        h.close()



@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [3, 8, 16])
def test_cooperative_mode_parity(R, dtype):
    """The cooperative launch mode (every AllReduce kernel a cooperative grid,
    the fused grids cooperative cluster grids that never run solo): the same
    bits as the oracle for both fused kernels and the plain AllReduce."""
    h = sfar.Sfar(R, 1 << 20, dtype)
    es = 2 if dtype == "bf16" else 4
    try:
        h.set_mode("cooperative")
        for path in ("oneshot", "twoshot", "auto"):
            assert sfar.sfar_test_set_fused_path(h.h, path) == sfar.SFAR_OK
            for rows, hidden in ((1, 8192), (4, 8192), (3, 7168), (2, 1000), (16, 4096 // es * 2)):
                if rows * hidden * es > (1 << 20):
                    continue
                x, res, w = draw_case(2000 + R + rows, R, rows, hidden, dtype)
                check(h, x, res, w, hidden, 1e-5, f"cooperative {path} R={R} {rows}x{hidden} {dtype}")
        x = inputs.draw(2100 + R, 0, R, 8192 + 5, "normal", 1.0, dtype)
        ins = [x[r].contiguous().cuda() for r in range(R)]
        for proto in ("ll", "sentinel", "twoshot_sent", "twoshot_tma"):
            outs = [torch.empty_like(t) for t in ins]
            h.allreduce(ins, outs, proto)
            torch.cuda.synchronize()
            status_ok(h.h, f"cooperative {proto}")
            want = oracle.allreduce(inputs.to_bits(x))
            for r in range(R):
                assert_equal_nan_aware(outs[r], want[r], f"cooperative {proto} R={R} rank {r}")
    finally:
        h.close()

@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [8, 16])
def test_norm_alone_parity(R, dtype):
    h = sfar.Sfar(R, 1 << 20, dtype)
    es = 2 if dtype == "bf16" else 4
    try:
        for rows, hidden in SHAPES[dtype]:
            if R > 8 and hidden * es > 65536:
                continue
            x, res, w = draw_case(600 + rows, R, rows, hidden, dtype, sigma=5.0)
            check(h, x, res, w, hidden, 1e-6, f"alone {rows}x{hidden} {dtype}", allreduce=False)
    finally:
        h.close()


def test_in_place_residual():
    R, rows, hidden = 8, 4, 8192
    h = sfar.Sfar(R, 1 << 20, "bf16")
    try:
        x, res, w = draw_case(700, R, rows, hidden, "bf16")
        check(h, x, res, w, hidden, 1e-5, "in place", in_place=True)
        check(h, x, res, w, hidden, 1e-5, "alone in place", allreduce=False, in_place=True)
    finally:
        h.close()


def test_special_rows_and_ranges():
    R, hidden = 4, 1024
    h = sfar.Sfar(R, 1 << 20, "fp32")
    try:
        x, res, w = draw_case(701, R, 6, hidden, "fp32")
        res[:, :hidden] = 0.0
        x[:, :hidden] = 0.0                          # row 0: all zero
        x[1, hidden + 7] = float("nan")              # row 1: NaN
        res[2, 2 * hidden + 9] = float("inf")        # row 2: an infinity on rank 2 only
        x[:, 3 * hidden:4 * hidden] *= 2.0 ** 60     # row 3: large
        x[:, 4 * hidden:5 * hidden] *= 2.0 ** -70    # row 4: tiny (subnormal squares)
        res[:, 4 * hidden:5 * hidden] *= 2.0 ** -70
        check(h, x, res, w, hidden, 1e-6, "special rows")
    finally:
        h.close()


@pytest.mark.parametrize("path", ["oneshot", "twoshot"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_rows_with_outliers(path, dtype):
    """Rows whose largest magnitude sits in one place, 2^k above the rest
    (k = 0 .. 12, also on one rank only): the kernels take the row's scale
    from the whole row whatever the spread between the parts of it that
    different warps hold, including spreads of 3 and 4 binades and beyond."""
    R = 8
    h = sfar.Sfar(R, 1 << 20, dtype)
    try:
        assert sfar.sfar_test_set_fused_path(h.h, path) == sfar.SFAR_OK
        for rows, hidden in ((1, 8192), (4, 8192), (6, 2048), (3, 7168), (5, 64)):
            code, got = sfar.sfar_test_query_fused_path(h.h, rows, hidden)
            if code != sfar.SFAR_OK or got != (1 if path == "oneshot" else 2):
                continue
            x, res, w = draw_case(1200 + rows, R, rows, hidden, dtype)
            for i in range(rows):
                k = (0, 3, 4, 5, 12, 2)[i % 6]
                j = i * hidden + (97 * i + 13) % hidden
                x[:, j] *= 2.0 ** k
                res[:, j] *= 2.0 ** k
                if i % 2:
                    x[i % R, (j + hidden // 2) % (rows * hidden)] *= 2.0 ** (k + 1)
            check(h, x, res, w, hidden, 1e-5, f"{path} outliers {rows}x{hidden} {dtype}")
    finally:
        h.close()


@pytest.mark.parametrize("mode", ["serial", "overlap", "cooperative"])
def test_fused_chain_1024_calls(mode):
    """The decode shape (R = 8, one row of 8192 bf16) for 1,024 graph-chained
    calls, each with its own inputs and residual."""
    R, hidden, calls = 8, 8192, 1024
    x = torch.stack([inputs.draw(800, c, R, hidden, "normal", 1.0, "bf16") for c in range(calls)])
    res = torch.stack([inputs.draw(801, c, R, hidden, "normal", 2.0, "bf16") for c in range(calls)])
    w = inputs.draw(802, 0, 1, hidden, "normal", 1.0, "bf16")[0]
    want_y, want_z = oracle.add_rmsnorm(inputs.to_bits(x.transpose(0, 1).reshape(R, calls * hidden)),
                                        inputs.to_bits(res.transpose(0, 1).reshape(R, calls * hidden)),
                                        inputs.to_bits(w[None, :])[0], 1e-5, hidden)
    h = sfar.Sfar(R, 2 * hidden, "bf16")
    try:
        h.set_mode(mode)
        xd, rd, wd = x.cuda(), res.cuda(), w.cuda()
        od, zd = torch.empty_like(xd), torch.empty_like(xd)
        # warm-up call outside the graph (sets up the launch shape)
        h.allreduce_add_rmsnorm([xd[0, r] for r in range(R)], [rd[0, r] for r in range(R)], wd,
                                [od[0, r] for r in range(R)], [zd[0, r] for r in range(R)], hidden, 1e-5)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in range(calls):
                code = sfar.sfar_allreduce_add_rmsnorm(h.h, [xd[c, r].data_ptr() for r in range(R)],
                                                       [rd[c, r].data_ptr() for r in range(R)], wd.data_ptr(),
                                                       [od[c, r].data_ptr() for r in range(R)],
                                                       [zd[c, r].data_ptr() for r in range(R)], 1, hidden, 1e-5)
                assert code == sfar.SFAR_OK
        for rep in range(2):
            od.view(torch.int16).fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            status_ok(h.h, f"chain {mode} replay {rep}")
            got_y = od.transpose(0, 1).reshape(R, calls * hidden)
            got_z = zd.transpose(0, 1).reshape(R, calls * hidden)
            for r in range(R):
                assert_equal_nan_aware(got_z[r], want_z[r], f"chain {mode} z rank {r}")
                assert_equal_nan_aware(got_y[r], want_y[r], f"chain {mode} y rank {r}")
    finally:
        h.close()


def test_shares_the_ll_region_with_plain_calls():
    R, hidden = 8, 8192
    h = sfar.Sfar(R, 1 << 20, "bf16")
    try:
        for i in range(12):
            x, res, w = draw_case(900 + i, R, 1 + i % 3, hidden, "bf16")
            if i % 2:
                check(h, x, res, w, hidden, 1e-5, f"interleaved fused {i}")
            else:
                xi = x.contiguous()
                ins = [xi[r].cuda() for r in range(R)]
                outs = [torch.empty_like(t) for t in ins]
                h.allreduce(ins, outs, "ll")
                torch.cuda.synchronize()
                status_ok(h.h, "ll")
                want = oracle.allreduce(inputs.to_bits(xi))
                for r in range(R):
                    assert np.array_equal(inputs.to_bits(outs[r].cpu()), want[r])
    finally:
        h.close()


def test_argument_checks():
    R, hidden = 4, 1024
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        x, res, w = draw_case(950, R, 2, hidden, "bf16")
        ins = [t.cuda() for t in x]
        rs = [t.cuda() for t in res]
        wd = w.cuda()
        outs = [torch.empty_like(t) for t in ins]
        zs = [torch.empty_like(t) for t in ins]
        P = lambda ts: [t.data_ptr() for t in ts]
        call = lambda i=P(ins), rr=P(rs), ww=wd.data_ptr(), o=P(outs), z=P(zs), rows=2, hid=hidden: \
            sfar.sfar_allreduce_add_rmsnorm(h.h, i, rr, ww, o, z, rows, hid, 1e-5)
        assert call() == sfar.SFAR_OK
        assert call(rows=0) == sfar.SFAR_OK
        assert call(hid=1020) == sfar.SFAR_ERR_INVALID                         # row not whole vectors
        assert call(ww=wd.data_ptr() + 2) == sfar.SFAR_ERR_INVALID             # misaligned weight
        assert call(o=[P(rs)[0]] + P(outs)[1:]) == sfar.SFAR_ERR_INVALID        # out over a residual
        assert call(z=[P(ins)[1]] + P(zs)[1:]) == sfar.SFAR_ERR_INVALID         # z over an input
        assert call(z=[P(rs)[1]] + P(zs)[1:]) == sfar.SFAR_ERR_INVALID         # z over another rank's residual
        assert call(rows=40) == sfar.SFAR_ERR_INVALID                          # over the handle's 64 KiB
        big = sfar.Sfar(2, 1 << 20, "bf16")
        try:
            t = torch.zeros(2 * 65544, dtype=torch.bfloat16, device="cuda")
            assert sfar.sfar_add_rmsnorm(big.h, [t.data_ptr()] * 2, [t.data_ptr()] * 2, t.data_ptr(),
                                         [t.data_ptr()] * 2, [t.data_ptr()] * 2, 1, 65544, 0.0) == \
                sfar.SFAR_ERR_INVALID                                          # row above 128 KiB
        finally:
            big.close()
        torch.cuda.synchronize()
        status_ok(h.h)
    finally:
        h.close()


def test_dropped_rank_times_out_and_reset_recovers():
    R, rows, hidden = 4, 2, 4096
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        assert sfar.sfar_test_set_fused_path(h.h, "oneshot") == sfar.SFAR_OK
        x, res, w = draw_case(960, R, rows, hidden, "bf16")
        check(h, x, res, w, hidden, 1e-5, "before")
        assert sfar.sfar_test_set_timeout(h.h, 2_000_000) == sfar.SFAR_OK
        assert sfar.sfar_test_drop_rank(h.h, 1) == sfar.SFAR_OK
        ins = [t.cuda() for t in x]
        rs = [t.cuda() for t in res]
        outs = [torch.empty_like(t) for t in ins]
        zs = [torch.empty_like(t) for t in ins]
        h.allreduce_add_rmsnorm(ins, rs, w.cuda(), outs, zs, hidden, 1e-5)
        torch.cuda.synchronize()
        code, f = sfar.sfar_status_get(h.h)
        assert code == sfar.SFAR_ERR_TIMEOUT and sfar.WAIT_NAMES[f.where] == "ll" and f.peer in (1, -1)
        h.reset()
        assert sfar.sfar_test_drop_rank(h.h, -1) == sfar.SFAR_OK
        torch.cuda.synchronize()
        check(h, x, res, w, hidden, 1e-5, "after reset")
    finally:
        h.close()


@pytest.mark.parametrize("phase", [0, 1])
def test_fused_chain_overlap_with_straggler(phase):
    """512 graph-chained calls in overlap mode with one rank (rotating) delayed
    by 0-20 us before its sends (phase 0) or between its sends and receives
    (phase 1): calls overtake one another across ranks, and the cluster
    statistics rounds see the skew; every call stays bit-exact."""
    R, hidden, calls, eps = 8, 8192, 512, 1e-5
    x = torch.stack([inputs.draw(810, c, R, hidden, "normal", 1.0, "bf16") for c in range(calls)])
    res = torch.stack([inputs.draw(811, c, R, hidden, "normal", 2.0, "bf16") for c in range(calls)])
    w = inputs.draw(812, 0, 1, hidden, "normal", 1.0, "bf16")[0]
    want_y, want_z = oracle.add_rmsnorm(inputs.to_bits(x.transpose(0, 1).reshape(R, calls * hidden)),
                                        inputs.to_bits(res.transpose(0, 1).reshape(R, calls * hidden)),
                                        inputs.to_bits(w[None, :])[0], eps, hidden)
    h = sfar.Sfar(R, 2 * hidden, "bf16")
    try:
        h.set_mode("overlap")
        xd, rd, wd = x.cuda(), res.cuda(), w.cuda()
        od, zd = torch.empty_like(xd), torch.empty_like(xd)
        h.allreduce_add_rmsnorm([xd[0, r] for r in range(R)], [rd[0, r] for r in range(R)], wd,
                                [od[0, r] for r in range(R)], [zd[0, r] for r in range(R)], hidden, eps)
        torch.cuda.synchronize()
        g = torch.Generator().manual_seed(813)
        delays = torch.randint(0, 20001, (calls,), generator=g).to(torch.int32).cuda()
        assert sfar.sfar_test_set_straggler(h.h, delays.data_ptr(), calls, -1, phase) == sfar.SFAR_OK
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in range(calls):
                assert sfar.sfar_allreduce_add_rmsnorm(h.h, [xd[c, r].data_ptr() for r in range(R)],
                                                       [rd[c, r].data_ptr() for r in range(R)], wd.data_ptr(),
                                                       [od[c, r].data_ptr() for r in range(R)],
                                                       [zd[c, r].data_ptr() for r in range(R)], 1, hidden,
                                                       eps) == sfar.SFAR_OK
        graph.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"straggler phase {phase}")
        got_y = od.transpose(0, 1).reshape(R, calls * hidden)
        got_z = zd.transpose(0, 1).reshape(R, calls * hidden)
        for r in range(R):
            assert_equal_nan_aware(got_z[r], want_z[r], f"straggler {phase} z rank {r}")
            assert_equal_nan_aware(got_y[r], want_y[r], f"straggler {phase} y rank {r}")
    finally:
        h.close()


# ------------------------------------------------------- two-shot fused kernel
def force_two_shot(h, rows, hidden):
    code, path = sfar.sfar_test_query_fused_path(h.h, rows, hidden)
    assert code == sfar.SFAR_OK and path == 2, (code, path)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [2, 3, 8, 16])
def test_two_shot_parity(R, dtype):
    """Every shape whose rows fit the two-shot kernel (at most 32 KB), with
    the kernel forced: the same bits as the oracle on every rank."""
    h = sfar.Sfar(R, 1 << 20, dtype)
    es = 2 if dtype == "bf16" else 4
    try:
        assert sfar.sfar_test_set_fused_path(h.h, "twoshot") == sfar.SFAR_OK
        for rows, hidden in SHAPES[dtype] + [(7, 2048 // es), (R + 1, 4096 // es)]:
            code, path = sfar.sfar_test_query_fused_path(h.h, rows, hidden)
            if hidden * es > 32768:
                assert code != sfar.SFAR_OK or path == 1              # rows above 32 KB keep the one-shot kernel
                continue
            if path == 1:
                # the two-shot grid cannot be resident at once: R = 16 with rows above 16 KB (clusters of
                # up to 8 CTAs of 256 threads, one CTA per SM)
                assert R == 16 and hidden * es > 16384, (R, rows, hidden, dtype)
                continue
            force_two_shot(h, rows, hidden)
            x, res, w = draw_case(1000 + R + rows, R, rows, hidden, dtype)
            check(h, x, res, w, hidden, 1e-5, f"two-shot R={R} {rows}x{hidden} {dtype}")
    finally:
        h.close()


def test_two_shot_in_place_and_special_rows():
    R, hidden = 4, 1024
    h = sfar.Sfar(R, 1 << 20, "fp32")
    try:
        assert sfar.sfar_test_set_fused_path(h.h, "twoshot") == sfar.SFAR_OK
        force_two_shot(h, 6, hidden)
        x, res, w = draw_case(1101, R, 6, hidden, "fp32")
        res[:, :hidden] = 0.0
        x[:, :hidden] = 0.0                          # row 0: all zero
        x[1, hidden + 7] = float("nan")              # row 1: NaN
        res[2, 2 * hidden + 9] = float("inf")        # row 2: an infinity on rank 2 only
        x[:, 3 * hidden:4 * hidden] *= 2.0 ** 60     # row 3: large
        x[:, 4 * hidden:5 * hidden] *= 2.0 ** -70    # row 4: tiny (subnormal squares)
        res[:, 4 * hidden:5 * hidden] *= 2.0 ** -70
        check(h, x, res, w, hidden, 1e-6, "two-shot special rows")
        check(h, x, res, w, hidden, 1e-6, "two-shot in place", in_place=True)
    finally:
        h.close()


def test_shape_chooses_the_kernel():
    R = 8
    h = sfar.Sfar(R, 2 << 20, "bf16")
    try:
        assert sfar.sfar_test_query_fused_path(h.h, 1, 8192) == (sfar.SFAR_OK, 1)
        assert sfar.sfar_test_query_fused_path(h.h, 64, 7168) == (sfar.SFAR_OK, 2)
        assert sfar.sfar_test_query_fused_path(h.h, 8, 32768)[1] == 1          # 64 KB rows: one-shot only
        assert sfar.sfar_test_set_fused_path(h.h, "oneshot") == sfar.SFAR_OK
        assert sfar.sfar_test_query_fused_path(h.h, 64, 7168) == (sfar.SFAR_OK, 1)
        assert sfar.sfar_test_set_fused_path(h.h, 3) == sfar.SFAR_ERR_INVALID
    finally:
        h.close()


@pytest.mark.parametrize("mode", ["serial", "overlap"])
def test_two_shot_chain_with_other_calls(mode):
    """256 graph-chained calls that cycle through the two-shot fused kernel
    (4 rows), the one-shot fused kernel (1 row), the two-shot TMA AllReduce
    (which shares the arrival and completion flags) and the LL AllReduce,
    each with its own inputs: every result bit for bit.  Each fused call has
    its kernel forced."""
    R, hidden, calls, eps = 8, 8192, 256, 1e-5
    rows_of = lambda c: 4 if c % 4 == 0 else 1
    x = torch.stack([inputs.draw(1200, c, R, 4 * hidden, "normal", 1.0, "bf16") for c in range(calls)])
    res = torch.stack([inputs.draw(1201, c, R, 4 * hidden, "normal", 2.0, "bf16") for c in range(calls)])
    w = inputs.draw(1202, 0, 1, hidden, "normal", 1.0, "bf16")[0]
    h = sfar.Sfar(R, 8 * hidden, "bf16")
    try:
        h.set_mode(mode)
        xd, rd, wd = x.cuda(), res.cuda(), w.cuda()
        od, zd = torch.empty_like(xd), torch.empty_like(xd)
        P = lambda t, c: [t[c, r].data_ptr() for r in range(R)]

        def call(c):
            kind = c % 4
            if kind in (0, 1):
                # the kernel is chosen when the call is enqueued (here: captured)
                assert sfar.sfar_test_set_fused_path(h.h, "twoshot" if kind == 0 else "oneshot") == sfar.SFAR_OK
                assert sfar.sfar_test_query_fused_path(h.h, rows_of(c), hidden) == (sfar.SFAR_OK, 2 - kind)
                return sfar.sfar_allreduce_add_rmsnorm(h.h, P(xd, c), P(rd, c), wd.data_ptr(), P(od, c), P(zd, c),
                                                       rows_of(c), hidden, eps)
            return sfar.sfar_allreduce(h.h, P(xd, c), P(od, c), 4 * hidden, "twoshot_tma" if kind == 2 else "ll")

        assert call(0) == sfar.SFAR_OK
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in range(calls):
                assert call(c) == sfar.SFAR_OK
        od.view(torch.int16).fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"mixed chain {mode}")
        wb = inputs.to_bits(w[None, :])[0]
        for c in range(calls):
            n = rows_of(c) * hidden
            xb = inputs.to_bits(x[c, :, :n]) if c % 4 in (0, 1) else inputs.to_bits(x[c])
            if c % 4 in (0, 1):
                want_y, want_z = oracle.add_rmsnorm(xb, inputs.to_bits(res[c, :, :n]), wb, eps, hidden)
                for r in range(R):
                    assert_equal_nan_aware(zd[c, r, :n], want_z[r], f"{mode} call {c} z rank {r}")
                    assert_equal_nan_aware(od[c, r, :n], want_y[r], f"{mode} call {c} y rank {r}")
            else:
                want = oracle.allreduce(xb)
                for r in range(R):
                    assert np.array_equal(inputs.to_bits(od[c, r].cpu()), want[r]), f"{mode} call {c} rank {r}"
    finally:
        h.close()


@pytest.mark.parametrize("phase", [0, 1])
def test_two_shot_chain_with_straggler(phase):
    """256 graph-chained two-shot calls (8 rows of 7168 bf16, R = 8) in
    overlap mode with one rank (rotating) delayed by 0-20 us before its
    arrival (phase 0) or between its arrival and its reads (phase 1)."""
    R, rows, hidden, calls, eps = 8, 8, 7168, 256, 1e-5
    n = rows * hidden
    x = torch.stack([inputs.draw(1300, c, R, n, "normal", 1.0, "bf16") for c in range(calls)])
    res = torch.stack([inputs.draw(1301, c, R, n, "normal", 2.0, "bf16") for c in range(calls)])
    w = inputs.draw(1302, 0, 1, hidden, "normal", 1.0, "bf16")[0]
    h = sfar.Sfar(R, 2 * n, "bf16")
    try:
        h.set_mode("overlap")
        assert sfar.sfar_test_set_fused_path(h.h, "twoshot") == sfar.SFAR_OK
        force_two_shot(h, rows, hidden)
        xd, rd, wd = x.cuda(), res.cuda(), w.cuda()
        od, zd = torch.empty_like(xd), torch.empty_like(xd)
        P = lambda t, c: [t[c, r].data_ptr() for r in range(R)]
        g = torch.Generator().manual_seed(1303)
        delays = torch.randint(0, 20001, (calls,), generator=g).to(torch.int32).cuda()
        assert sfar.sfar_allreduce_add_rmsnorm(h.h, P(xd, 0), P(rd, 0), wd.data_ptr(), P(od, 0), P(zd, 0), rows,
                                               hidden, eps) == sfar.SFAR_OK
        torch.cuda.synchronize()
        assert sfar.sfar_test_set_straggler(h.h, delays.data_ptr(), calls, -1, phase) == sfar.SFAR_OK
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in range(calls):
                assert sfar.sfar_allreduce_add_rmsnorm(h.h, P(xd, c), P(rd, c), wd.data_ptr(), P(od, c), P(zd, c),
                                                       rows, hidden, eps) == sfar.SFAR_OK
        graph.replay()
        torch.cuda.synchronize()
        status_ok(h.h, f"two-shot straggler phase {phase}")
        want_y, want_z = oracle.add_rmsnorm(inputs.to_bits(x.transpose(0, 1).reshape(R, calls * n)),
                                            inputs.to_bits(res.transpose(0, 1).reshape(R, calls * n)),
                                            inputs.to_bits(w[None, :])[0], eps, hidden)
        got_y = od.transpose(0, 1).reshape(R, calls * n)
        got_z = zd.transpose(0, 1).reshape(R, calls * n)
        for r in range(R):
            assert_equal_nan_aware(got_z[r], want_z[r], f"two-shot straggler {phase} z rank {r}")
            assert_equal_nan_aware(got_y[r], want_y[r], f"two-shot straggler {phase} y rank {r}")
    finally:
        h.close()


def test_two_shot_dropped_rank_times_out_and_reset_recovers():
    R, rows, hidden = 4, 8, 4096
    h = sfar.Sfar(R, 1 << 17, "bf16")
    try:
        assert sfar.sfar_test_set_fused_path(h.h, "twoshot") == sfar.SFAR_OK
        force_two_shot(h, rows, hidden)
        x, res, w = draw_case(1400, R, rows, hidden, "bf16")
        check(h, x, res, w, hidden, 1e-5, "two-shot before")
        assert sfar.sfar_test_set_timeout(h.h, 2_000_000) == sfar.SFAR_OK
        assert sfar.sfar_test_drop_rank(h.h, 1) == sfar.SFAR_OK
        ins = [t.cuda() for t in x]
        rs = [t.cuda() for t in res]
        outs = [torch.empty_like(t) for t in ins]
        zs = [torch.empty_like(t) for t in ins]
        h.allreduce_add_rmsnorm(ins, rs, w.cuda(), outs, zs, hidden, 1e-5)
        torch.cuda.synchronize()
        code, f = sfar.sfar_status_get(h.h)
        assert code == sfar.SFAR_ERR_TIMEOUT and sfar.WAIT_NAMES[f.where] in ("arrive", "complete")
        h.reset()
        assert sfar.sfar_test_drop_rank(h.h, -1) == sfar.SFAR_OK
        torch.cuda.synchronize()
        check(h, x, res, w, hidden, 1e-5, "two-shot after reset")
    finally:
        h.close()


@pytest.mark.parametrize("mode", ["serial", "cooperative"])
def test_large_grid_chain_does_not_stall(mode):
    """A one-shot grid that fills most of the device (R = 8, eight rows of
    8192 bf16: 32 clusters of 8 CTAs) chained in a graph: launched as a plain
    programmatic dependent it sometimes had a cluster that never started (its
    peers timed out).  In serial mode such a grid runs solo; in cooperative
    mode it is a cooperative grid, which the device places whole, and keeps
    the programmatic launch.  Twenty replays of 32 calls with a 50 ms wait
    limit, then the last call against the oracle."""
    R, rows, hidden, calls, eps = 8, 8, 8192, 32, 1e-5
    n = rows * hidden
    x = torch.stack([inputs.draw(1500, c, R, n, "normal", 1.0, "bf16") for c in range(calls)])
    res = torch.stack([inputs.draw(1501, c, R, n, "normal", 2.0, "bf16") for c in range(calls)])
    w = inputs.draw(1502, 0, 1, hidden, "normal", 1.0, "bf16")[0]
    h = sfar.Sfar(R, 2 * n, "bf16")
    try:
        h.set_mode(mode)
        assert sfar.sfar_test_set_fused_path(h.h, "oneshot") == sfar.SFAR_OK
        code, k, cl, t = sfar.sfar_test_query_norm_launch(h.h, rows, hidden)
        assert code == sfar.SFAR_OK and k * R // cl >= 24, (k, cl)          # a grid of most of the device
        assert sfar.sfar_test_set_timeout(h.h, 50_000_000) == sfar.SFAR_OK
        xd, rd, wd = x.cuda(), res.cuda(), w.cuda()
        od, zd = torch.empty_like(xd), torch.empty_like(xd)
        P = lambda t, c: [t[c, r].data_ptr() for r in range(R)]
        f = lambda c: sfar.sfar_allreduce_add_rmsnorm(h.h, P(xd, c), P(rd, c), wd.data_ptr(), P(od, c), P(zd, c),
                                                       rows, hidden, eps)
        assert f(0) == sfar.SFAR_OK
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in range(calls):
                assert f(c) == sfar.SFAR_OK
        for rep in range(20):
            for _ in range(32):
                graph.replay()
            torch.cuda.synchronize()
            status_ok(h.h, f"large grid replay batch {rep}")
        c = calls - 1
        want_y, want_z = oracle.add_rmsnorm(inputs.to_bits(x[c]), inputs.to_bits(res[c]),
                                            inputs.to_bits(w[None, :])[0], eps, hidden)
        for r in range(R):
            assert_equal_nan_aware(zd[c, r], want_z[r], f"large grid z rank {r}")
            assert_equal_nan_aware(od[c, r], want_y[r], f"large grid y rank {r}")
    finally:
        h.close()


def test_solo_grid_between_overlapped_calls():
    """Overlap mode: LL calls, a fused call whose grid runs solo (8 rows of
    8192 bf16, one-shot forced) and more LL calls, all on one handle and in
    one graph; the calls around the solo grid must not overtake it.  Every
    result bit for bit."""
    R, rows, hidden, eps = 8, 8, 8192, 1e-5
    n = rows * hidden
    seq = ["ll", "ll", "fused", "ll", "ll", "fused", "fused", "ll"] * 8
    x = torch.stack([inputs.draw(1600, c, R, n, "normal", 1.0, "bf16") for c in range(len(seq))])
    res = torch.stack([inputs.draw(1601, c, R, n, "normal", 2.0, "bf16") for c in range(len(seq))])
    w = inputs.draw(1602, 0, 1, hidden, "normal", 1.0, "bf16")[0]
    h = sfar.Sfar(R, 2 * n, "bf16")
    try:
        h.set_mode("overlap")
        assert sfar.sfar_test_set_fused_path(h.h, "oneshot") == sfar.SFAR_OK
        xd, rd, wd = x.cuda(), res.cuda(), w.cuda()
        od, zd = torch.empty_like(xd), torch.empty_like(xd)
        P = lambda t, c: [t[c, r].data_ptr() for r in range(R)]

        def call(c):
            if seq[c] == "ll":
                return sfar.sfar_allreduce(h.h, P(xd, c), P(od, c), n, "ll")
            return sfar.sfar_allreduce_add_rmsnorm(h.h, P(xd, c), P(rd, c), wd.data_ptr(), P(od, c), P(zd, c),
                                                   rows, hidden, eps)

        assert call(0) == sfar.SFAR_OK
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in range(len(seq)):
                assert call(c) == sfar.SFAR_OK
        for rep in range(4):
            od.view(torch.int16).fill_(-1)
            graph.replay()
            torch.cuda.synchronize()
            status_ok(h.h, f"solo between overlapped calls, replay {rep}")
        wb = inputs.to_bits(w[None, :])[0]
        for c in range(len(seq)):
            xb = inputs.to_bits(x[c])
            if seq[c] == "ll":
                want = oracle.allreduce(xb)
                for r in range(R):
                    assert np.array_equal(inputs.to_bits(od[c, r].cpu()), want[r]), f"call {c} rank {r}"
            else:
                want_y, want_z = oracle.add_rmsnorm(xb, inputs.to_bits(res[c]), wb, eps, hidden)
                for r in range(R):
                    assert_equal_nan_aware(zd[c, r], want_z[r], f"call {c} z rank {r}")
                    assert_equal_nan_aware(od[c, r], want_y[r], f"call {c} y rank {r}")
    finally:
        h.close()
