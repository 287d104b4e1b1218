"""The fused normalisation kernels and the row-parallel projection against
plain mathematics, independently of the oracle.

The oracle's residual-add + RMSNorm uses an order-free fixed-point mean
square, and its projection sums in 8 row segments; the kernels are checked
bit for bit against those definitions elsewhere.  Here the same kernels are
held to definitions that share neither choice:

* fused AllReduce + residual add + RMSNorm (both kernels, forced): the
  AllReduce sum a is a numpy binary32 left fold in rank order, z = a + res
  rounded by torch's conversion (bit for bit), and y against a float64
  RMS normalisation of z, y64 = z / sqrt(mean(z^2) + eps) * w, within the
  bound that the binary32 roundings of any mean-square summation allow:
  relative 2^-21 for fp32 outputs, 2^-8 for bf16 (the final rounding and a
  flip at a near-tie), as derived in ``norm_pins.check_vs_float64``;
* the projection: y against the float64 product x W within the bound of
  recursive summation in any order, 2 (k + 1) 2^-24 sum |x_i W_ij| (Higham,
  "Accuracy and Stability of Numerical Algorithms", section 4.2, doubled for
  second-order terms), plus 2^-8 |y64| for the bf16 rounding.
"""
import numpy as np
import pytest
import torch

from barrier_free_message_gb300 import inputs, sfar
from gpu_helpers import ensure_built, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def f32(t):
    return t.detach().cpu().float().numpy()


def narrow(a32, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R,rows,hidden,path", [(8, 1, 8192, "oneshot"), (4, 3, 4096, "oneshot"),
                                                (8, 64, 7168, "twoshot"), (16, 8, 2048, "twoshot")])
def test_fused_against_float64_rmsnorm(R, rows, hidden, path, dtype):
    if dtype == "fp32" and rows * hidden * 4 > (1 << 20):
        rows = (1 << 20) // (hidden * 4)
    n, eps = rows * hidden, 1e-5
    x = inputs.draw(80, 0, R, n, "normal", 1.0, dtype)
    res = inputs.draw(80, 1, R, n, "normal", 2.0, dtype)
    w = inputs.draw(80, 2, 1, hidden, "normal", 1.0, dtype)[0]
    h = sfar.Sfar(R, 1 << 20, dtype)
    try:
        assert sfar.sfar_test_set_fused_path(h.h, path) == sfar.SFAR_OK
        code, chosen = sfar.sfar_test_query_fused_path(h.h, rows, hidden)
        assert code == sfar.SFAR_OK and chosen == (1 if path == "oneshot" else 2)
        ins = [x[r].contiguous().cuda() for r in range(R)]
        rs = [res[r].contiguous().cuda() for r in range(R)]
        outs = [torch.empty_like(t) for t in ins]
        zs = [torch.empty_like(t) for t in ins]
        h.allreduce_add_rmsnorm(ins, rs, w.cuda(), outs, zs, hidden, eps)
        torch.cuda.synchronize()
        status_ok(h.h, "fused")
    finally:
        h.close()
    xs = f32(x)
    acc = xs[0].copy()
    for q in range(1, R):
        acc = (acc + xs[q]).astype(np.float32)          # binary32, round to nearest even
    a = f32(narrow(acc, dtype))
    z_want = narrow((a[None, :] + f32(res)).astype(np.float32), dtype)
    wf = f32(w).astype(np.float64)
    rel = 2.0 ** -21 if dtype == "fp32" else 2.0 ** -8
    for r in range(R):
        assert np.array_equal(bits(zs[r]), bits(z_want[r])), f"{path} R={R} {dtype}: z of rank {r} != T(a + res)"
        zz = f32(z_want[r]).astype(np.float64).reshape(rows, hidden)
        rstd = 1.0 / np.sqrt((zz * zz).mean(axis=1, keepdims=True) + np.float64(np.float32(eps)))
        y64 = (zz * rstd * wf[None, :]).reshape(-1)
        y = f32(outs[r]).astype(np.float64)
        bad = np.abs(y - y64) > rel * np.abs(y64) + 2.0 ** -130
        assert not bad.any(), f"{path} R={R} {dtype}: rank {r}: {int(bad.sum())} of {n} off the float64 RMSNorm"


@pytest.mark.parametrize("R,k,hidden", [(8, 1024, 8192), (8, 3584, 8192), (2, 1000, 2056), (4, 7, 264)])
def test_projection_against_float64_product(R, k, hidden):
    x = inputs.draw(81, 0, R, k, "normal", 1.0, "bf16")
    W = inputs.draw(81, 1, R, k * hidden, "normal", 0.02, "bf16").reshape(R, k, hidden)
    h = sfar.Sfar(R, 1 << 16, "bf16")
    try:
        xs = [x[r].contiguous().cuda() for r in range(R)]
        ws = [W[r].contiguous().cuda() for r in range(R)]
        ys = [torch.empty(hidden, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        h.rowpar_gemv(xs, ws, ys)
        torch.cuda.synchronize()
    finally:
        h.close()
    xf = f32(x).astype(np.float64)
    Wf = W.float().numpy().astype(np.float64)
    y64 = np.einsum("rk,rkh->rh", xf, Wf)
    mag = np.einsum("rk,rkh->rh", np.abs(xf), np.abs(Wf))
    y = np.stack([f32(t) for t in ys]).astype(np.float64)
    bad = np.abs(y - y64) > 2 * (k + 1) * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(y64)
    assert not bad.any(), f"R={R} k={k} h={hidden}: {int(bad.sum())} outputs off the float64 product"
    # and not trivially: a projection that dropped the last eighth of the
    # rows would fail the bound in most outputs
    c = -(-k // 8)
    y_drop = y64 - np.einsum("rk,rkh->rh", xf[:, k - c:], Wf[:, k - c:, :])
    miss = np.abs(y_drop - y64) > 2 * (k + 1) * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(y64)
    assert miss.mean() > 0.5, "the bound is too loose to see a dropped segment"
