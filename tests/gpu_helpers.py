"""Helpers of the GPU tests: device buffers, calls through the C ABI, and
bit-exact comparison with the CPU oracle."""
import numpy as np
import torch

import oracle
from barrier_free_message_gb300 import _build, inputs, sfar

TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}
ONESHOT = ["ll", "ll128", "sentinel", "db", "baseline"]
ALL_PROTOS = ONESHOT + ["twoshot", "twoshot_sent", "twoshot_tma"]
DOUBLE_BUFFERED = ["ll", "ll128", "sentinel", "db", "twoshot", "twoshot_sent"]


def ensure_built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    sfar.lib()


def device_io(x_cpu: torch.Tensor, pad_outputs=0xA5):
    """[R, n] CPU tensor -> separate device allocations per rank, outputs prefilled."""
    R = x_cpu.shape[0]
    ins = [x_cpu[r].contiguous().cuda() for r in range(R)]
    outs = [torch.empty_like(t) for t in ins]
    for o in outs:
        o.view(torch.uint8).fill_(pad_outputs)
    return ins, outs


def expected_bits(x_cpu: torch.Tensor) -> np.ndarray:
    return oracle.allreduce(inputs.to_bits(x_cpu))


def as_uint(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def assert_bits_equal(outs, exp: np.ndarray, ctx=""):
    for r, o in enumerate(outs):
        got = as_uint(inputs.to_bits(o.cpu()))
        want = as_uint(exp[r])
        if not np.array_equal(got, want):
            bad = np.nonzero(got != want)[0]
            i = int(bad[0])
            raise AssertionError(f"{ctx} rank {r}: {bad.size} of {got.size} elements differ; first at {i}: "
                                 f"got {int(got[i]):#x} want {int(want[i]):#x}")


def status_ok(h, ctx=""):
    code, f = sfar.sfar_status_get(h)
    assert code == sfar.SFAR_OK, (f"{ctx}: device status {code} ({sfar.strerror(code)}), rank {f.rank} cta {f.cta} "
                                  f"peer {f.peer} epoch {f.epoch} where {sfar.WAIT_NAMES.get(f.where, f.where)}")


def run_once(handle: sfar.Sfar, x_cpu: torch.Tensor, proto: str):
    ins, outs = device_io(x_cpu)
    handle.allreduce(ins, outs, proto)
    torch.cuda.synchronize()
    status_ok(handle.h, proto)
    return outs
