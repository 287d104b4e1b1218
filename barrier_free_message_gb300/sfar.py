"""Thin ctypes binding of libsfar (``include/sfar.h``, ``include/sfar_test.h``).

Argument marshalling only: every step of the AllReduce runs in the library's
CUDA kernels.  The functions keep the C names; pointers are plain integers
(``tensor.data_ptr()``) and streams are CUDA stream handles as integers
(``torch.cuda.current_stream().cuda_stream``; ``None`` means the current
torch stream).  The library must have been built (``_build.build()``);
loading it otherwise raises, and there is no CPU fallback.
"""
import ctypes
import os

from . import _build

SFAR_BF16, SFAR_FP32 = 0, 1
SFAR_BASELINE, SFAR_DB, SFAR_LL, SFAR_LL128, SFAR_SENTINEL, SFAR_TWOSHOT, SFAR_TWOSHOT_TMA, \
    SFAR_LL128_ATOMIC, SFAR_TWOSHOT_SENTINEL = range(9)
PROTOS = {"baseline": SFAR_BASELINE, "db": SFAR_DB, "ll": SFAR_LL, "ll128": SFAR_LL128,
          "sentinel": SFAR_SENTINEL, "twoshot": SFAR_TWOSHOT, "twoshot_tma": SFAR_TWOSHOT_TMA,
          "ll128_atomic": SFAR_LL128_ATOMIC, "twoshot_sent": SFAR_TWOSHOT_SENTINEL}
# every protocol but ll128_atomic returns the rank-order fold bit for bit
EXACT_PROTOS = [p for p in PROTOS if p != "ll128_atomic"]
DTYPES = {"bf16": SFAR_BF16, "fp32": SFAR_FP32}
SFAR_OK, SFAR_ERR_INVALID, SFAR_ERR_CUDA, SFAR_ERR_OOM, SFAR_ERR_TIMEOUT, SFAR_ERR_UNSUPPORTED, \
    SFAR_ERR_POISONED = range(7)
SFAR_LAUNCH_SERIAL, SFAR_LAUNCH_OVERLAP, SFAR_LAUNCH_PLAIN, SFAR_LAUNCH_COOPERATIVE = 0, 1, 2, 3
MODES = {"serial": SFAR_LAUNCH_SERIAL, "overlap": SFAR_LAUNCH_OVERLAP, "plain": SFAR_LAUNCH_PLAIN,
         "cooperative": SFAR_LAUNCH_COOPERATIVE}
WAIT_NAMES = {1: "done", 2: "ll", 3: "sentinel", 4: "ready", 5: "bottom", 6: "ll128", 7: "rs", 8: "ag",
              9: "arrive", 10: "complete", 11: "copy", 12: "counter",
              13: "cluster"}


class SfarFault(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int), ("rank", ctypes.c_int), ("cta", ctypes.c_int), ("peer", ctypes.c_int),
                ("epoch", ctypes.c_uint32), ("where", ctypes.c_int)]


class SfarError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})")


_lib = None

# (name, restype, argtypes) of every exported entry point
_SIGS = [
    ("sfar_create", ctypes.c_void_p, [ctypes.c_int, ctypes.c_size_t, ctypes.c_int]),
    ("sfar_last_error", ctypes.c_int, []),
    ("sfar_allreduce", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                      ctypes.c_int, ctypes.c_void_p]),
    ("sfar_status_get", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(SfarFault)]),
    ("sfar_reset", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("sfar_destroy", None, [ctypes.c_void_p]),
    ("sfar_strerror", ctypes.c_char_p, [ctypes.c_int]),
    ("sfar_query_launch", ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    ("sfar_max_bytes", ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int]),
    ("sfar_allreduce_noalloc", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t,
                                              ctypes.c_int, ctypes.c_void_p]),
    ("sfar_noalloc_status", ctypes.c_int, [ctypes.POINTER(SfarFault), ctypes.c_int]),
    ("sfar_test_noalloc_record_failure", ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    ("sfar_allreduce_add_rmsnorm", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                                  ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p]),
    ("sfar_add_rmsnorm", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t,
                                        ctypes.c_float, ctypes.c_void_p]),
    ("sfar_test_set_straggler", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_void_p]),
    ("sfar_test_drop_rank", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    ("sfar_test_set_timeout", ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]),
    ("sfar_test_force_single_buffer", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    ("sfar_set_launch_mode", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    ("sfar_test_set_geometry", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]),
    ("sfar_test_set_trace", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32]),
    ("sfar_rowpar_gemv", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_void_p]),
    ("sfar_test_query_norm_launch", ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                                   ctypes.POINTER(ctypes.c_int)]),
    ("sfar_test_set_fused_path", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    ("sfar_test_query_fused_path", ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t,
                                                  ctypes.POINTER(ctypes.c_int)]),
    ("sfar_probe_empty", ctypes.c_int, [ctypes.c_void_p]),
    ("sfar_probe_pingpong", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_void_p]),
]


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libsfar (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libsfar is not built ({path} missing); run barrier_free_message_gb300._build.build()")
        L = ctypes.CDLL(path)
        for name, res, args in _SIGS:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def strerror(code: int) -> str:
    if _lib is None:
        return f"status {code}"
    return _lib.sfar_strerror(code).decode()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(stream)


def _ptr_array(ptrs):
    return (ctypes.c_void_p * len(ptrs))(*[int(p) for p in ptrs])


def _check(code, what):
    if code != SFAR_OK:
        raise SfarError(code, what)


# ------------------------------------------------------------- C-named calls
def sfar_create(R: int, max_bytes: int, dtype="bf16"):
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    h = lib().sfar_create(R, max_bytes, dt)
    if not h:
        raise SfarError(lib().sfar_last_error(), "sfar_create")
    return h


def sfar_allreduce(h, in_ptrs, out_ptrs, n: int, proto="ll", stream=None) -> int:
    p = PROTOS[proto] if isinstance(proto, str) else int(proto)
    return lib().sfar_allreduce(h, _ptr_array(in_ptrs), _ptr_array(out_ptrs), n, p, _stream(stream))


def sfar_allreduce_add_rmsnorm(h, in_ptrs, res_ptrs, weight_ptr: int, out_ptrs, res_out_ptrs, rows: int,
                               hidden: int, eps: float, stream=None) -> int:
    return lib().sfar_allreduce_add_rmsnorm(h, _ptr_array(in_ptrs), _ptr_array(res_ptrs), int(weight_ptr),
                                            _ptr_array(out_ptrs), _ptr_array(res_out_ptrs), rows, hidden, eps,
                                            _stream(stream))


def sfar_add_rmsnorm(h, a_ptrs, res_ptrs, weight_ptr: int, out_ptrs, res_out_ptrs, rows: int, hidden: int,
                     eps: float, stream=None) -> int:
    return lib().sfar_add_rmsnorm(h, _ptr_array(a_ptrs), _ptr_array(res_ptrs), int(weight_ptr),
                                  _ptr_array(out_ptrs), _ptr_array(res_out_ptrs), rows, hidden, eps, _stream(stream))


def sfar_rowpar_gemv(h, x_ptrs, w_ptrs, y_ptrs, k: int, hidden: int, prefetch_rows: int = 0, stream=None) -> int:
    return lib().sfar_rowpar_gemv(h, _ptr_array(x_ptrs), _ptr_array(w_ptrs), _ptr_array(y_ptrs), k, hidden,
                                  prefetch_rows, _stream(stream))


def sfar_test_query_norm_launch(h, rows: int, hidden: int, allreduce: bool = True):
    """(status, ctas_per_rank, cluster_size, threads_per_cta) of a fused call."""
    k, cl, t = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    code = lib().sfar_test_query_norm_launch(h, rows, hidden, 1 if allreduce else 0, ctypes.byref(k),
                                             ctypes.byref(cl), ctypes.byref(t))
    return code, k.value, cl.value, t.value


FUSED_PATHS = {"auto": 0, "oneshot": 1, "twoshot": 2}


def sfar_test_set_fused_path(h, path="auto") -> int:
    return lib().sfar_test_set_fused_path(h, FUSED_PATHS[path] if isinstance(path, str) else int(path))


def sfar_test_query_fused_path(h, rows: int, hidden: int):
    """(status, path) of sfar_allreduce_add_rmsnorm: 1 one-shot, 2 two-shot."""
    p = ctypes.c_int(0)
    code = lib().sfar_test_query_fused_path(h, rows, hidden, ctypes.byref(p))
    return code, p.value


def sfar_allreduce_noalloc(in_ptrs, out_ptrs, R: int, n: int, dtype="bf16", stream=None) -> int:
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    return lib().sfar_allreduce_noalloc(_ptr_array(in_ptrs), _ptr_array(out_ptrs), R, n, dt, _stream(stream))


def sfar_noalloc_status(clear: bool = False):
    """(code, fault) of sfar_allreduce_noalloc on the current device; clear
    erases a recorded failure."""
    f = SfarFault()
    code = lib().sfar_noalloc_status(ctypes.byref(f), 1 if clear else 0)
    return code, f


def sfar_test_noalloc_record_failure(rank: int, peer: int, where: int) -> int:
    return lib().sfar_test_noalloc_record_failure(rank, peer, where)


def sfar_status_get(h):
    f = SfarFault()
    code = lib().sfar_status_get(h, ctypes.byref(f))
    return code, f


def sfar_reset(h, stream=None) -> int:
    return lib().sfar_reset(h, _stream(stream))


def sfar_destroy(h) -> None:
    if h:
        lib().sfar_destroy(h)


def sfar_query_launch(h, n: int, proto="ll"):
    p = PROTOS[proto] if isinstance(proto, str) else int(proto)
    k, t = ctypes.c_int(), ctypes.c_int()
    _check(lib().sfar_query_launch(h, n, p, ctypes.byref(k), ctypes.byref(t)), "sfar_query_launch")
    return k.value, t.value


def sfar_max_bytes(h, proto="ll") -> int:
    p = PROTOS[proto] if isinstance(proto, str) else int(proto)
    return lib().sfar_max_bytes(h, p)


def sfar_test_set_straggler(h, delays_ptr: int, length: int, rank: int = -1, phase: int = 0, stream=None) -> int:
    return lib().sfar_test_set_straggler(h, delays_ptr, length, rank, phase, _stream(stream))


def sfar_test_drop_rank(h, rank: int, stream=None) -> int:
    return lib().sfar_test_drop_rank(h, rank, _stream(stream))


def sfar_test_set_timeout(h, ns: int, stream=None) -> int:
    return lib().sfar_test_set_timeout(h, ns, _stream(stream))


def sfar_test_force_single_buffer(h, on: bool, stream=None) -> int:
    return lib().sfar_test_force_single_buffer(h, 1 if on else 0, _stream(stream))


def sfar_set_launch_mode(h, mode) -> int:
    m = MODES.get(mode, mode)
    return lib().sfar_set_launch_mode(h, int(m))


def sfar_test_set_geometry(h, ctas_per_rank: int = 0, threads_per_cta: int = 0) -> int:
    return lib().sfar_test_set_geometry(h, ctas_per_rank, threads_per_cta)


def sfar_test_set_trace(h, trace_ptr: int, calls: int) -> int:
    return lib().sfar_test_set_trace(h, trace_ptr, calls)


def sfar_probe_empty(stream=None) -> int:
    return lib().sfar_probe_empty(_stream(stream))


def sfar_probe_pingpong(flags_ptr: int, trips: int, out_ptr: int, relaxed: bool = False, partner: int = 1,
                        stream=None) -> int:
    return lib().sfar_probe_pingpong(flags_ptr, trips, 1 if relaxed else 0, partner, out_ptr, _stream(stream))


# --------------------------------------------------------- convenience class
class Sfar:
    """A handle for R simulated ranks; ``allreduce`` takes lists of CUDA tensors."""

    def __init__(self, R: int, max_bytes: int, dtype: str = "bf16"):
        self.R, self.max_bytes, self.dtype = R, max_bytes, dtype
        self.h = sfar_create(R, max_bytes, dtype)

    def allreduce(self, ins, outs, proto="ll", n=None, stream=None) -> None:
        if len(ins) != self.R or len(outs) != self.R:
            raise ValueError(f"need {self.R} inputs and outputs")
        if n is None:
            n = ins[0].numel()
        code = sfar_allreduce(self.h, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs], n, proto, stream)
        _check(code, "sfar_allreduce")

    def allreduce_add_rmsnorm(self, ins, residuals, weight, outs, residual_outs, hidden: int, eps: float,
                              stream=None) -> None:
        """Tensors of rows * hidden elements per rank; weight of hidden elements."""
        rows = ins[0].numel() // hidden
        code = sfar_allreduce_add_rmsnorm(self.h, [t.data_ptr() for t in ins], [t.data_ptr() for t in residuals],
                                          weight.data_ptr(), [t.data_ptr() for t in outs],
                                          [t.data_ptr() for t in residual_outs], rows, hidden, eps, stream)
        _check(code, "sfar_allreduce_add_rmsnorm")

    def add_rmsnorm(self, a, residuals, weight, outs, residual_outs, hidden: int, eps: float, stream=None) -> None:
        rows = a[0].numel() // hidden
        code = sfar_add_rmsnorm(self.h, [t.data_ptr() for t in a], [t.data_ptr() for t in residuals],
                                weight.data_ptr(), [t.data_ptr() for t in outs], [t.data_ptr() for t in residual_outs],
                                rows, hidden, eps, stream)
        _check(code, "sfar_add_rmsnorm")

    def rowpar_gemv(self, x, w, y, prefetch_rows: int = 0, stream=None) -> None:
        """x: R tensors of k; w: R tensors of k x hidden; y: R tensors of hidden (bf16, on the device)."""
        k, hidden = w[0].shape[0], w[0].shape[1]
        code = sfar_rowpar_gemv(self.h, [t.data_ptr() for t in x], [t.data_ptr() for t in w],
                                [t.data_ptr() for t in y], k, hidden, prefetch_rows, stream)
        _check(code, "sfar_rowpar_gemv")

    def status(self):
        return sfar_status_get(self.h)

    def reset(self, stream=None) -> None:
        _check(sfar_reset(self.h, stream), "sfar_reset")

    def set_mode(self, mode) -> None:
        _check(sfar_set_launch_mode(self.h, mode), "sfar_set_launch_mode")

    def launch(self, n: int, proto="ll"):
        return sfar_query_launch(self.h, n, proto)

    def close(self) -> None:
        if self.h:
            sfar_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
