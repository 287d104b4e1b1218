"""CPU oracle for the barrier-free small-message AllReduce.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the GPU library (``barrier_free_message_gb300``) and never imports
it; the GPU library never imports this package.

The arithmetic lives in ``sfar_oracle.c`` (plain C99): for every element the
R ranks' values are widened to binary32, folded left to right in rank order
0..R-1 with round-to-nearest-even binary32 adds, and rounded once to the
output type; every rank receives the same result.  This module only loads the
compiled object and marshals numpy arrays.

Arrays: bf16 data is carried as ``numpy.uint16`` bit patterns, fp32 as
``numpy.float32``.  ``x`` has shape ``[R, n]``.
"""
import ctypes
import numpy as np

from .build import build_oracle

BF16 = 0
FP32 = 1

_libs = {}


def _lib(mutant: int = 0):
    if mutant not in _libs:
        lib = ctypes.CDLL(build_oracle(mutant))
        vpp = ctypes.POINTER(ctypes.c_void_p)
        lib.sfar_oracle_allreduce.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_int, vpp, vpp]
        lib.sfar_oracle_allreduce.restype = ctypes.c_int
        lib.sfar_oracle_allreduce_mt.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_int, vpp, vpp,
                                                 ctypes.c_int]
        lib.sfar_oracle_allreduce_mt.restype = ctypes.c_int
        lib.sfar_oracle_narrow_bf16.argtypes = [ctypes.c_float]
        lib.sfar_oracle_narrow_bf16.restype = ctypes.c_uint16
        lib.sfar_oracle_widen_bf16.argtypes = [ctypes.c_uint16]
        lib.sfar_oracle_widen_bf16.restype = ctypes.c_float
        lib.sfar_oracle_mutant.restype = ctypes.c_int
        lib.sfar_oracle_narrow_bf16_n.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
        lib.sfar_oracle_narrow_bf16_n.restype = None
        lib.sfar_oracle_add_rmsnorm.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, vpp,
                                                vpp, ctypes.c_void_p, ctypes.c_float, vpp, vpp, ctypes.c_int]
        lib.sfar_oracle_add_rmsnorm.restype = ctypes.c_int
        lib.sfar_oracle_gemv.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_size_t, vpp, vpp, vpp]
        lib.sfar_oracle_gemv.restype = ctypes.c_int
        _libs[mutant] = lib
    return _libs[mutant]


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return FP32
    raise TypeError(f"oracle takes uint16 (bf16 bits) or float32 arrays, got {x.dtype}")


def allreduce(x: np.ndarray, threads: int = 1, mutant: int = 0) -> np.ndarray:
    """Reduce ``x[R, n]`` over its first axis; return ``[R, n]`` with the sum on every rank."""
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must have shape [R, n]")
    R, n = x.shape
    code = _dtype_code(x)
    out = np.empty_like(x)
    ins = (ctypes.c_void_p * R)(*[x[r].ctypes.data for r in range(R)])
    outs = (ctypes.c_void_p * R)(*[out[r].ctypes.data for r in range(R)])
    lib = _lib(mutant)
    if threads > 1:
        rc = lib.sfar_oracle_allreduce_mt(R, n, code, ins, outs, threads)
    else:
        rc = lib.sfar_oracle_allreduce(R, n, code, ins, outs)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (R={R}, n={n})")
    return out


def allreduce_ptrs(R: int, n: int, code: int, in_ptrs, out_ptrs, threads: int = 1) -> None:
    """Same as :func:`allreduce` on raw host addresses (used to time the oracle without copies)."""
    ins = (ctypes.c_void_p * R)(*in_ptrs)
    outs = (ctypes.c_void_p * R)(*out_ptrs)
    lib = _lib()
    rc = (lib.sfar_oracle_allreduce_mt(R, n, code, ins, outs, threads) if threads > 1
          else lib.sfar_oracle_allreduce(R, n, code, ins, outs))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")


def narrow_bf16(f: float, mutant: int = 0) -> int:
    """binary32 -> bf16 bits, round to nearest even (the oracle's own conversion)."""
    return int(_lib(mutant).sfar_oracle_narrow_bf16(f))


def widen_bf16(b: int, mutant: int = 0) -> float:
    return float(_lib(mutant).sfar_oracle_widen_bf16(b))


def narrow_bf16_array(f: np.ndarray, mutant: int = 0) -> np.ndarray:
    """binary32 array -> bf16 bits (uint16), element by element with :func:`narrow_bf16`."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _lib(mutant).sfar_oracle_narrow_bf16_n(f.ctypes.data, out.ctypes.data, f.size)
    return out


def add_rmsnorm(x: np.ndarray, res: np.ndarray, weight: np.ndarray, eps: float, hidden: int,
                allreduce_first: bool = True, mutant: int = 0):
    """AllReduce (or not) + residual add + RMS normalisation, as defined in
    ``sfar_oracle.c``.  x, res: [R, rows * hidden]; weight: [hidden]; same
    dtype (uint16 bf16 bits or float32).  Returns (out, res_out), each
    [R, rows * hidden]."""
    x = np.ascontiguousarray(x)
    res = np.ascontiguousarray(res)
    weight = np.ascontiguousarray(weight)
    if x.ndim != 2 or res.shape != x.shape or weight.shape != (hidden,) or x.shape[1] % hidden:
        raise ValueError("x, res must be [R, rows * hidden] and weight [hidden]")
    if res.dtype != x.dtype or weight.dtype != x.dtype:
        raise TypeError("x, res and weight must share one dtype")
    R, total = x.shape
    code = _dtype_code(x)
    out = np.empty_like(x)
    res_out = np.empty_like(x)
    vp = ctypes.c_void_p * R
    rc = _lib(mutant).sfar_oracle_add_rmsnorm(
        R, total // hidden, hidden, code, vp(*[x[r].ctypes.data for r in range(R)]),
        vp(*[res[r].ctypes.data for r in range(R)]), weight.ctypes.data, float(eps),
        vp(*[out[r].ctypes.data for r in range(R)]), vp(*[res_out[r].ctypes.data for r in range(R)]),
        1 if allreduce_first else 0)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out, res_out


def gemv(x: np.ndarray, W: np.ndarray, mutant: int = 0) -> np.ndarray:
    """Row-parallel projection of every rank, as defined in ``sfar_oracle.c``.
    x: [R, k] bf16 bits (uint16); W: [R, k, h] bf16 bits.  Returns [R, h]."""
    x = np.ascontiguousarray(x)
    W = np.ascontiguousarray(W)
    if x.dtype != np.uint16 or W.dtype != np.uint16:
        raise TypeError("gemv takes bf16 bit patterns (uint16)")
    if x.ndim != 2 or W.ndim != 3 or W.shape[:2] != x.shape:
        raise ValueError("x must be [R, k] and W [R, k, h]")
    R, k = x.shape
    h = W.shape[2]
    y = np.empty((R, h), dtype=np.uint16)
    vp = ctypes.c_void_p * R
    rc = _lib(mutant).sfar_oracle_gemv(R, k, h, vp(*[x[r].ctypes.data for r in range(R)]),
                                       vp(*[W[r].ctypes.data for r in range(R)]),
                                       vp(*[y[r].ctypes.data for r in range(R)]))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return y
