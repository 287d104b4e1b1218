"""The C-ABI library without a GPU: it builds, loads, exports every entry
point the headers declare, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from barrier_free_message_gb300 import _build, sfar

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


def declared_functions():
    names = set()
    for path in HEADERS:
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        for m in re.finditer(r"\b(sfar_[a-z0-9_]+)\s*\(", text):
            if not re.search(r"typedef[^;]*\b" + m.group(1) + r"\b", text):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sfar.lib()


def test_headers_declare_the_boundary():
    names = declared_functions()
    for required in ("sfar_create", "sfar_allreduce", "sfar_destroy", "sfar_status_get", "sfar_reset",
                     "sfar_strerror", "sfar_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = sorted(n for n in declared_functions() if n not in exported)
    assert not missing, missing
    for n in declared_functions():
        getattr(lib, n)   # dlsym through ctypes


def test_binding_covers_every_symbol():
    bound = {name for name, _, _ in sfar._SIGS}
    assert declared_functions() <= bound


def test_create_rejects_bad_arguments_before_cuda(lib):
    for R, mb, dt in [(1, 1024, 0), (17, 1024, 0), (0, 1024, 0), (4, 0, 0), (4, 1024, 2), (4, 1024, -1)]:
        assert lib.sfar_create(R, mb, dt) is None
        assert lib.sfar_last_error() == sfar.SFAR_ERR_INVALID


def test_null_handle_calls(lib):
    ins = (ctypes.c_void_p * 2)()
    assert lib.sfar_allreduce(None, ins, ins, 16, 2, None) == sfar.SFAR_ERR_INVALID
    assert lib.sfar_reset(None, None) == sfar.SFAR_ERR_INVALID
    assert lib.sfar_status_get(None, None) == sfar.SFAR_ERR_INVALID
    assert lib.sfar_set_launch_mode(None, 0) == sfar.SFAR_ERR_INVALID
    assert lib.sfar_max_bytes(None, 2) == 0
    assert lib.sfar_probe_pingpong(None, 1, 0, 1, None, None) == sfar.SFAR_ERR_INVALID
    assert lib.sfar_test_set_geometry(None, 0, 0) == sfar.SFAR_ERR_INVALID
    lib.sfar_destroy(None)


def test_strerror_is_total(lib):
    for code in range(-1, 9):
        s = lib.sfar_strerror(code)
        assert isinstance(s, bytes) and s


def test_create_without_a_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.sfar_create(4, 1 << 16, 0) is None
    assert lib.sfar_last_error() in (sfar.SFAR_ERR_CUDA, sfar.SFAR_ERR_UNSUPPORTED)
