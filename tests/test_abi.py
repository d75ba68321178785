"""The C-ABI library builds, loads and exports what include/linattn.h
declares; argument errors come back before anything touches a GPU."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    from kernelised_causal_linear_gb300 import build

    return ctypes.CDLL(str(build.build()))


def declared_functions():
    names = []
    for h in sorted((ROOT / "include").glob("*.h")):
        names += re.findall(r"^LA_API\s+[\w\s\*]+?\b(la_\w+)\s*\(", h.read_text(), re.M)
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ("la_forward", "la_state", "la_decode_step", "la_get_device_status",
              "la_status_string", "la_forward_workspace_size", "la_state_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings_and_version(lib):
    lib.la_status_string.restype = ctypes.c_char_p
    for code in range(8):
        s = lib.la_status_string(code).decode()
        assert s.startswith("LA_")
    assert lib.la_version() >= 100


I64, I, SZ, VP = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
FAKE = VP(0x10000)  # 256-aligned, never dereferenced: every call below fails validation first


def fwd(lib, q=FAKE, B=1, H=1, N=8, d=64, dv=64, causal=1, fm=0, gamma=None, dtype=0,
        ws=FAKE, ws_bytes=1 << 30):
    lib.la_forward.restype = I
    lib.la_forward.argtypes = [VP, VP, VP, VP, I64, I64, I64, I, I, I, I,
                               ctypes.POINTER(ctypes.c_float), I, VP, SZ, VP]
    return lib.la_forward(q, FAKE, FAKE, FAKE, B, H, N, d, dv, causal, fm, gamma, dtype, ws,
                          ws_bytes, None)


def test_forward_argument_errors(lib):
    assert fwd(lib, B=0) == 1
    assert fwd(lib, N=-1) == 1
    assert fwd(lib, fm=7) == 1
    assert fwd(lib, dtype=9) == 1
    assert fwd(lib, causal=2) == 1
    assert fwd(lib, d=48) == 2
    assert fwd(lib, dv=256) == 2
    assert fwd(lib, q=None) == 1
    assert fwd(lib, q=VP(0x10004)) == 1                # misaligned
    assert fwd(lib, ws=None) == 6
    assert fwd(lib, ws_bytes=16) == 6
    # a workspace 16-aligned but not 256-aligned is refused before any launch
    assert fwd(lib, ws=VP(0x10010)) == 6
    assert fwd(lib, ws=VP(0x10080)) == 6
    g = (ctypes.c_float * 1)(0.5)
    assert fwd(lib, causal=0, gamma=g) == 2             # decay undefined non-causal
    bad = (ctypes.c_float * 1)(1.5)
    assert fwd(lib, gamma=bad) == 1
    zero = (ctypes.c_float * 1)(0.0)
    assert fwd(lib, gamma=zero) == 1
    big = (ctypes.c_float * 300)(*([0.9] * 300))
    assert fwd(lib, H=300, gamma=big) == 2


def test_workspace_size_queries(lib):
    lib.la_forward_workspace_size.restype = SZ
    lib.la_forward_workspace_size.argtypes = [I64, I64, I64, I, I, I, I]
    assert lib.la_forward_workspace_size(1, 1, 0, 64, 64, 1, 0) == 0
    assert lib.la_forward_workspace_size(1, 1, 8, 48, 64, 1, 0) == 0
    a = lib.la_forward_workspace_size(2, 16, 32768, 64, 64, 1, 0)
    b = lib.la_forward_workspace_size(2, 16, 65536, 64, 64, 1, 0)
    assert 0 < a < b


def test_decode_argument_errors(lib):
    lib.la_decode_step.restype = I
    lib.la_decode_step.argtypes = [VP, VP, VP, VP, VP, VP, I64, I64, I, I, I,
                                   ctypes.POINTER(ctypes.c_float), I, VP]
    assert lib.la_decode_step(None, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, None, 0,
                              None) == 1
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 96, 64, 0, None, 0,
                              None) == 2
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 64, 0, None, 0,
                              None) == 1


def test_binding_refuses_cpu_tensors():
    import torch

    import kernelised_causal_linear_gb300 as la

    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        la.la_forward(q, q, q, out=torch.zeros(1, 1, 4, 64), workspace=torch.zeros(1 << 20, dtype=torch.uint8))
