"""Thin ctypes binding of liblinattn.so with the C ABI's own names.

Only argument marshalling happens here: tensors become device pointers and
sizes, enums become ints, and a non-zero status becomes an exception.  Every
step of the computation runs in the library's CUDA kernels.  There is no
fallback: if the library has not been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from . import build as _build

LIB_PATH: Path = _build.LIB

if not LIB_PATH.exists():
    raise ImportError(
        f"liblinattn.so not found at {LIB_PATH}; build it first with "
        "`python -c 'import __graft_entry__ as g; g.build()'` "
        "(kernelised_causal_linear_gb300.build.build())")

_lib = ctypes.CDLL(str(LIB_PATH))

LA_OK = 0
STATUS_NAMES = {0: "LA_OK", 1: "LA_ERR_INVALID_ARG", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_CUDA",
                4: "LA_ERR_TIMEOUT", 5: "LA_ERR_DEVICE_CHECK", 6: "LA_ERR_WORKSPACE",
                7: "LA_ERR_TOO_LARGE"}
FEATURE_MAPS = {"elu1": 0, "identity_norm": 1, "none": 2}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}

_vp, _i64, _i, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_fp = ctypes.POINTER(ctypes.c_float)

_lib.la_version.restype = _i
_lib.la_version.argtypes = []
_lib.la_status_string.restype = ctypes.c_char_p
_lib.la_status_string.argtypes = [_i]
_lib.la_forward_workspace_size.restype = _sz
_lib.la_forward_workspace_size.argtypes = [_i64, _i64, _i64, _i, _i, _i, _i]
_lib.la_state_workspace_size.restype = _sz
_lib.la_state_workspace_size.argtypes = [_i64, _i64, _i64, _i, _i, _i]
_lib.la_forward.restype = _i
_lib.la_forward.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _i, _i, _fp, _i, _vp,
                            _sz, _vp]
_lib.la_state.restype = _i
_lib.la_state.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _i, _fp, _i, _vp, _sz,
                          _vp]
_lib.la_decode_step.restype = _i
_lib.la_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _i, _i, _fp, _i,
                                _vp]
_lib.la_forward_with_state.restype = _i
_lib.la_forward_with_state.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                       _i, _i, _i, _fp, _i, _vp, _sz, _vp]
_lib.la_gla_workspace_size.restype = _sz
_lib.la_gla_workspace_size.argtypes = [_i64, _i64, _i64, _i, _i]
_lib.la_forward_gla.restype = _i
_lib.la_forward_gla.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _i, _i, _vp,
                                _sz, _vp]
_lib.la_decode_step_gla.restype = _i
_lib.la_decode_step_gla.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _i, _i, _i,
                                    _vp]
_lib.la_state_prefix.restype = _i
_lib.la_state_prefix.argtypes = [_vp, _vp, _i, ctypes.POINTER(ctypes.c_int64), _i, _vp, _vp, _i64,
                                 _i64, _i, _i, _fp, _vp]
_lib.la_favor_features.restype = _i
_lib.la_favor_features.argtypes = [_vp, _vp, _vp, _i64, _i, _i, _i, _i, _vp]
_lib.la_forward_noalloc.restype = _i
_lib.la_forward_noalloc.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _i, _i, _fp,
                                    _i, _vp]
_lib.la_forward_path.restype = ctypes.c_char_p
_lib.la_forward_path.argtypes = [_i64, _i64, _i64, _i, _i, _i, _i, _i, _i]
_lib.la_debug_set_tc_faults.restype = _i
_lib.la_debug_set_tc_faults.argtypes = [ctypes.c_uint64, _i]
_lib.la_launch_count.restype = ctypes.c_uint64
_lib.la_launch_count.argtypes = []
_lib.la_get_device_status.restype = _i
_lib.la_get_device_status.argtypes = [_vp]


class LinAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {la_status_string(code)}")


def la_version() -> int:
    return _lib.la_version()


def la_status_string(code: int) -> str:
    return _lib.la_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != LA_OK:
        raise LinAttnError(code, where)


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _gamma_arg(gamma, H: int):
    if gamma is None:
        return None, None
    g = torch.as_tensor(gamma, dtype=torch.float32, device="cpu").contiguous().reshape(-1)
    if g.numel() != H:
        raise ValueError(f"gamma must have H={H} entries, got {g.numel()}")
    return ctypes.cast(g.data_ptr(), _fp), g  # keep g alive for the call


def _fm(feature_map) -> int:
    return FEATURE_MAPS[feature_map] if isinstance(feature_map, str) else int(feature_map)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in DTYPES:
        raise TypeError(f"unsupported input dtype {t.dtype}; use bfloat16 or float32")
    return DTYPES[t.dtype]


def _dev_ptr(t: torch.Tensor | None, name: str) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def la_forward_workspace_size(B, H, N, d, dv, causal=True, dtype=torch.bfloat16) -> int:
    return int(_lib.la_forward_workspace_size(B, H, N, d, dv, int(bool(causal)),
                                              DTYPES[dtype]))


def la_state_workspace_size(B, H, N, d, dv, dtype=torch.bfloat16) -> int:
    return int(_lib.la_state_workspace_size(B, H, N, d, dv, DTYPES[dtype]))


def la_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None,
               *, causal: bool = True, feature_map="elu1", gamma=None,
               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q, k: [B,H,N,d]; v: [B,H,N,dv] (bf16 or fp32, CUDA) -> out [B,H,N,dv] fp32.

    ``workspace`` may be passed to reuse scratch across calls (a uint8 CUDA
    tensor of at least la_forward_workspace_size() bytes); otherwise one is
    allocated by PyTorch for this call.
    """
    B, H, N, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    need = la_forward_workspace_size(B, H, N, d, dv, causal, q.dtype) if q.dtype in DTYPES else 0
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    gp, _keep = _gamma_arg(gamma, H)
    code = _lib.la_forward(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                           _dev_ptr(out, "out"), B, H, N, d, dv, int(bool(causal)),
                           _fm(feature_map), gp, _dtype(q), _dev_ptr(workspace, "workspace"),
                           workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(code, "la_forward")
    return out


def la_forward_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                       *, causal: bool = True, feature_map="elu1", gamma=None,
                       stream=None) -> torch.Tensor:
    """la_forward with no workspace argument and no allocation anywhere: for
    callers that cannot allocate device memory (their host application owns
    all of it, or they must not risk the device-wide synchronisation of
    cudaMalloc / cudaFree).  Scratch comes from a fixed device array inside the
    library; ``out`` must be given, since creating it would allocate.  Calls
    that overlap on the GPU share that array and race."""
    B, H, N, d = q.shape
    dv = v.shape[-1]
    gp, _keep = _gamma_arg(gamma, H)
    code = _lib.la_forward_noalloc(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                   _dev_ptr(out, "out"), B, H, N, d, dv, int(bool(causal)),
                                   _fm(feature_map), gp, _dtype(q), _stream_handle(stream))
    _check(code, "la_forward_noalloc")
    return out


def la_forward_with_state(q: torch.Tensor | None, k: torch.Tensor, v: torch.Tensor,
                          out: torch.Tensor | None = None, *, S0: torch.Tensor | None = None,
                          z0: torch.Tensor | None = None, S_out: torch.Tensor | None = None,
                          z_out: torch.Tensor | None = None, return_state: bool = True,
                          feature_map="elu1", gamma=None, workspace: torch.Tensor | None = None,
                          stream=None):
    """Causal forward continued from (S0, z0) [B,H,d,dv] / [B,H,d] (None: zero
    state), returning (out, S_out, z_out).  q = None computes the final state
    only (out is then None).  S_out / z_out may be S0 / z0 (in-place)."""
    B, H, N, d = k.shape
    dv = v.shape[-1]
    if q is not None and out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=k.device)
    if return_state and S_out is None:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32, device=k.device)
        z_out = torch.empty((B, H, d), dtype=torch.float32, device=k.device)
    need = la_forward_workspace_size(B, H, N, d, dv, True, k.dtype) if k.dtype in DTYPES else 0
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=k.device)
    gp, _keep = _gamma_arg(gamma, H)
    code = _lib.la_forward_with_state(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(out, "out"),
        _dev_ptr(S0, "S0"), _dev_ptr(z0, "z0"), _dev_ptr(S_out, "S_out"), _dev_ptr(z_out, "z_out"),
        B, H, N, d, dv, _fm(feature_map), gp, _dtype(k), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(code, "la_forward_with_state")
    return out, S_out, z_out


def la_state(k: torch.Tensor, v: torch.Tensor, S: torch.Tensor | None = None,
             z: torch.Tensor | None = None, *, feature_map="elu1", gamma=None,
             workspace: torch.Tensor | None = None, stream=None):
    """State after the N tokens of k [B,H,N,d], v [B,H,N,dv] -> (S [B,H,d,dv], z [B,H,d])."""
    B, H, N, d = k.shape
    dv = v.shape[-1]
    if S is None:
        S = torch.empty((B, H, d, dv), dtype=torch.float32, device=k.device)
    if z is None:
        z = torch.empty((B, H, d), dtype=torch.float32, device=k.device)
    need = la_state_workspace_size(B, H, N, d, dv, k.dtype) if k.dtype in DTYPES else 0
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=k.device)
    gp, _keep = _gamma_arg(gamma, H)
    code = _lib.la_state(_dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(S, "S"), _dev_ptr(z, "z"),
                         B, H, N, d, dv, _fm(feature_map), gp, _dtype(k),
                         _dev_ptr(workspace, "workspace"),
                         workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(code, "la_state")
    return S, z


def la_decode_step(S: torch.Tensor, z: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
                   v: torch.Tensor, out: torch.Tensor | None = None, *, feature_map="elu1",
                   gamma=None, stream=None) -> torch.Tensor:
    """One token per sequence: q, k [B,H,d], v [B,H,dv]; S, z updated in place."""
    B, H, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    gp, _keep = _gamma_arg(gamma, H)
    code = _lib.la_decode_step(_dev_ptr(S, "S"), _dev_ptr(z, "z"), _dev_ptr(q, "q"),
                               _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(out, "out"), B, H, d,
                               dv, _fm(feature_map), gp, _dtype(q), _stream_handle(stream))
    _check(code, "la_decode_step")
    return out


def la_gla_workspace_size(B, H, N, d, dv) -> int:
    return int(_lib.la_gla_workspace_size(B, H, N, d, dv))


def la_forward_gla(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor,
                   out: torch.Tensor | None = None, *, feature_map="elu1",
                   workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal forward with per-key-channel decay alpha [B,H,N,d] (fp32, in (0, 1])."""
    B, H, N, d = q.shape
    dv = v.shape[-1]
    if alpha.dtype != torch.float32:
        raise TypeError("alpha must be float32")
    if out is None:
        out = torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    need = int(_lib.la_gla_workspace_size(B, H, N, d, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    code = _lib.la_forward_gla(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                               _dev_ptr(alpha, "alpha"), _dev_ptr(out, "out"), B, H, N, d, dv,
                               _fm(feature_map), _dtype(q), _dev_ptr(workspace, "workspace"),
                               workspace.numel() * workspace.element_size(),
                               _stream_handle(stream))
    _check(code, "la_forward_gla")
    return out


def la_decode_step_gla(S, z, q, k, v, alpha, out=None, *, feature_map="elu1", stream=None):
    """One token per sequence with per-key-channel decay alpha [B,H,d] (fp32)."""
    B, H, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    code = _lib.la_decode_step_gla(_dev_ptr(S, "S"), _dev_ptr(z, "z"), _dev_ptr(q, "q"),
                                   _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(alpha, "alpha"),
                                   _dev_ptr(out, "out"), B, H, d, dv, _fm(feature_map), _dtype(q),
                                   _stream_handle(stream))
    _check(code, "la_decode_step_gla")
    return out


def la_state_prefix(S_parts: torch.Tensor, z_parts: torch.Tensor, part_len, upto: int,
                    S_out: torch.Tensor | None = None, z_out: torch.Tensor | None = None, *,
                    gamma=None, stream=None):
    """State before part `upto` from every part's own state: S_parts
    [P,B,H,d,dv], z_parts [P,B,H,d], part_len P token counts -> (S, z)."""
    P, B, H, d, dv = S_parts.shape
    if S_out is None:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32, device=S_parts.device)
    if z_out is None:
        z_out = torch.empty((B, H, d), dtype=torch.float32, device=S_parts.device)
    lens = (ctypes.c_int64 * P)(*[int(x) for x in part_len])
    gp, _keep = _gamma_arg(gamma, H)
    code = _lib.la_state_prefix(_dev_ptr(S_parts, "S_parts"), _dev_ptr(z_parts, "z_parts"), P,
                                lens, int(upto), _dev_ptr(S_out, "S_out"), _dev_ptr(z_out, "z_out"),
                                B, H, d, dv, gp, _stream_handle(stream))
    _check(code, "la_state_prefix")
    return S_out, z_out


def la_favor_features(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None, *,
                      out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """Positive random features of x [..., d] with Gaussian rows w [r, d]
    (fp32): exp(w . x' - |x'|^2 / 2) / sqrt(r), x' = x / d^(1/4) -> [..., r]."""
    d = x.shape[-1]
    r = w.shape[0]
    if w.dtype != torch.float32 or tuple(w.shape) != (r, d):
        raise ValueError("w must be a float32 [r, d] tensor")
    if out is None:
        out = torch.empty(x.shape[:-1] + (r,), dtype=out_dtype, device=x.device)
    code = _lib.la_favor_features(_dev_ptr(x, "x"), _dev_ptr(w, "w"), _dev_ptr(out, "out"),
                                  x.numel() // d, d, r, _dtype(x), DTYPES[out.dtype],
                                  _stream_handle(stream))
    _check(code, "la_favor_features")
    return out


def la_forward_path(B, H, N, d, dv, causal=True, feature_map="elu1", has_decay=False,
                    dtype=torch.bfloat16) -> str:
    return _lib.la_forward_path(B, H, N, d, dv, int(bool(causal)), _fm(feature_map),
                                int(bool(has_decay)), DTYPES[dtype]).decode()


def la_debug_set_tc_faults(wait_ns: int, withheld_segment: int = -1) -> None:
    """Test hook of the single-pass kernel's give-up path (see linattn.h)."""
    _check(_lib.la_debug_set_tc_faults(int(wait_ns), int(withheld_segment)),
           "la_debug_set_tc_faults")


def la_launch_count() -> int:
    return int(_lib.la_launch_count())


def la_get_device_status(stream=None) -> int:
    return int(_lib.la_get_device_status(_stream_handle(stream)))


# raw handle, for callers that want the C functions directly (tests of the ABI)
raw = _lib
