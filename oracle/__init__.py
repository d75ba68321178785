"""fp64 CPU oracle for causal kernelised linear attention -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never loads it and it never loads the CUDA library; the two share no
code.  The arithmetic lives in ``la_oracle.c`` (plain C, fp64, one thread per
(batch, head) sequence); this module only compiles it with gcc and marshals
numpy arrays through ctypes.

Every function takes the exact input values the GPU reads (bf16 or fp32 data
upcast to fp64 without rounding) and returns fp64 results.

Page citations for each computation are in the header of ``la_oracle.c``:
the causal recurrence ("Efficient Attention Variants", section 5), the
non-causal reassociation (same page, section 4), the RetNet scalar decay
(same page, section 7.1), the GLA per-channel decay (same page, section
7.2), the Performer positive random features (same page, section 6) and the
explicit masked kernel matrix (same page, section 10).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "la_oracle.c"
_BUILD = _HERE / "_build"

FM_ELU1 = 0            # phi = elu + 1, normalised
FM_IDENTITY_NORM = 1   # phi = identity, normalised (hand-worked examples)
FM_NONE = 2            # phi = identity, no normaliser (RetNet decay)

ORC_OK = 0
ORC_ERR_ARG = 1
ORC_ERR_NONPOSITIVE_DEN = 2

_FM_NAMES = {"elu1": FM_ELU1, "identity_norm": FM_IDENTITY_NORM, "none": FM_NONE}

# -ffp-contract=off keeps x86_64 and aarch64 builds bit-identical (no fused
# multiply-add contraction on one machine only).
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread"]


class OracleError(RuntimeError):
    pass


def build(defines: tuple[str, ...] = (), out_dir: Path | None = None, force: bool = False) -> Path:
    """Compile la_oracle.c into a shared library and return its path.

    ``defines`` (e.g. ``("ORC_PLANT_READ_BEFORE_WRITE",)``) is used only by the
    tests that build deliberately broken variants to prove the pins catch them.
    """
    out_dir = Path(out_dir) if out_dir is not None else _BUILD
    out_dir.mkdir(parents=True, exist_ok=True)
    tag = "_".join(d.lower() for d in defines) or "base"
    so = out_dir / f"liblaoracle_{tag}.so"
    if force or not so.exists() or so.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = so.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", *_CFLAGS, *[f"-D{d}" for d in defines], str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, so)
    return so


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, so_path: Path):
        lib = ctypes.CDLL(str(so_path))
        dp = ctypes.POINTER(ctypes.c_double)
        L, I = ctypes.c_long, ctypes.c_int
        lib.orc_phi.argtypes = [dp, dp, L, I]
        lib.orc_phi.restype = None
        lib.orc_forward.argtypes = [dp, dp, dp, dp, L, L, L, L, L, I, I, dp, dp, dp, dp, I]
        lib.orc_forward.restype = I
        lib.orc_state.argtypes = [dp, dp, dp, dp, L, L, L, L, L, I, dp, dp, I, I]
        lib.orc_state.restype = I
        lib.orc_decode_step.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, L, I, dp, dp, I]
        lib.orc_decode_step.restype = I
        lib.orc_favor.argtypes = [dp, dp, dp, L, L, L]
        lib.orc_favor.restype = None
        lib.orc_dense.argtypes = [dp, dp, dp, dp, dp, L, L, L, I, I, ctypes.c_double]
        lib.orc_dense.restype = I
        self.lib = lib
        self.path = Path(so_path)

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _arr(x) -> np.ndarray:
        if hasattr(x, "detach"):  # a torch tensor (CPU); bf16 -> fp32 is exact
            import torch

            x = x.detach().to("cpu")
            if x.dtype == torch.bfloat16 or x.dtype == torch.float16:
                x = x.float()
            x = x.numpy()
        return np.ascontiguousarray(x, dtype=np.float64)

    @staticmethod
    def _p(a: np.ndarray | None):
        if a is None:
            return None
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))

    @staticmethod
    def _fm(fm) -> int:
        return _FM_NAMES[fm] if isinstance(fm, str) else int(fm)

    @staticmethod
    def _check(rc: int, allow_den: bool) -> None:
        if rc == ORC_ERR_ARG:
            raise OracleError("oracle rejected its arguments")
        if rc == ORC_ERR_NONPOSITIVE_DEN and not allow_den:
            raise OracleError("normalised read met a non-positive denominator")

    # -- API -------------------------------------------------------------
    def phi(self, x, fm="elu1") -> np.ndarray:
        x = self._arr(x)
        y = np.empty_like(x)
        self.lib.orc_phi(self._p(x), self._p(y), x.size, self._fm(fm))
        return y

    def forward(self, q, k, v, causal=True, fm="elu1", gamma=None, alpha=None, S0=None,
                z0=None, nthreads=0, allow_nonpositive_den=False) -> np.ndarray:
        """q, k: [B,H,N,d]; v: [B,H,N,dv] -> out [B,H,N,dv] (fp64).

        gamma: [H] scalar decay per head; alpha: [B,H,N,d] per-key-channel
        decay; S0, z0: [B,H,d,dv], [B,H,d] state before the first token."""
        q, k, v = self._arr(q), self._arr(k), self._arr(v)
        B, H, N, d = q.shape
        dv = v.shape[-1]
        assert k.shape == (B, H, N, d) and v.shape == (B, H, N, dv)
        g = None if gamma is None else self._arr(gamma).reshape(H)
        a = None if alpha is None else self._arr(alpha).reshape(B, H, N, d)
        s0 = None if S0 is None else self._arr(S0).reshape(B, H, d, dv)
        zz0 = None if z0 is None else self._arr(z0).reshape(B, H, d)
        out = np.empty((B, H, N, dv), dtype=np.float64)
        rc = self.lib.orc_forward(self._p(q), self._p(k), self._p(v), self._p(out), B, H, N, d,
                                  dv, int(bool(causal)), self._fm(fm), self._p(g), self._p(a),
                                  self._p(s0), self._p(zz0), nthreads)
        self._check(rc, allow_nonpositive_den)
        return out

    def state(self, k, v, fm="elu1", gamma=None, alpha=None, S0=None, z0=None, nthreads=0):
        """State (S [B,H,d,dv], z [B,H,d]) after the N tokens of k, v [B,H,N,*],
        starting from zero or from (S0, z0)."""
        k, v = self._arr(k), self._arr(v)
        B, H, N, d = k.shape
        dv = v.shape[-1]
        g = None if gamma is None else self._arr(gamma).reshape(H)
        a = None if alpha is None else self._arr(alpha).reshape(B, H, N, d)
        init = S0 is not None
        S = self._arr(S0).copy() if init else np.zeros((B, H, d, dv))
        z = self._arr(z0).copy() if init else np.zeros((B, H, d))
        rc = self.lib.orc_state(self._p(k), self._p(v), self._p(S), self._p(z), B, H, N, d, dv,
                                self._fm(fm), self._p(g), self._p(a), int(init), nthreads)
        self._check(rc, True)
        return S, z

    def decode_step(self, S, z, q, k, v, fm="elu1", gamma=None, alpha=None, nthreads=0,
                    allow_nonpositive_den=False):
        """One token per sequence: q, k [B,H,d], v [B,H,dv], alpha [B,H,d] or
        None; returns (out [B,H,dv], S', z') without modifying the arrays
        passed in."""
        q, k, v = self._arr(q), self._arr(k), self._arr(v)
        S, z = self._arr(S).copy(), self._arr(z).copy()
        B, H, d = q.shape
        dv = v.shape[-1]
        g = None if gamma is None else self._arr(gamma).reshape(H)
        a = None if alpha is None else self._arr(alpha).reshape(B, H, d)
        out = np.empty((B, H, dv))
        rc = self.lib.orc_decode_step(self._p(S), self._p(z), self._p(q), self._p(k), self._p(v),
                                      self._p(out), B, H, d, dv, self._fm(fm), self._p(g),
                                      self._p(a), nthreads)
        self._check(rc, allow_nonpositive_den)
        return out, S, z

    def favor(self, x, w) -> np.ndarray:
        """Positive random features: x [..., d], w [r, d] -> [..., r]."""
        x, w = self._arr(x), self._arr(w)
        d = x.shape[-1]
        r = w.shape[0]
        assert w.shape == (r, d)
        xf = np.ascontiguousarray(x.reshape(-1, d))
        y = np.empty((xf.shape[0], r))
        self.lib.orc_favor(self._p(xf), self._p(w), self._p(y), xf.shape[0], d, r)
        return y.reshape(x.shape[:-1] + (r,))

    def dense(self, q, k, v, causal=True, fm="elu1", gamma=1.0, return_weights=False,
              allow_nonpositive_den=False):
        """Explicit N x N evaluation of one sequence: q, k [N,d], v [N,dv]."""
        q, k, v = self._arr(q), self._arr(k), self._arr(v)
        N, d = q.shape
        dv = v.shape[-1]
        out = np.empty((N, dv))
        w = np.empty((N, N)) if return_weights else None
        rc = self.lib.orc_dense(self._p(q), self._p(k), self._p(v), self._p(out), self._p(w), N,
                                d, dv, int(bool(causal)), self._fm(fm), float(gamma))
        self._check(rc, allow_nonpositive_den)
        return (out, w) if return_weights else out


_DEFAULT: Oracle | None = None


def load(defines: tuple[str, ...] = (), out_dir: Path | None = None) -> Oracle:
    """Build (if needed) and load an oracle.  With no defines the result is
    cached and shared."""
    global _DEFAULT
    if not defines and out_dir is None:
        if _DEFAULT is None:
            _DEFAULT = Oracle(build())
        return _DEFAULT
    return Oracle(build(defines, out_dir))
