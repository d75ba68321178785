"""la_forward_noalloc: the forward for callers that cannot allocate.

Such callers (a plugin whose host application owns all device memory, or
serving code that must not risk the device-wide synchronisation of
cudaMalloc / cudaFree) hand over only inputs and outputs; the scratch comes
from a fixed array inside the library.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from gpu_util import TOL, rel_err_rows, to_np

pytestmark = pytest.mark.gpu

la = pytest.importorskip("kernelised_causal_linear_gb300")
from kernelised_causal_linear_gb300 import _binding, synth  # noqa: E402


def _raw_noalloc(q, k, v, out, causal, gamma=None):
    """Call the C entry point directly through ctypes."""
    B, H, N, d = q.shape
    dv = v.shape[-1]
    g = None
    keep = None
    if gamma is not None:
        keep = torch.as_tensor(gamma, dtype=torch.float32).contiguous()
        g = ctypes.cast(keep.data_ptr(), ctypes.POINTER(ctypes.c_float))
    return _binding.raw.la_forward_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, d, dv, int(causal), 0,
        g, 0 if q.dtype == torch.bfloat16 else 1, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_matches_la_forward_twice(causal):
    w = synth.WORKLOADS["causal_n2048_d64_bf16"]
    q, k, v = synth.qkv(w, device="cuda")
    ref = la.la_forward(q, k, v, causal=causal)
    for _ in range(2):  # the second call reuses scratch left by the first
        out = torch.full_like(ref, float("nan"))
        assert _raw_noalloc(q, k, v, out, causal) == 0
        torch.cuda.synchronize()
        assert rel_err_rows(out, to_np(ref)) <= TOL[torch.bfloat16]
    assert la.la_get_device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    w = synth.WORKLOADS["causal_n32768_d64_bf16"]
    need = la.la_forward_workspace_size(w.B, w.H, w.N, w.d, w.dv, True, w.dtype)
    assert need > (64 << 20)
    q = torch.empty((w.B, w.H, w.N, w.d), dtype=w.dtype, device="cuda")
    out = torch.empty((w.B, w.H, w.N, w.dv), dtype=torch.float32, device="cuda")
    assert _raw_noalloc(q, q, q, out, True) == 7  # LA_ERR_TOO_LARGE
