"""Causal kernelised linear attention for GB300 (sm_103a).

The compute lives in ``liblinattn.so`` (hand-written CUDA behind the C ABI of
``include/linattn.h``).  This package holds that library's sources
(``csrc/``), its build step (``build``), a ctypes binding with the C names
(``la_forward``, ``la_state``, ``la_decode_step``, ...) and the seeded
synthetic-input generator (``synth``) shared by tests and benchmark.

The binding is imported lazily so that ``build`` and ``synth`` can be used
before the library exists; touching any ``la_*`` name without a built
library raises ImportError -- there is no CPU fallback.
"""
from __future__ import annotations

_EXPORTS = {
    "la_forward", "la_forward_noalloc", "la_forward_with_state", "la_favor_features", "la_state_prefix", "la_forward_gla", "la_gla_workspace_size", "la_decode_step_gla", "la_state", "la_decode_step", "la_get_device_status", "la_status_string",
    "la_version", "la_launch_count", "la_debug_set_tc_faults", "la_forward_path", "la_forward_workspace_size", "la_state_workspace_size", "LinAttnError",
}


def __getattr__(name):
    if name in _EXPORTS:
        from . import _binding

        return getattr(_binding, name)
    raise AttributeError(name)
