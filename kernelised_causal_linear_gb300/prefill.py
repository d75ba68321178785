"""Prefill helper: the decode state of a batched-decode workload.

Runs la_state over the seeded prefix of every sequence, a slice of sequences
at a time so that the prefix tokens never all sit in device memory at once
(8192 sequences x 4096 tokens x 128 x 2 operands in bf16 would be 17 GB).
"""
from __future__ import annotations

import torch

from . import synth


def prefill_decode_state(w: synth.Workload, device="cuda", batch: int = 512):
    """S [B,H,d,dv] and z [B,H,d] (fp32) after `w.prefix` seeded tokens."""
    from ._binding import la_state, la_state_workspace_size

    BH = w.B * w.H
    S = torch.empty((BH, 1, w.d, w.dv), dtype=torch.float32, device=device)
    z = torch.empty((BH, 1, w.d), dtype=torch.float32, device=device)
    ws = torch.empty(max(16, la_state_workspace_size(batch, 1, w.prefix, w.d, w.dv, w.dtype)),
                     dtype=torch.uint8, device=device)
    g = w.gamma()
    for lo in range(0, BH, batch):
        hi = min(BH, lo + batch)
        k, v = synth.decode_prefix(w, lo, hi, device=device)
        # the flattened sequences of one slice may span several heads: the
        # per-head decay is not supported on this path (none of the decode
        # workloads decays)
        assert g is None
        la_state(k, v, S[lo:hi], z[lo:hi], feature_map=w.feature_map, workspace=ws)
    return S.view(w.B, w.H, w.d, w.dv), z.view(w.B, w.H, w.d)
