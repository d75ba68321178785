"""Sequence split (LASP-2) on the library's kernels, one GPU standing in for
the ranks: every part's own state (la_state), the exclusive prefix of the
gathered states (la_state_prefix) and each part's forward from it
(la_forward_with_state) reproduce the forward over the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, rel_err_rows, to_np

pytestmark = pytest.mark.gpu

la = pytest.importorskip("kernelised_causal_linear_gb300")
from kernelised_causal_linear_gb300 import lasp, synth  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    yield
    assert la.la_get_device_status() == 0


@pytest.mark.parametrize("d,fm,decay,dtype", [(64, "elu1", False, torch.bfloat16),
                                              (128, "none", True, torch.bfloat16),
                                              (64, "elu1", True, torch.float32),
                                              (32, "identity_norm", False, torch.float32)])
def test_emulated_ranks_match_whole_sequence(orc, d, fm, decay, dtype):
    parts = [1000, 1, 3000, 129, 1966]
    w = synth.Workload("lasp", 1, 4, sum(parts), d, d, dtype, q_scale=0.5, k_scale=0.5,
                       v_scale=1 / np.sqrt(d) if fm == "none" else 1.0, feature_map=fm,
                       decay=decay, seed_id=95)
    q, k, v = synth.qkv(w, device="cuda")
    if fm == "identity_norm":
        q, k = q.abs() + 0.01, k.abs() + 0.01
    g = w.gamma()
    out = lasp.lasp2_forward_emulated(q, k, v, parts, feature_map=fm, gamma=g)
    torch.cuda.synchronize()
    ref = orc.forward(to_np(q), to_np(k), to_np(v), fm=fm,
                      gamma=None if g is None else g.double().numpy())
    assert rel_err_rows(out, ref) <= TOL[dtype]


def test_state_prefix_matches_oracle(orc):
    parts = [300, 0, 517, 64]
    w = synth.Workload("lasp2", 2, 3, sum(parts), 64, 128, torch.float32, seed_id=96)
    q, k, v = synth.qkv(w, device="cuda")
    g = torch.tensor([0.99, 0.9, 1.0])
    states, lo = [], 0
    for n in parts:
        states.append(la.la_state(k[:, :, lo:lo + n].contiguous(), v[:, :, lo:lo + n].contiguous(),
                                  gamma=g))
        lo += n
    S_all = torch.stack([s for s, _ in states])
    z_all = torch.stack([z for _, z in states])
    for upto in range(len(parts) + 1):
        S, z = la.la_state_prefix(S_all, z_all, parts, upto, gamma=g)
        n = sum(parts[:upto])
        Sr, zr = orc.state(to_np(k[:, :, :n]), to_np(v[:, :, :n]), gamma=g.double().numpy())
        if n:
            assert rel_err_rows(S, Sr) <= 1e-5 and rel_err_rows(z, zr) <= 1e-5
        else:
            assert torch.count_nonzero(S) == 0 and torch.count_nonzero(z) == 0
