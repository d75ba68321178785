"""Per-key-channel decay (GLA, "Efficient Attention Variants" s.7.2) on the
GPU against the fp64 oracle: forward and decode."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, rel_err_rows, to_np

pytestmark = pytest.mark.gpu

la = pytest.importorskip("kernelised_causal_linear_gb300")
from kernelised_causal_linear_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    yield
    assert la.la_get_device_status() == 0


@pytest.mark.parametrize("d,dv", [(32, 32), (64, 64), (128, 128), (64, 128), (128, 32)])
@pytest.mark.parametrize("N", [1, 31, 129, 1000])
@pytest.mark.parametrize("fm", ["elu1", "none"])
def test_gla_forward(orc, d, dv, N, fm):
    for dtype in (torch.float32, torch.bfloat16):
        w = synth.Workload("gla", 2, 3, N, d, dv, dtype, q_scale=0.5, k_scale=0.5,
                           feature_map=fm, seed_id=97)
        q, k, v = synth.qkv(w, device="cuda")
        a = synth.gates((2, 3, N, d), seed=98, lo=0.5, hi=1.0, device="cuda")
        out = la.la_forward_gla(q, k, v, a, feature_map=fm)
        ref = orc.forward(to_np(q), to_np(k), to_np(v), fm=fm, alpha=to_np(a))
        err = rel_err_rows(out, ref)
        assert err <= TOL[dtype], (dtype, err)


def test_gla_strong_and_constant_gates(orc):
    """Gates down to 0.01 (state nearly reset every token) stay finite and
    exact; a gate constant per head equals the scalar decay of that value."""
    w = synth.Workload("gla2", 1, 4, 700, 64, 64, torch.float32, q_scale=0.5, k_scale=0.5,
                       feature_map="none", seed_id=99)
    q, k, v = synth.qkv(w, device="cuda")
    a = synth.gates((1, 4, 700, 64), seed=100, lo=0.01, hi=1.0, device="cuda")
    out = la.la_forward_gla(q, k, v, a, feature_map="none")
    ref = orc.forward(to_np(q), to_np(k), to_np(v), fm="none", alpha=to_np(a))
    assert rel_err_rows(out, ref) <= TOL[torch.float32]
    g = torch.tensor([0.99, 0.9, 0.8, 1.0])
    const = g.view(1, 4, 1, 1).expand(1, 4, 700, 64).contiguous().cuda()
    out_g = la.la_forward_gla(q, k, v, const, feature_map="none")
    out_s = la.la_forward(q, k, v, feature_map="none", gamma=g)
    assert rel_err_rows(out_g, to_np(out_s)) <= 1e-5


def test_gla_decode_continues_forward(orc):
    B, H, N, d = 2, 3, 40, 128
    w = synth.Workload("gla3", B, H, N, d, d, torch.bfloat16, seed_id=101)
    q, k, v = synth.qkv(w, device="cuda")
    a = synth.gates((B, H, N, d), seed=102, lo=0.8, hi=1.0, device="cuda")
    full = la.la_forward_gla(q, k, v, a)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    for t in range(N):
        o = la.la_decode_step_gla(S, z, q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                  v[:, :, t].contiguous(), a[:, :, t].contiguous())
        # bf16 inputs at d = 128: the forward's sub-chunk products run on the
        # tensor cores (bf16 operands, the bf16 tolerance); the decode step is
        # fp32 throughout and meets 1e-5 against the oracle below
        assert rel_err_rows(o, to_np(full[:, :, t])) <= TOL[torch.bfloat16]
    ref = orc.forward(to_np(q), to_np(k), to_np(v), alpha=to_np(a))
    assert rel_err_rows(o, ref[:, :, -1]) <= 1e-5


@pytest.mark.parametrize("lo", [0.5, 0.01])
def test_gla_tensor_core_sub_chunks(orc, lo):
    """bf16 inputs at d = dv = 128 take the tensor-core products in every
    sub-chunk whose decay splits (gates >= 0.5 over 32 tokens) and the fp32
    products where it does not (gates down to 0.01); both forms in one call,
    several blocks and a ragged tail."""
    w = synth.Workload("gla4", 2, 2, 777, 128, 128, torch.bfloat16, q_scale=0.5, k_scale=0.5,
                       feature_map="none", seed_id=103)
    q, k, v = synth.qkv(w, device="cuda")
    a = synth.gates((2, 2, 777, 128), seed=104, lo=lo, hi=1.0, device="cuda")
    for fm in ("none", "elu1"):
        out = la.la_forward_gla(q, k, v, a, feature_map=fm)
        ref = orc.forward(to_np(q), to_np(k), to_np(v), fm=fm, alpha=to_np(a))
        assert rel_err_rows(out, ref) <= TOL[torch.bfloat16], fm
