"""Positive random features (Performer, "Efficient Attention Variants" s.6)
on the GPU against the fp64 oracle, then linear attention over them."""
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


@pytest.mark.parametrize("d,r", [(64, 64), (64, 128), (128, 128), (32, 200), (100, 37)])
@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
def test_features_match_oracle(orc, d, r, in_dtype):
    x = synth.normal((3, 5, 77, d), seed=91, scale=0.7, dtype=in_dtype, device="cuda")
    w = synth.gaussian_rows(r, d, seed=92, orthogonal=(r % d == 0), device="cuda")
    f32 = la.la_favor_features(x, w)
    ref = orc.favor(to_np(x), to_np(w))
    assert np.all(to_np(f32) > 0)
    # the exponent is an fp32 sum of d products; its rounding (about
    # sqrt(d) 2^-24 sum |w_c x_c|, tens of 2^-24 here) is the relative error
    # of the feature
    rel = np.max(np.abs(to_np(f32) - ref) / ref)
    assert rel < 3e-5, rel
    fbf = la.la_favor_features(x, w, out_dtype=torch.bfloat16)
    relb = np.max(np.abs(to_np(fbf) - ref) / ref)
    assert relb <= 2.0 ** -8, relb


def test_features_many_tiles(orc):
    """Enough rows for every CTA of the tensor-core form to reuse its x stages
    and both accumulators several times (128k rows, 1000 tiles of 128)."""
    x = synth.normal((8, 16, 1000, 64), seed=93, scale=0.7, dtype=torch.bfloat16, device="cuda")
    w = synth.gaussian_rows(128, 64, seed=94, device="cuda")
    f = la.la_favor_features(x, w)
    ref = orc.favor(to_np(x), to_np(w))
    assert np.max(np.abs(to_np(f) - ref) / ref) < 3e-5


@pytest.mark.parametrize("causal", [True, False])
def test_performer_attention(orc, causal):
    """The Performer workload: features of q and k (r = 128), then the
    identity-normalised forward; fp32 features through the CUDA-core path
    (1e-5) and bf16 features through the tensor-core path (2e-3)."""
    w_ = synth.WORKLOADS["favor_n4096_d64_r128_bf16"]
    r = w_.extra["favor_r"]
    q, k, v = synth.qkv(w_, device="cuda", B=1, H=4, N=1500)
    W = synth.gaussian_rows(r, w_.d, seed=w_.seed(30), device="cuda")
    fq_ref, fk_ref = orc.favor(to_np(q), to_np(W)), orc.favor(to_np(k), to_np(W))
    ref = orc.forward(fq_ref, fk_ref, to_np(v), causal=causal, fm="identity_norm")
    fq, fk = la.la_favor_features(q, W), la.la_favor_features(k, W)
    out = la.la_forward(fq, fk, v.float(), causal=causal, feature_map="identity_norm")
    assert rel_err_rows(out, ref) <= TOL[torch.float32] * 10
    # bf16 features (rounded once, checked against the oracle's features in
    # test_features_match_oracle) through the tensor-core path: compared with
    # the oracle's forward over those same bf16 features
    fq, fk = (la.la_favor_features(t, W, out_dtype=torch.bfloat16) for t in (q, k))
    out = la.la_forward(fq, fk, v, causal=causal, feature_map="identity_norm")
    ref_b = orc.forward(to_np(fq), to_np(fk), to_np(v), causal=causal, fm="identity_norm")
    assert rel_err_rows(out, ref_b) <= TOL[torch.bfloat16]


def test_kernel_estimate_converges():
    """With many features the GPU features estimate exp(q.k / sqrt(d))."""
    d, r = 64, 4096 * 8
    gen = torch.Generator().manual_seed(5)
    q = (torch.randn(d, generator=gen) * 0.3).cuda()
    k = (torch.randn(d, generator=gen) * 0.3).cuda()
    W = synth.gaussian_rows(256, d, seed=6, device="cuda")
    ests = []
    for i in range(r // 256):
        W = synth.gaussian_rows(256, d, seed=100 + i, device="cuda")
        ests.append(float((la.la_favor_features(q[None], W) * la.la_favor_features(k[None], W)).sum()))
    est = np.mean(ests)
    exact = float(torch.exp((q * k).sum() / np.sqrt(d)))
    assert abs(est - exact) / exact < 0.01, (est, exact)
