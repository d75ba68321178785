"""Parity of la_decode_step on the GPU against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, rel_err_rows, to_np

pytestmark = pytest.mark.gpu

la = pytest.importorskip("kernelised_causal_linear_gb300")
from kernelised_causal_linear_gb300 import prefill, synth  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_decode_workload_sampled_heads(orc):
    """Full batched-decode workload (256 x 32 heads, d=dv=128, 4096-token
    prefix, 1000 steps) in the launch configuration the benchmark times;
    64 sampled sequences are replayed by the oracle from the same bytes and
    compared at every step, plus their final state."""
    w = synth.WORKLOADS["decode_b256_h32_d128_bf16"]
    S, z = prefill.prefill_decode_state(w)
    qs, ks, vs = synth.decode_tokens(w, w.steps, device="cuda")
    BH = w.B * w.H
    rng = np.random.default_rng(99)
    sample = np.sort(rng.choice(BH, size=64, replace=False))
    sample[0], sample[-1] = 0, BH - 1
    outs = torch.empty((w.steps, len(sample), w.dv), dtype=torch.float32, device="cuda")
    idx = torch.as_tensor(sample, device="cuda")
    out = torch.empty((w.B, w.H, w.dv), dtype=torch.float32, device="cuda")
    for t in range(w.steps):
        la.la_decode_step(S, z, qs[t], ks[t], vs[t], out)
        outs[t] = out.view(BH, w.dv)[idx]
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0

    # oracle: the same prefix bytes, then the same tokens
    kp, vp = [], []
    for s in sample:
        a, b = synth.decode_prefix(w, int(s), int(s) + 1, device="cuda")
        kp.append(to_np(a)[0, 0])
        vp.append(to_np(b)[0, 0])
    kp = np.stack(kp)[:, None]
    vp = np.stack(vp)[:, None]
    So, zo = orc.state(kp, vp)
    qn = to_np(qs.view(w.steps, BH, w.d)[:, idx])[:, :, None]
    kn = to_np(ks.view(w.steps, BH, w.d)[:, idx])[:, :, None]
    vn = to_np(vs.view(w.steps, BH, w.dv)[:, idx])[:, :, None]
    ref = np.empty((w.steps, len(sample), w.dv))
    for t in range(w.steps):
        o, So, zo = orc.decode_step(So, zo, qn[t], kn[t], vn[t])
        ref[t] = o[:, 0]
    err = rel_err_rows(outs, ref)
    print(f"decode: max row-relative error over {w.steps} steps: {err:.3e}")
    assert err <= TOL[w.dtype]
    assert rel_err_rows(S.view(BH, w.d, w.dv)[idx], So[:, 0]) <= 1e-5
    assert rel_err_rows(z.view(BH, w.d)[idx][..., None], zo[:, 0][..., None]) <= 1e-5


@pytest.mark.parametrize("d,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("fm,decay", [("elu1", False), ("none", True), ("elu1", True)])
def test_decode_after_prefix_equals_forward(orc, d, dv, fm, decay):
    """Prefill P tokens with la_state, decode M more: the outputs equal
    la_forward over the whole sequence at those positions."""
    P, M = 77, 9
    w = synth.Workload("dec", 2, 3, P + M, d, dv, torch.float32, q_scale=0.5, k_scale=0.5,
                       feature_map=fm, decay=decay, seed_id=50)
    q, k, v = synth.qkv(w, device="cuda")
    g = w.gamma()
    full = la.la_forward(q, k, v, feature_map=fm, gamma=g)
    S, z = la.la_state(k[:, :, :P].contiguous(), v[:, :, :P].contiguous(), feature_map=fm,
                       gamma=g)
    for t in range(P, P + M):
        o = la.la_decode_step(S, z, q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                              v[:, :, t].contiguous(), feature_map=fm, gamma=g)
        assert rel_err_rows(o, to_np(full[:, :, t])) <= 1e-5
    ref = orc.forward(to_np(q), to_np(k), to_np(v), fm=fm,
                      gamma=None if g is None else g.double().numpy())
    assert rel_err_rows(o, ref[:, :, -1]) <= 1e-5


def test_decode_resume_bitwise():
    """Stop, copy the state, resume: identical bits to running straight through."""
    w = synth.Workload("resume", 4, 8, 40, 128, 128, torch.bfloat16, seed_id=51)
    q, k, v = synth.qkv(w, device="cuda")
    S0, z0 = la.la_state(k[:, :, :20].contiguous(), v[:, :, :20].contiguous())
    Sa, za = S0.clone(), z0.clone()
    for t in range(20, 40):
        oa = la.la_decode_step(Sa, za, q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                               v[:, :, t].contiguous())
    Sb, zb = S0.clone(), z0.clone()
    for t in range(20, 30):
        la.la_decode_step(Sb, zb, q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                          v[:, :, t].contiguous())
    Sc, zc = Sb.clone(), zb.clone()  # checkpoint
    del Sb, zb
    for t in range(30, 40):
        ob = la.la_decode_step(Sc, zc, q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                               v[:, :, t].contiguous())
    assert torch.equal(oa, ob) and torch.equal(Sa, Sc) and torch.equal(za, zc)
