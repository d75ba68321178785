"""Parity of la_forward / la_state on the GPU against the fp64 oracle."""
from __future__ import annotations

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
    torch.cuda.init()
    yield
    assert la.la_get_device_status() == 0


def _run_workload(orc, w, causal=None, **over):
    causal = w.causal if causal is None else causal
    q, k, v = synth.qkv(w, device="cuda", **over)
    gamma = w.gamma()
    out = la.la_forward(q, k, v, causal=causal, feature_map=w.feature_map, gamma=gamma)
    torch.cuda.synchronize()
    ref = orc.forward(to_np(q), to_np(k), to_np(v), causal=causal, fm=w.feature_map,
                      gamma=None if gamma is None else gamma.double().numpy())
    return out, ref


@pytest.mark.parametrize("name,causal", [
    ("causal_n256_d32_fp32", True),
    ("causal_n2048_d64_bf16", True),
    ("causal_n2048_d64_bf16", False),
    ("causal_n32768_d64_bf16", True),
    ("retnet_n8192_d128_bf16", True),
])
def test_workload_parity(orc, name, causal):
    w = synth.WORKLOADS[name]
    out, ref = _run_workload(orc, w, causal)
    err = rel_err_rows(out, ref)
    print(f"{name} causal={causal}: max row-relative error {err:.3e}")
    assert err <= TOL[w.dtype], err


@pytest.mark.parametrize("d,dv", [(64, 64), (32, 64), (64, 32), (128, 64), (64, 128), (128, 128)])
@pytest.mark.parametrize("N", [1, 31, 129, 1000])
def test_ragged_shapes(orc, d, dv, N):
    """Lengths that are not a multiple of any tile, d != dv, both dtypes."""
    for dtype in (torch.bfloat16, torch.float32):
        w = synth.Workload("ragged", 1, 2, N, d, dv, dtype, q_scale=0.5, k_scale=0.5, seed_id=40)
        for causal in (True, False):
            out, ref = _run_workload(orc, w, causal)
            assert rel_err_rows(out, ref) <= TOL[dtype]


def test_decay_normalised_and_identity(orc):
    """Decay with the normaliser, and the identity feature maps."""
    for fm in ("elu1", "identity_norm", "none"):
        w = synth.Workload("fm", 2, 3, 300, 64, 64, torch.float32, seed_id=41, feature_map=fm,
                           decay=fm != "identity_norm", q_scale=0.3, k_scale=0.3)
        if fm == "identity_norm":
            # positive features keep the normaliser well defined
            q, k, v = (t.abs() + 0.01 for t in synth.qkv(w, device="cuda"))
        else:
            q, k, v = synth.qkv(w, device="cuda")
        g = w.gamma()
        out = la.la_forward(q, k, v, feature_map=fm, gamma=g)
        ref = orc.forward(to_np(q), to_np(k), to_np(v), fm=fm,
                          gamma=None if g is None else g.double().numpy())
        assert rel_err_rows(out, ref) <= 1e-5, fm


def test_worked_example_on_gpu():
    """The hand-worked example (Efficient Attention Variants, section 5.1),
    zero-padded from 2 to 32 features: identity features, normalised."""
    import pins

    g = pins.golden("worked_example_s5_1.json")
    d = 32
    fk = torch.zeros(1, 1, 3, d)
    fk[0, 0, :, :2] = torch.tensor(g["phi_k"], dtype=torch.float32)
    v = torch.zeros(1, 1, 3, d)
    v[0, 0, :, :2] = torch.tensor(g["v"], dtype=torch.float32)
    fq = torch.zeros(1, 1, 3, d)
    fq[0, 0, :, :2] = torch.tensor([[1.0, 1.0], [2.0, 1.0], g["phi_q3"]])
    fk, v, fq = fk.cuda(), v.cuda(), fq.cuda()
    out = la.la_forward(fq, fk, v, feature_map="identity_norm").cpu()
    expect = torch.tensor(g["o3_numerator"], dtype=torch.float32) / g["o3_denominator"]
    assert torch.allclose(out[0, 0, 2, :2], expect, rtol=1e-6, atol=0)
    S, z = la.la_state(fk, v, feature_map="identity_norm")
    assert torch.equal(S[0, 0, :2, :2].cpu(), torch.tensor(g["S3"], dtype=torch.float32))
    assert torch.equal(z[0, 0, :2].cpu(), torch.tensor(g["z3"], dtype=torch.float32))


def test_no_future_leakage_bitwise():
    w = synth.WORKLOADS["causal_n2048_d64_bf16"]
    q, k, v = synth.qkv(w, device="cuda", B=1, H=2)
    base = la.la_forward(q, k, v)
    m = 777
    k2, v2 = k.clone(), v.clone()
    k2[:, :, m:] += 5
    v2[:, :, m:] -= 7
    pert = la.la_forward(q, k2, v2)
    assert torch.equal(base[:, :, :m], pert[:, :, :m])
    assert not torch.equal(base[:, :, m:], pert[:, :, m:])


def test_last_rows_agree_and_determinism():
    w = synth.WORKLOADS["causal_n2048_d64_bf16"]
    q, k, v = synth.qkv(w, device="cuda")
    c1 = la.la_forward(q, k, v, causal=True)
    c2 = la.la_forward(q, k, v, causal=True)
    assert torch.equal(c1, c2), "two runs differ"
    nc = la.la_forward(q, k, v, causal=False)
    assert rel_err_rows(c1[:, :, -1], to_np(nc[:, :, -1])) <= TOL[torch.bfloat16]


def test_state_matches_oracle(orc):
    for name in ("causal_n2048_d64_bf16", "retnet_n8192_d128_bf16"):
        w = synth.WORKLOADS[name]
        q, k, v = synth.qkv(w, device="cuda", B=1)
        g = w.gamma()
        S, z = la.la_state(k, v, feature_map=w.feature_map, gamma=g)
        Sr, zr = orc.state(to_np(k), to_np(v), fm=w.feature_map,
                           gamma=None if g is None else g.double().numpy())
        assert rel_err_rows(S, Sr) <= 1e-5
        assert rel_err_rows(z, zr) <= 1e-5


def test_output_guard_band():
    """Nothing is written outside out[B,H,N,dv]."""
    w = synth.Workload("guard", 1, 3, 257, 64, 64, torch.bfloat16, seed_id=42)
    q, k, v = synth.qkv(w, device="cuda")
    n = w.B * w.H * w.N * w.dv
    buf = torch.full((n + 2048,), 12345.0, device="cuda")
    out = buf[1024:1024 + n].view(w.B, w.H, w.N, w.dv)
    la.la_forward(q, k, v, out=out)
    assert torch.all(buf[:1024] == 12345.0) and torch.all(buf[1024 + n:] == 12345.0)


def test_argument_errors_on_device():
    w = synth.Workload("err", 1, 1, 64, 64, 64, torch.bfloat16, seed_id=43)
    q, k, v = synth.qkv(w, device="cuda")
    with pytest.raises(la.LinAttnError):
        la.la_forward(q, k, v, causal=False, gamma=[0.5])
    with pytest.raises(la.LinAttnError):
        la.la_forward(q, k, v, gamma=[1.5])
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(la.LinAttnError) as e:
        la.la_forward(q, k, v, workspace=ws)
    assert e.value.code == 6
    # N = 0 is a no-op
    z0 = q[:, :, :0]
    la.la_forward(z0, z0, z0)


def test_tensor_core_path_is_taken():
    """The bf16, d = dv = 64 causal workloads run on the single-pass tcgen05
    kernel; the RetNet workload and the non-causal form on the chunked one."""
    for name in ("causal_n2048_d64_bf16", "causal_n32768_d64_bf16"):
        w = synth.WORKLOADS[name]
        assert la.la_forward_path(w.B, w.H, w.N, w.d, w.dv, True, "elu1", False, w.dtype) == "tcgen05"
    w = synth.WORKLOADS["retnet_n8192_d128_bf16"]
    assert la.la_forward_path(w.B, w.H, w.N, w.d, w.dv, True, "none", True,
                              w.dtype) == "tcgen05_chunked"
    assert la.la_forward_path(1, 1, 100, 64, 64, False, "elu1", False,
                              torch.bfloat16) == "tcgen05_chunked"
    assert la.la_forward_path(1, 1, 100, 64, 64, True, "none", True,
                              torch.bfloat16) == "tcgen05_chunked"
    assert la.la_forward_path(1, 1, 100, 64, 64, True, "elu1", False, torch.float32) == "simt"
    # one long sequence: the chunked path uses the whole GPU
    assert la.la_forward_path(1, 1, 1 << 20, 64, 64, True, "elu1", False,
                              torch.bfloat16) == "tcgen05_chunked"


@pytest.mark.parametrize("fm", ["elu1", "identity_norm", "none"])
def test_tensor_core_feature_maps(orc, fm):
    w = synth.Workload("tcfm", 2, 3, 700, 64, 64, torch.bfloat16, q_scale=0.3, k_scale=0.3,
                       feature_map=fm, seed_id=44)
    q, k, v = synth.qkv(w, device="cuda")
    if fm == "identity_norm":
        q, k = q.abs() + 0.01, k.abs() + 0.01
    out = la.la_forward(q, k, v, feature_map=fm)
    ref = orc.forward(to_np(q), to_np(k), to_np(v), fm=fm)
    err = rel_err_rows(out, ref)
    print(f"tcgen05 fm={fm}: {err:.3e}")
    assert err <= TOL[torch.bfloat16]


@pytest.mark.parametrize("B,H,N", [(1, 1, 40000), (3, 1, 5000), (1, 7, 3000), (1, 8, 60000),
                                   (2, 5, 20000), (1, 4, 65536)])
def test_tensor_core_few_sequences_long(orc, B, H, N):
    """Few sequences: with fewer than a GPU's worth the chunked path splits
    each sequence over every SM; from four sequences on the single-pass
    kernel runs them, with many chunks of one sequence in flight at once and
    deep look-backs."""
    w = synth.Workload("few", B, H, N, 64, 64, torch.bfloat16, seed_id=45)
    out, ref = _run_workload(orc, w)
    assert rel_err_rows(out, ref) <= TOL[torch.bfloat16]
    q, k, v = synth.qkv(w, device="cuda")
    assert torch.equal(la.la_forward(q, k, v), la.la_forward(q, k, v))


@pytest.mark.parametrize("B,H,N", [(1, 16, 32768 + 3 * 128), (2, 12, 32700), (5, 8, 32768),
                                   (8, 8, 32768)])
def test_tensor_core_segment_lengths(orc, B, H, N):
    """Enough chunks that a segment holds 4, 5 and 8 chunks on a 152-SM GPU
    (one output group then runs a segment's chunks in order, carrying S_prev
    from chunk to chunk), with ragged and short last segments."""
    w = synth.Workload("seglen", B, H, N, 64, 64, torch.bfloat16, seed_id=46)
    out, ref = _run_workload(orc, w)
    err = rel_err_rows(out, ref)
    print(f"B={B} H={H} N={N}: max row-relative error {err:.3e}")
    assert err <= TOL[torch.bfloat16], err
