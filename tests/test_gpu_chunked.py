"""Parity of the chunked tensor-core path (segment aggregates, scan, outputs)
against the fp64 oracle: every feature map, d and dv in {64, 128}, causal
and not, the scalar decay, initial and final states, ragged lengths."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL, rel_err_rows, to_np

pytestmark = pytest.mark.gpu

la = pytest.importorskip("kernelised_causal_linear_gb300")
from kernelised_causal_linear_gb300 import synth  # noqa: E402

BF = torch.bfloat16


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


def _inputs(B, H, N, d, dv, fm, seed, scale=0.5):
    w = synth.Workload("chunked", B, H, N, d, dv, BF, q_scale=scale, k_scale=scale,
                       feature_map=fm, seed_id=seed)
    q, k, v = synth.qkv(w, device="cuda")
    if fm == "identity_norm":  # positive features keep the normaliser defined
        q, k = q.abs() + 0.01, k.abs() + 0.01
    return q, k, v


def _gamma(H):
    return torch.tensor([1.0 - 2.0 ** (-5 - (h % 8)) for h in range(H)], dtype=torch.float32)


def test_paths_reported():
    assert la.la_forward_path(4, 8, 8192, 128, 128, True, "none", True, BF) == "tcgen05_chunked"
    assert la.la_forward_path(4, 8, 2048, 64, 64, False, "elu1", False, BF) == "tcgen05_chunked"
    assert la.la_forward_path(1, 1, 100, 128, 64, True, "elu1", False, BF) == "tcgen05_chunked"
    assert la.la_forward_path(4, 8, 100, 64, 64, True, "elu1", False, BF) == "tcgen05"
    assert la.la_forward_path(1, 1, 100, 64, 64, True, "elu1", False, BF) == "tcgen05_chunked"
    # decay with a normalised map and the d = 32 shapes stay on the CUDA cores
    assert la.la_forward_path(1, 1, 100, 64, 64, True, "elu1", True, BF) == "simt"
    assert la.la_forward_path(1, 1, 100, 32, 64, True, "elu1", False, BF) == "simt"


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("fm", ["elu1", "identity_norm", "none"])
@pytest.mark.parametrize("causal", [True, False])
def test_chunked_forward(orc, d, dv, fm, causal):
    """Ragged length spanning several chunks and segments."""
    N = 1000 if causal else 777
    q, k, v = _inputs(2, 3, N, d, dv, fm, seed=60)
    if causal and d == 64 and dv == 64:  # route around the single-pass kernel
        out, _, _ = la.la_forward_with_state(q, k, v, feature_map=fm)
    else:
        out = la.la_forward(q, k, v, causal=causal, feature_map=fm)
    torch.cuda.synchronize()
    ref = orc.forward(to_np(q), to_np(k), to_np(v), causal=causal, fm=fm)
    err = rel_err_rows(out, ref)
    print(f"d={d} dv={dv} fm={fm} causal={causal}: {err:.3e}")
    assert err <= TOL[BF], err


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128)])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 3000])
def test_chunked_decay(orc, d, dv, N):
    """RetNet form: no feature map, no normaliser, per-head gamma."""
    q, k, v = _inputs(1, 4, N, d, dv, "none", seed=61, scale=1 / np.sqrt(d))
    g = _gamma(4)
    out = la.la_forward(q, k, v, feature_map="none", gamma=g)
    torch.cuda.synchronize()
    ref = orc.forward(to_np(q), to_np(k), to_np(v), fm="none", gamma=g.double().numpy())
    err = rel_err_rows(out, ref)
    print(f"decay d={d} N={N}: {err:.3e}")
    assert err <= TOL[BF], err


def test_fast_decay_takes_the_cuda_cores(orc):
    """gamma < 2^-1/2 is served by the CUDA-core path (the tensor-core form
    factors gamma^(i-j) into gamma^(i+1) gamma^-(j+1)), with the same results."""
    q, k, v = _inputs(1, 2, 700, 128, 128, "none", seed=70, scale=1 / np.sqrt(128))
    for g in ([0.5, 0.9], [0.7072, 0.75]):
        g = torch.tensor(g, dtype=torch.float32)
        out = la.la_forward(q, k, v, feature_map="none", gamma=g)
        ref = orc.forward(to_np(q), to_np(k), to_np(v), fm="none", gamma=g.double().numpy())
        assert rel_err_rows(out, ref) <= TOL[BF]


@pytest.mark.parametrize("B,H,N", [(1, 1, 40000), (2, 3, 9000), (1, 16, 4096)])
def test_chunked_many_segments(orc, B, H, N):
    """Long sequences: many segments per sequence, the scan carries the state
    across all of them."""
    q, k, v = _inputs(B, H, N, 128, 128, "none", seed=62, scale=1 / np.sqrt(128))
    g = _gamma(H)
    out = la.la_forward(q, k, v, feature_map="none", gamma=g)
    ref = orc.forward(to_np(q), to_np(k), to_np(v), fm="none", gamma=g.double().numpy())
    assert rel_err_rows(out, ref) <= TOL[BF]
    q, k, v = _inputs(B, H, N, 64, 64, "elu1", seed=63)
    out, _, _ = la.la_forward_with_state(q, k, v)
    ref = orc.forward(to_np(q), to_np(k), to_np(v))
    assert rel_err_rows(out, ref) <= TOL[BF]


@pytest.mark.parametrize("fm,decay", [("elu1", False), ("none", True), ("elu1", True),
                                      ("identity_norm", False)])
@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128)])
def test_chunked_state(orc, fm, decay, d, dv):
    """la_state on the tensor cores (the prefill that hands over to decode)."""
    q, k, v = _inputs(2, 4, 2500, d, dv, fm, seed=64)
    g = _gamma(4) if decay else None
    S, z = la.la_state(k, v, feature_map=fm, gamma=g)
    Sr, zr = orc.state(to_np(k), to_np(v), fm=fm, gamma=None if g is None else g.double().numpy())
    assert rel_err_rows(S, Sr) <= 1e-5
    assert rel_err_rows(z, zr) <= 1e-5


@pytest.mark.parametrize("fm,decay,d,dv", [("elu1", False, 64, 64), ("none", True, 128, 128),
                                           ("elu1", True, 128, 64), ("identity_norm", False, 64, 128)])
def test_state_many_sequences(orc, fm, decay, d, dv):
    """la_state over hundreds of sequences (the prefill before decode), with
    and without an initial state: the totals are summed one row per thread."""
    B, H, N = 40, 8, 700
    q, k, v = _inputs(B, H, N, d, dv, fm, seed=71)
    g = _gamma(H) if decay else None
    gd = None if g is None else g.double().numpy()
    S, z = la.la_state(k, v, feature_map=fm, gamma=g)
    Sr, zr = orc.state(to_np(k), to_np(v), fm=fm, gamma=gd)
    assert rel_err_rows(S, Sr) <= 1e-5 and rel_err_rows(z, zr) <= 1e-5
    # continued from a state: the second half from the first half's state
    P = 300
    _, S1, z1 = la.la_forward_with_state(None, k[:, :, :P].contiguous(), v[:, :, :P].contiguous(),
                                         feature_map=fm, gamma=g)
    _, S2, z2 = la.la_forward_with_state(None, k[:, :, P:].contiguous(), v[:, :, P:].contiguous(),
                                         S0=S1, z0=z1, feature_map=fm, gamma=g)
    assert rel_err_rows(S2, Sr) <= 1e-5 and rel_err_rows(z2, zr) <= 1e-5


@pytest.mark.parametrize("fm,decay,d", [("elu1", False, 64), ("none", True, 128),
                                        ("elu1", False, 128), ("identity_norm", False, 64)])
def test_forward_with_state_continues(orc, fm, decay, d):
    """A prefix through la_forward_with_state, the rest continued from its
    final state: outputs and the final state equal those of the whole
    sequence (the state summarises the prefix)."""
    B, H, P, M = 2, 3, 1300, 900
    q, k, v = _inputs(B, H, P + M, d, d, fm, seed=65)
    g = _gamma(H) if decay else None
    gd = None if g is None else g.double().numpy()
    out1, S1, z1 = la.la_forward_with_state(q[:, :, :P].contiguous(), k[:, :, :P].contiguous(),
                                            v[:, :, :P].contiguous(), feature_map=fm, gamma=g)
    out2, S2, z2 = la.la_forward_with_state(q[:, :, P:].contiguous(), k[:, :, P:].contiguous(),
                                            v[:, :, P:].contiguous(), S0=S1, z0=z1,
                                            feature_map=fm, gamma=g)
    torch.cuda.synchronize()
    ref = orc.forward(to_np(q), to_np(k), to_np(v), fm=fm, gamma=gd)
    assert rel_err_rows(out1, ref[:, :, :P]) <= TOL[BF]
    assert rel_err_rows(out2, ref[:, :, P:]) <= TOL[BF]
    Sr, zr = orc.state(to_np(k), to_np(v), fm=fm, gamma=gd)
    assert rel_err_rows(S2, Sr) <= 1e-5
    assert rel_err_rows(z2, zr) <= 1e-5
    # the continuation against the oracle's own continued forward
    S0r, z0r = orc.state(to_np(k[:, :, :P]), to_np(v[:, :, :P]), fm=fm, gamma=gd)
    ref2 = orc.forward(to_np(q[:, :, P:]), to_np(k[:, :, P:]), to_np(v[:, :, P:]), fm=fm,
                       gamma=gd, S0=S0r, z0=z0r)
    assert rel_err_rows(out2, ref2) <= TOL[BF]


def test_forward_with_state_in_place_and_state_only(orc):
    B, H, N, d = 1, 2, 700, 64
    q, k, v = _inputs(B, H, 2 * N, d, d, "elu1", seed=66)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    # state only (q = None), in place, two pieces
    for lo in (0, N):
        o, S, z = la.la_forward_with_state(None, k[:, :, lo:lo + N].contiguous(),
                                           v[:, :, lo:lo + N].contiguous(), S0=S, z0=z,
                                           S_out=S, z_out=z)
        assert o is None
    Sr, zr = orc.state(to_np(k), to_np(v))
    assert rel_err_rows(S, Sr) <= 1e-5 and rel_err_rows(z, zr) <= 1e-5
    # N = 0 copies the initial state
    e = q[:, :, :0]
    _, S2, z2 = la.la_forward_with_state(e, e, e, S0=S, z0=z)
    assert torch.equal(S2, S) and torch.equal(z2, z)


def test_forward_with_state_simt_path(orc):
    """fp32 inputs and d = 32 take the CUDA-core path, which carries the
    states the same way."""
    for dtype, d in ((torch.float32, 64), (BF, 32)):
        w = synth.Workload("simt_state", 1, 2, 600, d, d, dtype, q_scale=0.5, k_scale=0.5,
                           seed_id=67)
        q, k, v = synth.qkv(w, device="cuda")
        P = 250
        _, S1, z1 = la.la_forward_with_state(q[:, :, :P].contiguous(), k[:, :, :P].contiguous(),
                                             v[:, :, :P].contiguous())
        out2, S2, z2 = la.la_forward_with_state(q[:, :, P:].contiguous(), k[:, :, P:].contiguous(),
                                                v[:, :, P:].contiguous(), S0=S1, z0=z1)
        ref = orc.forward(to_np(q), to_np(k), to_np(v))
        assert rel_err_rows(out2, ref[:, :, P:]) <= TOL[dtype]
        Sr, zr = orc.state(to_np(k), to_np(v))
        assert rel_err_rows(S2, Sr) <= 1e-5 and rel_err_rows(z2, zr) <= 1e-5


def test_chunked_deterministic_and_causal():
    q, k, v = _inputs(1, 4, 3000, 128, 128, "none", seed=68, scale=1 / np.sqrt(128))
    g = _gamma(4)
    a = la.la_forward(q, k, v, feature_map="none", gamma=g)
    b = la.la_forward(q, k, v, feature_map="none", gamma=g)
    assert torch.equal(a, b)
    m = 1111
    k2, v2 = k.clone(), v.clone()
    k2[:, :, m:] += 5
    v2[:, :, m:] -= 7
    c = la.la_forward(q, k2, v2, feature_map="none", gamma=g)
    assert torch.equal(a[:, :, :m], c[:, :, :m])


def test_chunked_guard_band():
    """Nothing is written outside out (dv = 128, two value tiles)."""
    q, k, v = _inputs(1, 3, 333, 128, 128, "elu1", seed=69)
    n = 3 * 333 * 128
    buf = torch.full((n + 2048,), 12345.0, device="cuda")
    out = buf[1024:1024 + n].view(1, 3, 333, 128)
    la.la_forward(q, k, v, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 12345.0) and torch.all(buf[1024 + n:] == 12345.0)
