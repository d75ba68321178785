"""The entry points inside CUDA graphs: a serving loop captures a decode step
(or a forward) once and replays it.  Every call only enqueues work on the
caller's stream (kernels, a workspace memset), so a captured call replayed N
times must equal N eager calls bit for bit."""
import pytest
import torch

pytestmark = pytest.mark.gpu

la = pytest.importorskip("kernelised_causal_linear_gb300")
from kernelised_causal_linear_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    yield
    assert la.la_get_device_status() == 0


def test_decode_step_graph_replay():
    B, H, d, steps = 8, 16, 128, 12
    gen = torch.Generator(device="cuda").manual_seed(7)
    S0 = torch.randn(B, H, d, d, device="cuda", generator=gen) * 0.1
    z0 = torch.rand(B, H, d, device="cuda", generator=gen) + 1.0
    toks = [synth.normal((3, B, H, d), seed=200 + t, device="cuda") for t in range(steps)]
    g = torch.tensor([0.99 - 0.01 * h for h in range(H)])

    # eager
    S, z = S0.clone(), z0.clone()
    eager = []
    for t in range(steps):
        q, k, v = toks[t]
        eager.append(la.la_decode_step(S, z, q, k, v, gamma=g).clone())

    # captured once, replayed with the step's tokens copied into static inputs
    Sg, zg = S0.clone(), z0.clone()
    qs, ks, vs = (torch.empty_like(toks[0][i]) for i in range(3))
    out = torch.empty(B, H, d, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm-up outside the graph (library load, attributes)
        la.la_decode_step(Sg.clone(), zg.clone(), qs.zero_(), ks.zero_(), vs.zero_(), out,
                          gamma=g)
    torch.cuda.current_stream().wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        la.la_decode_step(Sg, zg, qs, ks, vs, out, gamma=g)
    for t in range(steps):
        qs.copy_(toks[t][0])
        ks.copy_(toks[t][1])
        vs.copy_(toks[t][2])
        graph.replay()
        assert torch.equal(out, eager[t]), t
    assert torch.equal(Sg, S) and torch.equal(zg, z)


@pytest.mark.parametrize("shape,fm,decay", [((2, 8, 3000, 64, 64), "elu1", False),
                                            ((1, 4, 2000, 128, 128), "none", True)])
def test_forward_graph_replay(shape, fm, decay):
    """The single-pass kernel (whose workspace flags are reset by a memset in
    the captured work) and the chunked path (three launches)."""
    B, H, N, d, dv = shape
    w = synth.Workload("graph", B, H, N, d, dv, torch.bfloat16, q_scale=0.5, k_scale=0.5,
                       feature_map=fm, seed_id=210)
    q, k, v = synth.qkv(w, device="cuda")
    g = torch.tensor([1.0 - 2.0 ** (-5 - h) for h in range(H)]) if decay else None
    ws = torch.empty(la.la_forward_workspace_size(B, H, N, d, dv, True, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    ref = la.la_forward(q, k, v, feature_map=fm, gamma=g, workspace=ws)
    out = torch.empty_like(ref)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        la.la_forward(q, k, v, out, feature_map=fm, gamma=g, workspace=ws)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
