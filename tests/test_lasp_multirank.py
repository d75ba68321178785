"""The sequence-split exchange of lasp.py on CPU: two and three gloo ranks,
each holding a consecutive part of one sequence, all-gather their part
states and continue from the exclusive prefix ("Linear Attention and SSM",
LASP-2).  The local steps are the fp64 oracle's (test infrastructure), so the
concatenated outputs must equal the oracle's forward over the whole sequence
to rounding; this checks the exchange (gather order, part lengths, the decay
of earlier parts) without a GPU.  tests/test_gpu_lasp.py runs the same split
on the library's kernels."""
import os
import socket
import sys
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]
TESTS = Path(__file__).resolve().parent


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_ops():
    import oracle
    from kernelised_causal_linear_gb300.lasp import LaspOps

    orc = oracle.load()

    def local_state(k, v, fm, g):
        S, z = orc.state(k.numpy(), v.numpy(), fm=fm, gamma=g)
        return torch.from_numpy(S), torch.from_numpy(z)

    def prefix(S_all, z_all, lens, upto, g):
        # P_{p+1} = gamma^len_p P_p + U_p, restated in fp64 for the test
        H = S_all.shape[2]
        gam = np.ones(H) if g is None else np.asarray(g, np.float64)
        S = np.zeros(S_all.shape[1:])
        z = np.zeros(z_all.shape[1:])
        for p in range(upto):
            dec = gam ** lens[p]
            S = dec[None, :, None, None] * S + S_all[p].numpy()
            z = dec[None, :, None] * z + z_all[p].numpy()
        return torch.from_numpy(S), torch.from_numpy(z)

    def forward(q, k, v, S0, z0, fm, g):
        return torch.from_numpy(orc.forward(q.numpy(), k.numpy(), v.numpy(), fm=fm, gamma=g,
                                            S0=S0.numpy(), z0=z0.numpy()))

    return LaspOps(local_state, prefix, forward)


def _rank(rank, world, port, parts, fm, gamma, out):
    for p in (str(ROOT), str(TESTS)):
        if p not in sys.path:
            sys.path.insert(0, p)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from kernelised_causal_linear_gb300 import lasp

        rng = np.random.default_rng(123)
        N = sum(parts)
        q, k, v = (torch.from_numpy(rng.normal(size=(2, 3, N, dd)) * 0.5) for dd in (5, 5, 4))
        lo = sum(parts[:rank])
        sl = slice(lo, lo + parts[rank])
        mine = lasp.lasp2_forward(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                                  v[:, :, sl].contiguous(), feature_map=fm, gamma=gamma,
                                  ops=_oracle_ops())
        out[rank] = mine.numpy()
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("parts,fm,gamma", [
    ([40, 25], "elu1", None),
    ([30, 1, 44], "none", [0.9, 0.6, 1.0]),
    ([17, 33, 20], "elu1", [0.95, 0.8, 0.7]),
])
def test_split_sequence_matches_whole(parts, fm, gamma):
    import oracle

    world = len(parts)
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), parts, fm, gamma, out), nprocs=world, join=True)
    rng = np.random.default_rng(123)
    N = sum(parts)
    q, k, v = (rng.normal(size=(2, 3, N, dd)) * 0.5 for dd in (5, 5, 4))
    ref = oracle.load().forward(q, k, v, fm=fm, gamma=None if gamma is None else np.array(gamma))
    got = np.concatenate([out[r] for r in range(world)], axis=2)
    assert np.allclose(got, ref, rtol=1e-11, atol=1e-11), np.max(np.abs(got - ref))
