"""Seeded synthetic inputs and the named workloads, shared by tests and bench.

This module holds none of the method's arithmetic: it only draws i.i.d.
normal numbers with a fixed seed, scales them and rounds them once to the
storage dtype.  Both the CUDA path and the fp64 oracle then read the very
same bytes (the oracle after an exact upcast), so parity never depends on two
random generators agreeing.

The workloads mirror the shapes the pages discuss (the capacity example of
"Efficient Attention Variants", section 1, is N=32768, d=dv=64 per head) and
the per-head RetNet decay rates gamma_h = 1 - 2^(-5-h).  None of them stands
in for a public dataset: the pages measure on none.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED_BASE = 0x4C410000


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dv: int
    dtype: torch.dtype
    q_scale: float = 1.0
    k_scale: float = 1.0
    v_scale: float = 1.0
    causal: bool = True
    feature_map: str = "elu1"
    decay: bool = False
    seed_id: int = 0
    # decode workloads: prefix length that builds the state, then steps
    prefix: int = 0
    steps: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def BH(self) -> int:
        return self.B * self.H

    def gamma(self):
        """Per-head decay gamma_h = 1 - 2^(-5-h), exact in fp32."""
        if not self.decay:
            return None
        return torch.tensor([1.0 - 2.0 ** (-5 - h) for h in range(self.H)], dtype=torch.float32)

    def seed(self, stream: int) -> int:
        return (SEED_BASE + self.seed_id) * 64 + stream


WORKLOADS = {
    # small fp32 case the oracle finishes instantly
    "causal_n256_d32_fp32": Workload("causal_n256_d32_fp32", 1, 1, 256, 32, 32, torch.float32,
                                     seed_id=1),
    # mid-size bf16, q and k scaled by 1/sqrt(d); run causal and non-causal
    "causal_n2048_d64_bf16": Workload("causal_n2048_d64_bf16", 4, 8, 2048, 64, 64, torch.bfloat16,
                                      q_scale=1 / 8, k_scale=1 / 8, seed_id=2),
    # the same shape, non-causal (every query reads the whole sequence's state)
    "noncausal_n2048_d64_bf16": Workload("noncausal_n2048_d64_bf16", 4, 8, 2048, 64, 64,
                                         torch.bfloat16, q_scale=1 / 8, k_scale=1 / 8,
                                         causal=False, seed_id=2),
    # long-context causal forward: the headline throughput workload
    "causal_n32768_d64_bf16": Workload("causal_n32768_d64_bf16", 2, 16, 32768, 64, 64,
                                       torch.bfloat16, seed_id=3),
    # RetNet scalar decay, no feature map and no normaliser, all inputs / sqrt(d)
    "retnet_n8192_d128_bf16": Workload("retnet_n8192_d128_bf16", 4, 8, 8192, 128, 128,
                                       torch.bfloat16, q_scale=1 / math.sqrt(128),
                                       k_scale=1 / math.sqrt(128), v_scale=1 / math.sqrt(128),
                                       feature_map="none", decay=True, seed_id=4),
    # per-key-channel decay (GLA), gates uniform in [0.95, 1), no feature map
    "gla_n8192_d128_bf16": Workload("gla_n8192_d128_bf16", 4, 8, 8192, 128, 128, torch.bfloat16,
                                    q_scale=1 / math.sqrt(128), k_scale=1 / math.sqrt(128),
                                    v_scale=1 / math.sqrt(128), feature_map="none", seed_id=7,
                                    extra={"gla_gates": (0.95, 1.0)}),
    # positive random features (Performer): d = 64 inputs, r = 128 features
    "favor_n4096_d64_r128_bf16": Workload("favor_n4096_d64_r128_bf16", 2, 8, 4096, 64, 64,
                                          torch.bfloat16, feature_map="identity_norm",
                                          seed_id=6, extra={"favor_r": 128}),
    # batched decode: 256 sequences x 32 heads, state from a 4096-token prefix
    "decode_b256_h32_d128_bf16": Workload("decode_b256_h32_d128_bf16", 256, 32, 1, 128, 128,
                                          torch.bfloat16, seed_id=5, prefix=4096, steps=1000),
}


def normal(shape, *, seed: int, scale: float = 1.0, dtype=torch.bfloat16, device="cpu"):
    """i.i.d. N(0,1) * scale, drawn in fp32 from a seeded generator and
    rounded once (round-to-nearest-even) to `dtype`."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def gates(shape, *, seed: int, lo: float = 0.9, hi: float = 1.0, device="cpu"):
    """Per-key-channel decay gates, i.i.d. uniform in [lo, hi) (lo > 0), fp32:
    the data-dependent alpha_t of a gated recurrence, here drawn instead of
    computed from the tokens."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    u = torch.rand(tuple(shape), generator=gen, dtype=torch.float64)
    return (lo + (hi - lo) * u).float().to(device)


def gaussian_rows(r: int, d: int, *, seed: int, orthogonal: bool = True, device="cpu"):
    """r random rows of length d for positive random features, fp32.

    orthogonal=True draws them in blocks of d mutually orthogonal rows (the QR
    factor of a Gaussian block), each row rescaled to the norm of an
    independent Gaussian vector, so every row is still marginally N(0, I);
    otherwise i.i.d. N(0, 1).  These are the random numbers the feature map
    consumes; the map itself is la_favor_features."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    if not orthogonal:
        return torch.randn(r, d, generator=gen, dtype=torch.float64).float().to(device)
    blocks = []
    for _ in range((r + d - 1) // d):
        g = torch.randn(d, d, generator=gen, dtype=torch.float64)
        qm, _ = torch.linalg.qr(g)
        norms = torch.randn(d, d, generator=gen, dtype=torch.float64).norm(dim=1)
        blocks.append(qm.T * norms[:, None])
    return torch.cat(blocks)[:r].float().contiguous().to(device)


def qkv(w: Workload, device="cpu", N: int | None = None, B: int | None = None,
        H: int | None = None):
    """The (q, k, v) tensors of a forward workload, [B,H,N,d] / [B,H,N,dv]."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    q = normal((B, H, N, w.d), seed=w.seed(0), scale=w.q_scale, dtype=w.dtype, device=device)
    k = normal((B, H, N, w.d), seed=w.seed(1), scale=w.k_scale, dtype=w.dtype, device=device)
    v = normal((B, H, N, w.dv), seed=w.seed(2), scale=w.v_scale, dtype=w.dtype, device=device)
    return q, k, v


def decode_prefix(w: Workload, head_lo: int, head_hi: int, device="cpu"):
    """Prefix (k, v) for the flattened sequences [head_lo, head_hi) of a
    decode workload, [n, 1, prefix, d] / [n, 1, prefix, dv].  Each flattened
    sequence has its own seed, so any subset can be regenerated alone."""
    ks, vs = [], []
    for s in range(head_lo, head_hi):
        ks.append(normal((w.prefix, w.d), seed=w.seed(8) * 1_000_003 + 2 * s, dtype=w.dtype,
                         device=device))
        vs.append(normal((w.prefix, w.dv), seed=w.seed(8) * 1_000_003 + 2 * s + 1,
                         dtype=w.dtype, device=device))
    return torch.stack(ks)[:, None], torch.stack(vs)[:, None]


def decode_tokens(w: Workload, steps: int, device="cpu"):
    """Per-step tokens of a decode workload: q, k [steps,B,H,d], v [steps,B,H,dv]."""
    shp = (steps, w.B, w.H)
    q = normal(shp + (w.d,), seed=w.seed(16), dtype=w.dtype, device=device)
    k = normal(shp + (w.d,), seed=w.seed(17), dtype=w.dtype, device=device)
    v = normal(shp + (w.dv,), seed=w.seed(18), dtype=w.dtype, device=device)
    return q, k, v
