"""Pins that tie the fp64 oracle to facts fixed outside the oracle itself.

Each pin is a plain function taking an ``oracle.Oracle`` handle and raising
``AssertionError`` on a mismatch.  ``test_oracle_pins.py`` runs all of them on
the real oracle; ``test_oracle_mutants.py`` builds deliberately broken
variants of the oracle source and checks that every variant fails at least
one pin, so a plausible slip (dropped term, wrong sign, read before write,
transposed operand, missing decay) cannot pass unnoticed.

The independent sides used here are: numbers printed on the pages (fixtures
under ``tests/golden/``), closed forms (gamma**n), a library ELU
(``torch.nn.functional.elu``), library matrix products over an explicit
N x N kernel matrix (brute force), and structural invariants of the method.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np

GOLDEN = Path(__file__).resolve().parent / "golden"


def golden(name: str) -> dict:
    return json.loads((GOLDEN / name).read_text())


def lib_phi(x: np.ndarray) -> np.ndarray:
    """elu(x) + 1 from torch's own ELU (alpha = 1), in fp64."""
    import torch

    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    return (torch.nn.functional.elu(t, alpha=1.0) + 1.0).numpy()


def brute_force(q, k, v, causal=True, fm="elu1", gamma=1.0):
    """Explicit N x N kernel matrix with library matmuls: A = (Fq Fk^T) o L,
    O = A V / rowsum(A) (normalised) or A V (fm == 'none')."""
    if fm == "elu1":
        fq, fk = lib_phi(q), lib_phi(k)
    else:
        fq, fk = np.asarray(q, float), np.asarray(k, float)
    a = fq @ fk.T
    n = a.shape[0]
    if causal:
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        mask = np.where(j <= i, np.power(float(gamma), np.maximum(i - j, 0)), 0.0)
        a = a * mask
    num = a @ np.asarray(v, float)
    if fm == "none":
        return num
    return num / a.sum(axis=1, keepdims=True)


def _close(a, b, rtol, atol, what):
    a, b = np.asarray(a, float), np.asarray(b, float)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert np.allclose(a, b, rtol=rtol, atol=atol), f"{what}: max abs err {err:.3e}"


# --------------------------------------------------------------- phi ------
def pin_phi_library(o):
    """phi equals torch's elu(x)+1 on a sweep, and the exact special values."""
    x = np.concatenate([np.linspace(-30, 30, 4001), [0.0, -0.0, 1e-300, -1e-300, -745.0, 700.0]])
    _close(o.phi(x), lib_phi(x), 1e-15, 4e-16, "phi vs library elu+1")
    y = o.phi(np.array([0.0, 3.0, -1.0, 0.5]))
    assert y[0] == 1.0 and y[1] == 4.0 and y[3] == 1.5, y
    assert abs(y[2] - math.exp(-1.0)) <= 1e-16, y
    assert np.all(o.phi(np.linspace(-50, 50, 101)) > 0.0), "phi must be positive"


# ---------------------------------------------------- worked example ------
def pin_worked_example(o):
    g = golden("worked_example_s5_1.json")
    fk = np.array(g["phi_k"], float)[None, None]
    v = np.array(g["v"], float)[None, None]
    S, z = o.state(fk, v, fm="identity_norm")
    _close(S[0, 0], g["S3"], 0, 1e-15, "S_3")
    _close(z[0, 0], g["z3"], 0, 1e-15, "z_3")
    # queries 1 and 2 are not given on the page; any positive features do.
    fq = np.array([[1.0, 1.0], [2.0, 1.0], g["phi_q3"]])[None, None]
    out = o.forward(fq, fk, v, causal=True, fm="identity_norm")
    expect = np.array(g["o3_numerator"], float) / g["o3_denominator"]
    _close(out[0, 0, 2], expect, 0, 1e-15, "o_3")
    _, w = o.dense(fq[0, 0], fk[0, 0], v[0, 0], causal=True, fm="identity_norm",
                   return_weights=True)
    wexp = [a / b for a, b in g["weights_row3"]]
    _close(w[2], wexp, 0, 1e-15, "row-3 weights")
    # the explicit path and the state path agree at every row
    _close(o.dense(fq[0, 0], fk[0, 0], v[0, 0], fm="identity_norm"), out[0, 0], 0, 1e-15,
           "dense vs state")


# ----------------------------------- dense vs recurrent, NumPy check ------
def _page_inputs():
    g = golden("numpy_check_s10.json")
    rng = np.random.default_rng(g["seed"])
    q = rng.normal(size=(g["N"], g["d"]))
    k = rng.normal(size=(g["N"], g["d"]))
    v = rng.normal(size=(g["N"], g["dv"]))
    return g, q, k, v


def pin_dense_equivalence(o):
    g, q, k, v = _page_inputs()
    rec = o.forward(q[None, None], k[None, None], v[None, None])[0, 0]
    bf = brute_force(q, k, v)
    _close(rec, bf, g["rtol"], g["atol"], "recurrence vs explicit matrix")
    # the page's own run lands at a few ulps; ours must be of that order too
    assert np.max(np.abs(rec - bf)) < 100 * g["printed_max_abs_error"]
    _close(o.dense(q, k, v), bf, g["rtol"], g["atol"], "oracle dense vs explicit matrix")
    # other shapes, d != dv so a transposed operand cannot pass, in a batch
    rng = np.random.default_rng(7)
    for (B, H, N, d, dv) in [(2, 3, 33, 8, 5), (1, 2, 1, 3, 6), (1, 1, 64, 16, 16)]:
        Q = rng.normal(size=(B, H, N, d))
        K = rng.normal(size=(B, H, N, d))
        V = rng.normal(size=(B, H, N, dv))
        out = o.forward(Q, K, V, nthreads=3)
        for b in range(B):
            for h in range(H):
                _close(out[b, h], brute_force(Q[b, h], K[b, h], V[b, h]), 1e-12, 1e-12,
                       f"batched slice {(b, h)}")


def pin_no_future_leakage(o):
    g, q, k, v = _page_inputs()
    m = g["leak_split"]
    base = o.forward(q[None, None], k[None, None], v[None, None])[0, 0]
    k2, v2 = k.copy(), v.copy()
    k2[m:] += g["k_shift"]
    v2[m:] += g["v_shift"]
    pert = o.forward(q[None, None], k2[None, None], v2[None, None])[0, 0]
    assert np.array_equal(base[:m], pert[:m]), "past outputs changed when only the future did"
    assert not np.allclose(base[m:], pert[m:]), "future outputs should change"


def pin_noncausal(o):
    g, q, k, v = _page_inputs()
    nc = o.forward(q[None, None], k[None, None], v[None, None], causal=False)[0, 0]
    _close(nc, brute_force(q, k, v, causal=False), g["rtol"], g["atol"], "non-causal vs explicit")
    c = o.forward(q[None, None], k[None, None], v[None, None], causal=True)[0, 0]
    _close(nc[-1], c[-1], 1e-13, 1e-13, "last causal row vs last non-causal row")
    # every non-causal query reads the full-sequence state: place it last
    for i in (0, 5, 11):
        q2 = q.copy()
        q2[-1] = q[i]
        ci = o.forward(q2[None, None], k[None, None], v[None, None], causal=True)[0, 0, -1]
        _close(nc[i], ci, 1e-13, 1e-13, f"non-causal row {i} vs causal read at the end")
    _close(o.dense(q, k, v, causal=False), nc, 1e-12, 1e-12, "oracle dense non-causal")


def pin_state_definition(o):
    rng = np.random.default_rng(11)
    k = rng.normal(size=(2, 2, 29, 6))
    v = rng.normal(size=(2, 2, 29, 4))
    S, z = o.state(k, v)
    for b in range(2):
        for h in range(2):
            fk = lib_phi(k[b, h])
            _close(S[b, h], fk.T @ v[b, h], 1e-13, 1e-13, "S = phi(K)^T V")
            _close(z[b, h], fk.sum(axis=0), 1e-13, 1e-13, "z = column sums of phi(K)")


# ------------------------------------------------------------- decay ------
def pin_decay_impulse(o):
    g = golden("retnet_decay_s7_1.json")
    n, gam, d = g["distance"], g["gamma"], 3
    k = np.zeros((n + 1, d))
    q = np.zeros((n + 1, d))
    v = np.zeros((n + 1, 1))
    k[0, 0] = 1.0
    v[0, 0] = 1.0
    q[:, 0] = 1.0
    out = o.forward(q[None, None], k[None, None], v[None, None], fm="none",
                    gamma=np.array([gam]))[0, 0, :, 0]
    assert abs(out[n] - g["coefficient_rounded"]) <= g["page_rounding"], out[n]
    assert abs(out[n] - gam ** n) <= 1e-13 * gam ** n, (out[n], gam ** n)
    _close(out, gam ** np.arange(n + 1), 1e-13, 0, "impulse response gamma^t")


def pin_decay_dense(o):
    rng = np.random.default_rng(3)
    B, H, N, d, dv = 1, 3, 40, 5, 3
    gam = np.array([0.9, 0.5, 1.0])
    q = rng.normal(size=(B, H, N, d))
    k = rng.normal(size=(B, H, N, d))
    v = rng.normal(size=(B, H, N, dv))
    out = o.forward(q, k, v, fm="none", gamma=gam)
    for h in range(H):
        _close(out[0, h], brute_force(q[0, h], k[0, h], v[0, h], fm="none", gamma=gam[h]),
               1e-12, 1e-12, f"decay head {h}")
    # gamma = 1 is plain unnormalised linear attention
    _close(out[0, 2], o.forward(q, k, v, fm="none")[0, 2], 0, 0, "gamma=1 equals no decay")
    # decay combined with the normaliser: the mask weights num and den alike
    outn = o.forward(q, k, v, fm="elu1", gamma=gam)
    for h in range(H):
        _close(outn[0, h], brute_force(q[0, h], k[0, h], v[0, h], fm="elu1", gamma=gam[h]),
               1e-12, 1e-12, f"normalised decay head {h}")


def pin_additive_vs_normalised(o):
    g = golden("delta_example_s7_3.json")
    kk = np.array([g["unit_key"]] * len(g["values_written"]), float)
    vv = np.array(g["values_written"], float)[:, None]
    qq = kk.copy()
    add = o.forward(qq[None, None], kk[None, None], vv[None, None], fm="none")[0, 0, -1, 0]
    nrm = o.forward(qq[None, None], kk[None, None], vv[None, None], fm="identity_norm")[0, 0, -1, 0]
    assert add == g["additive_read"], add
    assert nrm == g["normalised_read"], nrm


# ------------------------------------------------------------ decode ------
def pin_decode(o):
    rng = np.random.default_rng(5)
    B, H, P, M, d, dv = 2, 2, 13, 6, 4, 6
    q = rng.normal(size=(B, H, P + M, d))
    k = rng.normal(size=(B, H, P + M, d))
    v = rng.normal(size=(B, H, P + M, dv))
    for fm, gam in (("elu1", None), ("none", np.array([0.95, 0.7]))):
        full = o.forward(q, k, v, fm=fm, gamma=gam)
        S, z = o.state(k[:, :, :P], v[:, :, :P], fm=fm, gamma=gam)
        for t in range(P, P + M):
            out, S, z = o.decode_step(S, z, q[:, :, t], k[:, :, t], v[:, :, t], fm=fm, gamma=gam)
            _close(out, full[:, :, t], 1e-12, 1e-12, f"decode step {t} ({fm})")
        # state after decode equals the state of the whole sequence
        S_all, z_all = o.state(k, v, fm=fm, gamma=gam)
        _close(S, S_all, 1e-12, 1e-12, "state after decode")
        _close(z, z_all, 1e-12, 1e-12, "normaliser after decode")
    # resume from a copied state is bitwise identical to running through
    S, z = o.state(k[:, :, :P], v[:, :, :P])
    Sa, za = S.copy(), z.copy()
    for t in range(P, P + M):
        oa, Sa, za = o.decode_step(Sa, za, q[:, :, t], k[:, :, t], v[:, :, t])
    Sb, zb = S.copy(), z.copy()
    for t in range(P, P + 3):
        ob, Sb, zb = o.decode_step(Sb, zb, q[:, :, t], k[:, :, t], v[:, :, t])
    Sc, zc = np.array(Sb), np.array(zb)  # checkpoint copy
    for t in range(P + 3, P + M):
        ob, Sc, zc = o.decode_step(Sc, zc, q[:, :, t], k[:, :, t], v[:, :, t])
    assert np.array_equal(oa, ob) and np.array_equal(Sa, Sc) and np.array_equal(za, zc)
    # a state continued from a given prefix state equals the whole-prefix state
    S1, z1 = o.state(k[:, :, :5], v[:, :, :5])
    S2, z2 = o.state(k[:, :, 5:P], v[:, :, 5:P], S0=S1, z0=z1)
    _close(S2, S, 1e-13, 1e-13, "continued state")
    _close(z2, z, 1e-13, 1e-13, "continued normaliser")


# ------------------------------------------------------ initial state ------
def pin_initial_state(o):
    """A forward continued from the state of a prefix equals the same rows of
    the forward over the whole sequence, and the explicit matrix over it
    (the state summarises the prefix, "Efficient Attention Variants" s.5)."""
    rng = np.random.default_rng(21)
    B, H, P, M, d, dv = 2, 2, 11, 9, 5, 3
    q = rng.normal(size=(B, H, P + M, d))
    k = rng.normal(size=(B, H, P + M, d))
    v = rng.normal(size=(B, H, P + M, dv))
    alpha = rng.uniform(0.6, 1.0, size=(B, H, P + M, d))
    for fm, gam, al in (("elu1", None, None), ("none", np.array([0.9, 0.6]), None),
                        ("elu1", np.array([0.8, 1.0]), None), ("elu1", None, alpha)):
        full = o.forward(q, k, v, fm=fm, gamma=gam, alpha=al)
        S0, z0 = o.state(k[:, :, :P], v[:, :, :P], fm=fm, gamma=gam,
                         alpha=None if al is None else al[:, :, :P])
        tail = o.forward(q[:, :, P:], k[:, :, P:], v[:, :, P:], fm=fm, gamma=gam,
                         alpha=None if al is None else al[:, :, P:], S0=S0, z0=z0)
        _close(tail, full[:, :, P:], 1e-12, 1e-12, f"continued forward ({fm})")
        if al is None:
            for b in range(B):
                for h in range(H):
                    bf = brute_force(q[b, h], k[b, h], v[b, h], fm=fm,
                                     gamma=1.0 if gam is None else gam[h])
                    _close(tail[b, h], bf[P:], 1e-11, 1e-11, f"continued vs explicit {(b, h)}")
    try:
        o.forward(q, k, v, causal=False, S0=np.zeros((B, H, d, dv)), z0=np.zeros((B, H, d)))
    except Exception:
        pass
    else:
        raise AssertionError("an initial state with the non-causal form must be rejected")


# ------------------------------------------------ per-channel decay -------
def gla_brute_force(q, k, v, alpha, fm="none"):
    """o_i = sum_{j<=i} sum_r fq_ir fk_jr (prod_{s=j+1..i} alpha_sr) v_j,
    written out with explicit products ("Efficient Attention Variants" s.7.2:
    alpha_t scales row r of the state, broadcast along the values)."""
    fq, fk = (lib_phi(q), lib_phi(k)) if fm == "elu1" else (q, k)
    n, d = q.shape
    out = np.zeros((n, v.shape[1]))
    den = np.zeros(n)
    for i in range(n):
        for j in range(i + 1):
            w = np.ones(d)
            for s_ in range(j + 1, i + 1):
                w = w * alpha[s_]
            a = float(np.sum(fq[i] * fk[j] * w))
            out[i] += a * v[j]
            den[i] += a
    return out if fm == "none" else out / den[:, None]


def pin_gla(o):
    rng = np.random.default_rng(23)
    B, H, N, d, dv = 1, 2, 14, 4, 6
    q = rng.normal(size=(B, H, N, d))
    k = rng.normal(size=(B, H, N, d))
    v = rng.normal(size=(B, H, N, dv))
    alpha = rng.uniform(0.3, 1.0, size=(B, H, N, d))
    for fm in ("none", "elu1"):
        out = o.forward(q, k, v, fm=fm, alpha=alpha)
        for h in range(H):
            _close(out[0, h], gla_brute_force(q[0, h], k[0, h], v[0, h], alpha[0, h], fm),
                   1e-12, 1e-12, f"per-channel decay head {h} ({fm})")
    # a constant alpha is the scalar decay of the same value; alpha = 1 is none
    gam = np.array([0.85, 0.55])
    const = np.broadcast_to(gam[None, :, None, None], (B, H, N, d)).copy()
    _close(o.forward(q, k, v, fm="none", alpha=const), o.forward(q, k, v, fm="none", gamma=gam),
           0, 0, "constant alpha equals gamma")
    _close(o.forward(q, k, v, alpha=np.ones((B, H, N, d))), o.forward(q, k, v), 0, 0,
           "alpha = 1 equals no decay")
    # the state: S = sum_j diag(prod_{s>j} alpha_s) phi(k_j) v_j^T
    S, z = o.state(k, v, fm="elu1", alpha=alpha)
    fk = lib_phi(k[0, 1])
    w = np.ones((N, d))
    for j in range(N):
        for s_ in range(j + 1, N):
            w[j] *= alpha[0, 1, s_]
    _close(S[0, 1], (fk * w).T @ v[0, 1], 1e-12, 1e-12, "per-channel decayed state")
    _close(z[0, 1], (fk * w).sum(axis=0), 1e-12, 1e-12, "per-channel decayed normaliser")
    # decode continues it token by token
    S0, z0 = o.state(k[:, :, :8], v[:, :, :8], fm="none", alpha=alpha[:, :, :8])
    full = o.forward(q, k, v, fm="none", alpha=alpha)
    for t in range(8, N):
        ot, S0, z0 = o.decode_step(S0, z0, q[:, :, t], k[:, :, t], v[:, :, t], fm="none",
                                   alpha=alpha[:, :, t])
        _close(ot, full[:, :, t], 1e-12, 1e-12, f"per-channel decode step {t}")


# ------------------------------------------------- random features --------
def pin_favor(o):
    """Positive random features estimate the exponential kernel without bias
    ("Efficient Attention Variants" s.6): the mean of phi(q).phi(k) over many
    Gaussian rows approaches exp(q.k / sqrt(d)), within a few standard errors
    of the sample itself; every feature is positive."""
    rng = np.random.default_rng(29)
    d, r = 4, 200_000
    q = np.array([0.7, -0.3, 0.5, 0.2])
    k = np.array([0.4, 0.6, -0.2, 0.8])
    w = rng.normal(size=(r, d))
    fq, fk = o.favor(q[None], w)[0], o.favor(k[None], w)[0]
    assert np.all(fq > 0) and np.all(fk > 0), "features must be positive"
    prod = fq * fk * r          # one unbiased estimate per Gaussian row
    est, se = prod.mean(), prod.std() / math.sqrt(r)
    exact = math.exp(float(q @ k) / math.sqrt(d))
    assert abs(est - exact) < 5 * se, (est, exact, se)
    assert abs(fq @ fk - est) <= 1e-12 * est
    # for given features the state form equals the explicit kernel matrix
    Q = rng.normal(size=(9, d)) * 0.5
    K = rng.normal(size=(9, d)) * 0.5
    V = rng.normal(size=(9, 3))
    w8 = rng.normal(size=(8, d))
    FQ, FK = o.favor(Q, w8), o.favor(K, w8)
    rec = o.forward(FQ[None, None], FK[None, None], V[None, None], fm="identity_norm")[0, 0]
    _close(rec, brute_force(FQ, FK, V, fm="identity_norm"), 1e-12, 1e-12,
           "random-feature state form vs explicit matrix")


ALL_PINS = [
    pin_phi_library,
    pin_worked_example,
    pin_dense_equivalence,
    pin_no_future_leakage,
    pin_noncausal,
    pin_state_definition,
    pin_decay_impulse,
    pin_decay_dense,
    pin_additive_vs_normalised,
    pin_decode,
    pin_initial_state,
    pin_gla,
    pin_favor,
]
