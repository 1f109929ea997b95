"""Pins of the oracle's mixer variants: FLARE (Section 3.1 eq. 2-4), FLARE++
with separate synthesis values (Appendix A.1 eq. 11) and simplified FLARE++
(Appendix A.8 eq. 20), all from the FLARE++ paper.

As for the main mixer, every expected value comes from outside the oracle:
scalar loops with the math module, scipy's softmax, closed forms, or the main
mixer's oracle where the paper states that a variant reduces to it (and that
oracle is pinned on its own).
"""
import math

import numpy as np
import scipy.special

import oracle
from rank_latent_routing_gb300 import workloads

RNG = np.random.default_rng(4321)


def _attend(qrow, keys, vals):
    """One SDPA output row (eq. 1) as scalar loops: softmax over the keys."""
    D = len(qrow)
    s = 1.0 / math.sqrt(D)
    sc = [s * sum(qrow[d] * key[d] for d in range(D)) for key in keys]
    mx = max(sc)
    w = [math.exp(x - mx) for x in sc]
    tot = sum(w)
    return [sum(w[j] * vals[j][d] for j in range(len(keys))) / tot for d in range(len(vals[0]))]


def _nrm(row, eps=1e-6):
    ms = sum(x * x for x in row) / len(row)
    return [x / math.sqrt(ms + eps) for x in row]


def _route_brute(q, K, V):
    z = [_attend(qm, K, V) for qm in q]
    y = [_attend(kn, q, z) for kn in K]
    return z, y


def _tiny(N=7, M=3, D=4, **kw):
    wl = workloads.config("tiny", N=N, M=M, D=D, **kw)
    return wl, workloads.variant_inputs(wl)


# ----------------------------------------------------------------------- FLARE
def test_flare_brute_force_tiny():
    """Eq. 3 as scalar loops: Z = SDPA(Q_h, K, V), Y = SDPA(K, Q_h, Z)."""
    wl, ex = _tiny()
    for h in range(2):
        q, K, V = ex["Qlat"][h], wl.K[0, h], wl.V[0, h]
        z, y = _route_brute(q.tolist(), K.tolist(), V.tolist())
        r = oracle.flare_forward_head(q, K, V)
        np.testing.assert_allclose(r["Z"], z, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Y"], y, rtol=1e-12, atol=1e-14)


def test_flare_effective_operator():
    """Y = W_dec W_enc V with W_enc = softmax over N of S and W_dec = softmax
    over M of S^T, S = Q K^T / sqrt(D) (eq. 4), built with scipy's softmax."""
    q = RNG.normal(size=(5, 8))
    k = RNG.normal(size=(13, 8)) * 1.5
    v = RNG.normal(size=(13, 8))
    s = q @ k.T / math.sqrt(8)
    w = scipy.special.softmax(s.T, axis=1) @ scipy.special.softmax(s, axis=1)
    np.testing.assert_allclose(oracle.flare_forward_head(q, k, v)["Y"], w @ v, rtol=1e-12,
                               atol=1e-14)
    # rows of the effective operator are probability vectors
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-13)


def test_flare_lse_matches_scipy():
    q = RNG.normal(size=(4, 16))
    k = RNG.normal(size=(40, 16)) * 2
    v = RNG.normal(size=(40, 16))
    r = oracle.flare_forward_head(q, k, v)
    np.testing.assert_allclose(r["L"], scipy.special.logsumexp(q @ k.T / 4.0, axis=1), rtol=1e-13)


def test_flare_is_flarepp_with_zero_gate():
    """With g = 0 the FLARE++ queries are N0(Q^f) (eq. 7): FLARE with those queries."""
    wl = workloads.config("tiny", N=90, M=8)
    gate0 = np.zeros_like(wl.gate)
    a = oracle.forward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, gate0)
    qn = np.stack([oracle.n0(wl.Qf[h]) for h in range(wl.shape.H)])
    b = oracle.flare_forward(qn, wl.K, wl.V)
    for key in ("Z", "L", "Y"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-13, atol=1e-15)


def test_flare_queries_are_per_head():
    """Each head routes with its own query set (eq. 2): swapping the heads'
    query sets swaps the heads' outputs."""
    wl, ex = _tiny(N=30, M=4, D=8)
    q = ex["Qlat"]
    a = oracle.flare_forward(q, wl.K, wl.V)
    b = oracle.flare_forward(q[::-1].copy(), wl.K[:, ::-1].copy(), wl.V[:, ::-1].copy())
    np.testing.assert_allclose(b["Y"][:, ::-1], a["Y"], rtol=1e-14, atol=1e-15)


# ------------------------------------------------- separate synthesis values
def test_unshared_brute_force_tiny():
    """Eq. 11 with N0 on the synthesis keys and the separate values as given."""
    wl, ex = _tiny()
    for h in range(2):
        ks = [_nrm(r) for r in wl.Ks_raw[0, h].tolist()]
        vs = ex["Vs"][0, h].tolist()
        qd = [_attend(qm, ks, vs) for qm in wl.Qseed[h].tolist()]
        qf = [_nrm(r) for r in wl.Qf[h].tolist()]
        g = float(wl.gate[h])
        q = [[qf[m][d] + g * qd[m][d] for d in range(4)] for m in range(3)]
        z, y = _route_brute(q, wl.K[0, h].tolist(), wl.V[0, h].tolist())
        r = oracle.forward_unshared(wl.K[:, h:h + 1], wl.V[:, h:h + 1], wl.Ks_raw[:, h:h + 1],
                                    ex["Vs"][:, h:h + 1], wl.Qseed[h:h + 1], wl.Qf[h:h + 1],
                                    wl.gate[h:h + 1])
        np.testing.assert_allclose(r["Qd"][0, 0], qd, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Q"][0, 0], q, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Z"][0, 0], z, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Y"][0, 0], y, rtol=1e-12, atol=1e-14)


def test_unshared_with_shared_values_is_default():
    """V~ = N0(K~) is the default configuration (Appendix A.6 eq. 19)."""
    wl = workloads.config("tiny", N=120, M=8)
    vs = np.stack([np.stack([oracle.n0(wl.Ks_raw[b, h]) for h in range(wl.shape.H)])
                   for b in range(wl.shape.B)])
    a = oracle.forward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate)
    b = oracle.forward_unshared(wl.K, wl.V, wl.Ks_raw, vs, wl.Qseed, wl.Qf, wl.gate)
    for key in a:
        np.testing.assert_allclose(b[key], a[key], rtol=1e-13, atol=1e-15)


def test_unshared_synthesis_linear_in_values():
    """The synthesis weights do not depend on V~, so Q^d is linear in V~, and
    constant value rows give that constant (eq. 12: Q^d = A~ V~, A~ row-stochastic)."""
    qs = RNG.normal(size=(6, 16))
    ks = RNG.normal(size=(50, 16)) * 3
    v1 = RNG.normal(size=(50, 16))
    v2 = RNG.normal(size=(50, 16))
    f = oracle.synthesis_unshared
    np.testing.assert_allclose(f(qs, ks, 2 * v1 - 3 * v2), 2 * f(qs, ks, v1) - 3 * f(qs, ks, v2),
                               rtol=1e-12, atol=1e-12)
    c = RNG.normal(size=16)
    np.testing.assert_allclose(f(qs, ks, np.tile(c, (50, 1))), np.tile(c, (6, 1)), rtol=1e-13)
    # the keys are normalised: scaling the raw synthesis keys changes nothing beyond eps
    np.testing.assert_allclose(f(qs, 5 * ks, v1), f(qs, ks, v1), rtol=1e-6, atol=1e-7)


# ------------------------------------------------------------ simplified form
def test_simplified_brute_force_tiny():
    """Eq. 20: Q = SDPA(Q~, K~, V~) with no N0, no reference and no gate."""
    wl, ex = _tiny()
    for h in range(2):
        ks, vs = wl.Ks_raw[0, h].tolist(), ex["Vs"][0, h].tolist()
        q = [_attend(qm, ks, vs) for qm in wl.Qseed[h].tolist()]
        z, y = _route_brute(q, wl.K[0, h].tolist(), wl.V[0, h].tolist())
        r = oracle.forward_simplified(wl.K[:, h:h + 1], wl.V[:, h:h + 1], wl.Ks_raw[:, h:h + 1],
                                      ex["Vs"][:, h:h + 1], wl.Qseed[h:h + 1])
        np.testing.assert_allclose(r["Q"][0, 0], q, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Z"][0, 0], z, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Y"][0, 0], y, rtol=1e-12, atol=1e-14)


def test_simplified_single_token():
    """N = 1: every route's query is that token's synthesis value, and the
    encode and decode softmaxes have one key each, so Y = Z = V."""
    K = RNG.normal(size=(1, 1, 1, 8))
    V = RNG.normal(size=(1, 1, 1, 8))
    Ks = RNG.normal(size=(1, 1, 1, 8))
    Vs = RNG.normal(size=(1, 1, 1, 8))
    Qs = RNG.normal(size=(1, 5, 8))
    r = oracle.forward_simplified(K, V, Ks, Vs, Qs)
    np.testing.assert_allclose(r["Q"][0, 0], np.tile(Vs[0, 0, 0], (5, 1)), rtol=1e-15)
    np.testing.assert_allclose(r["Z"][0, 0], np.tile(V[0, 0, 0], (5, 1)), rtol=1e-15)
    np.testing.assert_allclose(r["Y"][0, 0, 0], V[0, 0, 0], rtol=1e-14)


def test_simplified_scores_are_bilinear():
    """No hidden normalisation of either operand of the synthesis scores:
    SDPA(Q~, c K~, V~) = SDPA(c Q~, K~, V~), and it differs from c = 1."""
    qs = RNG.normal(size=(6, 16))
    ks = RNG.normal(size=(40, 16))
    vs = RNG.normal(size=(40, 16))
    f = oracle.synthesis_simplified
    np.testing.assert_allclose(f(qs, 3 * ks, vs), f(3 * qs, ks, vs), rtol=1e-12, atol=1e-14)
    assert np.max(np.abs(f(qs, 3 * ks, vs) - f(qs, ks, vs))) > 1e-2


def test_variant_inputs_statistics():
    """Separate values are drawn like the other tokens; FLARE queries are N(0,1)."""
    wl = workloads.config("pde2d", B=1, H=2, N=4096)
    ex = workloads.variant_inputs(wl)
    assert ex["Vs"].shape == wl.V.shape and ex["Qlat"].shape == wl.Qseed.shape
    assert abs(float(ex["Vs"].std()) - 1.0) < 0.03 and abs(float(ex["Vs"].mean())) < 0.03
    assert abs(float(ex["Qlat"].std()) - 1.0) < 0.1
    # a stream of its own: not a copy of V or of the synthesis keys
    assert not np.allclose(ex["Vs"], wl.V) and not np.allclose(ex["Vs"], wl.Ks_raw)
