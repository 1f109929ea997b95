"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Every check here comes from the FLARE++ paper's mathematics, a closed form, a
library routine computing the same textbook quantity, or brute force on tiny
inputs written as plain scalar loops. Each is chosen so that a plausible slip
in the oracle (a dropped term, a wrong sign, a transposed operand, the softmax
over the wrong axis, a wrong scale or eps) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from rank_latent_routing_gb300 import workloads

RNG = np.random.default_rng(1234)


def _rms(x):
    return np.sqrt(np.mean(np.asarray(x) ** 2, axis=-1))


# --------------------------------------------------------------------------- N0
def test_n0_closed_form():
    """N0 divides by sqrt(mean square + eps) (paper Section 3.2, eq. 5)."""
    x = np.array([[3.0, 4.0], [1.0, 1.0], [-2.0, 0.0]])
    expect = np.array([[3.0, 4.0] / np.sqrt(12.5 + 1e-6),
                       [1.0, 1.0] / np.sqrt(1.0 + 1e-6),
                       [-2.0, 0.0] / np.sqrt(2.0 + 1e-6)])
    np.testing.assert_allclose(oracle.n0(x), expect, rtol=0, atol=1e-15)


def test_n0_unit_rms_and_scale_invariance():
    x = RNG.normal(size=(50, 32)) * RNG.uniform(0.1, 10, size=(50, 1))
    y = oracle.n0(x)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(_rms(y), np.sqrt(ms / (ms + oracle.EPS)), rtol=1e-13)
    # scale invariance holds up to the eps term: relative change <= eps / (2 ms)
    np.testing.assert_allclose(oracle.n0(7.0 * x), y, rtol=oracle.EPS / (2 * ms.min()) + 1e-13)
    # a zero row stays zero (no NaN)
    assert np.all(oracle.n0(np.zeros((1, 16))) == 0)


# ------------------------------------------------------------------- SDPA, LSE
def test_sdpa_matches_torch_library():
    """SDPA of eq. 1 against torch's scaled_dot_product_attention in float64."""
    import torch
    q = RNG.normal(size=(7, 16))
    k = RNG.normal(size=(11, 16)) * 2.0
    v = RNG.normal(size=(11, 16))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None])[0].numpy()
    np.testing.assert_allclose(oracle.sdpa(q, k, v), ref, rtol=1e-12, atol=1e-13)
    # row blocking changes nothing beyond the matmul library's own rounding order
    np.testing.assert_allclose(oracle.sdpa(q, k, v, rows=3), oracle.sdpa(q, k, v), rtol=1e-14,
                               atol=1e-15)


def test_lse_matches_scipy_library():
    from scipy.special import logsumexp
    s = RNG.normal(size=(5, 40)) * 30.0
    np.testing.assert_allclose(oracle.logsumexp_rows(s), logsumexp(s, axis=-1), rtol=1e-14)
    q = RNG.normal(size=(4, 8))
    k = RNG.normal(size=(9, 8))
    _, lse = oracle.sdpa(q, k, RNG.normal(size=(9, 8)), with_lse=True)
    np.testing.assert_allclose(lse, logsumexp(q @ k.T / math.sqrt(8), axis=-1), rtol=1e-14)


def test_two_token_softmax_closed_form():
    """With two keys the softmax weight of key 1 is sigmoid of the score gap."""
    q = np.array([[0.5, -1.0, 2.0, 0.25]])
    k = np.array([[1.0, 0.0, 1.0, 0.0], [0.0, 2.0, 0.0, -1.0]])
    v = np.array([[1.0, 2.0, 3.0, 4.0], [-1.0, 0.0, 5.0, 2.0]])
    gap = (q @ (k[0] - k[1])) / 2.0  # scale 1/sqrt(4)
    w1 = 1.0 / (1.0 + math.exp(-gap[0]))
    np.testing.assert_allclose(oracle.sdpa(q, k, v), (w1 * v[0] + (1 - w1) * v[1])[None], rtol=1e-14)


# ------------------------------------------------------------------- synthesis
def test_synthesis_rms_bound():
    """RMS(Q^d_m) <= 1 (Appendix A.4 eq. 17): rows of Q^d are convex
    combinations of unit-RMS rows."""
    for scale in (1.0, 8.0, 50.0):
        qseed = RNG.normal(size=(16, 32)) * scale / math.sqrt(32)
        ks = RNG.normal(size=(300, 32)) * RNG.uniform(0.1, 5, size=(300, 1))
        qd = oracle.synthesis(qseed, ks)
        assert np.all(_rms(qd) <= 1.0 + 1e-12)


def test_synthesis_equal_rows_attain_bound():
    """All synthesis keys equal to u: every Q^d row is N0(u) (bound attained)."""
    u = RNG.normal(size=(1, 16))
    ks = np.repeat(u, 37, axis=0)
    qd = oracle.synthesis(RNG.normal(size=(5, 16)), ks)
    np.testing.assert_allclose(qd, np.repeat(oracle.n0(u), 5, axis=0), rtol=1e-13)
    u_rms = np.sqrt(np.mean(u * u))
    np.testing.assert_allclose(_rms(qd), u_rms / np.sqrt(u_rms ** 2 + oracle.EPS), rtol=1e-13)


def test_synthesis_zero_seed_is_mean():
    """Qseed = 0 gives uniform attention, so Q^d is the mean of the N0 rows."""
    ks = RNG.normal(size=(29, 8)) * 3.0
    kt = ks / np.sqrt(np.mean(ks * ks, axis=1, keepdims=True) + 1e-6)
    qd = oracle.synthesis(np.zeros((4, 8)), ks)
    np.testing.assert_allclose(qd, np.repeat(kt.mean(axis=0, keepdims=True), 4, axis=0), rtol=1e-13)


def test_synthesis_uses_shared_normalised_values():
    """The values of the synthesis call are N0(Ks_raw), not Ks_raw (eq. 5, 19):
    scaling one raw key row must not change Q^d except through eps."""
    ks = RNG.normal(size=(40, 16))
    qseed = RNG.normal(size=(6, 16)) * 2
    ks2 = ks.copy()
    ks2[3] *= 100.0
    np.testing.assert_allclose(oracle.synthesis(qseed, ks2), oracle.synthesis(qseed, ks), rtol=5e-6,
                               atol=1e-7)


# -------------------------------------------------------------------- the gate
def test_gate_bounds():
    """1 - g <= RMS(Q_m) <= 1 + g (Appendix A.4), up to the eps slack of N0."""
    for g in (0.0, 0.25, 0.5622, 0.99):
        qd = oracle.synthesis(RNG.normal(size=(32, 16)) * 3, RNG.normal(size=(200, 16)))
        q = oracle.routing_queries(RNG.normal(size=(32, 16)) / 4, qd, g)
        r = _rms(q)
        assert np.all(r <= 1 + g + 1e-12)
        assert np.all(r >= 1 - g - 1e-4)


def test_gate_zero_is_fixed_query_routing():
    """g = 0: Q = N0(Q^f), and Y no longer depends on Ks_raw or Qseed (eq. 7)."""
    wl = workloads.config("tiny", N=100, M=8)
    K, V = wl.K[0, 0], wl.V[0, 0]
    a = oracle.forward_head(K, V, wl.Ks_raw[0, 0], wl.Qseed[0], wl.Qf[0], 0.0)
    b = oracle.forward_head(K, V, wl.Ks_raw[0, 1] * 3, wl.Qseed[1] * 5, wl.Qf[0], 0.0)
    np.testing.assert_array_equal(a["Q"], oracle.n0(wl.Qf[0]))
    np.testing.assert_array_equal(a["Y"], b["Y"])
    # and it is FLARE with the normalised queries (eq. 3)
    z = oracle.sdpa(oracle.n0(wl.Qf[0]), K, V)
    np.testing.assert_allclose(a["Y"], oracle.sdpa(K, oracle.n0(wl.Qf[0]), z), rtol=1e-13)


# ---------------------------------------------------------------- encode/decode
def test_encode_constant_values_and_zero_keys():
    q = RNG.normal(size=(6, 16))
    k = RNG.normal(size=(50, 16))
    c = RNG.normal(size=(1, 16))
    z, _ = oracle.encode(q, k, np.repeat(c, 50, axis=0))
    np.testing.assert_allclose(z, np.repeat(c, 6, axis=0), rtol=1e-13)
    v = RNG.normal(size=(50, 16))
    z, lse = oracle.encode(q, np.zeros((50, 16)), v)
    np.testing.assert_allclose(z, np.repeat(v.mean(axis=0, keepdims=True), 6, axis=0), rtol=1e-12)
    np.testing.assert_allclose(lse, np.full(6, math.log(50)), rtol=1e-14)


def test_decode_single_route_and_single_token():
    """M = 1: every token gets Z_1. N = 1: the whole mixer returns V."""
    k = RNG.normal(size=(20, 8))
    z = RNG.normal(size=(1, 8))
    y = oracle.decode(k, RNG.normal(size=(1, 8)), z)
    np.testing.assert_allclose(y, np.repeat(z, 20, axis=0), rtol=1e-14)
    v = RNG.normal(size=(1, 8))
    r = oracle.forward_head(RNG.normal(size=(1, 8)), v, RNG.normal(size=(1, 8)),
                            RNG.normal(size=(5, 8)), RNG.normal(size=(5, 8)), 0.4)
    np.testing.assert_allclose(r["Y"], v, rtol=1e-13)
    np.testing.assert_allclose(r["Z"], np.repeat(v, 5, axis=0), rtol=1e-13)


def test_decode_softmax_is_over_routes():
    """Decode weights sum to one over the M routes for each token (Figure 1)."""
    q = RNG.normal(size=(6, 16))
    k = RNG.normal(size=(30, 16))
    # one-hot Z rows expose the decode weights directly
    w = oracle.decode(k, q, np.eye(6, 16))[:, :6]
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-13)
    s = k @ q.T / 4.0
    e = np.exp(s - s.max(axis=1, keepdims=True))
    np.testing.assert_allclose(w, e / e.sum(axis=1, keepdims=True), rtol=1e-12)


# -------------------------------------------------------------- whole operator
def test_rank_and_materialised_operator():
    """Y = W_dec W_enc V with rank(W_dec W_enc) <= M (eq. 4, eq. 9)."""
    N, M, D = 64, 16, 16
    wl = workloads.config("tiny", N=N, M=M, D=D)
    r = oracle.forward_head(wl.K[0, 0], wl.V[0, 0], wl.Ks_raw[0, 0], wl.Qseed[0], wl.Qf[0],
                            wl.gate[0])
    w = oracle.w_eff(r["Q"], wl.K[0, 0])
    np.testing.assert_allclose(w @ wl.V[0, 0], r["Y"], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-13)
    sv = np.linalg.svd(w, compute_uv=False)
    assert sv[M] / sv[0] < 1e-10
    assert sv[M - 1] / sv[0] > 1e-8


def test_permutation_equivariance():
    """Token order carries no meaning: permuting K, V, Ks_raw permutes Y."""
    wl = workloads.config("tiny", N=77, M=8)
    perm = np.random.default_rng(5).permutation(77)
    a = oracle.forward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate)
    b = oracle.forward(wl.K[:, :, perm], wl.V[:, :, perm], wl.Ks_raw[:, :, perm], wl.Qseed,
                       wl.Qf, wl.gate)
    np.testing.assert_allclose(b["Y"], a["Y"][:, :, perm], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["Z"], a["Z"], rtol=1e-12, atol=1e-14)


def test_lse_merge_equals_unsplit_encoder():
    """Appendix B.2-B.3: the merge of shard results is the unsplit encoder,
    including an empty shard (L_r = -inf, Z_r = 0)."""
    q = RNG.normal(size=(9, 16)) * 2
    k = RNG.normal(size=(103, 16)) * 2
    v = RNG.normal(size=(103, 16))
    z, lse = oracle.encode(q, k, v)
    cuts = [0, 10, 10, 57, 103]  # second shard is empty
    parts = [oracle.encode_partial(q, k[a:b], v[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    assert np.all(np.isneginf(parts[1][1])) and np.all(parts[1][0] == 0)
    zm, lm = oracle.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(zm, z, rtol=1e-12)
    np.testing.assert_allclose(lm, lse, rtol=1e-13)


# ----------------------------------------------------------------- brute force
def _brute_force_head(K, V, Ks, Qs, Qf, g, eps=1e-6):
    """Eq. 5-8 as scalar loops with the math module only (tiny sizes)."""
    N, D = len(K), len(K[0])
    M = len(Qs)
    s = 1.0 / math.sqrt(D)

    def nrm(row):
        ms = sum(x * x for x in row) / len(row)
        return [x / math.sqrt(ms + eps) for x in row]

    def attend(qrow, keys, vals):
        sc = [s * sum(qrow[d] * key[d] for d in range(D)) for key in keys]
        mx = max(sc)
        w = [math.exp(x - mx) for x in sc]
        tot = sum(w)
        return [sum(w[j] * vals[j][d] for j in range(len(keys))) / tot for d in range(len(vals[0]))]

    kt = [nrm(r) for r in Ks]
    qd = [attend(Qs[m], kt, kt) for m in range(M)]
    qf = [nrm(r) for r in Qf]
    q = [[qf[m][d] + g * qd[m][d] for d in range(D)] for m in range(M)]
    z = [attend(q[m], K, V) for m in range(M)]
    y = [attend(K[n], q, z) for n in range(N)]
    return qd, q, z, y


def test_brute_force_tiny():
    wl = workloads.config("tiny", N=7, M=3, D=4)
    for h in range(2):
        args = [wl.K[0, h].tolist(), wl.V[0, h].tolist(), wl.Ks_raw[0, h].tolist(),
                wl.Qseed[h].tolist(), wl.Qf[h].tolist(), float(wl.gate[h])]
        qd, q, z, y = _brute_force_head(*args)
        r = oracle.forward_head(wl.K[0, h], wl.V[0, h], wl.Ks_raw[0, h], wl.Qseed[h], wl.Qf[h],
                                wl.gate[h])
        np.testing.assert_allclose(r["Qd"], qd, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Q"], q, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Z"], z, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["Y"], y, rtol=1e-12, atol=1e-14)


def test_brute_force_peaked_synthesis():
    """Large seeds make the synthesis attention concentrate; brute force agrees."""
    wl = workloads.config("tiny", N=9, M=4, D=4, qseed_scale=8.0)
    h = 1
    qd, q, z, y = _brute_force_head(wl.K[0, h].tolist(), wl.V[0, h].tolist(),
                                    wl.Ks_raw[0, h].tolist(), wl.Qseed[h].tolist(),
                                    wl.Qf[h].tolist(), float(wl.gate[h]))
    r = oracle.forward_head(wl.K[0, h], wl.V[0, h], wl.Ks_raw[0, h], wl.Qseed[h], wl.Qf[h],
                            wl.gate[h])
    np.testing.assert_allclose(r["Qd"], qd, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["Y"], y, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("name", ["tiny", "pde2d", "mesh3d", "lra", "aero"])
def test_workload_statistics(name):
    """Synthetic inputs have the stated marginals (about N(0,1) tokens)."""
    wl = workloads.config(name, B=1, H=2, N=2048)
    for t in (wl.K, wl.V, wl.Ks_raw):
        assert abs(float(t.mean())) < 0.1
        assert 0.85 < float(t.std()) < 1.15
    D = wl.shape.D
    assert 0.8 < float(wl.Qseed.std()) * math.sqrt(D) < 1.2
    assert np.all((wl.gate > 0) & (wl.gate < 1))
