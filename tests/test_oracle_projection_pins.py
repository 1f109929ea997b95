"""Pins of the oracle's token projections (FLARE++ paper, Section 3.2 and
Appendix A.5-A.7: K = N_a(X W_K), V = X W_V, K~ = X W~_K, per-head RMSNorm
over D), each against something other than the oracle's own code."""
import math

import numpy as np

import oracle
from rank_latent_routing_gb300 import workloads

RNG = np.random.default_rng(99)


def _brute(X, W, bias, norms, scales, H, eps=1e-6):
    """The projections as scalar loops with the math module (tiny sizes)."""
    B, N, C = len(X), len(X[0]), len(X[0][0])
    D = C // H
    P = len(norms)
    out = [[[[None] * N for _ in range(H)] for _ in range(B)] for _ in range(P)]
    for p in range(P):
        for b in range(B):
            for n in range(N):
                for h in range(H):
                    row = []
                    for d in range(D):
                        o = p * C + h * D + d
                        acc = sum(X[b][n][k] * W[o][k] for k in range(C))
                        row.append(acc + (bias[o] if bias is not None else 0.0))
                    if norms[p] != 0:
                        ms = sum(v * v for v in row) / D
                        r = 1.0 / math.sqrt(ms + eps)
                        row = [v * r for v in row]
                        if norms[p] == 2:
                            row = [v * scales[p][d] for d, v in enumerate(row)]
                    out[p][b][h][n] = row
    return out


def test_projection_brute_force_tiny():
    pr = workloads.projection_inputs(2, 2, 3, 4, dtype="fp32", norms=(2, 0, 1, 0))
    got = oracle.project(pr.X, pr.W, pr.bias, pr.norms, pr.scales, pr.H)
    want = _brute(pr.X.tolist(), pr.W.tolist(), pr.bias.tolist(), pr.norms, pr.scales.tolist(),
                  pr.H)
    for p in range(4):
        np.testing.assert_allclose(got[p], want[p], rtol=1e-12, atol=1e-14)


def test_identity_weights_split_heads():
    """W = I and no bias (eq. 18 with dW = 0): V is X cut into heads, K is
    N_a of each head's slice, and a head-major reshape puts channel h*D + d at
    [h, :, d]."""
    B, N, H, D = 2, 5, 3, 4
    C = H * D
    X = RNG.normal(size=(B, N, C))
    W = np.concatenate([np.eye(C), np.eye(C)])
    a = RNG.uniform(0.5, 2.0, size=(2, D))
    K, V = oracle.project(X, W, None, (oracle.NORM_NA, oracle.NORM_NONE), a, H)
    for b in range(B):
        for h in range(H):
            sl = X[b, :, h * D:(h + 1) * D]
            np.testing.assert_allclose(V[b, h], sl, rtol=0, atol=0)
            ms = np.mean(sl * sl, axis=-1, keepdims=True)
            np.testing.assert_allclose(K[b, h], sl / np.sqrt(ms + 1e-6) * a[0], rtol=1e-14)


def test_norm_codes():
    """N_a with unit scale is N0; N_a scales N0 per element; N0 is invariant
    to scaling the input (up to eps); NONE is linear in X."""
    pr = workloads.projection_inputs(1, 2, 40, 8, dtype="fp32", norms=(1, 2, 0))
    C = pr.H * pr.D
    W = np.tile(pr.W[:C], (3, 1))  # the same map for all three outputs
    ones = np.ones_like(pr.scales)
    n0, na1, _ = oracle.project(pr.X, W, None, (1, 2, 0), ones, pr.H)
    np.testing.assert_allclose(na1, n0, rtol=1e-14)
    _, na, _ = oracle.project(pr.X, W, None, (1, 2, 0), pr.scales, pr.H)
    np.testing.assert_allclose(na, n0 * pr.scales[1], rtol=1e-14)
    X64 = pr.X.astype(np.float64)
    n0_big, _, lin_big = oracle.project(5 * X64, W, None, (1, 2, 0), ones, pr.H)
    np.testing.assert_allclose(n0_big, n0, rtol=2e-5)  # eps / (2 ms) for rows with ms >= 0.05
    _, _, lin = oracle.project(pr.X, W, None, (1, 2, 0), ones, pr.H)
    np.testing.assert_allclose(lin_big, 5 * lin, rtol=1e-13)
    # unit RMS rows up to eps
    rms = np.sqrt(np.mean(n0 ** 2, axis=-1))
    assert np.all(np.abs(rms - 1) < 1e-4)


def test_bias_before_norm():
    """The bias enters before the normalisation: with X = 0 the N0 output is
    N0(bias) per head and the NONE output is the bias itself."""
    H, D = 2, 8
    C = H * D
    X = np.zeros((1, 3, C))
    W = RNG.normal(size=(2 * C, C))
    bias = RNG.normal(size=2 * C)
    a, b = oracle.project(X, W, bias, (oracle.NORM_N0, oracle.NORM_NONE), None, H)
    for h in range(H):
        bh = bias[h * D:(h + 1) * D]
        np.testing.assert_allclose(a[0, h, 0], bh / np.sqrt(np.mean(bh * bh) + 1e-6), rtol=1e-14)
        np.testing.assert_allclose(b[0, h, 1], bias[C + h * D:C + (h + 1) * D], rtol=0)


def test_projection_inputs_statistics():
    pr = workloads.projection_inputs(2, 8, 512, 16)
    C = 128
    dw = pr.W.reshape(3, C, C) - np.eye(C)[None]
    assert abs(float(dw.std()) - 0.02) < 0.002 and float(np.abs(dw).max()) <= 0.0401
    assert abs(float(pr.X.std()) - 1.0) < 0.02
    assert pr.norms == (2, 0, 0)
