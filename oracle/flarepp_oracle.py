"""CPU fp64 oracle of the FLARE++ mixer forward. TEST INFRASTRUCTURE ONLY.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import this module. The library path never calls it; it shares no code
with the CUDA kernels (both sides are only fed from the seeded input module).

It is the plain definition written out in float64 with numpy, following the
FLARE++ paper ("FLARE++: Low-rank attention with attention-synthesized
routing", arXiv 2608.11519 v2):

* SDPA(Q, K, V) = softmax(Q K^T / sqrt(D)) V, softmax over the keys
  (Section 3.1, eq. 1), evaluated with the max shift of Appendix B.3 eq. 29.
* synthesis keys K~ = N0(Ks_raw), shared as values (Section 3.2 eq. 5,
  Appendix A.3 eq. 14, A.6 eq. 19).
* Q^d = SDPA(Qseed, K~, K~) (eq. 6 / eq. 19).
* Q = N0(Q^f) + g * Q^d (eq. 7 / eq. 15).
* Z = SDPA(Q, K, V), L = log-sum-exp of the encode scores (eq. 8, B.2 eq. 25).
* Y = SDPA(K, Q, Z), softmax over the M routes (eq. 8, Figure 1 caption).
* the mixer variants the paper defines beside it, at the end of the module:
  FLARE (Section 3.1 eq. 3), separate synthesis values (Appendix A.1 eq. 11)
  and simplified FLARE++ (Appendix A.8 eq. 20);
* the token projections that produce the mixer's inputs, with their per-head
  normalisations (Section 3.2, Appendix A.7);
* the mixer's backward pass (Appendix B.5 eq. 46-49 for each attention call,
  the chain rule through the gate and N0).

Readings where the paper is silent (each one is also listed in the design
notes of the repository):

1. N0 is RMSNorm without scale over the head width D with eps = 1e-6 inside the
   square root; the paper gives no eps.
2. Qseed arrives with its learned-scale normalisation N_a already applied, and
   K with its N_a applied (eq. 6 and the routing keys of eq. 8); the oracle uses
   both as given.
3. ``gate`` is g = sigmoid(gamma) itself, one value per head.
4. All three calls use the scale 1/sqrt(D), so the decode scores are the
   transpose of the encode scores.
5. No intermediate rounding: the oracle takes the (already dtype-rounded)
   inputs to float64 and rounds nothing afterwards.

Row blocking (``rows``) only splits independent softmax rows into groups to
bound memory; every row is computed by the same formula.

Parity status: every function here is pinned by tests against closed forms,
invariants, library routines and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

EPS = 1e-6


def n0(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    """Affine-free RMSNorm over the last axis, N0 (Section 3.2, eq. 5).

    Each row is divided by sqrt(mean of squares + eps), so it has unit RMS up to
    the eps term.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax over the last axis with the max shift (Appendix B.3 eq. 29)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def logsumexp_rows(s: np.ndarray) -> np.ndarray:
    """log sum_j exp(s_j) over the last axis, via the shift identity (eq. 29)."""
    m = np.max(s, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(s - m), axis=-1, keepdims=True)))[..., 0]


def sdpa(q: np.ndarray, k: np.ndarray, v: np.ndarray, with_lse: bool = False,
         rows: int | None = None):
    """SDPA(Q, K, V) of eq. 1 for one head: q [Nq, D], k [Nk, D], v [Nk, Dv].

    Scores are q k^T / sqrt(D) with D = q.shape[-1]; the softmax runs over the
    Nk keys. With ``with_lse`` it also returns the row log-normaliser L of
    Appendix B.2 eq. 25. ``rows`` caps how many query rows are scored at once.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, d = q.shape
    scale = 1.0 / math.sqrt(d)
    step = nq if rows is None else max(1, rows)
    out = np.empty((nq, v.shape[1]), dtype=np.float64)
    lse = np.empty(nq, dtype=np.float64)
    for r0 in range(0, nq, step):
        r1 = min(nq, r0 + step)
        s = (q[r0:r1] @ k.T) * scale
        out[r0:r1] = softmax_rows(s) @ v
        if with_lse:
            lse[r0:r1] = logsumexp_rows(s)
    return (out, lse) if with_lse else out


def synthesis(qseed_h: np.ndarray, ks_raw_bh: np.ndarray, rows: int | None = None) -> np.ndarray:
    """Synthesised corrections Q^d = SDPA(Qseed, N0(Ks_raw), N0(Ks_raw)).

    Section 3.2 eq. 5-6 with shared keys and values (Appendix A.6 eq. 19).
    qseed_h [M, D], ks_raw_bh [N, D] -> [M, D].
    """
    kt = n0(ks_raw_bh)
    return sdpa(qseed_h, kt, kt, rows=rows)


def routing_queries(qf_h: np.ndarray, qd: np.ndarray, g: float) -> np.ndarray:
    """Q = N0(Q^f) + g Q^d (Section 3.2 eq. 7, Appendix A.4 eq. 15)."""
    return n0(qf_h) + float(g) * np.asarray(qd, dtype=np.float64)


def encode(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: int | None = None):
    """Z = SDPA(Q, K, V) and its log-normaliser L (eq. 8; Appendix B.2 eq. 23-25).

    q [M, D], k [N, D], v [N, D] -> Z [M, D], L [M]; softmax over the N tokens.
    """
    return sdpa(q, k, v, with_lse=True, rows=rows)


def decode(k: np.ndarray, q: np.ndarray, z: np.ndarray, rows: int | None = None) -> np.ndarray:
    """Y = SDPA(K, Q, Z): each token attends over the M routes (eq. 8).

    k [N, D], q [M, D], z [M, D] -> [N, D]; softmax over M (Figure 1 caption).
    """
    return sdpa(k, q, z, rows=rows)


def forward_head(k, v, ks_raw, qseed_h, qf_h, g, rows: int | None = None) -> dict:
    """The whole mixer for one (batch, head): returns Qd, Q, Z, L and Y."""
    qd = synthesis(qseed_h, ks_raw, rows=rows)
    q = routing_queries(qf_h, qd, g)
    z, lse = encode(q, k, v, rows=rows)
    y = decode(k, q, z, rows=rows)
    return {"Qd": qd, "Q": q, "Z": z, "L": lse, "Y": y}


def forward(K, V, Ks_raw, Qseed, Qf, gate, rows: int | None = None) -> dict:
    """The mixer over all batches and heads.

    K, V, Ks_raw [B,H,N,D]; Qseed, Qf [H,M,D]; gate [H]. Returns float64 arrays
    Qd, Q, Z [B,H,M,D], L [B,H,M] and Y [B,H,N,D].
    """
    B, H, N, D = K.shape
    M = Qseed.shape[1]
    res = {"Qd": np.empty((B, H, M, D)), "Q": np.empty((B, H, M, D)),
           "Z": np.empty((B, H, M, D)), "L": np.empty((B, H, M)), "Y": np.empty((B, H, N, D))}
    for b in range(B):
        for h in range(H):
            r = forward_head(K[b, h], V[b, h], Ks_raw[b, h], Qseed[h], Qf[h], gate[h], rows=rows)
            for key in res:
                res[key][b, h] = r[key]
    return res


def encode_partial(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """Encoder on one token shard: (Z_r, L_r) of Appendix B.2 eq. 24-26.

    An empty shard returns Z_r = 0 and L_r = -inf (Appendix B.3, last paragraph).
    """
    q = np.asarray(q, dtype=np.float64)
    if k.shape[0] == 0:
        return np.zeros((q.shape[0], v.shape[1])), np.full(q.shape[0], -np.inf)
    return sdpa(q, k, v, with_lse=True)


def lse_merge(z_parts, l_parts):
    """Exact merge of shard results by the stable schedule of Appendix B.3.

    L_max = max_r L_r (eq. 30); d_r = exp(L_r - L_max), U_r = d_r Z_r (eq. 31);
    d = sum d_r, U = sum U_r (eq. 32); Z = U / d, L = L_max + log d (eq. 33).
    Shards with L_r = -inf contribute d_r = U_r = 0.
    """
    l_stack = np.stack([np.asarray(x, dtype=np.float64) for x in l_parts])  # [R, M]
    z_stack = np.stack([np.asarray(x, dtype=np.float64) for x in z_parts])  # [R, M, D]
    l_max = np.max(l_stack, axis=0)
    d_r = np.exp(l_stack - l_max[None, :])
    u_r = d_r[:, :, None] * z_stack
    d = np.sum(d_r, axis=0)
    u = np.sum(u_r, axis=0)
    return u / d[:, None], l_max + np.log(d)


def w_eff(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """The N x N operator W_dec W_enc of eq. 4 / eq. 9, materialised.

    W_enc = softmax over N of Q K^T / sqrt(D) ([M, N]); W_dec = softmax over M
    of K Q^T / sqrt(D) ([N, M]). Only for tiny N: it is what the fused path
    never builds.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    s = (q @ k.T) / math.sqrt(q.shape[1])
    w_enc = softmax_rows(s)
    w_dec = softmax_rows(s.T)
    return w_dec @ w_enc


# ------------------------------------------------------------------ variants
# The FLARE++ paper also defines the mixer it improves on (FLARE, Section 3.1
# eq. 2-3), the general form with a separate synthesis value projection
# (Appendix A.1 eq. 11) and the simplified variant (Appendix A.8 eq. 20).
# Readings where the paper leaves a step open (also in the design notes):
#
# 6. FLARE's learned queries Q_h are used as given; the caller owns any
#    normalisation of Q_h and of K.
# 7. In the general form the library applies N0 to the synthesis keys only;
#    the separate values V~ are used as given. V~ = N0(Ks_raw) is the default
#    shared configuration.
# 8. In the simplified variant the learned-scale normalisations N_a of the
#    seeds and of the synthesis keys are applied by the caller (as for K in
#    the main mixer); V~ is unnormalised; there is no reference and no gate,
#    so Q = Q^d.


def flare_forward_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: int | None = None) -> dict:
    """FLARE for one (batch, head): Z = SDPA(Q_h, K, V), Y = SDPA(K, Q_h, Z)
    (Section 3.1 eq. 3). q [M, D] is the head's learned query set."""
    z, lse = encode(q, k, v, rows=rows)
    y = decode(k, q, z, rows=rows)
    return {"Q": np.asarray(q, dtype=np.float64), "Z": z, "L": lse, "Y": y}


def flare_forward(Q, K, V, rows: int | None = None) -> dict:
    """FLARE over all batches and heads. Q [H,M,D]; K, V [B,H,N,D].

    Returns Q, Z [B,H,M,D], L [B,H,M] and Y [B,H,N,D] (float64)."""
    B, H, N, D = K.shape
    M = Q.shape[1]
    res = {"Q": np.empty((B, H, M, D)), "Z": np.empty((B, H, M, D)), "L": np.empty((B, H, M)),
           "Y": np.empty((B, H, N, D))}
    for b in range(B):
        for h in range(H):
            r = flare_forward_head(Q[h], K[b, h], V[b, h], rows=rows)
            for key in res:
                res[key][b, h] = r[key]
    return res


def synthesis_unshared(qseed_h: np.ndarray, ks_raw_bh: np.ndarray, vs_bh: np.ndarray,
                       rows: int | None = None) -> np.ndarray:
    """Q^d = SDPA(Qseed, N0(Ks_raw), V~) with a separate value projection V~
    (Appendix A.1 eq. 11, keys normalised as in Section 3.2 eq. 5)."""
    return sdpa(qseed_h, n0(ks_raw_bh), vs_bh, rows=rows)


def synthesis_simplified(qseed_h: np.ndarray, ks_bh: np.ndarray, vs_bh: np.ndarray,
                         rows: int | None = None) -> np.ndarray:
    """Q = Q^d = SDPA(N_a(Q~), N_a(K~), V~) (Appendix A.8 eq. 20), with the
    N_a already applied to ``qseed_h`` and ``ks_bh`` by the caller."""
    return sdpa(qseed_h, ks_bh, vs_bh, rows=rows)


def _route(q, k, v, rows):
    z, lse = encode(q, k, v, rows=rows)
    return z, lse, decode(k, q, z, rows=rows)


def forward_unshared(K, V, Ks_raw, Vs, Qseed, Qf, gate, rows: int | None = None) -> dict:
    """FLARE++ with separate synthesis values (eq. 11): Q^d from
    ``synthesis_unshared``, then Q = N0(Q^f) + g Q^d and eq. 8 as in ``forward``.
    Vs [B,H,N,D]; the other arguments as in ``forward``."""
    B, H, N, D = K.shape
    M = Qseed.shape[1]
    res = {"Qd": np.empty((B, H, M, D)), "Q": np.empty((B, H, M, D)),
           "Z": np.empty((B, H, M, D)), "L": np.empty((B, H, M)), "Y": np.empty((B, H, N, D))}
    for b in range(B):
        for h in range(H):
            qd = synthesis_unshared(Qseed[h], Ks_raw[b, h], Vs[b, h], rows=rows)
            q = routing_queries(Qf[h], qd, gate[h])
            z, lse, y = _route(q, K[b, h], V[b, h], rows)
            for key, val in (("Qd", qd), ("Q", q), ("Z", z), ("L", lse), ("Y", y)):
                res[key][b, h] = val
    return res


def forward_simplified(K, V, Ks, Vs, Qseed, rows: int | None = None) -> dict:
    """Simplified FLARE++ (eq. 20): Q = SDPA(Qseed, Ks, Vs), then eq. 8.
    Ks, Vs [B,H,N,D] as used (N_a applied to Ks by the caller); Qseed [H,M,D]."""
    B, H, N, D = K.shape
    M = Qseed.shape[1]
    res = {"Q": np.empty((B, H, M, D)), "Z": np.empty((B, H, M, D)), "L": np.empty((B, H, M)),
           "Y": np.empty((B, H, N, D))}
    for b in range(B):
        for h in range(H):
            q = synthesis_simplified(Qseed[h], Ks[b, h], Vs[b, h], rows=rows)
            z, lse, y = _route(q, K[b, h], V[b, h], rows)
            for key, val in (("Q", q), ("Z", z), ("L", lse), ("Y", y)):
                res[key][b, h] = val
    return res


# ---------------------------------------------------------------- projection
# The pointwise projections that produce the mixer's inputs (Section 3.2 and
# Appendix A.7 Table 2: K = N_a(X W_K), V = X W_V, K~ = X W~_K, each a plain
# linear map per token, heads split along the output channels). Readings (also
# in the design notes):
#
# 9.  The output channels of one projection are ordered head-major:
#     channel h*D + d is element d of head h (D = C / H).
# 10. A bias, when present, is added before the normalisation.
# 11. N_a is RMSNorm over D with a learned scale of D values shared by all
#     heads (Appendix A.7 counts D parameters for an affine per-head norm);
#     eps = 1e-6 as N0.

NORM_NONE, NORM_N0, NORM_NA = 0, 1, 2


def project(X, W, bias, norms, scales, H: int) -> list:
    """Fused projections of the mixer's token inputs.

    X [B, N, C]; W [P*C, C] (P stacked projections, torch Linear layout
    out x in); bias [P*C] or None; norms: P codes (NORM_NONE, NORM_N0,
    NORM_NA); scales [P, D] (row p used when norms[p] == NORM_NA) or None.
    Returns P float64 arrays [B, H, N, D]:
    out_p = norm_p(X W_p^T + b_p), normalised per head over D.
    """
    X = np.asarray(X, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    B, N, C = X.shape
    P = len(norms)
    D = C // H
    y = X @ W.T  # [B, N, P*C]
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)
    outs = []
    for p in range(P):
        part = y[:, :, p * C:(p + 1) * C].reshape(B, N, H, D).transpose(0, 2, 1, 3)
        if norms[p] == NORM_N0:
            part = n0(part)
        elif norms[p] == NORM_NA:
            part = n0(part) * np.asarray(scales[p], dtype=np.float64)
        elif norms[p] != NORM_NONE:
            raise ValueError(norms[p])
        outs.append(np.ascontiguousarray(part))
    return outs


# ------------------------------------------------------------------ backward
# Reverse mode of the mixer (the training direction). For each attention call
# out = softmax(s q k^T) v the local backward of Appendix B.5 eq. 46-49 is
# used with a single shard (the merged L, so P = exp(S - L)) and no cotangent
# on L (the mixer's output does not depend on L):
#   dv = P^T dout,  c = <dout, out>_D per row,  dS = P o (dout v^T - c),
#   dk = s dS^T q,  dq = s dS k.
# The decode is the same call with the softmax over the M routes (queries K,
# keys Q, values Z). The gate and N0 follow by the chain rule; the per-head
# parameters (Qseed, Qf, g) collect their gradient over the batch.
# Reading (also in the design notes):
# 12. Gradients flow through Q as the forward computed it, unrounded; the
#     routing queries, seeds and fixed queries are treated as exact.


def sdpa_backward(q, k, v, dout):
    """Gradients (dq, dk, dv) of out = SDPA(q, k, v) for the cotangent dout
    (Appendix B.5 eq. 46-49 with one shard and zero cotangent on L)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    s = 1.0 / math.sqrt(q.shape[1])
    scores = s * (q @ k.T)
    lse = logsumexp_rows(scores)
    p = np.exp(scores - lse[:, None])
    out = p @ v
    dv = p.T @ dout
    c = np.sum(dout * out, axis=1)
    ds = p * (dout @ v.T - c[:, None])
    return s * (ds @ k), s * (ds.T @ q), dv


def n0_backward(x, dy, eps: float = EPS):
    """Gradient of y = N0(x) row-wise: dx = r (dy - y <dy, y> / D), r = (ms + eps)^-1/2."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    y = x * r
    return r * (dy - y * np.mean(dy * y, axis=-1, keepdims=True))


def backward_head(k, v, ks_raw, qseed_h, qf_h, g, dy) -> dict:
    """Gradients of the mixer for one (batch, head) given dY [N, D]:
    dK, dV, dKs_raw [N, D], dQseed, dQf [M, D] and dgate (a float)."""
    kt = n0(ks_raw)
    qd = sdpa(qseed_h, kt, kt)
    q = routing_queries(qf_h, qd, g)
    z = sdpa(q, k, v)
    dk_dec, dq_dec, dz = sdpa_backward(k, q, z, dy)   # decode: queries K, keys Q, values Z
    dq_enc, dk_enc, dv = sdpa_backward(q, k, v, dz)   # encode
    dq = dq_dec + dq_enc
    dqd = float(g) * dq
    dgate = float(np.sum(dq * qd))
    dqf = n0_backward(qf_h, dq)
    dqseed, dkt_keys, dkt_vals = sdpa_backward(qseed_h, kt, kt, dqd)
    dks = n0_backward(ks_raw, dkt_keys + dkt_vals)
    return {"dK": dk_dec + dk_enc, "dV": dv, "dKs_raw": dks, "dQseed": dqseed, "dQf": dqf,
            "dgate": dgate}


def backward(K, V, Ks_raw, Qseed, Qf, gate, dY) -> dict:
    """Gradients over all batches and heads: dK, dV, dKs_raw [B,H,N,D];
    dQseed, dQf [H,M,D] and dgate [H], summed over the batch."""
    B, H, N, D = K.shape
    M = Qseed.shape[1]
    res = {"dK": np.empty((B, H, N, D)), "dV": np.empty((B, H, N, D)),
           "dKs_raw": np.empty((B, H, N, D)), "dQseed": np.zeros((H, M, D)),
           "dQf": np.zeros((H, M, D)), "dgate": np.zeros(H)}
    for b in range(B):
        for h in range(H):
            r = backward_head(K[b, h], V[b, h], Ks_raw[b, h], Qseed[h], Qf[h], gate[h], dY[b, h])
            for key in ("dK", "dV", "dKs_raw"):
                res[key][b, h] = r[key]
            res["dQseed"][h] += r["dQseed"]
            res["dQf"][h] += r["dQf"]
            res["dgate"][h] += r["dgate"]
    return res
