"""Pins of the oracle's backward pass (FLARE++ paper, Appendix B.5 eq. 46-49
for each attention call, the chain rule through the gate and N0).

Expected values come from outside the backward code: central finite
differences of the (separately pinned) forward oracle, torch's autograd in
float64 for the library attention routine, and identities of the softmax."""
import numpy as np
import pytest

import oracle
from rank_latent_routing_gb300 import workloads

RNG = np.random.default_rng(2024)


def _loss(fwd_y, w):
    return float(np.sum(fwd_y * w))


def _fd(fun, x, h=1e-6):
    """Central differences of the scalar fun over every element of x."""
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = fun()
        x[i] = old - h
        fm = fun()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("qseed_scale", [1.0, 6.0])
def test_backward_matches_finite_differences(qseed_scale):
    """Every gradient of the whole mixer against central differences of the
    forward oracle, for the loss <Y, W> with a random W (tiny sizes)."""
    wl = workloads.config("tiny", B=2, H=2, N=6, M=3, D=4, qseed_scale=qseed_scale)
    K, V, Ks = (wl.K.astype(np.float64), wl.V.astype(np.float64), wl.Ks_raw.astype(np.float64))
    Qs, Qf = wl.Qseed.astype(np.float64), wl.Qf.astype(np.float64)
    g = wl.gate.astype(np.float64)
    W = RNG.normal(size=K.shape)
    got = oracle.backward(K, V, Ks, Qs, Qf, g, W)

    def f():
        return _loss(oracle.forward(K, V, Ks, Qs, Qf, g)["Y"], W)

    for name, arr in (("dK", K), ("dV", V), ("dKs_raw", Ks), ("dQseed", Qs), ("dQf", Qf),
                      ("dgate", g)):
        want = _fd(f, arr)
        np.testing.assert_allclose(got[name], want, rtol=1e-6, atol=1e-8, err_msg=name)


def test_sdpa_backward_matches_torch_autograd():
    """The attention backward against torch's autograd of its own float64
    scaled_dot_product_attention (a library routine)."""
    import torch
    q = torch.tensor(RNG.normal(size=(5, 8)), requires_grad=True)
    k = torch.tensor(RNG.normal(size=(9, 8)) * 1.5, requires_grad=True)
    v = torch.tensor(RNG.normal(size=(9, 8)), requires_grad=True)
    dout = RNG.normal(size=(5, 8))
    out = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None])[0]
    out.backward(torch.tensor(dout))
    dq, dk, dv = oracle.sdpa_backward(q.detach().numpy(), k.detach().numpy(),
                                      v.detach().numpy(), dout)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-11, atol=1e-13)


def test_sdpa_backward_identities():
    """Three softmax identities: rows of P sum to 1, so sum_n dV_n =
    sum_m dout_m; the score cotangent rows sum to 0 (shift invariance), so
    with identical query rows the key gradients sum to 0; and constant value
    rows make the output independent of q and k (dq = dk = 0)."""
    q = RNG.normal(size=(4, 8))
    k = RNG.normal(size=(7, 8))
    v = RNG.normal(size=(7, 8))
    dout = RNG.normal(size=(4, 8))
    dq, dk, dv = oracle.sdpa_backward(q, k, v, dout)
    np.testing.assert_allclose(dv.sum(axis=0), dout.sum(axis=0), rtol=1e-12)
    # identical query rows: the key gradients sum to zero
    q1 = np.tile(q[:1], (4, 1))
    _, dk1, _ = oracle.sdpa_backward(q1, k, v, dout)
    np.testing.assert_allclose(dk1.sum(axis=0), 0.0, atol=1e-12)
    # constant values: the output does not depend on q or k
    vc = np.tile(RNG.normal(size=(1, 8)), (7, 1))
    dqc, dkc, _ = oracle.sdpa_backward(q, k, vc, dout)
    np.testing.assert_allclose(dqc, 0.0, atol=1e-12)
    np.testing.assert_allclose(dkc, 0.0, atol=1e-12)


def test_n0_backward_matches_finite_differences_and_is_orthogonal():
    x = RNG.normal(size=(3, 8)) * 2
    dy = RNG.normal(size=(3, 8))
    got = oracle.n0_backward(x, dy)

    def f():
        return float(np.sum(oracle.n0(x) * dy))

    np.testing.assert_allclose(got, _fd(f, x), rtol=1e-7, atol=1e-9)
    # N0 is scale invariant up to eps: the gradient is orthogonal to x up to eps
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.sum(got * x, axis=-1), 0.0, atol=1e-5 * np.max(np.abs(dy)) / ms.min())


def test_backward_zero_cotangent_and_gate_zero():
    """dY = 0 gives zero gradients; with g = 0 the synthesis receives no
    gradient, so dQseed = dKs_raw = 0 (eq. 7)."""
    wl = workloads.config("tiny", N=20, M=4, D=8)
    z = oracle.backward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate, np.zeros(wl.K.shape))
    for key in ("dK", "dV", "dKs_raw", "dQseed", "dQf", "dgate"):
        assert np.all(z[key] == 0), key
    g0 = np.zeros_like(wl.gate)
    r = oracle.backward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, g0, RNG.normal(size=wl.K.shape))
    assert np.all(r["dQseed"] == 0) and np.all(r["dKs_raw"] == 0)
    assert np.any(r["dgate"] != 0) and np.any(r["dQf"] != 0)
