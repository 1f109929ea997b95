"""GPU parity of the mixer variants against the fp64 oracle: FLARE (Section 3.1
eq. 3), separate synthesis values (Appendix A.1 eq. 11) and simplified FLARE++
(Appendix A.8 eq. 20), through the library's C ABI.

Mid-size cases compare every element of Y and of the intermediates; two
full-size workloads compare sampled rows computed by the oracle head by head.
"""
import numpy as np
import pytest

import oracle
from rank_latent_routing_gb300 import workloads
from tests.helpers import assert_parity, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_latent_routing_gb300 import flarepp
    return flarepp


def _extra_to_device(wl, ex, device="cuda"):
    import torch
    out = {}
    for k in ("Vs", "Qlat"):
        if wl.dtype == "bf16":
            bits = np.ascontiguousarray(ex[k + "_bits"]).view(np.int16)
            out[k] = torch.from_numpy(bits).to(device).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(ex[k])).to(device)
    return out


def _host(r):
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in r.items()}


def _run(fp, variant, wl, ex, host=True):
    import torch
    t = to_device(wl)
    e = _extra_to_device(wl, ex)
    if variant == "flare":
        r = fp.flare_forward(e["Qlat"], t["K"], t["V"], debug=True)
    elif variant == "unshared":
        r = fp.forward_variant("unshared", t["K"], t["V"], t["Ks_raw"], e["Vs"], t["Qseed"],
                               t["Qf"], t["gate"], debug=True)
    else:
        r = fp.forward_variant("simplified", t["K"], t["V"], t["Ks_raw"], e["Vs"], t["Qseed"],
                               debug=True)
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    return _host(r) if host else r


def _oracle(variant, wl, ex):
    if variant == "flare":
        return oracle.flare_forward(ex["Qlat"], wl.K, wl.V)
    if variant == "unshared":
        return oracle.forward_unshared(wl.K, wl.V, wl.Ks_raw, ex["Vs"], wl.Qseed, wl.Qf, wl.gate)
    return oracle.forward_simplified(wl.K, wl.V, wl.Ks_raw, ex["Vs"], wl.Qseed)


# (structure, B, H, N, M, D, dtype): every slot mode of the kernels (M <= 64,
# one 128-row block, pairs of blocks, an odd block count), ragged token tails,
# N = 1, and the fp32 build
CASES = [
    ("iid", 1, 2, 999, 40, 32, "fp32"),
    ("iid", 2, 1, 1, 16, 16, "fp32"),
    ("iid", 1, 3, 1000, 64, 16, "bf16"),
    ("iid", 2, 2, 3001, 128, 32, "bf16"),
    ("lowrank", 1, 2, 2500, 256, 32, "bf16"),
    ("points", 1, 1, 4097, 512, 32, "bf16"),
    ("iid", 1, 2, 5000, 192, 16, "bf16"),
    ("iid", 1, 2, 129, 48, 16, "bf16"),
    ("iid", 1, 1, 1, 64, 32, "bf16"),
]
VARIANTS = ["flare", "unshared", "simplified"]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_variant_parity_against_oracle(fp, variant, case):
    structure, B, H, N, M, D, dtype = case
    wl = workloads.make(workloads.Shape(B, H, N, M, D), dtype, structure, seed=29 + N + M)
    ex = workloads.variant_inputs(wl)
    got = _run(fp, variant, wl, ex)
    want = _oracle(variant, wl, ex)
    assert_parity(got["Y"], want["Y"], dtype, f"{variant} Y")
    assert_parity(got["Z"], want["Z"], dtype, f"{variant} Z")
    if variant != "flare":
        assert_parity(got["Q"], want["Q"], dtype, f"{variant} Q")
    if variant == "unshared":
        assert_parity(got["Qd"], want["Qd"], dtype, f"{variant} Qd")
    # bf16 routing queries move the encode scores by about 2^-9 of their size
    np.testing.assert_allclose(got["L"], want["L"], rtol=0 if dtype == "bf16" else 1e-6,
                               atol=2e-2 if dtype == "bf16" else 1e-6)


def test_simplified_leaves_qd_untouched(fp):
    """The simplified variant has no separate Qd (Q is Qd): the debug copy of
    Qd is not written, Q is."""
    import torch
    wl = workloads.make(workloads.Shape(1, 2, 700, 64, 16), "bf16", "iid", seed=3)
    ex = workloads.variant_inputs(wl)
    t = to_device(wl)
    e = _extra_to_device(wl, ex)
    qd = torch.full((1, 2, 64, 16), 7.0, device="cuda")
    q = torch.zeros((1, 2, 64, 16), device="cuda")
    out = torch.empty_like(t["K"])
    from ctypes import c_void_p
    with torch.cuda.device(0):
        rc = fp.raw_call("flarepp_forward_variant", 2, c_void_p(t["K"].data_ptr()),
                         c_void_p(t["V"].data_ptr()), c_void_p(t["Ks_raw"].data_ptr()),
                         c_void_p(e["Vs"].data_ptr()), c_void_p(t["Qseed"].data_ptr()), None, None,
                         1, 2, 700, 64, 16, 0, c_void_p(out.data_ptr()), c_void_p(qd.data_ptr()),
                         c_void_p(q.data_ptr()), None, None,
                         c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    assert bool((qd == 7.0).all())
    want = oracle.forward_simplified(wl.K, wl.V, wl.Ks_raw, ex["Vs"], wl.Qseed)
    assert_parity(q.cpu().numpy(), want["Q"], "bf16", "simplified Q")


def test_flare_matches_default_mixer_with_zero_gate(fp):
    """FLARE with Q_h = N0(Q^f) (as bf16) and the default mixer with g = 0
    route identically (eq. 7): the two GPU results agree to rounding."""
    import torch
    wl = workloads.make(workloads.Shape(1, 2, 2000, 128, 32), "bf16", "iid", seed=8)
    wl.gate[:] = 0.0
    dflt = _host(fp.forward_debug(*[to_device(wl)[k] for k in
                                    ("K", "V", "Ks_raw", "Qseed", "Qf", "gate")]))
    q = torch.from_numpy(dflt["Q"][0].astype(np.float32)).cuda().to(torch.bfloat16)
    t = to_device(wl)
    fl = _host(fp.flare_forward(q.contiguous(), t["K"], t["V"], debug=True))
    np.testing.assert_allclose(fl["Z"], dflt["Z"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(fl["Y"], dflt["Y"], rtol=0, atol=1e-6)


def _sampled_rows(N, count, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=min(count, N), replace=False).tolist())
    rows.update({0, N - 1})
    return np.array(sorted(rows))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["pde2d", "lra"])
def test_variant_full_size_sampled(fp, variant, name):
    """Full-size workloads: Q, Z, L of two heads in full and Y on sampled
    token rows, against the oracle one head at a time."""
    import torch
    wl = workloads.config(name)
    ex = workloads.variant_inputs(wl)
    dev = _run(fp, variant, wl, ex, host=False)
    got = {k: dev[k].cpu().numpy().astype(np.float64) for k in ("Q", "Z", "L") if k in dev}
    s = wl.shape
    rows = _sampled_rows(s.N, 256, 5)
    for b, h in [(0, 0), (s.B - 1, s.H - 1)]:
        K, V = wl.K[b, h], wl.V[b, h]
        if variant == "flare":
            q = ex["Qlat"][h].astype(np.float64)
        elif variant == "unshared":
            qd = oracle.synthesis_unshared(wl.Qseed[h], wl.Ks_raw[b, h], ex["Vs"][b, h], rows=64)
            q = oracle.routing_queries(wl.Qf[h], qd, wl.gate[h])
        else:
            q = oracle.synthesis_simplified(wl.Qseed[h], wl.Ks_raw[b, h], ex["Vs"][b, h], rows=64)
        if variant != "flare":
            assert_parity(got["Q"][b, h], q, wl.dtype, f"{name} {variant} Q[{b},{h}]")
        z, lse = oracle.encode(q, K, V, rows=64)
        assert_parity(got["Z"][b, h], z, wl.dtype, f"{name} {variant} Z[{b},{h}]")
        np.testing.assert_allclose(got["L"][b, h], lse, rtol=1e-6, atol=2e-2)
        y = oracle.decode(K[rows], q, z)
        y_got = dev["Y"][b, h][torch.from_numpy(rows).to(dev["Y"].device)].float().cpu().numpy()
        assert_parity(y_got, y, wl.dtype, f"{name} {variant} Y[{b},{h}] sampled")
    assert bool(torch.isfinite(dev["Y"].float()).all())
