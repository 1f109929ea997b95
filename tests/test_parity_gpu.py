"""GPU parity: the CUDA path against the fp64 oracle on the same seeded inputs.

Small and mid-size cases compare every element of Y and of the intermediate
results (Q^d, Q, Z, L) through the debug entry point; the five full-size
workloads compare sampled output rows that the oracle computes one head at a
time.
"""
import numpy as np
import pytest

import oracle
from rank_latent_routing_gb300 import workloads
from tests.helpers import assert_parity, max_abs, rel_l2, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_latent_routing_gb300 import flarepp
    return flarepp


def _run_debug(fp, wl, host=True):
    import torch
    t = to_device(wl)
    r = fp.forward_debug(t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"])
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    if not host:
        return r
    return {k: v.float().cpu().numpy().astype(np.float64) for k, v in r.items()}


# (structure, B, H, N, M, D, dtype): several tiles and a ragged token tail each
CASES = [
    ("iid", 1, 2, 1024, 32, 16, "fp32"),     # the tiny workload itself
    ("iid", 1, 2, 999, 40, 32, "fp32"),      # ragged M and N, fp32
    ("iid", 2, 1, 1, 16, 16, "fp32"),        # N = 1
    ("iid", 1, 1, 300, 1, 16, "fp32"),       # M = 1
    ("iid", 1, 3, 1000, 64, 16, "bf16"),
    ("iid", 2, 2, 3001, 128, 32, "bf16"),
    ("lowrank", 1, 2, 2500, 256, 32, "bf16"),
    ("vocab", 2, 2, 1537, 128, 32, "bf16"),
    ("points", 1, 1, 4097, 512, 32, "bf16"),
    ("iid", 1, 2, 777, 16, 16, "bf16"),
    ("iid", 1, 2, 129, 48, 16, "bf16"),
    ("iid", 1, 1, 1, 64, 32, "bf16"),        # N = 1
    ("iid", 1, 2, 5000, 192, 16, "bf16"),    # M not a multiple of 128
    ("iid", 1, 2, 2000, 80, 32, "bf16"),     # last 64-route block of the decode has 16 routes
    ("lowrank", 2, 1, 1500, 144, 16, "bf16"),  # two latent blocks, the second 16 rows; ragged route block
    ("iid", 80, 4, 100, 32, 16, "bf16"),     # 320 heads of one tile: each decode CTA spans three heads
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_parity_against_oracle(fp, case):
    structure, B, H, N, M, D, dtype = case
    wl = workloads.make(workloads.Shape(B, H, N, M, D), dtype, structure, seed=11 + N + M)
    got = _run_debug(fp, wl)
    want = oracle.forward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate)
    assert_parity(got["Y"], want["Y"], dtype, "Y")
    assert_parity(got["Z"], want["Z"], dtype, "Z")
    assert_parity(got["Q"], want["Q"], dtype, "Q")
    assert_parity(got["Qd"], want["Qd"], dtype, "Qd")
    # bf16: the encode scores use Q rounded to bf16 (relative 2^-9), so L moves
    # by up to about 2^-9 times the score magnitudes (|S| < 5 here): atol 1e-2
    np.testing.assert_allclose(got["L"], want["L"], rtol=0 if dtype == "bf16" else 1e-6,
                               atol=1e-2 if dtype == "bf16" else 1e-6)


def test_peaked_synthesis_stage(fp):
    """Large seeds and low-rank synthesis keys concentrate the synthesis
    attention, so a wrong synthesis cannot hide behind a near-uniform average."""
    s = workloads.Shape(1, 2, 3000, 128, 32)
    wl = workloads.make(s, "bf16", "lowrank", seed=5, qseed_scale=8.0)
    got = _run_debug(fp, wl)
    want = oracle.forward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate)
    # the synthesis output is far from its mean here
    assert np.linalg.norm(want["Qd"] - want["Qd"].mean(axis=2, keepdims=True)) > \
        0.3 * np.linalg.norm(want["Qd"])
    assert_parity(got["Qd"], want["Qd"], "bf16", "Qd")
    assert_parity(got["Y"], want["Y"], "bf16", "Y")


def _sampled_rows(N, count, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=min(count, N), replace=False).tolist())
    rows.update({0, N - 1})
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["tiny", "pde2d", "mesh3d", "lra", "aero"])
def test_full_size_workload_sampled(fp, name):
    """Each workload at its full size: Q, Z, L of two heads in full and Y on
    sampled token rows, against the oracle computed head by head."""
    import torch
    wl = workloads.config(name)
    dev = _run_debug(fp, wl, host=False)
    got = {k: dev[k].cpu().numpy().astype(np.float64) for k in ("Qd", "Q", "Z", "L")}
    s = wl.shape
    heads = [(0, 0), (s.B - 1, s.H - 1)]
    rows = _sampled_rows(s.N, 256, 3)
    for b, h in heads:
        qd = oracle.synthesis(wl.Qseed[h], wl.Ks_raw[b, h], rows=64)
        q = oracle.routing_queries(wl.Qf[h], qd, wl.gate[h])
        z, lse = oracle.encode(q, wl.K[b, h], wl.V[b, h], rows=64)
        y = oracle.decode(wl.K[b, h][rows], q, z)
        assert_parity(got["Qd"][b, h], qd, wl.dtype, f"{name} Qd[{b},{h}]")
        assert_parity(got["Q"][b, h], q, wl.dtype, f"{name} Q[{b},{h}]")
        assert_parity(got["Z"][b, h], z, wl.dtype, f"{name} Z[{b},{h}]")
        y_got = dev["Y"][b, h][torch.from_numpy(rows).to(dev["Y"].device)].float().cpu().numpy()
        assert_parity(y_got, y, wl.dtype, f"{name} Y[{b},{h}] sampled")
        np.testing.assert_allclose(got["L"][b, h], lse, rtol=1e-6, atol=1e-2)
    # properties that hold at any size, on every head
    assert bool(torch.isfinite(dev["Y"].float()).all())
    rms_q = np.sqrt(np.mean(got["Q"] ** 2, axis=-1))
    g = wl.gate[None, :, None]
    assert np.all(rms_q <= 1 + g + 2e-2) and np.all(rms_q >= 1 - g - 2e-2)
    assert np.all(np.sqrt(np.mean(got["Qd"] ** 2, axis=-1)) <= 1 + 1e-2)
