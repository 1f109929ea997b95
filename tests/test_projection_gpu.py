"""GPU parity of the fused token projections (flarepp_project) against the
fp64 oracle: every element at small and mid sizes with ragged token tails,
and sampled tokens of a full-size workload."""
import numpy as np
import pytest

import oracle
from rank_latent_routing_gb300 import workloads
from tests.helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_latent_routing_gb300 import flarepp
    return flarepp


def _upload(pr, with_bias=True):
    import torch
    if pr.dtype == "bf16":
        X = torch.from_numpy(np.ascontiguousarray(pr.bits["X"]).view(np.int16)).cuda().view(torch.bfloat16)
        W = torch.from_numpy(np.ascontiguousarray(pr.bits["W"]).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        X = torch.from_numpy(pr.X).cuda()
        W = torch.from_numpy(pr.W).cuda()
    bias = torch.from_numpy(pr.bias).cuda() if with_bias else None
    scales = torch.from_numpy(pr.scales).cuda() if 2 in pr.norms else None
    return X, W, bias, scales


def _bound(got, want, dtype):
    """bf16 outputs: one rounding (2^-9 relative) plus fp32 accumulation of
    C bf16 products; fp32: accumulation order only."""
    rel, absolute = (2.0 ** -8, 2e-3) if dtype == "bf16" else (1e-5, 1e-5)
    err = np.abs(got - want)
    lim = rel * np.abs(want) + absolute
    assert np.all(err <= lim), f"max excess {float(np.max(err - lim)):.3e}"


# (B, H, N, D, dtype, norms, bias): C = H D in {64, 128, 256} for bf16, ragged
# token tails, P from 1 to 4, every norm code, with and without bias
CASES = [
    (2, 8, 1000, 16, "bf16", (2, 0, 0), True),
    (1, 8, 4097, 32, "bf16", (2, 0, 0), True),
    (3, 4, 300, 16, "bf16", (1, 2, 0, 0), True),
    (2, 2, 129, 32, "bf16", (0,), False),
    (1, 8, 127, 32, "bf16", (2, 0, 1, 0), True),
    (2, 16, 513, 16, "bf16", (2, 0, 0), False),
    (1, 4, 1, 16, "bf16", (2, 0), True),
    (2, 3, 100, 16, "fp32", (2, 0, 1), True),
    (1, 2, 77, 32, "fp32", (0, 2), False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_projection_parity(fp, case):
    import torch
    B, H, N, D, dtype, norms, with_bias = case
    pr = workloads.projection_inputs(B, H, N, D, dtype=dtype, seed=N + H, norms=norms)
    X, W, bias, scales = _upload(pr, with_bias)
    outs = fp.project(X, W, H, norms, bias=bias, scales=scales)
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    want = oracle.project(pr.X, pr.W, pr.bias if with_bias else None, norms, pr.scales, H)
    for p, (o, w) in enumerate(zip(outs, want)):
        got = o.float().cpu().numpy().astype(np.float64)
        assert_parity(got, w, dtype, f"output {p}")
        _bound(got, w, dtype)


def test_projection_feeds_the_mixer(fp):
    """The projection's outputs are the mixer's inputs as they stand: K, V
    and the raw synthesis keys go straight into flarepp_forward."""
    import torch
    B, H, N, D, M = 1, 8, 3000, 16, 64
    pr = workloads.projection_inputs(B, H, N, D, seed=5)
    X, W, bias, scales = _upload(pr)
    K, V, Ks = fp.project(X, W, H, pr.norms, bias=bias, scales=scales)
    wl = workloads.make(workloads.Shape(B, H, N, M, D), "bf16", "iid", seed=6)
    lat = {k: torch.from_numpy(np.ascontiguousarray(wl.bits[k]).view(np.int16)).cuda()
           .view(torch.bfloat16) for k in ("Qseed", "Qf")}
    gate = torch.from_numpy(wl.gate).cuda()
    y = fp.forward(K, V, Ks, lat["Qseed"], lat["Qf"], gate)
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    k64 = [o.float().cpu().numpy() for o in (K, V, Ks)]
    want = oracle.forward(k64[0], k64[1], k64[2], wl.Qseed, wl.Qf, wl.gate)
    assert_parity(y.float().cpu().numpy(), want["Y"], "bf16", "Y")


def test_projection_full_size_sampled(fp):
    """aero-sized projection (B=1, N=2^20, C=256): every output element is
    finite; sampled tokens (both ends and 254 in between) match the oracle."""
    import torch
    B, H, N, D = 1, 8, 1 << 20, 32
    pr = workloads.projection_inputs(B, H, N, D, seed=11)
    X, W, bias, scales = _upload(pr)
    outs = fp.project(X, W, H, pr.norms, bias=bias, scales=scales)
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 254, replace=False)]))
    want = oracle.project(pr.X[:, rows], pr.W, pr.bias, pr.norms, pr.scales, H)
    idx = torch.from_numpy(rows).cuda()
    for p, o in enumerate(outs):
        assert bool(torch.isfinite(o.float()).all())
        got = o[:, :, idx].float().cpu().numpy().astype(np.float64)
        assert_parity(got, want[p], "bf16", f"output {p} sampled")
        _bound(got, want[p], "bf16")
