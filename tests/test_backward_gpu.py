"""GPU parity of the backward pass (flarepp_backward) against the fp64
oracle's gradients (FLARE++ paper, Appendix B.5 eq. 46-49 per attention call,
the chain rule through the gate and N0), every element, on seeded inputs with
ragged token tails, N = 1, M = 1 and every latent-block layout."""
import numpy as np
import pytest

import oracle
from rank_latent_routing_gb300 import workloads
from tests.helpers import to_device

pytestmark = pytest.mark.gpu

# The forward's bars: relative L2 1e-2 for bf16 (Q and Z enter the backward
# rounded to bf16 as in the forward, relative 2^-9; the cases here measure at
# most 3.5e-3, the score cotangents dA - c partly cancelling) and 1e-5 for
# fp32 (accumulation order only; measured at most 9e-7)
REL = {"bf16": 1e-2, "fp32": 1e-5}
# absolute RMS floor, for gradients that vanish (N = 1: the output is V
# whatever K and Q are, so dK = 0 up to the cancellation in dA - c)
ATOL = {"bf16": 1e-4, "fp32": 1e-6}


@pytest.fixture(scope="module")
def fp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_latent_routing_gb300 import flarepp
    return flarepp


def _dy_device(wl, ct):
    import torch
    if wl.dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(ct["dY_bits"]).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(ct["dY"]).cuda()


CASES = [
    ("iid", 1, 2, 999, 40, 32, "fp32"),
    ("iid", 2, 1, 1, 16, 16, "fp32"),
    ("iid", 1, 1, 300, 1, 16, "fp32"),
    ("iid", 1, 3, 1000, 64, 16, "bf16"),
    ("iid", 2, 2, 3001, 128, 32, "bf16"),
    ("lowrank", 1, 2, 2500, 256, 32, "bf16"),
    ("points", 1, 1, 4097, 512, 32, "bf16"),
    ("iid", 1, 2, 129, 48, 16, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_parity(fp, case):
    import torch
    structure, B, H, N, M, D, dtype = case
    wl = workloads.make(workloads.Shape(B, H, N, M, D), dtype, structure, seed=41 + N + M)
    ct = workloads.cotangent(wl, seed=N)
    t = to_device(wl)
    got = fp.backward(t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"], _dy_device(wl, ct))
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    want = oracle.backward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate, ct["dY"])
    for key in ("dK", "dV", "dKs_raw", "dQseed", "dQf", "dgate"):
        g = got[key].cpu().numpy().astype(np.float64)
        w = np.asarray(want[key], dtype=np.float64)
        assert np.all(np.isfinite(g)), key
        err = float(np.linalg.norm(g - w))
        bound = REL[dtype] * float(np.linalg.norm(w)) + ATOL[dtype] * np.sqrt(w.size)
        assert err <= bound, f"{key}: error {err:.3e}, bound {bound:.3e}"


def test_backward_repeatable(fp):
    """Two calls give bitwise identical gradients (fixed reduction order)."""
    import torch
    wl = workloads.make(workloads.Shape(1, 2, 2000, 128, 32), "bf16", "iid", seed=3)
    ct = workloads.cotangent(wl)
    t = to_device(wl)
    dy = _dy_device(wl, ct)
    a = fp.backward(t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"], dy)
    b = fp.backward(t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"], dy)
    torch.cuda.synchronize()
    for key in a:
        assert torch.equal(a[key], b[key]), key
