"""The allocation-free entry point, flarepp_forward_static, called through the
C ABI: its output must match flarepp_forward's on the same inputs, on two
calls in a row with different inputs (its fixed scratch keeps the previous
call's contents), and it must refuse sizes whose scratch exceeds its fixed
maximum. Collected last so a failure here leaves the rest of the suite run."""
import pytest

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


def test_static_scratch_matches_allocating_entry_point(fp):
    import torch
    cases = [(workloads.Shape(2, 3, 3001, 128, 32), "bf16", 31),
             (workloads.Shape(4, 2, 5000, 64, 16), "bf16", 32)]
    for shape, dtype, seed in cases:  # two calls in a row, different inputs and sizes
        wl = workloads.make(shape, dtype, "iid", seed=seed)
        t = to_device(wl)
        ref = fp.forward(t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"])
        out = torch.full_like(ref, float("nan"))
        fp.forward_static(t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"], out)
        torch.cuda.synchronize()
        assert fp.sync_status() == 0
        assert_parity(out.float().cpu().numpy(), ref.float().cpu().numpy(), dtype,
                      f"static vs allocating {shape}")


def test_static_scratch_rejects_oversize(fp):
    import torch
    B, H, N, M, D = 1024, 1, 1024, 512, 32
    assert fp.workspace_size(B, H, N, M, D) > 32 << 20
    big = dict(device="cuda", dtype=torch.bfloat16)
    K = torch.zeros(B, H, N, D, **big)
    lat = torch.zeros(H, M, D, **big)
    gate = torch.zeros(H, device="cuda")
    out = torch.empty_like(K)
    with pytest.raises(fp.FlareppError) as err:
        fp.forward_static(K, K.clone(), K.clone(), lat, lat.clone(), gate, out)
    assert err.value.code == 4  # FLAREPP_ERR_NO_MEMORY
