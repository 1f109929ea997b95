"""The device-side failure path, forced from the host: with the test hook
flarepp_test_fail_wait set, one barrier of the chosen pass never completes.
The kernels' bounded waits give up, the call ends within seconds, and
flarepp_sync_status reports FLAREPP_ERR_TIMEOUT; the next call on the same
context is correct. Nothing here faults, traps or waits without a bound."""
import time

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


@pytest.mark.parametrize("pass_id", [1, 2, 3], ids=["synthesis", "encode", "decode"])
def test_a_wait_that_never_completes_ends_the_call_with_a_timeout(fp, pass_id):
    import torch
    wl = workloads.make(workloads.Shape(1, 2, 1500, 64, 16), "bf16", "iid", seed=77)
    t = to_device(wl)
    args = (t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"])
    fp.test_fail_wait(pass_id)
    try:
        t0 = time.monotonic()
        fp.forward(*args)
        rc = fp.sync_status()
        elapsed = time.monotonic() - t0
    finally:
        fp.test_fail_wait(0)
    assert rc == 6, rc  # FLAREPP_ERR_TIMEOUT
    assert elapsed < 30.0, elapsed
    # the context stays usable, and the next call is correct
    y = fp.forward(*args)
    torch.cuda.synchronize()
    assert fp.sync_status() == 0
    want = oracle.forward(wl.K, wl.V, wl.Ks_raw, wl.Qseed, wl.Qf, wl.gate)["Y"]
    assert_parity(y.float().cpu().numpy(), want, "bf16", f"after a timeout in pass {pass_id}")
