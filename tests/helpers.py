"""Shared test helpers: device upload of seeded workloads and error metrics."""
import numpy as np

from rank_latent_routing_gb300 import workloads

# Parity bars: bf16 relative L2 <= 1e-2 and max-abs <= 3e-2 against the fp64
# oracle; the fp32 verification build relative L2 <= 1e-5.
BF16_REL_L2 = 1e-2
BF16_MAX_ABS = 3e-2
FP32_REL_L2 = 1e-5


def to_device(wl: workloads.Workload, device="cuda"):
    import torch
    out = {}
    for k in ("K", "V", "Ks_raw", "Qseed", "Qf"):
        if wl.dtype == "bf16":
            bits = np.ascontiguousarray(wl.bits[k]).view(np.int16)
            out[k] = torch.from_numpy(bits).to(device).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(getattr(wl, k))).to(device)
    out["gate"] = torch.from_numpy(wl.gate).to(device)
    return out


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def assert_parity(got, want, dtype, what=""):
    r = rel_l2(got, want)
    if dtype == "bf16":
        m = max_abs(got, want)
        assert r <= BF16_REL_L2 and m <= BF16_MAX_ABS, f"{what}: rel-L2 {r:.3e}, max-abs {m:.3e}"
    else:
        assert r <= FP32_REL_L2, f"{what}: rel-L2 {r:.3e}"
    return r
