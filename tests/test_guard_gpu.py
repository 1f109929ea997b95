"""Bounds checks in place of a memory sanitizer: every buffer a call writes
(the output, the caller's workspace, the fp32 intermediates, the projection
outputs) is carved out of a larger allocation whose bytes before and after it
hold a sentinel pattern. After the call, every guard byte must still hold the
pattern, so no TMA store past the last token, no merge row past M and no
partial-result write past the workspace leaves its tensor. Shapes cover ragged
N, N = 1, M below, between and above multiples of 128, D in {16, 32}, both
dtypes and every pass kind (the default mixer, the two synthesis variants,
FLARE), plus the fused projections."""
import numpy as np
import pytest

from rank_latent_routing_gb300 import workloads
from tests.helpers import to_device

pytestmark = pytest.mark.gpu

GUARD = 1 << 16  # bytes of sentinel on each side
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def fp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_latent_routing_gb300 import flarepp
    return flarepp


class Guarded:
    """A tensor of `shape` and `dtype` at byte offset GUARD of a sentinel-filled
    buffer (256-byte aligned), with GUARD sentinel bytes after it."""

    def __init__(self, shape, dtype, fill=SENTINEL):
        import torch
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), fill, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        import torch
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        return bool(torch.all(head == SENTINEL)) and bool(torch.all(tail == SENTINEL))


# (B, H, N, M, D, dtype)
SHAPES = [
    (1, 2, 1000, 48, 16, "bf16"),   # ragged N, M <= 64 (two token streams per slot)
    (2, 1, 777, 144, 32, "bf16"),   # M between 128 and 256, ragged N
    (1, 2, 300, 272, 32, "bf16"),   # M above 256: a pair of latent blocks and a single one
    (1, 1, 1, 16, 16, "bf16"),      # one token
    (1, 1, 4097, 512, 32, "bf16"),  # the largest M, a one-token tail
    (2, 2, 333, 40, 16, "fp32"),
    (1, 1, 1, 7, 32, "fp32"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_forward_ws_writes_only_its_output_and_workspace(fp, shape):
    import torch
    B, H, N, M, D, dtype = shape
    wl = workloads.make(workloads.Shape(B, H, N, M, D), dtype, "iid", seed=404)
    t = to_device(wl)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ws_bytes = fp.workspace_size(B, H, N, M, D, tdt)
    out = Guarded((B, H, N, D), tdt)
    ws = Guarded((ws_bytes,), torch.uint8, fill=0x5A)
    ws.buf[:GUARD].fill_(SENTINEL)
    ws.buf[GUARD + ws_bytes:].fill_(SENTINEL)
    fp.forward_ws(t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"], ws.t, out=out.t)
    assert fp.sync_status() == 0
    assert out.intact(), "a write landed outside out"
    assert ws.intact(), "a write landed outside the workspace"
    assert torch.isfinite(out.t.float()).all()


@pytest.mark.parametrize("shape", SHAPES[:5], ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("variant", ["unshared", "simplified", "flare"])
def test_variants_write_only_their_outputs(fp, shape, variant):
    import torch
    B, H, N, M, D, dtype = shape
    wl = workloads.make(workloads.Shape(B, H, N, M, D), dtype, "iid", seed=405)
    t = to_device(wl)
    ex = workloads.variant_inputs(wl)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def dev(name):
        bits = np.ascontiguousarray(ex[name + "_bits"]).view(np.int16)
        return torch.from_numpy(bits).cuda().view(torch.bfloat16)

    out = Guarded((B, H, N, D), tdt)
    f32 = torch.float32
    dbg = {"Qd": Guarded((B, H, M, D), f32), "Q": Guarded((B, H, M, D), f32),
           "Z": Guarded((B, H, M, D), f32), "L": Guarded((B, H, M), f32)}
    if variant == "flare":
        rc = fp.raw_call("flare_forward", fp._ptr(dev("Qlat")), fp._ptr(t["K"]), fp._ptr(t["V"]),
                         B, H, N, M, D, fp.BF16, fp._ptr(out.t), fp._ptr(dbg["Z"].t),
                         fp._ptr(dbg["L"].t), fp._stream())
        used = ("Z", "L")
    else:
        code = fp.VARIANT_UNSHARED if variant == "unshared" else fp.VARIANT_SIMPLIFIED
        qf = None if variant == "simplified" else t["Qf"]
        gate = None if variant == "simplified" else t["gate"]
        qd = None if variant == "simplified" else dbg["Qd"].t
        rc = fp.raw_call("flarepp_forward_variant", code, fp._ptr(t["K"]), fp._ptr(t["V"]),
                         fp._ptr(t["Ks_raw"]), fp._ptr(dev("Vs")), fp._ptr(t["Qseed"]), fp._ptr(qf),
                         fp._ptr(gate), B, H, N, M, D, fp.BF16, fp._ptr(out.t), fp._ptr(qd),
                         fp._ptr(dbg["Q"].t), fp._ptr(dbg["Z"].t), fp._ptr(dbg["L"].t), fp._stream())
        used = ("Q", "Z", "L") + (() if variant == "simplified" else ("Qd",))
    assert rc == 0, fp.status_string(rc)
    assert fp.sync_status() == 0
    assert out.intact(), "a write landed outside out"
    for k in used:
        assert dbg[k].intact(), f"a write landed outside {k}"
    for k in set(dbg) - set(used):
        assert bool(torch.all(dbg[k].buf == SENTINEL)), f"{k} was not requested but written"


# (B, H, N, D, P): ragged tails, C = H D in {64, 128, 256}
PROJ = [(2, 8, 1000, 16, 3), (1, 8, 4097, 32, 3), (1, 4, 1, 16, 2), (3, 2, 129, 32, 4)]


@pytest.mark.parametrize("case", PROJ, ids=lambda c: "-".join(map(str, c)))
def test_projection_writes_only_its_outputs(fp, case):
    import torch
    B, H, N, D, P = case
    norms = (2, 0, 1, 0)[:P]
    pr = workloads.projection_inputs(B, H, N, D, dtype="bf16", seed=9, norms=norms)
    X = torch.from_numpy(np.ascontiguousarray(pr.bits["X"]).view(np.int16)).cuda().view(torch.bfloat16)
    W = torch.from_numpy(np.ascontiguousarray(pr.bits["W"]).view(np.int16)).cuda().view(torch.bfloat16)
    bias = torch.from_numpy(pr.bias).cuda()
    scales = torch.from_numpy(pr.scales).cuda()
    outs = [Guarded((B, H, N, D), torch.bfloat16) for _ in range(P)]
    fp.project(X, W, H, list(norms), bias=bias, scales=scales, outs=[o.t for o in outs])
    assert fp.sync_status() == 0
    for i, o in enumerate(outs):
        assert o.intact(), f"a write landed outside output {i}"


def test_binding_refuses_a_mismatched_out(fp):
    import torch
    wl = workloads.make(workloads.Shape(1, 2, 256, 32, 16), "bf16", "iid", seed=406)
    t = to_device(wl)
    args = (t["K"], t["V"], t["Ks_raw"], t["Qseed"], t["Qf"], t["gate"])
    bad = [torch.empty(1, 2, 255, 16, dtype=torch.bfloat16, device="cuda"),     # shape
           torch.empty(1, 2, 256, 16, dtype=torch.float32, device="cuda"),      # dtype
           torch.empty(1, 2, 16, 256, dtype=torch.bfloat16, device="cuda").transpose(2, 3),  # layout
           torch.empty(1, 2, 256, 16, dtype=torch.bfloat16)]                    # host memory
    for o in bad:
        for call in (fp.forward, fp.forward_static):
            with pytest.raises((ValueError, TypeError)):
                call(*args, out=o)
    with pytest.raises(ValueError):
        fp.forward_static(*args, out=None)
