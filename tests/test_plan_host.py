"""Host logic of the launch plan, without a GPU: flarepp_plan_info reports the
plan that flarepp_forward would use for given sizes and SM count. The split
passes' token splits cover every token with no empty split; the decode CTAs'
tile ranges, walked with the decode kernel's own mapping restated here, cover
every (batch, head, 128-token tile) exactly once, and no CTA spans more heads
than it keeps Q and Z for."""
import ctypes

import pytest

FIELDS = ("splits", "split_len", "latent_groups", "decode_tiles_per_cta",
          "decode_ctas_per_head", "decode_heads", "decode_ctas", "workspace_bytes")
BF16, FP32 = 0, 1

# the five workloads, the GPU parity shapes, and a few edge cases
SHAPES = [
    (1, 2, 1024, 32, 16), (4, 8, 16384, 64, 16), (2, 8, 65536, 256, 32), (32, 8, 4096, 128, 32),
    (1, 8, 1048576, 512, 32),
    (1, 2, 999, 40, 32), (2, 1, 1, 16, 16), (1, 3, 1000, 64, 16), (2, 2, 3001, 128, 32),
    (1, 2, 2500, 256, 32), (2, 2, 1537, 128, 32), (1, 1, 4097, 512, 32), (1, 2, 777, 16, 16),
    (1, 2, 129, 48, 16), (1, 1, 1, 64, 32), (1, 2, 5000, 192, 16), (1, 2, 2000, 80, 32),
    (2, 1, 1500, 144, 16), (80, 4, 100, 32, 16), (40, 4, 300, 64, 16), (4, 2, 5000, 64, 16),
    (300, 2, 130, 512, 32), (1, 1, 128, 512, 16), (7, 3, 257, 96, 32),
]


@pytest.fixture(scope="module")
def lib():
    from rank_latent_routing_gb300 import build
    lib = ctypes.CDLL(build.build())
    lib.flarepp_plan_info.argtypes = [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_int), ctypes.c_int]
    lib.flarepp_plan_info.restype = ctypes.c_int
    lib.flarepp_set_splits.argtypes = [ctypes.c_int]
    lib.flarepp_set_splits.restype = None
    return lib


def plan(lib, B, H, N, M, D, dtype=BF16, sms=152):
    arr = (ctypes.c_int * len(FIELDS))()
    rc = lib.flarepp_plan_info(B, H, N, M, D, dtype, sms, arr, len(FIELDS))
    assert rc == 0, rc
    return dict(zip(FIELDS, arr))


def decode_ranges(p, BH, n_tiles):
    """(first flattened tile, tile count) of every decode CTA, as the decode
    kernel derives them from its block index."""
    per, cph = p["decode_tiles_per_cta"], p["decode_ctas_per_head"]
    for c in range(p["decode_ctas"]):
        if cph > 0:
            hh, j = divmod(c, cph)
            g0, T = hh * n_tiles + j * per, max(0, min(per, n_tiles - j * per))
        else:
            g0 = c * per
            T = max(0, min(per, BH * n_tiles - g0))
        yield g0, T


@pytest.mark.parametrize("sms", [152, 148, 132, 7])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_decode_ranges_cover_every_tile_once(lib, shape, sms):
    B, H, N, M, D = shape
    if M % 16:
        pytest.skip("the tensor-core path (and its decode plan) needs M % 16 == 0")
    p = plan(lib, B, H, N, M, D, sms=sms)
    BH, n_tiles = B * H, -(-N // 128)
    assert 1 <= p["decode_heads"] <= 4
    assert p["decode_ctas_per_head"] == 0 or p["decode_heads"] == 1
    seen = [0] * (BH * n_tiles)
    for g0, T in decode_ranges(p, BH, n_tiles):
        assert T >= 1
        heads = (g0 % n_tiles + T - 1) // n_tiles + 1
        assert heads <= p["decode_heads"], (g0, T, heads)
        for g in range(g0, g0 + T):
            seen[g] += 1
    assert all(v == 1 for v in seen)


@pytest.mark.parametrize("dtype", [BF16, FP32])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_split_ranges_cover_the_tokens(lib, shape, dtype):
    B, H, N, M, D = shape
    if dtype == BF16 and M % 16:
        pytest.skip("bf16 needs M % 16 == 0")
    p = plan(lib, B, H, N, M, D, dtype=dtype)
    s, L = p["splits"], p["split_len"]
    assert s >= 1 and L >= 1
    assert s * L >= N > (s - 1) * L  # every token in a split, no split empty
    if dtype == BF16:
        assert L % 128 == 0
        assert p["latent_groups"] == (1 if M <= 64 else -(-M // 128))  # one 128-row latent block per CTA
    assert p["workspace_bytes"] > 0


def test_one_balanced_decode_wave_on_the_workloads(lib):
    for shape in [(4, 8, 16384, 64, 16), (2, 8, 65536, 256, 32), (32, 8, 4096, 128, 32)]:
        p = plan(lib, *shape)
        assert p["decode_ctas_per_head"] == 0 and p["decode_ctas"] == 152, (shape, p)
    # aero: two heads' Q and Z (M = 512) do not fit beside the ring; 8 heads x 19 CTAs
    p = plan(lib, 1, 8, 1048576, 512, 32)
    assert (p["decode_ctas_per_head"], p["decode_heads"], p["decode_ctas"]) == (19, 1, 152)


def test_forced_splits_reach_the_plan(lib):
    auto = plan(lib, 1, 2, 4000, 128, 32)
    try:
        lib.flarepp_set_splits(3)
        forced = plan(lib, 1, 2, 4000, 128, 32)
        assert forced["splits"] == 3 and forced["split_len"] == 11 * 128  # 32 tiles in 3 splits
    finally:
        lib.flarepp_set_splits(0)
    assert plan(lib, 1, 2, 4000, 128, 32) == auto


def test_plan_info_rejects_bad_arguments(lib):
    arr = (ctypes.c_int * 8)()
    assert lib.flarepp_plan_info(1, 1, 64, 32, 16, BF16, 152, None, 8) == 1
    assert lib.flarepp_plan_info(1, 1, 64, 32, 16, BF16, 0, arr, 8) == 1
    assert lib.flarepp_plan_info(1, 1, 64, 32, 16, BF16, 152, arr, 0) == 1
    assert lib.flarepp_plan_info(1, 1, 64, 32, 64, BF16, 152, arr, 8) == 2  # D = 64 unsupported
    assert lib.flarepp_plan_info(1, 1, 64, 24, 16, BF16, 152, arr, 8) == 2  # bf16 M % 16 != 0
