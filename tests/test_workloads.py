"""The seeded input generator, which feeds both the oracle and the CUDA path,
against what its recipes promise: SplitMix64 as published, in the counter
form used here; uniform and normal moments; bf16 round-to-nearest-even; the
five workloads' shapes, dtypes and seeds; and each token-value structure
(i.i.d., rank-8 component plus noise, a 256-row vocabulary, sin/cos of
random 3-D points). The generator holds none of the mixer's arithmetic, so
nothing here involves the oracle."""
import numpy as np
import pytest

from rank_latent_routing_gb300 import workloads as W

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def splitmix64(state, n):
    """Sequential SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) in plain
    integer arithmetic: state += golden gamma, then the output mix."""
    out = []
    for _ in range(n):
        state = (state + GOLDEN) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_first_outputs_from_state_zero():
    # the outputs published with the algorithm's reference code
    assert splitmix64(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_form_is_the_sequential_generator():
    # output i of a sub-stream is mix(key + i * gamma): the sequential
    # generator started from state key - gamma, and any window of it
    key = int(W._key(123, 4, 5))
    want = splitmix64((key - GOLDEN) & M64, 64)
    assert [int(v) for v in W.uniform_bits(123, 4, 0, 64, sub=5)] == want
    assert [int(v) for v in W.uniform_bits(123, 4, 17, 5, sub=5)] == want[17:22]
    # streams and sub-streams are different sequences
    assert int(W._key(123, 4, 5)) != int(W._key(123, 4, 6)) != int(W._key(123, 5, 5))


def test_uniform_and_normal_moments_and_windows():
    u = W.uniform(7, 1, 1_000_000)
    assert 0.0 < u.min() and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 2e-3 and abs(u.var() - 1.0 / 12.0) < 1e-3
    z = W.normal(7, 2, 1_000_000)
    assert abs(z.mean()) < 5e-3 and abs(z.var() - 1.0) < 1e-2
    assert abs(np.mean(z ** 4) - 3.0) < 6e-2  # a normal's fourth moment
    assert abs(np.mean(np.abs(z) < 1.0) - 0.6826894921) < 2e-3
    # the two normals of a Box-Muller pair are independent
    assert abs(np.corrcoef(z[0::2], z[1::2])[0, 1]) < 5e-3
    assert abs(np.corrcoef(z[0::2] ** 2, z[1::2] ** 2)[0, 1]) < 5e-3
    # values do not depend on how the draw is cut into windows or chunks
    assert np.array_equal(W.normal(7, 2, 10, start=300_000), z[300_000:300_010])
    assert np.array_equal(W.uniform(7, 1, 7, start=999_990), u[999_990:999_997])


def test_round_to_bf16_is_nearest_even():
    hand = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 3 * 2 ** -8),
                     0.0, -0.0, 2 ** -130, 65504.0, 1e30], dtype=np.float64)
    want = np.array([1.0, 1.0, 1 + 2 ** -6, 1 + 2 ** -7, -(1 + 2 ** -6), 0.0, -0.0, 2 ** -130,
                     65536.0, None], dtype=object)
    bits, vals = W.round_to_bf16(hand)
    for i in range(len(hand) - 1):  # ties go to the even mantissa
        assert vals[i] == np.float32(want[i]), (hand[i], vals[i])
    assert np.signbit(vals[6])
    torch = pytest.importorskip("torch")
    x = np.concatenate([hand, W.normal(3, 1, 200_000) * 10.0 ** (6 * W.uniform(3, 2, 200_000) - 3)])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bits, vals = W.round_to_bf16(x)
    assert np.array_equal(bits, ref)
    assert np.array_equal(vals.view(np.uint32) >> 16, bits.astype(np.uint32))


def test_the_five_workloads():
    want = {"tiny": ((1, 2, 1024, 32, 16), "fp32", "iid"),
            "pde2d": ((4, 8, 16384, 64, 16), "bf16", "iid"),
            "mesh3d": ((2, 8, 65536, 256, 32), "bf16", "lowrank"),
            "lra": ((32, 8, 4096, 128, 32), "bf16", "vocab"),
            "aero": ((1, 8, 1048576, 512, 32), "bf16", "points")}
    for i, name in enumerate(("tiny", "pde2d", "mesh3d", "lra", "aero")):
        shape, dtype, structure, seed = W.CONFIGS[name]
        s = (shape.B, shape.H, shape.N, shape.M, shape.D)
        assert (s, dtype, structure) == want[name] and seed == 1000 + i


def test_latents_and_gate():
    wl = W.make(W.Shape(1, 4, 64, 128, 32), "bf16", "iid", seed=11)
    for q in (wl.Qseed, wl.Qf):  # N(0, 1) / sqrt(D)
        assert q.shape == (4, 128, 32)
        assert abs(q.std() * np.sqrt(32) - 1.0) < 0.05 and abs(q.mean()) < 0.01
    assert wl.gate.shape == (4,) and np.all((wl.gate > 0) & (wl.gate < 1))
    # bf16 values are exactly the uploaded bits
    for k in ("K", "V", "Ks_raw", "Qseed", "Qf"):
        assert np.array_equal(getattr(wl, k).view(np.uint32) >> 16, wl.bits[k].astype(np.uint32))
    # the stress input scales the seeds only
    wl8 = W.make(W.Shape(1, 4, 64, 128, 32), "fp32", "iid", seed=11, qseed_scale=8.0)
    wl1 = W.make(W.Shape(1, 4, 64, 128, 32), "fp32", "iid", seed=11)
    assert np.allclose(wl8.Qseed, 8 * wl1.Qseed) and np.array_equal(wl8.K, wl1.K)


def _top_energy(X, r):
    sv = np.linalg.svd(X - X.mean(axis=0), compute_uv=False)
    return float(np.sum(sv[:r] ** 2) / np.sum(sv ** 2))


def test_lowrank_structure():
    # 0.5 U W (rank 8, entry variance 0.25) plus sqrt(0.75) noise: unit entry
    # variance, and the top 8 of 32 directions hold 0.25 + 0.75 * 8/32 of it
    s = W.Shape(1, 2, 8192, 64, 32)
    low = W.make(s, "fp32", "lowrank", seed=5)
    iid = W.make(s, "fp32", "iid", seed=5)
    X = low.K[0, 0].astype(np.float64)
    assert abs(X.var() - 1.0) < 0.05
    assert 0.40 < _top_energy(X, 8) < 0.48
    assert _top_energy(iid.K[0, 0].astype(np.float64), 8) < 0.30
    # each head has its own factors
    assert not np.allclose(low.K[0, 0], low.K[0, 1])


def test_vocab_structure():
    s = W.Shape(2, 2, 3000, 64, 16)
    wl = W.make(s, "fp32", "vocab", seed=3)
    rows, inv = np.unique(wl.K[0, 0], axis=0, return_inverse=True)
    assert len(rows) == 256  # 3000 draws from 256 symbols hit every one
    inv = inv.reshape(-1)
    # the token ids are shared by K, V and Ks_raw and by the heads of an entry
    for other in (wl.V[0, 0], wl.Ks_raw[0, 0], wl.K[0, 1]):
        _, inv2 = np.unique(other, axis=0, return_inverse=True)
        inv2 = inv2.reshape(-1)
        assert len(np.unique(np.stack([inv, inv2]), axis=1)[0]) == 256  # a bijection of symbols
    # per-head tables; different batch entries draw different ids
    assert not np.allclose(wl.K[0, 0], wl.K[0, 1])
    assert not np.array_equal(wl.K[0, 0], wl.K[1, 0])


def test_points_structure():
    s = W.Shape(1, 2, 2000, 64, 32)
    seed = 4
    wl = W.make(s, "fp32", "points", seed=seed)
    X = wl.K[0, 0].astype(np.float64)
    assert np.max(np.abs(X)) < np.sqrt(2) + 0.1 * 6
    assert abs(X.var() - 1.01) < 0.1  # sqrt(2) sin/cos has variance 1; noise 0.01
    # the values vary smoothly over the points: nearest neighbours in [0, 1]^3
    # differ far less than random pairs
    pts = W.uniform(seed, W.STREAM_AUX, s.N * 3).reshape(s.N, 3)
    d2 = ((pts[:, None, :] - pts[None, :, :]) ** 2).sum(-1)
    np.fill_diagonal(d2, np.inf)
    nn = d2.argmin(axis=1)
    near = np.mean((X - X[nn]) ** 2)
    far = np.mean((X - X[np.random.default_rng(0).permutation(s.N)]) ** 2)
    assert near < 0.6 * far


def test_a_head_drawn_alone_matches_the_full_draw():
    wl = W.config("lra", B=2, H=3, N=300, M=64)
    one = W.make_head("lra", 1, 2, B=2, H=3, N=300, M=64)
    for k in ("K", "V", "Ks_raw"):
        assert np.array_equal(one[k], getattr(wl, k)[1, 2])
    for k in ("Qseed", "Qf"):
        assert np.array_equal(one[k], getattr(wl, k)[2])
    assert one["gate"] == float(wl.gate[2])
