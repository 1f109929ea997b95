"""Seeded synthetic inputs for the FLARE++ mixer forward.

This module only draws numbers. It holds none of the mixer's arithmetic, so
both the CPU oracle (under ``oracle/``) and the CUDA path can be fed from it
without sharing any of the method's code.

Random numbers come from a counter-based generator written out here from its
published definition: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) applied to ``key + counter``.
Uniforms take the top 53 bits; normals use the Box-Muller transform. Every
value is a pure function of (seed, stream, index), so the same workload comes
out on x86 and Arm hosts and for any chunking.

Shapes and value structure follow the five workloads of the FLARE++ paper's
experiments, as synthetic stand-ins (no dataset is used):

* ``tiny``   B=1 H=2  N=1024     M=32  D=16  fp32, i.i.d. N(0,1) tokens
* ``pde2d``  B=4 H=8  N=16384    M=64  D=16  bf16, i.i.d. N(0,1) tokens (2-D
  PDE meshes of Section 4.1, points in random order)
* ``mesh3d`` B=2 H=8  N=65536    M=256 D=32  bf16, per-head rank-8 component at
  amplitude 0.5 plus noise (3-D meshes)
* ``lra``    B=32 H=8 N=4096     M=128 D=32  bf16, rows looked up from a
  256-symbol table by uniform token ids (Long Range Arena, Section D.5)
* ``aero``   B=1 H=8  N=1048576  M=512 D=32  bf16, sin/cos of random 3-D
  points plus 0.1 N(0,1) noise (DrivAerML, Section 4.2)

Seeds Qseed and Qf are N(0,1)/sqrt(D) of shape [H, M, D]; the gate is
U(0,1) per head (already the post-sigmoid value g).

The mixer variants take two more tensors (``variant_inputs``): separate
synthesis values Vs [B, H, N, D], drawn like the other token tensors, and
FLARE's learned queries [H, M, D], N(0,1) (unit RMS rows, the magnitude of
N0(Qf) that the default mixer routes with).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

# sub-stream ids of the tensors of one workload
STREAM_K, STREAM_V, STREAM_KS, STREAM_QSEED, STREAM_QF, STREAM_GATE = 1, 2, 3, 4, 5, 6
STREAM_AUX = 7  # tokens ids, points, low-rank factors and similar structure
STREAM_VS, STREAM_QLAT = 8, 9  # separate synthesis values; FLARE's learned queries
STREAM_X, STREAM_W, STREAM_B, STREAM_A = 10, 11, 12, 13  # projection inputs and parameters
STREAM_DY = 14  # output cotangents of the backward pass

_CHUNK = 1 << 18


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function, applied in place to an array of uint64 states."""
    t = np.empty_like(z)
    np.right_shift(z, np.uint64(30), out=t)
    z ^= t
    z *= _C1
    np.right_shift(z, np.uint64(27), out=t)
    z ^= t
    z *= _C2
    np.right_shift(z, np.uint64(31), out=t)
    z ^= t
    return z


def _key(seed: int, stream: int, sub: int = 0) -> np.uint64:
    """Key of one sub-stream: two SplitMix64 rounds over (seed, stream, sub)."""
    s = np.array([(seed * 1_000_003 + stream * 7919 + sub) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    s += _GOLDEN
    return _mix(_mix(s))[0]


def uniform_bits(seed: int, stream: int, start: int, count: int, sub: int = 0) -> np.ndarray:
    """uint64 outputs number ``start .. start+count-1`` of one sub-stream."""
    key = _key(seed, stream, sub)
    z = np.arange(start, start + count, dtype=np.uint64)
    z *= _GOLDEN
    z += key
    return _mix(z)


def uniform(seed: int, stream: int, count: int, sub: int = 0, start: int = 0) -> np.ndarray:
    """Doubles in (0, 1): (top 53 bits + 0.5) / 2**53."""
    out = np.empty(count, dtype=np.float64)
    for c0 in range(0, count, _CHUNK):
        c1 = min(count, c0 + _CHUNK)
        b = uniform_bits(seed, stream, start + c0, c1 - c0, sub)
        out[c0:c1] = ((b >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    return out


def normal(seed: int, stream: int, count: int, sub: int = 0, start: int = 0) -> np.ndarray:
    """Standard normals ``start .. start+count-1`` of one sub-stream, by
    Box-Muller: elements 2i and 2i+1 share uniforms 2i and 2i+1 (``start`` even)."""
    if start % 2:
        raise ValueError("start must be even")
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        u = uniform(seed, stream, 2 * (p1 - p0), sub, start=start + 2 * p0)
        u = u.reshape(-1, 2)
        r = np.sqrt(-2.0 * np.log(u[:, 0]))
        t = (2.0 * math.pi) * u[:, 1]
        pair = np.empty((p1 - p0, 2), dtype=np.float64)
        np.multiply(r, np.cos(t), out=pair[:, 0])
        np.multiply(r, np.sin(t), out=pair[:, 1])
        pair = pair.reshape(-1)
        n0 = 2 * p0
        n1 = min(count, 2 * p1)
        out[n0:n1] = pair[: n1 - n0]
    return out


def round_to_bf16(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round to bfloat16 (nearest, ties to even).

    Returns (bits as uint16, the same values as float32). Inputs are finite.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    hi = (u >> np.uint64(16)).astype(np.uint16)
    vals = (hi.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return hi, vals


@dataclass(frozen=True)
class Shape:
    B: int
    H: int
    N: int
    M: int
    D: int

    @property
    def tokens(self) -> int:
        return self.B * self.N

    @property
    def flops(self) -> float:
        """Three token-latent attention calls, 2 matmuls of 2*N*M*D each."""
        return 12.0 * self.B * self.H * self.N * self.M * self.D


@dataclass
class Workload:
    """Inputs of one forward call, already rounded to the working dtype.

    ``K, V, Ks_raw`` are [B,H,N,D]; ``Qseed, Qf`` are [H,M,D]; ``gate`` is [H].
    Arrays hold float32 values exactly representable in ``dtype``; for bf16 the
    ``*_bits`` uint16 arrays hold the same values for upload.
    """
    name: str
    shape: Shape
    dtype: str  # "bf16" or "fp32"
    K: np.ndarray
    V: np.ndarray
    Ks_raw: np.ndarray
    Qseed: np.ndarray
    Qf: np.ndarray
    gate: np.ndarray
    bits: dict = field(default_factory=dict)
    structure: str | None = None  # value structure and seed it was drawn with
    seed: int | None = None

    def device_arrays(self) -> dict:
        """Host arrays in the layout the library takes (uint16 bits for bf16)."""
        out = {}
        for k in ("K", "V", "Ks_raw", "Qseed", "Qf"):
            out[k] = self.bits[k] if self.dtype == "bf16" else getattr(self, k)
        out["gate"] = self.gate
        return out


CONFIGS = {
    "tiny": (Shape(1, 2, 1024, 32, 16), "fp32", "iid", 1000),
    "pde2d": (Shape(4, 8, 16384, 64, 16), "bf16", "iid", 1001),
    "mesh3d": (Shape(2, 8, 65536, 256, 32), "bf16", "lowrank", 1002),
    "lra": (Shape(32, 8, 4096, 128, 32), "bf16", "vocab", 1003),
    "aero": (Shape(1, 8, 1048576, 512, 32), "bf16", "points", 1004),
}


def _tokens_iid(seed, stream, s: Shape, b: int, h: int):
    n = s.N * s.D
    return normal(seed, stream, n, start=(b * s.H + h) * n).reshape(s.N, s.D)


def _tokens_lowrank(seed, stream, s: Shape, b: int, h: int, rank=8, amp=0.5):
    noise_amp = math.sqrt(1.0 - amp * amp)
    sub = 1 + b * s.H + h
    U = normal(seed, stream, s.N * rank, sub=sub).reshape(s.N, rank)
    W = normal(seed, stream + 100, rank * s.D, sub=sub).reshape(rank, s.D) / math.sqrt(rank)
    E = normal(seed, stream + 200, s.N * s.D, sub=sub).reshape(s.N, s.D)
    return amp * (U @ W) + noise_amp * E


def _tokens_vocab(seed, stream, s: Shape, b: int, h: int, vocab=256):
    ids = (uniform_bits(seed, STREAM_AUX, b * s.N, s.N) % np.uint64(vocab)).astype(np.int64)
    table = normal(seed, stream, vocab * s.D, sub=1 + h).reshape(vocab, s.D)
    return table[ids]


def _tokens_points(seed, stream, s: Shape, b: int, h: int, noise=0.1):
    pts = uniform(seed, STREAM_AUX, s.N * 3, start=b * s.N * 3).reshape(s.N, 3)
    omega = normal(seed, stream, s.D * 3, sub=1 + h).reshape(s.D, 3) * (2.0 * math.pi)
    phi = uniform(seed, stream + 100, s.D, sub=1 + h) * (2.0 * math.pi)
    arg = pts @ omega.T + phi  # [N, D]
    val = np.empty_like(arg)
    val[:, 0::2] = np.sin(arg[:, 0::2])
    val[:, 1::2] = np.cos(arg[:, 1::2])
    eps = normal(seed, stream + 200, s.N * s.D, sub=1 + b * s.H + h).reshape(s.N, s.D)
    return math.sqrt(2.0) * val + noise * eps


_STRUCTURES = {
    "iid": _tokens_iid,
    "lowrank": _tokens_lowrank,
    "vocab": _tokens_vocab,
    "points": _tokens_points,
}


def _round(a, dtype):
    if dtype == "bf16":
        return round_to_bf16(a)
    if dtype == "fp32":
        return None, np.ascontiguousarray(a, dtype=np.float32)
    raise ValueError(dtype)


def make(shape: Shape, dtype: str = "bf16", structure: str = "iid", seed: int = 1,
         name: str = "custom", qseed_scale: float = 1.0) -> Workload:
    """Draw one workload. ``qseed_scale`` multiplies Qseed (stress inputs).

    Token tensors are drawn one (batch, head) slice at a time and rounded per
    slice, so ``make_head`` reproduces any slice without drawing the rest."""
    s = shape
    gen = _STRUCTURES[structure]
    vals, bits = {}, {}
    for k, stream in (("K", STREAM_K), ("V", STREAM_V), ("Ks_raw", STREAM_KS)):
        v = np.empty((s.B, s.H, s.N, s.D), dtype=np.float32)
        bt = np.empty((s.B, s.H, s.N, s.D), dtype=np.uint16) if dtype == "bf16" else None
        for b in range(s.B):
            for h in range(s.H):
                hb, hv = _round(gen(seed, stream, s, b, h), dtype)
                v[b, h] = hv
                if bt is not None:
                    bt[b, h] = hb
        vals[k] = v
        if bt is not None:
            bits[k] = bt
    for k, a in _latents(shape, seed, qseed_scale).items():
        hb, hv = _round(a, dtype)
        vals[k] = hv
        if hb is not None:
            bits[k] = hb
    gate = uniform(seed, STREAM_GATE, s.H).astype(np.float32)
    return Workload(name, s, dtype, vals["K"], vals["V"], vals["Ks_raw"], vals["Qseed"],
                    vals["Qf"], gate, bits, structure, seed)


def _latents(s: Shape, seed: int, qseed_scale: float = 1.0) -> dict:
    return {
        "Qseed": normal(seed, STREAM_QSEED, s.H * s.M * s.D).reshape(s.H, s.M, s.D)
        * (qseed_scale / math.sqrt(s.D)),
        "Qf": normal(seed, STREAM_QF, s.H * s.M * s.D).reshape(s.H, s.M, s.D) / math.sqrt(s.D),
    }


def make_head(name: str, b: int, h: int, **overrides) -> dict:
    """The (b, h) slice of a named workload, drawn alone: K, V, Ks_raw [N, D],
    Qseed, Qf [M, D] and the gate g (float), the same values as in ``config``."""
    shape, dtype, structure, seed = CONFIGS[name]
    dims = {k: overrides.pop(k, getattr(shape, k)) for k in ("B", "H", "N", "M", "D")}
    s = Shape(**dims)
    dtype = overrides.pop("dtype", dtype)
    seed = overrides.pop("seed", seed)
    gen = _STRUCTURES[structure]
    out = {}
    for k, stream in (("K", STREAM_K), ("V", STREAM_V), ("Ks_raw", STREAM_KS)):
        out[k] = _round(gen(seed, stream, s, b, h), dtype)[1]
    for k, a in _latents(s, seed).items():
        out[k] = _round(a, dtype)[1][h]
    out["gate"] = float(uniform(seed, STREAM_GATE, s.H).astype(np.float32)[h])
    return out


def from_arrays(name: str, shape: Shape, dtype: str, K, V, Ks_raw, Qseed, Qf, gate) -> Workload:
    """Round given arrays to ``dtype`` and wrap them as a workload."""
    vals, bits = {}, {}
    for k, a in (("K", K), ("V", V), ("Ks_raw", Ks_raw), ("Qseed", Qseed), ("Qf", Qf)):
        if dtype == "bf16":
            bits[k], vals[k] = round_to_bf16(a)
        elif dtype == "fp32":
            vals[k] = np.ascontiguousarray(a, dtype=np.float32)
        else:
            raise ValueError(dtype)
    return Workload(name, shape, dtype, vals["K"], vals["V"], vals["Ks_raw"], vals["Qseed"],
                    vals["Qf"], np.ascontiguousarray(gate, dtype=np.float32), bits)


def config(name: str, **overrides) -> Workload:
    """One of the five named workloads; ``overrides`` may change B, H, N, M, D,
    dtype or seed (smaller parity cases keep the value structure)."""
    shape, dtype, structure, seed = CONFIGS[name]
    dims = {k: overrides.pop(k, getattr(shape, k)) for k in ("B", "H", "N", "M", "D")}
    dtype = overrides.pop("dtype", dtype)
    seed = overrides.pop("seed", seed)
    return make(Shape(**dims), dtype, structure, seed, name=name, **overrides)


def variant_inputs(wl: Workload) -> dict:
    """The extra inputs of the mixer variants for workload ``wl`` (same shape,
    dtype, structure and seed): ``Vs`` [B,H,N,D] and ``Qlat`` [H,M,D] as float32
    values exactly representable in the dtype, with ``Vs_bits``/``Qlat_bits``
    (uint16) for bf16."""
    s = wl.shape
    if wl.structure is None:
        raise ValueError("variant inputs need a drawn workload (not from_arrays)")
    seed = wl.seed
    gen = _STRUCTURES[wl.structure]
    vs = np.empty((s.B, s.H, s.N, s.D), dtype=np.float32)
    vb = np.empty((s.B, s.H, s.N, s.D), dtype=np.uint16)
    for b in range(s.B):
        for h in range(s.H):
            hb, hv = _round(gen(seed, STREAM_VS, s, b, h), wl.dtype)
            vs[b, h] = hv
            if hb is not None:
                vb[b, h] = hb
    ql = normal(seed, STREAM_QLAT, s.H * s.M * s.D).reshape(s.H, s.M, s.D)
    qb, qv = _round(ql, wl.dtype)
    out = {"Vs": vs, "Qlat": qv}
    if wl.dtype == "bf16":
        out["Vs_bits"] = vb
        out["Qlat_bits"] = qb
    return out




def make_variant_head(name: str, b: int, h: int) -> dict:
    """The (b, h) slice of ``variant_inputs`` for a named workload, drawn
    alone: Vs [N, D] and the head's FLARE queries Qlat [M, D]."""
    shape, dtype, structure, seed = CONFIGS[name]
    gen = _STRUCTURES[structure]
    ql = normal(seed, STREAM_QLAT, shape.H * shape.M * shape.D).reshape(shape.H, shape.M, shape.D)
    return {"Vs": _round(gen(seed, STREAM_VS, shape, b, h), dtype)[1],
            "Qlat": _round(ql, dtype)[1][h]}


@dataclass
class Projection:
    """Inputs of the fused token projections: X [B, N, C] (C = H D), the
    stacked weights W [P*C, C] (torch Linear layout, out x in), bias [P*C]
    fp32, the per-head norm codes of the P outputs and the N_a scales [P, D]
    fp32. X and W hold values exact in ``dtype``; ``bits`` has their uint16
    patterns for bf16."""
    B: int
    H: int
    N: int
    D: int
    dtype: str
    X: np.ndarray
    W: np.ndarray
    bias: np.ndarray
    norms: tuple
    scales: np.ndarray
    bits: dict = field(default_factory=dict)


def projection_inputs(B: int, H: int, N: int, D: int, dtype: str = "bf16", seed: int = 7,
                      norms=(2, 0, 0)) -> Projection:
    """X ~ N(0,1) (a pre-normalised block input); W = I + dW per stacked
    projection with dW ~ 0.02 N(0,1) clipped at two standard deviations (the
    near-identity initialisation of the FLARE++ paper, Appendix A.5 eq. 18);
    bias ~ 0.02 N(0,1); N_a scales ~ 1 + 0.1 N(0,1). The default norms are
    those of the FLARE++ mixer's inputs: K = N_a(X W_K), V = X W_V and the raw
    synthesis keys X W~_K."""
    C = H * D
    P = len(norms)
    x = normal(seed, STREAM_X, B * N * C).reshape(B, N, C)
    dw = np.clip(normal(seed, STREAM_W, P * C * C), -2.0, 2.0).reshape(P, C, C) * 0.02
    w = (dw + np.eye(C)[None]).reshape(P * C, C)
    bias = (normal(seed, STREAM_B, P * C) * 0.02).astype(np.float32)
    scales = (1.0 + 0.1 * normal(seed, STREAM_A, P * D)).reshape(P, D).astype(np.float32)
    xb, xv = _round(x, dtype)
    wb, wv = _round(w, dtype)
    bits = {"X": xb, "W": wb} if dtype == "bf16" else {}
    return Projection(B, H, N, D, dtype, xv, wv, bias, tuple(int(n) for n in norms), scales, bits)


def cotangent(wl: Workload, seed: int = 5) -> dict:
    """An output cotangent dY ~ N(0,1) of the shape of the mixer's output,
    exact in the workload's dtype: {"dY": float32 values, "dY_bits": uint16
    (bf16 only)}."""
    s = wl.shape
    hb, hv = _round(normal(seed, STREAM_DY, s.B * s.H * s.N * s.D).reshape(s.B, s.H, s.N, s.D), wl.dtype)
    out = {"dY": hv}
    if hb is not None:
        out["dY_bits"] = hb
    return out
