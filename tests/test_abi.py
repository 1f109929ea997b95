"""The C-ABI library loads and exports every entry point of include/flarepp.h;
argument validation works without a GPU (no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    text = open(os.path.join(ROOT, "include", "flarepp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flare(?:pp)?_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from rank_latent_routing_gb300 import build
    path = build.build()
    return ctypes.CDLL(path), path


def test_header_declares_the_boundary():
    names = _header_functions()
    for want in ("flarepp_forward", "flarepp_forward_ws", "flarepp_forward_debug",
                 "flarepp_workspace_size", "flarepp_sync_status", "flarepp_status_string",
                 "flarepp_forward_variant", "flare_forward", "flarepp_project",
                 "flarepp_backward"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    _, path = lib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (flare(?:pp)?_\w+)", out))
    missing = [n for n in _header_functions() if n not in exported]
    assert not missing, missing
    for n in _header_functions():
        getattr(lib[0], n)


def test_status_strings(lib):
    l = lib[0]
    l.flarepp_status_string.restype = ctypes.c_char_p
    seen = set()
    for code in range(7):
        s = l.flarepp_status_string(code).decode()
        assert s and s not in seen
        seen.add(s)
    assert l.flarepp_status_string(99).decode() == "unknown status"


def _forward(l, ptrs, B=1, H=2, N=64, M=32, D=16, dtype=0, out=None):
    f = l.flarepp_forward
    vp = ctypes.c_void_p
    f.argtypes = [vp] * 6 + [ctypes.c_int] * 6 + [vp, vp]
    f.restype = ctypes.c_int
    return f(*ptrs, B, H, N, M, D, dtype, out, None)


def test_argument_validation_without_gpu(lib):
    l = lib[0]
    good = [0x10000 * (i + 1) for i in range(6)]
    out = 0x900000
    assert _forward(l, [None] + good[1:], out=out) == 1          # null K
    assert _forward(l, good, out=None) == 1                      # null out
    assert _forward(l, good, N=0, out=out) == 1                  # N <= 0
    assert _forward(l, good, D=64, out=out) == 2                 # D unsupported
    assert _forward(l, good, M=520, out=out) == 2                # M > 512
    assert _forward(l, good, M=40, out=out) == 2                 # bf16 needs M % 16 == 0
    assert _forward(l, good, dtype=7, out=out) == 2              # unknown dtype
    assert _forward(l, [good[0] + 8] + good[1:], out=out) == 3   # misaligned K
    assert _forward(l, good, out=good[1]) == 1                   # out aliases V


def test_workspace_size_rejects_unsupported(lib):
    l = lib[0]
    l.flarepp_workspace_size.restype = ctypes.c_size_t
    assert l.flarepp_workspace_size(1, 1, 64, 32, 64, 0) == 0
    assert l.flarepp_workspace_size(1, 1, 0, 32, 16, 0) == 0


def _variant(l, variant, K, V, Ks, Vs, Qs, Qf, gate, out, B=1, H=2, N=64, M=32, D=16, dtype=0):
    f = l.flarepp_forward_variant
    vp = ctypes.c_void_p
    f.argtypes = [ctypes.c_int] + [vp] * 7 + [ctypes.c_int] * 6 + [vp] * 5 + [vp]
    f.restype = ctypes.c_int
    return f(variant, K, V, Ks, Vs, Qs, Qf, gate, B, H, N, M, D, dtype, out, None, None, None,
             None, None)


def test_variant_argument_validation_without_gpu(lib):
    """Each variant takes exactly the inputs it reads (include/flarepp.h)."""
    l = lib[0]
    K, V, Ks, Vs, Qs, Qf, g = [0x10000 * (i + 1) for i in range(7)]
    out = 0x900000
    assert _variant(l, 3, K, V, Ks, None, Qs, Qf, g, out) == 1      # unknown variant
    assert _variant(l, 0, K, V, Ks, Vs, Qs, Qf, g, out) == 1        # shared takes no Vs
    assert _variant(l, 1, K, V, Ks, None, Qs, Qf, g, out) == 1      # unshared needs Vs
    assert _variant(l, 2, K, V, Ks, Vs, Qs, Qf, g, out) == 1        # simplified: no Qf, gate
    assert _variant(l, 2, K, V, Ks, Vs, Qs, None, g, out) == 1
    assert _variant(l, 2, K, V, None, Vs, Qs, None, None, out) == 1  # simplified needs Ks
    assert _variant(l, 1, K, V, Ks, Vs + 8, Qs, Qf, g, out) == 3    # misaligned Vs
    assert _variant(l, 1, K, V, Ks, Vs, Qs, Qf, g, Vs) == 1         # out aliases Vs
    assert _variant(l, 2, K, V, Ks, Vs, Qs, None, None, out, D=64) == 2


def test_flare_argument_validation_without_gpu(lib):
    l = lib[0]
    f = l.flare_forward
    vp = ctypes.c_void_p
    f.argtypes = [vp] * 3 + [ctypes.c_int] * 6 + [vp] * 4
    f.restype = ctypes.c_int
    Q, K, V, out = 0x10000, 0x20000, 0x30000, 0x900000

    def call(q, k, v, o, M=32, D=16):
        return f(q, k, v, 1, 2, 64, M, D, 0, o, None, None, None)

    assert call(None, K, V, out) == 1        # null Q
    assert call(Q, K, None, out) == 1        # null V
    assert call(Q + 4, K, V, out) == 3       # misaligned Q
    assert call(Q, K, V, Q) == 1             # out aliases Q
    assert call(Q, K, V, out, M=600) == 2    # M > 512


def test_project_argument_validation_without_gpu(lib):
    l = lib[0]
    f = l.flarepp_project
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, vp] + [ctypes.c_int] * 5 + [vp]
    f.restype = ctypes.c_int
    X, W, bias, sc = 0x100000, 0x200000, 0x300000, 0x400000
    outs = (ctypes.c_void_p * 3)(0x1000000, 0x2000000, 0x3000000)

    def call(norms, scales=sc, P=3, H=8, D=16, dtype=0, x=X, o=outs):
        arr = (ctypes.c_int * len(norms))(*norms)
        return f(x, W, bias, P, ctypes.cast(arr, vp), scales, ctypes.cast(o, vp), 2, H, 64, D, dtype,
                 None)

    assert call([2, 0, 0], P=0) == 1                    # P out of range
    assert call([2, 0, 0], P=5) == 1
    assert call([3, 0, 0]) == 1                         # unknown norm code
    assert call([0, 0, 0]) == 1                         # scales given but no N_a output
    assert call([2, 0, 0], scales=None) == 1            # N_a output without scales
    assert call([2, 0, 0], H=3) == 2                    # bf16 needs C in {64, 128, 256}
    assert call([2, 0, 0], D=64) == 2                   # D unsupported
    assert call([2, 0, 0], x=X + 8) == 3                # misaligned X
    assert call([2, 0, 0], x=None) == 1                 # null X
    same = (ctypes.c_void_p * 3)(0x1000000, 0x1000000, 0x3000000)
    assert call([2, 0, 0], o=same) == 1                 # outputs overlap
    onx = (ctypes.c_void_p * 3)(X, 0x2000000, 0x3000000)
    assert call([2, 0, 0], o=onx) == 1                  # output aliases X


def test_backward_argument_validation_without_gpu(lib):
    l = lib[0]
    f = l.flarepp_backward
    vp = ctypes.c_void_p
    f.argtypes = [vp] * 7 + [ctypes.c_int] * 6 + [vp] * 7
    f.restype = ctypes.c_int
    ins = [0x100000 * (i + 1) for i in range(7)]
    outs = [0x10000000 * (i + 1) for i in range(6)]

    def call(i=ins, o=outs, M=32, D=16):
        return f(*i, 1, 2, 64, M, D, 0, *o, None)

    assert call(i=[None] + ins[1:]) == 1                 # null K
    assert call(o=outs[:5] + [None]) == 1                # null dgate
    assert call(D=64) == 2                               # D unsupported
    assert call(i=ins[:6] + [ins[6] + 4]) == 3           # misaligned dY
    assert call(o=[ins[6]] + outs[1:]) == 1              # dK aliases dY
    assert call(o=[outs[0], outs[0]] + outs[2:]) == 1    # dK and dV overlap
