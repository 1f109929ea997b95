"""Python binding of the FLARE++ C-ABI library (argument marshalling only).

Every step of the mixer runs in the library's CUDA kernels; this module only
checks tensor properties, passes device pointers, sizes and the current CUDA
stream through ctypes, and turns status codes into exceptions. PyTorch is
used for device memory and streams. There is no CPU path: if the library is
not built, importing this module raises.

The names follow include/flarepp.h: ``forward``, ``forward_ws``,
``forward_debug``, ``forward_static``, ``forward_variant``, ``flare_forward``, ``project``,
``backward``,
``workspace_size``, ``sync_status``, ``status_string``, ``set_splits``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

BF16, FP32 = 0, 1
VARIANT_SHARED, VARIANT_UNSHARED, VARIANT_SIMPLIFIED = 0, 1, 2
_VARIANTS = {"shared": VARIANT_SHARED, "unshared": VARIANT_UNSHARED,
             "simplified": VARIANT_SIMPLIFIED}
_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "ALIGNMENT", 4: "NO_MEMORY",
           5: "CUDA", 6: "TIMEOUT"}


class FlareppError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = _lib.flarepp_last_error().decode() if code == 5 else status_string(code)
        super().__init__(f"{where}: FLAREPP_ERR_{_STATUS.get(code, code)} ({detail})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB):
        raise ImportError(
            f"FLARE++ CUDA library not found at {LIB}; build it first "
            "(python -m rank_latent_routing_gb300.build, or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB)
    vp, i, f32p, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
    lib.flarepp_forward.argtypes = [vp, vp, vp, vp, vp, f32p, i, i, i, i, i, i, vp, st]
    lib.flarepp_forward.restype = ctypes.c_int
    lib.flarepp_forward_ws.argtypes = [vp, vp, vp, vp, vp, f32p, i, i, i, i, i, i, vp, vp,
                                       ctypes.c_size_t, st]
    lib.flarepp_forward_ws.restype = ctypes.c_int
    lib.flarepp_forward_debug.argtypes = [vp, vp, vp, vp, vp, f32p, i, i, i, i, i, i, vp,
                                          f32p, f32p, f32p, f32p, st]
    lib.flarepp_forward_debug.restype = ctypes.c_int
    lib.flarepp_forward_static.argtypes = [vp, vp, vp, vp, vp, f32p, i, i, i, i, i, i, vp, st]
    lib.flarepp_forward_static.restype = ctypes.c_int
    lib.flarepp_forward_variant.argtypes = [i, vp, vp, vp, vp, vp, vp, f32p, i, i, i, i, i, i,
                                            vp, f32p, f32p, f32p, f32p, st]
    lib.flarepp_forward_variant.restype = ctypes.c_int
    lib.flare_forward.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp, f32p, f32p, st]
    lib.flare_forward.restype = ctypes.c_int
    lib.flarepp_project.argtypes = [vp, vp, f32p, i, vp, f32p, vp, i, i, i, i, i, st]
    lib.flarepp_project.restype = ctypes.c_int
    lib.flarepp_backward.argtypes = [vp, vp, vp, vp, vp, f32p, vp, i, i, i, i, i, i,
                                     f32p, f32p, f32p, f32p, f32p, f32p, st]
    lib.flarepp_backward.restype = ctypes.c_int
    lib.flarepp_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.flarepp_workspace_size.restype = ctypes.c_size_t
    lib.flarepp_sync_status.argtypes = [st]
    lib.flarepp_sync_status.restype = ctypes.c_int
    lib.flarepp_status_string.argtypes = [ctypes.c_int]
    lib.flarepp_status_string.restype = ctypes.c_char_p
    lib.flarepp_last_error.argtypes = []
    lib.flarepp_last_error.restype = ctypes.c_char_p
    lib.flarepp_set_splits.argtypes = [i]
    lib.flarepp_set_splits.restype = None
    lib.flarepp_set_stage_events.argtypes = [vp, i]
    lib.flarepp_set_stage_events.restype = None
    lib.flarepp_plan_info.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int), i]
    lib.flarepp_plan_info.restype = ctypes.c_int
    lib.flarepp_test_fail_wait.argtypes = [i]
    lib.flarepp_test_fail_wait.restype = None
    return lib


_lib = _load()


def status_string(code: int) -> str:
    return _lib.flarepp_status_string(int(code)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}; use torch.bfloat16 or torch.float32")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(K, V, Ks_raw, Qseed, Qf, gate):
    B, H, N, D = K.shape
    M = Qseed.shape[1]
    for name, t, shape in (("K", K, (B, H, N, D)), ("V", V, (B, H, N, D)),
                           ("Ks_raw", Ks_raw, (B, H, N, D)), ("Qseed", Qseed, (H, M, D)),
                           ("Qf", Qf, (H, M, D)), ("gate", gate, (H,))):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != K.device:
            raise ValueError(f"{name} is on {t.device}, K on {K.device}")
    if gate.dtype != torch.float32:
        raise TypeError("gate must be float32")
    code = _dtype_code(K)
    for name, t in (("V", V), ("Ks_raw", Ks_raw), ("Qseed", Qseed), ("Qf", Qf)):
        if _dtype_code(t) != code:
            raise TypeError(f"{name} dtype {t.dtype} differs from K dtype {K.dtype}")
    return B, H, N, M, D, code


def forward(K, V, Ks_raw, Qseed, Qf, gate, out=None, stream=None):
    """The FLARE++ mixer forward; returns ``out`` [B,H,N,D] (allocated if None)."""
    B, H, N, M, D, code = _check(K, V, Ks_raw, Qseed, Qf, gate)
    _check_tensors(K, [("out", out, (B, H, N, D), False)])
    if out is None:
        out = torch.empty_like(K)
    with torch.cuda.device(K.device):
        rc = _lib.flarepp_forward(_ptr(K), _ptr(V), _ptr(Ks_raw), _ptr(Qseed), _ptr(Qf),
                                  _ptr(gate), B, H, N, M, D, code, _ptr(out), _stream(stream))
    if rc:
        raise FlareppError(rc, "flarepp_forward")
    return out


def workspace_size(B, H, N, M, D, dtype=torch.bfloat16, device=None) -> int:
    code = BF16 if dtype == torch.bfloat16 else FP32
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(_lib.flarepp_workspace_size(B, H, N, M, D, code))


def forward_ws(K, V, Ks_raw, Qseed, Qf, gate, workspace, out=None, stream=None):
    """As ``forward`` with a caller-owned workspace (uint8 CUDA tensor)."""
    B, H, N, M, D, code = _check(K, V, Ks_raw, Qseed, Qf, gate)
    _check_tensors(K, [("out", out, (B, H, N, D), False)])
    if out is None:
        out = torch.empty_like(K)
    with torch.cuda.device(K.device):
        rc = _lib.flarepp_forward_ws(_ptr(K), _ptr(V), _ptr(Ks_raw), _ptr(Qseed), _ptr(Qf),
                                     _ptr(gate), B, H, N, M, D, code, _ptr(out), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    if rc:
        raise FlareppError(rc, "flarepp_forward_ws")
    return out


def forward_static(K, V, Ks_raw, Qseed, Qf, gate, out, stream=None):
    """As ``forward``, for callers that cannot allocate device memory: scratch
    comes from a fixed 32 MiB array inside the library and ``out`` must be
    given. Calls that overlap on the GPU share that array and race."""
    B, H, N, M, D, code = _check(K, V, Ks_raw, Qseed, Qf, gate)
    if out is None:
        raise ValueError("forward_static writes into a caller-given out (it allocates nothing)")
    _check_tensors(K, [("out", out, (B, H, N, D), False)])
    with torch.cuda.device(K.device):
        rc = _lib.flarepp_forward_static(_ptr(K), _ptr(V), _ptr(Ks_raw), _ptr(Qseed), _ptr(Qf),
                                         _ptr(gate), B, H, N, M, D, code, _ptr(out),
                                         _stream(stream))
    if rc:
        raise FlareppError(rc, "flarepp_forward_static")
    return out


def forward_debug(K, V, Ks_raw, Qseed, Qf, gate, stream=None) -> dict:
    """The forward plus the intermediate results Qd, Q, Z (fp32 [B,H,M,D]) and
    L (fp32 [B,H,M]); returns a dict with those and ``Y``."""
    B, H, N, M, D, code = _check(K, V, Ks_raw, Qseed, Qf, gate)
    out = torch.empty_like(K)
    f = dict(device=K.device, dtype=torch.float32)
    res = {"Qd": torch.empty(B, H, M, D, **f), "Q": torch.empty(B, H, M, D, **f),
           "Z": torch.empty(B, H, M, D, **f), "L": torch.empty(B, H, M, **f)}
    with torch.cuda.device(K.device):
        rc = _lib.flarepp_forward_debug(_ptr(K), _ptr(V), _ptr(Ks_raw), _ptr(Qseed), _ptr(Qf),
                                        _ptr(gate), B, H, N, M, D, code, _ptr(out),
                                        _ptr(res["Qd"]), _ptr(res["Q"]), _ptr(res["Z"]),
                                        _ptr(res["L"]), _stream(stream))
    if rc:
        raise FlareppError(rc, "flarepp_forward_debug")
    res["Y"] = out
    return res


def _check_tensors(ref, named):
    code = _dtype_code(ref)
    for name, t, shape, float_only in named:
        if t is None:
            continue
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
        if not t.is_cuda or t.device != ref.device:
            raise ValueError(f"{name} must be a CUDA tensor on {ref.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if float_only:
            if t.dtype != torch.float32:
                raise TypeError(f"{name} must be float32")
        elif _dtype_code(t) != code:
            raise TypeError(f"{name} dtype {t.dtype} differs from K dtype {ref.dtype}")
    return code


def forward_variant(variant, K, V, Ks, Vs, Qseed, Qf=None, gate=None, out=None, stream=None,
                    debug=False):
    """One of the mixer variants of include/flarepp.h: ``variant`` is
    "shared" (the default mixer), "unshared" (separate synthesis values Vs)
    or "simplified" (Q = SDPA(Qseed, Ks, Vs), no reference and no gate: pass
    Qf = gate = None). Returns ``Y`` [B,H,N,D], or with ``debug`` a dict of Y and
    the fp32 intermediates Q, Z, L (and Qd except for "simplified"). ``out`` is
    allocated if None."""
    code_v = _VARIANTS[variant] if isinstance(variant, str) else int(variant)
    B, H, N, D = K.shape
    M = Qseed.shape[1]
    code = _check_tensors(K, [("V", V, (B, H, N, D), False), ("Ks", Ks, (B, H, N, D), False),
                              ("Vs", Vs, (B, H, N, D), False), ("Qseed", Qseed, (H, M, D), False),
                              ("Qf", Qf, (H, M, D), False), ("gate", gate, (H,), True),
                              ("out", out, (B, H, N, D), False)])
    if out is None:
        out = torch.empty_like(K)
    res = {}
    if debug:
        f = dict(device=K.device, dtype=torch.float32)
        res = {"Q": torch.empty(B, H, M, D, **f), "Z": torch.empty(B, H, M, D, **f),
               "L": torch.empty(B, H, M, **f)}
        if code_v != VARIANT_SIMPLIFIED:
            res["Qd"] = torch.empty(B, H, M, D, **f)
    with torch.cuda.device(K.device):
        rc = _lib.flarepp_forward_variant(code_v, _ptr(K), _ptr(V), _ptr(Ks), _ptr(Vs),
                                          _ptr(Qseed), _ptr(Qf), _ptr(gate), B, H, N, M, D, code,
                                          _ptr(out), _ptr(res.get("Qd")), _ptr(res.get("Q")),
                                          _ptr(res.get("Z")), _ptr(res.get("L")), _stream(stream))
    if rc:
        raise FlareppError(rc, "flarepp_forward_variant")
    if not debug:
        return out
    res["Y"] = out
    return res


def flare_forward(Q, K, V, out=None, stream=None, debug=False):
    """FLARE (fixed learned queries Q [H,M,D]): Z = SDPA(Q_h, K, V),
    Y = SDPA(K, Q_h, Z). Returns ``Y`` [B,H,N,D], or with ``debug`` a dict of Y
    and the fp32 Z [B,H,M,D] and L [B,H,M]. ``out`` is allocated if None."""
    B, H, N, D = K.shape
    M = Q.shape[1]
    code = _check_tensors(K, [("V", V, (B, H, N, D), False), ("Q", Q, (H, M, D), False),
                              ("out", out, (B, H, N, D), False)])
    if out is None:
        out = torch.empty_like(K)
    res = {}
    if debug:
        f = dict(device=K.device, dtype=torch.float32)
        res = {"Z": torch.empty(B, H, M, D, **f), "L": torch.empty(B, H, M, **f)}
    with torch.cuda.device(K.device):
        rc = _lib.flare_forward(_ptr(Q), _ptr(K), _ptr(V), B, H, N, M, D, code, _ptr(out),
                                _ptr(res.get("Z")), _ptr(res.get("L")), _stream(stream))
    if rc:
        raise FlareppError(rc, "flare_forward")
    if not debug:
        return out
    res["Y"] = out
    return res


def backward(K, V, Ks_raw, Qseed, Qf, gate, dY, stream=None) -> dict:
    """Gradients of the mixer for the output cotangent dY [B,H,N,D]: a dict
    of fp32 tensors dK, dV, dKs_raw [B,H,N,D], dQseed, dQf [H,M,D] and dgate
    [H] (include/flarepp.h ``flarepp_backward``)."""
    B, H, N, M, D, code = _check(K, V, Ks_raw, Qseed, Qf, gate)
    _check_tensors(K, [("dY", dY, (B, H, N, D), False)])
    f = dict(device=K.device, dtype=torch.float32)
    g = {"dK": torch.empty(B, H, N, D, **f), "dV": torch.empty(B, H, N, D, **f),
         "dKs_raw": torch.empty(B, H, N, D, **f), "dQseed": torch.empty(H, M, D, **f),
         "dQf": torch.empty(H, M, D, **f), "dgate": torch.empty(H, **f)}
    with torch.cuda.device(K.device):
        rc = _lib.flarepp_backward(_ptr(K), _ptr(V), _ptr(Ks_raw), _ptr(Qseed), _ptr(Qf),
                                   _ptr(gate), _ptr(dY), B, H, N, M, D, code, _ptr(g["dK"]),
                                   _ptr(g["dV"]), _ptr(g["dKs_raw"]), _ptr(g["dQseed"]),
                                   _ptr(g["dQf"]), _ptr(g["dgate"]), _stream(stream))
    if rc:
        raise FlareppError(rc, "flarepp_backward")
    return g


NORM_NONE, NORM_N0, NORM_NA = 0, 1, 2
_NORMS = {"none": NORM_NONE, "n0": NORM_N0, "na": NORM_NA}


def project(X, W, H, norms, bias=None, scales=None, outs=None, stream=None):
    """Fused token projections (include/flarepp.h ``flarepp_project``).

    X [B,N,C], W [P*C, C] (stacked, out x in), ``norms`` P codes or names
    ("none", "n0", "na"), bias [P*C] fp32 or None, scales [P,D] fp32 or None.
    Returns the P outputs [B,H,N,D] (allocated unless ``outs`` is given)."""
    B, N, C = X.shape
    if C % H:
        raise ValueError(f"C={C} is not a multiple of H={H}")
    D = C // H
    P = len(norms)
    codes = [_NORMS[n] if isinstance(n, str) else int(n) for n in norms]
    code = _check_tensors(X, [("W", W, (P * C, C), False), ("bias", bias, (P * C,), True),
                              ("scales", scales, (P, D), True)])
    if outs is None:
        outs = [torch.empty(B, H, N, D, dtype=X.dtype, device=X.device) for _ in range(P)]
    for k, o in enumerate(outs):
        _check_tensors(X, [(f"outs[{k}]", o, (B, H, N, D), False)])
    norm_arr = (ctypes.c_int * P)(*codes)
    out_arr = (ctypes.c_void_p * P)(*[o.data_ptr() for o in outs])
    with torch.cuda.device(X.device):
        rc = _lib.flarepp_project(_ptr(X), _ptr(W), _ptr(bias), P,
                                  ctypes.cast(norm_arr, ctypes.c_void_p), _ptr(scales),
                                  ctypes.cast(out_arr, ctypes.c_void_p), B, H, N, D, code,
                                  _stream(stream))
    if rc:
        raise FlareppError(rc, "flarepp_project")
    return outs


def sync_status(stream=None) -> int:
    """Waits for the stream; returns the library status code (0 = OK)."""
    return int(_lib.flarepp_sync_status(_stream(stream)))


def set_splits(splits: int) -> None:
    """Test hook: force the token split count (0 = automatic)."""
    _lib.flarepp_set_splits(int(splits))


def test_fail_wait(pass_id: int) -> None:
    """Test hook: make one barrier of pass 1 (synthesis), 2 (encode) or 3
    (decode) of the next bf16 forward calls never complete, so that the call
    ends with a recorded timeout; 0 switches it off."""
    _lib.flarepp_test_fail_wait(int(pass_id))


PLAN_FIELDS = ("splits", "split_len", "latent_groups", "decode_tiles_per_cta",
               "decode_ctas_per_head", "decode_heads", "decode_ctas", "workspace_bytes")


def plan_info(B, H, N, M, D, dtype=torch.bfloat16, sms=152) -> dict:
    """The launch plan of a forward call for these sizes on a GPU with ``sms``
    multiprocessors, computed on the host (no device needed)."""
    code = BF16 if dtype == torch.bfloat16 else FP32
    arr = (ctypes.c_int * len(PLAN_FIELDS))()
    rc = _lib.flarepp_plan_info(B, H, N, M, D, code, int(sms), arr, len(PLAN_FIELDS))
    if rc:
        raise FlareppError(rc, "flarepp_plan_info")
    return dict(zip(PLAN_FIELDS, arr))


class StageTimer:
    """Device time of the three passes of each forward call (synthesis,
    encode, decode), from CUDA events the library records on the call's
    stream. Use as a context manager around one call at a time."""

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in self.events:  # torch creates the CUDA event on first record
            e.record()
        handles = [e.cuda_event for e in self.events]
        if not all(handles):
            raise RuntimeError("CUDA events were not created")
        self._arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(h) for h in handles])

    def __enter__(self):
        _lib.flarepp_set_stage_events(ctypes.cast(self._arr, ctypes.c_void_p), 4)
        return self

    def __exit__(self, *exc):
        _lib.flarepp_set_stage_events(None, 0)
        return False

    def elapsed_ms(self):
        """[synthesis, encode, decode] milliseconds of the last call (synchronises)."""
        self.events[3].synchronize()
        return [self.events[i].elapsed_time(self.events[i + 1]) for i in range(3)]


def raw_call(name: str, *args):
    """Calls a C-ABI function by name with raw ctypes arguments (tests only)."""
    return getattr(_lib, name)(*args)
