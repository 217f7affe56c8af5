"""Python access to the CPU oracle (TEST INFRASTRUCTURE ONLY).

The oracle is the plain single-threaded C++ statement of the MoE layer in
``oracle/oracle.cpp``.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  It never imports the CUDA library
and the CUDA library never imports it.

``MOE_ORACLE_LIB``, when set, names another build of the oracle's source to
load instead; the test that plants mistakes in the oracle uses it to run the
pins against each altered copy.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None

_f32p = C.POINTER(C.c_float)
_f64p = C.POINTER(C.c_double)
_i32p = C.POINTER(C.c_int32)
_u8p = C.POINTER(C.c_uint8)
_u16p = C.POINTER(C.c_uint16)


class _Layer(C.Structure):
    _fields_ = [
        ("hidden", C.c_int), ("inter", C.c_int), ("n_experts", C.c_int),
        ("top_k", C.c_int), ("n_group", C.c_int), ("topk_group", C.c_int),
        ("rsf", C.c_float), ("n_shared", C.c_int), ("shared_inter", C.c_int),
        ("router_w", _f32p), ("router_b", _f32p),
        ("gate_q", C.POINTER(_u8p)), ("gate_s", C.POINTER(_u16p)),
        ("up_q", C.POINTER(_u8p)), ("up_s", C.POINTER(_u16p)),
        ("down_q", C.POINTER(_u8p)), ("down_s", C.POINTER(_u16p)),
        ("sh_gate_q", _u8p), ("sh_gate_s", _u16p),
        ("sh_up_q", _u8p), ("sh_up_s", _u16p),
        ("sh_down_q", _u8p), ("sh_down_s", _u16p),
        ("wfmt", C.c_int), ("gsz", C.c_int),
    ]


# weight formats of the oracle (R22)
FMT_INT4, FMT_INT8 = 0, 1


def shape_format(shape) -> tuple[int, int]:
    """(fmt, gsz) of a layer shape: its weight format and scale group."""
    fmt = FMT_INT8 if getattr(shape, "weight_format", "int4") == "int8" else FMT_INT4
    return fmt, int(getattr(shape, "group_size", 32))


def lib():
    global _lib
    if _lib is None:
        path = os.environ.get("MOE_ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        L.oracle_router_exp.restype = C.c_float
        L.oracle_router_exp.argtypes = [C.c_float]
        L.oracle_router_sigmoid.restype = C.c_float
        L.oracle_router_sigmoid.argtypes = [C.c_float]
        L.oracle_half_to_float.restype = C.c_float
        L.oracle_half_to_float.argtypes = [C.c_uint16]
        L.oracle_dequant.restype = C.c_float
        L.oracle_dequant.argtypes = [_u8p, _u16p, C.c_int]
        L.oracle_router_logits.argtypes = [_f32p, C.c_int, C.c_int, _f32p, C.c_int, _f32p]
        L.oracle_select.argtypes = [_f32p, _f32p, C.c_int, C.c_int, C.c_int, C.c_int,
                                    C.c_int, C.c_float, _i32p, _f32p]
        L.oracle_plan.argtypes = [_i32p, C.c_int, C.c_int, C.c_int, _i32p, _i32p, _i32p,
                                  _i32p, _i32p]
        L.oracle_rmsnorm.argtypes = [_f32p, C.c_int, C.c_int, _f32p, C.c_double, _f32p]
        L.oracle_expert.argtypes = [_f32p, C.c_int, C.c_int, _u8p, _u16p, _u8p, _u16p,
                                    _u8p, _u16p, C.c_int, _f64p]
        L.oracle_dequant_fmt.restype = C.c_float
        L.oracle_dequant_fmt.argtypes = [_u8p, _u16p, C.c_int, C.c_int, C.c_int]
        L.oracle_expert_fmt.argtypes = [_f32p, C.c_int, C.c_int, C.c_int, C.c_int, _u8p, _u16p,
                                        _u8p, _u16p, _u8p, _u16p, C.c_int, _f64p]
        L.oracle_moe_forward.argtypes = [C.POINTER(_Layer), _f32p, C.c_int, C.c_double,
                                         _f32p, _f32p, C.c_int, _i32p, _f32p, _f32p, _f32p]
        _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(t)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def router_exp(t: float) -> float:
    return float(lib().oracle_router_exp(C.c_float(t)))


def router_sigmoid(z: float) -> float:
    return float(lib().oracle_router_sigmoid(C.c_float(z)))


def half_to_float(h: int) -> float:
    return float(lib().oracle_half_to_float(C.c_uint16(h)))


def dequant(row_q: np.ndarray, row_s: np.ndarray, k: int) -> float:
    row_q = np.ascontiguousarray(row_q, dtype=np.uint8)
    row_s = np.ascontiguousarray(row_s, dtype=np.uint16)
    return float(lib().oracle_dequant(_p(row_q, _u8p), _p(row_s, _u16p), k))


def dequant_fmt(row_q: np.ndarray, row_s: np.ndarray, k: int, fmt: int, gsz: int) -> float:
    """Element k of one row in weight format fmt and scale group gsz (R22)."""
    row_q = np.ascontiguousarray(row_q, dtype=np.uint8)
    row_s = np.ascontiguousarray(row_s, dtype=np.uint16)
    return float(lib().oracle_dequant_fmt(_p(row_q, _u8p), _p(row_s, _u16p), k, fmt, gsz))


def router_logits(x: np.ndarray, Wr: np.ndarray) -> np.ndarray:
    x, Wr = _f32(x), _f32(Wr)
    T, H = x.shape
    E = Wr.shape[0]
    out = np.empty((T, E), np.float32)
    rc = lib().oracle_router_logits(_p(x, _f32p), T, H, _p(Wr, _f32p), E, _p(out, _f32p))
    if rc:
        raise ValueError("oracle_router_logits: bad shape")
    return out


def select(logits, bias, k, n_group, topk_group, rsf):
    logits, bias = _f32(logits), _f32(bias)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    rc = lib().oracle_select(_p(logits, _f32p), _p(bias, _f32p), T, E, k, n_group,
                             topk_group, C.c_float(rsf), _p(ids, _i32p), _p(w, _f32p))
    if rc:
        raise ValueError("oracle_select: bad configuration")
    return ids, w


def plan(ids: np.ndarray, E: int) -> dict:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    active = np.zeros(E, np.int32)
    na = np.zeros(1, np.int32)
    rc = lib().oracle_plan(_p(ids, _i32p), T, k, E, _p(counts, _i32p), _p(offsets, _i32p),
                           _p(perm, _i32p), _p(active, _i32p), _p(na, _i32p))
    if rc:
        raise ValueError("oracle_plan: expert id out of range")
    return {"counts": counts, "offsets": offsets, "perm": perm,
            "active": active[: int(na[0])].copy(), "n_active": int(na[0])}


def rmsnorm(h: np.ndarray, gamma=None, eps: float = 1e-5) -> np.ndarray:
    h = _f32(h)
    T, H = h.shape
    out = np.empty_like(h)
    g = None if gamma is None else _f32(gamma)
    gp = _p(g, _f32p) if g is not None else None
    if lib().oracle_rmsnorm(_p(h, _f32p), T, H, gp, C.c_double(eps), _p(out, _f32p)):
        raise ValueError("oracle_rmsnorm: bad shape")
    return out


def expert(x: np.ndarray, inter: int, mats, prec: int = 0) -> np.ndarray:
    """One expert's SwiGLU on one token; mats = (gq, gs, uq, us, dq, ds)."""
    x = _f32(x).reshape(-1)
    H = x.shape[0]
    gq, gs, uq, us, dq, ds = [np.ascontiguousarray(m) for m in mats]
    out = np.empty(H, np.float64)
    rc = lib().oracle_expert(_p(x, _f32p), H, inter, _p(gq, _u8p), _p(gs, _u16p),
                             _p(uq, _u8p), _p(us, _u16p), _p(dq, _u8p), _p(ds, _u16p),
                             prec, _p(out, _f64p))
    if rc:
        raise ValueError("oracle_expert: bad shape")
    return out


def expert_fmt(x: np.ndarray, inter: int, mats, fmt: int, gsz: int,
               prec: int = 0) -> np.ndarray:
    """One expert of weight format fmt and scale group gsz (R22) on one token."""
    x = _f32(x).reshape(-1)
    H = x.shape[0]
    gq, gs, uq, us, dq, ds = [np.ascontiguousarray(m) for m in mats]
    out = np.empty(H, np.float64)
    rc = lib().oracle_expert_fmt(_p(x, _f32p), H, inter, fmt, gsz, _p(gq, _u8p), _p(gs, _u16p),
                                 _p(uq, _u8p), _p(us, _u16p), _p(dq, _u8p), _p(ds, _u16p),
                                 prec, _p(out, _f64p))
    if rc:
        raise ValueError("oracle_expert_fmt: bad shape or format")
    return out


def route(shape, router_w, router_b, x, eps: float = 0.0, gamma=None):
    """(x_hat, logits, ids, w) for activations x [T, H] (fp32 view)."""
    x = _f32(x)
    xh = rmsnorm(x, gamma, eps) if eps > 0 else x
    lg = router_logits(xh, router_w)
    ids, w = select(lg, router_b, shape.top_k, shape.n_group, shape.topk_group,
                    shape.routed_scaling_factor)
    return xh, lg, ids, w


def moe_forward(shape, router_w, router_b, get_expert, shared, x, eps: float = 0.0,
                gamma=None, resid=None, prec: int = 0):
    """Full layer on x [T, H]; returns (y, ids, w, logits).

    ``get_expert(e)`` returns the six host arrays of routed expert e;
    ``shared`` the six arrays of the shared expert (or None).  Only the
    experts the router selects are requested.
    """
    x = _f32(x)
    T, H = x.shape
    E = shape.n_experts
    _, _, ids0, _ = route(shape, router_w, router_b, x, eps, gamma)
    keep = []
    tabs = [(C.POINTER(C.c_uint8) * E)() if i % 2 == 0 else (C.POINTER(C.c_uint16) * E)()
            for i in range(6)]
    for e in sorted(set(int(v) for v in ids0.reshape(-1))):
        mats = [np.ascontiguousarray(m) for m in get_expert(e)]
        keep.append(mats)
        for i, m in enumerate(mats):
            tabs[i][e] = _p(m, _u8p if i % 2 == 0 else _u16p)
    rw, rb = _f32(router_w), _f32(router_b)
    L = _Layer()
    L.hidden, L.inter, L.n_experts, L.top_k = H, shape.inter, E, shape.top_k
    L.n_group, L.topk_group, L.rsf = shape.n_group, shape.topk_group, shape.routed_scaling_factor
    L.wfmt, L.gsz = shape_format(shape)
    L.router_w, L.router_b = _p(rw, _f32p), _p(rb, _f32p)
    L.gate_q, L.gate_s, L.up_q, L.up_s, L.down_q, L.down_s = tabs
    if shared is not None and shape.n_shared > 0:
        sh = [np.ascontiguousarray(m) for m in shared]
        keep.append(sh)
        L.n_shared, L.shared_inter = 1, shape.i_shared
        (L.sh_gate_q, L.sh_gate_s, L.sh_up_q, L.sh_up_s, L.sh_down_q,
         L.sh_down_s) = [_p(m, _u8p if i % 2 == 0 else _u16p) for i, m in enumerate(sh)]
    else:
        L.n_shared, L.shared_inter = 0, 0
    ids = np.empty((T, shape.top_k), np.int32)
    w = np.empty((T, shape.top_k), np.float32)
    lg = np.empty((T, E), np.float32)
    y = np.empty((T, H), np.float32)
    g = None if gamma is None else _f32(gamma)
    r = None if resid is None else _f32(resid)
    rc = lib().oracle_moe_forward(C.byref(L), _p(x, _f32p), T, C.c_double(eps),
                                  _p(g, _f32p) if g is not None else None,
                                  _p(r, _f32p) if r is not None else None, prec,
                                  _p(ids, _i32p), _p(w, _f32p), _p(lg, _f32p), _p(y, _f32p))
    if rc:
        raise RuntimeError(f"oracle_moe_forward failed ({rc})")
    del keep
    return y, ids, w, lg


__all__ = ["router_exp", "router_sigmoid", "half_to_float", "dequant", "dequant_fmt",
           "router_logits", "select", "plan", "rmsnorm", "expert", "expert_fmt", "route",
           "moe_forward", "shape_format", "FMT_INT4", "FMT_INT8", "lib"]
