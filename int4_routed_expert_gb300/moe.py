"""ctypes binding of libmoe.so, with the C ABI's names (argument marshalling only).

Every step of the layer runs in the library's CUDA kernels.  If the library
is missing or cannot be loaded, ``load`` raises; there is no Python or CPU
fallback.

Low-level functions mirror include/moe.h one to one:
    moe_layer_create, moe_route, moe_forward, moe_destroy, moe_last_error,
    moe_workspace_bytes, moe_trace_enable, moe_trace_read,
    moe_trace_phase_name, moe_device_status, moe_selftest_bounded_wait,
    moe_selftest_desync, moe_route_noalloc, the expert slot cache
    (moe_slot_cache_*) and the expert tier (moe_tier_*)
``MoELayer`` wraps a handle around torch tensors (device memory and streams
only) for the tests and the benchmark; ``ExpertTier`` does the same for an
expert tier (routed experts in pinned host memory, a bounded set in HBM) and
``SlotCache`` for the tier's host-side residency policy.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CAPACITY = -3
MOE_ERR_CUDA = -4
MOE_ERR_OOM = -5
MOE_F32 = 0
MOE_BF16 = 1

_STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
           -3: "MOE_ERR_CAPACITY", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_OOM"}


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


class moe_config_t(C.Structure):
    _fields_ = [("hidden", C.c_int), ("inter", C.c_int), ("n_experts", C.c_int),
                ("top_k", C.c_int), ("n_group", C.c_int), ("topk_group", C.c_int),
                ("routed_scaling_factor", C.c_float), ("n_shared", C.c_int),
                ("shared_inter", C.c_int), ("group_size", C.c_int),
                ("max_tokens", C.c_int), ("weight_format", C.c_int)]


MOE_W_INT4, MOE_W_INT8 = 0, 1


class moe_weights_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "router_w", "router_bias", "gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
        "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q", "sh_down_s")]


class moe_plan_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "topk_ids", "topk_w", "counts", "offsets", "perm", "active", "n_active")]


class moe_tier_config_t(C.Structure):
    _fields_ = [("n_slots", C.c_int), ("n_pinned", C.c_int)]


class moe_slot_cache_stats_t(C.Structure):
    _fields_ = [("hits_pinned", C.c_uint64), ("hits_lru", C.c_uint64), ("misses", C.c_uint64),
                ("loads", C.c_uint64), ("evictions", C.c_uint64), ("n_resident", C.c_int32),
                ("n_pinned", C.c_int32)]


# kinds of an admitted expert (moe_slot_cache_admit)
SLOT_HIT_PINNED, SLOT_HIT_LRU, SLOT_LOAD = 0, 1, 2

EXPORTED = ("moe_layer_create", "moe_route", "moe_forward", "moe_destroy",
            "moe_last_error", "moe_workspace_bytes", "moe_trace_enable", "moe_trace_read",
            "moe_trace_phase_name", "moe_device_status", "moe_route_noalloc",
            "moe_selftest_bounded_wait", "moe_selftest_desync",
            "moe_slot_cache_create", "moe_slot_cache_admit", "moe_slot_cache_prefetch",
            "moe_slot_cache_pin", "moe_slot_cache_repin", "moe_slot_cache_query",
            "moe_slot_cache_destroy", "moe_tier_create", "moe_tier_forward",
            "moe_tier_prefetch", "moe_tier_prefetch_routed", "moe_tier_pin", "moe_tier_repin",
            "moe_tier_query", "moe_tier_last_error", "moe_tier_destroy")

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libmoe.so (build it first with int4_routed_expert_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: run `python -m int4_routed_expert_gb300.build` "
                          "(there is no fallback implementation)")
    L = C.CDLL(path)
    L.moe_layer_create.restype = C.c_int
    L.moe_layer_create.argtypes = [C.POINTER(moe_config_t), C.POINTER(moe_weights_t),
                                   C.POINTER(C.c_void_p)]
    L.moe_route.restype = C.c_int
    L.moe_route.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_float,
                            C.POINTER(moe_plan_t), C.c_void_p]
    L.moe_forward.restype = C.c_int
    L.moe_forward.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p,
                              C.c_void_p, C.c_float, C.c_int, C.POINTER(moe_plan_t),
                              C.c_void_p]
    L.moe_destroy.restype = None
    L.moe_destroy.argtypes = [C.c_void_p]
    L.moe_last_error.restype = C.c_char_p
    L.moe_last_error.argtypes = [C.c_void_p]
    L.moe_workspace_bytes.restype = C.c_size_t
    L.moe_workspace_bytes.argtypes = [C.POINTER(moe_config_t)]
    L.moe_trace_enable.restype = C.c_int
    L.moe_trace_enable.argtypes = [C.c_void_p, C.c_int]
    L.moe_trace_read.restype = C.c_int
    L.moe_trace_read.argtypes = [C.c_void_p, C.POINTER(C.c_float), C.c_int,
                                 C.POINTER(C.c_int), C.POINTER(C.c_int)]
    L.moe_trace_phase_name.restype = C.c_char_p
    L.moe_trace_phase_name.argtypes = [C.c_int]
    L.moe_device_status.restype = C.c_int
    L.moe_device_status.argtypes = [C.c_void_p, C.POINTER(C.c_int32)]
    L.moe_selftest_desync.restype = C.c_int
    L.moe_selftest_desync.argtypes = [C.c_void_p]
    L.moe_selftest_bounded_wait.restype = C.c_int
    L.moe_selftest_bounded_wait.argtypes = [C.c_int, C.POINTER(C.c_int32)]
    L.moe_route_noalloc.restype = C.c_int
    L.moe_route_noalloc.argtypes = [C.POINTER(moe_config_t), C.c_void_p, C.c_void_p, C.c_void_p,
                                    C.c_int, C.c_int, C.c_void_p, C.c_float,
                                    C.POINTER(moe_plan_t), C.c_void_p]
    i32p = C.POINTER(C.c_int32)
    u64p = C.POINTER(C.c_uint64)
    L.moe_slot_cache_create.restype = C.c_int
    L.moe_slot_cache_create.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int,
                                        C.POINTER(C.c_void_p)]
    for fn in ("moe_slot_cache_admit", "moe_slot_cache_prefetch", "moe_slot_cache_pin"):
        getattr(L, fn).restype = C.c_int
        getattr(L, fn).argtypes = [C.c_void_p, i32p, C.c_int, i32p, i32p]
    L.moe_slot_cache_repin.restype = C.c_int
    L.moe_slot_cache_repin.argtypes = [C.c_void_p, C.c_int]
    L.moe_slot_cache_query.restype = C.c_int
    L.moe_slot_cache_query.argtypes = [C.c_void_p, C.POINTER(moe_slot_cache_stats_t), i32p,
                                       u64p]
    L.moe_slot_cache_destroy.restype = None
    L.moe_slot_cache_destroy.argtypes = [C.c_void_p]
    L.moe_tier_create.restype = C.c_int
    L.moe_tier_create.argtypes = [C.POINTER(moe_config_t), C.POINTER(moe_weights_t),
                                  C.POINTER(moe_tier_config_t), C.POINTER(C.c_void_p)]
    L.moe_tier_forward.restype = C.c_int
    L.moe_tier_forward.argtypes = L.moe_forward.argtypes
    L.moe_tier_prefetch.restype = C.c_int
    L.moe_tier_prefetch.argtypes = [C.c_void_p, i32p, C.c_int]
    L.moe_tier_prefetch_routed.restype = C.c_int
    L.moe_tier_prefetch_routed.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p,
                                           C.c_float, C.c_void_p]
    L.moe_tier_pin.restype = C.c_int
    L.moe_tier_pin.argtypes = [C.c_void_p, i32p, C.c_int]
    L.moe_tier_repin.restype = C.c_int
    L.moe_tier_repin.argtypes = [C.c_void_p, C.c_int, C.POINTER(C.c_int)]
    L.moe_tier_query.restype = C.c_int
    L.moe_tier_query.argtypes = [C.c_void_p, C.POINTER(moe_slot_cache_stats_t), i32p, u64p,
                                 u64p]
    L.moe_tier_last_error.restype = C.c_char_p
    L.moe_tier_last_error.argtypes = [C.c_void_p]
    L.moe_tier_destroy.restype = None
    L.moe_tier_destroy.argtypes = [C.c_void_p]
    _lib = L
    return L


def moe_last_error(h) -> str:
    return (load().moe_last_error(h) or b"").decode()


def _check(st: int, h=None):
    if st != MOE_OK:
        raise MoeError(st, moe_last_error(h))


def moe_workspace_bytes(cfg: moe_config_t) -> int:
    return int(load().moe_workspace_bytes(C.byref(cfg)))


def moe_layer_create(cfg: moe_config_t, w: moe_weights_t) -> C.c_void_p:
    h = C.c_void_p()
    _check(load().moe_layer_create(C.byref(cfg), C.byref(w), C.byref(h)), None)
    return h


def moe_route(h, x: int, dtype: int, T: int, gamma: int | None, eps: float,
              plan: moe_plan_t | None, stream: int | None) -> None:
    _check(load().moe_route(h, x, dtype, T, gamma, eps,
                            C.byref(plan) if plan is not None else None, stream), h)


def moe_forward(h, x: int, dtype: int, T: int, y: int, gamma: int | None, eps: float,
                accumulate: int, plan: moe_plan_t | None, stream: int | None) -> None:
    _check(load().moe_forward(h, x, dtype, T, y, gamma, eps, accumulate,
                              C.byref(plan) if plan is not None else None, stream), h)


def moe_route_noalloc(cfg: moe_config_t, router_w: int, router_bias: int, x: int, dtype: int,
                      T: int, gamma: int | None, eps: float, plan: moe_plan_t | None,
                      stream: int | None) -> None:
    """Routing of T tokens without a handle and without any allocation."""
    _check(load().moe_route_noalloc(C.byref(cfg), router_w, router_bias, x, dtype, T, gamma, eps,
                                    C.byref(plan) if plan is not None else None, stream), None)


def moe_destroy(h) -> None:
    if h:
        load().moe_destroy(h)


def moe_trace_enable(h, n_calls: int) -> None:
    _check(load().moe_trace_enable(h, n_calls), h)


def moe_trace_phase_name(p: int) -> str | None:
    r = load().moe_trace_phase_name(p)
    return r.decode() if r else None


def moe_device_status(h) -> int:
    """Device error flags of the handle (0 = fine); raises MoeError if set."""
    f = C.c_int32(0)
    _check(load().moe_device_status(h, C.byref(f)), h)
    return f.value


def moe_selftest_bounded_wait(which: int) -> int:
    """Error word of a one-warp kernel whose wait never completes (0: grid
    barrier, 1: mbarrier); bit 0 set when the wait gave up.  Takes ~1 s."""
    f = C.c_int32(0)
    _check(load().moe_selftest_bounded_wait(which, C.byref(f)))
    return f.value


def moe_selftest_desync(h) -> None:
    """Put the handle in the state a call that gave up leaves (self-test of
    the recovery in moe_device_status)."""
    _check(load().moe_selftest_desync(h), h)


def moe_trace_read(h, cap: int):
    """-> (phase names, list of per-call lists of phase milliseconds)."""
    buf = (C.c_float * max(1, cap * 16))()
    n, npha = C.c_int(), C.c_int()
    _check(load().moe_trace_read(h, buf, cap, C.byref(n), C.byref(npha)), h)
    names = [moe_trace_phase_name(p) for p in range(npha.value)]
    rows = [[buf[c * npha.value + p] for p in range(npha.value)] for c in range(n.value)]
    return names, rows


# ---------------------------------------------------------- torch wrapper --

def config_for(shape, max_tokens: int) -> moe_config_t:
    fmt = MOE_W_INT8 if getattr(shape, "weight_format", "int4") == "int8" else MOE_W_INT4
    return moe_config_t(shape.hidden, shape.inter, shape.n_experts, shape.top_k,
                        shape.n_group, shape.topk_group, shape.routed_scaling_factor,
                        shape.n_shared, shape.i_shared if shape.n_shared else 0,
                        shape.group_size, max_tokens, fmt)


def weights_for(L) -> moe_weights_t:
    """moe_weights_t from a workloads.gen.LayerInputs living on the device."""
    p = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    return moe_weights_t(p(L.router_w), p(L.router_b), p(L.gate_q), p(L.gate_s), p(L.up_q),
                         p(L.up_s), p(L.down_q), p(L.down_s), p(L.sh_gate_q), p(L.sh_gate_s),
                         p(L.sh_up_q), p(L.sh_up_s), p(L.sh_down_q), p(L.sh_down_s))


class Plan:
    """Device buffers for the routing outputs of T tokens."""

    def __init__(self, T: int, k: int, E: int, device):
        import torch
        i32 = dict(dtype=torch.int32, device=device)
        self.topk_ids = torch.empty(T, k, **i32)
        self.topk_w = torch.empty(T, k, dtype=torch.float32, device=device)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm = torch.empty(T * k, **i32)
        self.active = torch.full((E,), -1, **i32)
        self.n_active = torch.empty(1, **i32)

    def c(self) -> moe_plan_t:
        return moe_plan_t(*(getattr(self, n).data_ptr() for n, _ in moe_plan_t._fields_))

    def check(self, T: int, k: int, E: int, device) -> None:
        """Raise unless every buffer is a contiguous int32/fp32 tensor on
        ``device`` large enough for T tokens of this layer."""
        import torch
        need = {"topk_ids": (torch.int32, T * k), "topk_w": (torch.float32, T * k),
                "counts": (torch.int32, E), "offsets": (torch.int32, E + 1),
                "perm": (torch.int32, T * k), "active": (torch.int32, E),
                "n_active": (torch.int32, 1)}
        for name, (dt, n) in need.items():
            t = getattr(self, name)
            if t.device != device or t.dtype != dt or not t.is_contiguous() or t.numel() < n:
                raise ValueError(f"plan.{name} must be a contiguous {dt} tensor on {device} "
                                 f"with at least {n} elements")


class _TensorIO:
    """Argument checks shared by the torch wrappers (shape, device, dtype)."""

    shape = None
    device = None

    @staticmethod
    def _dtype(x) -> int:
        import torch
        if x.dtype == torch.float32:
            return MOE_F32
        if x.dtype == torch.bfloat16:
            return MOE_BF16
        raise TypeError(f"x must be fp32 or bf16, got {x.dtype}")

    @staticmethod
    def _io_ok(t) -> bool:
        """x and y may live on a CUDA device or in pinned host memory (the
        kernels then read and write it across the host link)."""
        return t.is_cuda or (t.device.type == "cpu" and t.is_pinned())

    def _check_x(self, x):
        """x: a contiguous [T][hidden] fp32/bf16 tensor on a CUDA device or in
        pinned host memory; returns T."""
        if not self._io_ok(x) or x.dim() != 2 or x.shape[1] != self.shape.hidden \
                or not x.is_contiguous():
            raise ValueError(f"x must be a contiguous CUDA or pinned host tensor of shape "
                             f"[T, {self.shape.hidden}], got {tuple(x.shape)} on {x.device}")
        return x.shape[0]

    def _check_vec(self, t, name: str, rows: int, device, host_ok: bool = False):
        """t: a contiguous fp32 tensor on ``device`` (or pinned host memory when
        host_ok) with rows * hidden elements."""
        import torch
        where_ok = t.device == device or (host_ok and self._io_ok(t))
        if not where_ok or t.dtype != torch.float32 or not t.is_contiguous() \
                or t.numel() != rows * self.shape.hidden:
            raise ValueError(f"{name} must be a contiguous fp32 tensor on {device} with "
                             f"{rows} x {self.shape.hidden} elements")

    @staticmethod
    def _stream(stream) -> int:
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        return s.cuda_stream

    def _forward_args(self, x, y, gamma, plan):
        """Checks forward's tensors; returns (T, y, plan struct or None)."""
        import torch
        T = self._check_x(x)
        if y is None:
            y = torch.empty(T, self.shape.hidden, dtype=torch.float32, device=self.device)
        self._check_vec(y, "y", T, self.device, host_ok=True)
        if gamma is not None:
            self._check_vec(gamma, "gamma", 1, self.device)
        if plan is not None:
            plan.check(T, self.shape.top_k, self.shape.n_experts, self.device)
        return T, y, (plan.c() if plan is not None else None)


class MoELayer(_TensorIO):
    """Handle + the tensors it borrows.  torch supplies memory and streams."""

    def __init__(self, layer_inputs, max_tokens: int):
        self.inputs = layer_inputs  # keeps the weights alive
        self.shape = layer_inputs.shape
        self.device = layer_inputs.router_w.device
        self.max_tokens = max_tokens
        self.cfg = config_for(self.shape, max_tokens)
        self.h = moe_layer_create(self.cfg, weights_for(layer_inputs))

    def close(self):
        if self.h:
            moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def route(self, x, gamma=None, eps: float = 1e-5, plan: Plan | None = None,
              stream=None) -> Plan:
        T = self._check_x(x)
        if gamma is not None:
            self._check_vec(gamma, "gamma", 1, self.device)
        plan = plan or Plan(T, self.shape.top_k, self.shape.n_experts, self.device)
        plan.check(T, self.shape.top_k, self.shape.n_experts, self.device)
        pc = plan.c()
        moe_route(self.h, x.data_ptr(), self._dtype(x), T,
                  gamma.data_ptr() if gamma is not None else None, eps, pc,
                  self._stream(stream))
        return plan

    def forward(self, x, y=None, gamma=None, eps: float = 1e-5, accumulate: bool = False,
                plan: Plan | None = None, stream=None):
        T, y, pc = self._forward_args(x, y, gamma, plan)
        moe_forward(self.h, x.data_ptr(), self._dtype(x), T, y.data_ptr(),
                    gamma.data_ptr() if gamma is not None else None, eps,
                    1 if accumulate else 0, pc, self._stream(stream))
        return y


# ------------------------------------------------------------ expert tier --

ROUTED_ARRAYS = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")


def _i32(ids):
    """ctypes int32 array of a sequence of expert ids, and its length."""
    v = [int(e) for e in ids]
    return (C.c_int32 * max(1, len(v)))(*v), len(v)


def _stats_dict(st: moe_slot_cache_stats_t) -> dict:
    return {n: int(getattr(st, n)) for n, _ in moe_slot_cache_stats_t._fields_}


class SlotCache:
    """The expert tier's residency policy on the host (moe_slot_cache_*)."""

    def __init__(self, n_experts: int, n_slots: int, n_pinned: int, call_slots: int):
        self.n_experts = n_experts
        h = C.c_void_p()
        _check(load().moe_slot_cache_create(n_experts, n_slots, n_pinned, call_slots,
                                            C.byref(h)))
        self.h = h

    def _op(self, fn, ids):
        a, n = _i32(ids)
        slot = (C.c_int32 * max(1, n))()
        kind = (C.c_int32 * max(1, n))()
        _check(fn(self.h, a, n, slot, kind))
        return list(slot[:n]), list(kind[:n])

    def admit(self, ids):
        """-> (slots, kinds) of one call's distinct experts."""
        return self._op(load().moe_slot_cache_admit, ids)

    def prefetch(self, ids):
        return self._op(load().moe_slot_cache_prefetch, ids)

    def pin(self, ids):
        return self._op(load().moe_slot_cache_pin, ids)

    def repin(self, max_swaps: int) -> int:
        r = load().moe_slot_cache_repin(self.h, max_swaps)
        if r < 0:
            raise MoeError(MOE_ERR_INVALID_ARG, "moe_slot_cache_repin: bad arguments")
        return r

    def query(self):
        """-> (counters, slot_of [E] (-(slot+2) when pinned, -1 absent), uses [E])."""
        st = moe_slot_cache_stats_t()
        slot_of = (C.c_int32 * self.n_experts)()
        uses = (C.c_uint64 * self.n_experts)()
        _check(load().moe_slot_cache_query(self.h, C.byref(st), slot_of, uses))
        return _stats_dict(st), list(slot_of), list(uses)

    def close(self):
        if self.h:
            load().moe_slot_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ExpertTier(_TensorIO):
    """Expert tier (moe_tier_*): the routed experts of ``layer_inputs`` are
    copied to pinned host memory (the slower tier); ``n_slots`` of them are
    held in HBM at a time.  The router and the shared expert stay on the
    device.  ``drop_device_routed`` releases the device copies of the routed
    arrays from ``layer_inputs`` afterwards."""

    def __init__(self, layer_inputs, max_tokens: int, n_slots: int, n_pinned: int = 0,
                 drop_device_routed: bool = False):
        import torch
        L = layer_inputs
        self.shape = L.shape
        self.device = L.router_w.device
        self.max_tokens = max_tokens
        self.cfg = config_for(self.shape, max_tokens)
        self.host = {}
        for n in ROUTED_ARRAYS:
            t = getattr(L, n)
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            self.host[n] = h
        w = weights_for(L)
        for n in ROUTED_ARRAYS:
            setattr(w, n, self.host[n].data_ptr())
        if drop_device_routed:
            for n in ROUTED_ARRAYS:
                setattr(L, n, None)
        self.inputs = L  # keeps the router and shared-expert tensors alive
        h = C.c_void_p()
        tc = moe_tier_config_t(n_slots, n_pinned)
        st = load().moe_tier_create(C.byref(self.cfg), C.byref(w), C.byref(tc), C.byref(h))
        if st != MOE_OK:
            raise MoeError(st, moe_last_error(None))
        self.h = h

    def _check(self, st):
        if st != MOE_OK:
            raise MoeError(st, (load().moe_tier_last_error(self.h) or b"").decode())

    def forward(self, x, y=None, gamma=None, eps: float = 1e-5, accumulate: bool = False,
                plan: Plan | None = None, stream=None):
        T, y, pc = self._forward_args(x, y, gamma, plan)
        self._check(load().moe_tier_forward(
            self.h, x.data_ptr(), self._dtype(x), T, y.data_ptr(),
            gamma.data_ptr() if gamma is not None else None, eps, 1 if accumulate else 0,
            C.byref(pc) if pc is not None else None, self._stream(stream)))
        return y

    def prefetch(self, ids) -> None:
        a, n = _i32(ids)
        self._check(load().moe_tier_prefetch(self.h, a, n))

    def prefetch_routed(self, x, gamma=None, eps: float = 1e-5, stream=None) -> None:
        T = self._check_x(x)
        if gamma is not None:
            self._check_vec(gamma, "gamma", 1, self.device)
        self._check(load().moe_tier_prefetch_routed(
            self.h, x.data_ptr(), self._dtype(x), T,
            gamma.data_ptr() if gamma is not None else None, eps, self._stream(stream)))

    def pin(self, ids) -> None:
        a, n = _i32(ids)
        self._check(load().moe_tier_pin(self.h, a, n))

    def repin(self, max_swaps: int) -> int:
        c = C.c_int(0)
        self._check(load().moe_tier_repin(self.h, max_swaps, C.byref(c)))
        return c.value

    def query(self):
        """-> (counters incl. h2d_bytes, slot_of [E], uses [E])."""
        E = self.shape.n_experts
        st = moe_slot_cache_stats_t()
        slot_of = (C.c_int32 * E)()
        uses = (C.c_uint64 * E)()
        h2d = C.c_uint64(0)
        self._check(load().moe_tier_query(self.h, C.byref(st), slot_of, uses, C.byref(h2d)))
        d = _stats_dict(st)
        d["h2d_bytes"] = int(h2d.value)
        return d, list(slot_of), list(uses)

    def close(self):
        if self.h:
            load().moe_tier_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
