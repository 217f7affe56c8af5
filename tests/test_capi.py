"""Host-side checks of the C ABI: the library builds, loads and exports what
include/moe.h declares, and argument validation happens before any CUDA
call.  None of these launch a kernel, so they run without a GPU."""
from __future__ import annotations

import ctypes as C
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    from int4_routed_expert_gb300 import build as b
    b.build()
    import int4_routed_expert_gb300 as mod
    mod.load()
    return mod


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for mt in re.finditer(r"\b(moe_[a-z_]+)\s*\(", text):
            names.add(mt.group(1))
    return names


def _cfg(m, **kw):
    c = dict(hidden=256, inter=128, n_experts=16, top_k=4, n_group=4, topk_group=2,
             routed_scaling_factor=2.5, n_shared=1, shared_inter=128, group_size=32,
             max_tokens=8)
    c.update(kw)
    return m.moe.moe_config_t(**c)


def _fake_weights(m, base=0x10000000, step=0x100000):
    return m.moe.moe_weights_t(*[base + i * step for i in range(14)])


def test_library_builds_and_loads(m):
    assert os.path.exists(m.moe.LIB_PATH)


def test_every_declared_symbol_is_exported(m):
    lib = m.load()
    names = _declared()
    assert {"moe_layer_create", "moe_route", "moe_forward", "moe_destroy"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(m.EXPORTED) <= names


def test_workspace_bytes(m):
    small = m.moe_workspace_bytes(_cfg(m))
    big = m.moe_workspace_bytes(_cfg(m, max_tokens=64))
    assert 0 < small < big
    assert m.moe_workspace_bytes(_cfg(m, group_size=64)) == 0


@pytest.mark.parametrize("bad", [
    dict(hidden=300), dict(hidden=128), dict(hidden=12544), dict(inter=100), dict(n_experts=0),
    dict(n_experts=2048), dict(n_group=3), dict(topk_group=5), dict(top_k=0),
    dict(top_k=33), dict(top_k=9, topk_group=2), dict(group_size=64), dict(max_tokens=0),
    dict(n_shared=2), dict(shared_inter=100), dict(routed_scaling_factor=float("nan")),
    dict(group_size=16), dict(group_size=-1), dict(weight_format=2), dict(weight_format=-1),
])
def test_bad_configs_are_unsupported(m, bad):
    h = C.c_void_p()
    st = m.load().moe_layer_create(C.byref(_cfg(m, **bad)), C.byref(_fake_weights(m)), C.byref(h))
    assert st == -2 and not h.value
    assert m.moe_last_error(None)


def test_null_or_misaligned_weights(m):
    lib = m.load()
    w = _fake_weights(m)
    w.gate_q = None
    h = C.c_void_p()
    assert lib.moe_layer_create(C.byref(_cfg(m)), C.byref(w), C.byref(h)) == -1
    w = _fake_weights(m)
    w.down_s = 0x10000008
    assert lib.moe_layer_create(C.byref(_cfg(m)), C.byref(w), C.byref(h)) == -1
    # shared pointers may be NULL without a shared expert
    w = _fake_weights(m)
    w.sh_gate_q = None
    assert lib.moe_layer_create(C.byref(_cfg(m)), C.byref(w), C.byref(h)) == -1


def test_create_without_gpu_fails_loudly(m):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = C.c_void_p()
    st = m.load().moe_layer_create(C.byref(_cfg(m)), C.byref(_fake_weights(m)), C.byref(h))
    assert st == -4 and not h.value  # MOE_ERR_CUDA: there is no CPU fallback


def test_null_handle(m):
    lib = m.load()
    assert lib.moe_forward(None, None, 0, 1, None, None, 0.0, 0, None, None) == -1
    assert lib.moe_route(None, None, 0, 1, None, 0.0, None, None) == -1
    assert lib.moe_trace_enable(None, 1) == -1
    flags = C.c_int32()
    assert lib.moe_device_status(None, C.byref(flags)) == -1
    lib.moe_destroy(None)


def test_bounded_wait_selftest_arguments(m):
    """Invalid arguments are refused before the device is touched."""
    lib = m.load()
    flags = C.c_int32(7)
    assert lib.moe_selftest_bounded_wait(2, C.byref(flags)) == -1
    assert lib.moe_selftest_bounded_wait(-1, C.byref(flags)) == -1
    assert lib.moe_selftest_bounded_wait(0, None) == -1
    assert lib.moe_selftest_desync(None) == -1
    assert flags.value == 7
    assert m.moe_last_error(None)


def test_phase_names(m):
    names = [m.moe_trace_phase_name(p) for p in range(12)]
    assert all(names) and len(set(names)) == 12
    assert {"tc_prep", "tc_gate_up", "tc_down"} <= set(names)
    assert m.moe_trace_phase_name(12) is None and m.moe_trace_phase_name(-1) is None


def test_binding_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "int4_routed_expert_gb300")
    for path in glob.glob(os.path.join(pkg, "*.py")) + glob.glob(os.path.join(pkg, "csrc", "*")):
        text = open(path, errors="replace").read()
        assert not re.search(r"^\s*(import|from)\s+(oracle|numpy)\b", text, re.M), path
        assert "liboracle" not in text and "oracle.cpp" not in text, path


def test_binding_checks_tensors_before_the_call(m):
    """MoELayer refuses x, y, gamma and plan tensors that the kernels would
    read or write out of bounds (wrong device, shape, dtype, layout or size),
    on the host, before any C call."""
    import torch

    class _Shape:
        hidden, top_k, n_experts = 256, 4, 16

    lay = m.MoELayer.__new__(m.MoELayer)  # no handle: only the host checks run
    lay.h = None
    lay.shape = _Shape
    with pytest.raises(ValueError):
        lay._check_x(torch.zeros(2, 256))  # host tensor
    cpu = torch.device("cpu")
    lay._check_vec(torch.zeros(3, 256), "y", 3, cpu)
    for bad in (torch.zeros(2, 256), torch.zeros(3, 256, dtype=torch.float64),
                torch.zeros(256, 3).t()):
        with pytest.raises(ValueError):
            lay._check_vec(bad, "y", 3, cpu)
    p = m.Plan(3, 4, 16, "cpu")
    p.check(3, 4, 16, cpu)
    p.check(2, 4, 16, cpu)  # more room than needed is fine
    for args in ((4, 4, 16, cpu), (3, 4, 17, cpu), (3, 4, 16, torch.device("meta"))):
        with pytest.raises(ValueError):
            p.check(*args)


def test_route_noalloc_config_checks(m):
    """moe_route_noalloc ignores max_tokens (any value is accepted) and
    reports the configuration check's own reason for a bad geometry."""
    f = m.load().moe_route_noalloc
    for mt in (0, -5, 10 ** 6):
        st = f(C.byref(_cfg(m, max_tokens=mt)), None, None, None, 0, 0, None, 0.0, None, None)
        assert st == 0, (mt, m.moe_last_error(None))  # T == 0: a no-op after the checks
    st = f(C.byref(_cfg(m, n_group=3, max_tokens=0)), None, None, None, 0, 0, None, 0.0, None,
           None)
    assert st == -2
    assert "multiple of n_group" in m.moe_last_error(None)
    st = f(None, None, None, None, 0, 0, None, 0.0, None, None)
    assert st == -2 and "cfg is NULL" in m.moe_last_error(None)


@pytest.mark.parametrize("fmt", [dict(group_size=0), dict(weight_format=1),
                                 dict(weight_format=1, group_size=0)])
def test_other_formats_are_accepted(m, fmt):
    """int8 experts and one scale a row are valid configurations (the
    workspace size does not depend on the format)."""
    lib = m.load()
    assert lib.moe_workspace_bytes(C.byref(_cfg(m, **fmt))) == \
        lib.moe_workspace_bytes(C.byref(_cfg(m)))


def test_tier_create_validates_before_any_cuda_call(m):
    """The expert tier's argument checks run on the host: NULL arguments,
    a bad geometry, and slot counts that cannot hold one call's union."""
    lib = m.load()
    h = C.c_void_p()
    w = _fake_weights(m)
    tc = m.moe.moe_tier_config_t
    assert lib.moe_tier_create(None, C.byref(w), C.byref(tc(8, 0)), C.byref(h)) == -1
    assert lib.moe_tier_create(C.byref(_cfg(m, hidden=300)), C.byref(w), C.byref(tc(8, 0)),
                               C.byref(h)) == -2
    # max_tokens 8 x top-4 over 16 experts: a union may hold all 16
    for slots, pinned in ((0, 0), (17, 0), (15, 0), (16, 1), (16, -1)):
        st = lib.moe_tier_create(C.byref(_cfg(m)), C.byref(w), C.byref(tc(slots, pinned)),
                                 C.byref(h))
        assert st == -1 and not h.value, (slots, pinned)
        assert b"n_slots" in lib.moe_last_error(None)
    assert lib.moe_tier_forward(None, None, 0, 1, None, None, 0.0, 0, None, None) == -1
    assert lib.moe_tier_repin(None, 1, None) == -1
    lib.moe_tier_destroy(None)


@pytest.mark.parametrize("E,k,T", [(16, 4, 1), (16, 4, 8), (256, 8, 1), (256, 8, 4), (64, 6, 3)])
def test_tier_slot_rule(m, E, k, T):
    """n_slots - n_pinned must hold one call's union, min(E, max_tokens * k):
    one slot fewer is refused for its slot count; exactly enough passes that
    check and stops at the next one (the fake routed pointers are not
    page-locked host memory)."""
    lib = m.load()
    need = min(E, T * k)
    cfg = _cfg(m, n_experts=E, top_k=k, n_group=1, topk_group=1, max_tokens=T)
    h = C.c_void_p()
    for pinned in (0, 2):
        if need + pinned > E:
            continue
        tc = m.moe.moe_tier_config_t(need + pinned - 1, pinned)
        assert lib.moe_tier_create(C.byref(cfg), C.byref(_fake_weights(m)), C.byref(tc),
                                   C.byref(h)) == -1
        assert b"n_slots" in lib.moe_last_error(None)
        tc = m.moe.moe_tier_config_t(need + pinned, pinned)
        assert lib.moe_tier_create(C.byref(cfg), C.byref(_fake_weights(m)), C.byref(tc),
                                   C.byref(h)) == -1
        assert b"page-locked" in lib.moe_last_error(None) and not h.value
