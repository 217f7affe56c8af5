"""GPU parity of the expert tier (moe_tier_*): the routed experts in pinned
host memory, a bounded set of them in HBM slots ("GLM-5.2 on a 32 GB Mac -
native MLX port of the Colibri hierarchy", "What Colibri is actually doing",
items 4-10).

The tier changes where the weights live, not the arithmetic.  Every call's
ids and gate weights are compared bit for bit with the oracle and its output
within the parity tolerance while slots are loaded, evicted, prefetched and
pinned.  The tier's counters and slot table are compared with the host slot
cache (checked against the plain statement of the rules on the CPU) driven by
the oracle's unions, so the tier took the policy's decisions.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, oracle_layer, rel_err_per_token, router_of
from workloads import CONFIGS
from workloads.configs import LayerShape, Workload
from workloads.gen import HostExpertCache, gen_activations, gen_layer

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
COUNTERS = ("hits_pinned", "hits_lru", "misses", "loads", "evictions", "n_resident", "n_pinned")


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_gb300 import build as b
    b.build()
    import int4_routed_expert_gb300 as mod
    mod.load()
    return mod


def _call(m, tier, wl, router, cache, x_cpu, ref, check_y=True):
    """One tier forward on x, checked against the oracle; the reference slot
    cache admits the oracle's union in the order the tier does (ascending)."""
    sh = wl.shape
    T = x_cpu.shape[0]
    plan = m.Plan(T, sh.top_k, sh.n_experts, DEV)
    y = tier.forward(x_cpu.to(DEV), plan=plan)
    torch.cuda.synchronize()
    x32 = x_cpu.float().numpy()
    _, _, ids_o, w_o = oracle.route(sh, router[0], router[1], x32)
    assert np.array_equal(plan.topk_ids.cpu().numpy(), ids_o)
    assert np.array_equal(plan.topk_w.cpu().numpy().view(np.uint32), w_o.view(np.uint32))
    if ref is not None:
        ref.admit(sorted(set(int(e) for e in ids_o.ravel())))
    if check_y:
        y_o, _, _, _ = oracle_layer(wl, 0, router, x32, list(range(T)), cache=cache)
        err = rel_err_per_token(y.cpu().numpy(), y_o)
        assert err.max() <= TOL, err
    return y


def _same_state(tier, ref):
    st, slot_of, uses = tier.query()
    rst, rslot, ruses = ref.query()
    for k in COUNTERS:
        assert st[k] == rst[k], (k, st, rst)
    assert list(slot_of) == list(rslot)
    assert list(uses) == list(ruses)
    return st


@pytest.mark.parametrize("fmt,gsz", [("int4", 32), ("int4", 0), ("int8", 32)])
def test_tier_lru_hot_store_and_formats(m, fmt, gsz):
    """16 experts, top-4, T = 1 or 2 (a call's union: up to 8), 10 slots of
    which 2 pinned: loads, LRU hits, evictions and pinned hits all happen."""
    sh = LayerShape(256, 128, 16, 4, 4, 2, 2.5, group_size=gsz, weight_format=fmt)
    wl = Workload("tier_small", sh, 2, 1, "f32", "zipf", 9400 + gsz + (7 if fmt == "int8" else 0))
    L = gen_layer(wl, device=DEV)
    tier = m.ExpertTier(L, max_tokens=2, n_slots=10, n_pinned=2)
    ref = m.SlotCache(16, 10, 2, 8)
    tier.pin([0, 5])
    ref.pin([0, 5])
    router, cache = router_of(wl, 0), HostExpertCache(wl, 0)
    for c in range(30):
        _call(m, tier, wl, router, cache, gen_activations(wl, 1 + c % 2, call=c), ref)
        if c == 14:
            assert tier.repin(2) == ref.repin(2)
    st = _same_state(tier, ref)
    assert st["misses"] > 0 and st["hits_lru"] > 0 and st["evictions"] > 0
    tier_stats = tier.query()[0]
    assert tier_stats["h2d_bytes"] == st["loads"] * sh.expert_bytes()
    tier.close()


def test_tier_prefetch_routed_makes_the_next_call_hit(m):
    sh = LayerShape(256, 128, 16, 4, 4, 2, 2.5)
    wl = Workload("tier_prefetch", sh, 1, 1, "f32", "zipf", 9410)
    L = gen_layer(wl, device=DEV)
    tier = m.ExpertTier(L, max_tokens=1, n_slots=6)
    ref = m.SlotCache(16, 6, 0, 4)
    router, cache = router_of(wl, 0), HostExpertCache(wl, 0)
    for c in range(12):
        x = gen_activations(wl, 1, call=c)
        tier.prefetch_routed(x.to(DEV))
        _, _, ids_o, _ = oracle.route(sh, router[0], router[1], x.float().numpy())
        ref.prefetch(sorted(set(int(e) for e in ids_o.ravel())))
        before = tier.query()[0]["misses"]
        _call(m, tier, wl, router, cache, x, ref)
        assert tier.query()[0]["misses"] == before
    _same_state(tier, ref)
    tier.close()


def test_tier_refill_waits_for_the_running_call(m):
    """Every slot holds an expert of the call just launched; a prefetch of
    other experts right after it (no synchronisation in between) must not
    overwrite them before that call has read them."""
    sh = LayerShape(2048, 1024, 16, 4, 4, 2, 2.5)
    wl = Workload("tier_hazard", sh, 1, 1, "f32", "uniform", 9420)
    L = gen_layer(wl, device=DEV)
    tier = m.ExpertTier(L, max_tokens=1, n_slots=4)
    router, cache = router_of(wl, 0), HostExpertCache(wl, 0)
    for c in range(6):
        x = gen_activations(wl, 1, call=c)
        x32 = x.float().numpy()
        _, _, ids_o, _ = oracle.route(sh, router[0], router[1], x32)
        others = [e for e in range(16) if e not in set(ids_o.ravel().tolist())][:4]
        y = tier.forward(x.to(DEV))
        tier.prefetch(others)
        torch.cuda.synchronize()
        y_o, _, _, _ = oracle_layer(wl, 0, router, x32, [0], cache=cache)
        assert rel_err_per_token(y.cpu().numpy(), y_o).max() <= TOL
        _, slot_of, _ = tier.query()
        assert all(slot_of[e] >= 0 for e in others)
    tier.close()


def test_tier_glm_decode(m):
    """GLM decode shape (256 experts, top-8), a quarter of the experts in
    HBM with 8 pinned: ids of 16 Zipf-routed tokens bit for bit, outputs of
    the first 4 within the tolerance."""
    wl = CONFIGS["glm_decode"]
    sh = wl.shape
    L = gen_layer(wl, device=DEV)
    tier = m.ExpertTier(L, max_tokens=1, n_slots=64, n_pinned=8, drop_device_routed=True)
    torch.cuda.empty_cache()
    ref = m.SlotCache(256, 64, 8, 8)
    router, cache = router_of(wl, 0), HostExpertCache(wl, 0)
    for c in range(16):
        _call(m, tier, wl, router, cache, gen_activations(wl, 1, call=c), ref, check_y=c < 4)
        if c == 7:
            assert tier.repin(4) == ref.repin(4)
    st = _same_state(tier, ref)
    assert st["misses"] > 0
    tier.close()


def test_tier_rejects_bad_arguments(m):
    sh = LayerShape(256, 128, 16, 4, 4, 2, 2.5)
    wl = Workload("tier_bad", sh, 1, 1, "f32", "uniform", 9430)
    L = gen_layer(wl, device=DEV)
    with pytest.raises(m.MoeError):
        m.ExpertTier(L, max_tokens=2, n_slots=7)           # a union of 8 does not fit
    with pytest.raises(m.MoeError):
        m.ExpertTier(L, max_tokens=1, n_slots=6, n_pinned=3)
    # routed arrays in device memory instead of page-locked host memory
    cfg = m.moe.config_for(sh, 1)
    w = m.moe.weights_for(L)
    import ctypes as C
    h = C.c_void_p()
    st = m.load().moe_tier_create(C.byref(cfg), C.byref(w),
                                  C.byref(m.moe.moe_tier_config_t(8, 0)), C.byref(h))
    assert st == m.moe.MOE_ERR_INVALID_ARG and not h.value
    tier = m.ExpertTier(L, max_tokens=1, n_slots=8)
    with pytest.raises(m.MoeError):
        tier.prefetch([3, 3])
    with pytest.raises(m.MoeError):
        tier.pin([16])
    x = gen_activations(wl, 2, call=0).to(DEV)
    with pytest.raises(m.MoeError):
        tier.forward(x)                                     # T = 2 > max_tokens
    tier.close()
