"""moe_route_noalloc (routing with static device scratch, no allocation)
against moe_route on a layer handle, through the C ABI, on a GPU.

Collected last on purpose: it must pass alone and after every other test,
so nothing in its static scratch may depend on earlier calls."""
from __future__ import annotations

import pytest
import torch

from workloads import CONFIGS
from workloads.configs import LayerShape, Workload
from workloads.gen import gen_activations, gen_layer, gen_norm_weight

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PLAN_FIELDS = ("topk_ids", "topk_w", "counts", "offsets", "perm", "n_active")


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_gb300 import build as b
    b.build()
    import int4_routed_expert_gb300 as mod
    mod.load()
    return mod


def _same_plan(p1, p2):
    for name in PLAN_FIELDS:
        assert torch.equal(getattr(p1, name), getattr(p2, name)), name
    n = int(p1.n_active.item())
    assert torch.equal(p1.active[:n], p2.active[:n])


def _noalloc(m, cfg, L, x, gamma, eps, plan):
    dt = m.MOE_BF16 if x.dtype == torch.bfloat16 else m.MOE_F32
    m.moe_route_noalloc(cfg, L.router_w.data_ptr(), L.router_b.data_ptr(), x.data_ptr(), dt,
                        x.shape[0], gamma.data_ptr() if gamma is not None else None, eps,
                        plan.c(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("which", ["tiny", "glm_like", "glm_like_rmsnorm"])
def test_noalloc_matches_handle_route_twice(m, which):
    if which == "tiny":
        wl = CONFIGS["tiny"]
    else:
        wl = Workload(which, LayerShape(1024, 512, 64, 6, 8, 3, 2.5), 4, 1, "bf16", "zipf", 8100,
                      rmsnorm_eps=1e-5 if which.endswith("rmsnorm") else 0.0)
    sh = wl.shape
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 64)
    cfg = m.moe.config_for(sh, 64)
    gamma = gen_norm_weight(wl, 0).to(DEV) if wl.rmsnorm_eps > 0 else None
    eps = 1e-5
    for T in (1, 5, 33):
        xs = [gen_activations(wl, T, call=c).to(DEV) for c in (T, T + 100)]
        plans = [m.Plan(T, sh.top_k, sh.n_experts, DEV) for _ in range(4)]
        # two calls in a row with different inputs, each checked against the handle
        for i, x in enumerate(xs):
            ref = h.route(x, gamma=gamma, eps=eps, plan=plans[2 * i])
            _noalloc(m, cfg, L, x, gamma, eps, plans[2 * i + 1])
            torch.cuda.synchronize()
            _same_plan(ref, plans[2 * i + 1])
    h.close()


def test_noalloc_allocates_nothing_and_rejects_oversize(m):
    sh = LayerShape(6144, 2048, 256, 8, 8, 4, 2.5)
    wl = Workload("glm_router_only", sh, 1, 1, "bf16", "zipf", 8200)
    from workloads.gen import gen_router
    rw, rb = gen_router(sh, wl.seed, 0, wl.bias_kind, wl.zipf_s)
    rw, rb = rw.to(DEV), rb.to(DEV)

    class R:  # the router-only view a prefetcher would hold
        router_w, router_b = rw, rb

    cfg = m.moe.config_for(sh, 64)
    T = 64
    x = gen_activations(wl, T, call=0).to(DEV)
    plan = m.Plan(T, sh.top_k, sh.n_experts, DEV)
    _noalloc(m, cfg, R, x, None, 0.0, plan)   # first call: per-device set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(m, cfg, R, x, None, 0.0, plan)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    counts = plan.counts.cpu()
    assert int(counts.sum()) == T * sh.top_k
    big = gen_activations(wl, 96, call=1).to(DEV)
    big_plan = m.Plan(96, sh.top_k, sh.n_experts, DEV)
    with pytest.raises(m.MoeError) as ei:
        _noalloc(m, cfg, R, big, None, 0.0, big_plan)
    assert ei.value.status == -3 and "2 MiB" in str(ei.value)


def test_noalloc_partial_plan_and_argument_checks(m):
    """Plan members left NULL (and a NULL plan) are kept in the scratch: the
    members that are given still match the handle's route.  max_tokens is
    ignored, and a router buffer shorter than E * H floats is refused before
    any launch."""
    import ctypes as C
    wl = Workload("glm_like_partial", LayerShape(1024, 512, 64, 6, 8, 3, 2.5), 4, 1, "bf16",
                  "zipf", 8300)
    sh = wl.shape
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 64)
    T = 9
    x = gen_activations(wl, T, call=3).to(DEV)
    ref = h.route(x, plan=m.Plan(T, sh.top_k, sh.n_experts, DEV))
    torch.cuda.synchronize()
    cfg = m.moe.config_for(sh, 0)  # max_tokens = 0: not used by this call
    stream = torch.cuda.current_stream().cuda_stream
    full = m.Plan(T, sh.top_k, sh.n_experts, DEV)
    part = full.c()
    for name in ("topk_w", "offsets", "perm", "active", "n_active"):
        setattr(part, name, None)
    for t in (full.topk_ids, full.counts):
        t.fill_(-1)
    m.moe_route_noalloc(cfg, L.router_w.data_ptr(), L.router_b.data_ptr(), x.data_ptr(),
                        m.MOE_BF16, T, None, 0.0, part, stream)
    torch.cuda.synchronize()
    assert torch.equal(full.topk_ids, ref.topk_ids)
    assert torch.equal(full.counts, ref.counts)
    # no plan at all, then the full plan again: still the handle's result
    m.moe_route_noalloc(cfg, L.router_w.data_ptr(), L.router_b.data_ptr(), x.data_ptr(),
                        m.MOE_BF16, T, None, 0.0, None, stream)
    again = m.Plan(T, sh.top_k, sh.n_experts, DEV)
    _noalloc(m, cfg, L, x, None, 0.0, again)
    torch.cuda.synchronize()
    _same_plan(ref, again)
    # router arrays outside device memory are refused on the host (a short
    # device buffer is refused the same way, but whether the addresses past a
    # caching-allocator tensor belong to some allocation depends on the pool)
    host_w = torch.zeros(sh.n_experts * sh.hidden, dtype=torch.float32).pin_memory()
    with pytest.raises(m.MoeError) as ei:
        m.moe_route_noalloc(cfg, host_w.data_ptr(), L.router_b.data_ptr(), x.data_ptr(),
                            m.MOE_BF16, T, None, 0.0, again.c(), stream)
    assert ei.value.status == -1 and "router_w" in str(ei.value)
    plain = C.create_string_buffer(sh.n_experts * 4 + 16)
    addr = (C.addressof(plain) + 15) & ~15
    with pytest.raises(m.MoeError) as ei:
        m.moe_route_noalloc(cfg, L.router_w.data_ptr(), addr, x.data_ptr(),
                            m.MOE_BF16, T, None, 0.0, again.c(), stream)
    assert ei.value.status == -1 and "router_bias" in str(ei.value)
    h.close()
