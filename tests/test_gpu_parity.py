"""Parity of the CUDA layer, called through the C ABI, with the CPU oracle.

Expert ids, gate weights and the whole routing plan must match bit for bit;
layer outputs must match within TOL (per-token max abs error / max abs
oracle output) of the fp32-accumulated oracle.  Every input is seeded and
synthetic (workloads/).  Runs only on a machine with a CUDA GPU.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from parity_util import (RMS_EPS, TOL, elem_err_per_token, oracle_layer, rel_err_per_token,
                         resid_err_per_token, router_of)
from workloads import CONFIGS
from workloads.configs import LayerShape, Workload
from workloads.gen import HostExpertCache, gen_activations, gen_layer, gen_norm_weight

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_gb300 import build as b
    b.build()
    import int4_routed_expert_gb300 as mod
    mod.load()
    return mod


def _check_plan(plan, ids_o, E):
    P = oracle.plan(ids_o, E)
    assert np.array_equal(plan.counts.cpu().numpy(), P["counts"])
    assert np.array_equal(plan.offsets.cpu().numpy(), P["offsets"])
    assert np.array_equal(plan.perm.cpu().numpy(), P["perm"])
    n = int(plan.n_active.cpu().numpy()[0])
    assert n == P["n_active"]
    assert np.array_equal(plan.active.cpu().numpy()[:n], P["active"])


def _run_full(m, wl, L, x_cpu, *, layer=0, sample=None, gamma=None, max_tokens=None,
              tol=TOL, cache=None, handle=None, report=None):
    """Forward x on the GPU with a plan; compare routing bit for bit and y."""
    sh = wl.shape
    T = x_cpu.shape[0]
    own = handle is None
    h = handle or m.MoELayer(L, max_tokens or T)
    x = x_cpu.to(DEV)
    g = gamma.to(DEV) if gamma is not None else None
    plan = m.Plan(T, sh.top_k, sh.n_experts, DEV)
    y = h.forward(x, gamma=g, eps=RMS_EPS, plan=plan)
    torch.cuda.synchronize()
    assert m.moe_device_status(h.h) == 0
    x32 = x_cpu.float().numpy()
    eps = RMS_EPS if gamma is not None else 0.0
    gnp = gamma.numpy() if gamma is not None else None
    router = router_of(wl, layer)
    _, _, ids_o, w_o = oracle.route(sh, router[0], router[1], x32, eps, gnp)
    ids = plan.topk_ids.cpu().numpy()
    wts = plan.topk_w.cpu().numpy()
    assert np.array_equal(ids, ids_o), (ids, ids_o)
    assert np.array_equal(wts.view(np.uint32), w_o.view(np.uint32))
    _check_plan(plan, ids_o, sh.n_experts)
    tokens = list(range(T)) if sample is None else [t for t in sample if t < T]
    y_o, _, _, _ = oracle_layer(wl, layer, router, x32, tokens, eps=eps, gamma=gnp, cache=cache)
    err = rel_err_per_token(y.cpu().numpy()[tokens], y_o)
    if report is not None:
        # the gate is the per-token figure; the element-wise one is reported
        ee = elem_err_per_token(y.cpu().numpy()[tokens], y_o)
        report(f"{wl.name}_T{T}", float(err.max()), float(ee.max()))
    assert err.max() <= tol, err
    if own:
        h.close()
    return y, plan, err


# ------------------------------------------------------------------ tiny layer

@pytest.mark.parametrize("T", [1, 2, 3, 17, 64, 100])
def test_tiny_layer(m, T):
    wl = CONFIGS["tiny"]
    L = gen_layer(wl, device=DEV)
    x = gen_activations(wl, T, call=T)
    _run_full(m, wl, L, x, tol=1e-4)


# ------------------------------------------------------------- shape sweep ---

SHAPES = [
    # H, I, E, k, n_group, topk_group, n_shared  (I % 64 == 0, I <= 2048 takes
    # the fused single-token kernel for T = 1; T > 1 with I % 256 == 0 takes
    # the grouped GEMM)
    (256, 256, 32, 4, 4, 2, 1),
    (512, 512, 64, 6, 8, 3, 1),
    (1024, 256, 128, 8, 8, 4, 1),
    (2048, 1024, 256, 8, 8, 4, 1),
    (1024, 512, 64, 4, 2, 1, 0),
    (256, 256, 32, 4, 32, 8, 1),    # one expert per group
    (768, 96, 27, 5, 9, 3, 1),      # general path only
    (256, 128, 1024, 8, 8, 4, 1),   # 1024 experts
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("T", [1, 3, 4, 9])
def test_shape_sweep(m, shape, T):
    H, I, E, k, ng, tg, ns = shape
    sh = LayerShape(H, I, E, k, ng, tg, 1.5, n_shared=ns)
    wl = Workload("sweep", sh, T, 1, "bf16" if T % 2 else "f32", "uniform",
                  7000 + H + I + E + k)
    L = gen_layer(wl, device=DEV)
    x = gen_activations(wl, T, call=0)
    _run_full(m, wl, L, x, max_tokens=max(T, 16))


LIMIT_CASES = [
    # H, I, E, k, n_group, topk_group, tokens per call: the largest hidden size
    # on the single-token tensor-core kernel (T = 1) and the grouped GEMM
    # (T = 2), and on the SIMT path (I = 96); the largest top_k (32 experts a
    # token: the single-token SIMT kernel at T = 1, the grouped GEMM at T = 6);
    # every expert selected (k = E); a single expert; a single group
    (12288, 1024, 32, 4, 4, 2, (1, 2)),
    (12288, 96, 16, 4, 4, 2, (1, 3)),
    (1024, 512, 64, 32, 4, 4, (1, 6)),
    (512, 256, 8, 8, 2, 2, (1, 4)),
    (256, 256, 1, 1, 1, 1, (1, 3)),
    (512, 256, 64, 8, 1, 1, (1, 2)),
]


@pytest.mark.parametrize("case", LIMIT_CASES, ids=lambda c: "x".join(map(str, c[:6])))
def test_limits_and_degenerate_routing(m, case):
    H, I, E, k, ng, tg, Ts = case
    sh = LayerShape(H, I, E, k, ng, tg, 2.5)
    wl = Workload("limits", sh, max(Ts), 1, "bf16", "zipf" if E >= 32 else "uniform",
                  7900 + H + I + E + k)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, max(Ts))
    for T in Ts:
        _run_full(m, wl, L, gen_activations(wl, T, call=T), handle=h)
    h.close()


def test_small_batch_with_rmsnorm(m):
    sh = LayerShape(1024, 512, 64, 6, 8, 3, 2.0)
    wl = Workload("norm", sh, 2, 1, "f32", "zipf", 7101, rmsnorm_eps=1e-5)
    L = gen_layer(wl, device=DEV)
    for T in (1, 2, 4):
        x = gen_activations(wl, T, call=T) * 3.0
        _run_full(m, wl, L, x, gamma=gen_norm_weight(wl, 0), max_tokens=8)


# -------------------------------------------------------- API behaviour ------

def _tiny_handle(m, max_tokens=8):
    wl = CONFIGS["tiny"]
    L = gen_layer(wl, device=DEV)
    return wl, L, m.MoELayer(L, max_tokens)


def test_device_status_clean(m):
    wl, L, h = _tiny_handle(m)
    h.forward(gen_activations(wl, 2, call=1).to(DEV))
    torch.cuda.synchronize()
    assert m.moe_device_status(h.h) == 0
    h.close()


def test_create_refuses_weights_outside_device_memory(m):
    """A weight array in host memory (pageable or pinned) is refused at create
    time with MOE_ERR_INVALID_ARG, naming the array; nothing is launched.  The
    same weights on the device are accepted."""
    wl = CONFIGS["tiny"]
    L = gen_layer(wl, device=DEV)
    cfg = m.moe.config_for(L.shape, 1)
    nbytes = L.gate_q.numel() + 16
    pageable = np.zeros(nbytes, dtype=np.uint8)
    pinned = torch.zeros(nbytes, dtype=torch.uint8, pin_memory=True)
    for addr in (pageable.ctypes.data, pinned.data_ptr()):
        w = m.moe.weights_for(L)
        w.gate_q = (addr + 15) & ~15
        with pytest.raises(m.MoeError) as e:
            m.moe_layer_create(cfg, w)
        assert e.value.status == m.moe.MOE_ERR_INVALID_ARG
        assert "gate_q" in str(e.value) and "device memory" in str(e.value)
    h = m.moe_layer_create(cfg, m.moe.weights_for(L))
    m.moe_destroy(h)


def test_bounded_wait_gives_up_and_device_stays_usable(m):
    """A wait that can never complete (grid-barrier counter below its target,
    mbarrier phase nobody arrives on) gives up after about one second, sets
    bit 0 of the error word, and leaves the device usable."""
    for which in (0, 1):
        assert m.moe_selftest_bounded_wait(which) & 1 == 1
    wl, L, h = _tiny_handle(m, 4)
    _run_full(m, wl, L, gen_activations(wl, 3, call=2), handle=h)
    h.close()


def test_handle_recovers_after_a_call_gives_up(m):
    """A call whose grid barrier cannot complete gives up (bit 0); the status
    call reports it and resets the barrier state; the next calls (one token,
    then a small batch through the routing front end) are correct again."""
    sh = LayerShape(1024, 512, 64, 6, 8, 3, 2.0)
    wl = Workload("recover", sh, 1, 1, "bf16", "zipf", 7606)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 4)
    _run_full(m, wl, L, gen_activations(wl, 1, call=0), handle=h)
    m.moe_selftest_desync(h.h)
    h.forward(gen_activations(wl, 1, call=1).to(DEV))
    torch.cuda.synchronize()
    with pytest.raises(m.MoeError):
        m.moe_device_status(h.h)
    _run_full(m, wl, L, gen_activations(wl, 1, call=2), handle=h)
    _run_full(m, wl, L, gen_activations(wl, 3, call=3), handle=h)
    h.close()


def test_zero_tokens_is_noop(m):
    wl, L, h = _tiny_handle(m)
    x = torch.zeros(0, wl.shape.hidden, device=DEV)
    y = torch.full((1, wl.shape.hidden), 7.0, device=DEV)
    m.moe_forward(h.h, x.data_ptr() if x.numel() else y.data_ptr(), m.MOE_F32, 0,
                  y.data_ptr(), None, 0.0, 0, None, None)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    h.close()


def test_capacity_and_argument_errors(m):
    wl, L, h = _tiny_handle(m, max_tokens=4)
    H = wl.shape.hidden
    x = torch.randn(5, H, device=DEV)
    with pytest.raises(m.MoeError) as ei:
        h.forward(x)
    assert ei.value.status == -3
    buf = torch.zeros(4 * H + 4, device=DEV)
    with pytest.raises(m.MoeError) as ei:  # misaligned x
        m.moe_forward(h.h, buf.data_ptr() + 4, m.MOE_F32, 1, buf.data_ptr() + 4 * H * 2,
                      None, 0.0, 0, None, None)
    assert ei.value.status == -1
    xx = torch.randn(2, H, device=DEV)
    with pytest.raises(m.MoeError) as ei:  # overlap outside the residual form
        m.moe_forward(h.h, xx.data_ptr(), m.MOE_F32, 2, xx.data_ptr(), None, 0.0, 1, None, None)
    assert ei.value.status == -1
    with pytest.raises(m.MoeError) as ei:
        m.moe_forward(h.h, xx.data_ptr(), 7, 2, buf.data_ptr(), None, 0.0, 0, None, None)
    assert ei.value.status == -1
    # the binding refuses tensors the kernels would read or write out of
    # bounds, before the C call
    bad = [dict(x=xx.cpu()), dict(x=xx[:, : H // 2]), dict(x=torch.randn(H, 2, device=DEV).t()),
           dict(x=xx, y=torch.empty(1, H, device=DEV)),
           dict(x=xx, y=torch.empty(2, H, device=DEV, dtype=torch.bfloat16)),
           dict(x=xx, gamma=torch.ones(H // 2, device=DEV)),
           dict(x=xx, plan=m.Plan(1, wl.shape.top_k, wl.shape.n_experts, DEV))]
    for kw in bad:
        with pytest.raises(ValueError):
            h.forward(**kw)
    with pytest.raises(ValueError):
        h.route(xx, plan=m.Plan(2, wl.shape.top_k, wl.shape.n_experts, "cpu"))
    h.close()


def test_deterministic_repeat(m):
    sh = LayerShape(1024, 512, 64, 6, 8, 3, 2.0)
    wl = Workload("det", sh, 4, 1, "bf16", "zipf", 7202)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 64)
    for T in (1, 4, 33):
        x = gen_activations(wl, T, call=T).to(DEV)
        y1 = h.forward(x).clone()
        y2 = h.forward(x).clone()
        assert torch.equal(y1, y2)
    h.close()


def test_route_matches_forward_plan(m):
    sh = LayerShape(512, 512, 64, 6, 8, 3, 2.0)
    wl = Workload("route", sh, 4, 1, "bf16", "zipf", 7303)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 64)
    for T in (1, 3, 40):
        x = gen_activations(wl, T, call=T).to(DEV)
        p1 = h.route(x)
        p2 = m.Plan(T, sh.top_k, sh.n_experts, DEV)
        h.forward(x, plan=p2)
        torch.cuda.synchronize()
        for name in ("topk_ids", "topk_w", "counts", "offsets", "perm", "n_active"):
            assert torch.equal(getattr(p1, name), getattr(p2, name)), name
        n = int(p1.n_active.item())
        assert torch.equal(p1.active[:n], p2.active[:n])
    h.close()


def test_residual_in_place(m):
    for sh in (CONFIGS["tiny"].shape, LayerShape(1024, 512, 64, 6, 8, 3, 2.0)):
        wl = Workload("resid", sh, 3, 1, "f32", "zipf", 7404, rmsnorm_eps=1e-5)
        L = gen_layer(wl, device=DEV)
        h = m.MoELayer(L, 8)
        gamma = gen_norm_weight(wl, 0)
        for T in (1, 3, 6):
            x0 = (gen_activations(wl, T, call=T) * 2.0).float()
            xd = x0.to(DEV)
            h.forward(xd, y=xd, gamma=gamma.to(DEV), eps=RMS_EPS, accumulate=True)
            torch.cuda.synchronize()
            y_o, _, _, _ = oracle_layer(wl, 0, router_of(wl), x0.numpy(), range(T), eps=RMS_EPS,
                                        gamma=gamma.numpy(), resid=x0.numpy())
            err = resid_err_per_token(xd.cpu().numpy(), y_o, x0.numpy())
            assert err.max() <= TOL
        h.close()


def test_trace_phases(m):
    sh = LayerShape(1024, 512, 64, 6, 8, 3, 2.0)
    wl = Workload("trace", sh, 4, 1, "bf16", "zipf", 7505)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 64)
    m.moe_trace_enable(h.h, 3)
    h.forward(gen_activations(wl, 1, call=0).to(DEV))
    h.forward(gen_activations(wl, 20, call=1).to(DEV))
    h.forward(gen_activations(wl, 3, call=2).to(DEV))
    names, rows = m.moe_trace_read(h.h, 3)
    assert len(rows) == 3 and len(names) == 12
    small = {n for n, v in zip(names, rows[0]) if v > 0}
    tc = {n for n, v in zip(names, rows[1]) if v > 0}
    assert small == {"decode_fused"}
    assert tc == {"prep", "router_logits", "select", "plan", "tc_prep", "tc_gate_up", "tc_down",
                  "combine"}
    batch = {n for n, v in zip(names, rows[2]) if v > 0}
    # small batches: routing in one cooperative kernel, then the grouped GEMM
    assert batch == {"tc_front", "tc_gate_up", "tc_down", "combine"}
    m.moe_trace_enable(h.h, 0)
    h.close()
    # intermediate size not a multiple of 256: the SIMT general path
    wl, L, h = _tiny_handle(m, 32)
    m.moe_trace_enable(h.h, 1)
    h.forward(gen_activations(wl, 20, call=1).to(DEV))
    names, rows = m.moe_trace_read(h.h, 1)
    general = {n for n, v in zip(names, rows[0]) if v > 0}
    assert general == {"prep", "router_logits", "select", "plan", "gate_up", "down", "combine"}
    m.moe_trace_enable(h.h, 0)
    h.close()


# ------------------------------------------------ tensor-core grouped GEMM ---

TC_SHAPES = [
    # H, I, E, k, n_group, topk_group, n_shared, shared_inter (0: = I)
    (512, 256, 16, 4, 4, 2, 1, 0),
    (1024, 512, 8, 2, 2, 1, 1, 768),   # shared expert wider than the routed ones
    (256, 256, 8, 2, 2, 1, 0, 0),      # no shared expert
    (768, 256, 32, 6, 8, 4, 1, 512),
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("T", [3, 5, 40, 150, 300])
def test_tc_grouped_gemm(m, shape, T):
    """T = 3 takes the small-batch routing front end where the shape allows
    (32 experts: 768 x 256 with a 512-wide shared expert), the five routing
    kernels otherwise; T = 300 gives most shapes >= 64 rows per expert, which
    selects 128-row chunks (N = 128 MMAs)."""
    H, I, E, k, ng, tg, ns, Is = shape
    sh = LayerShape(H, I, E, k, ng, tg, 2.5, n_shared=ns, shared_inter=Is)
    wl = Workload("tc", sh, T, 1, "bf16" if T % 2 else "f32", "zipf", 7700 + H + I + E + T)
    L = gen_layer(wl, device=DEV)
    x = gen_activations(wl, T, call=0)
    _run_full(m, wl, L, x, max_tokens=T + 3)


def test_single_token_wide_intermediate(m):
    """One token with an intermediate size the SIMT single-token kernel
    does not keep in registers (I = 4096): with H a multiple of 1024 the
    tensor-core single-token kernel takes it; with H = 512 the grouped GEMM."""
    sh = LayerShape(1024, 4096, 32, 4, 4, 2, 2.5)
    wl = Workload("tc_t1", sh, 1, 1, "bf16", "zipf", 7803)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 2)
    m.moe_trace_enable(h.h, 1)
    _run_full(m, wl, L, gen_activations(wl, 1, call=0), handle=h)
    names, rows = m.moe_trace_read(h.h, 1)
    assert {n for n, v in zip(names, rows[0]) if v > 0} == {"decode_fused"}
    h.close()
    sh = LayerShape(512, 4096, 32, 4, 4, 2, 2.5)
    wl = Workload("tc_t1b", sh, 1, 1, "bf16", "zipf", 7804)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 2)
    m.moe_trace_enable(h.h, 1)
    _run_full(m, wl, L, gen_activations(wl, 1, call=0), handle=h)
    names, rows = m.moe_trace_read(h.h, 1)
    assert "tc_gate_up" in {n for n, v in zip(names, rows[0]) if v > 0}
    m.moe_trace_enable(h.h, 0)
    h.close()


def test_tc_multi_chunk_experts(m):
    """Experts with more than 64 rows (several chunks) and a 300-token
    shared expert (five chunks, the last one ragged)."""
    sh = LayerShape(512, 256, 4, 2, 1, 1, 2.5)
    wl = Workload("tc_chunks", sh, 300, 1, "bf16", "zipf", 7801)
    L = gen_layer(wl, device=DEV)
    x = gen_activations(wl, 300, call=0)
    _, plan, _ = _run_full(m, wl, L, x, sample=list(range(0, 300, 7)) + [299])
    assert plan.counts.cpu().numpy().max() > 128


def test_tc_rmsnorm_residual(m):
    sh = LayerShape(512, 512, 16, 4, 4, 2, 2.5)
    wl = Workload("tc_resid", sh, 24, 1, "f32", "zipf", 7802, rmsnorm_eps=1e-5)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 64)
    gamma = gen_norm_weight(wl, 0)
    for T in (9, 64):
        x0 = (gen_activations(wl, T, call=T) * 2.0).float()
        xd = x0.to(DEV)
        h.forward(xd, y=xd, gamma=gamma.to(DEV), eps=RMS_EPS, accumulate=True)
        torch.cuda.synchronize()
        assert m.moe_device_status(h.h) == 0
        y_o, _, _, _ = oracle_layer(wl, 0, router_of(wl), x0.numpy(), range(T), eps=RMS_EPS,
                                    gamma=gamma.numpy(), resid=x0.numpy())
        err = resid_err_per_token(xd.cpu().numpy(), y_o, x0.numpy())
        assert err.max() <= TOL
    h.close()


# ------------------------------------- single-token tensor-core kernel ---

DM_SHAPES = [
    # H, I, E, k, n_group, topk_group, n_shared: H and I multiples of 1024
    # with I beyond what the SIMT single-token kernel keeps in registers
    # (I > 2048) take the single-token tensor-core kernel at T = 1
    (1024, 3072, 32, 4, 4, 2, 1),    # fewer blocks and tiles than CTAs
    (2048, 4096, 64, 6, 8, 3, 1),    # blocks and tiles cut by CTA ranges
    (3072, 3072, 32, 8, 4, 2, 1),
    (2048, 4096, 32, 4, 8, 4, 0),    # no shared expert
]


@pytest.mark.parametrize("shape", DM_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_token_tensor_core(m, shape, dtype):
    H, I, E, k, ng, tg, ns = shape
    sh = LayerShape(H, I, E, k, ng, tg, 2.5, n_shared=ns)
    wl = Workload("dm", sh, 1, 1, dtype, "uniform", 9100 + H + I + E + k)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 1)
    m.moe_trace_enable(h.h, 4)
    # several calls of one handle: grid-barrier targets and part counters
    for call in range(4):
        _run_full(m, wl, L, gen_activations(wl, 1, call=call), handle=h)
    names, rows = m.moe_trace_read(h.h, 4)
    for row in rows:
        assert {n for n, v in zip(names, row) if v > 0} == {"decode_fused"}
    m.moe_trace_enable(h.h, 0)
    h.close()


def test_single_token_tensor_core_rmsnorm_residual(m):
    sh = LayerShape(2048, 3072, 64, 6, 8, 3, 2.0)
    wl = Workload("dm_resid", sh, 1, 1, "f32", "zipf", 9201, rmsnorm_eps=1e-5)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 4)
    gamma = gen_norm_weight(wl, 0)
    for call in range(3):
        x0 = (gen_activations(wl, 1, call=call) * 2.0).float()
        xd = x0.to(DEV)
        h.forward(xd, y=xd, gamma=gamma.to(DEV), eps=RMS_EPS, accumulate=True)
        torch.cuda.synchronize()
        assert m.moe_device_status(h.h) == 0
        y_o, _, _, _ = oracle_layer(wl, 0, router_of(wl), x0.numpy(), [0], eps=RMS_EPS,
                                    gamma=gamma.numpy(), resid=x0.numpy())
        err = resid_err_per_token(xd.cpu().numpy(), y_o, x0.numpy())
        assert err.max() <= TOL, err
    h.close()


def test_single_token_tensor_core_deterministic(m):
    sh = LayerShape(3072, 4096, 32, 8, 4, 2, 2.5)
    wl = Workload("dm_det", sh, 1, 1, "bf16", "zipf", 9202)
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 1)
    x = gen_activations(wl, 1, call=0).to(DEV)
    y1 = h.forward(x).clone()
    for _ in range(3):
        assert torch.equal(h.forward(x), y1)
    h.close()


# -------------------------------------------------- GLM-5.2-shaped layers ----

_GLM_CACHE: dict = {}


def _glm(name):
    if name not in _GLM_CACHE:
        _GLM_CACHE.clear()
        torch.cuda.empty_cache()
        wl = CONFIGS[name]
        _GLM_CACHE[name] = (wl, gen_layer(wl, device=DEV), HostExpertCache(wl))
    return _GLM_CACHE[name]


@pytest.fixture
def report(record_property):
    """Records (and prints) the gated per-token error and the element-wise
    companion figure of a parity case."""
    def rec(name, per_token, elementwise):
        record_property(f"{name}_per_token", per_token)
        record_property(f"{name}_elementwise", elementwise)
        print(f"parity {name}: per-token {per_token:.3e}, element-wise {elementwise:.3e}")
    return rec


def test_glm_decode_tokens(m, report):
    """Outputs of three tokens against the oracle; the routing (ids, gate
    weights, plan) of all 256 tokens of the benchmark's decode step."""
    wl, L, cache = _glm("glm_decode")
    h = m.MoELayer(L, 1)
    for call in (0, 1, 2):
        x = gen_activations(wl, 1, call=call)
        _run_full(m, wl, L, x, cache=cache, handle=h, report=report)
    router = router_of(wl, 0)
    sh = wl.shape
    plan = m.Plan(1, sh.top_k, sh.n_experts, DEV)
    for call in range(wl.calls):
        x = gen_activations(wl, 1, call=call)
        h.forward(x.to(DEV), plan=plan)
        _, _, ids_o, w_o = oracle.route(sh, router[0], router[1], x.float().numpy())
        assert np.array_equal(plan.topk_ids.cpu().numpy(), ids_o), call
        assert np.array_equal(plan.topk_w.cpu().numpy().view(np.uint32), w_o.view(np.uint32))
        _check_plan(plan, ids_o, sh.n_experts)
    assert m.moe_device_status(h.h) == 0
    h.close()


def test_glm_verify_batch(m, report):
    wl, L, cache = _glm("glm_verify")
    x = gen_activations(wl, 4, call=0)
    _run_full(m, wl, L, x, cache=cache, report=report)


def test_glm_prefill_sampled(m, report):
    wl, L, cache = _glm("glm_prefill")
    x = gen_activations(wl, 512, call=0)
    _, plan, _ = _run_full(m, wl, L, x, sample=[0, 1, 77, 255, 300, 511], cache=cache,
                           report=report)
    counts = plan.counts.cpu().numpy()
    assert counts.max() >= 40 and (counts == 0).sum() >= 1  # uneven, Zipf-skewed load


def test_glm_ragged_batch(m):
    wl, L, cache = _glm("glm_prefill")
    x = gen_activations(wl, 37, call=5)
    _run_full(m, wl, L, x, sample=[0, 18, 36], cache=cache, max_tokens=64)


def test_glm_stack_teacher_forced(m):
    """24 resident layers, RMSNorm + residual, one token; layers checked
    against the oracle on the GPU's own layer inputs."""
    _GLM_CACHE.clear()
    torch.cuda.empty_cache()
    wl = CONFIGS["glm_stack"]
    free, _ = torch.cuda.mem_get_info()
    per = 5.6e9
    n_layers = wl.layers if free > per * wl.layers + 20e9 else max(2, int((free - 20e9) // per))
    layers = [gen_layer(wl, layer=i, device=DEV) for i in range(n_layers)]
    handles = [m.MoELayer(L, 1) for L in layers]
    gammas = [gen_norm_weight(wl, i).to(DEV) for i in range(n_layers)]
    x = gen_activations(wl, 1, call=0, dtype="f32").to(DEV)
    check = sorted({0, 1, n_layers // 2, n_layers - 1})
    inputs = {}
    for i in range(n_layers):
        if i in check:
            inputs[i] = x.clone()
        handles[i].forward(x, y=x, gamma=gammas[i], eps=RMS_EPS, accumulate=True)
    torch.cuda.synchronize()
    final = x.cpu().numpy()
    assert np.all(np.isfinite(final))
    for i in check:
        x_in = inputs[i].cpu().numpy()
        g = gammas[i].cpu().numpy()
        xd = inputs[i].clone()
        plan = m.Plan(1, wl.shape.top_k, wl.shape.n_experts, DEV)
        handles[i].forward(xd, y=xd, gamma=gammas[i], eps=RMS_EPS, accumulate=True, plan=plan)
        torch.cuda.synchronize()
        router = router_of(wl, i)
        y_o, ids_o, w_o, _ = oracle_layer(wl, i, router, x_in, [0], eps=RMS_EPS, gamma=g,
                                          resid=x_in)
        assert np.array_equal(plan.topk_ids.cpu().numpy(), ids_o)
        assert np.array_equal(plan.topk_w.cpu().numpy().view(np.uint32), w_o.view(np.uint32))
        err = resid_err_per_token(xd.cpu().numpy(), y_o, x_in)
        assert err.max() <= TOL, (i, err)
    for h in handles:
        h.close()


def test_two_handles_after_a_larger_shared_memory_shape(m):
    """The single-token kernel's shared-memory opt-in is kept per kernel and
    device: a handle whose shape needs more dynamic shared memory runs first,
    then a handle of a smaller shape on the same device, then the first one
    again; every call matches the oracle."""
    big = LayerShape(6144, 1024, 64, 4, 4, 2, 2.5)    # ~197 KB: x_hat and rings of H = 6144
    small = LayerShape(1024, 512, 32, 4, 4, 2, 2.5)
    wb = Workload("smem_big", big, 1, 1, "bf16", "zipf", 9601)
    ws_ = Workload("smem_small", small, 1, 1, "bf16", "zipf", 9602)
    Lb, Ls = gen_layer(wb, device=DEV), gen_layer(ws_, device=DEV)
    hb, hs = m.MoELayer(Lb, 1), m.MoELayer(Ls, 1)
    for wl, L, h in ((wb, Lb, hb), (ws_, Ls, hs), (wb, Lb, hb), (ws_, Ls, hs)):
        m.moe_trace_enable(h.h, 1)
        _run_full(m, wl, L, gen_activations(wl, 1, call=0), handle=h)
        names, rows = m.moe_trace_read(h.h, 1)
        m.moe_trace_enable(h.h, 0)
        assert {n for n, v in zip(names, rows[0]) if v > 0} == {"decode_fused"}
    hb.close()
    hs.close()


def test_pinned_host_inputs_and_outputs(m):
    """x and y in pinned host memory (read and written by the kernels across
    the host link) give the same outputs bit for bit as device buffers, on
    the single-token kernel (T = 1), the routing front end (T = 3), the
    routing kernels with the grouped GEMM (T = 9) and the SIMT batch path
    (an int8 layer); unpinned host memory is refused before any launch."""
    import ctypes as C
    cases = [(LayerShape(1024, 512, 64, 6, 8, 3, 2.5), (1, 3, 9)),
             (LayerShape(512, 256, 32, 4, 4, 2, 2.5, weight_format="int8"), (1, 9))]
    for sh, Ts in cases:
        wl = Workload("pinned_io", sh, 9, 1, "bf16", "zipf", 9801)
        L = gen_layer(wl, device=DEV)
        h = m.MoELayer(L, 16)
        for T in Ts:
            x = gen_activations(wl, T, call=T)
            y_dev = h.forward(x.to(DEV))
            xh = x.pin_memory()
            yh = torch.empty(T, sh.hidden, dtype=torch.float32).pin_memory()
            h.forward(xh, y=yh)
            torch.cuda.synchronize()
            assert torch.equal(yh, y_dev.cpu()), (sh, T)
        assert m.moe_device_status(h.h) == 0
        # the binding refuses unpinned host tensors ...
        with pytest.raises(ValueError):
            h.forward(gen_activations(wl, 1, call=0))
        # ... and the C ABI refuses unregistered host memory before a launch
        buf = np.zeros((1, sh.hidden), np.float32)
        yd = torch.empty(1, sh.hidden, dtype=torch.float32, device=DEV)
        st = m.load().moe_forward(h.h, C.c_void_p(buf.ctypes.data), m.MOE_F32, 1,
                                  C.c_void_p(yd.data_ptr()), None, C.c_float(0.0), 0, None, None)
        assert st == -1 and "pinned host memory" in m.moe_last_error(h.h)
        h.close()
