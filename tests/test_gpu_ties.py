"""The selection's tie rules on every CUDA selection implementation.

The rule is fixed by "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri
hierarchy", "G2 implementation status": on an exact tie of selection keys the
lower expert id wins.  Groups tied on their score go to the lower group index
(the group reading of the router).  Random fp32 keys almost never tie, so these
cases build ties on purpose: a zero router weight makes every logit exactly 0
and every score sigmoid(0) = 0.5 exactly, and biases that are binary fractions
make the keys 0.5 + b exact in fp32.  Each case is routed through every kernel
that selects experts, and ids, gate weights (as bits) and the whole plan are
compared with the CPU oracle; where the call also runs the experts, the output
is compared too.

Which kernel selects depends on the call (the library's path choice):
  T = 1                  the single-token kernels (CTA 0 selects and publishes)
  T = 3                  the small-batch routing front end
  T = 9, moe_route       the register selection kernel (E <= 512)
  E = 1024               the shared-memory selection kernel
  moe_route_noalloc      the same router kernels with static scratch
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, oracle_layer, rel_err_per_token
from tie_cases import KINDS, expected_ids_t1, tie_bias
from workloads.configs import LayerShape, Workload
from workloads.gen import gen_activations, gen_layer

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


def _tie_layer(shape, seed, bias):
    wl = Workload("ties", shape, 16, 1, "bf16", "uniform", seed)
    L = gen_layer(wl, device=DEV)
    L.router_w.zero_()
    L.router_b.copy_(torch.from_numpy(bias))
    router = (np.zeros((shape.n_experts, shape.hidden), np.float32), bias)
    return wl, L, router


def _check_routing(plan, shape, router, x32):
    _, _, ids_o, w_o = oracle.route(shape, router[0], router[1], x32)
    ids = plan.topk_ids.cpu().numpy()
    wts = plan.topk_w.cpu().numpy()
    assert np.array_equal(ids, ids_o), (ids, ids_o)
    assert np.array_equal(wts.view(np.uint32), w_o.view(np.uint32))
    P = oracle.plan(ids_o, shape.n_experts)
    assert np.array_equal(plan.counts.cpu().numpy(), P["counts"])
    assert np.array_equal(plan.offsets.cpu().numpy(), P["offsets"])
    assert np.array_equal(plan.perm.cpu().numpy(), P["perm"])
    n = int(plan.n_active.cpu().numpy()[0])
    assert n == P["n_active"]
    assert np.array_equal(plan.active.cpu().numpy()[:n], P["active"])
    return ids_o


def _forward_checked(m, h, wl, L, router, x_cpu, expect_phases, check_y=True):
    sh = wl.shape
    T = x_cpu.shape[0]
    x = x_cpu.to(DEV)
    plan = m.Plan(T, sh.top_k, sh.n_experts, DEV)
    m.moe_trace_enable(h.h, 1)
    y = h.forward(x, plan=plan)
    torch.cuda.synchronize()
    names, rows = m.moe_trace_read(h.h, 1)
    m.moe_trace_enable(h.h, 0)
    ran = {n for n, v in zip(names, rows[0]) if v > 0}
    assert expect_phases <= ran, (expect_phases, ran)
    assert m.moe_device_status(h.h) == 0
    x32 = x_cpu.float().numpy()
    ids = _check_routing(plan, sh, router, x32)
    if check_y:
        y_o, _, _, _ = oracle_layer(wl, 0, router, x32, list(range(T)))
        err = rel_err_per_token(y.cpu().numpy(), y_o)
        assert err.max() <= TOL, err
    return ids


@pytest.mark.parametrize("kind", KINDS)
def test_ties_single_token_and_small_batches(m, kind):
    """E = 256, top-8, 8 groups, 4 kept: T = 1 (single-token kernel), T = 3
    (routing front end), T = 9 (register selection), moe_route and
    moe_route_noalloc."""
    sh = LayerShape(1024, 256, 256, 8, 8, 4, 2.5)
    bias = tie_bias(sh.n_experts, sh.n_group, kind)
    wl, L, router = _tie_layer(sh, 9100, bias)
    h = m.MoELayer(L, 16)
    ids = _forward_checked(m, h, wl, L, router, gen_activations(wl, 1, call=0),
                           {"decode_fused"})
    # the worked expectation, by hand from the rule, beside the oracle
    assert list(ids[0]) == expected_ids_t1(kind, sh.n_experts, sh.n_group, sh.top_k)
    _forward_checked(m, h, wl, L, router, gen_activations(wl, 3, call=1), {"tc_front"})
    _forward_checked(m, h, wl, L, router, gen_activations(wl, 9, call=2), {"select"})
    x = gen_activations(wl, 5, call=3)
    plan = h.route(x.to(DEV), plan=m.Plan(5, sh.top_k, sh.n_experts, DEV))
    torch.cuda.synchronize()
    _check_routing(plan, sh, router, x.float().numpy())
    cfg = m.moe.config_for(sh, 16)
    p2 = m.Plan(5, sh.top_k, sh.n_experts, DEV)
    xd = x.to(DEV)
    m.moe_route_noalloc(cfg, L.router_w.data_ptr(), L.router_b.data_ptr(), xd.data_ptr(),
                        m.MOE_BF16, 5, None, 0.0, p2.c(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    _check_routing(p2, sh, router, x.float().numpy())
    h.close()


@pytest.mark.parametrize("kind", KINDS)
def test_ties_single_token_wide_intermediate(m, kind):
    """I = 3072 (the single-token tensor-core kernel's shapes)."""
    sh = LayerShape(1024, 3072, 256, 8, 8, 4, 2.5)
    bias = tie_bias(sh.n_experts, sh.n_group, kind)
    wl, L, router = _tie_layer(sh, 9200, bias)
    h = m.MoELayer(L, 4)
    ids = _forward_checked(m, h, wl, L, router, gen_activations(wl, 1, call=0),
                           {"decode_fused"})
    assert list(ids[0]) == expected_ids_t1(kind, sh.n_experts, sh.n_group, sh.top_k)
    h.close()


@pytest.mark.parametrize("kind", KINDS)
def test_ties_1024_experts(m, kind):
    """E = 1024 (128 experts a group): the shared-memory selection kernel."""
    sh = LayerShape(256, 256, 1024, 8, 8, 4, 2.5)
    bias = tie_bias(sh.n_experts, sh.n_group, kind)
    wl, L, router = _tie_layer(sh, 9300, bias)
    h = m.MoELayer(L, 16)
    for T in (1, 9):
        ids = _forward_checked(m, h, wl, L, router, gen_activations(wl, T, call=T), {"select"}
                               if T > 4 else set())
        if T == 1:
            assert list(ids[0]) == expected_ids_t1(kind, sh.n_experts, sh.n_group, sh.top_k)
    h.close()
