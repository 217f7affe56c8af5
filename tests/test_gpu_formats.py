"""GPU parity of the other expert formats: signed int8 weights and one fp16
scale per row ("GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri
hierarchy", N2 and "G2 implementation status").

Routing is compared bit for bit with the oracle, the outputs within the
parity tolerance; the kernels each call ran are checked from the trace:
per-row int4 on the single-token SIMT kernel (T = 1) and the tensor-core
grouped GEMM (T > 1); int8 on the SIMT batch path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from parity_util import RMS_EPS, TOL, oracle_layer, resid_err_per_token, router_of
from workloads import CONFIGS
from workloads.configs import LayerShape, Workload
from workloads.gen import gen_activations, gen_layer, gen_norm_weight

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SIMT = {"prep", "router_logits", "select", "plan", "gate_up", "down", "combine"}


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_routed_expert_gb300 import build as b
    b.build()
    import int4_routed_expert_gb300 as mod
    mod.load()
    return mod


def _check(m, h, wl, L, x_cpu, expect):
    """expect: the exact set of phases, or a callable judging the set."""
    sh = wl.shape
    T = x_cpu.shape[0]
    plan = m.Plan(T, sh.top_k, sh.n_experts, DEV)
    m.moe_trace_enable(h.h, 1)
    y = h.forward(x_cpu.to(DEV), plan=plan)
    torch.cuda.synchronize()
    names, rows = m.moe_trace_read(h.h, 1)
    m.moe_trace_enable(h.h, 0)
    ran = {n for n, v in zip(names, rows[0]) if v > 0}
    assert expect(ran) if callable(expect) else ran == expect, ran
    assert m.moe_device_status(h.h) == 0
    router = router_of(wl, 0)
    x32 = x_cpu.float().numpy()
    _, _, ids_o, w_o = oracle.route(sh, router[0], router[1], x32)
    assert np.array_equal(plan.topk_ids.cpu().numpy(), ids_o)
    assert np.array_equal(plan.topk_w.cpu().numpy().view(np.uint32), w_o.view(np.uint32))
    y_o, _, _, _ = oracle_layer(wl, 0, router, x32, list(range(T)))
    err = np.abs(y.cpu().numpy().astype(np.float64) - y_o).max(axis=1) / \
        np.maximum(np.abs(y_o).max(axis=1), 1e-30)
    assert err.max() <= TOL, err
    return y


FORMATS = [("int4", 0), ("int8", 32), ("int8", 0)]


@pytest.mark.parametrize("fmt,gsz", FORMATS, ids=lambda v: str(v))
@pytest.mark.parametrize("shape", [(512, 256, 32, 4, 4, 2, 1), (1024, 512, 64, 6, 8, 3, 0)],
                         ids=lambda s: "x".join(map(str, s)))
def test_formats_match_the_oracle(m, fmt, gsz, shape):
    H, I, E, k, ng, tg, ns = shape
    sh = LayerShape(H, I, E, k, ng, tg, 2.5, n_shared=ns, group_size=gsz, weight_format=fmt)
    wl = Workload("fmt", sh, 9, 1, "bf16", "zipf", 8100 + H + E + gsz + (fmt == "int8"))
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 16)
    def tensor_path(ran):
        return {"tc_gate_up", "tc_down", "combine"} <= ran and "gate_up" not in ran
    t1 = {"decode_fused"} if fmt == "int4" else SIMT
    tb = tensor_path if fmt == "int4" else SIMT
    for T in (1, 3, 9):
        _check(m, h, wl, L, gen_activations(wl, T, call=T), t1 if T == 1 else tb)
    h.close()


def test_row_scaled_equals_grouped_with_repeated_scales(m):
    """The pages' identity on the GPU: a per-row int4 layer and the same
    layer with each row's scale repeated over its groups give the same
    outputs bit for bit on the single-token kernel (T = 1: the same
    arithmetic), and within the parity tolerance on the tensor-core grouped
    GEMM (T = 3, 9), which rounds (u - 8) * s to f16 with grouped scales but
    applies a row's scale to the f32 accumulator."""
    sh_r = LayerShape(1024, 512, 32, 4, 4, 2, 2.5, group_size=0)
    wl = Workload("rowscale", sh_r, 1, 1, "bf16", "zipf", 8201)
    Lr = gen_layer(wl, device=DEV)
    import dataclasses
    rep = {}
    for name, K in (("gate_s", sh_r.hidden), ("up_s", sh_r.hidden), ("down_s", sh_r.inter),
                    ("sh_gate_s", sh_r.hidden), ("sh_up_s", sh_r.hidden),
                    ("sh_down_s", sh_r.inter)):
        rep[name] = getattr(Lr, name).repeat_interleave(K // 32, dim=-1).contiguous()
    sh_g = dataclasses.replace(sh_r, group_size=32)
    Lg = dataclasses.replace(Lr, shape=sh_g, **rep)
    hr, hg = m.MoELayer(Lr, 16), m.MoELayer(Lg, 16)
    for c, T in ((0, 1), (1, 1), (2, 3), (3, 9)):
        x = gen_activations(wl, T, call=c).to(DEV)
        yr, yg = hr.forward(x), hg.forward(x)
        torch.cuda.synchronize()
        if T == 1:
            assert torch.equal(yr, yg)
        else:
            d = (yr - yg).abs().amax(dim=1) / yg.abs().amax(dim=1)
            assert float(d.max()) <= TOL, (T, d)
    hr.close()
    hg.close()


def test_glm_decode_row_scaled(m):
    """The GLM decode layer with one scale a row: routing of 8 tokens and the
    outputs of 2 sampled tokens against the oracle."""
    wl = CONFIGS["glm_decode_rowscale"]
    L = gen_layer(wl, device=DEV)
    h = m.MoELayer(L, 1)
    router = router_of(wl, 0)
    for c in range(8):
        x_cpu = gen_activations(wl, 1, call=c)
        plan = m.Plan(1, wl.shape.top_k, wl.shape.n_experts, DEV)
        y = h.forward(x_cpu.to(DEV), plan=plan)
        torch.cuda.synchronize()
        x32 = x_cpu.float().numpy()
        _, _, ids_o, _ = oracle.route(wl.shape, router[0], router[1], x32)
        assert np.array_equal(plan.topk_ids.cpu().numpy(), ids_o)
        if c < 2:
            y_o, _, _, _ = oracle_layer(wl, 0, router, x32, [0])
            err = np.abs(y.cpu().numpy() - y_o).max() / np.abs(y_o).max()
            assert err <= TOL, err
    assert m.moe_device_status(h.h) == 0
    h.close()
