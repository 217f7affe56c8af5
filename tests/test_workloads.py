"""The seeded synthetic inputs follow their stated recipe (CPU).

Uniform int4 codes, fp16 scales inside U(0.005, 0.02), router weight
N(0, 0.02), the tiny layer's U(-0.1, 0.1) bias and the Zipf-ranked bias of the
GLM-shaped layers (a 512-token batch gives its busiest expert about 100 tokens
and leaves some experts idle), correlated verify tokens, and generation that
is deterministic and independent per expert.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import CONFIGS
from workloads.gen import (DOWN, GATE, SHARED_EXPERT, UP, ZIPF_KAPPA, gen_activations,
                           gen_expert_matrix, gen_router)


def test_nibbles_uniform_and_scales_in_range():
    q, s = gen_expert_matrix(1234, 0, GATE, [0, 5], 256, 1024)
    b = q.numpy().reshape(-1)
    nib = np.concatenate([b & 0xF, b >> 4])
    counts = np.bincount(nib, minlength=16)
    expect = nib.size / 16
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 50.0, chi2  # 15 degrees of freedom: p < 1e-5 beyond 50
    sv = s.float().numpy()
    assert sv.min() >= 0.005 and sv.max() <= 0.02
    assert abs(sv.mean() - 0.0125) < 0.0125 * 0.01


def test_generation_is_deterministic_and_per_expert():
    q1, s1 = gen_expert_matrix(77, 2, UP, [3], 64, 256)
    q3, s3 = gen_expert_matrix(77, 2, UP, [2, 3, 4], 64, 256)
    assert torch.equal(q1[0], q3[1]) and torch.equal(s1[0], s3[1])
    again, _ = gen_expert_matrix(77, 2, UP, [3], 64, 256)
    assert torch.equal(q1, again)
    others = [gen_expert_matrix(77, 2, UP, [4], 64, 256)[0],      # another expert
              gen_expert_matrix(77, 3, UP, [3], 64, 256)[0],      # another layer
              gen_expert_matrix(77, 2, DOWN, [3], 64, 256)[0],    # another matrix
              gen_expert_matrix(78, 2, UP, [3], 64, 256)[0],      # another seed
              gen_expert_matrix(77, 2, UP, [SHARED_EXPERT], 64, 256)[0]]
    for o in others:
        assert (o != q1).float().mean() > 0.9


def test_router_weight_and_bias_recipe():
    sh = CONFIGS["glm_decode"].shape
    w, b = gen_router(sh, 1002, 0, "zipf")
    assert abs(float(w.std()) - 0.02) < 0.02 * 0.01 and abs(float(w.mean())) < 1e-4
    assert abs(float(b.double().mean())) < 1e-6
    # b_e = c - kappa * s * ln(rank_e): the ranks come back as 1..E
    b64 = b.double().numpy()
    rank = np.exp((b64.max() - b64) / (ZIPF_KAPPA * 1.1))
    assert np.allclose(np.sort(rank), np.arange(1, sh.n_experts + 1), rtol=1e-3)
    _, bu = gen_router(CONFIGS["tiny"].shape, 1001, 0, "uniform")
    assert float(bu.min()) >= -0.1 and float(bu.max()) <= 0.1


def test_zipf_prefill_load():
    # 512 tokens of the prefill workload through the oracle router: uneven
    # per-expert counts from 0 to about 100
    wl = CONFIGS["glm_prefill"]
    sh = wl.shape
    rw, rb = gen_router(sh, wl.seed, 0, wl.bias_kind, wl.zipf_s)
    x = gen_activations(wl, 512, call=0).float().numpy()
    _, _, ids, _ = oracle.route(sh, rw.numpy(), rb.numpy(), x, 0.0, None)
    counts = np.bincount(ids.reshape(-1), minlength=sh.n_experts)
    assert counts.sum() == 512 * sh.top_k
    assert 80 <= counts.max() <= 120, counts.max()
    assert (counts == 0).sum() >= 1


def test_verify_tokens_correlated_and_activation_types():
    wl = CONFIGS["glm_verify"]
    x = gen_activations(wl, 4, call=0)
    assert x.dtype == torch.bfloat16 and tuple(x.shape) == (4, wl.shape.hidden)
    c = np.corrcoef(x.float().numpy())
    off = c[~np.eye(4, dtype=bool)]
    # base + 0.3 * noise: correlation 1 / (1 + 0.09) = 0.917
    assert np.all((off > 0.89) & (off < 0.94)), off
    assert gen_activations(CONFIGS["glm_decode"], 1, call=0).dtype == torch.bfloat16
    assert gen_activations(CONFIGS["tiny"], 1, call=0).dtype == torch.float32
    xs = gen_activations(CONFIGS["glm_decode"], 2, call=1).float()
    assert abs(float(xs.std()) - 1.0) < 0.03
