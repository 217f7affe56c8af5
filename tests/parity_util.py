"""Shared helpers of the parity tests: tolerance, error measure, oracle runs.

The tolerance is the layer's stated accuracy bar: per token, the largest
absolute difference between the CUDA output and the fp32-accumulated oracle,
divided by the largest absolute oracle output of that token, must not exceed
2e-3.  Expert ids, gate weights and the routing plan are compared bit for bit.
"""
from __future__ import annotations

import numpy as np

import oracle
from workloads.gen import SHARED_EXPERT, HostExpertCache, gen_router

TOL = 2e-3
RMS_EPS = float(np.float32(1e-5))  # the fp32 eps the C ABI receives, widened


def rel_err_per_token(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    y = np.asarray(y, np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    den = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    return np.abs(y - ref).max(axis=1) / den


def elem_err_per_token(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """The element-wise companion figure (reported, not gated): per token, the
    largest |y_i - ref_i| / max(|ref_i|, 1e-2 * max_j |ref_j|).  The floor keeps
    elements near zero from dividing by almost nothing."""
    y = np.asarray(y, np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    floor = np.maximum(1e-2 * np.abs(ref).max(axis=1, keepdims=True), 1e-30)
    return (np.abs(y - ref) / np.maximum(np.abs(ref), floor)).max(axis=1)


def resid_err_per_token(y: np.ndarray, y_ref: np.ndarray, resid: np.ndarray) -> np.ndarray:
    """Error of a residual-form output y = resid + MoE(...).

    Both sides round resid + v once in fp32, so a difference d in v can
    move y by d plus one unit in the last place of y: that ulp is allowed on
    top, and the rest is measured against the MoE output y_ref - resid."""
    y = np.asarray(y, np.float64).reshape(y_ref.shape[0], -1)
    ref = np.asarray(y_ref, np.float64).reshape(y_ref.shape[0], -1)
    delta = ref - np.asarray(resid, np.float64).reshape(ref.shape)
    ulp = np.spacing(np.abs(np.asarray(y_ref, np.float32))).astype(np.float64).reshape(ref.shape)
    excess = np.maximum(np.abs(y - ref) - ulp, 0.0)
    den = np.maximum(np.abs(delta).max(axis=1), 1e-30)
    return excess.max(axis=1) / den


def router_of(workload, layer: int = 0):
    seed = workload.seed + layer if workload.layers > 1 else workload.seed
    rw, rb = gen_router(workload.shape, seed, layer, workload.bias_kind, workload.zipf_s)
    return rw.numpy(), rb.numpy()


def oracle_layer(workload, layer: int, router, x_f32: np.ndarray, tokens, eps: float = 0.0,
                 gamma=None, resid=None, cache: HostExpertCache | None = None):
    """Oracle outputs (y, ids, w, logits) of the given token rows of x."""
    rw, rb = router
    cache = cache or HostExpertCache(workload, layer)
    xs = np.ascontiguousarray(x_f32[list(tokens)], np.float32)
    rs = None if resid is None else np.ascontiguousarray(resid[list(tokens)], np.float32)
    shared = cache.expert(SHARED_EXPERT) if workload.shape.n_shared else None
    return oracle.moe_forward(workload.shape, rw, rb, cache.expert, shared, xs, eps=eps,
                              gamma=gamma, resid=rs)
