"""Seeded generators for the MoE layer's weights and activations.

Two kinds of randomness are used:

* Packed int4 expert weights and their fp16 group scales come from a
  counter-based integer hash evaluated with torch integer ops.  The same call
  gives the same bytes on any device, so the GPU can hold a whole 24-layer
  stack that was generated in place while the CPU oracle regenerates only the
  experts it needs, byte for byte.
* Activations, router weights and the score-correction bias are small; they
  are drawn on the CPU with a seeded ``torch.Generator`` and copied wherever
  they are needed.

Distributions (from the workload definitions): nibbles uniform over the 16
codes (symmetric int4 q in [-8, 7] stored offset-binary as q+8), fp16 scales
~U(0.005, 0.02), router weight ~N(0, 0.02), activations ~N(0, 1) (bf16 for the
GLM-shaped workloads), bias ~U(-0.1, 0.1) for the tiny layer and a
Zipf-ranked bias for the GLM-shaped ones.  Verify batches share one N(0,1)
base row plus 0.3 N(0,1) per-token noise.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from .configs import LayerShape, Workload

_M32 = 0xFFFFFFFF
_MUL = 0x045D9F3B  # odd multiplier of a 32-bit integer finaliser (< 2**27)

# matrix ids for the hash streams
GATE, UP, DOWN = 0, 1, 2
SHARED_EXPERT = -1


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """32-bit integer finaliser on int64 tensors holding values in [0, 2**32).

    Products stay below 2**59, so int64 arithmetic is exact on every device.
    """
    x = ((x ^ (x >> 16)) * _MUL) & _M32
    x = ((x ^ (x >> 16)) * _MUL) & _M32
    return x ^ (x >> 16)


def _stream_keys(seed: int, layer: int, mat: int, experts: torch.Tensor, salt: int):
    """Per-expert 32-bit stream keys (int64 tensor, one per expert row)."""
    e = experts.to(torch.int64) & _M32
    k = torch.full_like(e, (seed * 0x9E3779B1 + 0x7F4A7C15) & _M32)
    k = _mix32(k)
    k = _mix32(k ^ ((layer * 0x85EBCA6B + salt) & _M32))
    k = _mix32(k ^ ((mat * 0xC2B2AE35 + 0x27D4EB2F) & _M32))
    k = _mix32(k ^ e)
    return k


def _words(seed, layer, mat, experts, n_words, device, salt):
    k1 = _stream_keys(seed, layer, mat, experts, salt).to(device)[:, None]
    k2 = _mix32(k1 ^ 0x68E31DA4)
    i = torch.arange(n_words, dtype=torch.int64, device=device)[None, :]
    return _mix32(_mix32(i ^ k1) ^ k2)


def _to_u32_bytes(words: torch.Tensor) -> torch.Tensor:
    w = torch.where(words >= 2**31, words - 2**32, words).to(torch.int32)
    return w.contiguous().view(torch.uint8)


def scale_table() -> np.ndarray:
    """1024 fp16 values evenly covering U(0.005, 0.02) (bin midpoints)."""
    k = np.arange(1024, dtype=np.float64)
    return (0.005 + 0.015 * (k + 0.5) / 1024.0).astype(np.float16)


_SCALE_TABLE_CACHE: dict = {}


def _scale_table_t(device) -> torch.Tensor:
    key = str(device)
    if key not in _SCALE_TABLE_CACHE:
        _SCALE_TABLE_CACHE[key] = torch.from_numpy(scale_table()).to(device)
    return _SCALE_TABLE_CACHE[key]


def gen_expert_matrix(seed: int, layer: int, mat: int, experts, rows: int,
                      cols: int, device="cpu", group_size: int = 32, fmt: str = "int4"):
    """Weights and fp16 scales of one matrix per listed expert.

    int4: packed nibbles [n, rows, cols/2] uint8; int8: signed bytes [n, rows,
    cols] (stored as uint8, uniform over all 256 codes).  Scales [n, rows,
    cols/g] for group size g, or [n, rows, 1] for group_size 0 (one scale a
    row).  int8 scales are the int4 table divided by 16 (exact in fp16), so
    the weights span about the same range in both formats.  ``experts``
    lists expert indices (``SHARED_EXPERT`` = -1 for the shared expert).
    Row-major, K (= cols) contiguous.  Each output row is independent of
    which other experts are generated in the same call.
    """
    experts = torch.as_tensor(experts, dtype=torch.int64)
    n = experts.numel()
    assert cols % 8 == 0 and (group_size == 0 or cols % group_size == 0)
    bpr = cols if fmt == "int8" else cols // 2  # weight bytes a row
    n_words = rows * bpr // 4
    q = _to_u32_bytes(_words(seed, layer, mat, experts, n_words, device, 0x1B873593))
    q = q.view(n, rows, bpr)
    spr = 1 if group_size == 0 else cols // group_size  # scales a row
    sidx = _words(seed, layer, mat, experts, rows * spr, device, 0x3C6EF372) & 1023
    table = _scale_table_t(device)
    if fmt == "int8":
        table = table / 16
    s = table[sidx].view(n, rows, spr)
    return q, s


def gen_router(shape: LayerShape, seed: int, layer: int, bias_kind: str,
               zipf_s: float = 1.1, zipf_kappa: float | None = None):
    """Router weight [E, H] fp32 ~N(0, 0.02) and score-correction bias [E] fp32."""
    g = torch.Generator().manual_seed(seed * 7919 + layer * 104729 + 17)
    w = torch.randn(shape.n_experts, shape.hidden, generator=g) * 0.02
    if bias_kind == "uniform":
        b = torch.rand(shape.n_experts, generator=g) * 0.2 - 0.1
    elif bias_kind == "zipf":
        kappa = ZIPF_KAPPA if zipf_kappa is None else zipf_kappa
        perm = torch.randperm(shape.n_experts, generator=g)
        rank = torch.empty(shape.n_experts, dtype=torch.float64)
        rank[perm] = torch.arange(1, shape.n_experts + 1, dtype=torch.float64)
        b64 = -kappa * zipf_s * torch.log(rank)
        b64 = b64 - b64.mean()
        b = b64.to(torch.float32)
    else:
        raise ValueError(bias_kind)
    return w.contiguous(), b.contiguous()


# Strength of the Zipf-ranked score-correction bias.  Chosen so that a
# 512-token prefill batch sends roughly 100 tokens to its busiest expert
# (the workload asks for uneven per-expert counts "0 to ~100");
# ``workloads/calibrate_zipf.py`` re-derives it with the oracle router.
ZIPF_KAPPA = 0.033


def gen_activations(w: Workload, T: int, call: int, layer: int = 0,
                    dtype: str | None = None) -> torch.Tensor:
    """Activations [T, H] on the CPU: fp32, or bf16 for the GLM-shaped layers."""
    dtype = dtype or w.x_dtype
    g = torch.Generator().manual_seed(w.seed * 1000003 + call * 9973 + layer * 31 + 5)
    H = w.shape.hidden
    if w.correlated > 0:
        base = torch.randn(1, H, generator=g)
        x = base + w.correlated * torch.randn(T, H, generator=g)
    else:
        x = torch.randn(T, H, generator=g)
    if dtype == "bf16":
        return x.to(torch.bfloat16).contiguous()
    return x.to(torch.float32).contiguous()


def gen_norm_weight(w: Workload, layer: int) -> torch.Tensor:
    """RMSNorm weight [H] fp32 ~U(0.5, 1.5) of one layer of a stacked workload."""
    g = torch.Generator().manual_seed(w.seed * 65537 + layer * 257 + 3)
    return (torch.rand(w.shape.hidden, generator=g) + 0.5).contiguous()


@dataclass
class LayerInputs:
    """All tensors of one MoE layer (device or host)."""
    shape: LayerShape
    router_w: torch.Tensor  # [E, H] f32
    router_b: torch.Tensor  # [E] f32
    gate_q: torch.Tensor  # [E, I, H/2] u8
    gate_s: torch.Tensor  # [E, I, H/32] f16
    up_q: torch.Tensor
    up_s: torch.Tensor
    down_q: torch.Tensor  # [E, H, I/2] u8
    down_s: torch.Tensor  # [E, H, I/32] f16
    sh_gate_q: torch.Tensor  # [I_s, H/2]
    sh_gate_s: torch.Tensor
    sh_up_q: torch.Tensor
    sh_up_s: torch.Tensor
    sh_down_q: torch.Tensor  # [H, I_s/2]
    sh_down_s: torch.Tensor


def _gen_mat_all(seed, layer, mat, E, rows, cols, device, chunk, group_size=32, fmt="int4"):
    bpr = cols if fmt == "int8" else cols // 2
    spr = 1 if group_size == 0 else cols // group_size
    q = torch.empty(E, rows, bpr, dtype=torch.uint8, device=device)
    s = torch.empty(E, rows, spr, dtype=torch.float16, device=device)
    for e0 in range(0, E, chunk):
        ex = list(range(e0, min(E, e0 + chunk)))
        qq, ss = gen_expert_matrix(seed, layer, mat, ex, rows, cols, device, group_size, fmt)
        q[e0:e0 + len(ex)] = qq
        s[e0:e0 + len(ex)] = ss
        del qq, ss
    return q, s


def gen_layer(w: Workload, layer: int = 0, device="cpu", chunk: int | None = None,
              zipf_kappa: float | None = None) -> LayerInputs:
    """Generate every tensor of one layer directly on ``device``."""
    sh = w.shape
    seed = w.seed + layer if w.layers > 1 else w.seed
    H, I, E, Is = sh.hidden, sh.inter, sh.n_experts, sh.i_shared
    if chunk is None:
        chunk = max(1, (1 << 25) // max(1, I * H // 8))
    rw, rb = gen_router(sh, seed, layer, w.bias_kind, w.zipf_s, zipf_kappa)
    f = (sh.group_size, sh.weight_format)
    gq, gs = _gen_mat_all(seed, layer, GATE, E, I, H, device, chunk, *f)
    uq, us = _gen_mat_all(seed, layer, UP, E, I, H, device, chunk, *f)
    dq, ds = _gen_mat_all(seed, layer, DOWN, E, H, I, device, chunk, *f)
    sgq, sgs = gen_expert_matrix(seed, layer, GATE, [SHARED_EXPERT], Is, H, device, *f)
    suq, sus = gen_expert_matrix(seed, layer, UP, [SHARED_EXPERT], Is, H, device, *f)
    sdq, sds = gen_expert_matrix(seed, layer, DOWN, [SHARED_EXPERT], H, Is, device, *f)
    return LayerInputs(sh, rw.to(device), rb.to(device), gq, gs, uq, us, dq, ds,
                       sgq[0].contiguous(), sgs[0].contiguous(), suq[0].contiguous(),
                       sus[0].contiguous(), sdq[0].contiguous(), sds[0].contiguous())


class HostExpertCache:
    """CPU copies of single experts of one layer, regenerated on demand.

    Lets the oracle touch only the experts a batch selects, without reading
    weights back from the device.
    """

    def __init__(self, w: Workload, layer: int = 0):
        self.w = w
        self.layer = layer
        self.seed = w.seed + layer if w.layers > 1 else w.seed
        self._cache: dict = {}

    def expert(self, e: int):
        """(gate_q, gate_s, up_q, up_s, down_q, down_s) numpy arrays; e=-1 shared."""
        if e not in self._cache:
            sh = self.w.shape
            H = sh.hidden
            I = sh.i_shared if e == SHARED_EXPERT else sh.inter
            out = []
            for mat, (r, c) in ((GATE, (I, H)), (UP, (I, H)), (DOWN, (H, I))):
                q, s = gen_expert_matrix(self.seed, self.layer, mat, [e], r, c, "cpu",
                                         sh.group_size, sh.weight_format)
                out.append(np.ascontiguousarray(q[0].numpy()))
                out.append(np.ascontiguousarray(s[0].view(torch.int16).numpy().view(np.uint16)))
            self._cache[e] = tuple(out)
        return self._cache[e]


def zipf_counts_summary(counts: np.ndarray) -> dict:
    c = np.sort(np.asarray(counts))[::-1]
    return {"max": int(c[0]), "min": int(c[-1]), "zero": int((c == 0).sum()),
            "top8": [int(v) for v in c[:8]],
            "gini": float(_gini(c))}


def _gini(c):
    c = np.sort(np.asarray(c, dtype=np.float64))
    n = len(c)
    if c.sum() == 0:
        return 0.0
    idx = np.arange(1, n + 1)
    return float((2 * (idx * c).sum() / (n * c.sum())) - (n + 1) / n)


def stack_bytes(w: Workload) -> int:
    sh = w.shape
    per = sh.n_experts * sh.expert_bytes() + sh.shared_bytes() + sh.router_bytes()
    return per * w.layers


assert math.isclose(float(scale_table()[0]), 0.005, rel_tol=2e-3)
