"""The five workloads of the MoE-layer hot path, by name and size.

tiny          H=256,  I=128,  E=16,  top-4, 4 groups / 2 kept, 1 token, fp32 x
glm_decode    H=6144, I=2048, E=256, top-8, 8 groups / 4 kept, T=1, 256 tokens
glm_verify    same layer, T=4 correlated tokens per step (1 accepted + 3 drafts)
glm_prefill   same layer, T=512 tokens in one call
glm_stack     24 such layers resident, T=1, RMSNorm before each router and a
              residual add after each layer
glm_prefill_uniform  the same layer, T=8192 without the Zipf skew (256 rows
              per expert on average): the grouped GEMM where it is compute-bound
glm_decode_rowscale  glm_decode with one fp16 scale per row (Colibri's whole-row
              group, "GLM-5.2 on a 32 GB Mac", G2 implementation status)
glm_prefill_rowscale glm_prefill with one fp16 scale per row

GLM-5.2 layer geometry (256 routed experts, top-8, one shared expert,
routed_scaling_factor, sigmoid noaux_tc routing): "GLM-5.2 on a 32 GB Mac"
section "What Colibri is actually doing" and "N1. GLM-5.2 graph"; the Colibri
README "What's implemented".  Hidden/intermediate sizes, group limits and the
int4 group-32 fp16-scale format are the workload's own fixed sizes.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class LayerShape:
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    n_group: int
    topk_group: int
    routed_scaling_factor: float
    n_shared: int = 1
    shared_inter: int = 0  # 0 -> same as inter
    group_size: int = 32   # 32, or 0 for one fp16 scale per row
    weight_format: str = "int4"  # "int4" (offset-binary nibbles) or "int8" (signed bytes)

    @property
    def i_shared(self) -> int:
        return self.shared_inter or self.inter

    def matrix_bytes(self, rows: int, cols: int) -> int:
        """Weights and fp16 scales of one rows x cols matrix in this format."""
        q = rows * cols if self.weight_format == "int8" else rows * cols // 2
        n_sc = rows if self.group_size == 0 else rows * (cols // self.group_size)
        return q + 2 * n_sc

    def expert_bytes(self) -> int:
        """Weights + scales of one routed expert (gate, up, down)."""
        h, i = self.hidden, self.inter
        return 2 * self.matrix_bytes(i, h) + self.matrix_bytes(h, i)

    def shared_bytes(self) -> int:
        h, i = self.hidden, self.i_shared
        return 2 * self.matrix_bytes(i, h) + self.matrix_bytes(h, i)

    def router_bytes(self) -> int:
        return self.n_experts * self.hidden * 4 + self.n_experts * 4


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    tokens_per_call: int  # T of one forward call
    calls: int  # forward calls in one pass of the workload
    x_dtype: str  # "f32" or "bf16"
    bias_kind: str  # "uniform" or "zipf"
    seed: int
    layers: int = 1
    correlated: float = 0.0  # per-token noise amplitude for verify batches
    rmsnorm_eps: float = 0.0  # >0: RMSNorm before the router + residual add
    zipf_s: float = 1.1
    extra: dict = field(default_factory=dict)


TINY = LayerShape(256, 128, 16, 4, 4, 2, 2.5)
GLM = LayerShape(6144, 2048, 256, 8, 8, 4, 2.5)
GLM_ROWSCALE = LayerShape(6144, 2048, 256, 8, 8, 4, 2.5, group_size=0)

CONFIGS = {
    "tiny": Workload("tiny", TINY, 1, 1, "f32", "uniform", 1001),
    "glm_decode": Workload("glm_decode", GLM, 1, 256, "bf16", "zipf", 1002),
    "glm_verify": Workload("glm_verify", GLM, 4, 64, "bf16", "zipf", 1003,
                           correlated=0.3),
    "glm_prefill": Workload("glm_prefill", GLM, 512, 1, "bf16", "zipf", 1004),
    "glm_stack": Workload("glm_stack", GLM, 1, 16, "f32", "zipf", 5000,
                          layers=24, rmsnorm_eps=1e-5),
    # calibration of the grouped GEMM where it is compute-bound: 8192 tokens
    # without the Zipf skew, 256 plan rows per expert on average
    "glm_prefill_uniform": Workload("glm_prefill_uniform", GLM, 8192, 1, "bf16", "uniform",
                                    1005, extra={"bound": "tensor"}),
    "glm_decode_rowscale": Workload("glm_decode_rowscale", GLM_ROWSCALE, 1, 256, "bf16", "zipf",
                                    1006),
    "glm_prefill_rowscale": Workload("glm_prefill_rowscale", GLM_ROWSCALE, 512, 1, "bf16", "zipf",
                                     1007),
}


def config_by_name(name: str) -> Workload:
    return CONFIGS[name]
