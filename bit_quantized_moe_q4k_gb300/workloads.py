"""The MoE layer workloads this library is measured and checked on.

Shapes follow the studied pages' statement of the problem: the tiny id-GEMV
case of the ferrum-kernels batched-GEMV tests (4 experts, N=64, K=256, 3
tokens, top_k=2) and three decode-shaped layers (a Qwen3-MoE-like layer with a
sigmoid-gated shared expert, a DeepSeek-V3-like layer with an unscaled shared
expert, and a Mixtral-like layer without one).
"""
from __future__ import annotations

from dataclasses import dataclass

QK = 256
BLOCK_BYTES = 144

SHARED_NONE, SHARED_SIGMOID, SHARED_UNSCALED = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int          # K of gate/up, N of down
    inter: int           # N of gate/up, K of down
    num_experts: int
    top_k: int
    m: int               # tokens
    ids: str             # "uniform" | "zipf" (distinct experts per token)
    shared_inter: int    # 0 when there is no shared expert
    shared_mode: int     # SHARED_NONE / SHARED_SIGMOID / SHARED_UNSCALED
    seed: int

    @property
    def pairs(self) -> int:
        return self.m * self.top_k

    def slab_bytes(self, n: int, k: int) -> int:
        """Bytes of one expert's [n, k] Q4_K projection."""
        return n * (k // QK) * BLOCK_BYTES

    def with_m(self, m: int) -> "Workload":
        return Workload(self.name, self.hidden, self.inter, self.num_experts, self.top_k, m, self.ids,
                        self.shared_inter, self.shared_mode, self.seed)


WORKLOADS = {
    # id-GEMV only (gate/up stride mode, and the down stride mode as a second case)
    "tiny_idgemv_e4_n64_k256_m3_t2": Workload("tiny_idgemv_e4_n64_k256_m3_t2", 256, 64, 4, 2, 3, "uniform",
                                              0, SHARED_NONE, 0x5EED + 1),
    "qwen3moe_h2048_i768_e128_t8_m1": Workload("qwen3moe_h2048_i768_e128_t8_m1", 2048, 768, 128, 8, 1,
                                               "uniform", 768, SHARED_SIGMOID, 0x5EED + 2),
    "qwen3moe_h2048_i768_e128_t8_m16_zipf": Workload("qwen3moe_h2048_i768_e128_t8_m16_zipf", 2048, 768, 128, 8,
                                                     16, "zipf", 768, SHARED_SIGMOID, 0x5EED + 3),
    "deepseekv3_h7168_i2048_e256_t8_m64": Workload("deepseekv3_h7168_i2048_e256_t8_m64", 7168, 2048, 256, 8, 64,
                                                   "uniform", 2048, SHARED_UNSCALED, 0x5EED + 4),
    "mixtral_h4096_i14336_e8_t2": Workload("mixtral_h4096_i14336_e8_t2", 4096, 14336, 8, 2, 1, "uniform",
                                           0, SHARED_NONE, 0x5EED + 5),
}

MIXTRAL_M_SWEEP = (1, 4, 16, 64, 256)
# Prefill-size batches of the same layers (the tensor-core grouped GEMM carries them).
PREFILL = (("mixtral_h4096_i14336_e8_t2", 512), ("mixtral_h4096_i14336_e8_t2", 2048),
           ("qwen3moe_h2048_i768_e128_t8_m1", 512))

# The headline decode layer: the Qwen3-MoE-like layer at m=1.
HEADLINE = "qwen3moe_h2048_i768_e128_t8_m1"
