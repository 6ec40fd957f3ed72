"""Workload shapes of the decode MoE layer (synthetic, seeded).

Each entry is one fine-grained MoE FFN layer shape plus the stack it is run
in.  Shapes follow the model sizes the pages discuss (a 35B MoE with d_model
2048, E=256, K=4 and a prerouter input of 2048+2*256=2560; an 8B MoE with
K=8; a 397B-A17B-like model with ~6.75 MB 4-bit experts).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class MoEConfig:
    name: str
    d: int                 # d_model
    E: int                 # routed experts per layer
    K: int                 # experts per token
    F: int                 # expert SwiGLU hidden size
    shared: bool           # one always-on shared expert (weight 1)
    L: int                 # distinct resident layers
    depth: int             # layers per decode step (resident layers cycled)
    H: int                 # prerouter head hidden size (0: plain router)
    bits: int = 4          # 4 or 2
    group: int = 64
    head_prec: str = "int4"   # "int4" (affine group-64) or "fp16"
    lora_r: int = 0
    lora_alpha: float = 0.0
    lora_on: str = ""      # "routed_down" or "shared_all"
    seed: int = 0
    steps: int = 64
    T: int = 1             # tokens per call (1 = decode)
    sigma_w: float = 0.02
    sigma_lora: float = 0.01
    sigma_bias: float = 0.01
    self_predict: bool = False   # L == 1: the head predicts the layer's own route

    @property
    def slots(self) -> int:
        return self.K + (1 if self.shared else 0)

    @property
    def lora_scale(self) -> float:
        return self.lora_alpha / self.lora_r if self.lora_r else 0.0

    def expert_bytes(self) -> int:
        """Algorithmic bytes of one expert: 3*d*F weights at bits/8 B plus an
        fp16 scale and bias per 64 weights."""
        return 3 * self.d * self.F * self.bits // 8 + 3 * self.d * self.F // self.group * 4

    def expert_bytes_per_layer(self) -> int:
        """Expert weight bytes one decode token reads in one layer."""
        return self.slots * self.expert_bytes()


TINY = MoEConfig("tiny-d256-E16-K2", d=256, E=16, K=2, F=128, shared=False, L=1,
                 depth=1, H=128, lora_r=8, lora_alpha=16.0, lora_on="routed_down",
                 seed=0, steps=64, self_predict=True)

MOE35B = MoEConfig("35b-like-d2048-E256-K4-F512-shared-L40", d=2048, E=256, K=4,
                   F=512, shared=True, L=40, depth=40, H=512, lora_r=16,
                   lora_alpha=32.0, lora_on="shared_all", seed=1, steps=256)


def k_sweep(K: int) -> MoEConfig:
    return replace(MOE35B, name=f"35b-like-K{K}", K=K)


MOE8B = MoEConfig("8b-like-d2048-E256-K8-F512-L24", d=2048, E=256, K=8, F=512,
                  shared=False, L=24, depth=24, H=512, seed=2, steps=256)


def wide(bits: int) -> MoEConfig:
    return MoEConfig(f"397b-like-d4096-E512-K4-F1024-int{bits}", d=4096, E=512, K=4,
                     F=1024, shared=False, L=12, depth=48, H=1024, bits=bits, seed=3,
                     steps=64)


def batched(T: int) -> MoEConfig:
    return replace(MOE35B, name=f"batched-T{T}", L=1, depth=1, T=T, seed=4, steps=1)


ALL = {
    "tiny": TINY,
    "35b": MOE35B,
    # the 35B-like stack with 4 resident layers (1.8 GB of experts): the
    # profiling case of the fused decode step (its traffic per layer is the
    # 40-layer stack's)
    "35b-L4": replace(MOE35B, name="35b-like-d2048-E256-K4-F512-shared-L4", L=4, depth=4),
    "35b-K2": k_sweep(2),
    "35b-K8": k_sweep(8),
    # the 35B-like stack with fp16 head matrices (per-call path only): the
    # head-bytes side of the expert-byte share
    "35b-fp16head": replace(MOE35B, name="35b-like-fp16-heads", head_prec="fp16"),
    "8b": MOE8B,
    "wide-int4": wide(4),
    "wide-int2": wide(2),
    "batched-T8": batched(8),
    "batched-T64": batched(64),
    "batched-T512": batched(512),
    "batched-T4096": batched(4096),
}
