"""The named attention workloads and their input recipe.

Every workload draws q, k and v i.i.d. N(0, 1) from ``ragen`` with
seed = 1000 * workload index and tensor ids 0 (q), 1 (k), 2 (v); the backward
draws dL/dout the same way with tensor id 3, shaped like q; bf16
workloads round each sample to bfloat16 (nearest even).  Tensors are laid out
shard-major: q is [B, Hq, S, D], k and v are [B, Hkv, S, D], and virtual
device i of N owns rows [i*S/N, (i+1)*S/N) of every (b, h) slice.  Under the
striped layout, row r of shard i holds token r*N + i.
"""
from __future__ import annotations

from dataclasses import dataclass

TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_DO = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    dtype: str  # "f32" or "bf16"
    B: int
    Hq: int
    Hkv: int
    S: int
    N: int
    D: int
    causal: bool
    striped: int  # layout: 0 contiguous, 1 striped, 2 zigzag

    @property
    def seed(self) -> int:
        return 1000 * self.index

    @property
    def Sb(self) -> int:
        return self.S // self.N

    def flops(self) -> float:
        """Attention FLOPs by the metric's convention: 4*B*Hq*S^2*D, halved if causal."""
        f = 4.0 * self.B * self.Hq * self.S * self.S * self.D
        return f / 2 if self.causal else f

    def flops_exact(self) -> float:
        """FLOPs over the visible (query, key) pairs only: S(S+1)/2 pairs if causal."""
        pairs = self.S * (self.S + 1) / 2 if self.causal else float(self.S) * self.S
        return 4.0 * self.B * self.Hq * pairs * self.D

    def shapes(self):
        return ((self.B, self.Hq, self.S, self.D), (self.B, self.Hkv, self.S, self.D))

    def describe(self) -> dict:
        return {
            "workload": self.name, "dtype": self.dtype, "B": self.B, "Hq": self.Hq,
            "Hkv": self.Hkv, "S": self.S, "N": self.N, "Sb": self.Sb, "D": self.D,
            "causal": self.causal,
            "layout": ("contiguous", "striped", "zigzag")[int(self.striped)],
        }


WORKLOADS = {
    "toy_f32": Workload(0, "toy_f32_N4_S32_D16", "f32", 1, 1, 1, 32, 4, 16, False, False),
    "noncausal_8k": Workload(1, "bf16_noncausal_B1_H8_S8192_N8_D128", "bf16",
                             1, 8, 8, 8192, 8, 128, False, False),
    "causal_32k_contig": Workload(2, "bf16_causal_B2_H32_S32768_N8_D128_contiguous", "bf16",
                                  2, 32, 32, 32768, 8, 128, True, False),
    "causal_32k_striped": Workload(2, "bf16_causal_B2_H32_S32768_N8_D128_striped", "bf16",
                                   2, 32, 32, 32768, 8, 128, True, True),
    # the same shape under the zigzag layout (2N chunks, device i holds chunks i and 2N-1-i)
    "causal_32k_zigzag": Workload(2, "bf16_causal_B2_H32_S32768_N8_D128_zigzag", "bf16",
                                  2, 32, 32, 32768, 8, 128, True, 2),
    "gqa_128k": Workload(3, "bf16_causal_gqa_B1_Hq32_Hkv8_S131072_N16_D128_striped", "bf16",
                         1, 32, 8, 131072, 16, 128, True, True),
    # the 128K GQA shape with ragged shards (8000 tokens each: the last tile of
    # every shard holds 64 rows)
    "gqa_128k_ragged": Workload(6, "bf16_causal_gqa_B1_Hq32_Hkv8_S128000_N16_D128_striped", "bf16",
                                1, 32, 8, 128000, 16, 128, True, 1),
    # profiling case: same kernel shape as gqa_128k, inputs larger than L2 but under 1 GB
    "prof_64k": Workload(5, "bf16_causal_gqa_B1_Hq16_Hkv4_S65536_N8_D128_striped", "bf16",
                         1, 16, 4, 65536, 8, 128, True, True),
    # the 128K GQA shape at head dimension 64 (a tensor-core kernel variant)
    "gqa_128k_d64": Workload(7, "bf16_causal_gqa_B1_Hq32_Hkv8_S131072_N16_D64_striped", "bf16",
                             1, 32, 8, 131072, 16, 64, True, 1),
    "long_1m": Workload(4, "bf16_causal_gqa_B1_Hq8_Hkv1_S1048576_N64_D128_striped", "bf16",
                        1, 8, 1, 1048576, 64, 128, True, True),
    # parity case for the forward's common ring entry at a size whose rows the
    # oracle checks by the shard: 16 shards of 24576 tokens, whose keys and
    # values (24 MiB per shard) together exceed the L2
    "long_shards_384k": Workload(8, "bf16_causal_gqa_B1_Hq2_Hkv1_S393216_N16_D128_striped",
                                 "bf16", 1, 2, 1, 393216, 16, 128, True, 1),
}
