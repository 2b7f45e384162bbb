"""Decode projection shapes of the w8a16 GEMV workloads.

Shapes are the GLM-5.2 checkpoint tensors read from the safetensors headers
on the "GLM-5.2 anatomy" page (section "weights measured", tensor table):
fused_qkv_a_proj is q_a_proj [2048, 6144] and kv_a_proj_with_mqa [576, 6144]
merged into one [2624, 6144] plane (section "one merge at construction");
o_proj [6144, 16384]; a shared expert is 6144 <-> 2048 (gate and up merged
into [4096, 6144], down [6144, 2048]); q_b_proj [16384, 2048]; kv_b_proj
[28672, 512]; the indexer's wq_b [4096, 2048], wk [128, 6144] and
weights_proj [32, 6144]; lm_head [154880, 6144] in bf16.

W is [N, K]: N output rows, K reduction columns, K contiguous in memory.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Projection:
    name: str
    n: int
    k: int
    dtype: str                  # "e4m3fn", "e4m3fn_b128", "bf16" or "mxfp4"
    ms: tuple                   # decode-token counts exercised
    ldw: int | None = None      # source row stride when the plane is padded
    act: str = ""               # "silu_mul": a merged gate_up plane (gate rows first)
                                # whose call returns silu(gate) * up, n / 2 columns

    @property
    def weight_bytes(self) -> int:
        if self.dtype == "mxfp4":  # codes, half a byte each, and one E8M0 byte per 32
            return self.n * self.k // 2 + self.n * -(-self.k // 32)
        if self.dtype == "e4m3fn_b128":  # codes and one fp32 factor per 128 x 128 block
            return self.n * self.k + 4 * -(-self.n // 128) * -(-self.k // 128)
        return self.n * self.k * (1 if self.dtype == "e4m3fn" else 2)

    @property
    def out_n(self) -> int:
        return self.n // 2 if self.act == "silu_mul" else self.n

    def algorithmic_bytes(self, m: int) -> int:
        """W + fp32 scales (FP8) + x + y, with the logical K (pad excluded)."""
        b = self.weight_bytes + 2 * m * self.k + 2 * m * self.out_n
        if self.dtype == "e4m3fn":
            b += 4 * self.n
        return b

    def flops(self, m: int) -> int:
        extra = (m * self.n if self.dtype == "e4m3fn" else
                 2 * m * self.n * -(-self.k // 128) if self.dtype == "e4m3fn_b128" else 0)
        return 2 * m * self.n * self.k + extra


SWEEP_M = (1, 2, 4, 8, 16, 32, 64)

TINY = Projection("tiny", 256, 512, "e4m3fn", (1,))
FUSED_QKV_A = Projection("fused_qkv_a_proj", 2624, 6144, "e4m3fn", (1, 4, 16))
O_PROJ = Projection("o_proj", 6144, 16384, "e4m3fn", (1, 2, 8, 32))
O_PROJ_BF16 = Projection("o_proj_bf16", 6144, 16384, "bf16", (1, 2, 8, 32))
SHARED_GATE_UP = Projection("shared_expert_gate_up", 4096, 6144, "e4m3fn", (8,))
SHARED_DOWN = Projection("shared_expert_down", 6144, 2048, "e4m3fn", (8,))
SHARED_GATE_UP_KPAD = Projection("shared_expert_gate_up_kpad", 4096, 6144, "e4m3fn", (8,),
                                 ldw=6144 + 128)
# The shared expert's gate_up with SiLU-and-multiply in the same kernel: its
# output h [M, 2048] is the down projection's input.
SHARED_GATE_UP_SILU = Projection("shared_expert_gate_up_silu", 4096, 6144, "e4m3fn", (8,),
                                 act="silu_mul")
Q_B = Projection("q_b_proj", 16384, 2048, "e4m3fn", SWEEP_M)
KV_B = Projection("kv_b_proj", 28672, 512, "e4m3fn", SWEEP_M)
WQ_B = Projection("indexer_wq_b", 4096, 2048, "e4m3fn", SWEEP_M)
WK = Projection("indexer_wk", 128, 6144, "bf16", SWEEP_M)
WEIGHTS_PROJ = Projection("indexer_weights_proj", 32, 6144, "bf16", SWEEP_M)
LM_HEAD = Projection("lm_head", 154880, 6144, "bf16", (1,))
# The indexer's wk and weights_proj read the same token rows (hidden states,
# K = 6144), so their bf16 planes bind as one [160, 6144] plane: one call
# instead of two, rows 0..127 = wk, 128..159 = weights_proj.
WK_WEIGHTS_PROJ = Projection("indexer_wk_weights_proj", 160, 6144, "bf16", SWEEP_M)
# q_b_proj and the indexer's wq_b read the same q_lora_rank latent (q_c, 2048
# wide, after q_a_layernorm: the GLM-5.2 anatomy page's config table notes
# that wq_b takes this rank too, and its layer diagram feeds q_c to both), and
# both are E4M3 planes with row scales, so they bind as one [20480, 2048]
# plane: rows 0..16383 = q_b, 16384..20479 = wq_b, one call instead of two.
Q_B_WQ_B = Projection("q_b_wq_b_proj", 20480, 2048, "e4m3fn", SWEEP_M)

# Above the decode range: draft rows and prefill chunks of 96..256 tokens on
# the largest attention projections (the tensor-memory kernel only).
LARGE_M = (96, 128, 192, 256)
O_PROJ_LARGE_M = Projection("o_proj_large_m", 6144, 16384, "e4m3fn", LARGE_M)
Q_B_LARGE_M = Projection("q_b_proj_large_m", 16384, 2048, "e4m3fn", LARGE_M)
KV_B_LARGE_M = Projection("kv_b_proj_large_m", 28672, 512, "e4m3fn", LARGE_M)

# w4a16: the same projections as MXFP4 planes (the GLM-5.2 anatomy page's
# deployments serve a GLM-5.2-MXFP4 checkpoint), on the register ring.
O_PROJ_MXFP4 = Projection("o_proj_mxfp4", 6144, 16384, "mxfp4", (1, 2, 8, 32))
Q_B_MXFP4 = Projection("q_b_proj_mxfp4", 16384, 2048, "mxfp4", (1, 8, 64))
FUSED_QKV_A_MXFP4 = Projection("fused_qkv_a_proj_mxfp4", 2624, 6144, "mxfp4", (1, 4, 16))

# Block-scaled FP8 (one fp32 factor per 128 x 128 block): the GLM-5.2 anatomy
# page runs fused_qkv_a_proj through a blockscale GEMM; o_proj as the largest
# attention plane.  Register ring, 1..64 tokens.
FUSED_QKV_A_B128 = Projection("fused_qkv_a_proj_b128", 2624, 6144, "e4m3fn_b128", (1, 4, 16))
O_PROJ_B128 = Projection("o_proj_b128", 6144, 16384, "e4m3fn_b128", (1, 2, 8, 32))

ALL = (TINY, FUSED_QKV_A, O_PROJ, O_PROJ_BF16, SHARED_GATE_UP, SHARED_DOWN,
       SHARED_GATE_UP_KPAD, SHARED_GATE_UP_SILU, Q_B, KV_B, WQ_B, WK, WEIGHTS_PROJ, WK_WEIGHTS_PROJ,
       Q_B_WQ_B, LM_HEAD,
       O_PROJ_LARGE_M, Q_B_LARGE_M, KV_B_LARGE_M, O_PROJ_MXFP4, Q_B_MXFP4, FUSED_QKV_A_MXFP4,
       FUSED_QKV_A_B128, O_PROJ_B128)
BY_NAME = {p.name: p for p in ALL}

# The bench's step, one call per plane and token count: o_proj as an FP8 and
# as a bf16 plane at M in {1, 2, 8, 32}; the GLM-5.2 layer sweep -- q_b, kv_b,
# the indexer's wq_b, and its wk and weights_proj bound as one [160, 6144]
# bf16 plane (both read the hidden states; one call gives both outputs) -- at
# M in {1, 2, 4, 8, 16, 32, 64}; and the bf16 lm_head at M = 1.
BENCH_STEP = (O_PROJ, O_PROJ_BF16, Q_B, KV_B, WQ_B, WK_WEIGHTS_PROJ, LM_HEAD)

# The workload groups, in order: the tiny correctness case, the fused
# qkv_a projection, o_proj (FP8 and bf16), the shared-expert pair with its
# K-padded variant and its gate_up with SiLU-and-multiply, the full-layer
# sweep, 96..256 tokens on the large attention projections, MXFP4 planes and
# block-scaled FP8 planes.
GROUPS = {
    "tiny": (TINY,),
    "fused_qkv_a_proj": (FUSED_QKV_A,),
    "o_proj": (O_PROJ, O_PROJ_BF16),
    "shared_expert": (SHARED_GATE_UP, SHARED_DOWN, SHARED_GATE_UP_KPAD, SHARED_GATE_UP_SILU),
    "layer_sweep": (Q_B, KV_B, WQ_B, WK, WEIGHTS_PROJ, WK_WEIGHTS_PROJ, Q_B_WQ_B, LM_HEAD),
    "large_m": (O_PROJ_LARGE_M, Q_B_LARGE_M, KV_B_LARGE_M),
    "mxfp4": (O_PROJ_MXFP4, Q_B_MXFP4, FUSED_QKV_A_MXFP4),
    "block_scaled": (FUSED_QKV_A_B128, O_PROJ_B128),
}
