"""The five MLA decode workloads, stated as data.

Every workload is one decode step of DeepSeek Multi-Head Latent Attention in
weight-absorbed form over a latent KV cache whose rows are
``[c_kv (d_c) || k_rope (d_rope)]`` (Multi-Head Latent Attention, section 3.6
"Decoupled RoPE": the cache holds (d_c + d_R) values per token).

Shapes follow DeepSeek-V2-Lite (16 heads, hidden 2048; "Deepseek V2 Lite
Inference Engine in C", MLA notes) and a DeepSeek-V3-style head count (128
heads, hidden 7168; Multi-Head Latent Attention, section 3.1).

This module holds no arithmetic of the method: only sizes and the seeded
recipe's parameters.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Tuple

D_C = 512       # latent width of c_kv
D_ROPE = 64     # decoupled RoPE key/query width
D_NOPE = 128    # per-head non-rotated query/key width
D_V = 128       # per-head value width
ROW = D_C + D_ROPE


@dataclass(frozen=True)
class MlaConfig:
    name: str
    dtype: str                 # "f32" or "bf16": storage type of cache, queries, weights;
                               # "fp8": an FP8 E4M3 cache with bf16 queries and weights
    batch: int
    heads: int
    s_max: int                 # cache capacity in rows per sequence
    hidden: int                # model width; used only by the operation counters
    # per-sequence lengths: None -> every sequence is s_max rows long;
    # (lo, hi) -> drawn uniformly in [lo, hi] from the seed
    ragged: Optional[Tuple[int, int]] = None
    num_splits: int = 0        # 0 -> the library chooses; else KV chunks per sequence
    scaled_row_frac: float = 0.0   # fraction of rows per sequence multiplied by scaled_row_gain
    scaled_row_gain: float = 1.0
    d_c: int = D_C
    d_rope: int = D_ROPE
    d_nope: int = D_NOPE
    d_v: int = D_V
    rope_base: float = 10000.0
    weight_std: float = 0.02
    # query tokens per sequence in one step (multi-token / speculative decode): the
    # last q_len cached rows of each sequence are the step's tokens
    q_len: int = 1

    @property
    def row(self) -> int:
        return self.d_c + self.d_rope

    @property
    def elt_bytes(self) -> int:
        """Bytes per cache element."""
        return {"f32": 4, "bf16": 2, "fp8": 1}[self.dtype]

    @property
    def softmax_scale(self) -> float:
        # 1/sqrt(d_h + d_R) with d_h = qk_nope width (Multi-Head Latent
        # Attention, section 3.6: scores are scaled by 1/sqrt(d_h + d_R)).
        return (self.d_nope + self.d_rope) ** -0.5

    def scaled(self, **kw) -> "MlaConfig":
        return replace(self, **kw)


# The five workloads.  Names say what they are.
V2LITE_F32_B1_S64 = MlaConfig(
    name="v2lite_f32_b1_s64", dtype="f32", batch=1, heads=16, s_max=64, hidden=2048)
V2LITE_BF16_B8_S4096 = MlaConfig(
    name="v2lite_bf16_b8_s4096", dtype="bf16", batch=8, heads=16, s_max=4096, hidden=2048)
V2LITE_BF16_B64_RAGGED = MlaConfig(
    name="v2lite_bf16_b64_ragged512_8192", dtype="bf16", batch=64, heads=16, s_max=8192,
    hidden=2048, ragged=(512, 8192))
V3_BF16_H128_B32_S16384 = MlaConfig(
    name="v3heads_bf16_h128_b32_s16384", dtype="bf16", batch=32, heads=128, s_max=16384,
    hidden=7168)
V2LITE_BF16_B4_S65536_LONG = MlaConfig(
    name="v2lite_bf16_b4_s65536_split128", dtype="bf16", batch=4, heads=16, s_max=65536,
    hidden=2048, num_splits=128, scaled_row_frac=0.01, scaled_row_gain=8.0)

ALL_CONFIGS = (
    V2LITE_F32_B1_S64,
    V2LITE_BF16_B8_S4096,
    V2LITE_BF16_B64_RAGGED,
    V3_BF16_H128_B32_S16384,
    V2LITE_BF16_B4_S65536_LONG,
)

# The same shapes with an FP8 (E4M3) cache: one byte per cached element
# (Multi-Head Latent Attention, section 3.1).  The cache values are the same
# N(0, 1) draws rounded to E4M3 instead of bf16.
V2LITE_FP8_B8_S4096 = V2LITE_BF16_B8_S4096.scaled(name="v2lite_fp8_b8_s4096", dtype="fp8")
V2LITE_FP8_B64_RAGGED = V2LITE_BF16_B64_RAGGED.scaled(
    name="v2lite_fp8_b64_ragged512_8192", dtype="fp8")
V3_FP8_H128_B32_S16384 = V3_BF16_H128_B32_S16384.scaled(
    name="v3heads_fp8_h128_b32_s16384", dtype="fp8")
V2LITE_FP8_B4_S65536_LONG = V2LITE_BF16_B4_S65536_LONG.scaled(
    name="v2lite_fp8_b4_s65536_split128", dtype="fp8")
FP8_CONFIGS = (V2LITE_FP8_B8_S4096, V2LITE_FP8_B64_RAGGED, V3_FP8_H128_B32_S16384,
               V2LITE_FP8_B4_S65536_LONG)

# Multi-token decode ("Transformer and KV Cache Basics", mask design for multi-token
# decoding): four new tokens per sequence in one step, on the bench shape.
V2LITE_BF16_B8_S4096_Q4 = V2LITE_BF16_B8_S4096.scaled(name="v2lite_bf16_b8_s4096_q4", q_len=4)
V2LITE_FP8_B8_S4096_Q4 = V2LITE_FP8_B8_S4096.scaled(name="v2lite_fp8_b8_s4096_q4", q_len=4)
MULTI_TOKEN_CONFIGS = (V2LITE_BF16_B8_S4096_Q4, V2LITE_FP8_B8_S4096_Q4)

BY_NAME = {c.name: c for c in ALL_CONFIGS + FP8_CONFIGS + MULTI_TOKEN_CONFIGS}

# Parity tolerances: bf16 operands with fp32 accumulation, and the fp32 path.
TOL_BF16_MAX_ABS = 2e-2
TOL_BF16_REL_L2 = 5e-3
TOL_F32_MAX_ABS = 1e-4
