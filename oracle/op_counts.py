"""Operation and memory-operation counters for one MLA decode step.

TEST INFRASTRUCTURE (same import rule as ``mla_oracle``).

"Deepseek V2 Lite Inference Engine in C" (MLA notes) lists, for three ways of
computing one decode step at cache length S, each matrix product with its
shapes, and totals them under a convention: a multiply-add counts as one
"flop", and a product's memory operations are the element counts of its two
operands plus its result.  The counters below apply that convention to the
same op lists, so that the printed totals can be checked, and to the fully
absorbed path this library computes.

Each op is (name, macs, memops) as functions of S.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Tuple

Op = Tuple[str, Callable[[int], int], Callable[[int], int]]


def _matvec(rows: int, cols: int):
    """(cols) @ (rows, cols)^T -> (rows): macs rows*cols; memops cols + rows*cols + rows."""
    return (lambda S: rows * cols), (lambda S: cols + rows * cols + rows)


def variant_ops(variant: str, hidden: int = 2048, heads: int = 16, d_c: int = 512,
                d_rope: int = 64, d_nope: int = 128, d_v: int = 128) -> List[Op]:
    """Op list of one decode step for variant "A" (original weights), "B"
    (materialised W_UK.W_Q per head) or "C" (absorbed without materialising), in
    the order the page lists them; the shared kv_a_proj step is skipped as on
    the page."""
    H = heads
    q_out = H * (d_nope + d_rope)          # 3072 for V2-Lite
    kvb_rows = H * (d_nope + d_v)          # 4096
    qk = d_nope + d_rope                   # 192
    ops: List[Op] = []
    if variant == "A":
        ops.append(("q_proj", *_matvec(q_out, hidden)))
        ops.append(("kv_b_proj decompress",
                    lambda S: S * d_c * kvb_rows,
                    lambda S: S * d_c + kvb_rows * d_c + S * kvb_rows))
        ops.append(("scores", lambda S: H * S * qk, lambda S: H * S * qk + H * qk + H * S))
        ops.append(("p @ v", lambda S: H * S * d_v, lambda S: H * S + H * S * d_v + H * d_v))
    elif variant == "B":
        ops.append(("q_nope via materialised WukWq",
                    lambda S: hidden * H * d_c,
                    lambda S: hidden + H * hidden * d_c + H * S * d_c))
        ops.append(("q_rope proj",
                    lambda S: hidden * H * d_rope,
                    lambda S: hidden + H * d_rope * hidden + H * d_rope))
        ops.append(("scores vs latent rows", lambda S: H * S * (d_c + d_rope),
                    lambda S: S * (d_c + d_rope) + H * (d_c + d_rope) + H * S))
        ops.append(("v decompress", lambda S: S * d_c * H * d_v,
                    lambda S: S * d_c + H * d_v * d_c + S * H * d_v))
        ops.append(("p @ v", lambda S: H * S * d_v, lambda S: H * S + H * S * d_v + H * d_v))
    elif variant == "C":
        ops.append(("q_proj", *_matvec(q_out, hidden)))
        ops.append(("absorb q_nope @ W_UK",
                    lambda S: H * d_nope * d_c,
                    lambda S: H * d_nope + H * d_nope * d_c + H * d_c))
        ops.append(("scores vs latent rows", lambda S: H * S * (d_c + d_rope),
                    lambda S: S * (d_c + d_rope) + H * (d_c + d_rope) + H * S))
        ops.append(("v decompress", lambda S: S * d_c * H * d_v,
                    lambda S: S * d_c + H * d_v * d_c + S * H * d_v))
        ops.append(("p @ v", lambda S: H * S * d_v, lambda S: H * S + H * S * d_v + H * d_v))
    elif variant == "latent":
        # Fully absorbed (W^UV applied after attention, Multi-Head Latent
        # Attention eq. 3.3.3): the three library calls, q_proj excluded.
        ops.append(("absorb q_nope @ W_UK",
                    lambda S: H * d_nope * d_c,
                    lambda S: H * d_nope + H * d_nope * d_c + H * d_c))
        ops.append(("scores vs latent rows", lambda S: H * S * (d_c + d_rope),
                    lambda S: S * (d_c + d_rope) + H * (d_c + d_rope) + H * S))
        ops.append(("p @ latent rows", lambda S: H * S * d_c,
                    lambda S: H * S + S * d_c + H * d_c))
        ops.append(("o_c @ W_UV", lambda S: H * d_c * d_v,
                    lambda S: H * d_c + H * d_v * d_c + H * d_v))
    else:
        raise ValueError(variant)
    return ops


def counts(variant: str, S: int, **dims) -> Dict[str, int]:
    ops = variant_ops(variant, **dims)
    return dict(flops=sum(f(S) for _, f, _ in ops), memops=sum(m(S) for _, _, m in ops))


def affine(variant: str, **dims) -> Dict[str, Tuple[int, int]]:
    """Counts as (constant, per-row coefficient) pairs; exact because every term is
    affine in S."""
    c0, c1 = counts(variant, 0, **dims), counts(variant, 1, **dims)
    return {k: (c0[k], c1[k] - c0[k]) for k in c0}


def mla_over_mha_ops(d_h: int, H: int, d_c: int, d: int) -> float:
    """Scalar-op ratio of creating K and V with MLA (down-projection to d_c, then two
    up-projections) over MHA (two d -> d_h*H projections), per token
    (Multi-Head Latent Attention, 3.1, eq. 3.1.2)."""
    mla = (d * d_c) + 2 * (d_c * d_h * H)
    mha = 2 * (d * d_h * H)
    return mla / mha
