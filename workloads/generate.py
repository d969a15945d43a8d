"""Seeded synthetic inputs for one MLA decode step.

One CPU ``torch.Generator`` per call, seeded, with a fixed draw order:

1. latent cache ``[B, S_max, d_c + d_rope]`` ~ N(0, 1)  (k_rope taken as already rotated)
2. ``q_nope [B, H, d_nope]`` ~ N(0, 1)
3. ``q_rope [B, H, d_rope]`` ~ N(0, 1)
4. ``W_UK [H, d_nope, d_c]`` ~ N(0, std^2)
5. ``W_UV [H, d_v, d_c]`` ~ N(0, std^2)
6. per-sequence lengths (ragged workloads only), uniform in [lo, hi]
7. the rows to scale (long-context workload only): round(frac * len_b) rows of
   sequence b chosen by a seeded permutation; whole 576-wide rows are scaled.

With ``q_len`` > 1 the queries have B * q_len rows (row b * q_len + i is token i
of sequence b) and ``positions[b * q_len + i] = len_b - q_len + i``.

Values are drawn in fp32 and then rounded once to the storage type (bf16 by
round-to-nearest-even; an FP8 cache to E4M3 by round-to-nearest-even, with
queries and weights bf16), so the CUDA path and the oracle read identical bits.
Positions are ``len_b - 1``: the cache already holds the current token's row.

This module holds none of the method's arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from .configs import MlaConfig


@dataclass
class MlaInputs:
    cfg: MlaConfig
    cache: torch.Tensor      # [B, S_max, row], storage dtype, CPU
    q_nope: torch.Tensor     # [B * q_len, H, d_nope]
    q_rope: torch.Tensor     # [B * q_len, H, d_rope]
    w_uk: torch.Tensor       # [H, d_nope, d_c]
    w_uv: torch.Tensor       # [H, d_v, d_c]
    lengths: torch.Tensor    # [B] int32
    positions: torch.Tensor  # [B * q_len] int32

    def as_float64_numpy(self, b: Optional[int] = None):
        """Exact fp64 copies (bf16 and fp32 values are exactly representable).

        An FP8 cache is handed over as its raw E4M3 codes (``cache_e4m3``,
        uint8) with ``cache`` None: decoding the format is left to the reader.
        """
        sl = slice(None) if b is None else slice(b, b + 1)
        f = lambda t: t.to(torch.float64).numpy()
        fp8 = self.cache.dtype == FP8
        return dict(
            cache=None if fp8 else f(self.cache[sl]),
            cache_e4m3=self.cache[sl].view(torch.uint8).numpy() if fp8 else None,
            q_nope=f(self.q_nope[sl]), q_rope=f(self.q_rope[sl]),
            w_uk=f(self.w_uk), w_uv=f(self.w_uv),
            lengths=self.lengths[sl].numpy().astype("int64"),
            positions=self.positions[sl].numpy().astype("int64"))


FP8 = torch.float8_e4m3fn


def _storage(cfg: MlaConfig) -> torch.dtype:
    """Storage type of queries and weights (bf16 also for an FP8 cache)."""
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def cache_storage(cfg: MlaConfig) -> torch.dtype:
    return FP8 if cfg.dtype == "fp8" else _storage(cfg)


def make_inputs(cfg: MlaConfig, seed: int = 0, poison_tail: bool = False,
                lengths: Optional[torch.Tensor] = None) -> MlaInputs:
    """Draw the inputs of ``cfg`` from ``seed``.

    ``poison_tail`` fills every cache row at or past ``lengths[b]`` with NaN, so
    that any read of the masked tail that reaches the arithmetic shows up.
    ``lengths`` overrides the drawn lengths (edge-case tests).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B, H, S = cfg.batch, cfg.heads, cfg.s_max
    st = _storage(cfg)

    cache = torch.randn((B, S, cfg.row), generator=g, dtype=torch.float32)
    q_nope = torch.randn((B * cfg.q_len, H, cfg.d_nope), generator=g, dtype=torch.float32)
    q_rope = torch.randn((B * cfg.q_len, H, cfg.d_rope), generator=g, dtype=torch.float32)
    w_uk = torch.randn((H, cfg.d_nope, cfg.d_c), generator=g, dtype=torch.float32) * cfg.weight_std
    w_uv = torch.randn((H, cfg.d_v, cfg.d_c), generator=g, dtype=torch.float32) * cfg.weight_std

    if cfg.ragged is not None:
        lo, hi = cfg.ragged
        drawn = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    else:
        drawn = torch.full((B,), S, dtype=torch.int32)
    if lengths is not None:
        drawn = lengths.to(torch.int32).clone()

    if cfg.scaled_row_frac > 0.0:
        for b in range(B):
            n = int(drawn[b])
            k = int(round(cfg.scaled_row_frac * n))
            rows = torch.randperm(n, generator=g)[:k]
            cache[b, rows, :] *= cfg.scaled_row_gain

    if poison_tail:
        for b in range(B):
            cache[b, int(drawn[b]):, :] = float("nan")
    cache = cache.to(cache_storage(cfg))

    tok = torch.arange(cfg.q_len, dtype=torch.int32)
    positions = (drawn[:, None] - cfg.q_len + tok[None, :]).clamp(min=0).reshape(-1).to(torch.int32)
    return MlaInputs(cfg=cfg, cache=cache, q_nope=q_nope.to(st), q_rope=q_rope.to(st),
                     w_uk=w_uk.to(st), w_uv=w_uv.to(st), lengths=drawn, positions=positions)


@dataclass
class AppendInputs:
    cfg: MlaConfig
    x: torch.Tensor          # [B, hidden] storage dtype: the new token's hidden state
    w_kva: torch.Tensor      # [d_c + d_rope, hidden] storage dtype
    positions: torch.Tensor  # [B] int32: the row each token goes to


def make_append_inputs(cfg: MlaConfig, seed: int = 0) -> AppendInputs:
    """Inputs of the cache-append step: x ~ N(0, 1), W_kva ~ N(0, std^2), positions
    uniform in [0, s_max) -- drawn in that order from one seeded CPU generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    st = _storage(cfg)
    x = torch.randn((cfg.batch, cfg.hidden), generator=g, dtype=torch.float32)
    w = torch.randn((cfg.row, cfg.hidden), generator=g, dtype=torch.float32) * cfg.weight_std
    pos = torch.randint(0, cfg.s_max, (cfg.batch,), generator=g, dtype=torch.int64).to(torch.int32)
    return AppendInputs(cfg=cfg, x=x.to(st), w_kva=w.to(st), positions=pos)


@dataclass
class OutProjInputs:
    cfg: MlaConfig
    o: torch.Tensor          # [B, H, d_v] fp32: the heads' value outputs (out_proj's result)
    w_o: torch.Tensor        # [hidden, H * d_v] storage dtype


def make_wo_inputs(cfg: MlaConfig, seed: int = 0) -> OutProjInputs:
    """Inputs of the W^O projection: o ~ N(0, 1) in fp32, W_O ~ N(0, std^2), in that
    order from one seeded CPU generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    o = torch.randn((cfg.batch, cfg.heads, cfg.d_v), generator=g, dtype=torch.float32)
    w = torch.randn((cfg.hidden, cfg.heads * cfg.d_v), generator=g, dtype=torch.float32) * cfg.weight_std
    return OutProjInputs(cfg=cfg, o=o, w_o=w.to(_storage(cfg)))


@dataclass
class MaterializedInputs:
    base: MlaInputs          # cache, q_rope, w_uk, w_uv, lengths, positions (q_nope unused)
    x: torch.Tensor          # [B, hidden] storage dtype: the decoded tokens' hidden states
    w_q_nope: torch.Tensor   # [H, d_nope, hidden] storage dtype: the nope rows of q_proj per head
    w_o: torch.Tensor        # [hidden, H * d_v] storage dtype


def make_materialized_inputs(cfg: MlaConfig, seed: int = 0, **kw) -> MaterializedInputs:
    """Inputs of the materialised (W^KQ, W^OV) step: ``make_inputs(cfg, seed, **kw)``,
    then, from a second CPU generator seeded with 10000 + seed, x ~ N(0, 1),
    W_Q's nope rows ~ N(0, std^2) and W_O ~ N(0, std^2), in that order."""
    base = make_inputs(cfg, seed, **kw)
    g = torch.Generator(device="cpu")
    g.manual_seed(10000 + seed)
    st = _storage(cfg)
    B, H = cfg.batch, cfg.heads
    x = torch.randn((B, cfg.hidden), generator=g, dtype=torch.float32)
    wq = torch.randn((H, cfg.d_nope, cfg.hidden), generator=g, dtype=torch.float32) * cfg.weight_std
    wo = torch.randn((cfg.hidden, H * cfg.d_v), generator=g, dtype=torch.float32) * cfg.weight_std
    return MaterializedInputs(base=base, x=x.to(st), w_q_nope=wq.to(st), w_o=wo.to(st))
