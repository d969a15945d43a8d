"""GB300 (sm_103a) MLA decode: weight-absorbed Multi-Head Latent Attention over a
latent KV cache, as a C-ABI CUDA library with a thin Python binding.

The three library calls (``absorb_q``, ``decode_attn``, ``out_proj``) are
re-exported from the binding.  ``DecodeStep`` owns the intermediate device
buffers of one decode step (allocated through PyTorch) and runs the three
calls on the current stream.
"""
from __future__ import annotations

from typing import Optional

from ._binding import (EXPORTED, LIB_PATH, MLA_BF16, MLA_DEV_LENGTH_OUT_OF_RANGE,
                       MLA_DEV_PIPELINE_TIMEOUT, MLA_F32, MlaDims, MlaError, absorb_q, decode_attn,
                       decode_attn_noalloc, decode_combine, decode_split, dims, dtype_code, load,
                       num_splits, out_proj, workspace_bytes)

__all__ = [
    "EXPORTED", "LIB_PATH", "MLA_BF16", "MLA_F32", "MLA_DEV_LENGTH_OUT_OF_RANGE",
    "MLA_DEV_PIPELINE_TIMEOUT", "MlaDims", "MlaError", "absorb_q", "decode_attn",
    "decode_attn_noalloc", "decode_split", "decode_combine", "dims",
    "dtype_code", "load", "num_splits", "out_proj", "workspace_bytes", "DecodeStep",
]


class DecodeStep:
    """One MLA decode step for a fixed (batch, heads, s_max, dtype).

    ``run`` takes device tensors: q_nope [B,H,128], q_rope [B,H,64],
    cache [B,s_max,576], lengths [B] int32, positions [B] int32,
    w_uk [H,128,512], w_uv [H,128,512]; it returns o [B,H,128] fp32 (a buffer
    reused by the next call).
    """

    def __init__(self, batch: int, heads: int, s_max: int, dtype, device="cuda",
                 num_splits_requested: int = 0, rope_base: float = 10000.0,
                 softmax_scale: Optional[float] = None):
        import torch
        self.dims = dims(batch, heads, s_max, dtype_code(dtype))
        self.splits_requested = num_splits_requested
        self.splits = num_splits(self.dims, num_splits_requested)
        self.rope_base = rope_base
        self.scale = softmax_scale if softmax_scale is not None else (128 + 64) ** -0.5
        dev = torch.device(device)
        self.q_abs = torch.empty((batch, heads, 512), dtype=torch.float32, device=dev)
        self.q_pe = torch.empty((batch, heads, 64), dtype=torch.float32, device=dev)
        self.o_c = torch.empty((batch, heads, 512), dtype=torch.float32, device=dev)
        self.lse = torch.empty((batch, heads), dtype=torch.float32, device=dev)
        self.out = torch.empty((batch, heads, 128), dtype=torch.float32, device=dev)
        nbytes = workspace_bytes(self.dims, num_splits_requested)
        self.workspace = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def run(self, q_nope, q_rope, cache, lengths, positions, w_uk, w_uv, stream=None):
        absorb_q(self.dims, q_nope, q_rope, w_uk, positions, self.q_abs, self.q_pe,
                 self.rope_base, stream)
        decode_attn(self.dims, self.q_abs, self.q_pe, cache, lengths, self.o_c, self.workspace,
                    self.scale, self.splits_requested, self.lse, self.status, stream)
        out_proj(self.dims, self.o_c, w_uv, self.out, stream)
        return self.out
