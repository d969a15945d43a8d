"""GB300 (sm_103a) MLA decode: weight-absorbed Multi-Head Latent Attention over a
latent KV cache, as a C-ABI CUDA library with a thin Python binding.

The three library calls (``absorb_q``, ``decode_attn``, ``out_proj``) are
re-exported from the binding.  ``DecodeStep`` owns the intermediate device
buffers of one decode step (allocated through PyTorch) and runs the three
calls on the current stream.
"""
from __future__ import annotations

from typing import Optional

from ._binding import (_check, _stream, step_call, EXPORTED, LIB_PATH, MLA_BF16, MLA_FP8_E4M3, MLA_DEV_LENGTH_OUT_OF_RANGE,
                       MLA_DEV_PIPELINE_TIMEOUT, MLA_F32, MlaDims, MlaError, absorb_q, cache_append,
                       decode_attn, decode_attn_multi, decode_step_multi, multi_num_splits,
                       multi_workspace_bytes,
                       query_dims, wo_proj,
                       materialize_wkq, materialize_wov, absorb_q_materialized, ov_proj,
                       decode_attn_noalloc, decode_combine, decode_split, decode_step, dims,
                       dtype_code, heads_per_cta, load, num_splits, out_proj, plan,
                       set_launch_overlap, set_split_parts,
                       workspace_bytes)

__all__ = [
    "EXPORTED", "LIB_PATH", "MLA_BF16", "MLA_F32", "MLA_FP8_E4M3", "MLA_DEV_LENGTH_OUT_OF_RANGE",
    "MLA_DEV_PIPELINE_TIMEOUT", "MlaDims", "MlaError", "absorb_q", "decode_attn",
    "decode_attn_multi", "decode_step_multi", "multi_num_splits", "multi_workspace_bytes",
    "query_dims", "materialize_wkq", "materialize_wov",
    "absorb_q_materialized", "ov_proj",
    "decode_attn_noalloc", "decode_split", "decode_combine", "decode_step", "dims",
    "dtype_code", "load", "num_splits", "out_proj", "workspace_bytes", "DecodeStep", "HostStep",
    "cache_append", "wo_proj", "set_launch_overlap", "plan", "set_split_parts", "heads_per_cta",
]


class DecodeStep:
    """One MLA decode step for a fixed (batch, heads, s_max, dtype).

    ``dtype`` is the cache's element type: torch.bfloat16, torch.float32, or
    torch.float8_e4m3fn (an E4M3 cache with bf16 queries and weights).

    ``run`` takes device tensors: q_nope [R,H,128], q_rope [R,H,64],
    cache [B,s_max,576], lengths [B] int32, positions [R] int32,
    w_uk [H,128,512], w_uv [H,128,512]; it returns o [R,H,128] fp32 (a buffer
    reused by the next call).  R = B * q_len: with ``q_len`` > 1 each sequence
    decodes q_len new tokens at once (row b * q_len + i is token i of sequence
    b, at position lengths[b] - q_len + i, causal within the block).
    """

    def __init__(self, batch: int, heads: int, s_max: int, dtype, device="cuda",
                 num_splits_requested: int = 0, rope_base: float = 10000.0,
                 softmax_scale: Optional[float] = None, q_len: int = 1):
        import torch
        self.dims = dims(batch, heads, s_max, dtype_code(dtype))
        self.q_len = q_len
        self.qdims = query_dims(self.dims, q_len)     # the query side: B * q_len rows
        self.splits_requested = num_splits_requested
        self.splits = (multi_num_splits(self.dims, q_len, num_splits_requested) if q_len > 1
                       else num_splits(self.dims, num_splits_requested))
        self.rope_base = rope_base
        self.scale = softmax_scale if softmax_scale is not None else (128 + 64) ** -0.5
        dev = torch.device(device)
        rows = batch * q_len
        self.q_abs = torch.empty((rows, heads, 512), dtype=torch.float32, device=dev)
        self.q_pe = torch.empty((rows, heads, 64), dtype=torch.float32, device=dev)
        self.o_c = torch.empty((rows, heads, 512), dtype=torch.float32, device=dev)
        self.lse = torch.empty((rows, heads), dtype=torch.float32, device=dev)
        self.out = torch.empty((rows, heads, 128), dtype=torch.float32, device=dev)
        nbytes = (multi_workspace_bytes(self.dims, q_len, num_splits_requested) if q_len > 1
                  else workspace_bytes(self.dims, num_splits_requested))
        self.workspace = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def run(self, q_nope, q_rope, cache, lengths, positions, w_uk, w_uv, stream=None, out=None):
        """The whole step in one library call (mla_decode_step, or
        mla_decode_step_multi for q_len > 1).

        q_nope, q_rope, lengths, positions and ``out`` (o, default: this step's
        device buffer) may be pinned host tensors, read and written by the
        kernels directly.
        """
        o = self.out if out is None else out
        if self.q_len > 1:
            decode_step_multi(self.dims, self.q_len, q_nope, q_rope, w_uk, positions, cache,
                              lengths, w_uv, self.workspace, self.q_abs, self.q_pe, self.o_c, o,
                              self.scale, self.rope_base, self.splits_requested, self.lse,
                              self.status, stream)
            return o
        decode_step(self.dims, q_nope, q_rope, w_uk, positions, cache, lengths, w_uv,
                    self.workspace, self.q_abs, self.q_pe, self.o_c, o, self.scale,
                    self.rope_base, self.splits_requested, self.lse, self.status, stream)
        return o

    def run_calls(self, q_nope, q_rope, cache, lengths, positions, w_uk, w_uv, stream=None):
        """The same step as the three separate calls absorb_q, decode_attn (or
        decode_attn_multi), out_proj."""
        absorb_q(self.qdims, q_nope, q_rope, w_uk, positions, self.q_abs, self.q_pe,
                 self.rope_base, stream)
        if self.q_len > 1:
            decode_attn_multi(self.dims, self.q_len, self.q_abs, self.q_pe, cache, lengths,
                              self.o_c, self.workspace, self.scale, self.splits_requested,
                              self.lse, self.status, stream)
        else:
            decode_attn(self.dims, self.q_abs, self.q_pe, cache, lengths, self.o_c,
                        self.workspace, self.scale, self.splits_requested, self.lse,
                        self.status, stream)
        out_proj(self.qdims, self.o_c, w_uv, self.out, stream)
        return self.out

    def capture(self, cache, w_uk, w_uv):
        """Capture one whole step from host memory as a CUDA graph.

        The returned ``HostStep`` keeps ``cache``, ``w_uk``, ``w_uv`` and this
        step alive for as long as it exists.

        Returns a ``HostStep``: pinned host tensors ``q_nope``, ``q_rope``,
        ``lengths``, ``positions`` (the step's inputs, filled by the caller) and
        ``out`` (o, written by the step), ``replay()`` and ``launch()``.  Both
        run mla_decode_step (mla_decode_step_multi for several tokens per
        sequence) on the host tensors themselves: its kernels read the inputs
        and write o over the host link, with no copies.  ``replay()`` replays
        the captured graph; ``launch()`` makes the call directly with arguments
        converted at capture, so that consecutive steps overlap.
        """
        return HostStep(self, cache, w_uk, w_uv)


class HostStep:
    """A decode step captured by ``DecodeStep.capture`` (see there)."""

    def __init__(self, step: DecodeStep, cache, w_uk, w_uv):
        import torch
        B, H, R = step.dims.batch, step.dims.heads, step.qdims.batch
        dt = torch.bfloat16 if cache.dtype == torch.float8_e4m3fn else cache.dtype
        elt = torch.tensor([], dtype=dt).element_size()
        pieces = [("q_nope", (R, H, 128), dt, elt), ("q_rope", (R, H, 64), dt, elt),
                  ("lengths", (B,), torch.int32, 4), ("positions", (R,), torch.int32, 4)]
        offs, off = [], 0
        for _, shape, _, e in pieces:
            n = 1
            for x in shape:
                n *= x
            offs.append(off)
            off += (n * e + 255) // 256 * 256        # every piece 256-byte aligned
        dev = step.q_abs.device
        self._h_block = torch.empty((off,), dtype=torch.uint8).pin_memory()

        def view(block, i):
            name, shape, dtype, e = pieces[i]
            n = 1
            for x in shape:
                n *= x
            return block[offs[i]:offs[i] + n * e].view(dtype).view(shape)

        self.q_nope, self.q_rope, self.lengths, self.positions = (view(self._h_block, i)
                                                                   for i in range(4))
        self.out = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
        # Bytes that cross the host link each step: the kernels read the inputs
        # and write o in place (mla_decode_step and mla_decode_step_multi accept
        # page-locked host buffers).
        self.h2d_bytes = sum(t.numel() * t.element_size()
                             for t in (self.q_nope, self.q_rope, self.lengths, self.positions))
        self.d2h_bytes = self.out.numel() * self.out.element_size()

        h = (self.q_nope, self.q_rope, self.lengths, self.positions)
        # The graph holds raw addresses: keep every tensor it reads or writes (and
        # the step that owns the intermediates) alive as long as this object.
        self._keep = (step, cache, w_uk, w_uv)

        def body():
            step.run(h[0], h[1], cache, h[2], h[3], w_uk, w_uv, out=self.out)

        # One run outside capture (module loading, kernel attributes); the inputs
        # are whatever the block holds, so start from valid lengths.
        self.lengths.fill_(step.q_len)
        self.positions.zero_()
        self.q_nope.zero_()
        self.q_rope.zero_()
        body()
        torch.cuda.synchronize(dev)
        self._graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        with torch.cuda.graph(self._graph, stream=side):
            body()

        # launch(): the same library call made directly, without the graph, its
        # arguments checked and converted once here.  Consecutive launches let
        # each step's first kernel overlap the previous step's last one
        # (programmatic dependent launch), which separate graph replays cannot.
        self._call = step_call(step.dims, step.q_len, h[0], h[1], w_uk, h[3], cache, h[2], w_uv,
                               step.workspace, step.q_abs, step.q_pe, step.o_c, self.out,
                               step.scale, step.rope_base, step.splits_requested, step.lse,
                               step.status)

    def replay(self):
        """The step as one replay of its CUDA graph."""
        self._graph.replay()

    def launch(self, stream=None):
        """The step as one direct mla_decode_step call (its kernels launched on
        ``stream``, default the current one), on the same host buffers."""
        fn, args = self._call
        _check(fn(*args, _stream(stream)))
