"""ctypes binding of the C ABI in ``include/mla.h``.

Argument marshalling only: every step of the decode runs in the CUDA library.
Tensors are torch tensors on a CUDA device (PyTorch provides device memory and
streams); their data pointers, sizes and the current stream are passed through.
If the shared library is missing the calls raise: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmla_gb300.so")
CHECK_LIB_PATH = os.path.join(PKG, "libmla_gb300_check.so")   # the checked build

MLA_F32, MLA_BF16, MLA_FP8_E4M3 = 0, 1, 2
MLA_DEV_LENGTH_OUT_OF_RANGE = 1
MLA_DEV_PIPELINE_TIMEOUT = 2
MLA_DEV_BOUNDS = 4
STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
          3: "MLA_ERR_WORKSPACE", 4: "MLA_ERR_CUDA"}
EXPORTED = ("mla_absorb_q", "mla_decode_num_splits", "mla_decode_workspace_bytes",
            "mla_decode_attn", "mla_decode_split", "mla_decode_combine",
            "mla_decode_attn_noalloc", "mla_decode_attn_multi", "mla_decode_multi_num_splits",
            "mla_decode_multi_workspace_bytes", "mla_decode_step", "mla_decode_step_multi",
            "mla_out_proj", "mla_cache_append",
            "mla_wo_proj", "mla_materialize_wkq", "mla_materialize_wov",
            "mla_absorb_q_materialized", "mla_ov_proj",
            "mla_status_string", "mla_last_error_message", "mla_test_set_split_hooks",
            "mla_set_launch_overlap", "mla_decode_plan", "mla_test_set_split_debug",
            "mla_test_set_split_form", "mla_built_with_checks", "mla_debug_bounds_word",
            "mla_set_split_parts", "mla_decode_heads_per_cta")


class MlaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("d_c", ctypes.c_int32),
                ("d_rope", ctypes.c_int32), ("d_nope", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("s_max", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class MlaError(RuntimeError):
    def __init__(self, code: int, detail: str):
        super().__init__(f"{STATUS.get(code, code)}: {detail}")
        self.code = code


_lib = None


def load(path: Optional[str] = None):
    """Load the shared library (once) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library {p} is not built; run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(MlaDims)
    lib.mla_absorb_q.argtypes = [D, P, P, P, P, ctypes.c_double, P, P, P]
    lib.mla_absorb_q.restype = ctypes.c_int
    lib.mla_decode_num_splits.argtypes = [D, I32]
    lib.mla_decode_num_splits.restype = I32
    lib.mla_decode_workspace_bytes.argtypes = [D, I32]
    lib.mla_decode_workspace_bytes.restype = SZ
    lib.mla_decode_attn.argtypes = [D, P, P, P, P, ctypes.c_float, I32, P, SZ, P, P, P, P]
    lib.mla_decode_attn.restype = ctypes.c_int
    lib.mla_decode_split.argtypes = [D, P, P, P, P, ctypes.c_float, I32, P, SZ, P, P]
    lib.mla_decode_split.restype = ctypes.c_int
    lib.mla_decode_combine.argtypes = [D, P, I32, P, SZ, P, P, P]
    lib.mla_decode_combine.restype = ctypes.c_int
    lib.mla_decode_attn_multi.argtypes = [D, I32, P, P, P, P, ctypes.c_float, I32, P, SZ, P, P, P,
                                          P]
    lib.mla_decode_attn_multi.restype = ctypes.c_int
    lib.mla_decode_multi_num_splits.argtypes = [D, I32, I32]
    lib.mla_decode_multi_num_splits.restype = I32
    lib.mla_decode_multi_workspace_bytes.argtypes = [D, I32, I32]
    lib.mla_decode_multi_workspace_bytes.restype = SZ
    lib.mla_decode_attn_noalloc.argtypes = [D, P, P, P, P, ctypes.c_float, I32, P, P, P, P]
    lib.mla_decode_attn_noalloc.restype = ctypes.c_int
    lib.mla_decode_step.argtypes = [D, P, P, P, P, ctypes.c_double, P, P, ctypes.c_float, I32, P,
                                    P, SZ, P, P, P, P, P, P, P]
    lib.mla_decode_step.restype = ctypes.c_int
    lib.mla_decode_step_multi.argtypes = [D, I32, P, P, P, P, ctypes.c_double, P, P, ctypes.c_float,
                                          I32, P, P, SZ, P, P, P, P, P, P, P]
    lib.mla_decode_step_multi.restype = ctypes.c_int
    lib.mla_cache_append.argtypes = [D, I32, P, P, P, ctypes.c_double, P, P, P]
    lib.mla_cache_append.restype = ctypes.c_int
    lib.mla_wo_proj.argtypes = [D, I32, P, P, P, P]
    lib.mla_wo_proj.restype = ctypes.c_int
    lib.mla_materialize_wkq.argtypes = [D, I32, P, P, P, P]
    lib.mla_materialize_wkq.restype = ctypes.c_int
    lib.mla_materialize_wov.argtypes = [D, I32, P, P, P, P]
    lib.mla_materialize_wov.restype = ctypes.c_int
    lib.mla_absorb_q_materialized.argtypes = [D, I32, P, P, P, P, ctypes.c_double, P, P, P]
    lib.mla_absorb_q_materialized.restype = ctypes.c_int
    lib.mla_ov_proj.argtypes = [D, I32, P, P, P, P]
    lib.mla_ov_proj.restype = ctypes.c_int
    lib.mla_out_proj.argtypes = [D, P, P, P, P]
    lib.mla_out_proj.restype = ctypes.c_int
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_last_error_message.argtypes = []
    lib.mla_last_error_message.restype = ctypes.c_char_p
    lib.mla_test_set_split_hooks.argtypes = [ctypes.c_uint64, I32]
    lib.mla_test_set_split_hooks.restype = None
    lib.mla_set_launch_overlap.argtypes = [I32]
    lib.mla_set_launch_overlap.restype = None
    lib.mla_test_set_split_debug.argtypes = [P]
    lib.mla_test_set_split_debug.restype = None
    lib.mla_test_set_split_form.argtypes = [I32]
    lib.mla_test_set_split_form.restype = None
    lib.mla_set_split_parts.argtypes = [I32]
    lib.mla_set_split_parts.restype = ctypes.c_int
    lib.mla_decode_heads_per_cta.argtypes = [D]
    lib.mla_decode_heads_per_cta.restype = I32
    lib.mla_built_with_checks.argtypes = []
    lib.mla_built_with_checks.restype = I32
    lib.mla_debug_bounds_word.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    lib.mla_debug_bounds_word.restype = ctypes.c_int
    lib.mla_decode_plan.argtypes = [D, I32, ctypes.POINTER(I32), ctypes.POINTER(I32),
                                    ctypes.POINTER(I32)]
    lib.mla_decode_plan.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def set_launch_overlap(enable: bool) -> None:
    """Programmatic dependent launch on (default) or off for later launches."""
    load().mla_set_launch_overlap(1 if enable else 0)


def set_split_parts(parts: int) -> None:
    """0: the library's choice (one bf16 part of the query and P at multiples of
    64 heads); 2: hi + lo parts everywhere."""
    _check(load().mla_set_split_parts(int(parts)))


def heads_per_cta(d: "MlaDims") -> int:
    """Heads per split CTA under the current set_split_parts (64: one part)."""
    return int(load().mla_decode_heads_per_cta(ctypes.byref(d)))


def _check(code: int):
    if code != 0:
        raise MlaError(code, load().mla_last_error_message().decode())


def dims(batch: int, heads: int, s_max: int, dtype: int, d_c: int = 512, d_rope: int = 64,
         d_nope: int = 128, d_v: int = 128) -> MlaDims:
    return MlaDims(batch, heads, d_c, d_rope, d_nope, d_v, s_max, dtype)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    """The raw cudaStream_t of ``stream``, default the current device's current
    stream (read without building a torch.cuda.Stream object: that costs a few
    microseconds per call, as much as a kernel launch)."""
    import torch
    if stream is not None:
        return stream.cuda_stream
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch._C._cuda_getDevice())
    return torch.cuda.current_stream().cuda_stream


def dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.bfloat16:
        return MLA_BF16
    if torch_dtype == torch.float32:
        return MLA_F32
    if torch_dtype == torch.float8_e4m3fn:   # an E4M3 cache; queries and weights bf16
        return MLA_FP8_E4M3
    raise TypeError(f"unsupported dtype {torch_dtype}")


def _require(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(*ts):
    for t in ts:
        if t is not None:
            _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")


def _cuda_or_pinned(*ts):
    for t in ts:
        if t is not None:
            _require(t.is_contiguous() and (t.is_cuda or t.is_pinned()),
                     "tensors must be contiguous CUDA tensors or pinned host tensors")


def num_splits(d: MlaDims, requested: int = 0) -> int:
    return int(load().mla_decode_num_splits(ctypes.byref(d), int(requested)))


def plan(d: MlaDims, requested: int = 0):
    """(splits, chunk rows, persistent) of the split for `requested` chunks."""
    sp, ch, pe = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().mla_decode_plan(ctypes.byref(d), int(requested), ctypes.byref(sp),
                                  ctypes.byref(ch), ctypes.byref(pe)))
    return sp.value, ch.value, bool(pe.value)


def workspace_bytes(d: MlaDims, requested: int = 0) -> int:
    return int(load().mla_decode_workspace_bytes(ctypes.byref(d), int(requested)))


def absorb_q(d: MlaDims, q_nope, q_rope, w_uk, positions, q_abs, q_pe, rope_base: float = 10000.0,
             stream=None) -> None:
    """q_abs = q_nope . W_UK per head; q_pe = RoPE(q_rope, positions)."""
    _cuda_contig(q_nope, q_rope, w_uk, positions, q_abs, q_pe)
    _check(load().mla_absorb_q(ctypes.byref(d), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk),
                               _ptr(positions), float(rope_base), _ptr(q_abs), _ptr(q_pe),
                               _stream(stream)))


def decode_attn(d: MlaDims, q_abs, q_pe, cache, lengths, o_c, workspace, softmax_scale: float,
                num_splits_requested: int = 0, lse=None, dev_status=None, stream=None) -> None:
    """Split-KV attention over the latent cache followed by the LSE combine."""
    _cuda_contig(q_abs, q_pe, cache, lengths, o_c, workspace, lse, dev_status)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().mla_decode_attn(ctypes.byref(d), _ptr(q_abs), _ptr(q_pe), _ptr(cache),
                                  _ptr(lengths), float(softmax_scale), int(num_splits_requested),
                                  _ptr(workspace), nbytes, _ptr(o_c), _ptr(lse),
                                  _ptr(dev_status), _stream(stream)))


def decode_split(d: MlaDims, q_abs, q_pe, cache, lengths, workspace, softmax_scale: float,
                 num_splits_requested: int = 0, dev_status=None, stream=None) -> None:
    """First half of decode_attn: per-chunk partial outputs into the workspace."""
    _cuda_contig(q_abs, q_pe, cache, lengths, workspace, dev_status)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().mla_decode_split(ctypes.byref(d), _ptr(q_abs), _ptr(q_pe), _ptr(cache),
                                   _ptr(lengths), float(softmax_scale),
                                   int(num_splits_requested), _ptr(workspace), nbytes,
                                   _ptr(dev_status), _stream(stream)))


def decode_combine(d: MlaDims, lengths, workspace, o_c, num_splits_requested: int = 0, lse=None,
                   stream=None) -> None:
    """Second half of decode_attn: log-sum-exp merge of the chunk partials."""
    _cuda_contig(lengths, workspace, o_c, lse)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().mla_decode_combine(ctypes.byref(d), _ptr(lengths), int(num_splits_requested),
                                     _ptr(workspace), nbytes, _ptr(o_c), _ptr(lse),
                                     _stream(stream)))


def query_dims(d: MlaDims, q_len: int) -> MlaDims:
    """The dims of the query side of a q_len-token step: batch B * q_len."""
    return MlaDims(d.batch * q_len, d.heads, d.d_c, d.d_rope, d.d_nope, d.d_v, d.s_max, d.dtype)


def multi_num_splits(d: MlaDims, q_len: int, requested: int = 0) -> int:
    """Chunks per sequence that decode_attn_multi uses (d: the cache's dims)."""
    return int(load().mla_decode_multi_num_splits(ctypes.byref(d), int(q_len), int(requested)))


def multi_workspace_bytes(d: MlaDims, q_len: int, requested: int = 0) -> int:
    """Workspace bytes decode_attn_multi needs (d: the cache's dims)."""
    return int(load().mla_decode_multi_workspace_bytes(ctypes.byref(d), int(q_len),
                                                       int(requested)))


def decode_attn_multi(d: MlaDims, q_len: int, q_abs, q_pe, cache, lengths, o_c, workspace,
                      softmax_scale: float, num_splits_requested: int = 0, lse=None,
                      dev_status=None, stream=None) -> None:
    """decode_attn for q_len new tokens per sequence, causal within the block.

    ``d`` describes the cache (B sequences); q_abs, q_pe, o_c and lse have
    B * q_len rows (row b * q_len + i is token i of sequence b).
    """
    _cuda_contig(q_abs, q_pe, cache, lengths, o_c, workspace, lse, dev_status)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().mla_decode_attn_multi(ctypes.byref(d), int(q_len), _ptr(q_abs), _ptr(q_pe),
                                        _ptr(cache), _ptr(lengths), float(softmax_scale),
                                        int(num_splits_requested), _ptr(workspace), nbytes,
                                        _ptr(o_c), _ptr(lse), _ptr(dev_status),
                                        _stream(stream)))


def decode_attn_noalloc(d: MlaDims, q_abs, q_pe, cache, lengths, o_c, softmax_scale: float,
                        num_splits_requested: int = 0, lse=None, dev_status=None,
                        stream=None) -> None:
    """decode_attn with the library's fixed scratch in place of a workspace.

    For hosts that cannot allocate device memory while decoding; the call
    allocates nothing.  Calls that overlap on the GPU share that scratch and race.
    """
    _cuda_contig(q_abs, q_pe, cache, lengths, o_c, lse, dev_status)
    _check(load().mla_decode_attn_noalloc(ctypes.byref(d), _ptr(q_abs), _ptr(q_pe), _ptr(cache),
                                          _ptr(lengths), float(softmax_scale),
                                          int(num_splits_requested), _ptr(o_c), _ptr(lse),
                                          _ptr(dev_status), _stream(stream)))


def decode_step(d: MlaDims, q_nope, q_rope, w_uk, positions, cache, lengths, w_uv, workspace,
                q_abs, q_pe, o_c, out, softmax_scale: float, rope_base: float = 10000.0,
                num_splits_requested: int = 0, lse=None, dev_status=None, stream=None) -> None:
    """absorb_q, decode_attn and out_proj in one call (bf16: fused combine + W_UV).

    q_nope, q_rope, positions, lengths and out may be pinned host tensors: the
    kernels then read and write them over the host link, with no copies.
    """
    _cuda_contig(w_uk, cache, w_uv, workspace, q_abs, q_pe, o_c, lse, dev_status)
    _cuda_or_pinned(q_nope, q_rope, positions, lengths, out)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().mla_decode_step(ctypes.byref(d), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk),
                                  _ptr(positions), float(rope_base), _ptr(cache), _ptr(lengths),
                                  float(softmax_scale), int(num_splits_requested), _ptr(w_uv),
                                  _ptr(workspace), nbytes, _ptr(q_abs), _ptr(q_pe), _ptr(o_c),
                                  _ptr(lse), _ptr(out), _ptr(dev_status), _stream(stream)))


def decode_step_multi(d: MlaDims, q_len: int, q_nope, q_rope, w_uk, positions, cache, lengths,
                      w_uv, workspace, q_abs, q_pe, o_c, out, softmax_scale: float,
                      rope_base: float = 10000.0, num_splits_requested: int = 0, lse=None,
                      dev_status=None, stream=None) -> None:
    """decode_step for q_len tokens per sequence (d: the cache's dims; the query
    side has B * q_len rows).  The step's inputs and out may be pinned host tensors."""
    _cuda_contig(w_uk, cache, w_uv, workspace, q_abs, q_pe, o_c, lse, dev_status)
    _cuda_or_pinned(q_nope, q_rope, positions, lengths, out)
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().mla_decode_step_multi(ctypes.byref(d), int(q_len), _ptr(q_nope), _ptr(q_rope),
                                        _ptr(w_uk), _ptr(positions), float(rope_base),
                                        _ptr(cache), _ptr(lengths), float(softmax_scale),
                                        int(num_splits_requested), _ptr(w_uv), _ptr(workspace),
                                        nbytes, _ptr(q_abs), _ptr(q_pe), _ptr(o_c), _ptr(lse),
                                        _ptr(out), _ptr(dev_status), _stream(stream)))


def step_call(d: MlaDims, q_len: int, q_nope, q_rope, w_uk, positions, cache, lengths, w_uv,
              workspace, q_abs, q_pe, o_c, out, softmax_scale: float, rope_base: float,
              num_splits_requested: int, lse, dev_status):
    """The checked arguments of mla_decode_step (q_len 1) or mla_decode_step_multi,
    converted once: returns (function, arguments without the stream), for callers
    that make the same call every step (HostStep.launch).  The tensors must stay
    alive and in place while the arguments are used."""
    _cuda_contig(w_uk, cache, w_uv, workspace, q_abs, q_pe, o_c, lse, dev_status)
    _cuda_or_pinned(q_nope, q_rope, positions, lengths, out)
    nbytes = workspace.numel() * workspace.element_size()
    lib = load()
    tail = (_ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(positions), float(rope_base),
            _ptr(cache), _ptr(lengths), float(softmax_scale), int(num_splits_requested),
            _ptr(w_uv), _ptr(workspace), nbytes, _ptr(q_abs), _ptr(q_pe), _ptr(o_c), _ptr(lse),
            _ptr(out), _ptr(dev_status))
    if q_len == 1:
        return lib.mla_decode_step, (ctypes.byref(d),) + tail
    return lib.mla_decode_step_multi, (ctypes.byref(d), int(q_len)) + tail


def out_proj(d: MlaDims, o_c, w_uv, out, stream=None) -> None:
    """o = W_UV . o_c per head."""
    _cuda_contig(o_c, w_uv, out)
    _check(load().mla_out_proj(ctypes.byref(d), _ptr(o_c), _ptr(w_uv), _ptr(out), _stream(stream)))


def cache_append(d: MlaDims, x, w_kva, positions, cache, rope_base: float = 10000.0,
                 dev_status=None, stream=None) -> None:
    """Write the new token of each sequence into the cache at positions[b]."""
    _cuda_contig(x, w_kva, positions, cache, dev_status)
    _check(load().mla_cache_append(ctypes.byref(d), int(x.shape[-1]), _ptr(x), _ptr(w_kva),
                                   _ptr(positions), float(rope_base), _ptr(cache),
                                   _ptr(dev_status), _stream(stream)))


def wo_proj(d: MlaDims, o, w_o, y, stream=None) -> None:
    """y = concat_h(o[:, h, :]) . W_O^T."""
    _cuda_contig(o, w_o, y)
    _check(load().mla_wo_proj(ctypes.byref(d), int(w_o.shape[0]), _ptr(o), _ptr(w_o), _ptr(y),
                              _stream(stream)))


def materialize_wkq(d: MlaDims, w_q_nope, w_uk, w_kq, stream=None) -> None:
    """W^KQ[h*512 + c, i] = sum_d w_uk[h, d, c] w_q_nope[h, d, i] (once per model)."""
    _cuda_contig(w_q_nope, w_uk, w_kq)
    _check(load().mla_materialize_wkq(ctypes.byref(d), int(w_q_nope.shape[-1]), _ptr(w_q_nope),
                                      _ptr(w_uk), _ptr(w_kq), _stream(stream)))


def materialize_wov(d: MlaDims, w_o, w_uv, w_ov, stream=None) -> None:
    """W^OV[n, h*512 + c] = sum_e w_o[n, h*128 + e] w_uv[h, e, c] (once per model)."""
    _cuda_contig(w_o, w_uv, w_ov)
    _check(load().mla_materialize_wov(ctypes.byref(d), int(w_o.shape[0]), _ptr(w_o), _ptr(w_uv),
                                      _ptr(w_ov), _stream(stream)))


def absorb_q_materialized(d: MlaDims, x, w_kq, q_rope, positions, q_abs, q_pe,
                          rope_base: float = 10000.0, stream=None) -> None:
    """q_abs = W^KQ x per head; q_pe = RoPE(q_rope, positions)."""
    _cuda_contig(x, w_kq, q_rope, positions, q_abs, q_pe)
    _check(load().mla_absorb_q_materialized(ctypes.byref(d), int(x.shape[-1]), _ptr(x),
                                            _ptr(w_kq), _ptr(q_rope), _ptr(positions),
                                            float(rope_base), _ptr(q_abs), _ptr(q_pe),
                                            _stream(stream)))


def ov_proj(d: MlaDims, o_c, w_ov, y, stream=None) -> None:
    """y = W^OV . concat_h(o_c[:, h, :])."""
    _cuda_contig(o_c, w_ov, y)
    _check(load().mla_ov_proj(ctypes.byref(d), int(w_ov.shape[0]), _ptr(o_c), _ptr(w_ov), _ptr(y),
                              _stream(stream)))
