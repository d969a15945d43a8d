/*
 * mla.h -- C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * One decode step of DeepSeek Multi-Head Latent Attention in weight-absorbed
 * form over a latent KV cache, as three calls:
 *
 *   mla_absorb_q     q_abs = q_nope . W_UK (per head), q_pe = RoPE(q_rope, pos)
 *   mla_decode_attn  split-KV online-softmax attention of [q_abs || q_pe] against
 *                    the cached rows [c_kv || k_rope], then a log-sum-exp combine;
 *                    the output o_c stays in the latent space
 *   mla_out_proj     o = W_UV . o_c (per head)
 *
 * Sources: "Multi-Head Latent Attention" (Lior Sinai) sections 3.1 (C cache),
 * 3.3 (absorption, eq. 3.3.3), 3.6 (decoupled RoPE: score = nope part + RoPE
 * part, scaled by 1/sqrt(d_h + d_R), k_rope shared by all heads) and 3.7
 * (RoPE on adjacent pairs); "Deepseek V2 Lite Inference Engine in C", MLA
 * notes (absorbing W_UK without materialising it, cache row order
 * (kv_lora, k_rope)); "Transformer and KV Cache Basics" (decode is bound by
 * memory bandwidth; overflowing the cache is an error).
 *
 * Conventions for every call
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous, and
 *    must be 16-byte aligned.  The caller owns every buffer; the library
 *    allocates no device memory, keeps no per-call state and never
 *    synchronises the stream.  Work is enqueued on `stream` (a cudaStream_t;
 *    NULL means the legacy default stream) on the current device.
 *  - Argument errors are detected on the host before anything is enqueued and
 *    are returned as a status; nothing is launched then.  A failed launch
 *    returns MLA_ERR_CUDA.  mla_last_error_message() gives a one-line detail
 *    for the calling thread's most recent failure.
 *  - Element types: with dtype MLA_BF16 the cache, q_nope, q_rope and the
 *    weights are bf16 and all arithmetic accumulates in fp32; with MLA_F32
 *    they are fp32 and every step runs in fp32 (no TF32).  With
 *    MLA_FP8_E4M3 the cache elements are one-byte FP8 E4M3 numbers, used as
 *    they are (no scale; "Multi-Head Latent Attention" 3.1: an element takes
 *    1-4 bytes, FP8 to FP32), and q_nope, q_rope and the weights are bf16.
 *    Every result -- the absorbed query q_abs, the rotated q_pe, o_c, lse,
 *    the output o -- and the workspace are fp32 in every case (the bf16
 *    decode kernel feeds the fp32 query and the softmax weights to the
 *    tensor cores as hi + lo bf16 pairs, the FP8 kernel as four and three
 *    E4M3 parts).
 *  - Launch overlap: the kernels of mla_decode_attn (and of its halves), the
 *    bf16 kernel of mla_out_proj, and the fused tail of mla_decode_step are
 *    launched with programmatic stream serialization, so each may begin while
 *    the kernel before it on the stream is still running -- but only if that
 *    kernel allows it explicitly (griddepcontrol.launch_dependents), as these
 *    kernels and mla_absorb_q's do; after any other kernel, or a copy, they
 *    start as usual.  Within mla_decode_step (bf16 and FP8), when its decode
 *    grid fits in one wave on the device, the absorb kernel is launched that
 *    way too.  Before waiting for their predecessor they read only the cache
 *    and lengths (mla_decode_attn; the absorb inside mla_decode_step) or the
 *    weights (that absorb: w_uk; mla_out_proj and the fused tail: w_uv);
 *    everything else is read, and everything is written, after the wait.  So
 *    a kernel of the caller that allows early launch must not write those
 *    inputs.  mla_absorb_q on its own starts as usual.
 *  - Supported sizes: d_c = 512, d_rope = 64, d_nope = 128, d_v = 128;
 *    batch >= 1; s_max >= 1; heads >= 1 (a multiple of 16 for MLA_BF16 and
 *    MLA_FP8_E4M3).
 *    Anything else returns MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null or misaligned pointer, non-positive size */
  MLA_ERR_UNSUPPORTED = 2,   /* a size or dtype this build has no kernel for */
  MLA_ERR_WORKSPACE = 3,     /* workspace smaller than mla_decode_workspace_bytes() */
  MLA_ERR_CUDA = 4           /* a CUDA runtime call or kernel launch failed */
} mla_status;

typedef enum mla_dtype { MLA_F32 = 0, MLA_BF16 = 1, MLA_FP8_E4M3 = 2 } mla_dtype;

/* Problem sizes shared by the three calls. */
typedef struct mla_dims {
  int32_t batch;    /* B: sequences decoded in this step                      */
  int32_t heads;    /* H: attention heads                                     */
  int32_t d_c;      /* latent width of c_kv (512)                             */
  int32_t d_rope;   /* decoupled RoPE width (64)                              */
  int32_t d_nope;   /* per-head non-rotated query width (128)                 */
  int32_t d_v;      /* per-head value width (128)                             */
  int32_t s_max;    /* cache capacity: rows allocated per sequence            */
  int32_t dtype;    /* mla_dtype                                              */
} mla_dims;

/* Bits a kernel ORs into the optional device status word (see mla_decode_attn). */
#define MLA_DEV_LENGTH_OUT_OF_RANGE 1  /* some lengths[b] < 1 (< q_len) or > s_max */
#define MLA_DEV_PIPELINE_TIMEOUT 2     /* a bounded wait in a kernel's pipeline gave up */
#define MLA_DEV_BOUNDS 4               /* checked build: an index outside its buffer (skipped) */

/*
 * mla_absorb_q -- absorbed query and rotated RoPE query for one decode step.
 *
 *   q_abs[b,h,c] = sum_{d < d_nope} q_nope[b,h,d] * w_uk[h,d,c]
 *       (W_UK absorbed into the query side without materialising W_UK^T W_Q:
 *        Multi-Head Latent Attention 3.3; "Deepseek V2 Lite Inference Engine
 *        in C", absorption "without materializing WukWq")
 *   q_pe[b,h,2i:2i+2] = rotation of the pair (q_rope[b,h,2i], q_rope[b,h,2i+1])
 *       by the angle positions[b] * rope_base^(-2i/d_rope)
 *       (Multi-Head Latent Attention 3.7: complex multiply of adjacent pairs;
 *        positions counted from 0; the angle is formed in fp64)
 *
 * q_nope   [B, H, d_nope]   dtype           q_rope [B, H, d_rope] dtype
 * w_uk     [H, d_nope, d_c] dtype           positions [B] int32 (device)
 * q_abs    [B, H, d_c]      fp32 (out)      q_pe   [B, H, d_rope] fp32 (out)
 */
mla_status mla_absorb_q(const mla_dims* dims, const void* q_nope, const void* q_rope,
                        const void* w_uk, const int32_t* positions, double rope_base,
                        void* q_abs, void* q_pe, void* stream);

/*
 * mla_decode_num_splits -- the number of KV chunks per sequence that
 * mla_decode_attn will use for `requested` (0 = let the library choose from
 * the current device's SM count).  Chunks hold a multiple of 8 rows (of 128
 * rows when the split kernel runs persistent, see mla_decode_plan), so the
 * result can differ from `requested`.  Returns 0 for invalid dims.
 */
int32_t mla_decode_num_splits(const mla_dims* dims, int32_t requested);

/*
 * mla_decode_plan -- how mla_decode_attn (and mla_decode_split, the step calls
 * and mla_decode_attn_noalloc) cut the rows for `requested` chunks on the
 * current device.  Any output pointer may be NULL.
 *
 * splits      chunks per sequence (as mla_decode_num_splits); a sequence of
 *             length S_b has ceil(S_b / chunk) partials
 * chunk       rows per chunk (a multiple of 8; of 128 when persistent)
 * persistent  1: the bf16 split kernel (16 heads per CTA) runs as one CTA per
 *             SM, each CTA working through the chunks whose first 128-row tile
 *             falls in its equal share of all tiles, back to back; chosen when
 *             one CTA per chunk would need several waves and the library's
 *             estimate favours it.  0: one CTA per (head group, chunk, sequence).
 *             Results do not depend on it beyond rounding order.
 *
 * A chunk's partial is the exact softmax-normalised output of its rows and its
 * log-sum-exp (Multi-Head Latent Attention, 3.6 restated per chunk); the
 * combine merges them.  Returns MLA_OK or the dims' error status.
 */
mla_status mla_decode_plan(const mla_dims* dims, int32_t requested, int32_t* splits,
                           int32_t* chunk, int32_t* persistent);

/* Bytes of device workspace mla_decode_attn needs for `requested` splits. */
size_t mla_decode_workspace_bytes(const mla_dims* dims, int32_t requested);

/*
 * mla_decode_attn -- attention of the absorbed query against the latent cache.
 *
 * For sequence b with S_b = lengths[b] cached rows, head h, row t < S_b:
 *   s[t]   = softmax_scale * (q_abs[b,h,:] . cache[b,t,0:d_c]
 *                             + q_pe[b,h,:] . cache[b,t,d_c:d_c+d_rope])
 *   o_c[b,h,:] = sum_t softmax(s)[t] * cache[b,t,0:d_c]
 *   lse[b,h]   = log(sum_t exp(s[t]))               (natural log)
 * (Multi-Head Latent Attention 3.3 and 3.6: the nope part of the score is
 *  the latent row against the absorbed query, k_rope is shared by every head,
 *  and the output stays latent until W_UV is applied.)  softmax_scale is
 *  normally 1/sqrt(d_nope + d_rope).
 *
 * The rows of a sequence are cut into chunks of equal size; one kernel
 * computes every chunk's normalised partial output and lse into `workspace`,
 * a second kernel merges them: L = log sum_j exp(lse_j),
 * o_c = sum_j exp(lse_j - L) o_j.  Rows t >= S_b are never part of any
 * result; their contents may be anything, including NaN.
 *
 * q_abs   [B, H, d_c]       fp32       q_pe  [B, H, d_rope] fp32
 * cache   [B, s_max, d_c + d_rope] dtype; row t of sequence b is
 *         [c_kv (d_c) || k_rope (d_rope)], k_rope already rotated
 * lengths [B] int32 (device); 1 <= lengths[b] <= s_max
 * num_splits  chunks per sequence requested (0 = library's choice)
 * workspace   >= mla_decode_workspace_bytes(dims, num_splits) bytes, device,
 *             owned by the caller, contents need not be initialised
 * o_c     [B, H, d_c] fp32 (out)       lse [B, H] fp32 (out, may be NULL)
 * dev_status  optional device int32 (may be NULL).  Kernels OR
 *             MLA_DEV_* bits into it and never clear it; the caller zeroes
 *             it.  A length outside [1, s_max] cannot be checked on the host:
 *             the kernels clamp it to [0, s_max] (the cache overflow of
 *             "Transformer and KV Cache Basics" becomes an error bit), and a
 *             sequence with no rows gets o_c = 0 and lse = -inf.
 */
mla_status mla_decode_attn(const mla_dims* dims, const void* q_abs, const void* q_pe,
                           const void* cache, const int32_t* lengths, float softmax_scale,
                           int32_t num_splits, void* workspace, size_t workspace_bytes,
                           float* o_c, float* lse, int32_t* dev_status, void* stream);

/*
 * mla_decode_split / mla_decode_combine -- the two halves of mla_decode_attn,
 * for callers that schedule them separately (for example to time or overlap
 * them).  mla_decode_attn(...) is exactly mla_decode_split(...) followed by
 * mla_decode_combine(...) on the same stream with the same dims, lengths,
 * num_splits and workspace.
 *
 * mla_decode_split writes, for every chunk j of every sequence b with rows,
 * the chunk's normalised partial output o_j[b,j,h,:] and lse_j[b,j,h] into
 * the workspace (layout private to the library); chunks past S_b are not
 * written.  mla_decode_combine reads them back and writes o_c and lse as
 * described for mla_decode_attn.  Arguments have the meaning, layout and
 * error behaviour given above.
 */
mla_status mla_decode_split(const mla_dims* dims, const void* q_abs, const void* q_pe,
                            const void* cache, const int32_t* lengths, float softmax_scale,
                            int32_t num_splits, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream);
mla_status mla_decode_combine(const mla_dims* dims, const int32_t* lengths, int32_t num_splits,
                              const void* workspace, size_t workspace_bytes, float* o_c,
                              float* lse, void* stream);

/*
 * mla_decode_attn_multi -- mla_decode_attn for q_len new tokens per sequence
 * in one step (multi-token or speculative decoding).
 *
 * The cache already holds the step's q_len new rows, so for sequence b with
 * S_b = lengths[b] rows, token i (0 <= i < q_len) sits at position
 * S_b - q_len + i and attends rows t <= S_b - q_len + i: a key past the
 * query's own position is masked ("Transformer and KV Cache Basics", mask
 * design for multi-token decoding: prefill and decode handled alike, the
 * small upper-right triangle of the score matrix masked).  Each token's
 * score, softmax and latent output are those of mla_decode_attn with the
 * sequence cut to its first S_b - q_len + 1 + i rows; with q_len = 1 this is
 * mla_decode_attn exactly.
 *
 * Query-side tensors have one row per (sequence, token): row b*q_len + i.
 *   q_abs [B*q_len, H, d_c] fp32      q_pe [B*q_len, H, d_rope] fp32
 *   o_c   [B*q_len, H, d_c] fp32 (out) lse [B*q_len, H] fp32 (out, may be NULL)
 * (mla_absorb_q and mla_out_proj called with batch B*q_len and positions
 * S_b - q_len + i produce and consume them.)
 * dims  describes the cache: dims->batch = B sequences, cache
 *       [B, s_max, d_c + d_rope]; lengths [B] int32 (device),
 *       q_len <= lengths[b] <= s_max
 * q_len >= 1
 * workspace  >= mla_decode_multi_workspace_bytes(dims, q_len, num_splits)
 *       bytes (mla_decode_multi_num_splits(dims, q_len, num_splits) gives the
 *       chunk count used).
 * A length below q_len or above s_max sets MLA_DEV_LENGTH_OUT_OF_RANGE in
 * dev_status; a token left with no rows gets o_c = 0 and lse = -inf.
 * With a bf16 cache, an even q_len and a head count that is not a multiple of
 * 32, one CTA of the decode kernel takes two tokens x 16 heads, so that a
 * chunk's rows are read by q_len / 2 CTAs; otherwise each token's CTAs read
 * them (the reads of a row meet in L2).
 */
int32_t mla_decode_multi_num_splits(const mla_dims* dims, int32_t q_len, int32_t requested);
size_t mla_decode_multi_workspace_bytes(const mla_dims* dims, int32_t q_len, int32_t requested);
mla_status mla_decode_attn_multi(const mla_dims* dims, int32_t q_len, const void* q_abs,
                                 const void* q_pe, const void* cache, const int32_t* lengths,
                                 float softmax_scale, int32_t num_splits, void* workspace,
                                 size_t workspace_bytes, float* o_c, float* lse,
                                 int32_t* dev_status, void* stream);

/*
 * mla_decode_attn_noalloc -- mla_decode_attn for callers that cannot allocate
 * device memory.  The paper has no counterpart: it is a convenience of this
 * library.
 *
 * Who needs it: a host that reserved all device memory for its own pool at
 * start-up (a cudaMalloc there fails or breaks the pool's accounting), or a
 * latency-critical loop in which cudaMalloc and cudaFree would synchronise the
 * device.  This call allocates nothing: the chunk partials go to one fixed
 * array of MLA_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.  The caller still passes
 * inputs and outputs, with the meaning, layout and error behaviour given for
 * mla_decode_attn (which this call runs, with the array as its workspace).
 *
 * Limit: a call whose partials need more than MLA_NOALLOC_SCRATCH_BYTES
 * (mla_decode_workspace_bytes(dims, num_splits) > MLA_NOALLOC_SCRATCH_BYTES)
 * returns MLA_ERR_WORKSPACE and launches nothing.
 *
 * First call on a device (and in each CUDA context): it asks the runtime for
 * the array's device address with that device current and keeps it together
 * with the context's unique ID; make that first call before any stream capture
 * begins.  A later call from another context (after cudaDeviceReset, or with
 * another context current on the same device) asks again before it launches
 * anything, since the library's module and the array are loaded anew there.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents (nothing needs clearing: a call reads only what it wrote).
 * Calls whose kernels overlap on the GPU (other streams, other host threads)
 * race on it; order them on one stream or use mla_decode_attn.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB per device */
mla_status mla_decode_attn_noalloc(const mla_dims* dims, const void* q_abs, const void* q_pe,
                                   const void* cache, const int32_t* lengths,
                                   float softmax_scale, int32_t num_splits, float* o_c,
                                   float* lse, int32_t* dev_status, void* stream);

/*
 * mla_out_proj -- per-head value up-projection applied after attention.
 *
 *   o[b,h,e] = sum_{c < d_c} w_uv[h,e,c] * o_c[b,h,c]
 * (Multi-Head Latent Attention eq. 3.3.3, with W^O left to the caller.)
 *
 * o_c [B, H, d_c] fp32     w_uv [H, d_v, d_c] dtype     o [B, H, d_v] fp32 (out)
 */
mla_status mla_out_proj(const mla_dims* dims, const float* o_c, const void* w_uv, void* out,
                        void* stream);

/*
 * mla_cache_append -- write each sequence's new token into the latent cache.
 *
 *   y[b, :]        = x[b, :] . w_kva^T             (d_c + d_rope outputs)
 *   cache[b, positions[b], 0:d_c]          = y[b, 0:d_c]
 *   cache[b, positions[b], d_c:d_c+d_rope] = RoPE(y[b, d_c:], positions[b])
 * ("Deepseek V2 Lite Inference Engine in C", MLA notes: kv_a_proj fuses the KV
 *  down-projection and the shared RoPE key; "Multi-Head Latent Attention" 3.5:
 *  the latent row is what the cache keeps, and 3.7: the key is rotated at its
 *  position -- adjacent pairs, angle in fp64 -- before it is cached, which is
 *  the form mla_decode_attn reads.)  The new row is then attended with
 *  lengths[b] = positions[b] + 1.  fp32 accumulation; the row is rounded once
 *  to the cache dtype (MLA_FP8_E4M3: to nearest even, saturating at +-448;
 *  x and w_kva are then bf16).  No normalisation is applied (none is defined on the
 *  pages for this step).
 *
 * x      [B, hidden] dtype           w_kva [d_c + d_rope, hidden] dtype
 * positions [B] int32 (device); a position outside [0, s_max) writes nothing
 *        and sets MLA_DEV_LENGTH_OUT_OF_RANGE in dev_status (may be NULL)
 * cache  [B, s_max, d_c + d_rope] dtype (in/out: only the new rows change)
 * hidden must be a multiple of 128.
 */
mla_status mla_cache_append(const mla_dims* dims, int32_t hidden, const void* x,
                            const void* w_kva, const int32_t* positions, double rope_base,
                            void* cache, int32_t* dev_status, void* stream);

/*
 * mla_wo_proj -- the attention layer's output projection.
 *
 *   y[b, n] = sum_{h, e} w_o[n, h d_v + e] * o[b, h, e]
 * ("Multi-Head Latent Attention" eq. 3.3.3: W^O applied to the concatenated
 *  head outputs; o is mla_out_proj's result.)  fp32 accumulation.
 *
 * o [B, H, d_v] fp32     w_o [hidden, H d_v] dtype     y [B, hidden] fp32 (out)
 * hidden must be a multiple of 8 (and H d_v a multiple of 128 for MLA_BF16).
 */
mla_status mla_wo_proj(const mla_dims* dims, int32_t hidden, const float* o, const void* w_o,
                       float* y, void* stream);

/*
 * Materialised absorption: the pages' other form of the weight absorption,
 * where the products of the weights are formed once as matrices instead of
 * being applied right to left at every step ("Multi-Head Latent Attention"
 * 3.3, eq. 3.3.3 and 3.5; "Deepseek V2 Lite Inference Engine in C", MLA
 * notes: the materialised WukWq, per head).  With them a step is
 *   mla_absorb_q_materialized -> mla_decode_attn -> mla_ov_proj
 * and needs neither q_nope nor mla_out_proj nor mla_wo_proj.  The materialised
 * matrices are larger than the factors they come from (W^KQ holds H d_c d_in
 * values against H d_nope (d_c + d_in)); their rows are streamed once per step.
 *
 * mla_materialize_wkq -- W^KQ[h, c, i] = sum_{d < d_nope} w_uk[h, d, c] w_q_nope[h, d, i]
 *   w_q_nope [H, d_nope, d_in] dtype: the rows of the query projection whose
 *            output is q_nope (q_nope[b, h, :] = w_q_nope[h] . x[b, :])
 *   w_uk     [H, d_nope, d_c] dtype
 *   w_kq     [H * d_c, d_in] dtype (out): row h d_c + c is W^KQ[h, c, :]
 * mla_materialize_wov -- W^OV[n, h d_c + c] = sum_{e < d_v} w_o[n, h d_v + e] w_uv[h, e, c]
 *   w_o  [d_out, H * d_v] dtype     w_uv [H, d_v, d_c] dtype
 *   w_ov [d_out, H * d_c] dtype (out)
 * Both accumulate in fp32 and round each result once to the weight type
 * (nearest even for bf16; MLA_FP8_E4M3 means bf16 weights).  They are weight
 * transforms made once per model.
 *
 * mla_absorb_q_materialized -- the absorbed query straight from the hidden state:
 *   q_abs[b, h, c] = sum_{i < d_in} w_kq[h d_c + c, i] x[b, i]     (fp32 accumulation)
 *   q_pe = RoPE(q_rope, positions) exactly as mla_absorb_q computes it.
 *   x [B, d_in] dtype; d_in a multiple of 64.  Other arguments as mla_absorb_q.
 *
 * mla_ov_proj -- the layer output straight from the latent attention output:
 *   y[b, n] = sum_{h, c} w_ov[n, h d_c + c] o_c[b, h, c]            (fp32 accumulation)
 *   o_c [B, H, d_c] fp32 (mla_decode_attn's result); y [B, d_out] fp32 (out);
 *   d_out a multiple of 8.
 */
mla_status mla_materialize_wkq(const mla_dims* dims, int32_t d_in, const void* w_q_nope,
                               const void* w_uk, void* w_kq, void* stream);
mla_status mla_materialize_wov(const mla_dims* dims, int32_t d_out, const void* w_o,
                               const void* w_uv, void* w_ov, void* stream);
mla_status mla_absorb_q_materialized(const mla_dims* dims, int32_t d_in, const void* x,
                                     const void* w_kq, const void* q_rope,
                                     const int32_t* positions, double rope_base, float* q_abs,
                                     float* q_pe, void* stream);
mla_status mla_ov_proj(const mla_dims* dims, int32_t d_out, const float* o_c, const void* w_ov,
                       float* y, void* stream);

/*
 * mla_decode_step -- one whole decode step: mla_absorb_q, mla_decode_attn and
 * mla_out_proj in one call, with the same arguments, meanings and results
 * (q_abs, q_pe, o_c, lse and out are all written).
 *
 * With dtype MLA_BF16 or MLA_FP8_E4M3 and batch x heads <= 256 the combine and
 * the value up-projection run as one kernel (each CTA merges one (sequence,
 * head)'s chunk partials and applies 32 rows of W_UV[h] to them in fp32),
 * launched with programmatic stream serialization after the split kernel;
 * before its wait it reads only w_uv and lengths.  Larger batches run
 * mla_decode_combine and mla_out_proj, which read W_UV once per step.
 * With MLA_F32 the three calls run in order.  Every argument is checked before
 * anything is enqueued.  lse may be NULL.
 *
 * Host buffers for the step's own inputs and output: q_nope, q_rope,
 * positions, lengths and out may also be page-locked host memory (allocated
 * with cudaHostAlloc or registered with cudaHostRegister, so that the device
 * can address it).  The kernels then read the inputs and write o over the
 * host link themselves, with no copy of their own to enqueue; on a GB300
 * (NVLink-C2C) this costs about 2 us per step for the inputs and nothing
 * measurable for o.  The caller must not touch those host buffers until the
 * stream has passed the step.  Pageable host memory is refused with
 * MLA_ERR_INVALID_ARG before anything is enqueued.  Every other tensor (the
 * cache, the weights, q_abs, q_pe, o_c, lse, the workspace) must be device
 * memory, as for the other calls.
 */
mla_status mla_decode_step(const mla_dims* dims, const void* q_nope, const void* q_rope,
                           const void* w_uk, const int32_t* positions, double rope_base,
                           const void* cache, const int32_t* lengths, float softmax_scale,
                           int32_t num_splits, const void* w_uv, void* workspace,
                           size_t workspace_bytes, float* q_abs, float* q_pe, float* o_c,
                           float* lse, float* out, int32_t* dev_status, void* stream);

/*
 * mla_decode_step_multi -- mla_decode_step for q_len new tokens per sequence:
 * mla_absorb_q and mla_out_proj over the B*q_len query rows around
 * mla_decode_attn_multi (causal within the block), with the same launch
 * overlap, cache prefetch and host-buffer rules as mla_decode_step.
 * q_nope, q_rope [B*q_len, H, .], positions [B*q_len]; lengths [B];
 * q_abs, q_pe, o_c, lse, out have B*q_len rows; workspace >=
 * mla_decode_multi_workspace_bytes(dims, q_len, num_splits).  q_len = 1 is
 * mla_decode_step.
 */
mla_status mla_decode_step_multi(const mla_dims* dims, int32_t q_len, const void* q_nope,
                                 const void* q_rope, const void* w_uk, const int32_t* positions,
                                 double rope_base, const void* cache, const int32_t* lengths,
                                 float softmax_scale, int32_t num_splits, const void* w_uv,
                                 void* workspace, size_t workspace_bytes, float* q_abs,
                                 float* q_pe, float* o_c, float* lse, float* out,
                                 int32_t* dev_status, void* stream);

/* Static English name of a status code. */
const char* mla_status_string(mla_status status);

/* Detail of the calling thread's most recent failed call ("" if none). */
const char* mla_last_error_message(void);

/*
 * mla_set_launch_overlap -- whether the library's kernels are launched with
 * programmatic dependent launch (1, the default) or as plain launches (0).
 *
 * With overlap, a kernel may start while its predecessor on the stream is
 * still running: it prepares (tensor memory, barriers, weight and cache
 * prefetches) and waits on the device before it reads that predecessor's
 * results.  Without it, every launch starts only after the previous one has
 * finished, so a graph of back-to-back launches times each launch whole.
 * Results are the same either way.  Process-wide; read when a kernel is
 * enqueued (a graph keeps the launch form of its capture).  Not an operation
 * of the pages: a measurement switch of this library.
 */
void mla_set_launch_overlap(int32_t enable);

/*
 * mla_set_split_parts -- how the bf16 split kernel hands the fp32 absorbed
 * query and the softmax weights P to the tensor core (bf16 operands, fp32
 * accumulation in both forms).
 *
 *   0 (default)  the library's choice: where the head count is a multiple of
 *                64, one bf16 part each (round to nearest), 64 heads per CTA;
 *                otherwise two parts, as below.
 *   2            two parts at every head count: bf16(x) and bf16(x - bf16(x)),
 *                a rounding near 2^-17 relative (32 heads per CTA where the
 *                head count is a multiple of 32, else 16).
 *
 * One part rounds each query element and weight to bf16 (2^-9 relative): on
 * the V3 shape with N(0,1) rows and N(0,0.02^2) weights (Multi-Head Latent
 * Attention, 3.1: 128 heads) o_c stays near 2e-3 relative L2 of the exact
 * result, and the CTAs that read each cache row are halved.  Rows of large
 * magnitude (scores spread over tens of units) want two parts.  Process-wide,
 * read when a split is enqueued (a graph keeps the form of its capture).
 * Returns MLA_OK, or MLA_ERR_INVALID_ARG for another value.
 */
mla_status mla_set_split_parts(int32_t parts);

/*
 * mla_decode_heads_per_cta -- heads each CTA of the split kernel takes for
 * these dims under the current mla_set_split_parts: 64 (one bf16 part), 32 or
 * 16 (two parts) for a bf16 cache, 16 for FP8 (four and three E4M3 parts), 1
 * for fp32.  Returns 0 for invalid dims.
 */
int32_t mla_decode_heads_per_cta(const mla_dims* dims);

/*
 * The checked build.  Compiled with -DMLA_CHECK (the package's
 * build(check=True) writes it beside the default library as
 * libmla_gb300_check.so), the kernels of mla_decode_attn and of
 * mla_decode_step's fused tail (the split kernels, the combines, the combine
 * with W_UV) test each shared-memory and global index they can compute before
 * the access: TMA rows of the cache, the query rows, the query and P tiles and
 * the zeroed rows in shared memory, the partials and chunk counts.  A failed
 * test skips the access, ORs MLA_DEV_BOUNDS into the call's dev_status (when
 * given) and into the library's bounds word.  Nothing asserts or traps.  In the
 * default build the tests compile away and the word is never written.
 *
 * mla_built_with_checks   1 in the checked build, 0 otherwise.
 * mla_debug_bounds_word   the device address (current device) of the bounds
 *                         word; the caller may zero it and read it back.
 */
int32_t mla_built_with_checks(void);
mla_status mla_debug_bounds_word(int32_t** word);

/*
 * mla_test_set_split_hooks -- test hooks of the bf16 split kernel; not for
 * production use.  The pages have no counterpart: this exists so that a test
 * can make the kernel's bounded waits run out without faulting or hanging the
 * GPU (the overflow-returns-an-error rule of "Transformer and KV Cache Basics",
 * applied to the kernel's own pipeline).
 *
 * wait_ns           limit of every bounded wait of the bf16 split kernel in ns
 *                   (0: the default of 2 s).
 * stop_after_tiles  > 0: the kernel's HBM ring issues only the first
 *                   stop_after_tiles 128-row tiles of each chunk, so a chunk
 *                   with more tiles leaves its consumers waiting; they give up
 *                   after wait_ns, set MLA_DEV_PIPELINE_TIMEOUT in dev_status,
 *                   write no partial, let the copies still in flight land, free
 *                   their tensor memory and return.  0: normal operation.
 *
 * Process-wide; read when a split is enqueued (launches captured in a graph
 * keep the values of their capture).  Reset with (0, 0) after the test.
 */
void mla_test_set_split_hooks(uint64_t wait_ns, int32_t stop_after_tiles);

/*
 * mla_test_set_split_debug -- test hook of the bf16 split kernel; not for
 * production use.  records: NULL (off) or a zeroed device array of 1 + 8 * 256
 * int32.  Every CTA whose bounded wait ran out appends one record of eight
 * words after atomically counting itself in records[0]: its block index, the
 * index of the barrier its first failed wait was on (-1: ring B's wait for the
 * score issuers), that wait's parity, the waiting thread, the CTA's work items
 * and tiles, and the tiles each score issuer had issued.  Process-wide; read
 * when a split is enqueued.
 */
void mla_test_set_split_debug(int32_t* records);

/*
 * mla_test_set_split_form -- test hook; not for production use.  0: the
 * library chooses the split's launch form (mla_decode_plan); 1: the persistent
 * grid wherever the kernel supports it (bf16, 16 heads per CTA); 2: never the
 * persistent grid.  Process-wide; read by every later planning call, so set it
 * before sizing a workspace and keep it until the calls that use it are done.
 */
void mla_test_set_split_form(int32_t form);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
