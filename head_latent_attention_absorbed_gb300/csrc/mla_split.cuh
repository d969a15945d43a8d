// Parameters shared by the split kernels (the per-chunk half of
// mla_decode_attn) and the kernels that read their partials.
#pragma once

#include "mla_common.cuh"

namespace mla {

struct SplitParams {
  const void* q_abs;
  const void* q_pe;
  const void* cache;        // used by the fp32 kernel
  const int32_t* lengths;
  float* part_o;            // [B, H, splits, 512]: one (b, h)'s chunks contiguous
  float* part_lse;          // [B, H, splits]
  int32_t* status;
  int B, H, s_max, splits, chunk;  // B counts query groups: cache sequences x q_len
  int q_len;                // query tokens per cache sequence (1: ordinary decode)
  int tpc;                  // bf16 kernel, 32 columns: query groups per CTA (2: two tokens
                            // x 16 heads; 1: 32 heads of one token)
  float scale_log2;         // softmax_scale * log2(e)
  uint8_t* q_img;           // FP8: the query's E4M3 image per (sequence, head group)
  int fill_early;           // bf16 kernel: issue tile 0's first boxes before the length
                            // is known (a one-wave grid)
  int persist;              // bf16 kernel, 16 heads per CTA: a persistent grid whose CTAs
                            // take several chunks each (chunk % 128 == 0)
  // Test hooks of the bf16 kernel (see mla_test_set_split_hooks), 0 in normal use:
  unsigned long long wait_ns;   // limit of each bounded wait (0: kWaitNs)
  int stop_after_tiles;         // ring A issues only this many tiles of a chunk (0: all)
  int32_t* debug;               // where timed-out CTAs record their first failed wait
};

// FP8 cache: the query of one (sequence, 16-head group) as the split kernel's
// shared memory holds it -- five 128-column boxes of 64 rows (4 E4M3 parts x
// 16 heads) x 128 bytes, 128-byte swizzled -- followed by the 16 per-head
// power-of-two scales (fp32).  Written once per step into the workspace.
constexpr size_t kFp8QBoxes = 5 * 64 * 128;
constexpr size_t kFp8QImage = kFp8QBoxes + 16 * sizeof(float);

// Query group v (one token of one sequence) reads cache sequence v / q_len.
__device__ __forceinline__ int cache_seq(const SplitParams& p, int v) { return v / p.q_len; }

// Rows query group v attends.  Token i of a q_len-token step sits at position
// lengths[b] - q_len + i (the cache already holds all q_len new rows), and a
// key past the query's own position is masked ("Transformer and KV Cache
// Basics", mask design for multi-token decoding), so the token sees the first
// lengths[b] - (q_len - 1 - i) rows.  A length outside [q_len, s_max] is
// reported and clamped.
__device__ __forceinline__ int clamp_length(const SplitParams& p, int v, bool report_it) {
  int full = p.lengths[v / p.q_len];
  const int back = p.q_len - 1 - v % p.q_len;
  if (full < p.q_len || full > p.s_max) {
    if (report_it) report(p.status, MLA_DEV_LENGTH_OUT_OF_RANGE);
    full = full < 0 ? 0 : (full > p.s_max ? p.s_max : full);
  }
  const int len = full - back;
  return len < 0 ? 0 : len;
}

// The FP8 (E4M3) cache's split kernel (mla_fp8.cu): same grid, partials and
// launch overlap as the bf16 one.
// It runs as two launches: the query's E4M3 image, then the split itself.
mla_status launch_split_fp8(const SplitParams& p, const void* cache, cudaStream_t stream,
                            const char* who);

// mla_absorb_q's work (named `who` in error messages), with the decode kernel's
// first cache rows prefetched into L2 when pf.cache is set, and (bf16, `early`)
// launched with programmatic stream serialization (mla_proj.cu).  `q_host`:
// whether q_nope is page-locked host memory, 1 or 0 when the caller knows it,
// -1 to ask the runtime.
mla_status absorb_q(const char* who, const mla_dims* dims, const void* q_nope, const void* q_rope,
                    const void* w_uk, const int32_t* positions, double rope_base, void* q_abs,
                    void* q_pe, void* stream, const CachePrefetch& pf, bool early,
                    int q_host = -1);

}  // namespace mla
