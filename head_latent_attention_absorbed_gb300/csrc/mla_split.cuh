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
  int B, H, s_max, splits, chunk;
  float scale_log2;         // softmax_scale * log2(e)
  uint8_t* q_img;           // FP8: the query's E4M3 image per (sequence, head group)
};

// FP8 cache: the query of one (sequence, 16-head group) as the split kernel's
// shared memory holds it -- five 128-column boxes of 64 rows (4 E4M3 parts x
// 16 heads) x 128 bytes, 128-byte swizzled -- followed by the 16 per-head
// power-of-two scales (fp32).  Written once per step into the workspace.
constexpr size_t kFp8QBoxes = 5 * 64 * 128;
constexpr size_t kFp8QImage = kFp8QBoxes + 16 * sizeof(float);

__device__ __forceinline__ int clamp_length(const SplitParams& p, int b, bool report_it) {
  int len = p.lengths[b];
  if (len < 1 || len > p.s_max) {
    if (report_it) report(p.status, MLA_DEV_LENGTH_OUT_OF_RANGE);
    len = len < 0 ? 0 : (len > p.s_max ? p.s_max : len);
  }
  return len;
}

// The FP8 (E4M3) cache's split kernel (mla_fp8.cu): same grid, partials and
// launch overlap as the bf16 one.
// It runs as two launches: the query's E4M3 image, then the split itself.
mla_status launch_split_fp8(const SplitParams& p, const void* cache, cudaStream_t stream,
                            const char* who);

}  // namespace mla
