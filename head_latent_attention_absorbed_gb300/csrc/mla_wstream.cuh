// Weight-streaming projection on the tensor cores: y[b, n] = sum_k x[b, k] w[n, k]
// for a bf16 weight stored [N, K] (K contiguous) and a small batch of rows x
// (bf16, or fp32 entering as bf16 hi + lo parts).  It is the shape of both
// steps around the attention: the cache append's fused down-projection
// kv_a_proj ("Deepseek V2 Lite Inference Engine in C", MLA notes) and the
// output projection W^O ("Multi-Head Latent Attention", eq. 3.3.3).
#pragma once

#include "mla_common.cuh"

namespace mla {

enum WStreamMode { kWsWriteY = 0, kWsAppendRow = 1 };

struct WStreamJob {
  int mode;                    // kWsWriteY or kWsAppendRow
  bool x_f32;                  // x is fp32 (else bf16)
  const void* x;               // [B, K], 16-byte aligned
  const void* w;               // [N, K] bf16, 16-byte aligned
  int B, K, N;                 // K a multiple of 64
  float* y;                    // kWsWriteY: [B, N] fp32
  void* cache;                 // kWsAppendRow: [B, s_max, N] bf16, or E4M3 with cache_fp8
  bool cache_fp8;              // kWsAppendRow: the cache holds FP8 E4M3 elements
  const int32_t* positions;    // kWsAppendRow: [B], the row written
  int s_max, d_c;              // kWsAppendRow: columns >= d_c are rotated
  double turns[kDr / 2];       // kWsAppendRow: RoPE frequencies / (2 pi)
  int32_t* status;             // device error word (may be NULL)
};

// Enqueues the projection on `stream`; the error message names `who`.
mla_status wstream_launch(const WStreamJob& job, cudaStream_t stream, const char* who);

}  // namespace mla
