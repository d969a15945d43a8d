// mla_decode_attn: split-KV attention of the absorbed query over the latent
// cache, plus the log-sum-exp combine of the chunks.
//
// Multi-Head Latent Attention (Lior Sinai), 3.3 and 3.6: per head h the score
// of cached row t is (q_abs_h . c_t + q_pe_h . k_rope_t) / sqrt(d_h + d_R), one
// latent row serves every head (virtual broadcast of C^KV across heads), and
// the attention output stays in the d_c-wide latent space.
//
// bf16 kernel (one CTA per (16-head group, KV chunk, sequence)):
//   * thread 0 streams 32-row tiles of the cache (32 x 1152 B) through a ring
//     of shared-memory stages with 2-D TMA loads (nine 64-column boxes per
//     tile, 128-byte swizzle), each stage completing on its own mbarrier;
//   * scores S[16 heads x 32 rows] on the tensor cores (mma.sync m16n8k16):
//     warp w contracts its 144-wide quarter of the 576 columns with the query
//     held in registers; the four partial score tiles meet in shared memory;
//   * every warp forms the full scores, runs the online softmax (exp2 domain)
//     and keeps P in registers as the A operand of the PV product;
//   * the fp32 query and P enter the bf16 mma as hi + lo parts (two mma per
//     product), which keeps their rounding near 2^-17 relative;
//   * warp w accumulates O[16 heads x 128 latent columns] += P . C in fp32
//     registers, reading the same swizzled stage through ldmatrix.trans;
//   * one CTA barrier per tile; the stage freed by the previous tile is
//     refilled right after it.
// fp32 kernel: plain SIMT, fp32 arithmetic throughout (no TF32).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "mla_common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kSubBytes = kTileRows * 128;        // one 32-row x 64-col bf16 box
constexpr int kStageBytes = 9 * kSubBytes;        // 32 rows x 576 cols
constexpr int kSStride = 40;                      // floats per head row of a partial-score tile
constexpr int kSTileFloats = kHeadGroup * kSStride;
constexpr int kNumStagesBf16 = 4;

struct SplitParams {
  const void* q_abs;
  const void* q_pe;
  const void* cache;        // used by the fp32 kernel
  const int32_t* lengths;
  float* part_o;            // [B, splits, H, 512]
  float* part_lse;          // [B, splits, H]
  int32_t* status;
  int B, H, s_max, splits, chunk;
  float scale_log2;         // softmax_scale * log2(e)
};

__device__ __forceinline__ int clamp_length(const SplitParams& p, int b, bool report_it) {
  int len = p.lengths[b];
  if (len < 1 || len > p.s_max) {
    if (report_it) report(p.status, MLA_DEV_LENGTH_OUT_OF_RANGE);
    len = len < 0 ? 0 : (len > p.s_max ? p.s_max : len);
  }
  return len;
}

constexpr size_t bf16_smem_bytes(int nstage) {
  return 1024 /*alignment slack*/ + size_t(nstage) * kStageBytes +
         2 * kWarps * kSTileFloats * sizeof(float) + 8 * nstage;
}

template <int NSTAGE>
__global__ void __launch_bounds__(kThreads, 1)
    split_bf16_kernel(const __grid_constant__ CUtensorMap tmap, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* sbuf = reinterpret_cast<float*>(smem + NSTAGE * kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(sbuf + 2 * kWarps * kSTileFloats);

  const int g = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = clamp_length(p, b, tid == 0 && g == 0 && j == 0);
  const int r0 = j * p.chunk;
  if (r0 >= len) return;  // chunk past the end of this sequence: nothing to do
  const int r1 = min(r0 + p.chunk, len);
  const int ntiles = (r1 - r0 + kTileRows - 1) / kTileRows;
  const int row_base = b * p.s_max + r0;

  const uint32_t full0 = smem_u32(full);
  const uint32_t stage0 = smem_u32(stages);
  uint64_t policy = 0;
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(full0 + 8 * s, 1);
    fence_mbarrier_init();
  }
  __syncthreads();

  auto issue = [&](int tile, int stage) {
    const uint32_t bar = full0 + 8 * stage;
    const uint32_t dst = stage0 + stage * kStageBytes;
    mbar_arrive_expect_tx(bar, kStageBytes);
#pragma unroll
    for (int k = 0; k < 9; ++k)
      tma_load_2d(dst + k * kSubBytes, &tmap, 64 * k, row_base + tile * kTileRows, bar, policy);
  };
  if (tid == 0) {
    prefetch_tmap(&tmap);
    policy = l2_evict_first_policy();
    for (int s = 0; s < NSTAGE && s < ntiles; ++s) issue(s, s);
  }

  // Query fragments for this warp's quarter of the 576 columns (9 k-steps of
  // 16).  The fp32 query enters the tensor cores as hi + lo bf16 parts, so its
  // rounding stays near 2^-17 relative (bf16 alone is not enough when a few
  // large rows dominate the softmax).
  const int gq = lane >> 2, cq = lane & 3;
  const int h0 = g * kHeadGroup;
  const float* qa_base = static_cast<const float*>(p.q_abs);
  const float* qp_base = static_cast<const float*>(p.q_pe);
  uint32_t qh[9][4], ql[9][4];
#pragma unroll
  for (int ks = 0; ks < 9; ++ks) {
    const int k0 = 144 * warp + 16 * ks;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int h = h0 + gq + ((e & 1) ? 8 : 0);
      const int k = k0 + 2 * cq + ((e & 2) ? 8 : 0);
      const float* src = (k < kDc) ? qa_base + (size_t(b) * p.H + h) * kDc + k
                                   : qp_base + (size_t(b) * p.H + h) * kDr + (k - kDc);
      const float2 v = *reinterpret_cast<const float2*>(src);
      split_bf16(v.x, v.y, qh[ks][e], ql[ks][e]);
    }
  }

  float o[16][4];
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int i = 0; i < ntiles; ++i) {
    const int s = i % NSTAGE;
    const uint32_t parity = (i / NSTAGE) & 1;
    const bool ok = mbar_wait_bounded(full0 + 8 * s, parity);
    const uint32_t st = stage0 + s * kStageBytes;

    // Partial scores over this warp's 144 columns, all 32 rows (4 n-blocks of 8).
    float acc[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 9; ++ks) {
      const int k0 = 144 * warp + 16 * ks;
      const int sub = k0 >> 6, kin = k0 & 63;
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int row = np * 16 + ((lane >> 4) << 3) + (lane & 7);
        const int ch = (kin >> 3) + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(st + sub * kSubBytes + sw128(row, ch), b0, b1, b2, b3);
        mma_bf16(acc[2 * np], qh[ks], b0, b1);
        mma_bf16(acc[2 * np], ql[ks], b0, b1);
        mma_bf16(acc[2 * np + 1], qh[ks], b2, b3);
        mma_bf16(acc[2 * np + 1], ql[ks], b2, b3);
      }
    }
    float* sb = sbuf + ((i & 1) * kWarps + warp) * kSTileFloats;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      *reinterpret_cast<float2*>(sb + gq * kSStride + nb * 8 + 2 * cq) =
          make_float2(acc[nb][0], acc[nb][1]);
      *reinterpret_cast<float2*>(sb + (gq + 8) * kSStride + nb * 8 + 2 * cq) =
          make_float2(acc[nb][2], acc[nb][3]);
    }

    const int valid = min(kTileRows, r1 - (r0 + i * kTileRows));
    if (__syncthreads_or(!ok)) {
      // A copy did not land in time: report, give in-flight copies a bounded
      // chance to finish, and leave without touching the outputs.
      if (tid == 0) {
        report(p.status, MLA_DEV_PIPELINE_TIMEOUT);
        for (int t = i; t < ntiles && t < i + NSTAGE; ++t)
          mbar_wait_bounded(full0 + 8 * (t % NSTAGE), (t / NSTAGE) & 1);
      }
      return;
    }
    // The previous tile's stage is free (every warp is past its PV product).
    if (tid == 0 && i >= 1 && i - 1 + NSTAGE < ntiles) {
      fence_proxy_async_smem();
      issue(i - 1 + NSTAGE, (i - 1) % NSTAGE);
    }
    if (valid < kTileRows) {
      // Rows past the sequence end may hold anything (NaN included): zero them
      // so that P = 0 times the row contributes exactly 0 to the PV product.
      const int nchunks = (kTileRows - valid) * 9 * 8;
      for (int c = tid; c < nchunks; c += kThreads) {
        const int sub = c / ((kTileRows - valid) * 8);
        const int rem = c % ((kTileRows - valid) * 8);
        const int row = valid + rem / 8, ch = rem % 8;
        *reinterpret_cast<uint4*>(stages + s * kStageBytes + sub * kSubBytes + row * 128 +
                                  ch * 16) = make_uint4(0, 0, 0, 0);
      }
      __syncthreads();
    }

    // Full scores for this thread's elements (heads gq, gq+8; rows nb*8+2cq+{0,1}).
    const float* sb0 = sbuf + (i & 1) * kWarps * kSTileFloats;
    float sc[4][4];
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float2 v = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float2 t = *reinterpret_cast<const float2*>(
              sb0 + w * kSTileFloats + (gq + 8 * hh) * kSStride + nb * 8 + 2 * cq);
          v.x += t.x;
          v.y += t.y;
        }
        const int row = nb * 8 + 2 * cq;
        sc[nb][2 * hh] = row < valid ? v.x * p.scale_log2 : -INFINITY;
        sc[nb][2 * hh + 1] = row + 1 < valid ? v.y * p.scale_log2 : -INFINITY;
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      mx0 = fmaxf(mx0, fmaxf(sc[nb][0], sc[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nb][2], sc[nb][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float a0 = ex2(m0 - mu0), a1 = ex2(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
      sc[nb][0] = ex2(sc[nb][0] - mu0);
      sc[nb][1] = ex2(sc[nb][1] - mu0);
      sc[nb][2] = ex2(sc[nb][2] - mu1);
      sc[nb][3] = ex2(sc[nb][3] - mu1);
      ps0 += sc[nb][0] + sc[nb][1];
      ps1 += sc[nb][2] + sc[nb][3];
    }
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
    // P as hi + lo bf16 parts (A operand of the PV product).
    uint32_t ph[2][4], pl[2][4];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      split_bf16(sc[2 * kk][0], sc[2 * kk][1], ph[kk][0], pl[kk][0]);
      split_bf16(sc[2 * kk][2], sc[2 * kk][3], ph[kk][1], pl[kk][1]);
      split_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[kk][2], pl[kk][2]);
      split_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[kk][3], pl[kk][3]);
    }
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
      o[nb][0] *= a0;
      o[nb][1] *= a0;
      o[nb][2] *= a1;
      o[nb][3] *= a1;
    }
    // O[16 x 128 (this warp's columns)] += P[16 x 32] . C[32 x 128]
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const int col0 = 128 * warp + 16 * np;
        const int sub = col0 >> 6, cin = col0 & 63;
        const int mi = lane >> 3;
        const int t = kk * 16 + ((mi & 1) << 3) + (lane & 7);
        const int ch = (cin >> 3) + (mi >> 1);
        uint32_t r0_, r1_, r2_, r3_;
        ldsm_x4_t(st + sub * kSubBytes + sw128(t, ch), r0_, r1_, r2_, r3_);
        mma_bf16(o[2 * np], ph[kk], r0_, r1_);
        mma_bf16(o[2 * np], pl[kk], r0_, r1_);
        mma_bf16(o[2 * np + 1], ph[kk], r2_, r3_);
        mma_bf16(o[2 * np + 1], pl[kk], r2_, r3_);
      }
    }
  }

  // Epilogue: normalise by the softmax denominator and write the chunk's partials.
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const size_t base = (size_t(b) * p.splits + j) * p.H + h0;
  float* po = p.part_o + base * kDc;
#pragma unroll
  for (int nb = 0; nb < 16; ++nb) {
    const int col = 128 * warp + nb * 8 + 2 * cq;
    *reinterpret_cast<float2*>(po + size_t(gq) * kDc + col) =
        make_float2(o[nb][0] * inv0, o[nb][1] * inv0);
    *reinterpret_cast<float2*>(po + size_t(gq + 8) * kDc + col) =
        make_float2(o[nb][2] * inv1, o[nb][3] * inv1);
  }
  if (warp == 0 && cq == 0) {
    p.part_lse[base + gq] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
    p.part_lse[base + gq + 8] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
  }
}

// fp32 path: one CTA per (head, chunk, sequence); each warp runs its own online
// softmax over every fourth row, then the four warp states are merged.
__global__ void __launch_bounds__(kThreads)
    split_f32_kernel(const SplitParams p) {
  const int h = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = clamp_length(p, b, tid == 0 && h == 0 && j == 0);
  const int r0 = j * p.chunk;
  if (r0 >= len) return;
  const int r1 = min(r0 + p.chunk, len);

  const float* qa = static_cast<const float*>(p.q_abs) + (size_t(b) * p.H + h) * kDc;
  const float* qp = static_cast<const float*>(p.q_pe) + (size_t(b) * p.H + h) * kDr;
  float q[18];
#pragma unroll
  for (int i = 0; i < 18; ++i) {
    const int k = lane + 32 * i;
    q[i] = k < kDc ? qa[k] : qp[k - kDc];
  }
  const float* cache = static_cast<const float*>(p.cache);
  const float scale = p.scale_log2;
  float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int t = r0 + warp; t < r1; t += kWarps) {
    const float* row = cache + (size_t(b) * p.s_max + t) * kRow;
    float c[18];
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 18; ++i) {
      c[i] = row[lane + 32 * i];
      dot = fmaf(q[i], c[i], dot);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float s = dot * scale;
    const float mn = fmaxf(m, s);
    const float alpha = exp2f(m - mn);
    const float pr = exp2f(s - mn);
    l = l * alpha + pr;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = fmaf(pr, c[i], acc[i] * alpha);
    m = mn;
  }
  __shared__ float wm[kWarps], wl[kWarps], wo[kWarps][kDc];
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = l;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) wo[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w]);
  float L = 0.f, f[kWarps];
  for (int w = 0; w < kWarps; ++w) {
    f[w] = wm[w] == -INFINITY ? 0.f : exp2f(wm[w] - M);
    L += f[w] * wl[w];
  }
  const size_t base = (size_t(b) * p.splits + j) * p.H + h;
  for (int c = tid; c < kDc; c += kThreads) {
    float v = 0.f;
    for (int w = 0; w < kWarps; ++w) v += f[w] * wo[w][c];
    p.part_o[base * kDc + c] = v / L;
  }
  if (tid == 0) p.part_lse[base] = (M + log2f(L)) * kLn2;
}

// Merge of the chunk partials of one (sequence, head):
//   L = log sum_j exp(lse_j),  o_c = sum_j exp(lse_j - L) o_j.
__global__ void __launch_bounds__(128)
    combine_kernel(const SplitParams p, float* o_c, float* lse_out) {
  extern __shared__ float wts[];  // [splits]
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int len = clamp_length(p, b, false);
  const int nsplit = (len + p.chunk - 1) / p.chunk;
  float* out = o_c + (size_t(b) * p.H + h) * kDc;
  if (nsplit == 0) {
    reinterpret_cast<float4*>(out)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0 && lse_out) lse_out[size_t(b) * p.H + h] = -INFINITY;
    return;
  }
  const size_t stride = size_t(p.H);  // between consecutive splits of one (b, h)
  const float* lse_bh = p.part_lse + size_t(b) * p.splits * p.H + h;
  __shared__ float red[4];
  float mx = -INFINITY;
  for (int s = tid; s < nsplit; s += 128) mx = fmaxf(mx, lse_bh[s * stride]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float sum = 0.f;
  for (int s = tid; s < nsplit; s += 128) {
    const float w = expf(lse_bh[s * stride] - mx);
    wts[s] = w;
    sum += w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if ((tid & 31) == 0) red[tid >> 5] = sum;
  __syncthreads();
  sum = red[0] + red[1] + red[2] + red[3];
  const float inv = 1.f / sum;
  const float* po = p.part_o + (size_t(b) * p.splits * p.H + h) * kDc;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; ++s) {
    const float w = wts[s] * inv;
    const float4 v = reinterpret_cast<const float4*>(po + size_t(s) * stride * kDc)[tid];
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  reinterpret_cast<float4*>(out)[tid] = acc;
  if (tid == 0 && lse_out) lse_out[size_t(b) * p.H + h] = mx + logf(sum);
}

// ------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Rows per KV chunk (a multiple of the 32-row tile) and the resulting chunk
// count.  With `requested` = 0 the count minimises a makespan estimate: waves
// of CTAs over the SMs times (rows per chunk + a fixed per-CTA cost), plus the
// combine's cost per chunk.  The bf16 kernel runs one CTA per SM.
int chunk_rows(const mla_dims* d, int requested, int* splits_out) {
  const int S = d->s_max;
  const int max_splits = (S + kTileRows - 1) / kTileRows;
  int splits = requested;
  if (splits <= 0) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool bf16 = d->dtype == MLA_BF16;
    const long long per_split = static_cast<long long>(d->batch) * (bf16 ? d->heads / kHeadGroup : d->heads);
    const long long slots = bf16 ? sms : 4ll * sms;
    double best = 1e300;
    splits = 1;
    for (int s = 1; s <= max_splits; ++s) {
      const int chunk = ((S + s - 1) / s + kTileRows - 1) / kTileRows * kTileRows;
      const int s_eff = (S + chunk - 1) / chunk;
      if (s_eff != s) continue;
      const long long waves = (per_split * s_eff + slots - 1) / slots;
      const double cost = double(waves) * (chunk + 96) + 4.0 * s_eff;
      if (cost < best) {
        best = cost;
        splits = s;
      }
    }
  }
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  int chunk = (S + splits - 1) / splits;
  chunk = (chunk + kTileRows - 1) / kTileRows * kTileRows;
  *splits_out = (S + chunk - 1) / chunk;
  return chunk;
}

size_t workspace_bytes(const mla_dims* d, int splits) {
  const size_t n = size_t(d->batch) * splits * d->heads;
  const size_t o_bytes = (n * kDc * sizeof(float) + 255) / 256 * 256;
  return o_bytes + (n * sizeof(float) + 255) / 256 * 256;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int32_t mla_decode_num_splits(const mla_dims* dims, int32_t requested) {
  if (check_dims(dims, "mla_decode_num_splits") != MLA_OK) return 0;
  int splits = 0;
  chunk_rows(dims, requested, &splits);
  return splits;
}

extern "C" size_t mla_decode_workspace_bytes(const mla_dims* dims, int32_t requested) {
  if (check_dims(dims, "mla_decode_workspace_bytes") != MLA_OK) return 0;
  int splits = 0;
  chunk_rows(dims, requested, &splits);
  return workspace_bytes(dims, splits);
}

// Validates the arguments shared by the split and combine halves and fills the
// kernel parameters.  Returns MLA_OK or the status to hand back.
static mla_status prepare(const char* who, const mla_dims* dims, const void* q_abs,
                          const void* q_pe, const void* cache, const int32_t* lengths,
                          float softmax_scale, int32_t num_splits, void* workspace,
                          size_t ws_bytes, int32_t* dev_status, SplitParams* p) {
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!lengths || !workspace) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned16(q_abs) || !aligned16(q_pe) || !aligned16(cache) || !aligned16(workspace)) {
    set_error("%s: q_abs, q_pe, cache, workspace and o_c must be 16-byte aligned", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) {
    set_error("%s: softmax_scale must be finite and > 0", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (num_splits < 0) {
    set_error("%s: num_splits must be >= 0", who);
    return MLA_ERR_INVALID_ARG;
  }
  int splits = 0;
  const int chunk = chunk_rows(dims, num_splits, &splits);
  const size_t need = workspace_bytes(dims, splits);
  if (ws_bytes < need) {
    set_error("%s: workspace %zu bytes < %zu needed", who, ws_bytes, need);
    return MLA_ERR_WORKSPACE;
  }
  p->q_abs = q_abs;
  p->q_pe = q_pe;
  p->cache = cache;
  p->lengths = lengths;
  p->part_o = static_cast<float*>(workspace);
  const size_t n = size_t(dims->batch) * splits * dims->heads;
  p->part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         (n * kDc * sizeof(float) + 255) / 256 * 256);
  p->status = dev_status;
  p->B = dims->batch;
  p->H = dims->heads;
  p->s_max = dims->s_max;
  p->splits = splits;
  p->chunk = chunk;
  p->scale_log2 = softmax_scale * kLog2e;
  return MLA_OK;
}

extern "C" mla_status mla_decode_split(const mla_dims* dims, const void* q_abs, const void* q_pe,
                                       const void* cache, const int32_t* lengths,
                                       float softmax_scale, int32_t num_splits, void* workspace,
                                       size_t ws_bytes, int32_t* dev_status, void* stream) {
  const char* who = "mla_decode_split";
  if (!q_abs || !q_pe || !cache) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  SplitParams p;
  mla_status st = prepare(who, dims, q_abs, q_pe, cache, lengths, softmax_scale, num_splits,
                          workspace, ws_bytes, dev_status, &p);
  if (st != MLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dims->dtype == MLA_BF16) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) {
      set_error("%s: cuTensorMapEncodeTiled is not available from the driver", who);
      return MLA_ERR_CUDA;
    }
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {cuuint64_t(kRow), cuuint64_t(dims->batch) * dims->s_max};
    const cuuint64_t gstride[1] = {cuuint64_t(kRow) * 2};
    const cuuint32_t box[2] = {64, cuuint32_t(kTileRows)};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), gdim,
                     gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      set_error("%s: cuTensorMapEncodeTiled failed (%d)", who, int(r));
      return MLA_ERR_CUDA;
    }
    constexpr size_t smem = bf16_smem_bytes(kNumStagesBf16);
    static bool attr_set = false;
    if (!attr_set) {
      if (cudaFuncSetAttribute(split_bf16_kernel<kNumStagesBf16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(smem)) != cudaSuccess) {
        set_error("%s: cannot reserve %zu bytes of shared memory", who, smem);
        return MLA_ERR_CUDA;
      }
      attr_set = true;
    }
    dim3 grid(dims->heads / kHeadGroup, p.splits, dims->batch);
    split_bf16_kernel<kNumStagesBf16><<<grid, kThreads, smem, s>>>(tmap, p);
  } else {
    dim3 grid(dims->heads, p.splits, dims->batch);
    split_f32_kernel<<<grid, kThreads, 0, s>>>(p);
  }
  return launch_status(who);
}

extern "C" mla_status mla_decode_combine(const mla_dims* dims, const int32_t* lengths,
                                         int32_t num_splits, const void* workspace,
                                         size_t ws_bytes, float* o_c, float* lse, void* stream) {
  const char* who = "mla_decode_combine";
  if (!o_c || !aligned16(o_c)) {
    set_error("%s: o_c must be a non-NULL 16-byte aligned pointer", who);
    return MLA_ERR_INVALID_ARG;
  }
  SplitParams p;
  mla_status st = prepare(who, dims, nullptr, nullptr, nullptr, lengths, 1.f, num_splits,
                          const_cast<void*>(workspace), ws_bytes, nullptr, &p);
  if (st != MLA_OK) return st;
  combine_kernel<<<dim3(dims->heads, dims->batch), 128, p.splits * sizeof(float),
                   static_cast<cudaStream_t>(stream)>>>(p, o_c, lse);
  return launch_status(who);
}

extern "C" mla_status mla_decode_attn(const mla_dims* dims, const void* q_abs, const void* q_pe,
                                      const void* cache, const int32_t* lengths,
                                      float softmax_scale, int32_t num_splits, void* workspace,
                                      size_t ws_bytes, float* o_c, float* lse,
                                      int32_t* dev_status, void* stream) {
  if (!o_c || !aligned16(o_c)) {
    set_error("mla_decode_attn: o_c must be a non-NULL 16-byte aligned pointer");
    return MLA_ERR_INVALID_ARG;
  }
  mla_status st = mla_decode_split(dims, q_abs, q_pe, cache, lengths, softmax_scale, num_splits,
                                   workspace, ws_bytes, dev_status, stream);
  if (st != MLA_OK) {
    // keep the caller-facing name in the detail message
    return st;
  }
  return mla_decode_combine(dims, lengths, num_splits, workspace, ws_bytes, o_c, lse, stream);
}
