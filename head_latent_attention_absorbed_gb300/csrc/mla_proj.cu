// mla_absorb_q and mla_out_proj: the two small per-head projections around the
// attention.
//
//   absorb:  q_abs[b,h,:] = q_nope[b,h,:] . W_UK[h]     (128 -> 512)
//            q_pe[b,h,:]  = RoPE(q_rope[b,h,:], positions[b])
//   out:     o[b,h,:]     = W_UV[h] . o_c[b,h,:]         (512 -> 128)
//
// Multi-Head Latent Attention (Lior Sinai) 3.3 (W^UK is absorbed into the query
// side, W^UV applied after the latent attention, eq. 3.3.3) and 3.7 (RoPE as a
// complex rotation of adjacent pairs).  Both products are small batched GEMMs
// whose time goes into reading the bf16 weights once; with at most a few
// hundred FLOPs per weight byte they are latency-bound, so the kernels spread
// the weights over many small CTAs, issue every global load of a CTA before
// its first use, and run the batch as the M side of mma.sync m16n8k16 with
// fp32 accumulation.
#include <math.h>

#include <algorithm>

#include "mla_common.cuh"
#include "mla_split.cuh"
#include "mla_wstream.cuh"

namespace mla {
namespace {

// ---------------------------------------------------------------------- RoPE
// theta_i = base^(-2i/d_rope) comes from the host in fp64 as turns,
// theta_i / (2 pi).  The angle pos * theta_i is reduced modulo 2 pi in fp64
// (rope_angle), so that positions up to 2^31 keep their fractional turns; the
// reduced angle (|r| <= pi) then goes through single-precision sincosf.
struct RopeTheta {
  double turns[kDr / 2];
};

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ void rope_pair(const T* q_rope, const int32_t* positions,
                                          const RopeTheta& th, float* q_pe, int H, int h, int it) {
  const int b = it / (kDr / 2), i = it % (kDr / 2);
  float sn, cs;
  sincosf(rope_angle(positions[b], th.turns[i]), &sn, &cs);
  const size_t off = (size_t(b) * H + h) * kDr + 2 * i;
  const float x0 = to_f(q_rope[off]), x1 = to_f(q_rope[off + 1]);
  q_pe[off] = cs * x0 - sn * x1;
  q_pe[off + 1] = sn * x0 + cs * x1;
}

// ---------------------------------------------------------------------- absorb, bf16
// grid (H, d_c/16), one warp per CTA: CTA (h, cb) owns output columns
// [16cb, 16cb+16) of head h for the whole batch.  The 128 x 16 slice of W_UK
// lands in shared memory through cp.async (all copies in flight at once); the
// batch rows are the M side of mma.sync m16n8k16.  The CTAs of head h also
// rotate that head's RoPE pairs, one pair per thread.
// Within mla_decode_step it may be launched with programmatic stream
// serialization: the W_UK copies (and the cache prefetch) are issued before the
// wait for the previous kernel of the stream, so that they overlap its end;
// everything else (q_nope, q_rope, positions, every write) comes after.  Launched
// as usual, the wait returns at once.
constexpr int kPfPiece = 16384;   // bytes per L2 prefetch instruction
// Bytes between two staged query rows (128 bf16 = 256 B of data): the pad of
// 16 B puts the eight rows of an ldmatrix in eight different bank quads.
constexpr int kQsRow = 2 * kDn + 16;

// Four 8x8 bf16 matrices from shared memory (lanes 8i..8i+7 address the rows
// of matrix i), one register each, untransposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Within mla_decode_step: start the decode kernel's cache stream.  The pieces
// of every chunk's first rows are spread over the grid's threads (thread `me`
// of `nthreads`), the first piece of every chunk first.  Callers number their
// threads CTA-fastest (thread t of CTA c is me = t * CTAs + c), so that
// consecutive pieces go to different CTAs, hence SMs: each piece is one bulk
// prefetch that the SM's copy unit turns into L2 requests, and a few SMs
// holding all of them issue them one after another (measured on 8 sequences x
// 4096 rows: its 1152 pieces on the first three CTAs of a 16-CTA grid made
// the step 27 us slower).  The cache and lengths are inputs, not results of
// the previous kernel, so this precedes the wait.
__device__ __forceinline__ void issue_cache_prefetch(const CachePrefetch& pf, int me, int nthreads) {
  if (!pf.cache) return;
  const int nchunk = pf.B * pf.splits;
  const int per_chunk = (pf.rows * pf.row_bytes + kPfPiece - 1) / kPfPiece;
  for (int id = me; id < nchunk * per_chunk; id += nthreads) {
    const int k = id / nchunk, c = id % nchunk;
    const int b = c / pf.splits, r0 = (c % pf.splits) * pf.chunk;
    const int len = min(max(pf.lengths[b], 0), pf.s_max);
    const int rows = min(min(pf.chunk, len - r0), pf.rows);
    if (rows <= 0) continue;
    const long long first = (static_cast<long long>(b) * pf.s_max + r0) * pf.row_bytes;
    const long long beg = first + static_cast<long long>(k) * kPfPiece;
    const long long end = first + static_cast<long long>(rows) * pf.row_bytes;
    if (beg >= end) continue;
    const uint32_t size = static_cast<uint32_t>(min(static_cast<long long>(kPfPiece), end - beg));
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(pf.cache + beg), "r"(size)
                 : "memory");
  }
}

// Queries in device memory: each lane loads its A fragments directly (32
// four-byte loads; the 32 CTAs of a head read its query rows from L2).
__global__ void __launch_bounds__(32)
    absorb_bf16_kernel(const __nv_bfloat16* __restrict__ q_nope,
                       const __nv_bfloat16* __restrict__ q_rope,
                       const __nv_bfloat16* __restrict__ w_uk, const int32_t* __restrict__ pos,
                       const RopeTheta th, float* __restrict__ q_abs, float* __restrict__ q_pe,
                       int B, int H, const CachePrefetch pf) {
  __shared__ __align__(128) uint8_t wt[kDn * 32];  // 128 k-rows x 16 bf16 columns
  const int h = blockIdx.x, cb = blockIdx.y, lane = threadIdx.x;
  pdl_launch_dependents();   // the decode kernel may start its set-up and cache stream now
  const int c0 = cb * 16;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int idx = lane + 32 * r;          // 256 chunks of 16 B
    const int k = idx >> 1, ch = idx & 1;
    const uint32_t dst = smem_u32(wt + k * 32 + ((ch ^ ((k >> 2) & 1)) << 4));
    const void* src = w_uk + (size_t(h) * kDn + k) * kDc + c0 + ch * 8;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  issue_cache_prefetch(pf, lane * (gridDim.x * gridDim.y) + blockIdx.y * gridDim.x + blockIdx.x,
                       gridDim.x * gridDim.y * 32);
  pdl_wait();
  for (int it = cb * 32 + lane; it < B * (kDr / 2); it += 32 * gridDim.y)
    rope_pair(q_rope, pos, th, q_pe, H, h, it);

  const int gq = lane >> 2, cq = lane & 3;
  const uint32_t wbase = smem_u32(wt);
  for (int mt = 0; mt * 16 < B; ++mt) {
    const int bA = mt * 16 + gq, bB = bA + 8;
    uint32_t a[8][4];
    const __nv_bfloat16* rA = q_nope + (size_t(bA) * H + h) * kDn + 2 * cq;
    const __nv_bfloat16* rB = q_nope + (size_t(bB) * H + h) * kDn + 2 * cq;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      a[ks][0] = bA < B ? *reinterpret_cast<const uint32_t*>(rA + 16 * ks) : 0u;
      a[ks][1] = bB < B ? *reinterpret_cast<const uint32_t*>(rB + 16 * ks) : 0u;
      a[ks][2] = bA < B ? *reinterpret_cast<const uint32_t*>(rA + 16 * ks + 8) : 0u;
      a[ks][3] = bB < B ? *reinterpret_cast<const uint32_t*>(rB + 16 * ks + 8) : 0u;
    }
    if (mt == 0) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      // B fragments of n-blocks 0 and 1 for k in [16ks, 16ks+16): ldmatrix.trans
      // of the [k][n] slice (32-byte rows, 16-byte chunks swizzled by bit 2 of k).
      const int mi = lane >> 3;
      const int k = 16 * ks + ((mi & 1) << 3) + (lane & 7);
      const int ch = mi >> 1;
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(wbase + k * 32 + ((ch ^ ((k >> 2) & 1)) << 4), b0, b1, b2, b3);
      mma_bf16(acc[0], a[ks], b0, b1);
      mma_bf16(acc[1], a[ks], b2, b3);
    }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const int c = c0 + 8 * nb + 2 * cq;
      if (bA < B)
        *reinterpret_cast<float2*>(q_abs + (size_t(bA) * H + h) * kDc + c) =
            make_float2(acc[nb][0], acc[nb][1]);
      if (bB < B)
        *reinterpret_cast<float2*>(q_abs + (size_t(bB) * H + h) * kDc + c) =
            make_float2(acc[nb][2], acc[nb][3]);
    }
  }
}

// Queries in page-locked host memory, read over the host link: a head's
// query rows are read by 16 / kWarps CTAs instead of 32 (the form above reads
// them once per 16-column block).  grid (H, 16 / kWarps), 32 kWarps threads:
// CTA (h, y) owns columns [32 kWarps y, 32 kWarps (y + 1)), warp w of them
// the 32 columns at 32 w.  Before the wait, its W_UK[h] slice (128 rows x
// 32 kWarps bf16) lands in shared memory as 16-column blocks in the layout
// above.  After it, the first half of the warps copies up to 64 query rows at
// a time into shared memory with whole-line 16-byte loads while the second
// half rotates the head's RoPE pairs (shared over the head's CTAs; 32 lanes
// over the 32 pairs of one row: one 128-byte line of q_rope); then each warp
// computes its columns from those rows with ldmatrix fragments.
constexpr int kHeadStageRows = 64;
template <int kWarps>
struct HeadPlan {
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kCols = 32 * kWarps;                    // columns per CTA
  static constexpr int kCtasPerHead = kDc / kCols;
  static constexpr size_t kWBytes = size_t(kCols / 16) * kDn * 32;
  static constexpr size_t kSmem = kWBytes + size_t(kHeadStageRows) * kQsRow;
  static_assert(kWarps >= 2 && kDc % kCols == 0, "whole column slices, two warp halves");
};

template <int kWarps>
__global__ void __launch_bounds__(32 * kWarps)
    absorb_bf16_head_kernel(const __nv_bfloat16* __restrict__ q_nope,
                            const __nv_bfloat16* __restrict__ q_rope,
                            const __nv_bfloat16* __restrict__ w_uk,
                            const int32_t* __restrict__ pos, const RopeTheta th,
                            float* __restrict__ q_abs, float* __restrict__ q_pe, int B, int H,
                            const CachePrefetch pf) {
  using P = HeadPlan<kWarps>;
  constexpr int kHalf = P::kThreads / 2;
  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t* wt = dsm;                  // block i (columns c0 + 16i ..) at i * kDn * 32
  uint8_t* qs = dsm + P::kWBytes;     // staged query rows, kQsRow bytes apart
  const int h = blockIdx.x, y = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = y * P::kCols;
  pdl_launch_dependents();   // the decode kernel may start its set-up and cache stream now
  // The slice as 16-byte pieces: piece j is piece j % (kCols / 8) of k-row
  // j / (kCols / 8), so consecutive threads read consecutive pieces of a row.
  constexpr int kPieces = P::kCols / 8;
  for (int j = tid; j < kDn * kPieces; j += P::kThreads) {
    const int k = j / kPieces, piece = j % kPieces, blk = piece >> 1, ch = piece & 1;
    const uint32_t dst =
        smem_u32(wt + blk * (kDn * 32) + k * 32 + ((ch ^ ((k >> 2) & 1)) << 4));
    const void* src = w_uk + (size_t(h) * kDn + k) * kDc + c0 + piece * 8;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  issue_cache_prefetch(pf, tid * (gridDim.x * gridDim.y) + blockIdx.y * gridDim.x + blockIdx.x,
                       gridDim.x * gridDim.y * P::kThreads);
  pdl_wait();

  const int gq = lane >> 2, cq = lane & 3;
  const uint32_t qbase = smem_u32(qs);
  for (int g0 = 0; g0 < B; g0 += kHeadStageRows) {
    const int tiles = (min(kHeadStageRows, B - g0) + 15) / 16;
    if (g0 > 0) __syncthreads();   // every warp has read the previous rows
    if (tid < kHalf) {
      // Rows g0 .. of q_nope[., h, :] (256 B each), whole 16-row tiles (rows
      // past B as zeros): load j is 16-byte chunk j % 16 of row j / 16.
      for (int j = tid; j < tiles * 16 * 16; j += kHalf) {
        const int row = j >> 4, ch = j & 15, b = g0 + row;
        const uint4 v = b < B ? reinterpret_cast<const uint4*>(q_nope + (size_t(b) * H + h) * kDn)[ch]
                              : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(qs + row * kQsRow + ch * 16) = v;
      }
    } else if (g0 == 0) {
      for (int it = y * kHalf + tid - kHalf; it < B * (kDr / 2); it += kHalf * P::kCtasPerHead)
        rope_pair(q_rope, pos, th, q_pe, H, h, it);
    }
    if (g0 == 0) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();   // the rows and (first pass) every thread's W_UK pieces are in place
    for (int mt = 0; mt < tiles; ++mt) {
      const int bA = g0 + mt * 16 + gq, bB = bA + 8;
      float acc[2][2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // A fragment of k in [16ks, 16ks+16): lanes 0-7 / 8-15 / 16-23 / 24-31
        // address rows 0-7 / 8-15 / 0-7 / 8-15 of the tile at columns 16ks /
        // 16ks / 16ks+8 / 16ks+8, the order of the mma's four A registers.
        uint32_t a[4];
        ldsm_x4(qbase + (16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1)) * kQsRow +
                    (16 * ks + 8 * (lane >> 4)) * 2,
                a[0], a[1], a[2], a[3]);
        const int mi = lane >> 3;
        const int k = 16 * ks + ((mi & 1) << 3) + (lane & 7);
        const int ch = mi >> 1;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const uint32_t wbase = smem_u32(wt + (2 * warp + blk) * (kDn * 32));
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(wbase + k * 32 + ((ch ^ ((k >> 2) & 1)) << 4), b0, b1, b2, b3);
          mma_bf16(acc[blk][0], a, b0, b1);
          mma_bf16(acc[blk][1], a, b2, b3);
        }
      }
#pragma unroll
      for (int blk = 0; blk < 2; ++blk)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          const int c = c0 + 32 * warp + 16 * blk + 8 * nb + 2 * cq;
          if (bA < B)
            *reinterpret_cast<float2*>(q_abs + (size_t(bA) * H + h) * kDc + c) =
                make_float2(acc[blk][nb][0], acc[blk][nb][1]);
          if (bB < B)
            *reinterpret_cast<float2*>(q_abs + (size_t(bB) * H + h) * kDc + c) =
                make_float2(acc[blk][nb][2], acc[blk][nb][3]);
        }
    }
  }
}

template <int kWarps>
mla_status launch_absorb_head(const char* who, bool early, cudaStream_t s,
                              const __nv_bfloat16* qn, const __nv_bfloat16* qr,
                              const __nv_bfloat16* wk, const int32_t* positions,
                              const RopeTheta& th, float* qa, float* qp, int B, int H,
                              const CachePrefetch& pf) {
  using P = HeadPlan<kWarps>;
  static DeviceFlags attr_done;
  const int dev = current_device();
  if (!attr_done.test(dev)) {
    if (cudaFuncSetAttribute(absorb_bf16_head_kernel<kWarps>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(P::kSmem)) != cudaSuccess) {
      set_error("%s: cannot reserve %zu bytes of shared memory", who, P::kSmem);
      return MLA_ERR_CUDA;
    }
    attr_done.set(dev);
  }
  const dim3 grid(H, P::kCtasPerHead);
  if (early)
    launch_pdl(absorb_bf16_head_kernel<kWarps>, grid, dim3(P::kThreads), P::kSmem, s, qn, qr, wk,
               positions, th, qa, qp, B, H, pf);
  else
    absorb_bf16_head_kernel<kWarps><<<grid, P::kThreads, P::kSmem, s>>>(qn, qr, wk, positions,
                                                                         th, qa, qp, B, H, pf);
  return MLA_OK;
}

// ---------------------------------------------------------------------- absorb, fp32
// grid (H, B): thread t computes columns t, t+128, t+256, t+384 of q_abs[b,h,:].
__global__ void __launch_bounds__(128)
    absorb_f32_kernel(const float* __restrict__ q_nope, const float* __restrict__ q_rope,
                      const float* __restrict__ w_uk, const int32_t* __restrict__ pos,
                      const RopeTheta th, float* __restrict__ q_abs, float* __restrict__ q_pe,
                      int B, int H) {
  __shared__ float q[kDn];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  q[tid] = q_nope[(size_t(b) * H + h) * kDn + tid];
  if (tid < kDr / 2) rope_pair(q_rope, pos, th, q_pe, H, h, b * (kDr / 2) + tid);
  __syncthreads();
  const float* w = w_uk + size_t(h) * kDn * kDc;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int k = 0; k < kDn; ++k) {
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[r] = fmaf(q[k], w[size_t(k) * kDc + tid + 128 * r], acc[r]);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) q_abs[(size_t(b) * H + h) * kDc + tid + 128 * r] = acc[r];
}

// ---------------------------------------------------------------------- out_proj, bf16
// grid (H, d_v / (8 kNB)): CTA (h, eb) owns outputs e in [8 kNB eb, 8 kNB (eb + 1))
// for the whole batch, as kNB blocks of 8 that share the o_c fragments; warp w
// contracts the 128-wide quarter [128w, 128w+128) of d_c and the four partial
// sums meet in shared memory.  W_UV's rows are K-contiguous, so its B fragments
// come straight from global memory; o_c (fp32) enters the mma as bf16 hi + lo
// parts, keeping its rounding near 2^-17 relative.  Every load of a batch tile
// is issued before the first mma.  kNB = 1 spreads the weights over the most
// CTAs (small batches); kNB = 4 reads each head's o_c rows 4 times instead of
// 16 (large batches).
template <int kNB>
__global__ void __launch_bounds__(128)
    out_proj_bf16_kernel(const float* __restrict__ o_c, const __nv_bfloat16* __restrict__ w_uv,
                         float* __restrict__ out, int B, int H) {
  constexpr int kE = 8 * kNB;   // outputs per CTA
  __shared__ float red[4][16][kE + 1];
  const int h = blockIdx.x, eb = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int kw = 128 * warp;
  uint32_t bf[kNB][8][2];
#pragma unroll
  for (int nb = 0; nb < kNB; ++nb) {
    const __nv_bfloat16* wrow =
        w_uv + (size_t(h) * kDv + kE * eb + 8 * nb + gq) * kDc + kw + 2 * cq;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      bf[nb][ks][0] = *reinterpret_cast<const uint32_t*>(wrow + 16 * ks);
      bf[nb][ks][1] = *reinterpret_cast<const uint32_t*>(wrow + 16 * ks + 8);
    }
  }
  // Launched after the combine with programmatic serialization: the weight
  // loads above overlap it; o_c is its result.
  pdl_wait();
  for (int mt = 0; mt * 16 < B; ++mt) {
    const int bA = mt * 16 + gq, bB = bA + 8;
    const float* rA = o_c + (size_t(bA) * H + h) * kDc + kw + 2 * cq;
    const float* rB = o_c + (size_t(bB) * H + h) * kDc + kw + 2 * cq;
    float2 x[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const float2 z = make_float2(0.f, 0.f);
      x[ks][0] = bA < B ? *reinterpret_cast<const float2*>(rA + 16 * ks) : z;
      x[ks][1] = bB < B ? *reinterpret_cast<const float2*>(rB + 16 * ks) : z;
      x[ks][2] = bA < B ? *reinterpret_cast<const float2*>(rA + 16 * ks + 8) : z;
      x[ks][3] = bB < B ? *reinterpret_cast<const float2*>(rB + 16 * ks + 8) : z;
    }
    float acc[kNB][4];
#pragma unroll
    for (int nb = 0; nb < kNB; ++nb)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[nb][r] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) split_bf16(x[ks][r].x, x[ks][r].y, hi[r], lo[r]);
#pragma unroll
      for (int nb = 0; nb < kNB; ++nb) {
        mma_bf16(acc[nb], hi, bf[nb][ks][0], bf[nb][ks][1]);
        mma_bf16(acc[nb], lo, bf[nb][ks][0], bf[nb][ks][1]);
      }
    }
#pragma unroll
    for (int nb = 0; nb < kNB; ++nb) {
      red[warp][gq][8 * nb + 2 * cq] = acc[nb][0];
      red[warp][gq][8 * nb + 2 * cq + 1] = acc[nb][1];
      red[warp][gq + 8][8 * nb + 2 * cq] = acc[nb][2];
      red[warp][gq + 8][8 * nb + 2 * cq + 1] = acc[nb][3];
    }
    __syncthreads();
#pragma unroll
    for (int i = tid; i < 16 * kE; i += 128) {   // 16 rows x kE outputs
      const int r = i / kE, e = i % kE;
      const int b = mt * 16 + r;
      if (b < B)
        out[(size_t(b) * H + h) * kDv + kE * eb + e] =
            red[0][r][e] + red[1][r][e] + red[2][r][e] + red[3][r][e];
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------- out_proj, fp32
// grid (H, B): o_c row in shared memory; warp w produces e = w, w+4, ...
__global__ void __launch_bounds__(128)
    out_proj_f32_kernel(const float* __restrict__ o_c, const float* __restrict__ w_uv,
                        float* __restrict__ out, int B, int H) {
  __shared__ float x[kDc];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int c = tid; c < kDc; c += 128) x[c] = o_c[(size_t(b) * H + h) * kDc + c];
  __syncthreads();
  for (int e = warp; e < kDv; e += 4) {
    const float* w = w_uv + (size_t(h) * kDv + e) * kDc;
    float acc = 0.f;
#pragma unroll 4
    for (int c = lane; c < kDc; c += 32) acc = fmaf(w[c], x[c], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) out[(size_t(b) * H + h) * kDv + e] = acc;
  }
}

// ---------------------------------------------------------------------- fp32 row projections
// y[b, n] = sum_k x[b, k] * w[n, k] with w stored [N, K] (K contiguous): the
// cache append's fused down-projection kv_a_proj ("Deepseek V2 Lite Inference
// Engine in C", MLA notes) and the output projection W^O ("Multi-Head Latent
// Attention" eq. 3.3.3), for fp32 weights.  (bf16 weights go through the
// tensor-core weight stream of mla_wstream.cu.)
enum RowGemmMode { kWriteY = 0, kAppendRow = 1 };

struct RowGemmArgs {
  const void* x;               // [B, K] fp32 or bf16
  const __nv_bfloat16* w;      // [N, K]
  int B, K, N;
  float* y;                    // kWriteY: [B, N] fp32
  void* cache;                 // kAppendRow: [B, s_max, N] bf16
  const int32_t* positions;    // kAppendRow: [B], row written
  int s_max, d_c;              // kAppendRow: columns >= d_c are rotated
  int32_t* status;
};

// fp32 weights and inputs: one warp per output (b, n), fp32 arithmetic throughout.
template <int kMode>
__global__ void __launch_bounds__(256) rowgemm_f32_kernel(const RowGemmArgs a, const RopeTheta th,
                                                          const float* __restrict__ w) {
  const int warp = (blockIdx.x * 256 + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int npairs = a.N / 2;
  if (warp >= a.B * npairs) return;
  const int b = warp / npairs, n = 2 * (warp % npairs);
  const float* x = static_cast<const float*>(a.x) + size_t(b) * a.K;
  float v0 = 0.f, v1 = 0.f;
  for (int k = lane; k < a.K; k += 32) {
    const float xv = x[k];
    v0 = fmaf(xv, w[size_t(n) * a.K + k], v0);
    v1 = fmaf(xv, w[size_t(n + 1) * a.K + k], v1);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    v0 += __shfl_xor_sync(0xffffffffu, v0, off);
    v1 += __shfl_xor_sync(0xffffffffu, v1, off);
  }
  if (lane != 0) return;
  if constexpr (kMode == kWriteY) {
    a.y[size_t(b) * a.N + n] = v0;
    a.y[size_t(b) * a.N + n + 1] = v1;
  } else {
    const int pos = a.positions[b];
    if (pos < 0 || pos >= a.s_max) {
      report(a.status, MLA_DEV_LENGTH_OUT_OF_RANGE);
      return;
    }
    if (n >= a.d_c) {
      float sn, cs;
      sincosf(rope_angle(pos, th.turns[(n - a.d_c) / 2]), &sn, &cs);
      const float x0 = v0, x1 = v1;
      v0 = cs * x0 - sn * x1;
      v1 = sn * x0 + cs * x1;
    }
    float* row = static_cast<float*>(a.cache) + (size_t(b) * a.s_max + pos) * a.N;
    row[n] = v0;
    row[n + 1] = v1;
  }
}

// ---------------------------------------------------------------------- materialised weights
// out(h, m, n) = sum_{k < K} A(h, m, k) B(h, k, n), accumulated in fp32 and rounded
// once to T: one head's slice of W^KQ = (W^UK)^T W^UQ or of W^OV = W^O W^UV
// ("Multi-Head Latent Attention" 3.3, eq. 3.3.3 and 3.5).  A is addressed by
// strides (either its m or its k stride is 1), B and out have unit n stride.
// A weight transform made once per model, not per step: a plain SIMT tiling,
// 64 x 64 outputs per CTA, 4 x 4 per thread, K staged 64 at a time.
struct MatArgs {
  const void* a;
  long long a_h, a_m, a_k;
  const void* b;
  long long b_h, b_k;
  void* out;
  long long o_h, o_m;
  int M, N, K;
};

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(256) materialize_kernel(const MatArgs p) {
  __shared__ float As[64][65], Bs[64][64];
  const int h = blockIdx.z, m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const T* a = static_cast<const T*>(p.a) + h * p.a_h;
  const T* b = static_cast<const T*>(p.b) + h * p.b_h;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < p.K; k0 += 64) {
    for (int idx = tid; idx < 64 * 64; idx += 256) {
      // walk A along its unit stride so that neighbouring threads read neighbouring words
      const int m = p.a_m == 1 ? idx & 63 : idx >> 6, k = p.a_m == 1 ? idx >> 6 : idx & 63;
      const bool in = m0 + m < p.M && k0 + k < p.K;
      As[k][m] = in ? to_f(a[(m0 + m) * p.a_m + (k0 + k) * p.a_k]) : 0.f;
      const int kb = idx >> 6, nb = idx & 63;
      const bool inb = k0 + kb < p.K && n0 + nb < p.N;
      Bs[kb][nb] = inb ? to_f(b[(k0 + kb) * p.b_k + n0 + nb]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < 64; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[k][4 * ty + i];
        bv[i] = Bs[k][4 * tx + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  T* out = static_cast<T*>(p.out) + h * p.o_h;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + 4 * ty + i, n = n0 + 4 * tx + j;
      if (m < p.M && n < p.N) out[m * p.o_m + n] = from_f<T>(acc[i][j]);
    }
}

// q_pe[b, h, :] = RoPE(q_rope[b, h, :], positions[b]): one pair per thread.
template <typename T>
__global__ void __launch_bounds__(256) rope_q_kernel(const T* __restrict__ q_rope,
                                                     const int32_t* __restrict__ pos,
                                                     const RopeTheta th, float* __restrict__ q_pe,
                                                     int B, int H) {
  const int it = blockIdx.x * 256 + threadIdx.x;
  if (it >= B * H * (kDr / 2)) return;
  const int i = it % (kDr / 2), h = (it / (kDr / 2)) % H, b = it / (H * (kDr / 2));
  rope_pair(q_rope, pos, th, q_pe, H, h, b * (kDr / 2) + i);
}

}  // namespace
}  // namespace mla

using namespace mla;

// Dynamic shared memory (unused) of the early-launched absorb: with its static
// shared memory (4 KB) and the 1 KB the SM reserves per CTA, a CTA takes 48-49
// KB, so at most four fit on an SM; the total stays within the 48 KB a launch
// may use without opting in.
constexpr size_t kAbsorbSpreadSmem = (44u << 10) - 16;
static_assert(kAbsorbSpreadSmem + kDn * 32 <= (48u << 10),
              "the early absorb's shared memory needs no opt-in");

// Whether `p` is page-locked host memory (read by the kernels over the host link).
static bool host_resident(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

extern "C" mla_status mla_absorb_q(const mla_dims* dims, const void* q_nope, const void* q_rope,
                                   const void* w_uk, const int32_t* positions, double rope_base,
                                   void* q_abs, void* q_pe, void* stream) {
  CachePrefetch none{};
  return absorb_q("mla_absorb_q", dims, q_nope, q_rope, w_uk, positions, rope_base, q_abs, q_pe,
                  stream, none, false);
}

// theta_i / (2 pi) for `rope_base`, kept per thread for the last base seen
// (a step's host work is a few microseconds; 32 fp64 powers are a visible part).
static const RopeTheta& rope_theta(double rope_base) {
  thread_local double base = 0.0;
  thread_local RopeTheta th;
  if (base != rope_base) {
    for (int i = 0; i < kDr / 2; ++i) th.turns[i] = pow(rope_base, -2.0 * i / kDr) / (2.0 * M_PI);
    base = rope_base;
  }
  return th;
}

mla_status mla::absorb_q(const char* who, const mla_dims* dims, const void* q_nope,
                         const void* q_rope, const void* w_uk, const int32_t* positions,
                         double rope_base, void* q_abs, void* q_pe, void* stream,
                         const CachePrefetch& pf, bool early, int q_host) {
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!q_nope || !q_rope || !w_uk || !positions || !q_abs || !q_pe) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_abs) ||
      !aligned16(q_pe)) {
    set_error("%s: tensor pointers must be 16-byte aligned", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!(rope_base > 0.0) || !isfinite(rope_base)) {
    set_error("%s: rope_base must be finite and > 0", who);
    return MLA_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int B = dims->batch, H = dims->heads;
  const RopeTheta th = rope_theta(rope_base);
  if (dims->dtype != MLA_F32) {
    const auto* qn = static_cast<const __nv_bfloat16*>(q_nope);
    const auto* qr = static_cast<const __nv_bfloat16*>(q_rope);
    const auto* wk = static_cast<const __nv_bfloat16*>(w_uk);
    auto* qa = static_cast<float*>(q_abs);
    auto* qp = static_cast<float*>(q_pe);
    if (q_host < 0 ? host_resident(q_nope) : q_host == 1) {
      // Queries in host memory: read by fewer CTAs per head, about 64 CTAs in
      // all (one per head from 64 heads up).  Measured end to end, one direct
      // mla_decode_step call per step, against the 32-CTA-per-head form with
      // staged loads: 8 x 4096 rows x 16 heads 23.5 -> 20.9 us (four CTAs per
      // head; 21.0 with eight, 22.3 with one); 64 ragged sequences 120.2 ->
      // 100.3 us (106 with eight or one); 32 x 16384 rows x 128 heads 448 ->
      // 290 us (312 with four).
      const int per_head = std::max(1, std::min(4, 64 / H));
      st = per_head == 4   ? launch_absorb_head<4>(who, early, s, qn, qr, wk, positions, th, qa,
                                                   qp, B, H, pf)
           : per_head == 2 ? launch_absorb_head<8>(who, early, s, qn, qr, wk, positions, th, qa,
                                                   qp, B, H, pf)
                           : launch_absorb_head<16>(who, early, s, qn, qr, wk, positions, th, qa,
                                                    qp, B, H, pf);
      if (st != MLA_OK) return st;
    } else if (early) {
      // Launched while the previous step's fused tail fills most SMs' register
      // files, the grid's small CTAs would all land on the few SMs left free
      // (measured on 8 sequences x 16 heads: 512 CTAs on 24 SMs, 22 per SM,
      // 3.3 us from the wait to the last exit).  Unused shared memory caps
      // them at four per SM, so the rest start on the SMs the tail leaves:
      // 128 SMs, 1.7 us, and the step 19.5 -> 18.5 us.
      launch_pdl(absorb_bf16_kernel, dim3(H, kDc / 16), dim3(32), kAbsorbSpreadSmem, s, qn, qr,
                 wk, positions, th, qa, qp, B, H, pf);
    } else {
      absorb_bf16_kernel<<<dim3(H, kDc / 16), 32, 0, s>>>(qn, qr, wk, positions, th, qa, qp, B,
                                                          H, pf);
    }
  } else {
    absorb_f32_kernel<<<dim3(H, B), 128, 0, s>>>(
        static_cast<const float*>(q_nope), static_cast<const float*>(q_rope),
        static_cast<const float*>(w_uk), positions, th, static_cast<float*>(q_abs),
        static_cast<float*>(q_pe), B, H);
  }
  return launch_status(who);
}

extern "C" mla_status mla_out_proj(const mla_dims* dims, const float* o_c, const void* w_uv,
                                   void* out, void* stream) {
  const char* who = "mla_out_proj";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!o_c || !w_uv || !out) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned16(o_c) || !aligned16(w_uv) || !aligned16(out)) {
    set_error("%s: tensor pointers must be 16-byte aligned", who);
    return MLA_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int B = dims->batch, H = dims->heads;
  if (dims->dtype != MLA_F32) {
    if (B > 16)
      launch_pdl(out_proj_bf16_kernel<4>, dim3(H, kDv / 32), dim3(128), 0, s, o_c,
                 static_cast<const __nv_bfloat16*>(w_uv), static_cast<float*>(out), B, H);
    else
      launch_pdl(out_proj_bf16_kernel<1>, dim3(H, kDv / 8), dim3(128), 0, s, o_c,
                 static_cast<const __nv_bfloat16*>(w_uv), static_cast<float*>(out), B, H);
  } else {
    out_proj_f32_kernel<<<dim3(H, B), 128, 0, s>>>(o_c, static_cast<const float*>(w_uv),
                                                   static_cast<float*>(out), B, H);
  }
  return launch_status(who);
}

extern "C" mla_status mla_cache_append(const mla_dims* dims, int32_t hidden, const void* x,
                                       const void* w_kva, const int32_t* positions,
                                       double rope_base, void* cache, int32_t* dev_status,
                                       void* stream) {
  const char* who = "mla_cache_append";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!x || !w_kva || !positions || !cache) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned16(x) || !aligned16(w_kva) || !aligned16(cache)) {
    set_error("%s: x, w_kva and cache must be 16-byte aligned", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (hidden <= 0 || hidden % 128 != 0) {
    set_error("%s: hidden = %d must be a positive multiple of 128", who, hidden);
    return hidden <= 0 ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED;
  }
  if (!(rope_base > 0.0) || !isfinite(rope_base)) {
    set_error("%s: rope_base must be finite and > 0", who);
    return MLA_ERR_INVALID_ARG;
  }
  RopeTheta th;
  for (int i = 0; i < kDr / 2; ++i) th.turns[i] = pow(rope_base, -2.0 * i / kDr) / (2.0 * M_PI);
  RowGemmArgs a{};
  a.x = x;
  a.w = static_cast<const __nv_bfloat16*>(w_kva);
  a.B = dims->batch;
  a.K = hidden;
  a.N = kRow;
  a.cache = cache;
  a.positions = positions;
  a.s_max = dims->s_max;
  a.d_c = kDc;
  a.status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dims->dtype != MLA_F32) {
    WStreamJob j{};
    j.mode = kWsAppendRow;
    j.x_f32 = false;
    j.x = x;
    j.w = w_kva;
    j.B = dims->batch;
    j.K = hidden;
    j.N = kRow;
    j.cache = cache;
    j.cache_fp8 = dims->dtype == MLA_FP8_E4M3;
    j.positions = positions;
    j.s_max = dims->s_max;
    j.d_c = kDc;
    for (int i = 0; i < kDr / 2; ++i) j.turns[i] = th.turns[i];
    j.status = dev_status;
    return wstream_launch(j, s, who);
  } else {
    const int warps = a.B * kRow / 2;
    rowgemm_f32_kernel<kAppendRow><<<(warps + 7) / 8, 256, 0, s>>>(a, th,
                                                                   static_cast<const float*>(w_kva));
  }
  return launch_status(who);
}

extern "C" mla_status mla_wo_proj(const mla_dims* dims, int32_t hidden, const float* o,
                                  const void* w_o, float* y, void* stream) {
  const char* who = "mla_wo_proj";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!o || !w_o || !y) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned16(o) || !aligned16(w_o) || !aligned16(y)) {
    set_error("%s: o, w_o and y must be 16-byte aligned", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (hidden <= 0 || hidden % 8 != 0) {
    set_error("%s: hidden = %d must be a positive multiple of 8", who, hidden);
    return hidden <= 0 ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED;
  }
  RowGemmArgs a{};
  a.x = o;
  a.w = static_cast<const __nv_bfloat16*>(w_o);
  a.B = dims->batch;
  a.K = dims->heads * kDv;
  a.N = hidden;
  a.y = y;
  RopeTheta th{};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dims->dtype != MLA_F32) {
    if (a.K % 128 != 0) {
      set_error("%s: heads * d_v = %d must be a multiple of 128", who, a.K);
      return MLA_ERR_UNSUPPORTED;
    }
    WStreamJob j{};
    j.mode = kWsWriteY;
    j.x_f32 = true;
    j.x = o;
    j.w = w_o;
    j.B = dims->batch;
    j.K = a.K;
    j.N = hidden;
    j.y = y;
    return wstream_launch(j, s, who);
  } else {
    const int warps = a.B * hidden / 2;
    rowgemm_f32_kernel<kWriteY><<<(warps + 7) / 8, 256, 0, s>>>(a, th, static_cast<const float*>(w_o));
  }
  return launch_status(who);
}

// ------------------------------------------------------------------ materialised absorption
static mla_status materialize(const char* who, const mla_dims* dims, const MatArgs& a,
                              cudaStream_t s) {
  const dim3 grid((a.N + 63) / 64, (a.M + 63) / 64, dims->heads);
  if (dims->dtype == MLA_F32)
    materialize_kernel<float><<<grid, 256, 0, s>>>(a);
  else
    materialize_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
  return launch_status(who);
}

extern "C" mla_status mla_materialize_wkq(const mla_dims* dims, int32_t d_in,
                                          const void* w_q_nope, const void* w_uk, void* w_kq,
                                          void* stream) {
  const char* who = "mla_materialize_wkq";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!w_q_nope || !w_uk || !w_kq || !aligned16(w_q_nope) || !aligned16(w_uk) ||
      !aligned16(w_kq)) {
    set_error("%s: w_q_nope, w_uk and w_kq must be non-NULL 16-byte aligned pointers", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (d_in <= 0) {
    set_error("%s: d_in = %d must be positive", who, d_in);
    return MLA_ERR_INVALID_ARG;
  }
  // W^KQ[h, c, i] = sum_d W^UK[h, d, c] W^UQ[h, d, i]
  MatArgs a{};
  a.a = w_uk;
  a.a_h = static_cast<long long>(kDn) * kDc;
  a.a_m = 1;
  a.a_k = kDc;
  a.b = w_q_nope;
  a.b_h = static_cast<long long>(kDn) * d_in;
  a.b_k = d_in;
  a.out = w_kq;
  a.o_h = static_cast<long long>(kDc) * d_in;
  a.o_m = d_in;
  a.M = kDc;
  a.N = d_in;
  a.K = kDn;
  return materialize(who, dims, a, static_cast<cudaStream_t>(stream));
}

extern "C" mla_status mla_materialize_wov(const mla_dims* dims, int32_t d_out, const void* w_o,
                                          const void* w_uv, void* w_ov, void* stream) {
  const char* who = "mla_materialize_wov";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!w_o || !w_uv || !w_ov || !aligned16(w_o) || !aligned16(w_uv) || !aligned16(w_ov)) {
    set_error("%s: w_o, w_uv and w_ov must be non-NULL 16-byte aligned pointers", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (d_out <= 0) {
    set_error("%s: d_out = %d must be positive", who, d_out);
    return MLA_ERR_INVALID_ARG;
  }
  // W^OV[n, h d_c + c] = sum_e W^O[n, h d_v + e] W^UV[h, e, c]
  const long long H = dims->heads;
  MatArgs a{};
  a.a = w_o;
  a.a_h = kDv;
  a.a_m = H * kDv;
  a.a_k = 1;
  a.b = w_uv;
  a.b_h = static_cast<long long>(kDv) * kDc;
  a.b_k = kDc;
  a.out = w_ov;
  a.o_h = kDc;
  a.o_m = H * kDc;
  a.M = d_out;
  a.N = kDc;
  a.K = kDv;
  return materialize(who, dims, a, static_cast<cudaStream_t>(stream));
}

extern "C" mla_status mla_absorb_q_materialized(const mla_dims* dims, int32_t d_in, const void* x,
                                                const void* w_kq, const void* q_rope,
                                                const int32_t* positions, double rope_base,
                                                float* q_abs, float* q_pe, void* stream) {
  const char* who = "mla_absorb_q_materialized";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!x || !w_kq || !q_rope || !positions || !q_abs || !q_pe) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned16(x) || !aligned16(w_kq) || !aligned16(q_rope) || !aligned16(q_abs) ||
      !aligned16(q_pe)) {
    set_error("%s: tensor pointers must be 16-byte aligned", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (d_in <= 0 || d_in % 64 != 0) {
    set_error("%s: d_in = %d must be a positive multiple of 64", who, d_in);
    return d_in <= 0 ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED;
  }
  if (!(rope_base > 0.0) || !isfinite(rope_base)) {
    set_error("%s: rope_base must be finite and > 0", who);
    return MLA_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int B = dims->batch, H = dims->heads;
  RopeTheta th;
  for (int i = 0; i < kDr / 2; ++i) th.turns[i] = pow(rope_base, -2.0 * i / kDr) / (2.0 * M_PI);
  // q_abs [B, H * d_c] = x . W^KQ^T, W^KQ stored [H * d_c, d_in]
  if (dims->dtype != MLA_F32) {
    WStreamJob j{};
    j.mode = kWsWriteY;
    j.x_f32 = false;
    j.x = x;
    j.w = w_kq;
    j.B = B;
    j.K = d_in;
    j.N = H * kDc;
    j.y = q_abs;
    st = wstream_launch(j, s, who);
    if (st != MLA_OK) return st;
  } else {
    RowGemmArgs a{};
    a.x = x;
    a.B = B;
    a.K = d_in;
    a.N = H * kDc;
    a.y = q_abs;
    const int warps = a.B * a.N / 2;
    RopeTheta none{};
    rowgemm_f32_kernel<kWriteY><<<(warps + 7) / 8, 256, 0, s>>>(a, none,
                                                               static_cast<const float*>(w_kq));
    st = launch_status(who);
    if (st != MLA_OK) return st;
  }
  const int pairs = B * H * (kDr / 2);
  if (dims->dtype == MLA_F32)
    rope_q_kernel<float><<<(pairs + 255) / 256, 256, 0, s>>>(static_cast<const float*>(q_rope),
                                                             positions, th, q_pe, B, H);
  else
    rope_q_kernel<__nv_bfloat16><<<(pairs + 255) / 256, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(q_rope), positions, th, q_pe, B, H);
  return launch_status(who);
}

extern "C" mla_status mla_ov_proj(const mla_dims* dims, int32_t d_out, const float* o_c,
                                  const void* w_ov, float* y, void* stream) {
  const char* who = "mla_ov_proj";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (!o_c || !w_ov || !y || !aligned16(o_c) || !aligned16(w_ov) || !aligned16(y)) {
    set_error("%s: o_c, w_ov and y must be non-NULL 16-byte aligned pointers", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (d_out <= 0 || d_out % 8 != 0) {
    set_error("%s: d_out = %d must be a positive multiple of 8", who, d_out);
    return d_out <= 0 ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // y [B, d_out] = concat_h(o_c[:, h, :]) . W^OV^T, W^OV stored [d_out, H * d_c]
  if (dims->dtype != MLA_F32) {
    WStreamJob j{};
    j.mode = kWsWriteY;
    j.x_f32 = true;
    j.x = o_c;
    j.w = w_ov;
    j.B = dims->batch;
    j.K = dims->heads * kDc;
    j.N = d_out;
    j.y = y;
    return wstream_launch(j, s, who);
  }
  RowGemmArgs a{};
  a.x = o_c;
  a.B = dims->batch;
  a.K = dims->heads * kDc;
  a.N = d_out;
  a.y = y;
  RopeTheta none{};
  const int warps = a.B * d_out / 2;
  rowgemm_f32_kernel<kWriteY><<<(warps + 7) / 8, 256, 0, s>>>(a, none, static_cast<const float*>(w_ov));
  return launch_status(who);
}
