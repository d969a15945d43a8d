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
// whose time goes into streaming the bf16 weights once; the bf16 kernels stage
// a weight tile in shared memory (XOR-swizzled 16-byte chunks) and run the
// batch as the M side of mma.sync m16n8k16 with fp32 accumulation.
#include <math.h>

#include "mla_common.cuh"

namespace mla {
namespace {

// ---------------------------------------------------------------------- RoPE
// theta_i = base^(-2i/d_rope); the angle pos * theta_i is formed in fp64 so
// that positions up to 2^31 keep their fractional turns.
template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ void rope_pairs(const T* q_rope, const int32_t* positions, double base, float* q_pe,
                           int B, int H, int h, int tid, int nthreads) {
  for (int it = tid; it < B * (kDr / 2); it += nthreads) {
    const int b = it / (kDr / 2), i = it % (kDr / 2);
    const double theta = pow(base, -2.0 * i / kDr);
    const double ang = static_cast<double>(positions[b]) * theta;
    double sn, cs;
    sincos(ang, &sn, &cs);
    const size_t off = (size_t(b) * H + h) * kDr + 2 * i;
    const double x0 = to_f(q_rope[off]), x1 = to_f(q_rope[off + 1]);
    q_pe[off] = static_cast<float>(cs * x0 - sn * x1);
    q_pe[off + 1] = static_cast<float>(sn * x0 + cs * x1);
  }
}

// ---------------------------------------------------------------------- absorb, bf16
// grid (H, d_c/64): CTA (h, cb) owns output columns [64cb, 64cb+64) of head h
// for the whole batch; warp w owns 16 of those columns.
__global__ void __launch_bounds__(128)
    absorb_bf16_kernel(const __nv_bfloat16* __restrict__ q_nope,
                       const __nv_bfloat16* __restrict__ q_rope,
                       const __nv_bfloat16* __restrict__ w_uk, const int32_t* __restrict__ pos,
                       double base, float* __restrict__ q_abs, float* __restrict__ q_pe, int B,
                       int H) {
  __shared__ __align__(128) uint8_t wt[kDn * 128];  // 128 k-rows x 64 bf16 columns
  const int h = blockIdx.x, cb = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = cb * 64;
  for (int idx = tid; idx < kDn * 8; idx += 128) {
    const int k = idx >> 3, ch = idx & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(w_uk + (size_t(h) * kDn + k) * kDc + c0 + ch * 8);
    *reinterpret_cast<uint4*>(wt + k * 128 + ((ch ^ (k & 7)) << 4)) = v;
  }
  if (cb == 0) rope_pairs(q_rope, pos, base, q_pe, B, H, h, tid, 128);
  __syncthreads();

  const int gq = lane >> 2, cq = lane & 3;
  const uint32_t wbase = smem_u32(wt);
  for (int mt = 0; mt * 16 < B; ++mt) {
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int bA = mt * 16 + gq, bB = bA + 8;
#pragma unroll
    for (int ks = 0; ks < kDn / 16; ++ks) {
      const int k0 = ks * 16;
      uint32_t a[4];
      const __nv_bfloat16* rA = q_nope + (size_t(bA) * H + h) * kDn + k0 + 2 * cq;
      const __nv_bfloat16* rB = q_nope + (size_t(bB) * H + h) * kDn + k0 + 2 * cq;
      a[0] = bA < B ? *reinterpret_cast<const uint32_t*>(rA) : 0u;
      a[1] = bB < B ? *reinterpret_cast<const uint32_t*>(rB) : 0u;
      a[2] = bA < B ? *reinterpret_cast<const uint32_t*>(rA + 8) : 0u;
      a[3] = bB < B ? *reinterpret_cast<const uint32_t*>(rB + 8) : 0u;
      const int mi = lane >> 3;
      const int k = k0 + ((mi & 1) << 3) + (lane & 7);
      const int ch = 2 * warp + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(wbase + k * 128 + ((ch ^ (k & 7)) << 4), b0, b1, b2, b3);
      mma_bf16(acc[0], a, b0, b1);
      mma_bf16(acc[1], a, b2, b3);
    }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const int c = c0 + 16 * warp + 8 * nb + 2 * cq;
      if (bA < B)
        *reinterpret_cast<float2*>(q_abs + (size_t(bA) * H + h) * kDc + c) =
            make_float2(acc[nb][0], acc[nb][1]);
      if (bB < B)
        *reinterpret_cast<float2*>(q_abs + (size_t(bB) * H + h) * kDc + c) =
            make_float2(acc[nb][2], acc[nb][3]);
    }
  }
}

// ---------------------------------------------------------------------- absorb, fp32
// grid (H, B): thread t computes columns t, t+128, t+256, t+384 of q_abs[b,h,:].
__global__ void __launch_bounds__(128)
    absorb_f32_kernel(const float* __restrict__ q_nope, const float* __restrict__ q_rope,
                      const float* __restrict__ w_uk, const int32_t* __restrict__ pos,
                      double base, float* __restrict__ q_abs, float* __restrict__ q_pe, int B,
                      int H) {
  __shared__ float q[kDn];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  q[tid] = q_nope[(size_t(b) * H + h) * kDn + tid];
  if (b == 0) rope_pairs(q_rope, pos, base, q_pe, B, H, h, tid, 128);
  __syncthreads();
  const float* w = w_uk + size_t(h) * kDn * kDc;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k = 0; k < kDn; ++k) {
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[r] = fmaf(q[k], w[size_t(k) * kDc + tid + 128 * r], acc[r]);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) q_abs[(size_t(b) * H + h) * kDc + tid + 128 * r] = acc[r];
}

// ---------------------------------------------------------------------- out_proj, bf16
// grid (H, d_v/32): CTA (h, eb) owns outputs e in [32eb, 32eb+32) for the whole
// batch; warp w owns 8 of them.  o_c (fp32) enters the mma as bf16 hi + lo
// halves, so its rounding stays below 2^-16 relative.
__global__ void __launch_bounds__(128)
    out_proj_bf16_kernel(const float* __restrict__ o_c, const __nv_bfloat16* __restrict__ w_uv,
                         float* __restrict__ out, int B, int H) {
  __shared__ __align__(128) uint8_t wt[32 * kDc * 2];  // 32 e-rows x 512 bf16
  const int h = blockIdx.x, eb = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = eb * 32;
  for (int idx = tid; idx < 32 * 64; idx += 128) {
    const int e = idx >> 6, ch = idx & 63;
    const uint4 v = *reinterpret_cast<const uint4*>(w_uv + (size_t(h) * kDv + e0 + e) * kDc + ch * 8);
    *reinterpret_cast<uint4*>(wt + e * 1024 + ((ch ^ (e & 7)) << 4)) = v;
  }
  __syncthreads();
  const int gq = lane >> 2, cq = lane & 3;
  const uint32_t wbase = smem_u32(wt);
  for (int mt = 0; mt * 16 < B; ++mt) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int bA = mt * 16 + gq, bB = bA + 8;
    const float* rA = o_c + (size_t(bA) * H + h) * kDc + 2 * cq;
    const float* rB = o_c + (size_t(bB) * H + h) * kDc + 2 * cq;
    for (int ks2 = 0; ks2 < kDc / 32; ++ks2) {
      const int e = 8 * warp + (lane & 7);
      const int ch = ks2 * 4 + (lane >> 3);
      uint32_t bf[4];
      ldsm_x4(wbase + e * 1024 + ((ch ^ (e & 7)) << 4), bf[0], bf[1], bf[2], bf[3]);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int k0 = ks2 * 32 + half * 16;
        float2 x[4];
        x[0] = bA < B ? *reinterpret_cast<const float2*>(rA + k0) : make_float2(0.f, 0.f);
        x[1] = bB < B ? *reinterpret_cast<const float2*>(rB + k0) : make_float2(0.f, 0.f);
        x[2] = bA < B ? *reinterpret_cast<const float2*>(rA + k0 + 8) : make_float2(0.f, 0.f);
        x[3] = bB < B ? *reinterpret_cast<const float2*>(rB + k0 + 8) : make_float2(0.f, 0.f);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const __nv_bfloat162 hv = __floats2bfloat162_rn(x[r].x, x[r].y);
          const float2 hf = __bfloat1622float2(hv);
          hi[r] = *reinterpret_cast<const uint32_t*>(&hv);
          lo[r] = pack_bf16(x[r].x - hf.x, x[r].y - hf.y);
        }
        mma_bf16(acc, hi, bf[2 * half], bf[2 * half + 1]);
        mma_bf16(acc, lo, bf[2 * half], bf[2 * half + 1]);
      }
    }
    const int e = e0 + 8 * warp + 2 * cq;
    if (bA < B)
      *reinterpret_cast<float2*>(out + (size_t(bA) * H + h) * kDv + e) = make_float2(acc[0], acc[1]);
    if (bB < B)
      *reinterpret_cast<float2*>(out + (size_t(bB) * H + h) * kDv + e) = make_float2(acc[2], acc[3]);
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
    for (int c = lane; c < kDc; c += 32) acc = fmaf(w[c], x[c], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) out[(size_t(b) * H + h) * kDv + e] = acc;
  }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_absorb_q(const mla_dims* dims, const void* q_nope, const void* q_rope,
                                   const void* w_uk, const int32_t* positions, double rope_base,
                                   void* q_abs, void* q_pe, void* stream) {
  const char* who = "mla_absorb_q";
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
  if (dims->dtype == MLA_BF16) {
    absorb_bf16_kernel<<<dim3(H, kDc / 64), 128, 0, s>>>(
        static_cast<const __nv_bfloat16*>(q_nope), static_cast<const __nv_bfloat16*>(q_rope),
        static_cast<const __nv_bfloat16*>(w_uk), positions, rope_base,
        static_cast<float*>(q_abs), static_cast<float*>(q_pe), B, H);
  } else {
    absorb_f32_kernel<<<dim3(H, B), 128, 0, s>>>(
        static_cast<const float*>(q_nope), static_cast<const float*>(q_rope),
        static_cast<const float*>(w_uk), positions, rope_base, static_cast<float*>(q_abs),
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
  if (dims->dtype == MLA_BF16) {
    out_proj_bf16_kernel<<<dim3(H, kDv / 32), 128, 0, s>>>(
        o_c, static_cast<const __nv_bfloat16*>(w_uv), static_cast<float*>(out), B, H);
  } else {
    out_proj_f32_kernel<<<dim3(H, B), 128, 0, s>>>(o_c, static_cast<const float*>(w_uv),
                                                   static_cast<float*>(out), B, H);
  }
  return launch_status(who);
}
