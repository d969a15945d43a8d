// The split kernel of mla_decode_attn for an FP8 (E4M3) latent cache.
//
// "Multi-Head Latent Attention" (Lior Sinai), 3.1: a cache element takes one to
// four bytes, FP8 to FP32; with one byte per element the cache row of 576 values
// is 576 bytes, half the bf16 stream.  The arithmetic is that of the bf16 path
// (3.3, 3.6): per head the score of row t is
// (q_abs . c_t + q_pe . k_rope_t) / sqrt(d_h + d_R), an online softmax over the
// chunk's rows, and the normalised latent output with its log-sum-exp.  The
// cache values are the E4M3 numbers themselves (no scale).
//
// Both products run on the tensor cores as tcgen05.mma kind::f8f6f4 with E4M3
// operands and fp32 accumulators:
//   scores  S[128 rows x 64] = C[128 x 576] . Q^T       (C K-major)
//   output  O^T[128 latent x 48] += C^T[128 x 128 rows] . P^T   per 128-column block
//           (C read MN-major from the same shared-memory boxes)
// A 128-row tile of E4M3 rows is five 128-column boxes (80 KB; the fifth holds
// the 64 RoPE columns and TMA's zero fill), so two tiles stay resident from
// their arrival to their PV product: no second pass over L2.
// The fp32 query enters as four E4M3 parts with a power-of-two scale per
// head, sigma (weights 1, 1/16, 1/256, 1/4096), P as three parts (1, 1/16,
// 1/256), so they keep about 16 and 12 significant bits against E4M3's 4
// (rows that dominate a softmax carry their rounding into the output
// unaveraged).
//
// The query parts are made once per step by fp8_q_prep_kernel (E4M3
// conversions run at an eighth of the fp32 rate, and every chunk's CTA would
// repeat them) and copied into each CTA's shared memory in one bulk copy.
//
// Warp roles of the split (352 threads, one CTA per SM):
//   warp 8      TMA producer (and TMEM allocation)
//   warp 9      score MMAs of each tile (18 instructions)
//   warp 10     the query image's bulk copy, then the PV MMAs of each tile (16)
//   warps 0-7   softmax (one tile row per thread, heads 0-7 in warps 0-3 and
//               8-15 in warps 4-7), P, epilogue
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include "mla_split.cuh"

namespace mla {
namespace {

constexpr int kF8Threads = 352;
constexpr int kF8Soft = 256;
constexpr int kF8Rows = 128;                  // rows per tile (the MMA's M)
constexpr int kF8Boxes = 5;                   // 128-column boxes per tile
constexpr int kF8Box = kF8Rows * 128;         // 16 KB
constexpr int kF8Tile = kF8Boxes * kF8Box;    // 80 KB
constexpr int kQParts = 4, kPParts = 3;
constexpr int kHalf = kHeadGroup / 2;         // heads per softmax warp group
constexpr int kQN = kQParts * kHeadGroup;     // query rows of the score MMA (part-major)
constexpr int kPN = kPParts * kHeadGroup;     // P rows of the PV MMA (part-major)
constexpr int kQBox = kQN * 128;              // 8 KB per 128-column box
static_assert(size_t(kF8Boxes) * kQBox == kFp8QBoxes, "query image layout");
constexpr int kPBuf = kPN * 128;              // 6 KB: 48 rows of 128 tile rows
constexpr int kOffTile = 0;
constexpr int kOffQ = kOffTile + 2 * kF8Tile;
constexpr int kOffP = kOffQ + kF8Boxes * kQBox;
constexpr int kOffRed = kOffP + 2 * kPBuf;                   // [2][16 heads][4 warps] maxima
constexpr int kOffLsum = kOffRed + 2 * kHeadGroup * 4 * 4;  // [16 heads][4 warps]
constexpr int kOffSigma = kOffLsum + kHeadGroup * 4 * 4;    // query scale per head
constexpr int kOffBar = kOffSigma + kHeadGroup * 4;
enum {
  B_FULL = 0,      // [2] tile landed
  B_EMPTY = 2,     // [2] tile's PV finished: buffer free
  B_SFULL = 4,     // [2] scores of the tile in S[t & 1]
  B_SFREE = 6,     // [2] softmax read S[t & 1]
  B_PFULL = 8,     // [2] P of the tile written (and the tile's dead rows zeroed)
  B_ODONE = 10,    // [2] PV of the tile finished
  B_QREADY = 12,   // query parts written
  B_DONE = 13,     // every MMA finished
  kNumBars = 14
};
constexpr int kOffSlot = kOffBar + 8 * kNumBars;
constexpr int kOffAbort = kOffSlot + 16;
constexpr size_t kF8Smem = 1024 + kOffAbort + 16;
constexpr uint32_t kTmemCols = 512;   // S[2] at 0 / 64 (64 columns each), O^T at 128..319
constexpr uint32_t kOCol = 128;       // O^T block mb at kOCol + kPN mb
constexpr float kRescaleLog2 = 8.f;

static_assert(kF8Smem <= 232448, "shared memory");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "128-byte swizzle atoms");

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format 0) and an
// fp32 accumulator; a_mn selects an MN-major A.
constexpr uint32_t idesc_e4m3(int M, int N, int a_mn) {
  return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ bool f8_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitNs) {
      *abort = 1;
      return false;
    }
  }
}

// E4M3 encoding (round to nearest even, saturating at +-448) and the exact
// values back, two at a time (the conversions run at an eighth of the fp32
// rate; the x2 forms convert two per instruction): codes of (x0, x1) as the
// low and high byte.
__device__ __forceinline__ uint16_t to_e4m3x2(float x0, float x1) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float2 from_e4m3x2(uint16_t v) {
  const __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return __half22float2(__half2(h));
}

// Byte offset of K index k (< 128) in row n of a K-major box of 128-byte rows
// with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_byte(int n, int k) {
  return static_cast<uint32_t>(n * 128 + ((((k >> 4) ^ n) & 7) << 4) + (k & 15));
}

// The query image of one (sequence b, head h): v = [q_abs ; q_pe] (576 values)
// becomes sigma (a1 + a2 / 16 + a3 / 256 + a4 / 4096), a_i E4M3 and sigma a power
// of two that puts max |v| / sigma in [128, 256); part i goes to row
// 16 i + (h mod 16) of the head group's image, columns 576..639 are zero.
// grid (H, B), 160 threads: thread t < 144 converts values 4t .. 4t + 3.
__global__ void __launch_bounds__(160) fp8_q_prep_kernel(const SplitParams p) {
  __shared__ float wmax[5];
  pdl_launch_dependents();   // the split may begin its set-up and cache stream
  const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x, lane = t & 31;
  const int hh = h % kHeadGroup;
  uint8_t* img = p.q_img + (size_t(b) * (p.H / kHeadGroup) + h / kHeadGroup) * kFp8QImage;
  pdl_wait();   // q_abs and q_pe come from the kernel before
  const size_t bh = size_t(b) * p.H + h;
  const int c = 4 * t;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < kRow)
    v = c < kDc ? *reinterpret_cast<const float4*>(static_cast<const float*>(p.q_abs) + bh * kDc + c)
                : *reinterpret_cast<const float4*>(static_cast<const float*>(p.q_pe) + bh * kDr +
                                                   (c - kDc));
  float mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) wmax[t >> 5] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3])), wmax[4]);
  int ex = 0;
  frexpf(mx, &ex);   // mx = f 2^ex, f in [0.5, 1)
  const float sg = mx > 0.f ? ldexpf(1.f, ex - 8) : 1.f;
  const float inv = 1.f / sg;   // exact: a power of two
  if (t == 0) reinterpret_cast<float*>(img + kFp8QBoxes)[hh] = sg;
  if (c < kRow) {
    float x0 = v.x * inv, x1 = v.y * inv, x2 = v.z * inv, x3 = v.w * inv;
    uint8_t* bx = img + (c >> 7) * kQBox;
#pragma unroll
    for (int part = 0; part < kQParts; ++part) {
      const uint16_t lo = to_e4m3x2(x0, x1), hi = to_e4m3x2(x2, x3);
      *reinterpret_cast<uint32_t*>(bx + sw128_byte(kHeadGroup * part + hh, c & 127)) =
          static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      const float2 f01 = from_e4m3x2(lo), f23 = from_e4m3x2(hi);
      // the residuals of a rounding are exact
      x0 = (x0 - f01.x) * 16.f;
      x1 = (x1 - f01.y) * 16.f;
      x2 = (x2 - f23.x) * 16.f;
      x3 = (x3 - f23.y) * 16.f;
    }
  } else if (t < 144 + 16) {
    const int u = t - 144, part = u >> 2, q = u & 3;
    *reinterpret_cast<uint4*>(img + 4 * kQBox + sw128_byte(kHeadGroup * part + hh, 64 + 16 * q)) =
        make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(kF8Threads, 1)
    split_fp8_kernel(const __grid_constant__ CUtensorMap tmap, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBar;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
  float* sigma = reinterpret_cast<float*>(smem + kOffSigma);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* slot_ptr = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  auto bar = [&](int i) { return bars + 8 * i; };

  const int g = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = clamp_length(p, b, tid == 0 && g == 0 && j == 0);
  const int r0 = j * p.chunk;
  if (r0 >= len) return;   // chunk past the end of this sequence: nothing to do
  const int r1 = min(r0 + p.chunk, len);
  const int T = (r1 - r0 + kF8Rows - 1) / kF8Rows;
  const int last_valid = r1 - (r0 + (T - 1) * kF8Rows);
  // Rows of the last tile past the sequence's end may hold anything (NaN
  // included); they are zeroed before its PV.  Rows past the chunk but inside
  // the sequence are finite and get P = 0.
  const int zero_from = len - (r0 + (T - 1) * kF8Rows);
  const bool zero_last = zero_from < kF8Rows;
  const int row_base = cache_seq(p, b) * p.s_max + r0;
  const int h0 = g * kHeadGroup;

  // The cache stream starts first: the producer sets up the barriers and
  // issues the first two tiles before the CTA-wide barrier.
  auto issue = [&](int t) {
    const int bf = t & 1;
    mbar_arrive_expect_tx(bar(B_FULL + bf), kF8Tile);
    const uint64_t pol = l2_evict_first_policy();
#pragma unroll
    for (int m = 0; m < kF8Boxes; ++m)
      tma_load_2d(sbase + kOffTile + bf * kF8Tile + m * kF8Box, &tmap, 128 * m,
                  row_base + t * kF8Rows, bar(B_FULL + bf), pol);
  };
  if (warp == 8 && lane == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_FULL + i), 1);
      mbar_init(bar(B_EMPTY + i), 1);
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SFREE + i), 8);
      mbar_init(bar(B_PFULL + i), 8);
      mbar_init(bar(B_ODONE + i), 1);
    }
    mbar_init(bar(B_QREADY), 1);
    mbar_init(bar(B_DONE), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tmap(&tmap);
    for (int t = 0; t < 2 && t < T; ++t) issue(t);
  }
  if (warp == 8) {
    __syncwarp();
    tmem_alloc(smem_u32(slot_ptr), kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = T < 2 ? T : 2;
      for (int t = 2; t < T; ++t) {
        if (!f8_wait(bar(B_EMPTY + (t & 1)), ((t - 2) >> 1) & 1, abort_flag)) break;
        issue(t);
        issued = t + 1;
      }
      // Tiles still in flight land before the CTA may leave (bounded waits).
      for (int t = issued > 2 ? issued - 2 : 0; t < issued; ++t) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(bar(B_FULL + (t & 1)), (t >> 1) & 1))
          if (globaltimer_ns() - t0 > kWaitNs) {
            *abort_flag = 1;
            break;
          }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ score MMAs
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_e4m3(128, kQN, 0);
      f8_wait(bar(B_QREADY), 0, abort_flag);
      for (int t = 0; t < T && !*abort_flag; ++t) {
        const int bf = t & 1;
        if (!f8_wait(bar(B_FULL + bf), (t >> 1) & 1, abort_flag)) break;
        if (t >= 2 && !f8_wait(bar(B_SFREE + bf), ((t - 2) >> 1) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + 64 * bf;
#pragma unroll
        for (int m = 0; m < kF8Boxes; ++m) {
          const uint64_t a = umma_desc_sw128(sbase + kOffTile + bf * kF8Tile + m * kF8Box, 16, 1024);
          const uint64_t q = umma_desc_sw128(sbase + kOffQ + m * kQBox, 16, 1024);
          // a K step of 32 E4M3 columns moves the start by 32 B; the fifth box
          // holds 64 real columns
          const int ks = m < 4 ? 4 : 2;
          for (int k = 0; k < ks; ++k)
            umma_e4m3(d, a + 2 * k, q + 2 * k, idesc_s, (m > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_SFULL + bf));
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ query image, PV MMAs
    if (lane == 0) {
      pdl_wait();   // the image is written by the kernel before
      const uint8_t* img = p.q_img + (size_t(b) * (p.H / kHeadGroup) + g) * kFp8QImage;
      mbar_arrive_expect_tx(bar(B_QREADY), static_cast<uint32_t>(kFp8QImage));
      bulk_g2s(sbase + kOffQ, img, static_cast<uint32_t>(kFp8QBoxes), bar(B_QREADY));
      bulk_g2s(sbase + kOffSigma, img + kFp8QBoxes, 16 * sizeof(float), bar(B_QREADY));
      constexpr uint32_t idesc_o = idesc_e4m3(128, kPN, 1);
      for (int t = 0; t < T && !*abort_flag; ++t) {
        const int bf = t & 1;
        if (!f8_wait(bar(B_PFULL + bf), (t >> 1) & 1, abort_flag)) break;
        tc_fence_after();
        const uint64_t pd = umma_desc_sw128(sbase + kOffP + bf * kPBuf, 16, 1024);
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
          // C^T block mb: latent columns 128 mb.. (MN-major, one 128-byte
          // span), K = tile rows in 8-row groups 1024 B apart
          const uint64_t c = umma_desc_sw128(sbase + kOffTile + bf * kF8Tile + mb * kF8Box,
                                             kF8Box, 1024);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)   // 32 tile rows per step: 4096 B of C^T, 32 B of P^T
            umma_e4m3(tmem + kOCol + kPN * mb, c + ((ks * 4096) >> 4), pd + ((ks * 32) >> 4),
                      idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_ODONE + bf));
        umma_commit(bar(B_EMPTY + bf));
      }
      umma_commit(bar(B_DONE));
      mbar_wait_bounded(bar(B_DONE), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int gp = warp >> 2, wq = warp & 3;
    const int hb = kHalf * gp;                          // first head of this group
    const int row = 32 * wq + lane;                     // tile row held by this thread
    const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;

    f8_wait(bar(B_QREADY), 0, abort_flag);   // the query image and its scales
    float qsig[kHalf];
#pragma unroll
    for (int h = 0; h < kHalf; ++h) qsig[h] = sigma[hb + h] * p.scale_log2;

    float m[kHalf], l[kHalf];
#pragma unroll
    for (int h = 0; h < kHalf; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    for (int t = 0; t < T; ++t) {
      const int sb = t & 1;
      const int valid = t == T - 1 ? last_valid : kF8Rows;
      f8_wait(bar(B_SFULL + sb), (t >> 1) & 1, abort_flag);
      tc_fence_after();
      float sc[kHalf], tt[kHalf];
      {
        uint32_t s1[8], s2[8], s3[8], s4[8];
        tmem_ld8_nowait(tmem + lane_base + 64 * sb + hb, s1);
        tmem_ld8_nowait(tmem + lane_base + 64 * sb + kHeadGroup + hb, s2);
        tmem_ld8_nowait(tmem + lane_base + 64 * sb + 2 * kHeadGroup + hb, s3);
        tmem_ld8_nowait(tmem + lane_base + 64 * sb + 3 * kHeadGroup + hb, s4);
        tmem_wait_ld();
        const bool rv = row < valid;
#pragma unroll
        for (int h = 0; h < kHalf; ++h) {
          const float s = __uint_as_float(s1[h]) +
                          (__uint_as_float(s2[h]) * 0.0625f +
                           (__uint_as_float(s3[h]) * 0.00390625f +
                            __uint_as_float(s4[h]) * 0.000244140625f));
          sc[h] = rv ? s * qsig[h] : -INFINITY;
          tt[h] = sc[h];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SFREE + sb));
      // tile maximum per head: warp, then the group's four warps
#pragma unroll
      for (int h = 0; h < kHalf; ++h)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          tt[h] = fmaxf(tt[h], __shfl_xor_sync(0xffffffffu, tt[h], off));
      float* rd = red + sb * kHeadGroup * 4;
      if (lane < kHalf) {
        float v = tt[0];
#pragma unroll
        for (int h = 1; h < kHalf; ++h) v = lane == h ? tt[h] : v;
        rd[(hb + lane) * 4 + wq] = v;
      }
      named_bar_sync(1, kF8Soft);
      bool need = false;
      float tmax[kHalf];
#pragma unroll
      for (int h = 0; h < kHalf; ++h) {
        const float4 q4 = *reinterpret_cast<const float4*>(rd + (hb + h) * 4);
        tmax[h] = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
        need |= tmax[h] > m[h] + kRescaleLog2;
      }
      if (need) {
        // Move this group's reference maxima; rescale its row sums and the O^T
        // columns it owns (in TMEM, after the previous PV finished).
        float alpha[kHalf];
#pragma unroll
        for (int h = 0; h < kHalf; ++h) {
          const float mn = fmaxf(m[h], tmax[h]);
          alpha[h] = m[h] == -INFINITY ? 0.f : ex2(m[h] - mn);
          m[h] = mn;
          l[h] *= alpha[h];
        }
        if (t > 0) {
          f8_wait(bar(B_ODONE + ((t - 1) & 1)), ((t - 1) >> 1) & 1, abort_flag);
          tc_fence_after();
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int part = 0; part < kPParts; ++part) {
              const uint32_t col = kOCol + kPN * mb + kHeadGroup * part + hb;
              uint32_t r[8];
              float o[8];
              tmem_ld8_nowait(tmem + lane_base + col, r);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < kHalf; ++h) o[h] = __uint_as_float(r[h]) * alpha[h];
              tmem_st8(tmem + lane_base + col, o);
            }
          }
          tmem_wait_st();
        }
      }
      // p in [0, 2^8] as three E4M3 parts, two heads per conversion; the row
      // sum takes the value the PV uses.
      uint16_t pp[kPParts][kHalf / 2];
#pragma unroll
      for (int h2 = 0; h2 < kHalf / 2; ++h2) {
        float v0, v1;
        {
          const float mu0 = m[2 * h2] == -INFINITY ? 0.f : m[2 * h2];
          const float mu1 = m[2 * h2 + 1] == -INFINITY ? 0.f : m[2 * h2 + 1];
          v0 = ex2(sc[2 * h2] - mu0);
          v1 = ex2(sc[2 * h2 + 1] - mu1);
        }
        float used0 = 0.f, used1 = 0.f, wgt = 1.f;
#pragma unroll
        for (int part = 0; part < kPParts; ++part) {
          pp[part][h2] = to_e4m3x2(v0, v1);
          const float2 f = from_e4m3x2(pp[part][h2]);
          used0 += f.x * wgt;
          used1 += f.y * wgt;
          v0 = (v0 - f.x) * 16.f;
          v1 = (v1 - f.y) * 16.f;
          wgt *= 0.0625f;
        }
        l[2 * h2] += used0;
        l[2 * h2 + 1] += used1;
      }
      // P^T buffer sb was last read by the PV of tile t-2.
      if (t >= 2) f8_wait(bar(B_ODONE + sb), ((t - 2) >> 1) & 1, abort_flag);
      {
        // P^T (B operand of the PV MMA, K-major, 128-byte swizzle): row
        // 16 part + n is part `part` of head n; the K index is the tile row.
        uint8_t* pbuf = smem + kOffP + sb * kPBuf;
#pragma unroll
        for (int part = 0; part < kPParts; ++part)
#pragma unroll
          for (int h2 = 0; h2 < kHalf / 2; ++h2) {
            pbuf[sw128_byte(kHeadGroup * part + hb + 2 * h2, row)] = pp[part][h2] & 0xFF;
            pbuf[sw128_byte(kHeadGroup * part + hb + 2 * h2 + 1, row)] = pp[part][h2] >> 8;
          }
      }
      if (t == T - 1 && zero_last) {
        // Latent boxes 0-3 of the last tile: rows past the sequence's end -> 0.
        uint8_t* tile = smem + kOffTile + (t & 1) * kF8Tile;
        const int nrow = kF8Rows - zero_from;
        for (int c = tid; c < 4 * nrow * 8; c += kF8Soft) {
          const int mb = c / (nrow * 8), rem = c % (nrow * 8);
          *reinterpret_cast<uint4*>(tile + mb * kF8Box + (zero_from + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + sb));
    }
    // The combine may start launching: it waits for this grid anyway.
    if (tid == 0) pdl_launch_dependents();
    // Softmax denominators over the chunk's rows.
#pragma unroll
    for (int h = 0; h < kHalf; ++h)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
    if (lane < kHalf) {
      float v = l[0];
#pragma unroll
      for (int h = 1; h < kHalf; ++h) v = lane == h ? l[h] : v;
      lsum[(hb + lane) * 4 + wq] = v;
    }
    // O^T after the last PV: this thread's latent row is 128 mb + 32 wq + lane.
    f8_wait(bar(B_ODONE + ((T - 1) & 1)), ((T - 1) >> 1) & 1, abort_flag);
    tc_fence_after();
    named_bar_sync(1, kF8Soft);
    if (!*abort_flag) {
      const size_t base = (size_t(b) * p.H + h0) * p.splits + j;
      // 1/L by the approximate reciprocal (within 2 ulp for the L > 0 reached
      // here, 1 <= L <= 2^8 x rows), branch-free; lane h of the first warp of
      // each group writes head h's log-sum-exp.
      float inv[kHalf], Lme = 0.f, mme = 0.f;
#pragma unroll
      for (int h = 0; h < kHalf; ++h) {
        const float4 q4 = *reinterpret_cast<const float4*>(lsum + (hb + h) * 4);
        const float L = (q4.x + q4.y) + (q4.z + q4.w);
        inv[h] = L > 0.f ? __fdividef(1.f, L) : 0.f;
        Lme = lane == h ? L : Lme;
        mme = lane == h ? m[h] : mme;
      }
      if (wq == 0 && lane < kHalf)
        p.part_lse[base + size_t(hb + lane) * p.splits] =
            Lme > 0.f ? (mme + log2f(Lme)) * kLn2 : -INFINITY;
      float* row0 = p.part_o + (base + size_t(hb) * p.splits) * kDc + 32 * wq + lane;
      const size_t head_stride = size_t(p.splits) * kDc;
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
        uint32_t o1[8], o2[8], o3[8];
        tmem_ld8_nowait(tmem + lane_base + kOCol + kPN * mb + hb, o1);
        tmem_ld8_nowait(tmem + lane_base + kOCol + kPN * mb + kHeadGroup + hb, o2);
        tmem_ld8_nowait(tmem + lane_base + kOCol + kPN * mb + 2 * kHeadGroup + hb, o3);
        tmem_wait_ld();
        float* row = row0 + 128 * mb;
#pragma unroll
        for (int h = 0; h < kHalf; ++h, row += head_stride)
          *row = (__uint_as_float(o1[h]) +
                  (__uint_as_float(o2[h]) * 0.0625f + __uint_as_float(o3[h]) * 0.00390625f)) *
                 inv[h];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_flag) report(p.status, MLA_DEV_PIPELINE_TIMEOUT);
}

}  // namespace

mla_status launch_split_fp8(const SplitParams& p, const void* cache, cudaStream_t stream,
                            const char* who) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) {
    set_error("%s: cuTensorMapEncodeTiled is not available from the driver", who);
    return MLA_ERR_CUDA;
  }
  // The cache [B * s_max rows, 576 bytes] in 128-row x 128-byte boxes (128-byte
  // swizzle); the fifth box of a row reaches past column 576 and reads zeros.
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {cuuint64_t(kRow), cuuint64_t(p.B / p.q_len) * p.s_max};
  const cuuint64_t gstride[1] = {cuuint64_t(kRow)};
  const cuuint32_t box[2] = {128, cuuint32_t(kF8Rows)};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), gdim,
                   gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("%s: cuTensorMapEncodeTiled failed (%d)", who, int(r));
    return MLA_ERR_CUDA;
  }
  static DeviceFlags attr_done;
  const int dev = current_device();
  if (!attr_done.test(dev)) {
    if (cudaFuncSetAttribute(split_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kF8Smem)) != cudaSuccess) {
      set_error("%s: cannot reserve %zu bytes of shared memory", who, kF8Smem);
      return MLA_ERR_CUDA;
    }
    attr_done.set(dev);
  }
  launch_pdl(fp8_q_prep_kernel, dim3(p.H, p.B), dim3(160), 0, stream, p);
  dim3 grid(p.H / kHeadGroup, p.splits, p.B);
  launch_pdl(split_fp8_kernel, grid, dim3(kF8Threads), kF8Smem, stream, tmap, p);
  return launch_status(who);
}

}  // namespace mla
