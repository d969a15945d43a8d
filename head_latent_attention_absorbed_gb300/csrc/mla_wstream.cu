// Weight-streaming projection y = x . w^T on the 5th-generation tensor cores.
//
// The weight is the only large operand (kv_a_proj: 576 x hidden; W^O: hidden x
// H d_v) and is read once, so the kernel is a stream of weight tiles through
// shared memory into tcgen05.mma, with the batch rows as the MMA's N side:
//   y^T[n, b] (TMEM, fp32) += W[n, k-box] (A, 128 x 64, K-major) . x[b, k-box]^T
// grid (KS, ceil(N / 128), batch chunks), clusters of KS CTAs along K: CTA r of
// a cluster contracts the r-th of KS equal K ranges of one 128-row weight tile.
// Each CTA owns 128 / KS rows of the tile: the others send it their partial
// sums of those rows with bulk copies into its shared memory, and it adds them
// in rank order and writes the rows out (so a RoPE pair and the bf16 rounding
// of a cache row see the full sum).  The host picks KS so that the grid is
// one wave of clusters.
//
// Warp roles (224 threads, one CTA per SM):
//   warp 0      TMA producer: one 16 KB weight box per stage (and the bf16 x box)
//   warps 1, 2  MMA issue, stages of even / odd index, into two accumulators
//               (a thread issues one tcgen05.mma only every ~100 cycles)
//   warps 3-6   fp32 x: each stage's staged fp32 box split into the bf16
//               hi | lo rows of the B operand; then the epilogue (TMEM ->
//               shared memory, the partial-sum exchange, output)
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_wstream.cuh"

namespace mla {
namespace {

constexpr int kWsThreads = 224;
constexpr int kWsBox = 64;                           // K elements per box
constexpr uint32_t kWsWBytes = 128u * kWsBox * 2u;   // one weight box: 128 rows x 64 bf16
constexpr int kWsMaxStages = 8;
constexpr uint32_t kWsBarBytes = 512;
constexpr size_t kWsSmemMax = 232448;                // dynamic shared memory per CTA

struct WsParams {
  int B, K, N;
  int Bc, Nc;               // batch rows per chunk (multiple of 16); MMA N (Bc, or hi | lo = 2 Bc)
  int stages;               // ring depth, even
  uint32_t stage_bytes;     // weight box at 0, B operand at ops_off, fp32 x box at raw_off
  uint32_t ops_off, raw_off;
  uint32_t recv_off;        // partial sums received from the cluster's other CTAs
  uint32_t slice_bytes;     // one sender's slice: (128 / KS) rows of Bc + 4 floats
  uint32_t pos_off;         // positions of the chunk's rows (append)
  uint32_t bar_off;         // barriers; the send buffer reuses the ring
  uint32_t tmem_cols;
  int ks;                   // K splits = cluster size
  float* y;
  void* cache;              // bf16, or E4M3 with cache_fp8
  int cache_fp8;
  const int32_t* positions;
  int s_max, d_c;
  double turns[kDr / 2];
  int32_t* status;
};

__device__ __forceinline__ bool ws_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
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

__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

__device__ __forceinline__ float comp(const float4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Relaxed arrival: the only thing published through this barrier is the
// barrier set-up, which thread 0 releases with fence.mbarrier_init first (a
// releasing arrive would also wait for the thread's copies in flight).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Bounded wait for a phase completed by bulk copies from other CTAs of the cluster.
__device__ __forceinline__ bool ws_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

template <bool kXf32, int kMode>
__global__ void __launch_bounds__(kWsThreads, 1)
    wstream_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
                   const WsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int n0 = 128 * blockIdx.y, z = blockIdx.z;
  const int nbt = p.K / kWsBox;
  const int kb0 = rank * nbt / p.ks, nb = (rank + 1) * nbt / p.ks - kb0;   // nb >= 1
  // Weight tiles start their K range at different boxes, so that the CTAs of
  // one K split do not all read the same x box at the same time.
  const int rot = static_cast<int>((static_cast<long long>(blockIdx.y) * nb) / gridDim.y);
  auto kbox = [&](int i) { return kb0 + (i + rot) % nb; };
  const int S = p.stages;
  const int R = 128 / p.ks, rs = p.Bc + 4;   // rows owned by each CTA; row stride (floats)
  const uint32_t bars = sbase + p.bar_off;
  auto full = [&](int s) { return bars + 8 * s; };
  auto empty = [&](int s) { return bars + 8 * (S + s); };
  auto conv = [&](int s) { return bars + 8 * (2 * S + s); };
  const uint32_t acc_bar = bars + 8 * (3 * S);
  const uint32_t recv_bar = bars + 8 * (3 * S + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.bar_off + 8 * (3 * S + 2));
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (3 * S + 3));
  int* pos_s = reinterpret_cast<int*>(smem + p.pos_off);
  const uint32_t xbytes = static_cast<uint32_t>(p.Bc) * (kXf32 ? 256u : 128u);
  const uint32_t xoff = kXf32 ? p.raw_off : p.ops_off;

  // The weight stream starts before anything else: thread 0 sets up the
  // barriers and issues the first fills before the CTA-wide barrier.
  const uint64_t pol_w = l2_evict_first_policy();   // read once
  const uint64_t pol_x = l2_evict_last_policy();    // read by every weight tile's CTAs
  auto issue = [&](int i) {
    const int s = i % S;
    const uint32_t st = sbase + s * p.stage_bytes;
    mbar_arrive_expect_tx(full(s), kWsWBytes + xbytes);
    tma_load_2d(st, &tw, kWsBox * kbox(i), n0, full(s), pol_w);
    tma_load_2d(st + xoff, &tx, kWsBox * kbox(i), z * p.Bc, full(s), pol_x);
  };
  constexpr int kEarly = 4;   // boxes issued before the CTA-wide barrier
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(conv(s), 128);
    }
    mbar_init(acc_bar, 2);   // one commit per issuer
    mbar_init(recv_bar, 1);
    *abort_flag = 0;
    // The other CTAs' slices of this CTA's rows complete one phase.
    if (p.ks > 1) mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(p.ks - 1) * p.slice_bytes);
    else mbar_arrive(recv_bar);
    fence_mbarrier_init();
    prefetch_tmap(&tw);
    prefetch_tmap(&tx);
    for (int i = 0; i < kEarly && i < S && i < nb; ++i) issue(i);
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(slot), p.tmem_cols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive_relaxed();   // every thread, after the CTA barrier
  const uint32_t tmem = *slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = S < nb ? S : nb;
      for (int i = kEarly; i < S && i < nb; ++i) issue(i);
      for (int i = S; i < nb; ++i) {
        if (!ws_wait(empty(i % S), ((i / S) - 1) & 1, abort_flag)) break;
        issue(i);
        issued = i + 1;
      }
      // Copies still in flight land before the CTA may leave (bounded waits).
      const int from = issued > S ? issued - S : 0;
      for (int i = from; i < issued; ++i) {
        if (mbar_try_wait(full(i % S), (i / S) & 1)) continue;
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(full(i % S), (i / S) & 1))
          if (globaltimer_ns() - t0 > kWaitNs) {
            *abort_flag = 1;
            break;
          }
      }
    }
  } else if (warp <= 2) {
    if (lane == 0) {
      const int e = warp - 1;
      const uint32_t idesc = umma_idesc_bf16(128, p.Nc, 0, 0);
      const uint32_t d = tmem + static_cast<uint32_t>(e * p.Nc);
      bool first = true;
      for (int i = e; i < nb; i += 2) {
        const int s = i % S;
        if (!ws_wait(full(s), (i / S) & 1, abort_flag)) break;
        if (kXf32 && !ws_wait(conv(s), (i / S) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t st = sbase + s * p.stage_bytes;
        const uint64_t a = umma_desc_sw128(st, 16, 1024);
        const uint64_t b = umma_desc_sw128(st + p.ops_off, 16, 1024);
#pragma unroll
        for (int k = 0; k < kWsBox / 16; ++k)   // a K step of 16 bf16 moves the start by 32 B
          umma_bf16(d, a + 2 * k, b + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
        umma_commit(empty(s));
        first = false;
      }
      umma_commit(acc_bar);
    }
  } else {
    const int et = tid - 96;
    if constexpr (kXf32) {
      // The B operand of box i: hi rows 0..Bc-1, lo rows Bc..2Bc-1, 128-byte
      // swizzle, split from the fp32 box staged in the same stage.
      const int units = p.Bc * 8;
      for (int i = 0; i < nb; ++i) {
        const int s = i % S;
        if (!ws_wait(full(s), (i / S) & 1, abort_flag)) break;
        uint8_t* st = smem + s * p.stage_bytes;
        const float* raw = reinterpret_cast<const float*>(st + p.raw_off);
        uint8_t* ops = st + p.ops_off;
        for (int u = et; u < units; u += 128) {
          const int row = u >> 3, c = u & 7;
          const float4 v0 = *reinterpret_cast<const float4*>(raw + row * kWsBox + 8 * c);
          const float4 v1 = *reinterpret_cast<const float4*>(raw + row * kWsBox + 8 * c + 4);
          uint4 hi, lo;
          split_bf16(v0.x, v0.y, hi.x, lo.x);
          split_bf16(v0.z, v0.w, hi.y, lo.y);
          split_bf16(v1.x, v1.y, hi.z, lo.z);
          split_bf16(v1.z, v1.w, hi.w, lo.w);
          *reinterpret_cast<uint4*>(ops + sw128(row, c)) = hi;
          *reinterpret_cast<uint4*>(ops + sw128(p.Bc + row, c)) = lo;
        }
        fence_proxy_async_smem();
        mbar_arrive(conv(s));
      }
    }
    if (kMode == kWsAppendRow) {
      for (int c = et; c < p.Bc; c += 128) {
        const int b = z * p.Bc + c;
        pos_s[c] = b < p.B ? p.positions[b] : 0;
      }
    }
    // Epilogue, part 1: this thread's TMEM lane (weight row) -> shared memory,
    // both accumulators (and hi + lo) summed.  The ring is free once every MMA
    // has completed.
    ws_wait(acc_bar, 0, abort_flag);
    __syncwarp();
    tc_fence_after();
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_addr = tmem + ((32u * static_cast<uint32_t>(warp & 3)) << 16);
    float* red = reinterpret_cast<float*>(smem);
    const bool two = nb >= 2;
    for (int cb = 0; cb < p.Bc; cb += 8) {
      uint32_t h0[8], h1[8], l0[8], l1[8];
      tmem_ld8_nowait(lane_addr + cb, h0);
      if (two) tmem_ld8_nowait(lane_addr + p.Nc + cb, h1);
      if constexpr (kXf32) {
        tmem_ld8_nowait(lane_addr + p.Bc + cb, l0);
        if (two) tmem_ld8_nowait(lane_addr + p.Nc + p.Bc + cb, l1);
      }
      tmem_wait_ld();
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float hsum = __uint_as_float(h0[j]) + (two ? __uint_as_float(h1[j]) : 0.f);
        if constexpr (kXf32)
          hsum += __uint_as_float(l0[j]) + (two ? __uint_as_float(l1[j]) : 0.f);
        v[j] = hsum;
      }
      *reinterpret_cast<float4*>(red + row * rs + cb) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(red + row * rs + cb + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
    tc_fence_before();
    fence_proxy_async_smem();   // the bulk copies read these rows
    named_bar_sync(1, 128);
    cluster_wait();             // every CTA of the cluster has its barriers set up
    // Rows [q R, (q + 1) R) go to CTA q; CTA q keeps them in its slot for this rank.
    if (et < p.ks && et != rank) {
      const int slot_q = rank < et ? rank : rank - 1;
      bulk_s2peer(mapa_shared(sbase + p.recv_off + slot_q * p.slice_bytes, et),
                  sbase + static_cast<uint32_t>(et * R * rs * 4), p.slice_bytes,
                  mapa_shared(recv_bar, et));
    }
    // Epilogue, part 2: this CTA's rows, the cluster's slices added in rank order.
    ws_wait_cluster(recv_bar, 0, abort_flag);
    const float* recv = reinterpret_cast<const float*>(smem + p.recv_off);
    const int c4n = p.Bc / 4;
    auto sum4 = [&](int lr, int c4) {   // lr: row within this CTA's R rows
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < p.ks; ++q) {
        const float* src = q == rank ? red + (rank * R + lr) * rs
                                     : recv + (q < rank ? q : q - 1) * (R * rs) + lr * rs;
        add4(acc, *reinterpret_cast<const float4*>(src + 4 * c4));
      }
      return acc;
    };
    if constexpr (kMode == kWsWriteY) {
      for (int idx = et; idx < R * c4n; idx += 128) {
        const int lr = idx % R, c4 = idx / R;
        const float4 acc = sum4(lr, c4);
        const int n = n0 + rank * R + lr;
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int b = z * p.Bc + 4 * c4 + j;
            if (b < p.B) p.y[size_t(b) * p.N + n] = comp(acc, j);
          }
        }
      }
    } else {
      const int R2 = R / 2;
      for (int idx = et; idx < R2 * c4n; idx += 128) {
        const int lr = 2 * (idx % R2), c4 = idx / R2;
        const float4 a0 = sum4(lr, c4), a1 = sum4(lr + 1, c4);
        const int n = n0 + rank * R + lr;   // even: (n, n + 1) is one RoPE pair
        if (n >= p.N) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * c4 + j, b = z * p.Bc + c;
          if (b >= p.B) continue;
          const int pos = pos_s[c];
          if (pos < 0 || pos >= p.s_max) {
            if (n == 0) report(p.status, MLA_DEV_LENGTH_OUT_OF_RANGE);
            continue;
          }
          float v0 = comp(a0, j), v1 = comp(a1, j);
          if (n >= p.d_c) {
            // RoPE on the key part: the pair as one complex number rotated by
            // pos * theta_i, reduced mod 2 pi in fp64.
            float sn, cs;
            sincosf(rope_angle(pos, p.turns[(n - p.d_c) / 2]), &sn, &cs);
            const float x0 = v0, x1 = v1;
            v0 = cs * x0 - sn * x1;
            v1 = sn * x0 + cs * x1;
          }
          const size_t at = (size_t(b) * p.s_max + pos) * p.N + n;
          if (p.cache_fp8)   // E4M3, round to nearest even, saturating at +-448
            *reinterpret_cast<__nv_fp8x2_storage_t*>(static_cast<uint8_t*>(p.cache) + at) =
                __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
          else
            *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.cache) + at) =
                __floats2bfloat162_rn(v0, v1);
        }
      }
    }
    if (et < p.ks && et != rank) bulk_wait_read();   // the send buffer is read before leaving
  }
  if (warp < 3) cluster_wait();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
  if (tid == 0 && *abort_flag) report(p.status, MLA_DEV_PIPELINE_TIMEOUT);
}

// Shared-memory layout for a cluster size: the ring (as many even stages as
// fit, at most kWsMaxStages), the receive slices, the chunk's positions, the
// barriers.  False if nothing fits.
bool plan_layout(WsParams& p, int ks, bool x_f32, size_t* smem) {
  p.ks = ks;
  p.ops_off = kWsWBytes;
  p.raw_off = kWsWBytes + static_cast<uint32_t>(p.Nc) * 128u;
  p.stage_bytes = p.raw_off + (x_f32 ? static_cast<uint32_t>(p.Bc) * 256u : 0u);
  p.slice_bytes = static_cast<uint32_t>(128 / ks) * static_cast<uint32_t>(p.Bc + 4) * 4u;
  const size_t recv = (size_t(p.slice_bytes) * (ks - 1) + 1023) & ~size_t(1023);
  const size_t fixed = recv + 512 + kWsBarBytes + 1024;
  if (fixed >= kWsSmemMax) return false;
  int S = static_cast<int>((kWsSmemMax - fixed) / p.stage_bytes);
  if (S > kWsMaxStages) S = kWsMaxStages;
  S &= ~1;
  const size_t send = size_t(128) * (p.Bc + 4) * 4;   // the send buffer over the ring
  if (S < 2 || send > size_t(S) * p.stage_bytes) return false;
  p.stages = S;
  p.recv_off = static_cast<uint32_t>(S) * p.stage_bytes;
  p.pos_off = p.recv_off + static_cast<uint32_t>(recv);
  p.bar_off = p.pos_off + 512;
  *smem = size_t(p.bar_off) + kWsBarBytes + 1024;
  return true;
}

template <bool kXf32, int kMode>
struct Kernel {
  // Clusters of `ks` CTAs that can be resident at once with `smem` bytes each
  // (0 if that cluster size cannot be launched); cached per (ks, smem).
  static int max_clusters(int ks, size_t smem) {
    static int cache_ks[8] = {0}, cache_val[8] = {0};
    static size_t cache_smem[8] = {0};
    static std::mutex cache_mutex;   // the cache is shared by every host thread
    std::lock_guard<std::mutex> lock(cache_mutex);
    for (int i = 0; i < 8; ++i)
      if (cache_ks[i] == ks && cache_smem[i] == smem) return cache_val[i];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ks), 1, 1);
    cfg.blockDim = dim3(kWsThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, wstream_kernel<kXf32, kMode>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    for (int i = 0; i < 8; ++i)
      if (cache_ks[i] == 0) {
        cache_ks[i] = ks;
        cache_smem[i] = smem;
        cache_val[i] = n;
        break;
      }
    return n;
  }

  static mla_status launch(const CUtensorMap& tw, const CUtensorMap& tx, WsParams& p,
                           int clusters_needed, dim3 grid_yz, cudaStream_t s, const char* who) {
    auto* kern = wstream_kernel<kXf32, kMode>;
    static DeviceFlags set_up, big_clusters;   // per device: attributes set; clusters of 16 allowed
    const int dev = current_device();
    if (!set_up.test(dev)) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(kWsSmemMax)) != cudaSuccess) {
        set_error("%s: cannot reserve %zu bytes of shared memory", who, kWsSmemMax);
        return MLA_ERR_CUDA;
      }
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
          cudaSuccess)
        big_clusters.set(dev);
      cudaGetLastError();
      set_up.set(dev);
    }
    const int attr_state = big_clusters.test(dev) ? 2 : 1;
    // K splits: the largest cluster size whose clusters are all resident at
    // once, at least two K boxes per CTA where K allows.
    const int nbt = p.K / kWsBox;
    size_t smem = 0;
    int ks = 0;
    for (int cand = attr_state == 2 ? 16 : 8; cand >= 1; cand /= 2) {
      if (cand > 1 && 2 * cand > nbt) continue;
      WsParams q = p;
      size_t sm = 0;
      if (!plan_layout(q, cand, kXf32, &sm)) continue;
      if (cand == 1 || max_clusters(cand, sm) >= clusters_needed) {
        p = q;
        smem = sm;
        ks = cand;
        break;
      }
    }
    if (ks == 0) {
      set_error("%s: no shared-memory layout for batch chunk %d", who, p.Bc);
      return MLA_ERR_UNSUPPORTED;
    }
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * p.Nc)) cols <<= 1;
    p.tmem_cols = cols;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ks), grid_yz.y, grid_yz.z);
    cfg.blockDim = dim3(kWsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tw, tx, p);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_error("%s: launch failed: %s", who, cudaGetErrorString(e));
      return MLA_ERR_CUDA;
    }
    return launch_status(who);
  }
};

}  // namespace

mla_status wstream_launch(const WStreamJob& j, cudaStream_t stream, const char* who) {
  if (j.K <= 0 || j.K % kWsBox != 0 || j.N <= 0 || j.B <= 0) {
    set_error("%s: projection sizes B=%d K=%d N=%d (K a multiple of %d)", who, j.B, j.K, j.N,
              kWsBox);
    return MLA_ERR_UNSUPPORTED;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) {
    set_error("%s: cuTensorMapEncodeTiled is not available from the driver", who);
    return MLA_ERR_CUDA;
  }
  WsParams p{};
  p.B = j.B;
  p.K = j.K;
  p.N = j.N;
  // Batch chunks of at most 128 bf16 rows (64 fp32 rows, which become 128 hi | lo
  // rows), balanced and rounded up to the MMA's granule of 16.
  const int max_rows = j.x_f32 ? 64 : 128;
  const int chunks = (j.B + max_rows - 1) / max_rows;
  p.Bc = ((j.B + chunks - 1) / chunks + 15) / 16 * 16;
  p.Nc = j.x_f32 ? 2 * p.Bc : p.Bc;
  const int mtiles = (j.N + 127) / 128;
  p.y = j.y;
  p.cache = j.cache;
  p.cache_fp8 = j.cache_fp8 ? 1 : 0;
  p.positions = j.positions;
  p.s_max = j.s_max;
  p.d_c = j.d_c;
  for (int i = 0; i < kDr / 2; ++i) p.turns[i] = j.turns[i];
  p.status = j.status;

  // Tensor maps: the weight [N rows, K] in 128-row x 64-column boxes; x [B rows,
  // K] in Bc-row x 64-column boxes, bf16 with the 128-byte swizzle of the MMA
  // operands, fp32 unswizzled for the hi | lo split.  Rows past N or B read as
  // zero.
  CUtensorMap tw, tx;
  const cuuint32_t estride[2] = {1, 1};
  {
    const cuuint64_t gdim[2] = {cuuint64_t(j.K), cuuint64_t(j.N)};
    const cuuint64_t gstride[1] = {cuuint64_t(j.K) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kWsBox), 128};
    CUresult r = enc(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(j.w), gdim,
                     gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      set_error("%s: cuTensorMapEncodeTiled failed for the weight (%d)", who, int(r));
      return MLA_ERR_CUDA;
    }
  }
  {
    const size_t esz = j.x_f32 ? 4 : 2;
    const cuuint64_t gdim[2] = {cuuint64_t(j.K), cuuint64_t(j.B)};
    const cuuint64_t gstride[1] = {cuuint64_t(j.K) * esz};
    const cuuint32_t box[2] = {cuuint32_t(kWsBox), cuuint32_t(p.Bc)};
    CUresult r = enc(&tx, j.x_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     2, const_cast<void*>(j.x), gdim, gstride, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     j.x_f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      set_error("%s: cuTensorMapEncodeTiled failed for x (%d)", who, int(r));
      return MLA_ERR_CUDA;
    }
  }
  const int clusters = mtiles * chunks;
  const dim3 yz(1, static_cast<unsigned>(mtiles), static_cast<unsigned>(chunks));
  if (j.mode == kWsWriteY)
    return j.x_f32 ? Kernel<true, kWsWriteY>::launch(tw, tx, p, clusters, yz, stream, who)
                   : Kernel<false, kWsWriteY>::launch(tw, tx, p, clusters, yz, stream, who);
  return j.x_f32 ? Kernel<true, kWsAppendRow>::launch(tw, tx, p, clusters, yz, stream, who)
                 : Kernel<false, kWsAppendRow>::launch(tw, tx, p, clusters, yz, stream, who);
}

}  // namespace mla
