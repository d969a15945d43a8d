// mla_decode_attn: split-KV attention of the absorbed query over the latent
// cache, plus the log-sum-exp combine of the chunks.
//
// Multi-Head Latent Attention (Lior Sinai), 3.3 and 3.6: per head h the score
// of cached row t is (q_abs_h . c_t + q_pe_h . k_rope_t) / sqrt(d_h + d_R), one
// latent row serves every head (virtual broadcast of C^KV across heads), and
// the attention output stays in the d_c-wide latent space.
//
// bf16: a tcgen05 kernel (see split_tc_kernel); each chunk of rows yields a
// normalised partial output and its log-sum-exp.
// fp32: plain SIMT, fp32 arithmetic throughout (no TF32).
// combine: L = log sum_j exp(lse_j), o_c = sum_j exp(lse_j - L) o_j.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "mla_common.cuh"
#include "mla_split.cuh"

namespace mla {
namespace {

// The checked build (compiled with -DMLA_CHECK): before an access whose index
// it can compute, a kernel of this file tests that the index lies inside its
// buffer; a failed test skips the access and ORs MLA_DEV_BOUNDS into the call's
// status word (when it has one) and into g_bounds_word, which
// mla_debug_bounds_word exposes.  In the default build the tests compile away.
__device__ int32_t g_bounds_word;
__device__ __forceinline__ bool bounds_ok(bool in_range, int32_t* status) {
#ifdef MLA_CHECK
  if (!in_range) {
    atomicOr(&g_bounds_word, MLA_DEV_BOUNDS);
    if (status) atomicOr(status, MLA_DEV_BOUNDS);
  }
  return in_range;
#else
  (void)status;
  (void)in_range;
  return true;
#endif
}
#define MLA_IN_BOUNDS(cond) bounds_ok((cond), p.status)

constexpr int kWarps = 4;
constexpr int kChunkAlign = 8;   // chunk sizes are multiples of 8 rows
constexpr int kThreads = kWarps * 32;

// ---------------------------------------------------------------------------- bf16 split kernel
// One CTA per (head group of 16 or 32, KV chunk, sequence).  Every tcgen05.mma covers
// 128 cache rows (a K=16 step costs the same for M=64 as for M=128 at N=32, so
// 128-row tiles halve the tensor time per row), but a 128-row tile (147 KB)
// cannot stay resident from its scores to its PV product.  The cache
// therefore streams twice per tile, from two decoupled rings:
//   ring A  score boxes (128 rows x 64 columns, 16 KB) from HBM; a slot is
//           free again as soon as its four score MMAs finish
//   ring B  pairs of latent boxes (64 rows x 128 columns, 16 KB) for the PV
//           product, re-read from L2 (the score pass loads with evict_last);
//           a tile's pairs are requested once its score MMAs are issued, so
//           they land about when its P does instead of holding slots early
// L2 serves the GPU's SMs at close to three times the HBM rate, so the
// second read costs L2 bandwidth, not HBM time.
constexpr int kBoxBytes = kTileRows * 128;            // 128 rows x 64 bf16 columns
constexpr int kHalfBox = kBoxBytes / 2;               // 64 rows x 64 bf16 columns
// Rescale threshold (log2 units): P may grow to 2^8 before O is rescaled.
constexpr float kRescaleLog2 = 8.f;

// One work item of a split CTA: one chunk of one query group's rows for one
// head group.  A CTA of an ordinary grid has one item (its blockIdx); a
// persistent CTA has the items plan_items gives it, streamed back to back.
struct SplitItem {
  int row0;        // cache row (of the [B*s_max, 576] view) of the item's first row
  int tiles;       // 128-row tiles
  int t0;          // index of its first tile in the CTA's tile stream
  int valid_last;  // rows of its last tile that belong to the item
  int zero_from;   // rows of its last tile before the sequence's end; from there on
                   // (< 128) rows may hold anything and are zeroed before the PV
  int part;        // partial row of its first head: (v * H + h0) * splits + j
  int qv;          // query group (row block of q_abs and q_pe)
  int h0;          // first head
};
// Items a persistent CTA can hold (the planner keeps within it).
constexpr int kMaxItems = 128;
// Test hook (mla_test_set_split_form): 0 the planner chooses the split's form,
// 1 persistent wherever the kernel allows it, 2 never persistent.
std::atomic<int> g_split_form{0};
// mla_set_split_parts: 0 the library's choice (one bf16 part of the query and P
// with 64 heads per CTA where the head count is a multiple of 64), 2 always
// hi + lo parts.
std::atomic<int> g_split_parts{0};

// The kernel's plan for kG heads per CTA.  With 16 or 32 heads the query and P
// enter the tensor core as bf16 hi and lo parts (N = 2 kG query rows); with 64
// as one bf16 part each (N = 64: bf16 operands, fp32 accumulation), which
// halves the CTAs that read each row at 128 heads.  N = 64 halves, per head,
// the MMAs and the tile reads (shared memory and L2) against N = 32; its query
// and accumulators need more room, so ring A has four slots, P one buffer and
// O^T one buffer.  kPersist: the persistent instance (16 heads per CTA) holds a
// table of work items and double-buffers O^T in tensor memory, so that a CTA's
// next item accumulates while the previous one's epilogue reads its result;
// the ordinary instance has one item and none of that code.
template <int kG, bool kPersist = false>
struct TcPlan {
  static constexpr int kParts = kG == 64 ? 1 : 2;      // bf16 parts of the query and of P
  static constexpr int kQN = kParts * kG;              // query rows: [hi | lo] or the heads
  static constexpr int kGroupHeads = 16 / kParts;      // heads per softmax group of four warps
  static constexpr int kSoftWarps = kQN / 4;
  static constexpr int kSoftThreads = 32 * kSoftWarps;
  static constexpr int kThreads = kSoftThreads + 6 * 32;   // + ring A, ring B, 2 score, 2 PV
  static constexpr int kSlotsA = kG == 16 ? 6 : 4;
  static constexpr int kSlotsB = 4;                    // each slot: two adjacent 64-row boxes
  static constexpr int kPBufs = kG == 16 ? 2 : 1;
  static constexpr int kOBufs = kPersist ? 2 : 1;      // O^T accumulators in tensor memory
  static constexpr int kItems = kPersist ? kMaxItems : 1;
  static constexpr int kQBoxBytes = kQN * 128;
  static constexpr int kPSub = kQN * 128;              // P^T: 64 tile rows of kQN rows
  static constexpr int kPBytes = 2 * kPSub;            // 128 tile rows
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kSlotsA * kBoxBytes;
  static constexpr int kOffQ = kOffB + kSlotsB * 2 * kHalfBox;
  static constexpr int kOffP = kOffQ + 9 * kQBoxBytes;
  static constexpr int kOffRed = kOffP + kPBufs * kPBytes;   // [2][kG heads][4 warps] tile maxima
  static constexpr int kOffLsum = kOffRed + 2 * kG * 4 * 4;
  static constexpr int kOffItems = kOffLsum + kG * 4 * 4;
  static constexpr int kOffBar =
      (kOffItems + kItems * static_cast<int>(sizeof(SplitItem)) + 127) / 128 * 128;
  static constexpr int BAR_FULLA = 0, BAR_EMPTYA = kSlotsA, BAR_FULLB = 2 * kSlotsA,
                       BAR_EMPTYB = BAR_FULLB + kSlotsB, BAR_ZEROB = BAR_EMPTYB + kSlotsB,
                       BAR_SFULL = BAR_ZEROB + kSlotsB, BAR_SFREE = BAR_SFULL + 2,
                       BAR_PFULL = BAR_SFREE + 2, BAR_PFULL1 = BAR_PFULL + 2,
                       BAR_P0FREE = BAR_PFULL1 + 2, BAR_ODONE = BAR_P0FREE + 2,
                       BAR_LASTA = BAR_ODONE + 2, BAR_FULLX = BAR_LASTA + 1,
                       BAR_ZEROX = BAR_FULLX + 8, BAR_ODONE2 = BAR_ZEROX + 8,
                       BAR_PVPREV = BAR_ODONE2 + 1, BAR_DONE = BAR_PVPREV + 1,
                       BAR_QFREE = BAR_DONE + 1, BAR_QREADY = BAR_QFREE + 1,
                       BAR_ODRAIN = BAR_QREADY + 1, kNumBars = BAR_ODRAIN + 2;
  static constexpr int kOffSlot = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffSlot + 16;
  static constexpr int kOffIssued = kOffAbort + 16;   // score tiles issued, per score issuer
  static constexpr int kOffCount = kOffIssued + 16;   // [items, tiles] of this CTA
  static constexpr size_t kSmem = 1024 + kOffCount + 16;
  // TMEM: S_0[2] at 0 / kQN, S_1[2] at kS1Col / kS1Col + kQN, O^T blocks of kQN
  // columns from kOCol (buffer x at kOCol + x kOBufCols).
  static constexpr uint32_t kS1Col = 2 * kQN;
  static constexpr uint32_t kOCol = 4 * kQN;
  static constexpr uint32_t kOBufCols = 4 * kQN;
  static constexpr uint32_t kTmemCols = kG == 16 && !kPersist ? 256 : 512;
  static_assert(kOCol + kOBufs * kOBufCols <= kTmemCols, "tensor memory plan");
  static_assert(kOffBar % 8 == 0 && kOffItems % 4 == 0 && kOffRed % 16 == 0 &&
                    kOffLsum % 16 == 0 && kOffSlot % 16 == 0 && kOffAbort % 4 == 0,
                "mbarriers need 8-byte alignment, the float4 reads of the maxima 16");
  static_assert(kSmem <= 232448, "shared memory plan exceeds 227 KB");
  static_assert(kSlotsA * kBoxBytes + 9 * kQBoxBytes >= 8 * kBoxBytes,
                "the last tile's eight latent pairs fit in ring A and the query area");
  static_assert(kSlotsA % 2 == 0, "each score issuer owns every other ring-A slot");
};

// Waits for a phase; gives up (and raises the CTA's abort flag) after limit_ns,
// or at once when another role has already raised it.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort,
                                              unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      // The words after the flag keep where the CTA's first wait gave up (the
      // barrier's address, its parity and the waiting thread), for a test hook.
      abort[1] = static_cast<int>(bar);
      abort[2] = static_cast<int>(parity | (threadIdx.x << 8));
      *abort = 1;
      return false;
    }
  }
}

// After an abort: waits (bounded) until the copy armed on `bar` for the phase
// with this parity has landed, so that no copy into shared memory is still in
// flight when the CTA leaves.  A phase that completed before returns at once.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity,
                                            unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return;
}

// Exclusive prefix sum of x over the warp's lanes, and the warp's total.
__device__ __forceinline__ int warp_exclusive_scan(int x, int lane, int* total) {
  int incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - x;
}

// Persistent grid: the items of CTA c of G, computed by one whole warp.  Every
// (head group, query group, chunk) with rows is an item; items are ordered by
// head group, then query group, then chunk, which numbers every tile of every
// item consecutively (TT tiles in all).  CTA c takes the items whose first tile
// falls in [c TT / G', (c + 1) TT / G'): an equal share of the tiles, give or
// take one chunk, and mostly consecutive chunks of one sequence (one query
// load).  G' = G, except when every chunk is whole (NI = TT / tiles per chunk
// items of equal size): then G' = ceil(NI / k), k = ceil(NI / G), the fewest
// CTAs that still give the busiest one k chunks, so that the shares are equal
// and fewer CTAs share HBM while they stream (measured on 4 x 65536 rows at 128
// chunks: 128 CTAs of four chunks, split 61.5 us against 65.0 with 152 CTAs of
// three or four); CTAs from G' on take nothing.
// Chunks are whole tiles here (chunk % 128 == 0), so a tile never straddles two
// items.  Writes items[0..n) with their first tile in the CTA's stream and
// counts[0] = n, counts[1] = tiles; n > kMaxItems (never planned) raises
// MLA_DEV_PIPELINE_TIMEOUT and keeps the first kMaxItems.
__device__ void plan_items(const SplitParams& p, SplitItem* items, volatile int* counts,
                           int lane) {
  const int groups = p.H / 16, ct = p.chunk / kTileRows;
  const long long G = gridDim.x, c = blockIdx.x;
  // Lengths of the first 32 query groups, one load per lane, kept for both passes.
  const int len_lane = lane < p.B ? clamp_length(p, lane, c == 0) : 0;
  auto length_of = [&](int v0, bool report_it) {
    const int v = v0 + lane;
    return v0 == 0 ? len_lane : v < p.B ? clamp_length(p, v, report_it) : 0;
  };
  // Non-negative quotients; 32-bit division when both operands fit (the
  // planner's tile counts always do in practice; 64-bit division is a long
  // subroutine on the CTA's start-up path).
  auto quot = [](long long a, long long b) {
    return a <= 0x7fffffffll && b <= 0x7fffffffll
               ? static_cast<long long>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b))
               : a / b;
  };
  // Tiles of one head group: the sum over query groups of ceil(len / 128).
  long long tg = 0;
  bool whole = true;   // every chunk of every query group whole
  for (int v0 = 0; v0 < p.B; v0 += 32) {
    const int len = length_of(v0, c == 0);
    const int tiles = (len + kTileRows - 1) / kTileRows;
    int tot;
    warp_exclusive_scan(tiles, lane, &tot);
    tg += tot;
    whole = __all_sync(0xffffffffu, tiles % ct == 0) && whole;
  }
  const long long TT = groups * tg;
  long long Ge = G;   // CTAs with work
  if (whole && TT > 0) {
    const long long NI = TT / ct, k = quot(NI + G - 1, G);
    Ge = quot(NI + k - 1, k);
  }
  const long long lo = c < Ge ? quot(c * TT, Ge) : TT, hi = c < Ge ? quot((c + 1) * TT, Ge) : TT;
  int n = 0;
  long long base = 0;   // first tile of the current block of query groups
  for (int g = 0; g < groups && base < hi; ++g) {
    for (int v0 = 0; v0 < p.B && base < hi; v0 += 32) {
      const int v = v0 + lane;
      const int len = length_of(v0, false);
      const int tiles = (len + kTileRows - 1) / kTileRows;
      int tot;
      const long long s = base + warp_exclusive_scan(tiles, lane, &tot);   // its first tile
      // chunks j of this query group whose first tile s + j ct is in [lo, hi)
      const int nch = (tiles + ct - 1) / ct;
      long long jlo = lo > s ? quot(lo - s + ct - 1, ct) : 0;
      long long jhi = hi > s ? quot(hi - s + ct - 1, ct) : 0;
      jlo = jlo < nch ? jlo : nch;
      jhi = jhi < nch ? jhi : nch;
      const int cnt = jhi > jlo ? static_cast<int>(jhi - jlo) : 0;
      int ctot;
      int pos = n + warp_exclusive_scan(cnt, lane, &ctot);
      for (long long jj = jlo; jj < jhi; ++jj, ++pos) {
        if (pos >= kMaxItems) break;
        const int j = static_cast<int>(jj);
        const int r0 = j * p.chunk, r1 = min(r0 + p.chunk, len);
        const int it = (r1 - r0 + kTileRows - 1) / kTileRows;
        SplitItem m;
        m.row0 = cache_seq(p, v) * p.s_max + r0;
        m.tiles = it;
        m.t0 = 0;
        m.valid_last = r1 - (r0 + (it - 1) * kTileRows);
        m.zero_from = len - (r0 + (it - 1) * kTileRows);
        m.part = (v * p.H + 16 * g) * p.splits + j;
        m.qv = v;
        m.h0 = 16 * g;
        items[pos] = m;
      }
      n += ctot;
      base += tot;
    }
  }
  __syncwarp();
  if (lane == 0) {
    if (n > kMaxItems) {
      report(p.status, MLA_DEV_PIPELINE_TIMEOUT);
      n = kMaxItems;
    }
    int t = 0;
    for (int i = 0; i < n; ++i) {
      items[i].t0 = t;
      t += items[i].tiles;
    }
    counts[0] = n;
    counts[1] = t;
  }
  __syncwarp();
}

// Per-head max (or sum) of v[0..7] over the 32 lanes of a warp: one exchange
// across the half-warps, a butterfly that halves the values held per lane
// each round, and a last pairwise exchange; afterwards lane l holds head
// (l >> 1) & 7.
template <bool kMax>
__device__ __forceinline__ float reduce8_heads(float v[8], int lane) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float o = __shfl_xor_sync(0xffffffffu, v[k], 16);
    v[k] = kMax ? fmaxf(v[k], o) : v[k] + o;
  }
#pragma unroll
  for (int half = 4, bit = 8; half >= 1; half >>= 1, bit >>= 1) {
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = upper ? v[k] : v[k + half];
      const float keep = upper ? v[k + half] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, bit);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  const float o = __shfl_xor_sync(0xffffffffu, v[0], 1);
  return kMax ? fmaxf(v[0], o) : v[0] + o;
}

// Roles, for kG heads per CTA (16: 448 threads; 32: 704), with W = kG / 2
// softmax warps and N = 2 kG:
//   warp W    : TMEM allocation; one lane runs ring A (9 score boxes per tile)
//   warp W+2  : one lane runs ring B (8 latent box pairs per tile: four
//               128-column blocks x two 64-row halves)
//   warps W+1, W+3: score MMAs, each over alternate boxes of the stream, into
//               two accumulators S_0, S_1 (summed by the softmax):
//               S[128 x N] = C[128 x 576] . Q^T  (M=128, N: the heads' hi and
//               lo query parts; S double-buffered in TMEM)
//   warps W+4, W+5: PV MMAs, each over two of the four O^T blocks:
//               O^T[512 x N] += C^T[512 x 128] . P^T[128 x N]  (M=128 blocks,
//               each in two 64-row halves; C read MN-major from a ring-B pair)
//             A thread issues one tcgen05.mma per ~100 cycles whatever the
//             shape (N = 32 or 64), so four issuing threads keep the tensor
//             pipe fed.
//   warps 0..W-1: one tile row per thread, a group of four warps per 8 heads
//             (heads 8i..8i+7 in warps 4i..4i+3): softmax across the rows, P^T
//             (hi | lo bf16) to shared memory; O^T accumulates in TMEM against a
//             reference maximum per head that moves only when a tile's maximum
//             exceeds it by 2^8 (then O^T is rescaled in TMEM).
// The fp32 query and P reach the tensor core as bf16 hi + lo pairs, so their
// rounding stays near 2^-17 relative.
//
// The CTA works through its items (SplitItem) as one stream of T tiles: the
// rings and MMA issuers run across item boundaries without a pause.  At the end
// of an item the softmax warps write its partial one tile later (its O^T buffer
// is done by then, and the next item accumulates into the other buffer), and
// when the next item belongs to another query group or head group they load
// that query into the query area once the score MMAs of the item are done (the
// score issuers wait for it).  Only the CTA's last tile takes the special tail
// path (its boxes read in place from ring A).
template <int kG, bool kPersist>
__global__ void __launch_bounds__(TcPlan<kG, kPersist>::kThreads, 1)
    split_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_half,
                    const SplitParams p) {
  // The plan's sizes under the names the body uses (kHeadGroup: heads per CTA).
  using L = TcPlan<kG, kPersist>;
  static_assert(!kPersist || kG == 16, "the persistent instance takes 16 heads per CTA");
  constexpr int kHeadGroup = kG, kGroupHeads = L::kGroupHeads, kSoftWarps = L::kSoftWarps;
  constexpr int kParts = L::kParts;
  // One P buffer: the softmax writes each 64-row half of P as soon as the
  // previous tile's PV is done with that half.
  constexpr bool kHalfP = L::kPBufs == 1;
  constexpr int kSoftThreads = L::kSoftThreads, kSlotsA = L::kSlotsA, kSlotsB = L::kSlotsB;
  constexpr int kPBufs = L::kPBufs, kQN = L::kQN, kQBoxBytes = L::kQBoxBytes, kPSub = L::kPSub;
  constexpr int kPBytes = L::kPBytes, kOffA = L::kOffA, kOffB = L::kOffB, kOffQ = L::kOffQ;
  constexpr int kOffP = L::kOffP, kOffRed = L::kOffRed, kOffLsum = L::kOffLsum;
  constexpr int kOffBar = L::kOffBar, kOffSlot = L::kOffSlot, kOffAbort = L::kOffAbort;
  constexpr int kOffIssued = L::kOffIssued, kOffItems = L::kOffItems, kOffCount = L::kOffCount;

  constexpr uint32_t kS1Col = L::kS1Col, kOCol = L::kOCol, kTmemCols = L::kTmemCols;
  constexpr uint32_t kOBufCols = L::kOBufCols;
  constexpr int BAR_FULLA = L::BAR_FULLA, BAR_EMPTYA = L::BAR_EMPTYA, BAR_FULLB = L::BAR_FULLB,
                BAR_EMPTYB = L::BAR_EMPTYB, BAR_ZEROB = L::BAR_ZEROB, BAR_SFULL = L::BAR_SFULL,
                BAR_SFREE = L::BAR_SFREE, BAR_PFULL = L::BAR_PFULL, BAR_PFULL1 = L::BAR_PFULL1,
                BAR_P0FREE = L::BAR_P0FREE, BAR_ODONE = L::BAR_ODONE,
                BAR_LASTA = L::BAR_LASTA, BAR_FULLX = L::BAR_FULLX, BAR_ZEROX = L::BAR_ZEROX,
                BAR_ODONE2 = L::BAR_ODONE2, BAR_PVPREV = L::BAR_PVPREV, BAR_DONE = L::BAR_DONE,
                BAR_QFREE = L::BAR_QFREE, BAR_QREADY = L::BAR_QREADY, BAR_ODRAIN = L::BAR_ODRAIN;
  // Role warps after the softmax warps.
  constexpr int kWarpA = kSoftWarps, kWarpS0 = kSoftWarps + 1, kWarpB = kSoftWarps + 2,
                kWarpS1 = kSoftWarps + 3, kWarpPV0 = kSoftWarps + 4, kWarpPV1 = kSoftWarps + 5;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBar;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
  SplitItem* items = reinterpret_cast<SplitItem*>(smem + kOffItems);
  volatile int* counts = reinterpret_cast<volatile int*>(smem + kOffCount);   // [items, tiles]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  volatile int* s_issued = reinterpret_cast<volatile int*>(smem + kOffIssued);   // [2]
  uint32_t* slot_ptr = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  // Limit of every bounded wait below (a test hook may shorten it).
  const unsigned long long wait_ns = p.wait_ns ? p.wait_ns : kWaitNs;

  // With 32 columns the CTA may hold two tokens of a multi-token step (pair):
  // columns 0-15 are the 16 heads of query group b, 16-31 those of b + 1, the
  // next token of the same sequence; the tiles follow the later token's rows
  // and each 8-head softmax group masks the rows past its own token.
  const bool pair = kG == 32 && p.tpc == 2;
  constexpr bool persist = kPersist;
  // Rows of the cache's [sequences * s_max, 576] view (index checks).
  const long long cache_rows = static_cast<long long>(p.B / p.q_len) * p.s_max;
  (void)cache_rows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return bars + 8 * i; };

  // The cache stream starts before anything else: ring A's producer sets up its
  // own barriers and issues tile 0's first six boxes (stream positions 0-5 hold
  // boxes 0-5; the RoPE-first order below applies only to a last tile after
  // another) before the CTA-wide barrier.  In a one-wave grid they need only the
  // chunk's first row and go out before the sequence length is known.
  const uint64_t keep = l2_evict_last_policy();   // read again by ring B
  // Boxes [from, to) of the first fills; from == 0 also sets up ring A's barriers.
  auto first_fills = [&](int row, int from = 0, int to = -1) {
    if (to < 0) to = kSlotsA;
    if (from == 0) {
      for (int i = 0; i < kSlotsA; ++i) {
        mbar_init(bar(BAR_FULLA + i), 1);
        mbar_init(bar(BAR_EMPTYA + i), 1);
      }
      fence_mbarrier_init();
      prefetch_tmap(&tmap);
    }
    for (int pos = from; pos < to; ++pos) {
      mbar_arrive_expect_tx(bar(BAR_FULLA + pos), kBoxBytes);
      if (MLA_IN_BOUNDS(row >= 0 && row < cache_rows))
        tma_load_2d(sbase + kOffA + pos * kBoxBytes, &tmap, 64 * pos, row,
                    bar(BAR_FULLA + pos), keep);
    }
  };
  // Query rows of the score MMA's B operand (K-major, 128-byte swizzle, one box
  // of kQN rows per 64 columns): with two parts row n < kG is bf16(q) of head n
  // and row kG + n is bf16(q - bf16(q)); with one part row n is bf16(q) of head
  // n.  q_abs[v, h0..h0+kG-1, :] and q_pe[v, h0.., :] are contiguous; each
  // softmax thread loads nine float4 at a time before converting them.
  // signal: arrive on named barrier 3 once the first pass's loads are issued.
  auto load_query = [&](int v, int h0, bool signal = false) {
    const float4* qa = reinterpret_cast<const float4*>(static_cast<const float*>(p.q_abs) +
                                                       (size_t(v) * p.H + h0) * kDc);
    const float4* qp = reinterpret_cast<const float4*>(static_cast<const float*>(p.q_pe) +
                                                       (size_t(v) * p.H + h0) * kDr);
    constexpr int kNA = kHeadGroup * kDc / 4, kNQ = kNA + kHeadGroup * kDr / 4;
    static_assert(kNQ % (9 * kSoftThreads) == 0, "nine float4 per softmax thread and pass");
#pragma unroll 1
    for (int pass = 0; pass < kNQ / (9 * kSoftThreads); ++pass) {
    float4 q4[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int idx = tid + (9 * pass + i) * kSoftThreads;
      // the query row (v', h) this load belongs to, for the index check
      const int n = idx < kNA ? idx / (kDc / 4) : (idx - kNA) / (kDr / 4);
      const size_t row = pair ? size_t(v + n / 16) * p.H + h0 + n % 16 : size_t(v) * p.H + h0 + n;
      q4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!MLA_IN_BOUNDS(row < size_t(p.B) * p.H)) continue;
      if (pair) {
        // column n: head h0 + n % 16 of query group v + n / 16
        q4[i] = idx < kNA ? reinterpret_cast<const float4*>(static_cast<const float*>(p.q_abs) +
                                                            row * kDc)[idx % (kDc / 4)]
                          : reinterpret_cast<const float4*>(static_cast<const float*>(p.q_pe) +
                                                            row * kDr)[(idx - kNA) % (kDr / 4)];
      } else {
        q4[i] = idx < kNA ? qa[idx] : qp[idx - kNA];
      }
    }
    if (signal && pass == 0) named_bar_arrive(3, kSoftThreads + 32);
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int idx = tid + (9 * pass + i) * kSoftThreads;
      const int h = idx < kNA ? idx / (kDc / 4) : (idx - kNA) / (kDr / 4);
      const int k = idx < kNA ? 4 * (idx % (kDc / 4)) : kDc + 4 * ((idx - kNA) % (kDr / 4));
      uint2 hi, lo;
      split_bf16(q4[i].x, q4[i].y, hi.x, lo.x);
      split_bf16(q4[i].z, q4[i].w, hi.y, lo.y);
      const int box = k >> 6, ch = (k & 63) >> 3, w = k & 7;
      const uint32_t o_hi = box * kQBoxBytes + sw128(h, ch) + 2 * w;
      const uint32_t o_lo = box * kQBoxBytes + sw128(h + kHeadGroup, ch) + 2 * w;
      if (MLA_IN_BOUNDS(o_hi + 8 <= 9u * kQBoxBytes &&
                        (kParts == 1 || o_lo + 8 <= 9u * kQBoxBytes))) {
        *reinterpret_cast<uint2*>(smem + kOffQ + o_hi) = hi;
        if (kParts == 2) *reinterpret_cast<uint2*>(smem + kOffQ + o_lo) = lo;
      }
    }
    }
    fence_proxy_async_smem();
  };
  const bool ring_a = warp == kWarpA && lane == 0;
  int len_first = 0, len_pair = 0;   // paired tokens: rows of the earlier and later token
  int r0_one = 0;                    // one-item CTA: the chunk's first row in its sequence
  int qv0 = 0, qh0 = 0;              // query group and first head of the CTA's first item
  if (persist) {
    if (warp == kWarpA) plan_items(p, items, counts, lane);
    __syncthreads();
    if (counts[0] == 0) return;   // no tile for this CTA
    qv0 = items[0].qv;
    qh0 = items[0].h0;
    // Two boxes at once; the other first boxes once the softmax warps have
    // issued the query's loads (named barrier 3), so that those do not queue
    // behind every CTA's first-fill burst.
    if (warp == kWarpA) {
      if (lane == 0) first_fills(items[0].row0, 0, 2);
      __syncwarp();
      named_bar_sync(3, kSoftThreads + 32);
      if (lane == 0) first_fills(items[0].row0, 2, kSlotsA);
    }
  } else {
    const int g = blockIdx.x, j = blockIdx.y, b = pair ? 2 * blockIdx.z : blockIdx.z;
    const int r0 = j * p.chunk;
    r0_one = r0;
    const int row_base = cache_seq(p, b) * p.s_max + r0;
    qv0 = b;
    qh0 = g * (pair ? kHeadGroup / 2 : kHeadGroup);
    if (ring_a && p.fill_early) first_fills(row_base);
    // Launched after mla_absorb_q with programmatic serialization: everything up
    // to the query load (set-up, TMEM, the cache stream) overlaps that kernel.
    const int len = clamp_length(p, pair ? b + 1 : b, tid == 0 && g == 0 && j == 0);
    len_pair = len;
    len_first = pair ? clamp_length(p, b, tid == 0 && g == 0 && j == 0) : len;
    if (r0 >= len) {
      // Chunk past the end of this sequence: nothing to do once early copies
      // (into this CTA's shared memory) have landed.
      if (ring_a && p.fill_early)
        for (int pos = 0; pos < kSlotsA; ++pos) mbar_wait_bounded(bar(BAR_FULLA + pos), 0);
      return;
    }
    if (ring_a && !p.fill_early) first_fills(row_base);
    if (tid == 0) {
      // The last tile may reach past the chunk into the next chunk's rows (finite
      // cache data; their scores are masked) and past the sequence's end, where
      // rows may hold anything (NaN included): those are zeroed before the PV.
      const int r1 = min(r0 + p.chunk, len);
      const int nt = (r1 - r0 + kTileRows - 1) / kTileRows;
      SplitItem m;
      m.row0 = row_base;
      m.tiles = nt;
      m.t0 = 0;
      m.valid_last = r1 - (r0 + (nt - 1) * kTileRows);
      m.zero_from = len - (r0 + (nt - 1) * kTileRows);
      m.h0 = qh0;
      m.part = (b * p.H + m.h0) * p.splits + j;
      m.qv = b;
      items[0] = m;
      counts[0] = 1;
      counts[1] = nt;
    }
  }
  if (tid == 0) {
    for (int i = 0; i < kSlotsB; ++i) {
      mbar_init(bar(BAR_FULLB + i), 1);
      mbar_init(bar(BAR_EMPTYB + i), 1);
      mbar_init(bar(BAR_ZEROB + i), kSoftWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BAR_SFULL + i), 2);   // one commit per score issuer
      mbar_init(bar(BAR_SFREE + i), kSoftWarps);
      // With one P buffer, P is handed over per 64-row half: BAR_PFULL the rows
      // 0-63 (or all of P with two buffers), BAR_PFULL1 the rows 64-127, and
      // BAR_P0FREE: the previous PV has finished with rows 0-63.
      mbar_init(bar(BAR_PFULL + i), kHalfP ? kSoftWarps / 2 : kSoftWarps);
      mbar_init(bar(BAR_PFULL1 + i), kSoftWarps / 2);
      mbar_init(bar(BAR_P0FREE + i), 2);   // one commit per PV issuer
      mbar_init(bar(BAR_ODONE + i), 2);   // one commit per PV issuer
      mbar_init(bar(BAR_ODRAIN + i), kSoftWarps);   // an O^T buffer's result has been read
    }
    mbar_init(bar(BAR_LASTA), 2);         // every score MMA has finished
    for (int i = 0; i < 8; ++i) {
      mbar_init(bar(BAR_FULLX + i), 1);   // the last tile's borrowed pairs: one use each
      mbar_init(bar(BAR_ZEROX + i), kSoftWarps);
    }
    mbar_init(bar(BAR_ODONE2), 2);        // the score issuers' share of the last PV
    mbar_init(bar(BAR_PVPREV), 2);        // the PV of tile T-2 has finished
    mbar_init(bar(BAR_DONE), 4);          // every issuer's last commit
    mbar_init(bar(BAR_QFREE), 2);         // an item's score MMAs are done with the query
    mbar_init(bar(BAR_QREADY), kSoftWarps);   // the next item's query is in place
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    abort_flag[2] = 0;
    s_issued[0] = 0;
    s_issued[1] = 0;
    fence_mbarrier_init();
  }
  if (warp == kWarpA) {
    __syncwarp();
    tmem_alloc(smem_u32(slot_ptr), kTmemCols);
  }
  // The first item's query comes from the previous kernel of the stream
  // (mla_absorb_q).  A persistent CTA loads it while the other roles set up, so
  // that it is in place when the CTA-wide barrier below passes (its first boxes
  // are in flight by then); a one-item CTA loads it after that barrier, so that
  // under programmatic launch the set-up and ring B do not wait for the
  // previous kernel, and its query loads do not join the first boxes' burst.
  if (kPersist && warp < kSoftWarps) {
    pdl_wait();
    load_query(qv0, qh0, true);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;
  const int n_items = counts[0];
  const int T = counts[1];
  const SplitItem fin = items[n_items - 1];   // the item of the CTA's last tile
  const int fin_item = n_items - 1;
  const int last_row = fin.row0 + (fin.tiles - 1) * kTileRows;
  const int zero_from = fin.zero_from;
  const bool zero_last = zero_from < kTileRows;
  const bool fin_first = T - 1 == fin.t0;     // the last tile is its item's first
  // Item i accumulates into O^T buffer i % kOBufs.
  auto obuf_col = [&](int i) { return kOCol + static_cast<uint32_t>(i % L::kOBufs) * kOBufCols; };
  // Walks the items along the tile stream: item index, and its tiles' end.
  struct Cursor {
    int i, end;
  };
  constexpr bool kMulti = kPersist;   // the ordinary instance has one item per CTA
  auto seek = [&](Cursor& c, int t) {
    while (kMulti && t >= c.end) {
      ++c.i;
      c.end = items[c.i].t0 + items[c.i].tiles;
    }
  };
  auto row_of = [&](const Cursor& c, int t) {
    return items[c.i].row0 + (t - items[c.i].t0) * kTileRows;
  };
  // Whether item i (> 0) needs another query than item i - 1.
  auto new_query = [&](int i) {
    return items[i].qv != items[i - 1].qv || items[i].h0 != items[i - 1].h0;
  };
  // A tile before the last one that ends an item at its sequence's end: its
  // ring-B pairs are zeroed past the end before the PV.
  auto zero_mid = [&](const Cursor& c, int t) {
    const SplitItem& it = items[c.i];
    return kMulti && t != T - 1 && t == it.t0 + it.tiles - 1 && it.zero_from < kTileRows;
  };
  // The last tile's latent pairs.  With T >= 2 all eight go to space that is free
  // once every score MMA has finished (ring-A slots 0-5, then the query area),
  // so none waits for ring B; with T == 1 pairs 0-3 use ring B from the start
  // and pairs 4-7 go to ring-A slots 0-3.
  auto borrowed = [&](int t, int u) { return t == T - 1 && (T >= 2 || u >= 4); };
  auto borrow_x = [&](int u) { return T >= 2 ? u : u - 4; };
  auto borrow_off = [&](int x) {
    return x < kSlotsA ? kOffA + x * kBoxBytes : kOffQ + (x - kSlotsA) * kBoxBytes;
  };
  // With six ring-A slots the stream ends with the last tile's positions 3-8
  // still in ring A (positions 0-2 share slots with 6-8).  After at least one
  // other tile the last tile streams its RoPE box first, so those positions hold
  // latent boxes 2-7; a single tile keeps the order 0-8 (its first boxes were
  // issued before T was known), leaving boxes 3-7.  O^T block mb (boxes 2mb,
  // 2mb + 1) takes its PV operand from ring A in place when both boxes are there
  // and sit in adjacent slots (9 (T-1) is 0 or 3 modulo 6): blocks 1 and 3, and
  // block 2 when T is even, after another tile; blocks 2 and 3 of a single tile.
  // The other blocks' boxes are read again, as whole 128-row boxes, into the
  // ring-B space.
  constexpr bool kResidentTail = kSlotsA == 6;
  const bool rope_first = kResidentTail && T >= 2;
  auto box_at = [&](int t, int j) {   // latent/RoPE box at position j of tile t
    return rope_first && t == T - 1 ? (j + 8) % 9 : j;
  };
  auto tail_pos = [&](int k) { return rope_first ? k + 1 : k; };   // of latent box k
  auto tail_slot = [&](int k) { return (9 * (T - 1) + tail_pos(k)) % kSlotsA; };
  auto tail_res = [&](int mb) {
    return tail_pos(2 * mb) >= 3 && tail_slot(2 * mb) != kSlotsA - 1;
  };
  // Block 0 is never in ring A at the end: its two boxes are read again into
  // the query area, free once every score MMA has finished; a second block read
  // again (a single tile, or T odd) goes to the ring-B space.
  static_assert(!kResidentTail || 2 * kBoxBytes <= 9 * kQBoxBytes,
                "block 0's boxes fit in the query area");
  auto tail_box_off = [&](int k) {   // the last tile's latent box k (0-7)
    return tail_res(k >> 1) ? kOffA + tail_slot(k) * kBoxBytes
                            : (k < 2 ? kOffQ : kOffB) + (k & 1) * kBoxBytes;
  };


  if (warp == kWarpA) {
    // ------------------------------------------------------------ ring A (HBM)
    if (lane == 0) {
      int issued = kSlotsA;   // stream positions issued so far (the first fills included)
      Cursor c{0, items[0].tiles};
      for (int t = 0; t < T && !*abort_flag; ++t) {
        if (p.stop_after_tiles > 0 && t >= p.stop_after_tiles) break;   // test hook
        seek(c, t);
        const int row = row_of(c, t);
        for (int k = 0; k < 9; ++k) {
          const int pos = 9 * t + k, sl = pos % kSlotsA, use = pos / kSlotsA;
          if (pos < kSlotsA) continue;   // issued before the CTA-wide barrier
          if (use > 0 && !wait_or_abort(bar(BAR_EMPTYA + sl), (use - 1) & 1, abort_flag, wait_ns)) break;
          mbar_arrive_expect_tx(bar(BAR_FULLA + sl), kBoxBytes);
          if (MLA_IN_BOUNDS(row >= 0 && row < cache_rows))
            tma_load_2d(sbase + kOffA + sl * kBoxBytes, &tmap, 64 * box_at(t, k), row,
                        bar(BAR_FULLA + sl), keep);
          issued = pos + 1;
        }
      }
      // After an abort, the boxes still in flight (at most the last use of each
      // slot) land before the CTA leaves.
      if (*abort_flag)
        for (int pos = issued > kSlotsA ? issued - kSlotsA : 0; pos < issued; ++pos)
          drain_phase(bar(BAR_FULLA + pos % kSlotsA), (pos / kSlotsA) & 1, wait_ns);
    }
  } else if (warp == kWarpB) {
    // ------------------------------------------------------------ ring B (L2)
    if (lane == 0) {
      prefetch_tmap(&tmap_half);
      const uint64_t stream = l2_evict_first_policy();
      int issued = 0;          // ring-B positions issued (8 per tile)
      uint32_t armed_x = 0;    // single-use barriers BAR_FULLX + k armed
      Cursor c{0, items[0].tiles};
      for (int t = 0; t < T && !*abort_flag; ++t) {
        seek(c, t);
        if (kResidentTail && t == T - 1) {
          // The last tile's boxes that left ring A: block 0's into the query
          // area once every score MMA has finished, a second block's into the
          // ring-B space once the PV of tile T-2 has finished too.
          if (!wait_or_abort(bar(BAR_LASTA), 0, abort_flag, wait_ns)) break;
          bool second = false;
          for (int k = 0; k < 8; ++k) {
            if (tail_res(k >> 1)) continue;
            if (k >= 2 && !second) {
              if (T >= 2 && !wait_or_abort(bar(BAR_PVPREV), 0, abort_flag, wait_ns)) break;
              second = true;
            }
            mbar_arrive_expect_tx(bar(BAR_FULLX + k), kBoxBytes);
            if (MLA_IN_BOUNDS(last_row >= 0 && last_row < cache_rows))
              tma_load_2d(sbase + tail_box_off(k), &tmap, 64 * k, last_row, bar(BAR_FULLX + k),
                          stream);
            armed_x |= 1u << k;
          }
          break;
        }
        // A tile's pairs go out as soon as their ring slots are free (pacing them
        // on the tile's score MMAs measured 1 % slower on the large caches); by
        // then ring A, which runs ahead of the scores, has brought the rows to L2.
        // Unit u holds O^T block mb = u % 4 (ring slot mb) for row half u / 4.
        bool lasta = false;
        const int trow = row_of(c, t);
        for (int u = 0; u < 8 && !*abort_flag; ++u) {
          const int mb = u & 3, kh = u >> 2;
          const int row = trow + 64 * kh;
          if (borrowed(t, u)) {
            const int x = borrow_x(u);
            if (!lasta && !wait_or_abort(bar(BAR_LASTA), 0, abort_flag, wait_ns)) break;
            lasta = true;
            mbar_arrive_expect_tx(bar(BAR_FULLX + x), 2 * kHalfBox);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (MLA_IN_BOUNDS(row >= 0 && row < cache_rows))
                tma_load_2d(sbase + borrow_off(x) + h * kHalfBox, &tmap_half, 64 * (2 * mb + h),
                            row, bar(BAR_FULLX + x), stream);
            armed_x |= 1u << x;
            continue;
          }
          const int pos = 8 * t + u, sl = pos % kSlotsB, use = pos / kSlotsB;
          if (use > 0 && !wait_or_abort(bar(BAR_EMPTYB + sl), (use - 1) & 1, abort_flag, wait_ns)) break;
          mbar_arrive_expect_tx(bar(BAR_FULLB + sl), 2 * kHalfBox);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (MLA_IN_BOUNDS(row >= 0 && row < cache_rows))
              tma_load_2d(sbase + kOffB + (2 * sl + h) * kHalfBox, &tmap_half, 64 * (2 * mb + h),
                          row, bar(BAR_FULLB + sl), stream);
          issued = pos + 1;
        }
      }
      // After an abort, the pairs still in flight land before the CTA leaves:
      // the last use of each ring slot, and every single-use barrier armed.
      if (*abort_flag) {
        for (int pos = issued > kSlotsB ? issued - kSlotsB : 0; pos < issued; ++pos)
          drain_phase(bar(BAR_FULLB + pos % kSlotsB), (pos / kSlotsB) & 1, wait_ns);
        for (int k = 0; k < 8; ++k)
          if (armed_x >> k & 1u) drain_phase(bar(BAR_FULLX + k), 0, wait_ns);
      }
    }
  } else if (!kPersist && (warp < kSoftWarps || warp == kWarpS0 || warp == kWarpS1)) {
    // A one-item CTA's query (see above), then the softmax warps and the score
    // issuers meet: query in place.
    if (warp < kSoftWarps) {
      pdl_wait();
      load_query(qv0, qh0);
    }
    named_bar_sync(2, kSoftThreads + 64);
  }

  // One PV unit: O^T block u % 4 (of the O^T buffer at column ocol) += C^T (pair
  // u of tile t) . P^T (row half u / 4); four MMAs; `fresh`: the tile is its
  // item's first (the block starts from zero); `zmid`: a tile before the last
  // whose pairs are zeroed past the sequence's end first.  false if a wait gave up.
  constexpr uint32_t idesc_o = umma_idesc_bf16(128, kQN, 1, 0);
  auto pv_unit = [&](int t, int u, bool fresh, uint32_t ocol, bool zmid) -> bool {
    const int mb = u & 3, kh = u >> 2;
    if (kResidentTail && t == T - 1) {
      // Block mb's two 64-column boxes 2mb, 2mb + 1 (128 rows each, kBoxBytes
      // apart): still in ring A or read again into the ring-B space.
      const int k0 = 2 * mb;
      if (zero_last && (!wait_or_abort(bar(BAR_ZEROX + k0), 0, abort_flag, wait_ns) ||
                        !wait_or_abort(bar(BAR_ZEROX + k0 + 1), 0, abort_flag, wait_ns)))
        return false;
      if (!tail_res(mb) && (!wait_or_abort(bar(BAR_FULLX + k0), 0, abort_flag, wait_ns) ||
                     !wait_or_abort(bar(BAR_FULLX + k0 + 1), 0, abort_flag, wait_ns)))
        return false;
      tc_fence_after();
      const uint64_t c = umma_desc_sw128(sbase + kOffA, kBoxBytes, 1024) +
                         static_cast<uint64_t>((tail_box_off(k0) + kh * kHalfBox - kOffA) >> 4);
      const uint64_t pd = umma_desc_sw128(sbase + kOffP, 16, 1024) +
                          static_cast<uint64_t>(((t % kPBufs) * kPBytes + kh * kPSub) >> 4);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tmem + ocol + kQN * mb, c + ((ks * 2048) >> 4), pd + ((ks * 32) >> 4), idesc_o,
                  (!fresh || kh > 0 || ks > 0) ? 1u : 0u);
      return true;
    }
    const int pos = 8 * t + u, sl = pos % kSlotsB;
    const bool bw = borrowed(t, u);
    const int x = bw ? borrow_x(u) : 0;
    if (t == T - 1 && zero_last &&
        !wait_or_abort(bw ? bar(BAR_ZEROX + x) : bar(BAR_ZEROB + sl), 0, abort_flag, wait_ns))
      return false;
    // A zeroed tile before the last zeroes each slot twice (units u and u + 4),
    // so the zeroing of unit u completes the phase of parity u / 4.
    if (zmid && !wait_or_abort(bar(BAR_ZEROB + sl), kh, abort_flag, wait_ns)) return false;
    if (!wait_or_abort(bw ? bar(BAR_FULLX + x) : bar(BAR_FULLB + sl), bw ? 0 : (pos / kSlotsB) & 1,
                       abort_flag, wait_ns))
      return false;
    tc_fence_after();
    // MN-major pair: two 64-column boxes kHalfBox apart; the descriptor's
    // start address moves by 16-byte units.
    const uint64_t c = umma_desc_sw128(sbase + kOffA, kHalfBox, 1024) +
                       static_cast<uint64_t>(((bw ? borrow_off(x) : kOffB + sl * 2 * kHalfBox) - kOffA) >> 4);
    const uint64_t pd = umma_desc_sw128(sbase + kOffP, 16, 1024) +
                        static_cast<uint64_t>(((t % kPBufs) * kPBytes + kh * kPSub) >> 4);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_bf16(tmem + ocol + kQN * mb, c + ((ks * 2048) >> 4), pd + ((ks * 32) >> 4), idesc_o,
                (!fresh || kh > 0 || ks > 0) ? 1u : 0u);
    if (!bw) umma_commit(bar(BAR_EMPTYB + sl));
    return true;
  };
  // Before item i's first PV: the epilogue of item i - kOBufs has read the O^T
  // buffer item i accumulates into.
  auto wait_drain = [&](int i) {
    return i < L::kOBufs || wait_or_abort(bar(BAR_ODRAIN + i % L::kOBufs),
                                          ((i - L::kOBufs) / L::kOBufs) & 1, abort_flag, wait_ns);
  };

  if (warp == kWarpS0 || warp == kWarpS1) {
    // ------------------------------------------------------------ score MMA issuers
    // Issuer i takes the boxes whose stream position 9t + k has parity i, so it
    // owns ring-A slots i, i + 2, i + 4 and meets each slot's phases in order;
    // it accumulates them into its own S_i and the softmax adds S_0 + S_1.  One
    // thread issues a tcgen05.mma only every ~100 cycles, so the work is spread
    // over threads.
    if (lane == 0) {
      const int i = warp == kWarpS0 ? 0 : 1;
      constexpr uint32_t idesc_s = umma_idesc_bf16(128, kQN, 0, 0);
      // Base descriptors; a K step only moves the 14-bit start-address field,
      // so each MMA adds an offset (16-byte units) to a base.
      const uint64_t dA0 = umma_desc_sw128(sbase + kOffA, 16, 1024);     // K-major box
      const uint64_t dQ0 = umma_desc_sw128(sbase + kOffQ, 16, 1024);     // Q hi|lo
      const uint32_t dS = tmem + kS1Col * i;
      Cursor c{0, items[0].tiles};
      int qk = 0;   // query changes so far
      for (int t = 0; t < T; ++t) {
        seek(c, t);
        if (kMulti && __builtin_expect(c.i > 0 && t == items[c.i].t0 && new_query(c.i), 0)) {
          // The previous item's score MMAs release the query area; the softmax
          // warps fill it with this item's query.
          umma_commit(bar(BAR_QFREE));
          if (!wait_or_abort(bar(BAR_QREADY), qk & 1, abort_flag, wait_ns)) break;
          ++qk;
        }
        const int sb = t & 1;
        if (t >= 2 && !wait_or_abort(bar(BAR_SFREE + sb), ((t - 2) >> 1) & 1, abort_flag, wait_ns)) break;
        bool ok = true, first = true;
        for (int k = (9 * t + i) & 1; k < 9; k += 2) {
          const int pos = 9 * t + k, sl = pos % kSlotsA;
          if (!wait_or_abort(bar(BAR_FULLA + sl), (pos / kSlotsA) & 1, abort_flag, wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a = dA0 + static_cast<uint64_t>((sl * kBoxBytes) >> 4);
          const uint64_t q = dQ0 + static_cast<uint64_t>((box_at(t, k) * kQBoxBytes) >> 4);
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4)
            umma_bf16(dS + kQN * sb, a + ((s4 * 32) >> 4), q + ((s4 * 32) >> 4), idesc_s,
                      (!first || s4 > 0) ? 1u : 0u);
          umma_commit(bar(BAR_EMPTYA + sl));
          first = false;
        }
        if (!ok) break;
        umma_commit(bar(BAR_SFULL + sb));
        s_issued[i] = t + 1;
      }
      umma_commit(bar(BAR_LASTA));   // ring A and the query area are free for the last pairs
      // The last tile's PV is the tail of the kernel: these two threads take O^T
      // blocks 2 and 3 of it (after the PV issuers have finished tile T-2, the
      // previous writers of those blocks).
      {
        const int t = T - 1;
        bool ok = !*abort_flag;
        if (ok && T >= 2 && !wait_or_abort(bar(BAR_PVPREV), 0, abort_flag, wait_ns)) ok = false;
        if (ok && fin_first && !wait_drain(fin_item)) ok = false;
        if (ok && !wait_or_abort(bar(BAR_PFULL + (t & 1)), (t >> 1) & 1, abort_flag, wait_ns)) ok = false;
        if (ok && pv_unit(t, 2 + i, fin_first, obuf_col(fin_item), false) &&
            (!kHalfP || wait_or_abort(bar(BAR_PFULL1 + (t & 1)), (t >> 1) & 1, abort_flag, wait_ns)))
          pv_unit(t, 6 + i, fin_first, obuf_col(fin_item), false);
        umma_commit(bar(BAR_ODONE2));
      }
      // Every MMA this thread issued has finished before TMEM is released.
      umma_commit(bar(BAR_DONE));
      mbar_wait_bounded(bar(BAR_DONE), 0);
    }
  } else if (warp == kWarpPV0 || warp == kWarpPV1) {
    // ------------------------------------------------------------ PV MMA issuers
    // Issuer i takes O^T blocks mb = i and i + 2 (ring-B slots i and i + 2); of
    // the last tile only block i (the score issuers take blocks 2 and 3).
    if (lane == 0) {
      const int i = warp - kWarpPV0;
      Cursor c{0, items[0].tiles};
      for (int t = 0; t < T; ++t) {
        seek(c, t);
        const bool fresh = t == items[c.i].t0;
        if (fresh && !wait_drain(c.i)) break;
        if (!wait_or_abort(bar(BAR_PFULL + (t & 1)), (t >> 1) & 1, abort_flag, wait_ns)) break;
        bool ok = true;
        const int step = t == T - 1 ? 4 : 2;
        const bool zmid = zero_mid(c, t);
        for (int u = i; u < 8 && ok; u += step) {
          if (kHalfP && u >= 4 && u - step < 4) {
            // Rows 0-63 of P are free once this thread's MMAs so far have
            // finished; rows 64-127 are needed from here on.
            umma_commit(bar(BAR_P0FREE + (t & 1)));
            if (!wait_or_abort(bar(BAR_PFULL1 + (t & 1)), (t >> 1) & 1, abort_flag, wait_ns)) {
              ok = false;
              break;
            }
          }
          ok = pv_unit(t, u, fresh, obuf_col(c.i), zmid);
        }
        if (!ok) break;
        umma_commit(bar(BAR_ODONE + (t & 1)));
        if (t == T - 2) umma_commit(bar(BAR_PVPREV));
      }
      umma_commit(bar(BAR_DONE));
      mbar_wait_bounded(bar(BAR_DONE), 0);
    }
  } else if (warp < kSoftWarps) {
    // ------------------------------------------------------------ softmax warps
    const int gp = warp >> 2, wq = warp & 3;
    const int hb = kGroupHeads * gp;                     // first head of this group
    const int row = 32 * wq + lane;                     // tile row held by this thread
    const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
    float m[kGroupHeads], l[kGroupHeads];
#pragma unroll
    for (int h = 0; h < kGroupHeads; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    // An item's result: its row sums and maxima (m, l), once its last PV
    // (tile t_end) has finished; O^T buffer at column ocol.
    auto finish_item = [&](int idx, int t_end, const float* mm, const float* ll, bool last) {
      const SplitItem it = items[idx];
      const uint32_t ocol = obuf_col(idx);
#pragma unroll
      for (int e = 0; e < kGroupHeads; e += 8) {
        float tt[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) tt[h] = ll[e + h];
        const float ws = reduce8_heads<false>(tt, lane);
        if (lane < 16 && (lane & 1) == 0) lsum[(hb + e + (lane >> 1)) * 4 + wq] = ws;
      }
      // O^T after the item's last PV: this thread's latent row is d = 128 mb + 32 wq + lane.
      // The CTA's last tile's PV is split: blocks 2 and 3 complete BAR_ODONE2 (score
      // issuers), blocks 0 and 1 BAR_ODONE (PV issuers; block 0 usually waits for
      // its re-read).  The one-item 16-head kernel stores blocks 2-3 first, then 0-1
      // (bench workload: split 12.59 -> 12.28 us); with the other instances' register
      // budgets the second pass of loads costs more than it saves.
      constexpr bool kEarlyBlocks = kG == 16 && !kPersist;
      if (!kEarlyBlocks || !last)
        wait_or_abort(bar(BAR_ODONE + (t_end & 1)), (t_end >> 1) & 1, abort_flag, wait_ns);
      if (last) wait_or_abort(bar(BAR_ODONE2), 0, abort_flag, wait_ns);
      tc_fence_after();
      named_bar_sync(1, kSoftThreads);
      if (!*abort_flag) {
        // Row (v, h, j) of the partials; heads h0 + hw + h are p.splits rows apart
        // (paired tokens: groups 2 and 3 belong to query group v + 1).
        const size_t base = size_t(it.part) + (pair ? size_t(gp >> 1) * p.H * p.splits : 0);
        const int hw = pair ? kGroupHeads * (gp & 1) : hb;
        // 1/L by the approximate reciprocal (within 2 ulp for the L > 0 reached
        // here, 1 <= L <= 2^8 x rows): a branch-free instruction, where eight
        // IEEE divisions in a row cost about 0.4 us of the CTA's critical path.
        // Lane h of the first warp of each group writes head h's log-sum-exp.
        float inv[kGroupHeads], Lme = 0.f, mme = 0.f;
#pragma unroll
        for (int h = 0; h < kGroupHeads; ++h) {
          const float4 q4 = *reinterpret_cast<const float4*>(lsum + (hb + h) * 4);
          const float Ls = (q4.x + q4.y) + (q4.z + q4.w);
          inv[h] = Ls > 0.f ? __fdividef(1.f, Ls) : 0.f;
          Lme = lane == h ? Ls : Lme;
          mme = lane == h ? mm[h] : mme;
        }
        const size_t n_part = size_t(p.B) * p.H * p.splits;   // rows of the partials
        if (wq == 0 && lane < kGroupHeads &&
            MLA_IN_BOUNDS(base + size_t(hw + lane) * p.splits < n_part))
          p.part_lse[base + size_t(hw + lane) * p.splits] =
              Lme > 0.f ? (mme + log2f(Lme)) * kLn2 : -INFINITY;
        // Two parts: columns hb.. (hi) and kG + hb.. (lo) of each O^T block, summed;
        // one part: columns hb..hb+15 (heads hb..hb+7, then hb+8..hb+15).
        const size_t head_stride = size_t(p.splits) * kDc;
        if (!kEarlyBlocks) {
          uint32_t x4[4][8], y4[4][8];
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
            tmem_ld8_nowait(tmem + lane_base + ocol + kQN * mb + hb, x4[mb]);
            tmem_ld8_nowait(tmem + lane_base + ocol + kQN * mb + (kParts == 2 ? kHeadGroup : 8) + hb,
                            y4[mb]);
          }
          tmem_wait_ld();
          float* orow = p.part_o + (base + size_t(hw) * p.splits) * kDc + 32 * wq + lane;
#pragma unroll
          for (int h = 0; h < kGroupHeads; ++h, orow += head_stride) {
            if (!MLA_IN_BOUNDS(base + size_t(hw + h) * p.splits < n_part)) continue;
#pragma unroll
            for (int mb = 0; mb < 4; ++mb)
              orow[128 * mb] = (kParts == 2 ? __uint_as_float(x4[mb][h]) + __uint_as_float(y4[mb][h])
                                : h < 8     ? __uint_as_float(x4[mb][h & 7])
                                            : __uint_as_float(y4[mb][h & 7])) *
                               inv[h];
          }
        }
        auto store_blocks = [&](int mb0) {   // O^T blocks mb0 and mb0 + 1
          uint32_t x4[2][8], y4[2][8];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t col = ocol + kQN * (mb0 + q) + hb;
            tmem_ld8_nowait(tmem + lane_base + col, x4[q]);
            tmem_ld8_nowait(tmem + lane_base + col + (kParts == 2 ? kHeadGroup : 8), y4[q]);
          }
          tmem_wait_ld();
          float* orow = p.part_o + (base + size_t(hw) * p.splits) * kDc + 128 * mb0 + 32 * wq + lane;
#pragma unroll
          for (int h = 0; h < kGroupHeads; ++h, orow += head_stride) {
            if (!MLA_IN_BOUNDS(base + size_t(hw + h) * p.splits < n_part)) continue;
#pragma unroll
            for (int q = 0; q < 2; ++q)
              orow[128 * q] = (kParts == 2 ? __uint_as_float(x4[q][h]) + __uint_as_float(y4[q][h])
                               : h < 8     ? __uint_as_float(x4[q][h & 7])
                                           : __uint_as_float(y4[q][h & 7])) *
                              inv[h];
          }
        };
        if (kEarlyBlocks) {
          store_blocks(2);
          if (last) {
            wait_or_abort(bar(BAR_ODONE + (t_end & 1)), (t_end >> 1) & 1, abort_flag, wait_ns);
            tc_fence_after();
          }
          store_blocks(0);
        }
      }
      if (!last) {
        // The O^T buffer may take a later item now.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_ODRAIN + idx % L::kOBufs));
      }
    };
    Cursor c{0, items[0].tiles};
    int qk = 0;                  // query changes so far
    int pend = -1, pend_t = 0;   // item whose partial is still to be written, its last tile
    float mp[kGroupHeads], lp[kGroupHeads];
    for (int t = 0; t < T; ++t) {
      seek(c, t);
      const SplitItem it = items[c.i];
      const bool first_t = t == it.t0, last_t = t == it.t0 + it.tiles - 1;
      const int sb = t & 1;
      int valid = last_t ? it.valid_last : kTileRows;
      if (pair)   // this group's token ends at its own length (one item: tile t of chunk r0)
        valid = min(max(min(r0_one + p.chunk, gp < 2 ? len_first : len_pair) -
                            (r0_one + t * kTileRows), 0),
                    kTileRows);
      if (kMulti && first_t && t > 0) {
#pragma unroll
        for (int h = 0; h < kGroupHeads; ++h) {
          m[h] = -INFINITY;
          l[h] = 0.f;
        }
      }
      wait_or_abort(bar(BAR_SFULL + sb), (t >> 1) & 1, abort_flag, wait_ns);
      tc_fence_after();
      float sc[kGroupHeads], tt[kGroupHeads];
      {
        // Two parts: S = hi + lo columns of each accumulator; one part: columns
        // hb..hb+7 and hb+8..hb+15 of each accumulator are 16 heads.
        constexpr int kY = kParts == 2 ? kHeadGroup : 8;
        uint32_t x0[8], y0[8], x1[8], y1[8];
        tmem_ld8_nowait(tmem + lane_base + kQN * sb + hb, x0);
        tmem_ld8_nowait(tmem + lane_base + kQN * sb + kY + hb, y0);
        tmem_ld8_nowait(tmem + lane_base + kS1Col + kQN * sb + hb, x1);
        tmem_ld8_nowait(tmem + lane_base + kS1Col + kQN * sb + kY + hb, y1);
        tmem_wait_ld();
        const bool rv = row < valid;
#pragma unroll
        for (int h = 0; h < kGroupHeads; ++h) {
          const float s0 = kParts == 2 ? __uint_as_float(x0[h]) + __uint_as_float(y0[h])
                                       : __uint_as_float(h < 8 ? x0[h & 7] : y0[h & 7]);
          const float s1 = kParts == 2 ? __uint_as_float(x1[h]) + __uint_as_float(y1[h])
                                       : __uint_as_float(h < 8 ? x1[h & 7] : y1[h & 7]);
          sc[h] = rv ? (s0 + s1) * p.scale_log2 : -INFINITY;
          tt[h] = sc[h];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_SFREE + sb));
      float* rd = red + sb * kHeadGroup * 4;
#pragma unroll
      for (int e = 0; e < kGroupHeads; e += 8) {
        const float wmax = reduce8_heads<true>(tt + e, lane);
        if (lane < 16 && (lane & 1) == 0) rd[(hb + e + (lane >> 1)) * 4 + wq] = wmax;
      }
      named_bar_sync(1, kSoftThreads);
      bool need = false;
      float tmax[kGroupHeads];
#pragma unroll
      for (int h = 0; h < kGroupHeads; ++h) {
        const float4 q4 = *reinterpret_cast<const float4*>(rd + (hb + h) * 4);
        tmax[h] = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
        need |= tmax[h] > m[h] + kRescaleLog2;
      }
      if (need) {
        // Move this group's reference maxima; rescale its row sums and the O^T
        // columns it owns (in TMEM, after the previous PV finished).  The first
        // tile of an item starts from nothing (its first PV overwrites).
        float alpha[kGroupHeads];
#pragma unroll
        for (int h = 0; h < kGroupHeads; ++h) {
          const float mn = fmaxf(m[h], tmax[h]);
          alpha[h] = m[h] == -INFINITY ? 0.f : ex2(m[h] - mn);
          m[h] = mn;
          l[h] *= alpha[h];
        }
        if (!first_t) {
          wait_or_abort(bar(BAR_ODONE + ((t - 1) & 1)), ((t - 1) >> 1) & 1, abort_flag, wait_ns);
          tc_fence_after();
          const uint32_t ocol = obuf_col(c.i);
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              // two parts: hi (half 0) and lo (half 1) of 8 heads; one part: heads
              // hb.. (half 0) and hb+8.. (half 1)
              const uint32_t col = ocol + kQN * mb + (kParts == 2 ? kHeadGroup : 8) * half + hb;
              const int a0 = kParts == 2 ? 0 : 8 * half;
              uint32_t r[8];
              float o[8];
              tmem_ld8_nowait(tmem + lane_base + col, r);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 8; ++h) o[h] = __uint_as_float(r[h]) * alpha[a0 + h];
              tmem_st8(tmem + lane_base + col, o);
            }
          }
          tmem_wait_st();
        }
      }
#pragma unroll
      for (int h = 0; h < kGroupHeads; ++h) {
        const float mu = m[h] == -INFINITY ? 0.f : m[h];
        sc[h] = ex2(sc[h] - mu);
        l[h] += sc[h];
      }
      // P^T buffer sb was last read by the PV of tile t - kPBufs (with one buffer,
      // its rows 0-63 by that PV's first half).
      if (t >= kPBufs) {
        if (kHalfP && wq < 2)
          wait_or_abort(bar(BAR_P0FREE + ((t - 1) & 1)), ((t - 1) >> 1) & 1, abort_flag, wait_ns);
        else
          wait_or_abort(bar(BAR_ODONE + ((t - kPBufs) & 1)), ((t - kPBufs) >> 1) & 1, abort_flag,
                        wait_ns);
      }
      {
        // P^T (B operand of the PV MMA, K-major 128-byte swizzle, two 64-row
        // halves): two parts: row n < kG is bf16(p) of head n, row kG + n is
        // bf16(p - bf16(p)); one part: row n is bf16(p) of head n.  The K index
        // is the tile row.
        const uint32_t pofs = (t % kPBufs) * kPBytes + (row >> 6) * kPSub;
        uint8_t* pbuf = smem + kOffP + pofs;
        const int ch = (row & 63) >> 3, w = row & 7;
#pragma unroll
        for (int h = 0; h < kGroupHeads; ++h) {
          const __nv_bfloat16 hi = __float2bfloat16_rn(sc[h]);
          const __nv_bfloat16 lo = __float2bfloat16_rn(sc[h] - __bfloat162float(hi));
          const int top = kParts == 2 ? kHeadGroup + hb + h : hb + h;   // highest row written
          if (!MLA_IN_BOUNDS(pofs + sw128(top, ch) + 2 * w + 2 <= uint32_t(kPBufs * kPBytes)))
            continue;
          *reinterpret_cast<__nv_bfloat16*>(pbuf + sw128(hb + h, ch) + 2 * w) = hi;
          if (kParts == 2)
            *reinterpret_cast<__nv_bfloat16*>(pbuf + sw128(kHeadGroup + hb + h, ch) + 2 * w) = lo;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar((kHalfP && wq >= 2 ? BAR_PFULL1 : BAR_PFULL) + sb));
      if (t == T - 1 && zero_last) {
        // The last tile reaches past the sequence's end.  As each of its latent
        // box pairs lands in ring B, zero the rows past the end (they may hold
        // anything, NaN included) so that P = 0 times such a row adds exactly 0.
        // Borrowed pairs have single-use barriers; ring-B pairs of the last tile
        // exist only when it is the first tile too (first fills).
        if (kResidentTail) {
          // Whole 128-row boxes: in ring A (landed before the scores this thread
          // has read) or once read again.
          const int nrow = kTileRows - zero_from;
          for (int k = 0; k < 8; ++k) {
            if (!tail_res(k >> 1)) wait_or_abort(bar(BAR_FULLX + k), 0, abort_flag, wait_ns);
            uint8_t* box = smem + tail_box_off(k) + zero_from * 128;
            for (int q = tid; q < nrow * 8; q += kSoftThreads)
              if (MLA_IN_BOUNDS(zero_from >= 0 && tail_box_off(k) + zero_from * 128 + q * 16 + 16 <=
                                                     tail_box_off(k) + kBoxBytes))
                *reinterpret_cast<uint4*>(box + q * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_ZEROX + k));
          }
        }
        for (int u = 0; u < 8 && !kResidentTail; ++u) {
          const int kh = u >> 2;
          const int first = max(0, zero_from - 64 * kh);   // first row of this half to clear
          const int nrow = 64 - first;
          const int pos = 8 * t + u, sl = pos % kSlotsB;
          const bool bw = borrowed(t, u);
          const int x = bw ? borrow_x(u) : 0;
          wait_or_abort(bw ? bar(BAR_FULLX + x) : bar(BAR_FULLB + sl), bw ? 0 : (pos / kSlotsB) & 1,
                        abort_flag, wait_ns);
          uint8_t* pr = smem + (bw ? borrow_off(x) : kOffB + 2 * sl * kHalfBox);
          for (int q = tid; q < 2 * nrow * 8; q += kSoftThreads) {
            const int h = q / (nrow * 8), rem = q % (nrow * 8);
            const int o = h * kHalfBox + (first + rem / 8) * 128 + (rem % 8) * 16;
            if (MLA_IN_BOUNDS(o >= 0 && o + 16 <= 2 * kHalfBox))
              *reinterpret_cast<uint4*>(pr + o) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bw ? bar(BAR_ZEROX + x) : bar(BAR_ZEROB + sl));
        }
      } else if (__builtin_expect(zero_mid(c, t), 0)) {
        // A tile before the last that ends its item at the sequence's end: the
        // same zeroing on its ring-B pairs (one phase of the slot's barrier per
        // pair, two pairs per slot).
        // Its slots' previous uses belong to tile t - 1: once that tile's PV has
        // finished, each slot's full barrier is at most one phase short of
        // this tile's pair, so the parity waits below cannot pass on an older
        // phase (the PV issuers, not this role, consume the ring in order).
        const int zf = it.zero_from;
        if (t > 0)
          wait_or_abort(bar(BAR_ODONE + ((t - 1) & 1)), ((t - 1) >> 1) & 1, abort_flag, wait_ns);
        for (int u = 0; u < 8; ++u) {
          const int kh = u >> 2;
          const int first = max(0, zf - 64 * kh);
          const int nrow = 64 - first;
          const int pos = 8 * t + u, sl = pos % kSlotsB;
          wait_or_abort(bar(BAR_FULLB + sl), (pos / kSlotsB) & 1, abort_flag, wait_ns);
          uint8_t* pr = smem + kOffB + 2 * sl * kHalfBox;
          for (int q = tid; q < 2 * nrow * 8; q += kSoftThreads) {
            const int h = q / (nrow * 8), rem = q % (nrow * 8);
            const int o = h * kHalfBox + (first + rem / 8) * 128 + (rem % 8) * 16;
            if (MLA_IN_BOUNDS(o >= 0 && o + 16 <= 2 * kHalfBox))
              *reinterpret_cast<uint4*>(pr + o) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_ZEROB + sl));
        }
      }
      // The previous item's partial, one tile late: its last PV has had this
      // tile's softmax to finish.
      if (kMulti && pend >= 0) {
        finish_item(pend, pend_t, mp, lp, false);
        pend = -1;
      }
      if (kMulti && last_t && t != T - 1) {
        // The next item's query, once this item's score MMAs are done with the
        // query area (the score issuers wait for it).
        if (__builtin_expect(new_query(c.i + 1), 0)) {
          wait_or_abort(bar(BAR_QFREE), qk & 1, abort_flag, wait_ns);
          load_query(items[c.i + 1].qv, items[c.i + 1].h0);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_QREADY));
          ++qk;
        }
        pend = c.i;
        pend_t = t;
#pragma unroll
        for (int h = 0; h < kGroupHeads; ++h) {
          mp[h] = m[h];
          lp[h] = l[h];
        }
      }
    }
    // The combine may start launching: it waits for this grid anyway, and a
    // dependent that starts much earlier only sleeps longer.
    if (tid == 0) pdl_launch_dependents();
    finish_item(fin_item, T - 1, m, l, true);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_flag) {
    report(p.status, MLA_DEV_PIPELINE_TIMEOUT);
    if (p.debug) {   // test hook: where this CTA's first wait gave up
      const int k = atomicAdd(p.debug, 1);
      if (k < 256) {
        int* r = p.debug + 1 + 8 * k;
        r[0] = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
        r[1] = (abort_flag[1] - static_cast<int>(bars)) / 8;   // barrier index
        r[2] = abort_flag[2] & 0xFF;                            // parity
        r[3] = abort_flag[2] >> 8;                              // thread
        r[4] = n_items;
        r[5] = T;
        r[6] = s_issued[0];
        r[7] = s_issued[1];
      }
    }
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
    const float* row = cache + (size_t(cache_seq(p, b)) * p.s_max + t) * kRow;
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
  const size_t base = (size_t(b) * p.H + h) * p.splits + j;
  for (int c = tid; c < kDc; c += kThreads) {
    float v = 0.f;
    for (int w = 0; w < kWarps; ++w) v += f[w] * wo[w][c];
    p.part_o[base * kDc + c] = v / L;
  }
  if (tid == 0) p.part_lse[base] = (M + log2f(L)) * kLn2;
}

// Merge of the chunk partials of one (sequence, head):
//   L = log sum_j exp(lse_j),  o_c = sum_j exp(lse_j - L) o_j.
// grid (H, B, 4), one warp per CTA: thread t of CTA z owns latent columns
// [128z + 4t, 128z + 4t + 4).  Chunks are taken kCombineChunk at a time with
// every load of a group in flight at once; a running maximum keeps the weights
// finite (each thread recomputes the group's weights itself, so there is no
// shared memory and no barrier).
constexpr int kCombineChunk = 20;
__global__ void __launch_bounds__(32)
    combine_kernel(const SplitParams p, float* o_c, float* lse_out) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = blockIdx.z * 32 + threadIdx.x;   // float4 column of the 512
  const int len = clamp_length(p, b, false);   // a caller input, not the split's output
  pdl_wait();   // the partials come from the split kernel just before
  int nsplit = (len + p.chunk - 1) / p.chunk;
  if (!MLA_IN_BOUNDS(nsplit <= p.splits)) nsplit = p.splits;   // partials past the workspace
  float* out = o_c + (size_t(b) * p.H + h) * kDc;
  if (nsplit == 0) {
    reinterpret_cast<float4*>(out)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0 && lse_out) lse_out[size_t(b) * p.H + h] = -INFINITY;
    if (threadIdx.x == 0) pdl_launch_dependents();
    return;
  }
  const size_t row0 = (size_t(b) * p.H + h) * p.splits;   // this (b, h)'s chunks, contiguous
  const float* lse_bh = p.part_lse + row0;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + row0 * kDc) + tid;
  float m = -INFINITY, sum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < nsplit; s0 += kCombineChunk) {
    float ls[kCombineChunk];
    float4 v[kCombineChunk];
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u) {
      const bool ok = s0 + u < nsplit;
      ls[u] = ok ? lse_bh[s0 + u] : -INFINITY;
      v[u] = ok ? po[size_t(s0 + u) * (kDc / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (s0 + kCombineChunk >= nsplit && threadIdx.x == 0) pdl_launch_dependents();
    float cm = m;
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u) cm = fmaxf(cm, ls[u]);
    // cm is finite: every chunk with rows has a finite lse.
    const float r = m == -INFINITY ? 0.f : expf(m - cm);
    sum *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u) {
      const float w = s0 + u < nsplit ? expf(ls[u] - cm) : 0.f;
      sum += w;
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
    m = cm;
  }
  const float inv = 1.f / sum;
  reinterpret_cast<float4*>(out)[tid] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (tid == 0 && lse_out) lse_out[size_t(b) * p.H + h] = m + logf(sum);
}

// The same merge for many chunks (more than 16): grid (H, B, 4), CTA z owns
// latent columns [128z, 128z + 128), lane t the float4 at 128z + 4t.  The CTA's
// W warps share the chunks (warp w takes chunks
// w, w + W, ...); each keeps up to kCombineChunk chunks' loads in flight and a
// running maximum that keeps the weights finite, and the W warp states are then
// merged through shared memory.  W grows with the chunk count (combine_warps),
// so that many chunks are not read one group after another by a single warp.
constexpr int kCombineMaxWarps = 8;
// Each warp keeps kCombineGroup chunks' loads in flight (fewer registers than
// the one-warp kernel's kCombineChunk, so that two 256-thread CTAs share an SM
// and 128 chunks of 4 x 16 heads take one wave).  The warp states are merged in
// dynamic shared memory.
constexpr int kCombineGroup = 16;
__global__ void __launch_bounds__(32 * kCombineMaxWarps, 2)
    combine_warps_kernel(const SplitParams p, float* o_c, float* lse_out) {
  extern __shared__ float4 s_acc[];   // [W][32], then s_m[W], s_sum[W]
  const int h = blockIdx.x, b = blockIdx.y;
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = blockIdx.z * 32 + lane;      // float4 column of the 512
  const int len = clamp_length(p, b, false);   // a caller input, not the split's output
  pdl_wait();   // the partials come from the split kernel just before
  int nsplit = (len + p.chunk - 1) / p.chunk;
  if (!MLA_IN_BOUNDS(nsplit <= p.splits)) nsplit = p.splits;   // partials past the workspace
  float* out = o_c + (size_t(b) * p.H + h) * kDc;
  if (nsplit == 0) {
    if (warp == 0) {
      reinterpret_cast<float4*>(out)[col] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (col == 0 && lse_out) lse_out[size_t(b) * p.H + h] = -INFINITY;
    }
    if (threadIdx.x == 0) pdl_launch_dependents();
    return;
  }
  const size_t row0 = (size_t(b) * p.H + h) * p.splits;   // this (b, h)'s chunks, contiguous
  const float* lse_bh = p.part_lse + row0;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + row0 * kDc) + col;
  float m = -INFINITY, sum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp; s0 < nsplit; s0 += W * kCombineGroup) {
    float ls[kCombineGroup];
    float4 v[kCombineGroup];
#pragma unroll
    for (int u = 0; u < kCombineGroup; ++u) {
      const int sj = s0 + W * u;
      const bool ok = sj < nsplit;
      ls[u] = ok ? lse_bh[sj] : -INFINITY;
      v[u] = ok ? po[size_t(sj) * (kDc / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (s0 + W * kCombineGroup >= nsplit && threadIdx.x == 0) pdl_launch_dependents();
    float cm = m;
#pragma unroll
    for (int u = 0; u < kCombineGroup; ++u) cm = fmaxf(cm, ls[u]);
    // cm is finite: every chunk with rows has a finite lse, and s0 < nsplit.
    const float r = m == -INFINITY ? 0.f : expf(m - cm);
    sum *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
#pragma unroll
    for (int u = 0; u < kCombineGroup; ++u) {
      const float w = s0 + W * u < nsplit ? expf(ls[u] - cm) : 0.f;
      sum += w;
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
    m = cm;
  }
  if (W > 1) {
    // Merge the warps' states (a warp without chunks has m = -inf, sum = 0).
    float* s_m = reinterpret_cast<float*>(s_acc + 32 * W);
    float* s_sum = s_m + W;
    s_acc[32 * warp + lane] = acc;
    if (lane == 0) {
      s_m[warp] = m;
      s_sum[warp] = sum;
    }
    __syncthreads();
    if (warp != 0) return;
    float M = -INFINITY;
    for (int w = 0; w < W; ++w) M = fmaxf(M, s_m[w]);
    sum = 0.f;
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < W; ++w) {
      const float f = s_m[w] == -INFINITY ? 0.f : expf(s_m[w] - M);
      const float4 a4 = s_acc[32 * w + lane];
      sum = fmaf(f, s_sum[w], sum);
      acc.x = fmaf(f, a4.x, acc.x);
      acc.y = fmaf(f, a4.y, acc.y);
      acc.z = fmaf(f, a4.z, acc.z);
      acc.w = fmaf(f, a4.w, acc.w);
    }
    m = M;
  }
  const float inv = 1.f / sum;
  reinterpret_cast<float4*>(out)[col] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (col == 0 && lse_out) lse_out[size_t(b) * p.H + h] = m + logf(sum);
}

// Warps per combine CTA for `splits` chunks: one up to 64 chunks (combine_kernel:
// few enough registers that many of its CTAs run at once, and launch beside the
// split's), then more (combine_warps_kernel), so that a warp takes at most about
// 16 chunks (128 chunks: 6.8 us against 7.9 for one warp per CTA).
int combine_warps(int splits) {
  if (splits <= 64) return 1;   // measured: 22 chunks over two warps 12.7 us against 5.8
  int w = 1;
  while (w < kCombineMaxWarps && splits > 16 * w) w *= 2;
  return w;
}

// Combine and value up-projection in one launch (bf16 weights), for the whole
// decode step:
//   o_c[b,h,:] = sum_j exp(lse_j - L) o_j     (as combine_kernel)
//   o[b,h,e]   = sum_c W_UV[h,e,c] o_c[b,h,c]   (Multi-Head Latent Attention eq. 3.3.3)
// grid (H, B, kDv / 32), 128 threads: CTA z produces o rows [32z, 32z + 32).
// It is small (a few KB of shared memory, moderate registers) so that its
// CTAs fit beside the split kernel's and launch before that kernel ends;
// before waiting they ask L2 for their 32 KB slice of W_UV[h].  Each CTA then
// merges the (b, h) chunk partials itself (each thread four columns, up to
// kCombineChunk chunks in flight), the one with z = 0 also writes o_c and lse.
// The slice is read coalesced: load k of thread t is 16-byte chunk 128 k + t,
// so a warp holds 32 consecutive chunks of one row half and sums its eight
// products per lane with shuffles.  fp32 arithmetic throughout.
constexpr int kOutRows = 32;
__global__ void __launch_bounds__(128)
    combine_out_kernel(const SplitParams p, const __nv_bfloat16* __restrict__ w_uv,
                       float* __restrict__ o_c, float* __restrict__ lse_out,
                       float* __restrict__ out) {
  __shared__ __align__(16) float oc[kDc];
  __shared__ float half_dot[kOutRows][2];
  const int h = blockIdx.x, b = blockIdx.y, z = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint4* wslice = reinterpret_cast<const uint4*>(w_uv + (size_t(h) * kDv + kOutRows * z) * kDc);
#pragma unroll
  for (int i = 0; i < 2; ++i)   // 256 lines of 128 bytes, two per thread
    asm volatile("prefetch.global.L2 [%0];" ::"l"(wslice + 8 * (tid + 128 * i)));
  const int len = clamp_length(p, b, false);   // a caller input, not the split's output
  pdl_wait();   // the partials come from the split kernel just before
  // The next kernel (the next step's mla_absorb_q) may launch now and fetch its
  // weights; it waits for this grid before it reads or writes anything else.
  if (tid == 0) pdl_launch_dependents();
  int nsplit = (len + p.chunk - 1) / p.chunk;
  if (!MLA_IN_BOUNDS(nsplit <= p.splits)) nsplit = p.splits;   // partials past the workspace
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse_v = -INFINITY;
  if (nsplit > 0) {
    const size_t row0 = (size_t(b) * p.H + h) * p.splits;
    const float* lse_bh = p.part_lse + row0;
    const float4* po = reinterpret_cast<const float4*>(p.part_o + row0 * kDc) + tid;
    float m = -INFINITY, sum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += kCombineChunk) {
      float ls[kCombineChunk];
      float4 v[kCombineChunk];
#pragma unroll
      for (int u = 0; u < kCombineChunk; ++u) {
        const bool ok = s0 + u < nsplit;
        ls[u] = ok ? lse_bh[s0 + u] : -INFINITY;
        v[u] = ok ? po[size_t(s0 + u) * (kDc / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float cm = m;
#pragma unroll
      for (int u = 0; u < kCombineChunk; ++u) cm = fmaxf(cm, ls[u]);
      const float rs = m == -INFINITY ? 0.f : expf(m - cm);
      sum *= rs;
      acc.x *= rs;
      acc.y *= rs;
      acc.z *= rs;
      acc.w *= rs;
#pragma unroll
      for (int u = 0; u < kCombineChunk; ++u) {
        const float w = s0 + u < nsplit ? expf(ls[u] - cm) : 0.f;
        sum += w;
        acc.x = fmaf(w, v[u].x, acc.x);
        acc.y = fmaf(w, v[u].y, acc.y);
        acc.z = fmaf(w, v[u].z, acc.z);
        acc.w = fmaf(w, v[u].w, acc.w);
      }
      m = cm;
    }
    const float inv = 1.f / sum;
    r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    lse_v = m + logf(sum);
  }
  reinterpret_cast<float4*>(oc)[tid] = r;
  if (z == 0) {
    reinterpret_cast<float4*>(o_c + (size_t(b) * p.H + h) * kDc)[tid] = r;
    if (tid == 0 && lse_out) lse_out[size_t(b) * p.H + h] = lse_v;
  }
  uint4 wv[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) wv[k] = wslice[128 * k + tid];
  __syncthreads();
  // Chunk 128 k + tid: row 2k + warp / 2, columns 8 (tid % 64) .. + 8.
  const float4* x = reinterpret_cast<const float4*>(oc) + 2 * (tid & 63);
  const float4 x0 = x[0], x1 = x[1];
  const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
    float d = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 wf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[q]));
      d = fmaf(wf.x, xs[2 * q], d);
      d = fmaf(wf.y, xs[2 * q + 1], d);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) half_dot[2 * k + (warp >> 1)][warp & 1] = d;
  }
  __syncthreads();
  if (tid < kOutRows)
    out[(size_t(b) * p.H + h) * kDv + kOutRows * z + tid] = half_dot[tid][0] + half_dot[tid][1];
}

// ------------------------------------------------------------------------- host side
// Heads per CTA of the decode kernel: 32 for a bf16 cache whose head count
// allows it, else 16 (the FP8 kernel always takes 16).
int tc_heads_per_cta(const mla_dims* d) {
  if (d->dtype != MLA_BF16) return kHeadGroup;
  if (d->heads % 64 == 0 && g_split_parts.load() != 2) return 64;
  return d->heads % 32 == 0 ? 32 : kHeadGroup;
}

// Whether the bf16 kernel pairs the tokens of a multi-token step: with fewer
// than 32 heads per 32-head slice (16, 48, ... heads) and an even q_len, one
// CTA takes two tokens x 16 heads, so that a chunk's rows are read by half as
// many CTAs.
bool pair_tokens(const mla_dims* cache_dims, int q_len) {
  return cache_dims->dtype == MLA_BF16 && cache_dims->heads % 32 != 0 && q_len % 2 == 0;
}

template <int kG, bool kPersist>
mla_status launch_split_tc(const CUtensorMap& tmap, const CUtensorMap& tmap_half,
                           const SplitParams& p, int heads, cudaStream_t s, const char* who) {
  using L = TcPlan<kG, kPersist>;
  static DeviceFlags attr_done;
  const int dev = current_device();
  if (!attr_done.test(dev)) {
    if (cudaFuncSetAttribute(split_tc_kernel<kG, kPersist>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(L::kSmem)) != cudaSuccess) {
      set_error("%s: cannot reserve %zu bytes of shared memory", who, L::kSmem);
      return MLA_ERR_CUDA;
    }
    attr_done.set(dev);
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 0;
  }
  // Paired tokens: 16-head slices, two query groups per CTA.  A persistent grid
  // has one CTA per SM.
  const dim3 grid = p.persist ? dim3(sms > 0 ? sms : 1)
                              : dim3(p.tpc == 2 ? heads / 16 : heads / kG, p.splits,
                                     p.tpc == 2 ? p.B / 2 : p.B);
  // A CTA whose chunk lies past its sequence's end would fetch its first boxes
  // for nothing; that costs little in a one-wave grid, but in several waves it
  // delays the CTAs behind it (measured: 64 ragged sequences, split 67.9 ->
  // 70.4 us with the early fetch everywhere).
  SplitParams q = p;
  q.fill_early = !p.persist && static_cast<long long>(grid.x) * grid.y * grid.z <= sms;
  launch_pdl(split_tc_kernel<kG, kPersist>, grid, dim3(L::kThreads), L::kSmem, s, tmap, tmap_half, q);
  return MLA_OK;
}
// How the split kernel cuts the rows: chunk rows, chunks per sequence, and
// whether the grid is persistent.
struct SplitPlan {
  int chunk, splits;
  bool persist;
};

int device_sms() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 148;
  }
  return sms;
}

// Rows per KV chunk and the resulting chunk count, and the launch form.
//  - One CTA per chunk.  With `requested` = 0 the count minimises a makespan
//    estimate (in units of cache rows): waves of CTAs over the SMs times (rows
//    per chunk + a fixed per-CTA cost), plus the combine's cost per chunk.  The
//    bf16 and FP8 kernels run one CTA per SM and work in 128-row tiles, and a
//    chunk's partial last tile costs about what a full one does (measured: 16
//    chunks of 256 rows beat 19 of 216 on 8 x 4096 rows), so for them a chunk's
//    rows count rounded up to whole tiles.  Chunks are multiples of
//    kChunkAlign rows.
//  - Persistent (the bf16 kernel with 16 heads per CTA), whenever that grid
//    would take more than one wave, or, with the count left to the library, when
//    its estimate is within 15 % of the best one-wave plan's (which balances only
//    if every sequence is full): one CTA per SM works through the chunks whose
//    first tile falls in its share of all tiles, so a CTA's start-up and
//    last-tile chain are paid once and its stream runs across chunk boundaries
//    (measured on 4 x 65536 rows at 128 chunks: 72.6 us in 3.4 waves).  Chunks
//    are whole tiles.  With `requested` = 0 the chunk minimises: the largest
//    share (all tiles over the SMs, counted for full-length sequences since the
//    lengths live on the device) plus one chunk less a tile (a share ends
//    mid-chunk), one start-up, each chunk's partial (32 KB written and read
//    again, about 56 rows' worth of traffic and epilogue; measured on 64 ragged
//    sequences: 16 chunks of 512 rows beat 22 of 384), and the combine's cost
//    per chunk.
SplitPlan plan_split_compute(const mla_dims* d, int requested, bool pair, long long sms);

// plan_split is a pure function of the dims, the request, the pairing, the two
// process-wide switches and the SM count; a decode step asks for it twice per
// call, and the search over chunk counts is the larger part of the step's host
// work (measured: 19.6 us of host time per mla_decode_step call with it, from
// Python with prepared arguments), so each thread keeps its last few answers.
SplitPlan plan_split(const mla_dims* d, int requested, bool pair = false) {
  struct Entry {
    int key[9];
    SplitPlan plan;
  };
  constexpr int kEntries = 8;
  thread_local Entry memo[kEntries];
  thread_local int filled = 0, next = 0;
  const long long sms = device_sms();
  const int key[9] = {d->batch, d->heads, d->s_max, d->dtype, requested, pair ? 1 : 0,
                      g_split_form.load(), g_split_parts.load(), static_cast<int>(sms)};
  for (int i = 0; i < filled; ++i) {
    bool same = true;
    for (int k = 0; k < 9; ++k) same = same && memo[i].key[k] == key[k];
    if (same) return memo[i].plan;
  }
  const SplitPlan plan = plan_split_compute(d, requested, pair, sms);
  Entry& e = memo[next];
  for (int k = 0; k < 9; ++k) e.key[k] = key[k];
  e.plan = plan;
  next = (next + 1) % kEntries;
  if (filled < kEntries) ++filled;
  return plan;
}

SplitPlan plan_split_compute(const mla_dims* d, int requested, bool pair, long long sms) {
  const int S = d->s_max;
  const int max_splits = (S + kChunkAlign - 1) / kChunkAlign;
  const bool tiled = d->dtype != MLA_F32;   // bf16 and FP8 kernels: one CTA per SM
  const long long groups = d->dtype == MLA_F32 ? d->heads : d->heads / tc_heads_per_cta(d);
  const long long per_split = pair ? static_cast<long long>(d->batch) * d->heads / 32
                                   : static_cast<long long>(d->batch) * groups;
  const bool can_persist = d->dtype == MLA_BF16 && !pair && tc_heads_per_cta(d) == 16;
  const long long slots = tiled ? sms : 4ll * sms;
  auto chunk_of = [&](int s, int align) {
    return ((S + s - 1) / s + align - 1) / align * align;
  };
  // One CTA per chunk.
  int np_chunk = 0, np_splits = 0;
  double np_cost = 1e300;
  {
    double& best = np_cost;
    const int lo = requested > 0 ? requested : 1, hi = requested > 0 ? requested : max_splits;
    for (int s = lo; s <= hi && s <= max_splits; ++s) {
      const int chunk = chunk_of(s, kChunkAlign);
      const int s_eff = (S + chunk - 1) / chunk;
      if (requested <= 0 && s_eff != s) continue;
      const long long waves = (per_split * s_eff + slots - 1) / slots;
      const int rows = tiled ? (chunk + kTileRows - 1) / kTileRows * kTileRows : chunk;
      const double cost = double(waves) * (rows + 96) + 4.0 * s_eff;
      if (cost < best) {
        best = cost;
        np_chunk = chunk;
        np_splits = s_eff;
      }
    }
    if (np_chunk == 0) {   // more chunks requested than row groups: one per 8 rows
      np_chunk = kChunkAlign;
      np_splits = (S + np_chunk - 1) / np_chunk;
    }
  }
  const bool np_one_wave = per_split * np_splits <= slots;
  const int form = g_split_form.load();
  if (!can_persist || form == 2 || (form == 0 && requested > 0 && np_one_wave))
    return {np_chunk, np_splits, false};
  // Persistent.
  const long long tt = groups * d->batch * ((S + kTileRows - 1) / kTileRows);   // tiles, at most
  const long long share = (tt + sms - 1) / sms;
  if (share + 1 > kMaxItems) return {np_chunk, np_splits, false};   // more chunks than a CTA holds
  int p_chunk = 0, p_splits = 0;
  double best = 1e300;
  const int lo = requested > 0 ? requested : 1, hi = requested > 0 ? requested : max_splits;
  for (int s = lo; s <= hi && s <= max_splits; ++s) {
    const int chunk = chunk_of(s, kTileRows);
    const int s_eff = (S + chunk - 1) / chunk;
    if (requested <= 0 && s_eff != s) continue;
    const long long ct = chunk / kTileRows;
    const long long max_tiles = share + ct - 1;
    const double cost = double(max_tiles) * kTileRows + 96 + 56.0 * ((max_tiles + ct - 1) / ct) +
                        4.0 * s_eff;
    if (cost < best) {
      best = cost;
      p_chunk = chunk;
      p_splits = s_eff;
    }
  }
  // The persistent estimate already counts its worst case (a share ending one
  // chunk short of a tile), and one CTA per chunk balances only when every
  // sequence is full, so near-ties (within 15 %) go to the persistent grid.
  if (p_chunk == 0 || (form == 0 && np_one_wave && best > 1.15 * np_cost))
    return {np_chunk, np_splits, false};
  return {p_chunk, p_splits, true};
}

int chunk_rows(const mla_dims* d, int requested, int* splits_out, bool pair = false) {
  const SplitPlan pl = plan_split(d, requested, pair);
  *splits_out = pl.splits;
  return pl.chunk;
}

// Partial outputs, their log-sum-exps, and (FP8 cache) the query images.
size_t workspace_bytes(const mla_dims* d, int splits) {
  const size_t n = size_t(d->batch) * splits * d->heads;
  const size_t o_bytes = (n * kDc * sizeof(float) + 255) / 256 * 256;
  const size_t lse_bytes = (n * sizeof(float) + 255) / 256 * 256;
  const size_t img = d->dtype == MLA_FP8_E4M3
                         ? (size_t(d->batch) * (d->heads / kHeadGroup) * kFp8QImage + 255) / 256 * 256
                         : 0;
  return o_bytes + lse_bytes + img;
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

extern "C" mla_status mla_debug_bounds_word(int32_t** word) {
  if (!word) {
    set_error("mla_debug_bounds_word: word is NULL");
    return MLA_ERR_INVALID_ARG;
  }
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_bounds_word);
  if (e != cudaSuccess) {
    set_error("mla_debug_bounds_word: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  *word = static_cast<int32_t*>(ptr);
  return MLA_OK;
}

extern "C" int32_t mla_built_with_checks(void) {
#ifdef MLA_CHECK
  return 1;
#else
  return 0;
#endif
}

extern "C" mla_status mla_decode_plan(const mla_dims* dims, int32_t requested, int32_t* splits,
                                      int32_t* chunk, int32_t* persistent) {
  mla_status st = check_dims(dims, "mla_decode_plan");
  if (st != MLA_OK) return st;
  const SplitPlan pl = plan_split(dims, requested);
  if (splits) *splits = pl.splits;
  if (chunk) *chunk = pl.chunk;
  if (persistent) *persistent = pl.persist ? 1 : 0;
  return MLA_OK;
}

extern "C" int32_t mla_decode_multi_num_splits(const mla_dims* dims, int32_t q_len,
                                               int32_t requested) {
  if (check_dims(dims, "mla_decode_multi_num_splits") != MLA_OK || q_len < 1) return 0;
  mla_dims qd = *dims;
  qd.batch = dims->batch * q_len;
  int splits = 0;
  chunk_rows(&qd, requested, &splits, pair_tokens(dims, q_len));
  return splits;
}

extern "C" size_t mla_decode_multi_workspace_bytes(const mla_dims* dims, int32_t q_len,
                                                   int32_t requested) {
  if (check_dims(dims, "mla_decode_multi_workspace_bytes") != MLA_OK || q_len < 1) return 0;
  mla_dims qd = *dims;
  qd.batch = dims->batch * q_len;
  int splits = 0;
  chunk_rows(&qd, requested, &splits, pair_tokens(dims, q_len));
  return workspace_bytes(&qd, splits);
}

extern "C" size_t mla_decode_workspace_bytes(const mla_dims* dims, int32_t requested) {
  if (check_dims(dims, "mla_decode_workspace_bytes") != MLA_OK) return 0;
  int splits = 0;
  chunk_rows(dims, requested, &splits);
  return workspace_bytes(dims, splits);
}

// Test hooks of the bf16 split kernel (mla_test_set_split_hooks); 0 in normal use.
static std::atomic<unsigned long long> g_hook_wait_ns{0};
static std::atomic<int> g_hook_stop_tiles{0};
static std::atomic<int32_t*> g_hook_debug{nullptr};
extern "C" void mla_test_set_split_form(int32_t form) { g_split_form.store(form); }

extern "C" mla_status mla_set_split_parts(int32_t parts) {
  if (parts != 0 && parts != 2) {
    set_error("mla_set_split_parts: parts must be 0 (the library's choice) or 2 (hi + lo)");
    return MLA_ERR_INVALID_ARG;
  }
  g_split_parts.store(parts);
  return MLA_OK;
}

extern "C" int32_t mla_decode_heads_per_cta(const mla_dims* dims) {
  if (check_dims(dims, "mla_decode_heads_per_cta") != MLA_OK) return 0;
  return dims->dtype == MLA_F32 ? 1 : tc_heads_per_cta(dims);
}

extern "C" void mla_test_set_split_debug(int32_t* records) { g_hook_debug.store(records); }

extern "C" void mla_test_set_split_hooks(uint64_t wait_ns, int32_t stop_after_tiles) {
  g_hook_wait_ns.store(wait_ns);
  g_hook_stop_tiles.store(stop_after_tiles > 0 ? stop_after_tiles : 0);
}

// Validates the arguments shared by the split and combine halves and fills the
// kernel parameters.  `dims` describes the cache (dims->batch sequences); with
// q_len query tokens per sequence the queries, partials and outputs have
// dims->batch * q_len rows, and chunks and workspace are planned for that many.
// Returns MLA_OK or the status to hand back.
static mla_status prepare(const char* who, const mla_dims* dims, int q_len, const void* q_abs,
                          const void* q_pe, const void* cache, const int32_t* lengths,
                          float softmax_scale, int32_t num_splits, void* workspace,
                          size_t ws_bytes, int32_t* dev_status, SplitParams* p) {
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (q_len < 1 || static_cast<long long>(dims->batch) * q_len > (1ll << 30)) {
    set_error("%s: q_len=%d must be >= 1 with batch*q_len <= 2^30", who, q_len);
    return MLA_ERR_INVALID_ARG;
  }
  const bool pair = pair_tokens(dims, q_len);
  mla_dims qd = *dims;   // one row of queries per (sequence, token)
  qd.batch = dims->batch * q_len;
  dims = &qd;
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
  const SplitPlan plan = plan_split(dims, num_splits, pair);
  const int splits = plan.splits, chunk = plan.chunk;
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
  p->q_img = dims->dtype == MLA_FP8_E4M3
                 ? reinterpret_cast<uint8_t*>(p->part_lse) + (n * sizeof(float) + 255) / 256 * 256
                 : nullptr;
  p->status = dev_status;
  p->B = dims->batch;
  p->q_len = q_len;
  p->tpc = pair ? 2 : 1;
  p->H = dims->heads;
  p->s_max = dims->s_max;
  p->splits = splits;
  p->chunk = chunk;
  p->scale_log2 = softmax_scale * kLog2e;
  p->fill_early = 0;
  p->persist = plan.persist ? 1 : 0;
  p->wait_ns = g_hook_wait_ns.load();
  p->debug = g_hook_debug.load();
  p->stop_after_tiles = g_hook_stop_tiles.load();
  return MLA_OK;
}

// The split half for q_len query tokens per cache sequence (1: ordinary decode).
static mla_status decode_split(const char* who, const mla_dims* dims, int q_len,
                               const void* q_abs, const void* q_pe, const void* cache,
                               const int32_t* lengths, float softmax_scale, int32_t num_splits,
                               void* workspace, size_t ws_bytes, int32_t* dev_status,
                               void* stream) {
  if (!q_abs || !q_pe || !cache) {
    set_error("%s: a required pointer is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  SplitParams p;
  mla_status st = prepare(who, dims, q_len, q_abs, q_pe, cache, lengths, softmax_scale,
                          num_splits, workspace, ws_bytes, dev_status, &p);
  if (st != MLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dims->dtype == MLA_FP8_E4M3) return launch_split_fp8(p, cache, s, who);
  if (dims->dtype == MLA_BF16) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) {
      set_error("%s: cuTensorMapEncodeTiled is not available from the driver", who);
      return MLA_ERR_CUDA;
    }
    // Two views of the cache [B * s_max rows, 576 columns]: 128-row boxes for
    // the score pass, 64-row boxes for the PV pass; 64 columns (128 bytes,
    // 128-byte swizzle) per box in both.  The score pass's L2 requests are
    // promoted to 256 bytes (a row's next box comes with it from HBM); the PV
    // pass re-reads rows already in L2 and asks for 128 bytes at a time
    // (measured: 256-byte promotion there costs 1.5 % on the large caches).
    CUtensorMap tmap, tmap_half;
    const cuuint64_t gdim[2] = {cuuint64_t(kRow), cuuint64_t(dims->batch) * dims->s_max};
    const cuuint64_t gstride[1] = {cuuint64_t(kRow) * 2};
    const cuuint32_t estride[2] = {1, 1};
    for (int v = 0; v < 2; ++v) {
      const cuuint32_t box[2] = {64, cuuint32_t(v == 0 ? kTileRows : kTileRows / 2)};
      CUresult r = enc(v == 0 ? &tmap : &tmap_half, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                       const_cast<void*>(cache), gdim, gstride, box, estride,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       v == 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                              : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) {
        set_error("%s: cuTensorMapEncodeTiled failed (%d)", who, int(r));
        return MLA_ERR_CUDA;
      }
    }
    const int per_cta = p.tpc == 2 ? 32 : tc_heads_per_cta(dims);
    st = per_cta == 64   ? launch_split_tc<64, false>(tmap, tmap_half, p, dims->heads, s, who)
         : per_cta == 32 ? launch_split_tc<32, false>(tmap, tmap_half, p, dims->heads, s, who)
         : p.persist     ? launch_split_tc<16, true>(tmap, tmap_half, p, dims->heads, s, who)
                         : launch_split_tc<16, false>(tmap, tmap_half, p, dims->heads, s, who);
    if (st != MLA_OK) return st;
  } else {
    dim3 grid(dims->heads, p.splits, p.B);
    split_f32_kernel<<<grid, kThreads, 0, s>>>(p);
  }
  return launch_status(who);
}

static mla_status decode_combine(const char* who, const mla_dims* dims, int q_len,
                                 const int32_t* lengths, int32_t num_splits,
                                 const void* workspace, size_t ws_bytes, float* o_c, float* lse,
                                 void* stream) {
  if (!o_c || !aligned16(o_c)) {
    set_error("%s: o_c must be a non-NULL 16-byte aligned pointer", who);
    return MLA_ERR_INVALID_ARG;
  }
  SplitParams p;
  mla_status st = prepare(who, dims, q_len, nullptr, nullptr, nullptr, lengths, 1.f, num_splits,
                          const_cast<void*>(workspace), ws_bytes, nullptr, &p);
  if (st != MLA_OK) return st;
  const int cw = combine_warps(p.splits);
  if (cw == 1)
    launch_pdl(combine_kernel, dim3(dims->heads, p.B, kDc / 128), dim3(32), 0,
               static_cast<cudaStream_t>(stream), p, o_c, lse);
  else
    launch_pdl(combine_warps_kernel, dim3(dims->heads, p.B, kDc / 128), dim3(32 * cw),
               size_t(cw) * (32 * sizeof(float4) + 2 * sizeof(float)),
               static_cast<cudaStream_t>(stream), p, o_c, lse);
  return launch_status(who);
}

extern "C" mla_status mla_decode_split(const mla_dims* dims, const void* q_abs, const void* q_pe,
                                       const void* cache, const int32_t* lengths,
                                       float softmax_scale, int32_t num_splits, void* workspace,
                                       size_t ws_bytes, int32_t* dev_status, void* stream) {
  return decode_split("mla_decode_split", dims, 1, q_abs, q_pe, cache, lengths, softmax_scale,
                      num_splits, workspace, ws_bytes, dev_status, stream);
}

extern "C" mla_status mla_decode_combine(const mla_dims* dims, const int32_t* lengths,
                                         int32_t num_splits, const void* workspace,
                                         size_t ws_bytes, float* o_c, float* lse, void* stream) {
  return decode_combine("mla_decode_combine", dims, 1, lengths, num_splits, workspace, ws_bytes,
                        o_c, lse, stream);
}

extern "C" mla_status mla_decode_attn_multi(const mla_dims* dims, int32_t q_len,
                                            const void* q_abs, const void* q_pe,
                                            const void* cache, const int32_t* lengths,
                                            float softmax_scale, int32_t num_splits,
                                            void* workspace, size_t ws_bytes, float* o_c,
                                            float* lse, int32_t* dev_status, void* stream) {
  const char* who = "mla_decode_attn_multi";
  if (!o_c || !aligned16(o_c)) {
    set_error("%s: o_c must be a non-NULL 16-byte aligned pointer", who);
    return MLA_ERR_INVALID_ARG;
  }
  // Check everything the combine needs before the split is enqueued.
  SplitParams p;
  mla_status st = prepare(who, dims, q_len, q_abs, q_pe, cache, lengths, softmax_scale,
                          num_splits, workspace, ws_bytes, dev_status, &p);
  if (st != MLA_OK) return st;
  st = decode_split(who, dims, q_len, q_abs, q_pe, cache, lengths, softmax_scale, num_splits,
                    workspace, ws_bytes, dev_status, stream);
  if (st != MLA_OK) return st;
  return decode_combine(who, dims, q_len, lengths, num_splits, workspace, ws_bytes, o_c, lse,
                        stream);
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

// Largest batch x heads for which mla_decode_step fuses the combine with W_UV.
constexpr long long kFusedTailMax = 256;

// Bytes of the cache mla_decode_step asks L2 to fetch during its absorb kernel.
constexpr long long kPrefetchBudget = 16ll << 20;

// Whether the device can address `ptr` directly: 1 for device or managed
// memory, 2 for page-locked host memory (mapped into the device's address
// space), 0 otherwise.  Pageable host memory is refused: a kernel touching it
// would fault.
static int device_addressable(const void* ptr) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return 1;
  return a.type == cudaMemoryTypeHost && a.devicePointer != nullptr ? 2 : 0;
}

// The whole step for q_len tokens per sequence (mla_decode_step: q_len = 1).
static mla_status decode_step(const char* who, const mla_dims* dims, int q_len,
                              const void* q_nope, const void* q_rope, const void* w_uk,
                              const int32_t* positions, double rope_base, const void* cache,
                              const int32_t* lengths, float softmax_scale, int32_t num_splits,
                              const void* w_uv, void* workspace, size_t ws_bytes, float* q_abs,
                              float* q_pe, float* o_c, float* lse, float* out,
                              int32_t* dev_status, void* stream) {
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (q_len < 1 || static_cast<long long>(dims->batch) * q_len > (1ll << 30)) {
    set_error("%s: q_len=%d must be >= 1 with batch*q_len <= 2^30", who, q_len);
    return MLA_ERR_INVALID_ARG;
  }
  mla_dims qd = *dims;   // the query side: one row per (sequence, token)
  qd.batch = dims->batch * q_len;
  if (!o_c || !out || !w_uv || !aligned16(o_c) || !aligned16(out) || !aligned16(w_uv)) {
    set_error("%s: o_c, out and w_uv must be non-NULL 16-byte aligned pointers", who);
    return MLA_ERR_INVALID_ARG;
  }
  // The per-step inputs and the output may live in page-locked host memory.
  const void* step_io[5] = {q_nope, q_rope, positions, lengths, out};
  const char* step_io_name[5] = {"q_nope", "q_rope", "positions", "lengths", "out"};
  int kind[5] = {-1, -1, -1, -1, -1};
  for (int i = 0; i < 5; ++i) {
    if (step_io[i] && (kind[i] = device_addressable(step_io[i])) == 0) {
      set_error("%s: %s is not memory the device can address (pageable host memory?); use "
                "device memory or page-locked host memory", who, step_io_name[i]);
      return MLA_ERR_INVALID_ARG;
    }
  }
  if (dims->dtype == MLA_F32) {
    // The fp32 path has no fused tail: the three calls in order.
    st = mla_absorb_q(&qd, q_nope, q_rope, w_uk, positions, rope_base, q_abs, q_pe, stream);
    if (st != MLA_OK) return st;
    st = q_len == 1 ? mla_decode_attn(dims, q_abs, q_pe, cache, lengths, softmax_scale,
                                      num_splits, workspace, ws_bytes, o_c, lse, dev_status,
                                      stream)
                    : mla_decode_attn_multi(dims, q_len, q_abs, q_pe, cache, lengths,
                                            softmax_scale, num_splits, workspace, ws_bytes, o_c,
                                            lse, dev_status, stream);
    if (st != MLA_OK) return st;
    return mla_out_proj(&qd, o_c, w_uv, out, stream);
  }
  // Validate everything before the first launch, so an argument error leaves
  // nothing half-enqueued.
  SplitParams p;
  st = prepare(who, dims, q_len, q_abs, q_pe, cache, lengths, softmax_scale, num_splits,
               workspace, ws_bytes, dev_status, &p);
  if (st != MLA_OK) return st;
  CachePrefetch pf{};
  bool single_wave = false;
  pf.cache = static_cast<const uint8_t*>(cache);
  pf.lengths = lengths;
  pf.B = dims->batch;
  pf.s_max = dims->s_max;
  pf.chunk = p.chunk;
  pf.splits = p.splits;
  pf.row_bytes = kRow * (dims->dtype == MLA_FP8_E4M3 ? 1 : 2);
  // Up to one tile per chunk, and at most kPrefetchBudget bytes in all: more
  // than the absorb's duration of HBM time only competes with the absorb's own
  // weight loads (and past L2's capacity is evicted before use).  Measured on
  // 8 x 4096 rows: step 20.8 -> 20.0 us with 64 or 128 rows per chunk, 22.2 us
  // with whole chunks; 4 x 65536 rows: 64 -> 83 us with 1024 rows per chunk.
  {
    const long long nchunk = static_cast<long long>(pf.B) * pf.splits;
    long long rows = p.chunk < kTileRows ? p.chunk : kTileRows;
    const long long budget_rows = kPrefetchBudget / (nchunk * pf.row_bytes);
    if (rows > budget_rows) rows = budget_rows / 8 * 8;
    pf.rows = static_cast<int>(rows);
    // Only when every split CTA runs in the first wave: data fetched for later
    // waves only competes with the first one (measured: 64 ragged sequences in
    // three waves, step 103 -> 123 us).
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      sms = 0;
    }
    const long long ctas =
        static_cast<long long>(p.splits) *
        (p.tpc == 2 ? static_cast<long long>(p.B / 2) * (dims->heads / 16)
                    : static_cast<long long>(p.B) * (dims->heads / tc_heads_per_cta(dims)));
    single_wave = !p.persist && ctas <= sms;
    if (pf.rows <= 0 || !single_wave) pf.cache = nullptr;
  }
  // The early launch of the absorb pays only with a one-wave decode grid: with
  // several waves the early decode CTAs crowd out the previous step's tail
  // (measured: 64 ragged sequences, step 103 -> 122 us with it).
  st = absorb_q(who, &qd, q_nope, q_rope, w_uk, positions, rope_base, q_abs, q_pe, stream, pf,
                single_wave, kind[0] < 0 ? -1 : kind[0] == 2 ? 1 : 0);
  if (st != MLA_OK) return st;
  st = decode_split(who, dims, q_len, q_abs, q_pe, cache, lengths, softmax_scale, num_splits,
                    workspace, ws_bytes, dev_status, stream);
  if (st != MLA_OK) return st;
  // The fused tail reads W_UV[h] once per sequence: for small batches that
  // saves a kernel boundary, for large ones the separate combine and out_proj,
  // which read W_UV once, win (measured: B*H = 128 fused 20.3 against 22.8 us;
  // B*H = 1024 102.6 against 99.5 us; B*H = 4096 501 against 446 us).
  if (static_cast<long long>(qd.batch) * dims->heads > kFusedTailMax) {
    st = decode_combine(who, dims, q_len, lengths, num_splits, workspace, ws_bytes, o_c, lse,
                        stream);
    if (st != MLA_OK) return st;
    return mla_out_proj(&qd, o_c, w_uv, out, stream);
  }
  launch_pdl(combine_out_kernel, dim3(dims->heads, qd.batch, kDv / kOutRows), dim3(128), 0,
             static_cast<cudaStream_t>(stream), p, static_cast<const __nv_bfloat16*>(w_uv), o_c,
             lse, out);
  return launch_status(who);
}

extern "C" mla_status mla_decode_step(const mla_dims* dims, const void* q_nope, const void* q_rope,
                                      const void* w_uk, const int32_t* positions, double rope_base,
                                      const void* cache, const int32_t* lengths, float softmax_scale,
                                      int32_t num_splits, const void* w_uv, void* workspace,
                                      size_t ws_bytes, float* q_abs, float* q_pe, float* o_c,
                                      float* lse, float* out, int32_t* dev_status, void* stream) {
  return decode_step("mla_decode_step", dims, 1, q_nope, q_rope, w_uk, positions, rope_base,
                     cache, lengths, softmax_scale, num_splits, w_uv, workspace, ws_bytes, q_abs,
                     q_pe, o_c, lse, out, dev_status, stream);
}

extern "C" mla_status mla_decode_step_multi(const mla_dims* dims, int32_t q_len,
                                            const void* q_nope, const void* q_rope,
                                            const void* w_uk, const int32_t* positions,
                                            double rope_base, const void* cache,
                                            const int32_t* lengths, float softmax_scale,
                                            int32_t num_splits, const void* w_uv,
                                            void* workspace, size_t ws_bytes, float* q_abs,
                                            float* q_pe, float* o_c, float* lse, float* out,
                                            int32_t* dev_status, void* stream) {
  return decode_step("mla_decode_step_multi", dims, q_len, q_nope, q_rope, w_uk, positions,
                     rope_base, cache, lengths, softmax_scale, num_splits, w_uv, workspace,
                     ws_bytes, q_abs, q_pe, o_c, lse, out, dev_status, stream);
}

// ------------------------------------------------------- fixed scratch, no allocation
// Some hosts cannot allocate device memory when they decode: an inference engine that
// reserved all device memory for its own pool at start-up (a cudaMalloc would fail or
// break its accounting), or a latency-critical loop where cudaMalloc and cudaFree would
// synchronise the device.  mla_decode_attn_noalloc serves them with the chunk partials
// in this fixed array instead of a caller-supplied workspace.  Every GPU that loads the
// library reserves MLA_NOALLOC_SCRATCH_BYTES for it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
// Device address of the array per device ordinal, and the context it belongs to.
struct NoallocAddr {
  unsigned long long ctx_id;
  void* ptr;
};
NoallocAddr g_noalloc_addr[kMaxDevices] = {};

// The array's name in host code is only a host-side handle, so the device address
// is asked from the runtime with the device current.  The address belongs to the
// library's module as loaded in one context: after cudaDeviceReset, or with another
// context current on the same device, the module is loaded again and the array may
// move.  So the address is kept together with the context's process-unique ID and
// asked again whenever the current context differs (or its ID is unknown).
mla_status noalloc_scratch(const char* who, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    set_error("%s: cudaGetDevice failed", who);
    return MLA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("%s: device ordinal %d is beyond the %d the library tracks", who, dev, kMaxDevices);
    return MLA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocAddr& a = g_noalloc_addr[dev];
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || a.ctx_id != ctx || !a.ptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      set_error("%s: cudaGetSymbolAddress of the fixed scratch failed: %s", who,
                cudaGetErrorString(e));
      return MLA_ERR_CUDA;
    }
    // The lookup may have created the device's primary context: take its ID now.
    a.ctx_id = current_context_id();
    a.ptr = ptr;
  }
  *out = a.ptr;
  return MLA_OK;
}
}  // namespace

extern "C" mla_status mla_decode_attn_noalloc(const mla_dims* dims, const void* q_abs,
                                              const void* q_pe, const void* cache,
                                              const int32_t* lengths, float softmax_scale,
                                              int32_t num_splits, float* o_c, float* lse,
                                              int32_t* dev_status, void* stream) {
  const char* who = "mla_decode_attn_noalloc";
  mla_status st = check_dims(dims, who);
  if (st != MLA_OK) return st;
  if (num_splits < 0) {
    set_error("%s: num_splits must be >= 0", who);
    return MLA_ERR_INVALID_ARG;
  }
  int splits = 0;
  chunk_rows(dims, num_splits, &splits);
  const size_t need = workspace_bytes(dims, splits);
  if (need > MLA_NOALLOC_SCRATCH_BYTES) {
    set_error("%s: %d sequences x %d heads x %d chunks need %zu bytes of scratch, more than "
              "the fixed %zu; use mla_decode_attn with a workspace, or fewer chunks",
              who, dims->batch, dims->heads, splits, need, size_t(MLA_NOALLOC_SCRATCH_BYTES));
    return MLA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  st = noalloc_scratch(who, &scratch);
  if (st != MLA_OK) return st;
  // Every partial the combine reads is written by this call's split kernel, so
  // nothing left in the array by an earlier call needs clearing.
  return mla_decode_attn(dims, q_abs, q_pe, cache, lengths, softmax_scale, num_splits, scratch,
                         size_t(MLA_NOALLOC_SCRATCH_BYTES), o_c, lse, dev_status, stream);
}
