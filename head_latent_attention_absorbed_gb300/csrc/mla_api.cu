// Host-side helpers of the C ABI: status strings, the per-thread error detail,
// argument checks shared by the three calls.
#include <stdarg.h>
#include <stdio.h>

#include "mla_common.cuh"

namespace mla {

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status check_dims(const mla_dims* d, const char* who) {
  if (!d) {
    set_error("%s: dims is NULL", who);
    return MLA_ERR_INVALID_ARG;
  }
  if (d->batch < 1 || d->heads < 1 || d->s_max < 1) {
    set_error("%s: batch=%d heads=%d s_max=%d must all be >= 1", who, d->batch, d->heads,
              d->s_max);
    return MLA_ERR_INVALID_ARG;
  }
  if (d->d_c != kDc || d->d_rope != kDr || d->d_nope != kDn || d->d_v != kDv) {
    set_error("%s: only d_c=512 d_rope=64 d_nope=128 d_v=128 are built (got %d %d %d %d)", who,
              d->d_c, d->d_rope, d->d_nope, d->d_v);
    return MLA_ERR_UNSUPPORTED;
  }
  if (d->dtype != MLA_F32 && d->dtype != MLA_BF16 && d->dtype != MLA_FP8_E4M3) {
    set_error("%s: dtype %d is not MLA_F32, MLA_BF16 or MLA_FP8_E4M3", who, d->dtype);
    return MLA_ERR_UNSUPPORTED;
  }
  if (d->dtype != MLA_F32 && d->heads % kHeadGroup != 0) {
    set_error("%s: bf16 and FP8 kernels need heads to be a multiple of %d (got %d)", who, kHeadGroup,
              d->heads);
    return MLA_ERR_UNSUPPORTED;
  }
  // Row indices of the cache must fit a 32-bit TMA coordinate.
  if (static_cast<long long>(d->batch) * d->s_max >= (1ll << 31)) {
    set_error("%s: batch*s_max = %lld rows exceeds 2^31", who,
              static_cast<long long>(d->batch) * d->s_max);
    return MLA_ERR_UNSUPPORTED;
  }
  return MLA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    cudaGetLastError();
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// A driver function by name and ABI version through the runtime's entry-point
// query; NULL if the driver does not provide it.
static void* driver_entry(const char* name, unsigned int version) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return f;
  cudaGetLastError();
  return nullptr;
}

unsigned long long current_context_id() {
  static const auto get_current =
      reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(driver_entry("cuCtxGetCurrent", 4000));
  static const auto get_id =
      reinterpret_cast<PFN_cuCtxGetId_v12000>(driver_entry("cuCtxGetId", 12000));
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

static std::atomic<int> g_launch_overlap{1};

bool launch_overlap_enabled() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }

mla_status launch_status(const char* who) {
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("%s: launch failed: %s", who, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace mla

extern "C" const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
  }
  return "MLA_ERR_UNKNOWN";
}

extern "C" const char* mla_last_error_message(void) { return mla::g_last_error; }

extern "C" void mla_set_launch_overlap(int32_t enable) {
  mla::g_launch_overlap.store(enable != 0 ? 1 : 0);
}
