// moe_permute_noalloc: moe_permute for callers that cannot hand the library a
// device workspace.
//
// Some callers can't allocate device memory at the point where they permute:
// plugin-style interfaces that give an operator only its input and output
// buffers, and processes whose device memory is reserved up front by their own
// pool allocator, where an extra cudaMalloc would fail or fragment that pool.
// For them this entry point keeps moe_permute's per-block expert counts in a
// fixed array of device memory that belongs to the library itself, so the call
// allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kNoallocScratchInts * 4 bytes) until the process exits.
// Its address is looked up once per device, on the first call made while that
// device is current; make that first call before any stream capture.  The
// lookup is tied to the device's context: after cudaDeviceReset() the array
// lives in a new context at a possibly different address, so the first call
// made in the new context looks it up again (also before any capture).  All
// calls share the one array, so calls whose kernels overlap on the GPU (two
// streams, or two host threads) race on it and must be serialised by the
// caller.  The counts are fully written by every call before they are read, so
// nothing left from an earlier call is ever used.
#include <cuda.h>

#include <mutex>

#include "internal.h"

static __device__ __align__(256) int32_t g_permute_scratch[32768];

namespace moe {
namespace {

// 32768 counters = 128 KB.  A call needs (number of count blocks) * E counters
// plus 64 of slack, with ceil(T / 256) count blocks for T <= 65536 and 256
// above: E <= 64 always fits; E = 256 fits up to T = 32512 tokens.
constexpr size_t kNoallocScratchInts = sizeof(g_permute_scratch) / sizeof(int32_t);

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int32_t *g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};  // context the address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current context (0 if there is none yet
// or the driver cannot tell); ids are never reused within a process.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array on the current device: looked up on
// the first call in the device's context, kept for the later ones.
cudaError_t scratch_address(int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  const unsigned long long ctx = current_context_id();
  if (g_scratch_ptr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t *>(ptr);
    // the lookup made the device's primary context current if it was not yet
    g_scratch_ctx[dev] = ctx != 0 ? ctx : current_context_id();
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_noalloc(const uint16_t *x, int64_t ldx,
                                            const int32_t *topk_idx, int T, int d, int E, int k,
                                            int align, int capacity, uint16_t *x_sorted,
                                            int64_t ld_xs, int64_t rows_cap,
                                            int32_t *group_sizes, int32_t *kept_counts,
                                            int32_t *group_offsets, int32_t *sorted_to_flat,
                                            int32_t *flat_to_sorted, int32_t *dev_status,
                                            moe_stream_t stream) {
  const size_t cap_bytes = moe::kNoallocScratchInts * sizeof(int32_t);
  const size_t need = moe_permute_workspace_bytes(T, E);
  if (T >= 0 && E > 0 && need > cap_bytes) {
    moe::set_error("moe_permute_noalloc: T=%d, E=%d need %zu bytes of scratch; the built-in "
                   "array holds %zu (use moe_permute with a workspace)",
                   T, E, need, cap_bytes);
    return MOE_ERR_UNSUPPORTED;
  }
  int32_t *scratch = nullptr;
  const cudaError_t e = moe::scratch_address(&scratch);
  if (e != cudaSuccess) {
    moe::set_error("moe_permute_noalloc: cannot find the scratch array on this device: %s",
                   cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return moe_permute(x, ldx, topk_idx, T, d, E, k, align, capacity, x_sorted, ld_xs, rows_cap,
                     group_sizes, kept_counts, group_offsets, sorted_to_flat, flat_to_sorted,
                     scratch, cap_bytes, dev_status, stream);
}
