// moe_permute_noalloc: the permute with its scratch in a fixed device array
// inside the library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory: code running inside a host
// framework whose pool allocator owns all device memory and forbids other
// cudaMalloc calls, or latency-critical paths where cudaMalloc's implicit
// device-wide synchronisation is unacceptable.  For them the counting-sort
// tables of the permute live in g_permute_scratch below.  The caller still
// passes every input and output buffer.
//
// Rules of the array:
//  * kNoAllocScratchBytes (8 MiB) on every GPU that loads the library, held
//    until the process exits.  A call whose tables need more is refused
//    (MOE_ERR_WORKSPACE) before anything is launched.
//  * In host code the name g_permute_scratch is a host-side stand-in, not a
//    device address.  The device address is looked up once per device with
//    that device current (cudaGetSymbolAddress) on the first call and
//    cached; that first call should come before any stream capture.  The
//    cached address is that of the device's context at the time: after a
//    cudaDeviceReset it is stale, and the entry point must not be called
//    on that device again in the same process.
//  * All calls on a device share the array and it keeps the last call's
//    contents.  Nothing in it has to start at zero: each call writes every
//    table entry before reading it.  Calls whose work overlaps on the GPU
//    (unordered streams) race on the array.
//  * No cudaMalloc, cudaFree or allocating library routine is called.
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char
    g_permute_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_permute_scratch on the current device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool ptr_ok(const void* p, bool need16) {
  if (p == nullptr) return false;
  const uintptr_t u = reinterpret_cast<uintptr_t>(p);
  return need16 ? (u & 15u) == 0 : (u & 3u) == 0;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_noalloc(
    const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
    int32_t capped, void* x_sorted, int32_t* row_of, int32_t* sorted_token,
    int32_t* group_offsets, int32_t* uniq_offsets, int32_t* uniq_tokens,
    int32_t* expand_idx, int32_t* n_dropped, moe_stream_t stream) {
  using namespace moe;
  const moe_status_t st = moe_validate_config(cfg);
  if (st != MOE_OK) return st;
  const size_t need = permute_scratch_bytes(cfg->T, cfg->E, cfg->k, cfg->S);
  if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  if (!ptr_ok(group_offsets, false) || !ptr_ok(uniq_offsets, false) ||
      !ptr_ok(n_dropped, false))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 &&
      (!ptr_ok(x, true) || !ptr_ok(topk_idx, false) ||
       !ptr_ok(x_sorted, true) || !ptr_ok(row_of, false) ||
       !ptr_ok(sorted_token, false) || !ptr_ok(uniq_tokens, false) ||
       !ptr_ok(expand_idx, false)))
    return MOE_ERR_INVALID_ARG;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
  Carve cv(base);
  const PermuteScratch ws =
      carve_permute_scratch(cv, cfg->T, cfg->E, cfg->k, cfg->S);
  const int64_t cap = capped ? capacity_rows(*cfg) : -1;
  const cudaError_t e = launch_permute(
      *cfg, x, topk_idx, cap, x_sorted, row_of, sorted_token, group_offsets,
      uniq_offsets, uniq_tokens, expand_idx, n_dropped, ws, nullptr, stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
