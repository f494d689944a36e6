// moe_permute_noalloc: the token permutation without a caller workspace.
//
// Some callers cannot hand this library any device memory beyond their
// inputs and outputs: code that runs with a fixed memory budget reserved at
// start-up, plugins inside a host framework that forbids allocating outside
// its own pools, and latency-critical paths that must not call cudaMalloc /
// cudaFree (those calls may synchronise the whole device).  This entry point
// serves them.  The only scratch the permutation needs -- one counter per
// (tile of 2048 token-slot pairs, expert) -- lives in the fixed array below,
// which every GPU that loads the library holds until the process exits.
//
// Limits and sharing:
//  * at most kScratchInts counters: ceil(T*k / 2048) * E <= 65536, otherwise
//    the call returns MOE_ERR_UNSUPPORTED before enqueuing anything;
//  * every call shares the array and it keeps the last call's contents.
//    Each call writes every counter it later reads, so nothing has to start
//    at zero; but calls whose kernels overlap on the GPU (different streams,
//    no ordering between them) race on the array and corrupt each other;
//  * expert ids outside [0, E) are skipped (their row_map entry is -1)
//    without being reported: there is no workspace to hold an error word;
//  * every call looks up the array's address on the current device
//    (cudaGetSymbolAddress) and keeps no copy of it, so no address survives a
//    cudaDeviceReset or any other re-creation of the device's context.  The
//    first call on a device may load the library's device code there, so
//    make that first call before any stream capture on the device.
#include "common.cuh"

namespace moe {
namespace {

constexpr int64_t kScratchInts = MOE_PERMUTE_NOALLOC_MAX_COUNTERS;  // 256 KB per device

static __device__ __align__(256) int32_t g_perm_scratch[kScratchInts];

// Device address of g_perm_scratch in the current device's context.  Looked
// up on every call: a cached address would outlive the context it was read
// in (a cudaDeviceReset makes a new one) and then point at freed memory.
// Returns nullptr and the CUDA error on failure.
int32_t* scratch_on_current_device(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_perm_scratch);
  return *err == cudaSuccess ? static_cast<int32_t*>(p) : nullptr;
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const moe_config* cfg, const void* x,
                                          const int32_t* topk_idx, const uint8_t* keep,
                                          void* x_perm, int32_t* row_map,
                                          int32_t* expert_offsets, moe_stream_t stream) {
  using namespace moe;
  if (cfg == nullptr) return MOE_ERR_INVALID_ARG;
  size_t ws_unused = 0;
  const moe_status v = moe_workspace_size(cfg, &ws_unused);  // validates the configuration
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  if (c.pad_to_capacity) return MOE_ERR_INVALID_ARG;  // padding rows come from the map
  const int64_t np = static_cast<int64_t>(c.num_tokens) * c.topk;
  const int64_t ntiles = perm_tiles(np);
  if (ntiles * c.num_experts > kScratchInts) return MOE_ERR_UNSUPPORTED;
  if (expert_offsets == nullptr || !aligned(expert_offsets, 4)) return MOE_ERR_INVALID_ARG;
  if (np > 0) {
    if (x == nullptr || topk_idx == nullptr || x_perm == nullptr || row_map == nullptr)
      return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(x_perm, 16) || !aligned(topk_idx, 4) || !aligned(row_map, 4))
      return MOE_ERR_INVALID_ARG;
  }
  cudaError_t err = cudaSuccess;
  int32_t* scratch = scratch_on_current_device(&err);
  if (scratch == nullptr) return MOE_ERR_CUDA;
  if (np == 0) {
    return cudaMemsetAsync(expert_offsets, 0, (c.num_experts + 1) * sizeof(int32_t), stream) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  }
  if (launch_perm_index(np, c.num_experts, topk_idx, keep, scratch, row_map, nullptr,
                        expert_offsets, nullptr, nullptr, stream) != cudaSuccess ||
      launch_perm_copy(c.num_tokens, c.hidden, c.topk, c.dtype, x, row_map, x_perm, stream) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
