// moe_permute_noalloc.cu -- moe_permute for callers that cannot allocate.
//
// Some callers of this library cannot call cudaMalloc or any allocating
// routine: code that runs inside a framework whose allocator is not reachable
// from the call site, a host that forbids device allocation after start-up,
// or a call made from a place where an allocation could block or fail.  They
// can still pass their own input and output buffers, but not the scratch
// workspace moe_permute needs for its per-chunk expert histogram.  This entry
// point uses a fixed scratch array in the library's own device memory instead.
//
// The scratch is a file-scope __device__ array of MOE_PERMUTE_NOALLOC_MAX_SCRATCH
// bytes (1 MiB).  Every GPU that loads the library holds it until the process
// exits.  The permute's histogram takes 4 bytes per expert for every chunk of
// 512 pairs, so the array serves P = T*K <= 512 * floor(2^18 / E) pairs
// (131072 at E = 1024, 524288 at E = 256).  All calls share it, so two calls whose kernels overlap on the GPU
// (different streams without ordering between them) race on it.  The array
// keeps the previous call's contents; nothing needs clearing, because the count
// kernel writes every histogram entry the later kernels read.
#include "moe_common.cuh"

namespace {

static __device__ __align__(256) int32_t g_permute_scratch[MOE_PERMUTE_NOALLOC_MAX_SCRATCH / 4];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// on every call, with the calling thread's current device: a cached address
// would go stale if the caller reset the device or its primary context was
// rebuilt, since the library's module (and the array) is then loaded anew.
int scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return moe::set_error(MOE_ERR_CUDA,
                          "moe_permute_noalloc: cudaGetSymbolAddress of the scratch failed: %s",
                          cudaGetErrorString(e));
  }
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t* topk_ids, const void* x_bf16, int T, int K,
                                   int E, int H, int32_t* expert_offsets, int32_t* sorted_pair,
                                   int32_t* pair_to_row, void* x_perm_bf16, void* stream) {
  moe::clear_error();
  const size_t need = moe_permute_workspace_size(T, K, E);
  if (need > static_cast<size_t>(MOE_PERMUTE_NOALLOC_MAX_SCRATCH))
    return moe::set_error(MOE_ERR_WORKSPACE,
                          "moe_permute_noalloc: T=%d, K=%d, E=%d need %zu bytes of scratch, more "
                          "than the fixed %d; use moe_permute with a workspace",
                          T, K, E, need, MOE_PERMUTE_NOALLOC_MAX_SCRATCH);
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_permute(topk_ids, x_bf16, T, K, E, H, expert_offsets, sorted_pair, pair_to_row,
                     x_perm_bf16, scratch, static_cast<size_t>(MOE_PERMUTE_NOALLOC_MAX_SCRATCH),
                     stream);
}
