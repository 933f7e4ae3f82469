// dcp_prune_step_noalloc: the prune step for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a custom device allocator's callback (re-entering the
// allocator would deadlock), engines that reserve all device memory up front and forbid any later allocation, and
// thin host programs in other languages that have no device allocator of their own.  They cannot provide the
// workspace dcp_prune_step needs.  This entry point uses a fixed scratch array compiled into the library instead.
// The array lives in device memory of every GPU that loads the library, until the process exits.  Its size is
// DCP_NOALLOC_WORKSPACE_BYTES; a cache and config whose workspace (dcp_workspace_size) is larger are rejected.
//
// In host code the array's name is only a host-side stand-in, not a device address, so its device address is
// looked up (cudaGetSymbolAddress) on the first call made in each CUDA context (one per device for the runtime's
// primary contexts), with that context current, and passed to the kernels.  Make that first call before any stream
// capture.  The lookup is remembered per context id, so a context created later (after cudaDeviceReset, say) gets a
// lookup of its own instead of a stale address.
//
// Every call shares the one array and leaves its contents behind.  The part that must start at zero, the scan's
// 256-byte control block (its completion counter and the atomically folded plane checks), is cleared on the stream
// once the call's arguments have passed every host check, right before its first kernel; a refused call launches
// nothing.  Calls whose work overlaps on the GPU (different streams, or different threads on one device) race on the
// array: order them.
#include <cuda.h>

#include <mutex>

#include "dcp_internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_ws[DCP_NOALLOC_WORKSPACE_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

constexpr int kMaxContexts = 64;
struct AddressCache {
  std::mutex m;
  bool resolved = false;
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
  int n = 0;
  unsigned long long ctx_id[kMaxContexts];
  void* addr[kMaxContexts];
};
AddressCache g_cache;

// The id of the calling thread's current context (the driver's own unique id for the process lifetime), or 0 when
// the thread has no current context yet.  The driver entry points come through the runtime, so the library does not
// link the driver library itself.
bool current_context_id(AddressCache& c, unsigned long long* id) {
  if (!c.resolved) {
    void *f1 = nullptr, *f2 = nullptr;
    cudaDriverEntryPointQueryResult q1{}, q2{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return false;
    c.get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    c.get_id = reinterpret_cast<CtxGetIdFn>(f2);
    c.resolved = true;
  }
  CUcontext ctx = nullptr;
  if (c.get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return ctx == nullptr || c.get_id(ctx, id) == CUDA_SUCCESS;
}

dcp_status noalloc_address(void** out) {
  std::lock_guard<std::mutex> guard(g_cache.m);
  unsigned long long id = 0;
  if (!current_context_id(g_cache, &id)) return DCP_ECUDA;
  for (int i = 0; id && i < g_cache.n; ++i)
    if (g_cache.ctx_id[i] == id) {
      *out = g_cache.addr[i];
      return DCP_OK;
    }
  void* p = nullptr;  // the lookup makes the device's primary context current when the thread had none
  if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) return DCP_ECUDA;
  if (!current_context_id(g_cache, &id) || id == 0) return DCP_ECUDA;
  const int slot = g_cache.n < kMaxContexts ? g_cache.n++ : (int)(id % kMaxContexts);
  g_cache.ctx_id[slot] = id;
  g_cache.addr[slot] = p;
  *out = p;
  return DCP_OK;
}

}  // namespace

extern "C" dcp_status dcp_prune_step_noalloc(const dcp_cache* cache, const dcp_config* cfg, const float* x0hat_dev,
                                             const float* xref_dev, int32_t d, int32_t evict_slot,
                                             int32_t evict_first_frame, int32_t q0_prev, int32_t q0,
                                             const uint8_t* head_is_static_dev, int32_t* kept_dev,
                                             int32_t* kept_host_pinned, void* stream) {
  const size_t need = dcp_workspace_size(cache, cfg);  // 0 for an invalid cache or config
  if (need == 0 || need > (size_t)DCP_NOALLOC_WORKSPACE_BYTES) return DCP_EINVAL;
  void* ws = nullptr;
  const dcp_status rc = noalloc_address(&ws);
  if (rc != DCP_OK) return rc;
  return dcp::prune_step_cleared(cache, cfg, x0hat_dev, xref_dev, d, evict_slot, evict_first_frame, q0_prev, q0,
                                 head_is_static_dev, kept_dev, kept_host_pinned, ws,
                                 (size_t)DCP_NOALLOC_WORKSPACE_BYTES, sizeof(dcp::Ctrl), stream);
}
