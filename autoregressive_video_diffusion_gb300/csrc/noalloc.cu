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
// looked up once per device (cudaGetSymbolAddress, with that device current) on the first call made with that
// device current, and passed to the kernels.  Make that first call before any stream capture.
//
// Every call shares the one array and leaves its contents behind; the parts that must start at zero (the scan's
// control block and its look-back tile states) are cleared on the stream at the start of each call.  Calls whose
// work overlaps on the GPU (different streams, or different threads on one device) race on the array: order them.
#include "dcp_internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_ws[DCP_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void* g_noalloc_addr[kMaxDevices] = {nullptr};

dcp_status noalloc_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DCP_ECUDA;
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) return DCP_ECUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
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
  const int64_t C = (int64_t)cfg->tokens_per_frame * cfg->frames_per_chunk;
  const dcp::Layout lay = dcp::make_layout(C, (int64_t)cache->L * cache->H, cfg->frames_per_chunk,
                                           cfg->n_temporal_pairs, cfg->max_frames);
  if (cudaMemsetAsync(ws, 0, lay.ell, (cudaStream_t)stream) != cudaSuccess) return DCP_ECUDA;
  return dcp_prune_step(cache, cfg, x0hat_dev, xref_dev, d, evict_slot, evict_first_frame, q0_prev, q0,
                        head_is_static_dev, kept_dev, kept_host_pinned, ws, (size_t)DCP_NOALLOC_WORKSPACE_BYTES,
                        stream);
}
