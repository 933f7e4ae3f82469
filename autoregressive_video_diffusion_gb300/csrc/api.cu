// Host side of libdcp: argument validation, workspace layout and the launch sequence of each entry point.
// The entry points and their contracts are documented in include/dcp.h.
#include <atomic>
#include <cmath>
#include <cstring>

#include "dcp_internal.cuh"

using namespace dcp;

namespace {

cudaEvent_t g_ev_after_scan = nullptr;
cudaEvent_t g_ev_after_gather = nullptr;

struct Derived {
  int64_t C, sink_rows, win_row0, n_planes;
  int esize;
  int T_s;
  Layout lay;
};

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

dcp_status check_cache_cfg(const dcp_cache* c, const dcp_config* g, Derived* d) {
  if (!c || !g) return DCP_EINVAL;
  if (!c->k || !c->v || !c->hist_len || !c->hist_t || !c->status) return DCP_EINVAL;
  if (c->L < 1 || c->H < 1 || c->D < 2 || (c->D & 1)) return DCP_EINVAL;
  if (c->dtype != DCP_BF16 && c->dtype != DCP_F32) return DCP_EINVAL;
  const int es = c->dtype == DCP_BF16 ? 2 : 4;
  // rows of at most 4 KiB (a CTA of the streaming kernels covers whole rows), a multiple of 16 bytes
  if (((int64_t)c->D * es) % 16 || (int64_t)c->D * es > 4096) return DCP_EINVAL;
  if (!aligned(c->k, 16) || !aligned(c->v, 16) || !aligned(c->hist_len, 4) || !aligned(c->hist_t, 4) ||
      !aligned(c->status, 4))
    return DCP_EINVAL;
  if (g->tokens_per_frame < 1 || g->frames_per_chunk < 1 || g->sink_chunks < 0 || g->window_chunks < 0)
    return DCP_EINVAL;
  const int64_t C = (int64_t)g->tokens_per_frame * g->frames_per_chunk;
  if (C > (int64_t(1) << 30)) return DCP_EINVAL;
  if (g->n_temporal_pairs < 0 || g->n_temporal_pairs > c->D / 2) return DCP_EINVAL;
  // the gather keeps the leaving chunk's cos/sin table (F x n_t entries of 16 bytes) in shared memory
  if ((int64_t)g->frames_per_chunk * g->n_temporal_pairs * 16 > 100 * 1024) return DCP_EINVAL;
  if (g->pair_layout != 0 || g->rephase_sink != 0) return DCP_EINVAL;
  if (!std::isfinite(g->rope_base) || !(g->rope_base > 0.0)) return DCP_EINVAL;
  if (!std::isfinite(g->g_recent_R) || !std::isfinite(g->g_span_S)) return DCP_EINVAL;
  if (g->g_mode != 0 && g->g_mode != 1) return DCP_EINVAL;
  if (g->g_recent_R < (double)g->window_chunks * g->frames_per_chunk) return DCP_EINVAL;
  if (g->g_mode == 0 && g->g_span_S < g->g_recent_R) return DCP_EINVAL;
  if (g->g_mode == 1 && g->g_span_S < 0.0) return DCP_EINVAL;
  if (g->keep_rule < 0 || g->keep_rule > 2) return DCP_EINVAL;
  if ((g->reindex_mode != 0 && g->reindex_mode != 1) || g->reserved != 0) return DCP_EINVAL;
  if (!std::isfinite(g->gamma)) return DCP_EINVAL;
  if (g->max_frames < 1) return DCP_EINVAL;
  if (c->hist_cap < 0 || c->hist_cap > INT32_MAX) return DCP_EINVAL;
  const int64_t sink_rows = (int64_t)g->sink_chunks * C;
  const int64_t need = sink_rows + c->hist_cap + ((int64_t)g->window_chunks + 1) * C;
  if (c->cap < need) return DCP_EINVAL;
  const int64_t T_s = (int64_t)g->sink_chunks * g->frames_per_chunk;
  if (T_s > INT32_MAX) return DCP_EINVAL;
  // offsets inside one chunk's rows and inside the history region are 32-bit in the kernels
  if (C * c->D * es >= (int64_t(1) << 31) || c->hist_cap * c->D * es >= (int64_t(1) << 31)) return DCP_EINVAL;
  if (d) {
    d->C = C;
    d->sink_rows = sink_rows;
    d->win_row0 = sink_rows + c->hist_cap;
    d->n_planes = (int64_t)c->L * c->H;
    d->esize = es;
    d->T_s = (int)T_s;
    d->lay = make_layout(C, d->n_planes, g->frames_per_chunk, g->n_temporal_pairs, g->max_frames);
  }
  return DCP_OK;
}

dcp_status check_ws(const void* ws, size_t bytes, size_t need) {
  if (!ws || !aligned(ws, 256) || bytes < need) return DCP_EINVAL;
  return DCP_OK;
}

dcp_status check_eviction(const dcp_config* g, const Derived& d, int32_t evict_slot, int32_t evict_first_frame,
                          int32_t q0) {
  if (evict_slot < 0 || evict_slot > g->window_chunks) return DCP_EINVAL;
  if (evict_first_frame < d.T_s) return DCP_EINVAL;
  if ((int64_t)evict_first_frame + g->frames_per_chunk > q0) return DCP_EINVAL;
  if (q0 > g->max_frames) return DCP_EINVAL;
  return DCP_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

void choose_tiling(int32_t d, const float* x0, const float* xr, int* lpt, int* tile) {
  const int nvec = d / 4;
  const bool vec_ok = d % 4 == 0 && nvec >= 1 && nvec <= 32 && (nvec & (nvec - 1)) == 0 && aligned(x0, 16) &&
                      aligned(xr, 16);
  if (vec_ok) {
    *lpt = nvec;
    *tile = 1024 / nvec < kMaxTile ? 1024 / nvec : kMaxTile;
  } else {
    *lpt = 0;
    *tile = 64;
  }
}

// Scan parameters shared by the calls that work on a cache.
ScanParams cache_scan_params(const dcp_cache* c, const dcp_config* g, const Derived& d, void* ws) {
  ScanParams sp{};
  sp.gamma = g->gamma;
  sp.keep_rule = g->keep_rule;
  sp.g_identity = g->reindex_mode == 1 ? 1 : 0;
  sp.ctrl = at<Ctrl>(ws, 0);
  sp.bits = at<uint32_t>(ws, d.lay.bits);
  sp.status = c->status;
  sp.hist_len = c->hist_len;
  sp.n_planes = (int32_t)d.n_planes;
  sp.n_plane_slices = (int32_t)((d.n_planes + kThreads - 1) / kThreads);
  sp.hist_cap = c->hist_cap;
  sp.trig_g = at<float4>(ws, d.lay.trig_g);
  sp.rot_g = at<uint8_t>(ws, d.lay.rot_g);
  sp.trig_h = at<float4>(ws, d.lay.trig_h);
  sp.rot_h = at<uint8_t>(ws, d.lay.rot_h);
  sp.n_t = g->n_temporal_pairs;
  sp.base = g->rope_base;
  sp.R = g->g_recent_R;
  sp.S = g->g_span_S;
  sp.g_mode = g->g_mode;
  sp.T_s = d.T_s;
  return sp;
}

void finish_tables(ScanParams& sp) {
  const int entries = (sp.g_frames + (sp.h_hi - sp.h_lo)) * sp.n_t;
  int per = (entries + kTableTargetCTAs - 1) / kTableTargetCTAs;
  per = per < kTableMinEntries ? kTableMinEntries : (per > kTableEntries ? kTableEntries : per);
  sp.tbl_per = per;
  sp.n_trig_blocks = (entries + per - 1) / per;
}

// 32-byte vector accesses need 32-byte aligned rows and bases; otherwise the kernels use 16-byte vectors.
int vector_bytes(const dcp_cache* c, int row_bytes) {
  return (row_bytes % 32 == 0 && aligned(c->k, 32) && aligned(c->v, 32)) ? 32 : 16;
}

GatherParams gather_params(const dcp_cache* c, const dcp_config* g, const Derived& d, void* ws, int32_t slot,
                           const uint8_t* head_is_static, int32_t evict_first_frame) {
  GatherParams gp{};
  gp.k = static_cast<char*>(c->k);
  gp.v = static_cast<char*>(c->v);
  gp.row_bytes = c->D * d.esize;
  gp.plane_bytes = c->cap * (int64_t)gp.row_bytes;
  gp.vb = vector_bytes(c, gp.row_bytes);
  gp.src_row0 = d.win_row0 + (int64_t)slot * d.C;
  gp.dst_row0 = d.sink_rows;
  gp.n_planes = (int32_t)d.n_planes;
  gp.ctrl = at<Ctrl>(ws, 0);
  gp.idx = at<int32_t>(ws, d.lay.idx);
  gp.head_is_static = head_is_static;
  gp.hist_len = c->hist_len;
  gp.hist_t = c->hist_t;
  gp.evict_first_frame = evict_first_frame;
  gp.trig_g = at<float4>(ws, d.lay.trig_g);
  gp.rot_g = at<uint8_t>(ws, d.lay.rot_g);
  gp.T = g->tokens_per_frame;
  gp.n_t = g->n_temporal_pairs;
  gp.dtype = c->dtype;
  gp.n_frames = g->frames_per_chunk;
  gp.no_turn = 0;  // set by the callers that know q0 (set_turn)
  gp.status = c->status;
  return gp;
}

RephaseParams rephase_params(const dcp_cache* c, const dcp_config* g, const Derived& d, void* ws, int h_lo,
                             int h_hi) {
  RephaseParams rp{};
  rp.k = static_cast<char*>(c->k);
  rp.row_bytes = c->D * d.esize;
  rp.plane_bytes = c->cap * (int64_t)rp.row_bytes;
  rp.vb = vector_bytes(c, rp.row_bytes);
  rp.nvt = (2 * g->n_temporal_pairs * d.esize + rp.vb - 1) / rp.vb;
  rp.hist_row0 = d.sink_rows;
  rp.n_planes = (int32_t)d.n_planes;
  rp.ctrl = at<Ctrl>(ws, 0);
  rp.hist_len = c->hist_len;
  rp.hist_t = c->hist_t;
  rp.trig_h = at<float4>(ws, d.lay.trig_h);
  rp.rot_h = at<uint8_t>(ws, d.lay.rot_h);
  rp.n_t = g->n_temporal_pairs;
  rp.dtype = c->dtype;
  rp.h_lo = h_lo;
  rp.h_hi = h_hi;
  rp.status = c->status;
  return rp;
}

dcp_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? DCP_OK : DCP_ECUDA; }

// No kept key of the leaving chunk changes phase: g is the identity on every offset q0 - t of the chunk's frames, which
// holds when the oldest non-sink offset already fits the span (g is then the identity everywhere) or when the chunk's
// oldest offset is within the recent range R.  Read-time re-index moves keys unturned.
// This decision is load-bearing, not only a choice of speed: when it holds, the scan builds no cos/sin table for the
// chunk and no gather form turns any key (the staged gather takes its copy-only form; the register-staged one skips
// its turn under no_turn).  It is exact because it restates g's closed form: g(delta) = delta for delta <= R, and everywhere when
// delta_max = q0 - T_s <= span end, so t~(t) = t for every frame of the chunk (the chunk's oldest offset is
// q0 - evict_first_frame, its largest).  The GPU sweep draws steps on both sides of each boundary
// (q0 - evict_first_frame = R, R + 1; q0 - T_s = span end, span end + 1) and compares them with the oracle.
bool chunk_keeps_phase(const dcp_config* g, const Derived& d, int32_t evict_first_frame, int32_t q0) {
  if (g->reindex_mode == 1 || g->n_temporal_pairs == 0) return true;
  const double span_end = g->g_mode == 0 ? g->g_span_S : g->g_recent_R + g->g_span_S;
  return (double)(q0 - d.T_s) <= span_end || (double)(q0 - evict_first_frame) <= g->g_recent_R;
}

// The turn of the leaving chunk's keys for a gather at q0: none (no_turn: the scan builds no table for the chunk), or
// the scan's table CTAs build it.
void set_turn(GatherParams& gp, ScanParams& sp, const dcp_config* g, const Derived& d, int32_t evict_first_frame,
              int32_t q0) {
  gp.no_turn = chunk_keeps_phase(g, d, evict_first_frame, q0) ? 1 : 0;
  sp.g_frames = gp.no_turn ? 0 : g->frames_per_chunk;
}

// ------------------------------------------------------------------------------------------ snapshot helpers
dcp_status check_live(const dcp_config* g, uint32_t live_slots, int* n_live) {
  if (g->window_chunks + 1 > 32) return DCP_EINVAL;
  if (g->window_chunks + 1 < 32 && (live_slots >> (g->window_chunks + 1)) != 0) return DCP_EINVAL;
  int n = 0;
  for (int s = 0; s < 32; ++s) n += (live_slots >> s) & 1u;
  *n_live = n;
  return DCP_OK;
}

// Where a kernel can read a caller's buffer: device memory as it is; page-locked host memory (cudaHostAlloc,
// cudaHostRegister) through its device address (the kernel then reads over the host link); nullptr for memory the
// device cannot reach (pageable host memory), which the caller gets back as DCP_EINVAL.
const void* device_view(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

// Device address of a host image: page-locked host memory (cudaHostAlloc, cudaHostRegister) that the device reaches
// through unified addressing.
char* image_device_ptr(const void* img) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, img) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  return static_cast<char*>(a.devicePointer);
}

int64_t img_i64(const void* img, int64_t off) {
  int64_t x;
  std::memcpy(&x, static_cast<const char*>(img) + off, 8);
  return x;
}

int32_t img_i32(const void* img, int64_t off) {
  int32_t x;
  std::memcpy(&x, static_cast<const char*>(img) + off, 4);
  return x;
}

// ------------------------------------------------------------------------------------------ paged caches
struct PagedView {
  Paging pg;
  const int32_t* window_blocks;
  int64_t n_blocks;
};

// A paged cache seen as a dcp_cache (for the shared checks and parameters) plus its addressing.  The shadow's cap
// is the row count of the contiguous layout with the same regions; the kernels never use it for a paged cache.
dcp_status paged_view(const dcp_paged_cache* c, const dcp_config* g, dcp_cache* shadow, PagedView* pv) {
  if (!c || !g) return DCP_EINVAL;
  if (!c->hist_blocks || !c->window_blocks || !aligned(c->hist_blocks, 4) || !aligned(c->window_blocks, 4))
    return DCP_EINVAL;
  if (c->block_size < 1 || c->n_blocks < 1 || c->n_blocks > INT32_MAX) return DCP_EINVAL;
  if (c->layout != DCP_PAGED_HND && c->layout != DCP_PAGED_NHD) return DCP_EINVAL;
  if (g->tokens_per_frame < 1 || g->frames_per_chunk < 1 || g->window_chunks < 0 || g->sink_chunks < 0)
    return DCP_EINVAL;
  const int64_t C = (int64_t)g->tokens_per_frame * g->frames_per_chunk;
  if (C % c->block_size || c->hist_cap < 0 || c->hist_cap % c->block_size) return DCP_EINVAL;
  std::memset(shadow, 0, sizeof(*shadow));
  shadow->k = c->k_pool;
  shadow->v = c->v_pool;
  shadow->L = c->L;
  shadow->H = c->H;
  shadow->D = c->D;
  shadow->dtype = c->dtype;
  shadow->hist_cap = c->hist_cap;
  shadow->cap = (int64_t)g->sink_chunks * C + c->hist_cap + ((int64_t)g->window_chunks + 1) * C;
  shadow->hist_len = c->hist_len;
  shadow->hist_t = c->hist_t;
  shadow->status = c->status;
  if (c->H < 1 || c->D < 2) return DCP_EINVAL;
  const int64_t rb = (int64_t)c->D * (c->dtype == DCP_BF16 ? 2 : 4);
  const int64_t bs = c->block_size, H = c->H;
  Paging pg{};
  pg.H = c->H;
  pg.bs = c->block_size;
  if (c->layout == DCP_PAGED_HND) {
    pg.s_row = rb;
    pg.s_head = bs * rb;
  } else {
    pg.s_row = H * rb;
    pg.s_head = rb;
  }
  pg.s_block = H * bs * rb;
  pg.s_layer = c->n_blocks * pg.s_block;
  pg.hist_blocks = c->hist_blocks;
  pv->pg = pg;
  pv->window_blocks = c->window_blocks;
  pv->n_blocks = c->n_blocks;
  return DCP_OK;
}

dcp_status prune_step_impl(const dcp_cache* cache, const PagedView* pv, const dcp_config* cfg, const float* x0hat,
                           const float* xref, int32_t dd, int32_t evict_slot, int32_t evict_first_frame,
                           int32_t q0_prev, int32_t q0, const uint8_t* head_is_static, int32_t* kept_dev,
                           int32_t* kept_host_pinned, void* ws, size_t ws_bytes, void* stream,
                           size_t ws_clear_bytes = 0);

// Read-time re-index: the scan kernel's table CTAs build the turn t -> t~(t; q0) for frames [T_s, q0) and its plane
// checks find the longest history; the read kernel follows on the stream.
dcp_status read_impl(const dcp_cache* cache, const PagedView* pv, const dcp_config* cfg, int32_t q0, int32_t plane0,
                     int32_t n_planes, void* out, void* ws, size_t ws_bytes, void* stream) {
  Derived d;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK || cfg->reindex_mode != 1) return DCP_EINVAL;
  if (q0 < d.T_s || q0 > cfg->max_frames) return DCP_EINVAL;
  if (plane0 < 0 || n_planes < 1 || (int64_t)plane0 + n_planes > d.n_planes) return DCP_EINVAL;
  if (!out || !aligned(out, 16) || check_ws(ws, ws_bytes, d.lay.total) != DCP_OK) return DCP_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  ScanParams sp = cache_scan_params(cache, cfg, d, ws);
  sp.g_identity = 0;
  sp.want_rephase = 1;
  sp.evict_first_frame = d.T_s;
  sp.g_frames = q0 - d.T_s;
  sp.trig_g = at<float4>(ws, d.lay.trig_h);
  sp.rot_g = at<uint8_t>(ws, d.lay.rot_h);
  sp.h_lo = sp.h_hi = d.T_s;
  sp.q0 = q0;
  sp.q0_prev = q0;
  finish_tables(sp);
  ReadParams rp{};
  rp.k = static_cast<char*>(cache->k);
  rp.row_bytes = cache->D * d.esize;
  rp.plane_bytes = cache->cap * (int64_t)rp.row_bytes;
  rp.vb = (vector_bytes(cache, rp.row_bytes) == 32 && aligned(out, 32)) ? 32 : 16;
  rp.nvt = (2 * cfg->n_temporal_pairs * d.esize + rp.vb - 1) / rp.vb;
  rp.vpr = rp.row_bytes / rp.vb;
  rp.hist_row0 = d.sink_rows;
  rp.plane0 = plane0;
  rp.n_planes = n_planes;
  rp.hist_cap = cache->hist_cap;
  rp.out = static_cast<char*>(out);
  rp.ctrl = at<Ctrl>(ws, 0);
  rp.hist_len = cache->hist_len;
  rp.hist_t = cache->hist_t;
  rp.trig = sp.trig_g;
  rp.rot = sp.rot_g;
  rp.f_lo = d.T_s;
  rp.f_hi = q0;
  rp.n_t = cfg->n_temporal_pairs;
  rp.dtype = cache->dtype;
  rp.status = cache->status;
  if (pv) {
    rp.pg = pv->pg;
    sp.tbl_a = pv->pg.hist_blocks;
    sp.n_tbl_a = (int32_t)(cache->hist_cap / pv->pg.bs);
    sp.n_blocks = pv->n_blocks;
    sp.n_tbl_slices = (sp.n_tbl_a + kThreads - 1) / kThreads;
  }
  dcp_status rc = cuda_ok(launch_scan(sp, st));
  if (rc != DCP_OK) return rc;
  return cuda_ok(launch_read(rp, st, pv != nullptr));
}

SnapParams snap_params(const dcp_cache* c, const dcp_config* g, const Derived& d, uint32_t live_slots, int n_live,
                       char* img_dev, size_t img_bytes, void* ws, int dir) {
  SnapParams p{};
  p.dir = dir;
  p.k = static_cast<char*>(c->k);
  p.v = static_cast<char*>(c->v);
  p.row_bytes = c->D * d.esize;
  p.plane_bytes = c->cap * (int64_t)p.row_bytes;
  p.n_planes = (int32_t)d.n_planes;
  p.sink_rows = d.sink_rows;
  p.hist_cap = c->hist_cap;
  p.C = d.C;
  p.live_slots = live_slots;
  p.n_live = n_live;
  p.hist_len = c->hist_len;
  p.hist_t = c->hist_t;
  p.img = img_dev;
  p.img_bytes = (int64_t)img_bytes;
  p.L = c->L;
  p.H = c->H;
  p.D = c->D;
  p.dtype = c->dtype;
  p.cap = c->cap;
  p.window_chunks = g->window_chunks;
  p.ctrl = at<Ctrl>(ws, 0);
  p.plane_off = at<int64_t>(ws, d.lay.plane_off);
  p.status = c->status;
  return p;
}

}  // namespace

namespace dcp {
dcp_status prune_step_cleared(const dcp_cache* cache, const dcp_config* cfg, const float* x0hat, const float* xref,
                              int32_t dd, int32_t evict_slot, int32_t evict_first_frame, int32_t q0_prev, int32_t q0,
                              const uint8_t* head_is_static, int32_t* kept_dev, int32_t* kept_host_pinned, void* ws,
                              size_t ws_bytes, size_t ws_clear_bytes, void* stream) {
  return prune_step_impl(cache, nullptr, cfg, x0hat, xref, dd, evict_slot, evict_first_frame, q0_prev, q0,
                         head_is_static, kept_dev, kept_host_pinned, ws, ws_bytes, stream, ws_clear_bytes);
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];  // zero until first read on that device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    const int n = cache[dev].load(std::memory_order_relaxed);
    if (n) return n;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (cached) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}
}  // namespace dcp

extern "C" {

size_t dcp_workspace_size(const dcp_cache* cache, const dcp_config* cfg) {
  Derived d;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK) return 0;
  return d.lay.total;
}

size_t dcp_score_workspace_size(int32_t n_tok) {
  if (n_tok < 1 || n_tok > (1 << 30)) return 0;
  return make_layout(n_tok, 0, 0, 0, 0).total;
}

dcp_status dcp_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(Ctrl)) return DCP_EINVAL;
  return cuda_ok(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

dcp_status dcp_score_mask(const float* x0hat, const float* xref, int32_t n_tok, int32_t d, float gamma,
                          int32_t keep_rule, uint64_t random_stream, float* ell_dev, uint8_t* mask_dev,
                          int32_t* idx_dev, int32_t* kept_dev, int32_t* status_dev, void* ws, size_t ws_bytes,
                          void* stream) {
  if (!x0hat || !xref || !status_dev || n_tok < 1 || n_tok > (1 << 30) || d < 1 || !std::isfinite(gamma) ||
      keep_rule < 0 || keep_rule > 2)
    return DCP_EINVAL;
  if (!aligned(status_dev, 4) || (idx_dev && !aligned(idx_dev, 4)) || (ell_dev && !aligned(ell_dev, 4)) ||
      (kept_dev && !aligned(kept_dev, 4)) || !aligned(x0hat, 4) || !aligned(xref, 4))
    return DCP_EINVAL;
  const Layout lay = make_layout(n_tok, 0, 0, 0, 0);
  if (check_ws(ws, ws_bytes, lay.total) != DCP_OK) return DCP_EINVAL;
  x0hat = static_cast<const float*>(device_view(x0hat));  // device memory or page-locked host memory
  xref = static_cast<const float*>(device_view(xref));
  if (!x0hat || !xref) return DCP_EINVAL;
  ScanParams sp{};
  sp.x0hat = x0hat;
  sp.xref = xref;
  sp.n_tok = n_tok;
  sp.d = d;
  sp.gamma = gamma;
  sp.keep_rule = keep_rule;
  sp.random_stream = random_stream;
  choose_tiling(d, x0hat, xref, &sp.lpt, &sp.tile);
  sp.n_tiles = (n_tok + sp.tile - 1) / sp.tile;
  sp.ell_out = ell_dev;
  sp.mask_out = mask_dev;
  sp.idx_out = idx_dev;
  sp.ctrl = at<Ctrl>(ws, 0);
  sp.bits = at<uint32_t>(ws, lay.bits);
  sp.status = status_dev;
  sp.kept_dev = kept_dev;
  return cuda_ok(launch_scan(sp, (cudaStream_t)stream));
}

dcp_status dcp_compact_layers(const dcp_cache* cache, const dcp_config* cfg, int32_t evict_slot,
                              int32_t evict_first_frame, const uint8_t* mask, const uint8_t* head_is_static,
                              int32_t q0, int32_t* kept_dev, void* ws, size_t ws_bytes, void* stream) {
  Derived d;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK) return DCP_EINVAL;
  if (check_eviction(cfg, d, evict_slot, evict_first_frame, q0) != DCP_OK) return DCP_EINVAL;
  if (!mask || check_ws(ws, ws_bytes, d.lay.total) != DCP_OK) return DCP_EINVAL;
  if (kept_dev && !aligned(kept_dev, 4)) return DCP_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  ScanParams sp = cache_scan_params(cache, cfg, d, ws);
  sp.mask_in = mask;
  sp.n_tok = (int32_t)d.C;
  sp.tile = kMaxTile;
  sp.lpt = 0;
  sp.n_tiles = (int32_t)((d.C + sp.tile - 1) / sp.tile);
  sp.mask_out = at<uint8_t>(ws, d.lay.mask);
  sp.idx_out = at<int32_t>(ws, d.lay.idx);
  sp.kept_dev = kept_dev;
  sp.update_cache = 1;
  sp.head_is_static = head_is_static;
  sp.evict_first_frame = evict_first_frame;
  sp.q0 = q0;
  sp.q0_prev = q0;
  GatherParams gp = gather_params(cache, cfg, d, ws, evict_slot, head_is_static, evict_first_frame);
  set_turn(gp, sp, cfg, d, evict_first_frame, q0);
  if (head_is_static) sp.dyn_list = at<int32_t>(ws, d.lay.dyn);  // the scan lists the receiving planes
  finish_tables(sp);
  dcp_status rc = cuda_ok(launch_scan(sp, st));
  if (rc != DCP_OK) return rc;
  if (head_is_static) gp.dyn_list = at<int32_t>(ws, d.lay.dyn);
  return cuda_ok(launch_gather(gp, st, true, false));
}

dcp_status dcp_rope_reindex(const dcp_cache* cache, const dcp_config* cfg, int32_t q0_prev, int32_t q0, void* ws,
                            size_t ws_bytes, void* stream) {
  Derived d;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK) return DCP_EINVAL;
  if (q0_prev > q0 || q0 > cfg->max_frames || q0_prev < d.T_s) return DCP_EINVAL;
  if (check_ws(ws, ws_bytes, d.lay.total) != DCP_OK) return DCP_EINVAL;
  // no key changes phase (or, with read-time re-index, keys keep their own frame's phase)
  if (q0_prev == q0 || cfg->n_temporal_pairs == 0 || cfg->reindex_mode == 1) return DCP_OK;
  cudaStream_t st = (cudaStream_t)stream;
  ScanParams sp = cache_scan_params(cache, cfg, d, ws);
  sp.want_rephase = 1;
  sp.h_lo = d.T_s;
  sp.h_hi = q0;
  sp.q0 = q0;
  sp.q0_prev = q0_prev;
  finish_tables(sp);
  dcp_status rc = cuda_ok(launch_scan(sp, st));
  if (rc != DCP_OK) return rc;
  return cuda_ok(launch_rephase(rephase_params(cache, cfg, d, ws, sp.h_lo, sp.h_hi), st, true, false));
}

dcp_status dcp_prune_step(const dcp_cache* cache, const dcp_config* cfg, const float* x0hat, const float* xref,
                          int32_t dd, int32_t evict_slot, int32_t evict_first_frame, int32_t q0_prev, int32_t q0,
                          const uint8_t* head_is_static, int32_t* kept_dev, int32_t* kept_host_pinned, void* ws,
                          size_t ws_bytes, void* stream) {
  return prune_step_impl(cache, nullptr, cfg, x0hat, xref, dd, evict_slot, evict_first_frame, q0_prev, q0,
                         head_is_static, kept_dev, kept_host_pinned, ws, ws_bytes, stream);
}

size_t dcp_paged_workspace_size(const dcp_paged_cache* cache, const dcp_config* cfg) {
  dcp_cache shadow;
  PagedView pv;
  if (paged_view(cache, cfg, &shadow, &pv) != DCP_OK) return 0;
  return dcp_workspace_size(&shadow, cfg);
}

dcp_status dcp_paged_prune_step(const dcp_paged_cache* cache, const dcp_config* cfg, const float* x0hat,
                                const float* xref, int32_t dd, int32_t evict_slot, int32_t evict_first_frame,
                                int32_t q0_prev, int32_t q0, const uint8_t* head_is_static, int32_t* kept_dev,
                                int32_t* kept_host_pinned, void* ws, size_t ws_bytes, void* stream) {
  dcp_cache shadow;
  PagedView pv;
  if (paged_view(cache, cfg, &shadow, &pv) != DCP_OK) return DCP_EINVAL;
  return prune_step_impl(&shadow, &pv, cfg, x0hat, xref, dd, evict_slot, evict_first_frame, q0_prev, q0,
                         head_is_static, kept_dev, kept_host_pinned, ws, ws_bytes, stream);
}

uint32_t dcp_abi_paged_cache_size(void) { return (uint32_t)sizeof(dcp_paged_cache); }

dcp_status dcp_phase_table(const dcp_config* g, int32_t q0, int32_t frame_lo, int32_t frame_hi, float* out,
                           void* stream) {
  if (!g || !out || !aligned(out, 16)) return DCP_EINVAL;
  if (g->tokens_per_frame < 1 || g->frames_per_chunk < 1 || g->sink_chunks < 0 || g->window_chunks < 0)
    return DCP_EINVAL;
  if (g->n_temporal_pairs < 1 || !std::isfinite(g->rope_base) || !(g->rope_base > 0.0)) return DCP_EINVAL;
  if (!std::isfinite(g->g_recent_R) || !std::isfinite(g->g_span_S) || (g->g_mode != 0 && g->g_mode != 1))
    return DCP_EINVAL;
  if (g->g_recent_R < (double)g->window_chunks * g->frames_per_chunk) return DCP_EINVAL;
  if ((g->g_mode == 0 && g->g_span_S < g->g_recent_R) || (g->g_mode == 1 && g->g_span_S < 0.0)) return DCP_EINVAL;
  const int64_t T_s = (int64_t)g->sink_chunks * g->frames_per_chunk;
  if (T_s > INT32_MAX || frame_lo < T_s || frame_lo > frame_hi || frame_hi > q0) return DCP_EINVAL;
  const int64_t n = (int64_t)(frame_hi - frame_lo) * g->n_temporal_pairs;
  if (n > INT32_MAX) return DCP_EINVAL;
  return cuda_ok(launch_phase_table(reinterpret_cast<float4*>(out), frame_lo, (int32_t)n, g->n_temporal_pairs,
                                    g->rope_base, g->g_recent_R, g->g_span_S, g->g_mode, (int32_t)T_s, q0,
                                    (cudaStream_t)stream));
}

dcp_status dcp_read_history_keys(const dcp_cache* cache, const dcp_config* cfg, int32_t q0, int32_t plane0,
                                 int32_t n_planes, void* out_dev, void* ws, size_t ws_bytes, void* stream) {
  return read_impl(cache, nullptr, cfg, q0, plane0, n_planes, out_dev, ws, ws_bytes, stream);
}

dcp_status dcp_paged_read_history_keys(const dcp_paged_cache* cache, const dcp_config* cfg, int32_t q0,
                                       int32_t plane0, int32_t n_planes, void* out_dev, void* ws, size_t ws_bytes,
                                       void* stream) {
  dcp_cache shadow;
  PagedView pv;
  if (paged_view(cache, cfg, &shadow, &pv) != DCP_OK) return DCP_EINVAL;
  return read_impl(&shadow, &pv, cfg, q0, plane0, n_planes, out_dev, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {

// ws_clear_bytes > 0: the first ws_clear_bytes of the workspace are zeroed on the stream after every host check has
// passed and before the first kernel (a workspace shared by every call, whose start must be zero).
dcp_status prune_step_impl(const dcp_cache* cache, const PagedView* pv, const dcp_config* cfg, const float* x0hat,
                           const float* xref, int32_t dd, int32_t evict_slot, int32_t evict_first_frame,
                           int32_t q0_prev, int32_t q0, const uint8_t* head_is_static, int32_t* kept_dev,
                           int32_t* kept_host_pinned, void* ws, size_t ws_bytes, void* stream,
                           size_t ws_clear_bytes) {
  Derived d;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK) return DCP_EINVAL;
  if (check_eviction(cfg, d, evict_slot, evict_first_frame, q0) != DCP_OK) return DCP_EINVAL;
  if (q0_prev > q0 || q0_prev < d.T_s) return DCP_EINVAL;
  if (!x0hat || !xref || dd < 1 || !aligned(x0hat, 4) || !aligned(xref, 4)) return DCP_EINVAL;
  if (kept_dev && !aligned(kept_dev, 4)) return DCP_EINVAL;
  if (kept_host_pinned && !aligned(kept_host_pinned, 4)) return DCP_EINVAL;
  if (check_ws(ws, ws_bytes, d.lay.total) != DCP_OK) return DCP_EINVAL;
  // score rows in device memory, or in page-locked host memory read over the host link by the scan kernel
  x0hat = static_cast<const float*>(device_view(x0hat));
  xref = static_cast<const float*>(device_view(xref));
  if (!x0hat || !xref) return DCP_EINVAL;
  int32_t* kept_host = nullptr;  // page-locked: written by the scan kernel itself
  if (kept_host_pinned) {
    kept_host = static_cast<int32_t*>(const_cast<void*>(device_view(kept_host_pinned)));
    if (!kept_host) return DCP_EINVAL;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const bool rephase = q0_prev != q0 && cfg->n_temporal_pairs > 0 && cfg->reindex_mode == 0;
  ScanParams sp = cache_scan_params(cache, cfg, d, ws);
  sp.x0hat = x0hat;
  sp.xref = xref;
  sp.n_tok = (int32_t)d.C;
  sp.d = dd;
  choose_tiling(dd, x0hat, xref, &sp.lpt, &sp.tile);
  sp.n_tiles = (int32_t)((d.C + sp.tile - 1) / sp.tile);
  sp.ell_out = at<float>(ws, d.lay.ell);
  sp.mask_out = at<uint8_t>(ws, d.lay.mask);
  sp.idx_out = at<int32_t>(ws, d.lay.idx);
  sp.kept_dev = kept_dev;
  sp.kept_host = kept_host;
  sp.update_cache = 1;
  sp.want_rephase = rephase ? 1 : 0;
  sp.head_is_static = head_is_static;
  sp.evict_first_frame = evict_first_frame;
  sp.random_stream = ((uint64_t)cfg->random_seed << 32) | (uint32_t)evict_first_frame;
  sp.h_lo = d.T_s;
  sp.h_hi = rephase ? evict_first_frame : d.T_s;
  sp.q0 = q0;
  sp.q0_prev = q0_prev;
  GatherParams gp = gather_params(cache, cfg, d, ws, evict_slot, head_is_static, evict_first_frame);
  set_turn(gp, sp, cfg, d, evict_first_frame, q0);
  if (head_is_static) {  // the scan lists the receiving planes; the gather splits that list only
    sp.dyn_list = at<int32_t>(ws, d.lay.dyn);
    gp.dyn_list = sp.dyn_list;
  }
  finish_tables(sp);
  RephaseParams rp = rephase_params(cache, cfg, d, ws, sp.h_lo, sp.h_hi);
  if (pv) {
    const int64_t per_chunk = d.C / pv->pg.bs;
    Paging pg = pv->pg;
    pg.src_blocks = pv->window_blocks + (int64_t)evict_slot * per_chunk;
    gp.pg = pg;
    rp.pg = pg;
    sp.tbl_a = pg.hist_blocks;
    sp.n_tbl_a = (int32_t)(cache->hist_cap / pg.bs);
    sp.tbl_b = pg.src_blocks;
    sp.n_tbl_b = (int32_t)per_chunk;
    sp.n_blocks = pv->n_blocks;
    sp.n_tbl_slices = (sp.n_tbl_a + sp.n_tbl_b + kThreads - 1) / kThreads;
  }
  if (ws_clear_bytes && cudaMemsetAsync(ws, 0, ws_clear_bytes, st) != cudaSuccess) return DCP_ECUDA;
  // scan -> re-index (reads the history lengths before the step) -> gather (grows them); when every plane receives,
  // the re-index and the gather run as one launch (their rows are disjoint, and every length before the step is the
  // scan's common length)
  dcp_status rc = cuda_ok(launch_scan(sp, st));
  if (rc != DCP_OK) return rc;
  const bool fused = rephase && !head_is_static;
  if (rephase && !fused) {
    rc = cuda_ok(launch_rephase(rp, st, true, pv != nullptr));
    if (rc != DCP_OK) return rc;
  }
  if (g_ev_after_scan && cudaEventRecord(g_ev_after_scan, st) != cudaSuccess) return DCP_ECUDA;
  if (fused)
    rc = cuda_ok(launch_step_fused(gp, rp, st, g_ev_after_scan == nullptr, pv != nullptr));
  else
    rc = cuda_ok(launch_gather(gp, st, g_ev_after_scan == nullptr, pv != nullptr));
  if (rc != DCP_OK) return rc;
  if (g_ev_after_gather && cudaEventRecord(g_ev_after_gather, st) != cudaSuccess) return DCP_ECUDA;
  return rc;
}

}  // namespace

extern "C" {

size_t dcp_snapshot_max_bytes(const dcp_cache* cache, const dcp_config* cfg, uint32_t live_slots) {
  Derived d;
  int n_live = 0;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK || check_live(cfg, live_slots, &n_live) != DCP_OK) return 0;
  const int64_t rows = d.n_planes * (d.sink_rows + cache->hist_cap + (int64_t)n_live * d.C);
  const int64_t data_off = (128 + 4 * d.n_planes + 4 * cache->hist_cap + 255) & ~(int64_t)255;
  return (size_t)(data_off + 2 * rows * (int64_t)cache->D * d.esize);
}

dcp_status dcp_snapshot(const dcp_cache* cache, const dcp_config* cfg, uint32_t live_slots, int32_t q0,
                        void* image_host, size_t image_bytes, void* ws, size_t ws_bytes, void* stream) {
  Derived d;
  int n_live = 0;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK || check_live(cfg, live_slots, &n_live) != DCP_OK) return DCP_EINVAL;
  if (check_ws(ws, ws_bytes, d.lay.total) != DCP_OK) return DCP_EINVAL;
  if (!image_host || !aligned(image_host, 16) || image_bytes < 128) return DCP_EINVAL;
  char* img = image_device_ptr(image_host);
  if (!img || !aligned(img, 16)) return DCP_EINVAL;
  SnapParams p = snap_params(cache, cfg, d, live_slots, n_live, img, image_bytes, ws, 0);
  p.q0 = q0;
  return cuda_ok(launch_snapshot(p, (cudaStream_t)stream));
}

dcp_status dcp_restore(const dcp_cache* cache, const dcp_config* cfg, const void* image_host, size_t image_bytes,
                       int32_t* q0_out, uint32_t* live_slots_out, void* ws, size_t ws_bytes, void* stream) {
  Derived d;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK) return DCP_EINVAL;
  if (check_ws(ws, ws_bytes, d.lay.total) != DCP_OK) return DCP_EINVAL;
  if (!image_host || !aligned(image_host, 16) || image_bytes < 128) return DCP_EINVAL;
  char* img = image_device_ptr(image_host);
  if (!img || !aligned(img, 16)) return DCP_EINVAL;
  // the image is complete in host memory: check it against this cache before anything is launched
  const char* h = static_cast<const char*>(image_host);
  const int64_t row_bytes = (int64_t)cache->D * d.esize;
  if (std::memcmp(h, "DCPSNAP1", 8) != 0) return DCP_EINVAL;
  if (img_i32(h, 8) != cache->L || img_i32(h, 12) != cache->H || img_i32(h, 16) != cache->D ||
      img_i32(h, 20) != cache->dtype || img_i64(h, 24) != cache->cap || img_i64(h, 32) != cache->hist_cap ||
      img_i64(h, 40) != d.sink_rows || img_i64(h, 48) != d.C || img_i32(h, 56) != cfg->window_chunks ||
      img_i64(h, 72) != row_bytes)
    return DCP_EINVAL;
  const uint32_t live = (uint32_t)img_i32(h, 60);
  int n_live = 0;
  if (check_live(cfg, live, &n_live) != DCP_OK) return DCP_EINVAL;
  if ((int64_t)image_bytes < 128 + 4 * d.n_planes) return DCP_EINVAL;
  int64_t rows = 0;
  int32_t longest = 0;
  for (int64_t p = 0; p < d.n_planes; ++p) {
    const int32_t len = img_i32(h, 128 + 4 * p);
    if (len < 0 || len > cache->hist_cap) return DCP_EINVAL;
    rows += d.sink_rows + len + (int64_t)n_live * d.C;
    if (len > longest) longest = len;
  }
  const int64_t data_off = (128 + 4 * d.n_planes + 4 * (int64_t)longest + 255) & ~(int64_t)255;
  const int64_t total = data_off + 2 * rows * row_bytes;
  if (img_i32(h, 68) != longest || img_i64(h, 80) != rows || img_i64(h, 88) != total ||
      (int64_t)image_bytes < total)
    return DCP_EINVAL;
  if (q0_out) *q0_out = img_i32(h, 64);
  if (live_slots_out) *live_slots_out = live;
  SnapParams p = snap_params(cache, cfg, d, live, n_live, img, image_bytes, ws, 1);
  return cuda_ok(launch_snapshot(p, (cudaStream_t)stream));
}

dcp_status dcp_workspace_outputs(const dcp_cache* cache, const dcp_config* cfg, void* ws, float** ell_dev,
                                 uint8_t** mask_dev, int32_t** idx_dev) {
  Derived d;
  if (check_cache_cfg(cache, cfg, &d) != DCP_OK || !ws) return DCP_EINVAL;
  if (ell_dev) *ell_dev = at<float>(ws, d.lay.ell);
  if (mask_dev) *mask_dev = at<uint8_t>(ws, d.lay.mask);
  if (idx_dev) *idx_dev = at<int32_t>(ws, d.lay.idx);
  return DCP_OK;
}

dcp_status dcp_get_status(const int32_t* status_dev, void* stream) {
  if (!status_dev) return DCP_EINVAL;
  int32_t v = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DCP_ECUDA;
  if (cudaMemcpy(&v, status_dev, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DCP_ECUDA;
  return v;
}

dcp_status dcp_reset_status(int32_t* status_dev, void* stream) {
  if (!status_dev) return DCP_EINVAL;
  return cuda_ok(cudaMemsetAsync(status_dev, 0, sizeof(int32_t), (cudaStream_t)stream));
}

const char* dcp_status_string(dcp_status s) {
  switch (s) {
    case DCP_OK: return "ok";
    case DCP_EINVAL: return "invalid argument";
    case DCP_ECAPACITY: return "history capacity exceeded";
    case DCP_ECUDA: return "CUDA runtime error";
    case DCP_ETIMEOUT: return "timed out (not produced by this version)";
    case DCP_EDEVICE: return "inconsistent cache state on the device";
    default: return "unknown status";
  }
}

void dcp_pr_add_chunk(dcp_pr_counter* acc, int64_t n_planes, int64_t hist_len_sum, int64_t sink_tokens_visible,
                      int64_t window_tokens_visible, int64_t prior_tokens) {
  if (!acc) return;
  acc->visible += n_planes * (sink_tokens_visible + window_tokens_visible) + hist_len_sum;
  acc->full += n_planes * prior_tokens;
}

double dcp_pr_value(const dcp_pr_counter* acc) {
  if (!acc || acc->full <= 0) return 0.0;
  return 1.0 - (double)acc->visible / (double)acc->full;
}

dcp_status dcp_set_phase_events(void* ev_after_scan, void* ev_after_gather) {
  g_ev_after_scan = (cudaEvent_t)ev_after_scan;
  g_ev_after_gather = (cudaEvent_t)ev_after_gather;
  return DCP_OK;
}

uint32_t dcp_abi_struct_sizes(void) { return ((uint32_t)sizeof(dcp_cache) << 16) | (uint32_t)sizeof(dcp_config); }


}  // extern "C"
