// Host snapshot and restore of the pruned cache.
//
// Page "기술 요약: 생성형 월드 모델을 위한 지속적 계산 상태" (gist.science/ko/paper/2607.21686), section "PCS contract":
// checkpoint and restore, where restore gives back the state (round trip) and the checkpoint holds exactly the state
// that cannot be re-derived (snapshot completeness).  For the pruned cache that is every plane's sink rows and
// history rows [0, hist_len), the live ring slots of the dense window, hist_len, hist_t and q0.  The image layout is
// documented with dcp_snapshot in dcp.h.
//
// Two launches on the caller's stream, no host synchronisation (the history lengths live on the device):
//   layout kernel  one CTA: block scan of the planes' saved row counts into the first image row of each plane,
//                  the longest history, and (snapshot) the header, hist_len and hist_t of the image, after checking
//                  that the image is large enough; (restore) hist_len and hist_t of the cache.
//   copy kernel    persistent grid, one CTA per SM: an item is (tensor, plane, 64 image rows); its image rows are one
//                  contiguous run, its cache rows are the plane's sink + history run followed by its live ring
//                  slots.  16-byte vectors, four in flight per thread.
// On GB300 the image moves over the host link (~194 GB/s device to host, ~211 GB/s host to device measured for both
// copy engines and SM stores), so one CTA per SM is enough to saturate it and leaves the SMs to other work.
#include "dcp_internal.cuh"

namespace dcp {

namespace {

constexpr int kRowsPerItem = 64;
constexpr int kInFlight = 4;
constexpr unsigned kFullMask = 0xFFFFFFFFu;

__device__ int64_t block_exclusive_scan64(int64_t x, long long* s_warp, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFullMask, v, o);
    if (lane >= o) v += y;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  long long base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const long long s = s_warp[w];
    if (w < warp) base += s;
    tot += s;
  }
  *total = tot;
  return base + v - x;
}

__device__ __forceinline__ void put32(char* img, int off, int32_t x) { *reinterpret_cast<int32_t*>(img + off) = x; }
__device__ __forceinline__ void put64(char* img, int off, int64_t x) { *reinterpret_cast<int64_t*>(img + off) = x; }

__global__ void __launch_bounds__(kThreads) snap_layout_kernel(const SnapParams p) {
  __shared__ long long s_warp[kThreads / 32];
  __shared__ int s_red[kThreads / 32][2];
  allow_dependents();  // the copy kernel may start early: it waits for this grid before reading anything
  int32_t* img_len = reinterpret_cast<int32_t*>(p.img + 128);
  const int64_t fixed = p.sink_rows + (int64_t)p.n_live * p.C;
  int64_t base = 0;
  int longest = 0, bad = 0;
  for (int p0 = 0; p0 < p.n_planes; p0 += kThreads) {
    const int pl = p0 + threadIdx.x;
    int len = 0;
    if (pl < p.n_planes) {
      len = p.dir == 0 ? p.hist_len[pl] : img_len[pl];
      if (len < 0 || len > p.hist_cap) {
        bad = 1;
        len = 0;
      }
    }
    int64_t total = 0;
    const int64_t excl = block_exclusive_scan64(pl < p.n_planes ? fixed + len : 0, s_warp, &total);
    if (pl < p.n_planes) p.plane_off[pl] = base + excl;
    base += total;
    longest = max(longest, len);
  }
  longest = __reduce_max_sync(kFullMask, longest);
  bad = __reduce_max_sync(kFullMask, bad);
  if ((threadIdx.x & 31) == 0) {
    s_red[threadIdx.x >> 5][0] = longest;
    s_red[threadIdx.x >> 5][1] = bad;
  }
  __syncthreads();
  longest = 0;
  bad = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    longest = max(longest, s_red[w][0]);
    bad = max(bad, s_red[w][1]);
  }
  const int64_t data_off = (128 + 4 * (int64_t)p.n_planes + 4 * (int64_t)longest + 255) & ~(int64_t)255;
  const int64_t total_bytes = data_off + 2 * base * p.row_bytes;
  int abort = 0;
  if (bad) abort = DCP_EDEVICE;
  else if (p.dir == 0 && total_bytes > p.img_bytes) abort = DCP_ECAPACITY;

  if (p.dir == 0) {
    if (threadIdx.x == 0) {
      put64(p.img, 0, 0x3150414E53504344ll);  // "DCPSNAP1" read as a little-endian int64
      put32(p.img, 8, p.L);
      put32(p.img, 12, p.H);
      put32(p.img, 16, p.D);
      put32(p.img, 20, p.dtype);
      put64(p.img, 24, p.cap);
      put64(p.img, 32, p.hist_cap);
      put64(p.img, 40, p.sink_rows);
      put64(p.img, 48, p.C);
      put32(p.img, 56, p.window_chunks);
      put32(p.img, 60, (int32_t)p.live_slots);
      put32(p.img, 64, p.q0);
      put32(p.img, 68, longest);
      put64(p.img, 72, p.row_bytes);
      put64(p.img, 80, base);
      put64(p.img, 88, total_bytes);
      for (int off = 96; off < 128; off += 8) put64(p.img, off, 0);
    }
    if (!abort) {
      for (int pl = threadIdx.x; pl < p.n_planes; pl += kThreads) img_len[pl] = p.hist_len[pl];
      for (int j = threadIdx.x; j < longest; j += kThreads) img_len[p.n_planes + j] = p.hist_t[j];
      const int64_t pad_from = 128 + 4 * (int64_t)p.n_planes + 4 * (int64_t)longest;
      for (int64_t b = pad_from + threadIdx.x; b < data_off; b += kThreads) p.img[b] = 0;
    }
  } else if (!abort) {
    for (int pl = threadIdx.x; pl < p.n_planes; pl += kThreads) p.hist_len[pl] = img_len[pl];
    for (int j = threadIdx.x; j < longest; j += kThreads) p.hist_t[j] = img_len[p.n_planes + j];
  }
  if (threadIdx.x == 0) {
    p.plane_off[p.n_planes] = base;
    Ctrl* c = p.ctrl;
    c->snap_abort = abort;
    c->snap_hist_t_len = longest;
    c->snap_rows = base;
    c->snap_data_off = data_off;
    if (abort) set_status(p.status, abort);
  }
}

template <int DIR>
__global__ void __launch_bounds__(kThreads) snap_copy_kernel(const SnapParams p) {
  __shared__ int s_slot[32];
  wait_for_predecessor();
  const Ctrl* c = p.ctrl;
  if (c->snap_abort) return;
  if (threadIdx.x == 0) {
    int i = 0;
    for (int s = 0; s < 32; ++s)
      if ((p.live_slots >> s) & 1u) s_slot[i++] = s;
  }
  __syncthreads();
  const int64_t rows_tensor = c->snap_rows, data_off = c->snap_data_off;
  const int64_t live_rows = (int64_t)p.n_live * p.C;
  const int64_t max_rows = p.sink_rows + c->snap_hist_t_len + live_rows;
  const int64_t cpp = (max_rows + kRowsPerItem - 1) / kRowsPerItem;
  const int64_t items = 2 * (int64_t)p.n_planes * cpp;
  const int vpr = p.row_bytes / 16;

  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int64_t pt = it / cpp;
    const int64_t r0 = (it - pt * cpp) * kRowsPerItem;
    const int pl = (int)(pt % p.n_planes), t = (int)(pt / p.n_planes);
    const int64_t off0 = p.plane_off[pl];
    const int64_t n_rows = p.plane_off[pl + 1] - off0;
    if (r0 >= n_rows) continue;
    const int rows = (int)min((int64_t)kRowsPerItem, n_rows - r0);
    const int64_t first_run = n_rows - live_rows;  // the plane's sink + history rows
    char* cache = (t ? p.v : p.k) + pl * p.plane_bytes;
    char* img = p.img + data_off + (t * rows_tensor + off0 + r0) * p.row_bytes;
    const int nvec = rows * vpr;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kInFlight * kThreads) {
      int4 x[kInFlight];
      int64_t coff[kInFlight];
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int v = v0 + u * kThreads;
        coff[u] = -1;
        if (v < nvec) {
          const int r = v / vpr, col = v - r * vpr;
          int64_t row = r0 + r;
          if (row >= first_run) {
            const int64_t r2 = row - first_run, i = r2 / p.C;
            row = p.sink_rows + p.hist_cap + s_slot[i] * p.C + (r2 - i * p.C);
          }
          coff[u] = row * p.row_bytes + col * 16;
          if (DIR == 0) x[u] = __ldcs(reinterpret_cast<const int4*>(cache + coff[u]));
          else x[u] = *reinterpret_cast<const int4*>(img + (int64_t)v * 16);
        }
      }
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        if (coff[u] < 0) continue;
        if (DIR == 0) *reinterpret_cast<int4*>(img + (int64_t)(v0 + u * kThreads) * 16) = x[u];
        else *reinterpret_cast<int4*>(cache + coff[u]) = x[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_snapshot(const SnapParams& p, cudaStream_t s) {
  snap_layout_kernel<<<1, kThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sm_count());
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.dir == 0 ? cudaLaunchKernelEx(&cfg, snap_copy_kernel<0>, p) : cudaLaunchKernelEx(&cfg, snap_copy_kernel<1>, p);
}

}  // namespace dcp
