// Read-time re-index kernel: the history keys as attention at query frame q0 sees them, for a cache whose history
// keys stay at their own frame's phase (reindex_mode 1).
//
// Page: DeCoPrune (onedev.kr/papers/726), section "what differs": old context keys take the temporal phase
// t~(t) = q0 - g(q0 - t); only the key phase changes.  Instead of turning every history key in place each time q0
// moves, the keys stay at the phase t they were generated with and each read turns them once, from t to
// t~(t; q0), so nothing accumulates rounding from one step to the next.
//
// Plane streaming as in the other kernels: an item is (block of history rows, range of planes), each CTA taking one
// contiguous, equal share of all (block, plane) pairs; each thread owns one
// (row, vector) of the block, so a warp reads whole rows; the vectors that hold temporal pairs load their cos/sin
// entries (which depend only on the row's frame) into registers once per item.  Four planes in flight per thread.
// Rows past a plane's own history length are skipped.  The phase table comes from the scan kernel's table CTAs,
// launched just before on the same stream.
#include <type_traits>

#include "dcp_internal.cuh"

namespace dcp {

namespace {

constexpr int kPlanesInFlight = 4;

template <int NW, bool PAGED>
__global__ void __launch_bounds__(kThreads, 3) read_kernel(const ReadParams p) {
  using Off = typename std::conditional<PAGED, int64_t, int>::type;
  constexpr int VB = NW * 4;
  wait_for_predecessor();
  const Ctrl* c = p.ctrl;
  if (c->abort) return;
  const int rp_max = c->rp_max;  // longest history of any plane
  const int rp_min = c->rp_min;  // rows below it are history in every plane
  if (rp_max <= 0) return;
  const int ppv = p.dtype == DCP_BF16 ? VB / 4 : VB / 8;
  const int rows_per_item = kThreads / p.vpr;  // vpr <= kThreads: rows are at most 4 KiB
  const int nblk = (rp_max + rows_per_item - 1) / rows_per_item;
  // One contiguous, equal share of the (row block, plane) units per CTA, block-major.
  const int64_t units = (int64_t)nblk * p.n_planes;
  const int64_t u_end = units * (blockIdx.x + 1) / gridDim.x;
  const int row_in_item = threadIdx.x / p.vpr, vec = threadIdx.x - row_in_item * p.vpr;
  const int64_t hist0 = PAGED ? 0 : p.hist_row0 * (int64_t)p.row_bytes;
  const int64_t out_plane = p.hist_cap * (int64_t)p.row_bytes;
  auto plane_base = [&](int pl) -> int64_t {
    if (PAGED) return (int64_t)(pl / p.pg.H) * p.pg.s_layer + (int64_t)(pl % p.pg.H) * p.pg.s_head;
    return (int64_t)pl * p.plane_bytes;
  };

  for (int64_t u = units * blockIdx.x / gridDim.x; u < u_end;) {
    const int jb = (int)(u / p.n_planes);
    const int p0 = (int)(u - (int64_t)jb * p.n_planes);
    const int p1 = (int)min((int64_t)p.n_planes, u_end - (int64_t)jb * p.n_planes);
    u = (int64_t)jb * p.n_planes + p1;
    const int row = jb * rows_per_item + row_in_item;

    bool valid = row_in_item < rows_per_item && row < rp_max;
    bool turn = false;
    float4 tr[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) tr[i] = make_float4(1.f, 0.f, 0.f, 0.f);
    if (valid) {
      const int t = __ldg(p.hist_t + row);
      if (t < p.f_lo || t >= p.f_hi) {
        set_status(p.status, DCP_EDEVICE);  // a history frame outside the table: corrupt hist_t, skip the row
        valid = false;
      } else if (vec < p.nvt && __ldg(p.rot + (t - p.f_lo))) {
        turn = true;
        const float4* tt = p.trig + (int64_t)(t - p.f_lo) * p.n_t + vec * ppv;
#pragma unroll
        for (int i = 0; i < NW; ++i)
          if (i < ppv && vec * ppv + i < p.n_t) tr[i] = __ldg(tt + i);
      }
    }
    if (!__syncthreads_or(valid)) continue;
    Off src;
    if (PAGED)  // the table covers history rows only: look up valid rows
      src = valid ? (int64_t)__ldg(p.pg.hist_blocks + row / p.pg.bs) * p.pg.s_block +
                        (int64_t)(row % p.pg.bs) * p.pg.s_row + vec * VB
                  : 0;
    else
      src = row * p.row_bytes + vec * VB;
    const int64_t dst = (int64_t)row * p.row_bytes + vec * VB;

    for (int pl = p0; pl < p1; pl += kPlanesInFlight) {
      Vec<NW> x[kPlanesInFlight];
      bool go[kPlanesInFlight];
#pragma unroll
      for (int q = 0; q < kPlanesInFlight; ++q) {
        const int plq = pl + q;
        go[q] = valid && plq < p1 && (row < rp_min || row < __ldg(p.hist_len + p.plane0 + min(plq, p1 - 1)));
        if (go[q]) ld_stream(x[q], p.k + plane_base(p.plane0 + plq) + hist0 + src);
      }
#pragma unroll
      for (int q = 0; q < kPlanesInFlight; ++q) {
        if (go[q]) {
          if (turn) dev_rotate_vec_regs(x[q], p.dtype, vec * ppv, p.n_t, tr);
          st_stream(p.out + (int64_t)(pl + q) * out_plane + dst, x[q]);
        }
      }
    }
  }
}

template <int NW, bool PAGED>
cudaError_t launch_read_w(const ReadParams& p, cudaStream_t s) {
  static LaunchCache lc;
  int blocks_per_sm = 1;
  const cudaError_t e = launch_setup(lc, read_kernel<NW, PAGED>, kThreads, 0, &blocks_per_sm);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, read_kernel<NW, PAGED>, p);
}

}  // namespace

cudaError_t launch_read(const ReadParams& p, cudaStream_t s, bool paged) {
  if (paged) return p.vb == 32 ? launch_read_w<8, true>(p, s) : launch_read_w<4, true>(p, s);
  return p.vb == 32 ? launch_read_w<8, false>(p, s) : launch_read_w<4, false>(p, s);
}

}  // namespace dcp
