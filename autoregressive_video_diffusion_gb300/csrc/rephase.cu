// History re-index kernel: when the query frame moves from q0_prev to q0, each history key whose temporal phase
// t~(t) changes turns its temporal rotary pairs by theta_p * (t~(t; q0) - t~(t; q0_prev)), in place.
//
// Page: DeCoPrune (onedev.kr/papers/726), section "what differs": old context keys are re-indexed to
// t~(t) = q0 - g(q0 - t) inside a fixed virtual span; g leaves recent offsets alone and compresses old ones linearly,
// and only the key phase changes.  Since g depends on q0, the phase of every compressed history key moves whenever
// q0 advances.
//
// Only the vectors of a row that hold temporal pairs are read and written (for bf16, D = 128 and n_t = 22 that is
// the first 96 bytes of each 256-byte row: three 32-byte vectors); values and the other key dims are never touched.
// Plane streaming as in the gather: an item is (block of history rows, range of planes), and each CTA takes one
// contiguous, equal share of all (block, plane) pairs.  Each thread owns one
// (row, vector) of the block; the cos/sin entries of that vector's pairs depend only on the row's frame, so they are
// loaded into registers once per item and reused for every plane.  Planes are taken four at a time, so four
// independent loads are in flight per thread.  Rows whose frame does not move, and rows past a plane's own history
// length, are skipped.  The kernel runs before the gather of the same step, so hist_len still holds the lengths
// before the step.  Paged caches look a row's block up in the history block table once per item.
#include <type_traits>

#include "dcp_internal.cuh"

namespace dcp {

namespace {

constexpr int kPlanesInFlight = 4;

template <int NW, bool PAGED>
__global__ void __launch_bounds__(kThreads, 3) rephase_kernel(const RephaseParams p) {
  using Off = typename std::conditional<PAGED, int64_t, int>::type;
  constexpr int VB = NW * 4;
  wait_for_predecessor();
  allow_dependents();
  const Ctrl* c = p.ctrl;
  if (c->abort) return;
  const int rp_max = c->rp_max;
  if (rp_max <= 0 || p.nvt <= 0) return;
  const int ppv = p.dtype == DCP_BF16 ? VB / 4 : VB / 8;
  const int rows_per_item = kThreads / p.nvt;  // nvt <= kThreads: rows are at most 4 KiB
  const int nblk = (rp_max + rows_per_item - 1) / rows_per_item;
  // Each CTA takes one contiguous share of the (row block, plane) units, block-major, so every CTA gets the same
  // number of planes give or take one: whole items dealt round-robin left a third of the CTAs a third item.
  const int64_t units = (int64_t)nblk * p.n_planes;
  const int64_t u_end = units * (blockIdx.x + 1) / gridDim.x;
  const int row_in_item = threadIdx.x / p.nvt, vec = threadIdx.x - row_in_item * p.nvt;
  const int64_t hist0 = PAGED ? 0 : p.hist_row0 * (int64_t)p.row_bytes;
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

    bool live = false;
    float4 tr[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) tr[i] = make_float4(1.f, 0.f, 0.f, 0.f);
    if (row_in_item < rows_per_item && row < rp_max) {
      const int t = __ldg(p.hist_t + row);
      if (t < p.h_lo || t >= p.h_hi) {
        set_status(p.status, DCP_EDEVICE);  // a history frame outside the table: corrupt hist_t, leave the row
      } else if (__ldg(p.rot_h + t)) {
        live = true;
        const float4* tt = p.trig_h + (int64_t)t * p.n_t + vec * ppv;
#pragma unroll
        for (int i = 0; i < NW; ++i)
          if (i < ppv && vec * ppv + i < p.n_t) tr[i] = __ldg(tt + i);
      }
    }
    if (!__syncthreads_or(live)) continue;
    Off off;
    if (PAGED)  // the table covers history rows only: look up live rows
      off = live ? (int64_t)__ldg(p.pg.hist_blocks + row / p.pg.bs) * p.pg.s_block +
                       (int64_t)(row % p.pg.bs) * p.pg.s_row + vec * VB
                 : 0;
    else
      off = row * p.row_bytes + vec * VB;

    for (int pl = p0; pl < p1; pl += kPlanesInFlight) {
      Vec<NW> x[kPlanesInFlight];
      bool go[kPlanesInFlight];
#pragma unroll
      for (int q = 0; q < kPlanesInFlight; ++q) {
        const int plq = pl + q;
        go[q] = live && plq < p1 && row < __ldg(p.hist_len + min(plq, p1 - 1));
        if (go[q]) ld_plain(x[q], p.k + plane_base(plq) + hist0 + off);
      }
#pragma unroll
      for (int q = 0; q < kPlanesInFlight; ++q) {
        if (go[q]) {
          dev_rotate_vec_regs(x[q], p.dtype, vec * ppv, p.n_t, tr);
          st_plain(p.k + plane_base(pl + q) + hist0 + off, x[q]);
        }
      }
    }
  }
}

template <int NW, bool PAGED>
cudaError_t launch_rephase_w(const RephaseParams& p, cudaStream_t s, bool overlap_launch) {
  static LaunchCache lc;
  int blocks_per_sm = 1;
  const cudaError_t e = launch_setup(lc, rephase_kernel<NW, PAGED>, kThreads, 0, &blocks_per_sm);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_launch ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, rephase_kernel<NW, PAGED>, p);
}

}  // namespace

cudaError_t launch_rephase(const RephaseParams& p, cudaStream_t s, bool overlap_launch, bool paged) {
  if (paged)
    return p.vb == 32 ? launch_rephase_w<8, true>(p, s, overlap_launch)
                      : launch_rephase_w<4, true>(p, s, overlap_launch);
  return p.vb == 32 ? launch_rephase_w<8, false>(p, s, overlap_launch) : launch_rephase_w<4, false>(p, s, overlap_launch);
}

}  // namespace dcp
