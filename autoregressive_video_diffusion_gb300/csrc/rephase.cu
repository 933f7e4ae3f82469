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
// Plane streaming as in the gather: an item is (block of history rows, range of planes); each thread owns a few fixed
// (row, vector) pairs, looks up their frame's table row once, and walks the planes of its range.  Rows whose frame
// does not move, and rows past a plane's own history length, are skipped.  The kernel runs before the gather of the
// same step, so hist_len still holds the lengths before the step.
#include "dcp_internal.cuh"

namespace dcp {

namespace {

template <int NW>
__global__ void __launch_bounds__(kThreads, 3) rephase_kernel(const RephaseParams p) {
  constexpr int VB = NW * 4;
  constexpr int SLOTS = kBytesPerThread / VB;
  wait_for_predecessor();
  allow_dependents();
  const Ctrl* c = p.ctrl;
  if (c->abort) return;
  const int rp_max = c->rp_max;
  if (rp_max <= 0 || p.nvt <= 0) return;
  const int ppv = p.dtype == DCP_BF16 ? VB / 4 : VB / 8;
  const int rows_per_item = (kThreads * SLOTS) / p.nvt;
  const int nblk = (rp_max + rows_per_item - 1) / rows_per_item;
  int ranges = (int)gridDim.x / nblk;
  if (ranges < 1) ranges = 1;
  if (ranges > p.n_planes) ranges = p.n_planes;
  const int ppr = (p.n_planes + ranges - 1) / ranges;
  const int items = nblk * ranges;

  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int jb = it % nblk, r = it / nblk;
    const int p0 = r * ppr, p1 = min(p.n_planes, p0 + ppr);
    const int j0 = jb * rows_per_item;

    int off[SLOTS];       // offset of the slot's vector from the first history row, -1 if it does not turn
    int row_of[SLOTS], vec_of[SLOTS];
    const float4* trig[SLOTS];
    bool any = false;
#pragma unroll
    for (int u = 0; u < SLOTS; ++u) {
      const int e = threadIdx.x + u * kThreads;
      const int row = e / p.nvt, vec = e - row * p.nvt;
      row_of[u] = j0 + row;
      vec_of[u] = vec;
      off[u] = -1;
      trig[u] = p.trig_h;
      if (row < rows_per_item && j0 + row < rp_max) {
        const int t = __ldg(p.hist_t + j0 + row);
        if (t < p.h_lo || t >= p.h_hi) {
          set_status(p.status, DCP_EDEVICE);  // a history frame outside the table: corrupt hist_t, leave the row
        } else if (__ldg(p.rot_h + t)) {
          trig[u] = p.trig_h + (int64_t)t * p.n_t;
          off[u] = (j0 + row) * p.row_bytes + vec * VB;
        }
      }
      any |= off[u] >= 0;
    }
    if (!__syncthreads_or(any)) continue;

    const int64_t hist0 = p.hist_row0 * (int64_t)p.row_bytes;
    for (int pl = p0; pl < p1; ++pl) {
      const int len = __ldg(p.hist_len + pl);
      if (len <= j0) continue;
      char* kb = p.k + pl * p.plane_bytes + hist0;
      Vec<NW> x[SLOTS];
#pragma unroll
      for (int u = 0; u < SLOTS; ++u)
        if (off[u] >= 0 && row_of[u] < len) ld_plain(x[u], kb + off[u]);
#pragma unroll
      for (int u = 0; u < SLOTS; ++u) {
        if (off[u] >= 0 && row_of[u] < len) {
          dev_rotate_vec(x[u], p.dtype, vec_of[u] * ppv, p.n_t, trig[u]);
          st_plain(kb + off[u], x[u]);
        }
      }
    }
  }
}

template <int NW>
cudaError_t launch_rephase_w(const RephaseParams& p, cudaStream_t s, bool overlap_launch) {
  static int blocks_per_sm = 0;
  if (!blocks_per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, rephase_kernel<NW>, kThreads, 0) !=
            cudaSuccess ||
        blocks_per_sm < 1)
      blocks_per_sm = 1;
  }
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
  return cudaLaunchKernelEx(&cfg, rephase_kernel<NW>, p);
}

}  // namespace

cudaError_t launch_rephase(const RephaseParams& p, cudaStream_t s, bool overlap_launch) {
  return p.vb == 32 ? launch_rephase_w<8>(p, s, overlap_launch) : launch_rephase_w<4>(p, s, overlap_launch);
}

}  // namespace dcp
