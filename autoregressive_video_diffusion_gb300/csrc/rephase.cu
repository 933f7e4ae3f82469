// History re-index kernel: when the query frame moves from q0_prev to q0, each history key whose temporal phase
// t~(t) changes turns its temporal rotary pairs by theta_p * (t~(t; q0) - t~(t; q0_prev)), in place.
//
// Page: DeCoPrune (onedev.kr/papers/726), section "what differs": old context keys are re-indexed to
// t~(t) = q0 - g(q0 - t) inside a fixed virtual span; g leaves recent offsets alone and compresses old ones linearly,
// and only the key phase changes.  Since g depends on q0, the phase of every compressed history key moves whenever
// q0 advances.
//
// Only the 16-byte vectors of a row that hold temporal pairs are read and written (for bf16, D = 128 and
// n_t = 22 that is the first 96 bytes of each 256-byte row); values and the other key dims are never touched.
// One thread per (plane, row, vector); rows of frames whose phase does not change are skipped.
#include "dcp_internal.cuh"

namespace dcp {

namespace {

__global__ void __launch_bounds__(kThreads) rephase_kernel(const RephaseParams p) {
  const Ctrl* c = p.ctrl;
  if (c->abort) return;
  const int n_rp = c->n_rp, rp_max = c->rp_max;
  if (n_rp <= 0 || rp_max <= 0) return;
  const int ppv = p.dtype == DCP_BF16 ? 4 : 2;
  const int64_t per_plane = (int64_t)rp_max * p.nvt;
  const int64_t total = (int64_t)n_rp * per_plane;
  for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < total; g += (int64_t)gridDim.x * kThreads) {
    const int i = (int)(g / per_plane);
    const int64_t rem = g - (int64_t)i * per_plane;
    const int row = (int)(rem / p.nvt);
    const int vec = (int)(rem - (int64_t)row * p.nvt);
    if (row >= __ldg(p.rp_len + i)) continue;
    const int t = __ldg(p.hist_t + row);
    if (t < p.h_lo || t >= p.h_hi) {
      set_status(p.status, DCP_EDEVICE);  // a history frame outside the table: corrupt hist_t, leave the row
      continue;
    }
    if (!__ldg(p.rot_h + t)) continue;
    const int plane = __ldg(p.rp_list + i);
    uint4* addr = reinterpret_cast<uint4*>(p.k + (int64_t)plane * p.plane_bytes + (p.hist_row0 + row) * p.row_bytes +
                                           vec * 16);
    uint4 x = *addr;
    x = dev_rotate_vec(x, p.dtype, vec * ppv, p.n_t, p.trig_h + (int64_t)t * p.n_t);
    *addr = x;
  }
}

}  // namespace

cudaError_t launch_rephase(const RephaseParams& p, cudaStream_t s) {
  static int blocks_per_sm = 0;
  if (!blocks_per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, rephase_kernel, kThreads, 0) != cudaSuccess ||
        blocks_per_sm < 1)
      blocks_per_sm = 1;
  }
  rephase_kernel<<<sm_count() * blocks_per_sm, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dcp
