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
// length, are skipped.  This kernel serves dcp_rope_reindex and the prune steps of head-specialised caches, where it
// runs before the gather of the same step, so hist_len still holds the lengths before the step; when every plane
// receives, a prune step runs the same body inside the gather's launch (step_kernel in gather.cu).  Paged caches look
// a row's block up in the history block table once per item.  The body is in rephase_body.cuh.
#include "rephase_body.cuh"

namespace dcp {

namespace {

constexpr int kPlanesInFlight = 4;

template <int NW, bool PAGED>
__global__ void __launch_bounds__(kThreads, 3) rephase_kernel(const RephaseParams p) {
  wait_for_predecessor();
  allow_dependents();
  const Ctrl* c = p.ctrl;
  if (c->abort) return;
  const int rp_max = c->rp_max;
  if (rp_max <= 0 || p.nvt <= 0) return;
  // Each CTA takes one contiguous share of the (row block, plane) units, block-major, so every CTA gets the same
  // number of planes give or take one: whole items dealt round-robin left a third of the CTAs a third item.
  int rows_per_item = 0;
  const int64_t units = rephase_unit_count(p, rp_max, &rows_per_item);
  rephase_units<NW, PAGED, kPlanesInFlight>(p, rp_max, rows_per_item, -1, units * blockIdx.x / gridDim.x,
                                            units * (blockIdx.x + 1) / gridDim.x);
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
