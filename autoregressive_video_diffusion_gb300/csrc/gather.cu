// Gather kernel of the prune step: physical compaction K[m], V[m] of the leaving chunk into the history region of
// every receiving (layer, head) plane, with the temporal RoPE re-phase of each moved key fused in.
//
// Page: DeCoPrune (onedev.kr/papers/726).  Section "how it works": when a non-sink chunk leaves the dense window,
// each layer keeps only the selected entries K[m], V[m], shortening the real KV sequence (the attention weights are
// not masked).  Section "what differs": keys of old context take the temporal phase t~(t) = q0 - g(q0 - t); only
// the key phase changes, values and the spatial coordinates are left as they are.  Static heads of the
// head-specialised variant follow the Streaming policy and receive nothing.
//
// Work decomposition ("plane streaming"): the mask is shared by every plane, so the kept rows of one block of the
// index list sit at the same offsets in every plane.  An item is (block of rows, range of planes).  Each thread owns
// kSlots fixed 16-byte vectors of the block (row, vector-in-row), computes their source and destination offsets once
// from the index list, then walks the planes of its range issuing 2 * kSlots independent 16-byte loads (K and V) per
// plane with no dependent load in between.  Stores of a block are contiguous (the history tail).  Every source
// vector is read once and every destination vector written once.  Key vectors that hold temporal pairs are turned
// with the frame's cos/sin table before they are stored.
//
// Bookkeeping folded in: the item holding the first block of a receiving plane sets its hist_len to
// common_len + k, and the items of the lowest receiving plane append the kept frames to hist_t.
#include "dcp_internal.cuh"

namespace dcp {

namespace {

__global__ void __launch_bounds__(kThreads, 4) gather_kernel(const GatherParams p) {
  wait_for_predecessor();
  const Ctrl* c = p.ctrl;
  if (c->abort || !c->has_dyn) return;
  const int k = c->k;
  if (k <= 0) return;
  const int64_t common = c->common_len;
  const int first_dyn = c->first_dyn;
  const int rows_per_item = (kThreads * kSlots) / p.vpr;
  const int nblk = (k + rows_per_item - 1) / rows_per_item;
  int ranges = (int)gridDim.x / nblk;
  if (ranges < 1) ranges = 1;
  if (ranges > p.n_planes) ranges = p.n_planes;
  const int ppr = (p.n_planes + ranges - 1) / ranges;
  const int items = nblk * ranges;
  const int ppv = p.dtype == DCP_BF16 ? 4 : 2;  // rotary pairs per 16-byte vector
  const int temporal_vecs = (p.n_t + ppv - 1) / ppv;

  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int jb = it % nblk, r = it / nblk;
    const int p0 = r * ppr, p1 = min(p.n_planes, p0 + ppr);
    const int j0 = jb * rows_per_item, nrows = min(rows_per_item, k - j0);

    // destination vectors of the block are contiguous: vector e of the block is at dst_block + 16 e
    const int64_t src_slot = p.src_row0 * (int64_t)p.row_bytes;
    const int64_t dst_block = (p.dst_row0 + common + j0) * (int64_t)p.row_bytes;
    int src_rel[kSlots];  // offset of the slot's source vector inside the leaving chunk's rows, -1 if unused
    int rot[kSlots];      // frame (inside the chunk) whose table turns this key vector, -1 if it is only copied
#pragma unroll
    for (int u = 0; u < kSlots; ++u) {
      const int e = threadIdx.x + u * kThreads;
      const int row = e / p.vpr, vec = e - row * p.vpr;
      src_rel[u] = -1;
      rot[u] = -1;
      if (row < nrows) {
        const int s = __ldg(p.idx + j0 + row);
        const int f = s / p.T;
        src_rel[u] = s * p.row_bytes + vec * 16;
        if (vec < temporal_vecs && __ldg(p.rot_g + f)) rot[u] = f;
        if (vec == 0 && first_dyn >= p0 && first_dyn < p1) p.hist_t[common + j0 + row] = p.evict_first_frame + f;
      }
    }

    for (int pl = p0; pl < p1; ++pl) {
      if (p.head_is_static && __ldg(p.head_is_static + pl)) continue;  // Streaming policy: keeps nothing
      char* kb = p.k + pl * p.plane_bytes;
      char* vb = p.v + pl * p.plane_bytes;
      uint4 xk[kSlots], xv[kSlots];
#pragma unroll
      for (int u = 0; u < kSlots; ++u) {
        if (src_rel[u] >= 0) {
          xk[u] = ld_stream(kb + src_slot + src_rel[u]);
          xv[u] = ld_stream(vb + src_slot + src_rel[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kSlots; ++u) {
        if (rot[u] >= 0) {
          const int e = threadIdx.x + u * kThreads;
          const int vec = e % p.vpr;
          xk[u] = dev_rotate_vec(xk[u], p.dtype, vec * ppv, p.n_t, p.trig_g + rot[u] * p.n_t);
        }
      }
#pragma unroll
      for (int u = 0; u < kSlots; ++u) {
        if (src_rel[u] >= 0) {
          const int64_t d = dst_block + (int64_t)(threadIdx.x + u * kThreads) * 16;
          st_stream(kb + d, xk[u]);
          st_stream(vb + d, xv[u]);
        }
      }
      if (jb == 0 && threadIdx.x == 0) p.hist_len[pl] = (int32_t)(common + k);
    }
  }
}

}  // namespace

cudaError_t launch_gather(const GatherParams& p, cudaStream_t s, bool overlap_launch) {
  static int blocks_per_sm = 0;
  if (!blocks_per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, gather_kernel, kThreads, 0) != cudaSuccess ||
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
  return cudaLaunchKernelEx(&cfg, gather_kernel, p);
}

}  // namespace dcp
