// Gather kernel of the prune step: physical compaction K[m], V[m] of the leaving chunk into the history region of
// every dynamic (layer, head) plane, with the temporal RoPE re-phase of each moved key fused in.
//
// Page: DeCoPrune (onedev.kr/papers/726).  Section "how it works": when a non-sink chunk leaves the dense window,
// each layer keeps only the selected entries K[m], V[m], shortening the real KV sequence (the attention weights are
// not masked).  Section "what differs": keys of old context take the temporal phase t~(t) = q0 - g(q0 - t); only
// the key phase changes, values and the spatial coordinates are left as they are.
//
// Work decomposition: an item is (tensor, dynamic plane, block of rows_per_item kept rows).  A persistent grid
// walks the items; inside an item each thread moves 16-byte vectors (4 loads in flight per thread), so a warp
// reads two 256-byte rows per instruction and the destination block is written contiguously.  Vectors of key rows
// that hold temporal pairs are turned with the frame's cos/sin table before they are stored.  Every source row is
// read once and every destination row written once.
#include "dcp_internal.cuh"

namespace dcp {

namespace {

constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherParams p) {
  const Ctrl* c = p.ctrl;
  if (c->abort) return;
  const int k = c->k, n_dyn = c->n_dyn;
  if (k <= 0 || n_dyn <= 0) return;
  const int64_t common = c->common_len;
  const int rpi = p.rows_per_item;
  const int nblk = (k + rpi - 1) / rpi;
  const int64_t per_tensor = (int64_t)n_dyn * nblk;
  const int64_t items = 2 * per_tensor;
  const int ppv = p.dtype == DCP_BF16 ? 4 : 2;  // rotary pairs per 16-byte vector
  const int temporal_vecs = (p.n_t + ppv - 1) / ppv;

  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int is_v = it >= per_tensor;
    const int64_t r = is_v ? it - per_tensor : it;
    const int hi = (int)(r / nblk), jb = (int)(r - (int64_t)hi * nblk);
    const int plane = __ldg(p.dyn_list + hi);
    const int j0 = jb * rpi, nrows = min(rpi, k - j0);
    char* base = (is_v ? p.v : p.k) + (int64_t)plane * p.plane_bytes;
    const char* src0 = base + p.src_row0 * p.row_bytes;
    char* dst0 = base + (p.dst_row0 + common + j0) * p.row_bytes;
    const int nvec = nrows * p.vpr;

    for (int e0 = threadIdx.x; e0 < nvec; e0 += kThreads * kUnroll) {
      uint4 x[kUnroll];
      int jj[kUnroll], vv[kUnroll], ss[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int e = e0 + u * kThreads;
        jj[u] = -1;
        if (e < nvec) {
          const int j = p.vpr_shift >= 0 ? (e >> p.vpr_shift) : e / p.vpr;
          const int vec = e - j * p.vpr;
          const int s = __ldg(p.idx + j0 + j);
          jj[u] = j;
          vv[u] = vec;
          ss[u] = s;
          x[u] = ld_stream(src0 + (int64_t)s * p.row_bytes + vec * 16);
        }
      }
      if (!is_v) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          if (jj[u] >= 0 && vv[u] < temporal_vecs) {
            const int f = ss[u] / p.T;
            if (__ldg(p.rot_g + f)) x[u] = dev_rotate_vec(x[u], p.dtype, vv[u] * ppv, p.n_t, p.trig_g + f * p.n_t);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (jj[u] >= 0) st_stream(dst0 + (int64_t)jj[u] * p.row_bytes + vv[u] * 16, x[u]);
    }
  }
}

}  // namespace

cudaError_t launch_gather(const GatherParams& p, cudaStream_t s) {
  static int blocks_per_sm = 0;
  if (!blocks_per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, gather_kernel, kThreads, 0) != cudaSuccess ||
        blocks_per_sm < 1)
      blocks_per_sm = 1;
  }
  gather_kernel<<<sm_count() * blocks_per_sm, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dcp
