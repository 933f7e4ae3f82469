// Body of the history re-index, shared by the re-index kernel (rephase.cu) and the fused re-index + gather kernel
// (gather.cu).  See rephase.cu for the method and the work decomposition.
#pragma once

#include <type_traits>

#include "dcp_internal.cuh"

namespace dcp {

#ifdef __CUDACC__

// Rows per work unit and the number of (row block, plane) units of a history of rp_max rows.
__device__ __forceinline__ int64_t rephase_unit_count(const RephaseParams& p, int rp_max, int* rows_per_item) {
  *rows_per_item = kThreads / p.nvt;  // nvt <= kThreads: rows are at most 4 KiB
  const int nblk = (rp_max + *rows_per_item - 1) / *rows_per_item;
  return (int64_t)nblk * p.n_planes;
}

// Re-index units [u_begin, u_end) of the (row block, plane) grid, block-major: a CTA's contiguous share.  Every
// thread of the CTA must call it (it synchronises the CTA once per row block).  uniform_len >= 0: every plane's
// history before the step has that many rows (the fused kernel, whose gather grows hist_len while this runs);
// uniform_len < 0: each plane's length is read from hist_len.  PIF planes are loaded before any is stored; with PIPE
// the next PIF planes' loads are also in flight while a group is turned and stored (twice the registers).
template <int NW, bool PAGED, int PIF, bool PIPE = false>
__device__ __forceinline__ void rephase_units(const RephaseParams& p, int rp_max, int rows_per_item, int uniform_len,
                                              int64_t u_begin, int64_t u_end) {
  using Off = typename std::conditional<PAGED, int64_t, int>::type;
  constexpr int VB = NW * 4;
  const int ppv = p.dtype == DCP_BF16 ? VB / 4 : VB / 8;
  const int row_in_item = threadIdx.x / p.nvt, vec = threadIdx.x - row_in_item * p.nvt;
  const int64_t hist0 = PAGED ? 0 : p.hist_row0 * (int64_t)p.row_bytes;
  auto plane_base = [&](int pl) -> int64_t {
    if (PAGED) return (int64_t)(pl / p.pg.H) * p.pg.s_layer + (int64_t)(pl % p.pg.H) * p.pg.s_head;
    return (int64_t)pl * p.plane_bytes;
  };

  for (int64_t u = u_begin; u < u_end;) {
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

    auto load_group = [&](int pl, Vec<NW>(&x)[PIF], bool(&go)[PIF]) {
#pragma unroll
      for (int q = 0; q < PIF; ++q) {
        const int plq = pl + q;
        go[q] = live && plq < p1 && row < (uniform_len >= 0 ? uniform_len : __ldg(p.hist_len + min(plq, p1 - 1)));
        if (go[q]) ld_plain(x[q], p.k + plane_base(plq) + hist0 + off);
      }
    };
    auto store_group = [&](int pl, Vec<NW>(&x)[PIF], const bool(&go)[PIF]) {
#pragma unroll
      for (int q = 0; q < PIF; ++q) {
        if (go[q]) {
          dev_rotate_vec_regs(x[q], p.dtype, vec * ppv, p.n_t, tr);
          st_plain(p.k + plane_base(pl + q) + hist0 + off, x[q]);
        }
      }
    };
    if (!PIPE) {
      for (int pl = p0; pl < p1; pl += PIF) {
        Vec<NW> x[PIF];
        bool go[PIF];
        load_group(pl, x, go);
        store_group(pl, x, go);
      }
    } else {
      // two register sets in turn: the next group's loads are issued before this group is turned and stored, and
      // no register holding a load in flight is ever copied (a copy would wait for the load)
      Vec<NW> xa[PIF], xb[PIF];
      bool ga[PIF], gb[PIF];
      int pl = p0;
      if (pl < p1) load_group(pl, xa, ga);
      while (pl < p1) {
        if (pl + PIF < p1) load_group(pl + PIF, xb, gb);
        store_group(pl, xa, ga);
        pl += PIF;
        if (pl >= p1) break;
        if (pl + PIF < p1) load_group(pl + PIF, xa, ga);
        store_group(pl, xb, gb);
        pl += PIF;
      }
    }
  }
}

#endif  // __CUDACC__

}  // namespace dcp
