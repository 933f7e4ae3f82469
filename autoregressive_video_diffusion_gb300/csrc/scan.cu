// Scan kernel of the prune step: discrepancy score, threshold mask, ordered index list, phase tables and the cache
// bookkeeping, in one launch.
//
// The page (DeCoPrune, onedev.kr/papers/726, section "how it works") scores each token of the chunk by
// l = (1/d) ||x0hat(tau*) - x_final||^2, keeps tokens whose l exceeds gamma (one mask for every layer) and keeps
// K[m], V[m] of the kept positions m.  This kernel produces l, the mask and m; the gather kernel moves the rows.
//
// Structure (one 256-thread CTA per tile of tokens, plus table CTAs, numbered in start order by a ticket):
//   tile CTAs   score their tokens (a group of lanes per token, 128-bit loads, fp32 shuffle reduction), vote the
//               mask bits with ballots, scan them inside the CTA and find the tile's global offset by decoupled
//               look-back over the predecessors' published counts (bounded wait: a tile that gives up records
//               DCP_ETIMEOUT and the whole call is abandoned), then write their kept positions.
//   table CTAs  build the cos/sin tables of the key re-phase (section "what differs": t~(t) = q0 - g(q0 - t)) in
//               double precision, stored as float hi/lo pairs.
//   plane checks the CTAs numbered below ceil(planes / 256) also read 256 planes' hist_len each and fold them into
//               warp-reduced atomic maxima (receiving planes' shortest and longest history, lowest receiving plane,
//               longest history of any plane).
//   final CTA   (the last to finish) reads the kept count and the plane checks, decides capacity and consistency,
//               publishes the verdict for the kernels that follow, and resets the scan state for the next call.
// The kernel lets its dependents launch early (programmatic dependent launch); they wait for it to finish before
// they read anything it wrote.
#include "dcp_internal.cuh"

namespace dcp {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long pack_state(uint32_t flag, int32_t value) {
  return ((unsigned long long)flag << 32) | (uint32_t)value;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Exclusive scan of one int per thread over the CTA.  Every thread must call it; s_warp holds 8 ints.
__device__ int block_exclusive_scan(int x, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  __syncthreads();  // s_warp may still be read by a previous call
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    int s = s_warp[w];
    if (w < warp) base += s;
    tot += s;
  }
  *total = tot;
  return base + v - x;
}

struct TileShared {
  float ell[kMaxTile];
  int warp_tmp[kThreads / 32];
  int excl;
  int timed_out;
};

__device__ void score_tile(const ScanParams& p, int t0, int ntok, float* s_ell) {
  if (p.lpt > 0) {
    // lpt lanes per token, one float4 of each input per lane, up to 4 token passes in flight per thread
    const int lpt = p.lpt, tpp = kThreads / lpt, passes = p.tile / tpp;
    const int sub = threadIdx.x & (lpt - 1), tk = threadIdx.x / lpt;
    float4 a[4], b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      b[i] = a[i];
      const int tok = i * tpp + tk;
      if (i < passes && tok < ntok) {
        const int64_t off = (int64_t)(t0 + tok) * p.d + sub * 4;
        a[i] = __ldcs(reinterpret_cast<const float4*>(p.x0hat + off));
        b[i] = __ldcs(reinterpret_cast<const float4*>(p.xref + off));
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float dx = a[i].x - b[i].x, dy = a[i].y - b[i].y, dz = a[i].z - b[i].z, dw = a[i].w - b[i].w;
      float acc = dx * dx + dy * dy + dz * dz + dw * dw;
      for (int o = lpt >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      const int tok = i * tpp + tk;
      if (i < passes && sub == 0 && tok < ntok) s_ell[tok] = acc / (float)p.d;
    }
  } else {
    // any d: one warp per token, scalar loads strided over the row
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int tok = warp; tok < ntok; tok += kThreads / 32) {
      const float* xa = p.x0hat + (int64_t)(t0 + tok) * p.d;
      const float* xb = p.xref + (int64_t)(t0 + tok) * p.d;
      float acc = 0.f;
      for (int j = lane; j < p.d; j += 32) {
        const float df = xa[j] - xb[j];
        acc += df * df;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      if (lane == 0) s_ell[tok] = acc / (float)p.d;
    }
  }
}

__device__ void tile_work(const ScanParams& p, int tile_id, TileShared& sh) {
  const int t0 = tile_id * p.tile;
  const int ntok = min(p.tile, p.n_tok - t0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (p.x0hat) score_tile(p, t0, ntok, sh.ell);
  __syncthreads();

  int keep = 0;
  if (tid < ntok) {
    if (p.x0hat) {
      const float l = sh.ell[tid];
      const bool large = l > p.gamma;
      keep = p.keep_rule == 0 ? (int)large : (int)!large;
      if (p.ell_out) p.ell_out[t0 + tid] = l;
    } else {
      keep = p.mask_in[t0 + tid] != 0;
    }
    if (p.mask_out) p.mask_out[t0 + tid] = (uint8_t)keep;
  }

  int total = 0;
  const int local = block_exclusive_scan(keep, sh.warp_tmp, &total);

  if (warp == 0) {
    int prefix = 0, timed_out = 0;
    if (tile_id == 0) {
      if (lane == 0 && !p.force_timeout) st_release_u64(p.tile_state, pack_state(kFlagPrefix, total));
    } else {
      if (lane == 0 && !p.force_timeout) st_release_u64(p.tile_state + tile_id, pack_state(kFlagAgg, total));
      const int limit = p.force_timeout ? kForcedSpinLimit : kSpinLimit;
      int pos = tile_id - 1, spins = 0, acc = 0;
      while (true) {
        const int j = pos - lane;
        const unsigned long long st =
            j >= 0 ? ld_acquire_u64(p.tile_state + j) : pack_state(kFlagPrefix, 0);  // nothing precedes tile 0
        const uint32_t flag = (uint32_t)(st >> 32);
        if (__any_sync(kFull, flag == 0u)) {
          if (++spins > limit) {
            timed_out = 1;
            break;
          }
          __nanosleep(64);
          continue;
        }
        const unsigned pm = __ballot_sync(kFull, flag == kFlagPrefix);
        const int first = pm ? __ffs(pm) - 1 : 32;
        acc += warp_sum(lane <= first ? (int)(uint32_t)st : 0);
        if (pm) break;
        pos -= 32;
      }
      if (!timed_out) {
        prefix = acc;
        if (lane == 0 && !p.force_timeout) st_release_u64(p.tile_state + tile_id, pack_state(kFlagPrefix, prefix + total));
      } else if (lane == 0) {
        atomicExch(&p.ctrl->tile_error, 1);
        set_status(p.status, DCP_ETIMEOUT);
      }
    }
    if (lane == 0) {
      sh.excl = prefix;
      sh.timed_out = timed_out;
    }
  }
  __syncthreads();
  if (keep && p.idx_out && !sh.timed_out) p.idx_out[sh.excl + local] = t0 + tid;
}

__device__ void plane_checks(const ScanParams& p, int slice) {
  const int pl = slice * kThreads + threadIdx.x;
  int len1 = 0, min_inv = 0, first_inv = 0, longest = 0, bad = 0;
  if (pl < p.n_planes) {
    const int len = p.hist_len[pl];
    if (len < 0 || len > p.hist_cap) {
      bad = 1;
    } else {
      longest = len;
      const bool receives = p.update_cache && !(p.head_is_static && p.head_is_static[pl]);
      if (receives) {
        len1 = len + 1;
        min_inv = INT32_MAX - len;
        first_inv = INT32_MAX - pl;
      }
    }
  }
  len1 = __reduce_max_sync(kFull, len1);
  min_inv = __reduce_max_sync(kFull, min_inv);
  first_inv = __reduce_max_sync(kFull, first_inv);
  longest = __reduce_max_sync(kFull, longest);
  bad = __reduce_max_sync(kFull, bad);
  if ((threadIdx.x & 31) == 0) {
    Ctrl* c = p.ctrl;
    if (len1) {
      atomicMax(&c->acc_len_max1, len1);
      atomicMax(&c->acc_len_min_inv, min_inv);
      atomicMax(&c->acc_first_inv, first_inv);
    }
    if (longest) atomicMax(&c->acc_rp_max, longest);
    if (bad) atomicMax(&c->acc_bad, 1);
  }
}

__device__ void table_work(const ScanParams& p, int block) {
  if (threadIdx.x >= kTableEntries) return;
  const int e = block * kTableEntries + threadIdx.x;
  const int n_g = p.g_frames * p.n_t;
  const int n_h = (p.h_hi - p.h_lo) * p.n_t;
  if (e < n_g) {
    const int f = e / p.n_t, pp = e - f * p.n_t;
    const double t = (double)(p.evict_first_frame + f);
    const double delta = __dsub_rn(dev_phase(t, (double)p.q0, (double)p.T_s, p.R, p.S, p.g_mode), t);
    const double theta = pow(p.base, -(double)pp / (double)p.n_t);
    p.trig_g[e] = dev_trig_entry(__dmul_rn(theta, delta));
    if (pp == 0) p.rot_g[f] = delta != 0.0;
  } else if (e - n_g < n_h) {
    const int e2 = e - n_g;
    const int f = e2 / p.n_t, pp = e2 - f * p.n_t;
    const int t = p.h_lo + f;
    const double before = dev_phase((double)t, (double)p.q0_prev, (double)p.T_s, p.R, p.S, p.g_mode);
    const double after = dev_phase((double)t, (double)p.q0, (double)p.T_s, p.R, p.S, p.g_mode);
    const double delta = __dsub_rn(after, before);
    const double theta = pow(p.base, -(double)pp / (double)p.n_t);
    p.trig_h[(int64_t)t * p.n_t + pp] = dev_trig_entry(__dmul_rn(theta, delta));
    if (pp == 0) p.rot_h[t] = after != before;
  }
}

__device__ __forceinline__ int vload(const int32_t* x) { return *reinterpret_cast<const volatile int32_t*>(x); }

__device__ void finalize(const ScanParams& p) {
  Ctrl* c = p.ctrl;
  if (threadIdx.x == 0) {
    int abort = vload(&c->tile_error) ? 1 : 0;
    int k = 0;
    if (!abort && p.n_tiles > 0) {
      const unsigned long long st = ld_acquire_u64(p.tile_state + p.n_tiles - 1);
      if ((uint32_t)(st >> 32) == kFlagPrefix) {
        k = (int)(uint32_t)st;
      } else {
        abort = 1;
        set_status(p.status, DCP_ETIMEOUT);
      }
    }
    const int len1 = vload(&c->acc_len_max1), min_inv = vload(&c->acc_len_min_inv);
    const int first_inv = vload(&c->acc_first_inv), longest = vload(&c->acc_rp_max), bad = vload(&c->acc_bad);
    const bool has_dyn = p.update_cache && len1 > 0;
    int common = 0, first = -1;
    if ((p.update_cache || p.want_rephase) && bad && !abort) {
      abort = 1;
      set_status(p.status, DCP_EDEVICE);
    }
    if (has_dyn) {
      const int max_len = len1 - 1, min_len = INT32_MAX - min_inv;
      common = min_len;
      first = INT32_MAX - first_inv;
      if (!abort && min_len != max_len) {
        abort = 1;
        set_status(p.status, DCP_EDEVICE);
      } else if (!abort && (int64_t)min_len + k > p.hist_cap) {
        abort = 1;
        set_status(p.status, DCP_ECAPACITY);
      }
    }
    c->k = k;
    c->has_dyn = has_dyn ? 1 : 0;
    c->common_len = common;
    c->first_dyn = first;
    c->rp_max = p.want_rephase ? longest : 0;
    c->abort = abort;
    if (p.kept_dev) *p.kept_dev = k;
    c->acc_len_max1 = 0;
    c->acc_len_min_inv = 0;
    c->acc_first_inv = 0;
    c->acc_rp_max = 0;
    c->acc_bad = 0;
    c->tile_error = 0;
    c->ticket = 0u;
    c->done = 0u;
  }
  __syncthreads();  // thread 0 has read the last tile's state; only now may the states be cleared
  for (int i = threadIdx.x; i < p.n_tiles; i += kThreads) p.tile_state[i] = 0ull;
}

__global__ void __launch_bounds__(kThreads) scan_kernel(const ScanParams p) {
  __shared__ TileShared sh;
  __shared__ int s_id, s_last;
  allow_dependents();
  if (threadIdx.x == 0) s_id = (int)atomicAdd(&p.ctrl->ticket, 1u);
  __syncthreads();
  const int id = s_id;
  if (id < p.n_plane_slices) plane_checks(p, id);
  if (id < p.n_tiles) tile_work(p, id, sh);
  else if (id - p.n_tiles < p.n_trig_blocks) table_work(p, id - p.n_tiles);

  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.ctrl->done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (s_last) {
    __threadfence();
    finalize(p);
  }
}

}  // namespace

cudaError_t launch_scan(const ScanParams& p, cudaStream_t s) {
  int grid = p.n_tiles + p.n_trig_blocks;
  if (grid < p.n_plane_slices) grid = p.n_plane_slices;
  if (grid < 1) grid = 1;
  scan_kernel<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dcp
