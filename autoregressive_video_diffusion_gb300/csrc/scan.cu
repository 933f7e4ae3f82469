// Scan kernel of the prune step: discrepancy score, threshold mask, ordered index list, phase tables and the plane
// checks, in one launch.
//
// The page (DeCoPrune, onedev.kr/papers/726, section "how it works") scores each token of the chunk by
// l = (1/d) ||x0hat(tau*) - x_final||^2, keeps tokens whose l exceeds gamma (one mask for every layer) and keeps
// K[m], V[m] of the kept positions m.  This kernel produces l, the mask and m; the gather kernel moves the rows.
//
// Roles of the 256-thread CTAs (by block index):
//   tile CTAs    [0, n_tiles): score a tile of tokens (a group of lanes per token, 128-bit loads, fp32 shuffle
//                reduction), threshold, and publish the keep bits as warp ballot words.
//   table CTAs   [n_tiles, n_tiles + n_trig_blocks): the cos/sin tables of the key re-phase (section "what
//                differs": t~(t) = q0 - g(q0 - t)) in double precision, stored as float hi/lo pairs.
//   check CTAs   [n_tiles + n_trig_blocks, ...): each folds 256 planes' hist_len into warp-reduced atomic maxima
//                (receiving planes' shortest and longest history, lowest receiving plane, longest history) and, for
//                paged caches, checks 256 block-table entries.  They have CTAs of their own so that no tile starts
//                late (measured: the tiles that also ran the checks finished 0.9 us later).
//   final CTA    the last tile or check CTA to finish (completion counter) turns the ballot words into the ordered
//                index list with one block-wide exclusive scan of their popcounts per 256 words, decides capacity
//                and consistency, publishes the verdict for the kernels that follow and resets the counters.  Under
//                the Random ablation (keep rule 2) it first draws the kept set (radix select, below).  The table
//                CTAs, whose fp64 chains are the slowest part of the kernel, take no part in the count: nothing in
//                the final CTA reads the tables, and the kernels that do wait for the whole grid, so the compaction
//                runs while the tables are still being built instead of after them.
// Every step of that chain is a fixed number of dependent memory round trips; no CTA waits on another.  (A
// decoupled look-back over 98 tiles measured 11.8 us for a 6240-token chunk on GB300, where each polling round is a
// cross-die L2 round trip; this single-pass form removes the polling.)  The kernel lets its dependents launch early
// (programmatic dependent launch); they wait for it to finish before they read anything it wrote.
#include "dcp_internal.cuh"

namespace dcp {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Exclusive scan of one int per thread over the CTA.  Every thread must call it; s_warp holds 8 ints.
__device__ int block_exclusive_scan(int x, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  __syncthreads();  // s_warp may still be read by a previous call
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int s = s_warp[w];
    if (w < warp) base += s;
    tot += s;
  }
  *total = tot;
  return base + v - x;
}

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

// Tiles are multiples of 32 tokens, so warp w of tile t owns ballot word t * tile / 32 + w.
__device__ void tile_work(const ScanParams& p, int tile_id, float* s_ell) {
  const int t0 = tile_id * p.tile;
  const int ntok = min(p.tile, p.n_tok - t0);
  const int tid = threadIdx.x;

  if (p.x0hat) score_tile(p, t0, ntok, s_ell);
  __syncthreads();

  bool keep = false;
  if (tid < ntok) {
    if (p.x0hat) {
      const float l = s_ell[tid];
      const bool large = l > p.gamma;
      keep = p.keep_rule == 1 ? !large : large;  // rule 2 publishes rule 0's bits: the final CTA draws that many
      if (p.ell_out) p.ell_out[t0 + tid] = l;
    } else {
      keep = p.mask_in[t0 + tid] != 0;
    }
    if (p.mask_out && !(p.x0hat && p.keep_rule == 2)) p.mask_out[t0 + tid] = (uint8_t)keep;
  }
  const unsigned word = __ballot_sync(kFull, keep);
  const int w = tid >> 5;
  if ((tid & 31) == 0 && w * 32 < ntok) p.bits[(t0 >> 5) + w] = word;
}

__device__ void plane_checks(const ScanParams& p, int slice, int* s_warp, int* s_base) {
  const int pl = slice * kThreads + threadIdx.x;
  int len1 = 0, min_inv = 0, first_inv = 0, longest = 0, bad = 0, all_min_inv = 0;
  if (pl < p.n_planes) {
    const int len = p.hist_len[pl];
    if (len < 0 || len > p.hist_cap) {
      bad = 1;
    } else {
      longest = len;
      all_min_inv = INT32_MAX - len;
      const bool receives = p.update_cache && !(p.head_is_static && p.head_is_static[pl]);
      if (receives) {
        len1 = len + 1;
        min_inv = INT32_MAX - len;
        first_inv = INT32_MAX - pl;
      }
    }
  }
  if (p.dyn_list) {  // list the receiving planes: in plane order within this CTA's 256, one atomic per CTA
    int total = 0;
    const int rank = block_exclusive_scan(len1 > 0 ? 1 : 0, s_warp, &total);
    if (threadIdx.x == 0) *s_base = total ? atomicAdd(&p.ctrl->acc_n_dyn, total) : 0;
    __syncthreads();
    if (len1 > 0) p.dyn_list[*s_base + rank] = pl;
  }
  len1 = __reduce_max_sync(kFull, len1);
  min_inv = __reduce_max_sync(kFull, min_inv);
  first_inv = __reduce_max_sync(kFull, first_inv);
  longest = __reduce_max_sync(kFull, longest);
  all_min_inv = __reduce_max_sync(kFull, all_min_inv);
  bad = __reduce_max_sync(kFull, bad);
  if ((threadIdx.x & 31) == 0) {
    Ctrl* c = p.ctrl;
    if (len1) {
      atomicMax(&c->acc_len_max1, len1);
      atomicMax(&c->acc_len_min_inv, min_inv);
      atomicMax(&c->acc_first_inv, first_inv);
    }
    if (longest) atomicMax(&c->acc_rp_max, longest);
    if (all_min_inv) atomicMax(&c->acc_all_min_inv, all_min_inv);
    if (bad) atomicMax(&c->acc_bad, 1);
  }
}

// Paged caches: every block-table entry the step uses must name a block of the pools.  A bad entry aborts the step
// before anything moves (the gather and re-index kernels read the tables only after the verdict).
__device__ void table_checks(const ScanParams& p, int slice) {
  const int e = slice * kThreads + threadIdx.x;
  int bad = 0;
  if (e < p.n_tbl_a + p.n_tbl_b) {
    const int32_t b = e < p.n_tbl_a ? p.tbl_a[e] : p.tbl_b[e - p.n_tbl_a];
    bad = b < 0 || (int64_t)b >= p.n_blocks;
  }
  bad = __reduce_max_sync(kFull, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicMax(&p.ctrl->acc_bad, 1);
}

// theta_p = base^(-p / n_t) is evaluated as exp2(log2(base) * (-p / n_t)) (dev_turn_entry).
__device__ void table_work(const ScanParams& p, int block) {
  if (threadIdx.x >= p.tbl_per) return;
  const double log2_base = log2(p.base);
  const int e = block * p.tbl_per + threadIdx.x;
  const int n_g = p.g_frames * p.n_t;
  const int n_h = (p.h_hi - p.h_lo) * p.n_t;
  if (e < n_g) {
    const int f = e / p.n_t, pp = e - f * p.n_t;
    bool moves = false;
    p.trig_g[e] = dev_turn_entry((double)(p.evict_first_frame + f), pp, p.n_t, log2_base, (double)p.q0,
                                 (double)p.T_s, p.R, p.S, p.g_mode, p.g_identity != 0, &moves);
    if (pp == 0) p.rot_g[f] = moves ? 1 : 0;
  } else if (e - n_g < n_h) {
    const int e2 = e - n_g;
    const int f = e2 / p.n_t, pp = e2 - f * p.n_t;
    const int t = p.h_lo + f;
    bool moves = false;
    p.trig_h[(int64_t)t * p.n_t + pp] = dev_reindex_entry((double)t, pp, p.n_t, log2_base, (double)p.q0_prev,
                                                          (double)p.q0, (double)p.T_s, p.R, p.S, p.g_mode, &moves);
    if (pp == 0) p.rot_h[t] = moves ? 1 : 0;
  }
}

// ------------------------------------------------------------------------------------------ Random ablation
// Section "premises and limits" of the page compares DeCoPrune with a Random policy at the same compression ratio.
// Keep rule 2 keeps as many tokens as the discrepancy rule would, drawn uniformly without replacement: token n gets
// the priority z_n, the n-th output (0-based) of a SplitMix64 sequence (Steele, Lea & Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014) seeded with the call's stream, and the tokens with the smallest
// priorities are kept.  The state steps by an odd constant and the output function is a bijection of 64-bit words,
// so the priorities of one chunk are distinct and the kept set is unique.
__device__ __forceinline__ uint64_t dev_splitmix64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

struct Pick {          // kept set of rule 2: any && (z >> shift) <= prefix
  uint64_t prefix;
  int shift;
  bool any;
};

// Radix select, most significant byte first, of the target-th smallest priority in one CTA (s_pick: kThreads + 3
// ints).  A pass histograms the next byte of the priorities that still match the chosen prefix; the byte whose
// bin holds the remaining rank extends the prefix.  It stops as soon as the whole bin is taken; with distinct
// priorities that happens at the latest when one priority is left (byte 0).  The count of rule 0 comes from the
// ballot words the tile CTAs published.
__device__ Pick random_pick(const ScanParams& p, int n_words, int* s_warp, int* s_pick) {
  int target = 0;  // same value in every thread
  for (int w0 = 0; w0 < n_words; w0 += kThreads) {
    const int wi = w0 + threadIdx.x;
    int total = 0;
    block_exclusive_scan(wi < n_words ? __popc(__ldcg(p.bits + wi)) : 0, s_warp, &total);
    target += total;
  }
  Pick pk{0ull, 0, target > 0};
  if (!pk.any) return pk;
  int r = target;
  uint64_t prefix = 0;
  for (int shift = 56; shift >= 0; shift -= 8) {
    s_pick[threadIdx.x] = 0;
    __syncthreads();
    for (int n = threadIdx.x; n < p.n_tok; n += kThreads) {
      const uint64_t z = dev_splitmix64(p.random_stream, (uint64_t)n);
      if (shift == 56 || (z >> (shift + 8)) == prefix) atomicAdd(&s_pick[(z >> shift) & 255], 1);
    }
    __syncthreads();
    const int h = s_pick[threadIdx.x];
    int total = 0;
    const int below = block_exclusive_scan(h, s_warp, &total);
    if (below < r && r <= below + h) {
      s_pick[kThreads] = threadIdx.x;
      s_pick[kThreads + 1] = below;
      s_pick[kThreads + 2] = h;
    }
    __syncthreads();
    const int digit = s_pick[kThreads], taken_below = s_pick[kThreads + 1], in_bin = s_pick[kThreads + 2];
    r -= taken_below;
    prefix = (prefix << 8) | (uint64_t)digit;
    pk.prefix = prefix;
    pk.shift = shift;
    if (r == in_bin) break;
  }
  return pk;
}

// Ballot word wi of rule 2's kept set; also writes those tokens' mask bytes.
__device__ unsigned random_word(const ScanParams& p, const Pick& pk, int wi) {
  unsigned word = 0u;
  for (int b = 0; b < 32; ++b) {
    const int n = wi * 32 + b;
    if (n >= p.n_tok) break;
    const bool keep = pk.any && (dev_splitmix64(p.random_stream, (uint64_t)n) >> pk.shift) <= pk.prefix;
    word |= (unsigned)keep << b;
    if (p.mask_out) p.mask_out[n] = (uint8_t)keep;
  }
  return word;
}

// The last CTA: ballot words -> ordered index list (block scan of popcounts), then the step's verdict.
__device__ void finalize(const ScanParams& p, int* s_warp, int* s_pick) {
  Ctrl* c = p.ctrl;
  const int n_words = p.n_tiles > 0 ? (p.n_tok + 31) >> 5 : 0;
  const bool random = p.x0hat && p.keep_rule == 2;
  // the check accumulators (other CTAs' atomics), read now so their round trip overlaps the ballot words' loads
  int len1 = 0, min_inv = 0, first_inv = 0, longest = 0, bad = 0, all_min_inv = 0, n_dyn = 0;
  if (threadIdx.x == 0) {
    n_dyn = __ldcg(&c->acc_n_dyn);
    len1 = __ldcg(&c->acc_len_max1);
    min_inv = __ldcg(&c->acc_len_min_inv);
    first_inv = __ldcg(&c->acc_first_inv);
    longest = __ldcg(&c->acc_rp_max);
    bad = __ldcg(&c->acc_bad);
    all_min_inv = __ldcg(&c->acc_all_min_inv);
  }
  Pick pk{0ull, 0, false};
  if (random) pk = random_pick(p, n_words, s_warp, s_pick);
  int k = 0;  // same value in every thread
  for (int w0 = 0; w0 < n_words; w0 += kThreads) {
    const int wi = w0 + threadIdx.x;
    unsigned word = 0u;
    if (wi < n_words) word = random ? random_word(p, pk, wi) : __ldcg(p.bits + wi);  // other CTAs' words: via L2
    int total = 0;
    const int excl = block_exclusive_scan(__popc(word), s_warp, &total);
    if (p.idx_out) {
      int pos = k + excl;
      while (word) {
        const int b = __ffs(word) - 1;
        p.idx_out[pos++] = wi * 32 + b;
        word &= word - 1u;
      }
    }
    k += total;
  }
  if (threadIdx.x == 0) {
    int abort = 0;
    const bool has_dyn = p.update_cache && len1 > 0;
    int common = 0, first = -1;
    if ((p.update_cache || p.want_rephase) && bad) {
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
    c->rp_min = (p.want_rephase && all_min_inv > 0 && !bad) ? INT32_MAX - all_min_inv : 0;
    c->abort = abort;
    if (p.kept_dev) *p.kept_dev = k;
    if (p.kept_host) *reinterpret_cast<volatile int32_t*>(p.kept_host) = k;  // over the host link
    c->acc_len_max1 = 0;
    c->acc_len_min_inv = 0;
    c->acc_first_inv = 0;
    c->acc_rp_max = 0;
    c->acc_all_min_inv = 0;
    c->acc_bad = 0;
    c->n_dyn = n_dyn;
    c->acc_n_dyn = 0;
    c->done = 0u;
  }
}

__global__ void __launch_bounds__(kThreads) scan_kernel(const ScanParams p) {
  __shared__ float s_ell[kMaxTile];
  __shared__ int s_warp[kThreads / 32];
  __shared__ int s_pick[kThreads + 3];
  __shared__ int s_last;
  allow_dependents();
  const int id = blockIdx.x;
  const int check0 = p.n_tiles + p.n_trig_blocks;  // the check CTAs follow the tile and table CTAs
  if (id < p.n_tiles) {
    tile_work(p, id, s_ell);
  } else if (id < check0) {
    table_work(p, id - p.n_tiles);
    if (p.n_counted < (int)gridDim.x) return;  // not counted: the tables are read by the later kernels only
  }
  if (id >= check0 && id - check0 < p.n_plane_slices) plane_checks(p, id - check0, s_warp, &s_last);
  if (id >= check0 && id - check0 < p.n_tbl_slices) table_checks(p, id - check0);

  // Completion: the final CTA reads the ballot words (stored by lane 0 of each tile warp) and the atomically folded
  // plane checks.  The barrier orders them before thread 0's fence, and the fence before the completion count.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&p.ctrl->done, 1u) == (unsigned)p.n_counted - 1;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (s_last) finalize(p, s_warp, s_pick);
}

// Phase table on its own (dcp_phase_table): one entry per thread, 64-thread CTAs to spread the fp64 work over SMs.
__global__ void __launch_bounds__(kTableEntries) phase_table_kernel(float4* out, int32_t frame_lo, int32_t n_entries,
                                                                    int32_t n_t, double base, double R, double S,
                                                                    int32_t g_mode, int32_t T_s, int32_t q0) {
  const int e = blockIdx.x * kTableEntries + threadIdx.x;
  if (e >= n_entries) return;
  const int f = e / n_t, pp = e - f * n_t;
  bool moves = false;
  out[e] = dev_turn_entry((double)(frame_lo + f), pp, n_t, log2(base), (double)q0, (double)T_s, R, S, g_mode, false,
                          &moves);
}

}  // namespace

cudaError_t launch_phase_table(float4* out, int32_t frame_lo, int32_t n_entries, int32_t n_t, double base, double R,
                               double S, int32_t g_mode, int32_t T_s, int32_t q0, cudaStream_t s) {
  if (n_entries <= 0) return cudaSuccess;
  phase_table_kernel<<<(n_entries + kTableEntries - 1) / kTableEntries, kTableEntries, 0, s>>>(
      out, frame_lo, n_entries, n_t, base, R, S, g_mode, T_s, q0);
  return cudaGetLastError();
}

cudaError_t launch_scan(const ScanParams& p, cudaStream_t s) {
  const int checks = p.n_plane_slices > p.n_tbl_slices ? p.n_plane_slices : p.n_tbl_slices;
  int grid = p.n_tiles + p.n_trig_blocks + checks;
  if (grid < 1) grid = 1;
  ScanParams q = p;
  q.n_counted = grid - p.n_trig_blocks;  // tile and check CTAs; all CTAs when there are none
  if (q.n_counted < 1) q.n_counted = grid;
  scan_kernel<<<grid, kThreads, 0, s>>>(q);
  return cudaGetLastError();
}

}  // namespace dcp
