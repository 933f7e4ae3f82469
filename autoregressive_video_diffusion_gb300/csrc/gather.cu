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
// a few fixed vectors of the block (32-byte vectors when rows and bases allow it, else 16-byte), computes their source
// and destination offsets once from the index list, then walks the planes of its range issuing independent loads of
// K and V per plane with no dependent load in between; a block's destination rows are one contiguous run.  Every
// source vector is read once and every destination vector written once.
//
// Slot mapping: the threads of one slot cover whole rows (vpr consecutive threads per row); slot u of lane l takes
// vector (l + u * vpr / slots) mod vpr of its row, so the vectors that hold temporal pairs (the first few of a row)
// are spread over the threads instead of landing on the same lanes in every slot.  Key vectors with temporal pairs
// are turned with the frame's cos/sin table before they are stored.
//
// Bookkeeping folded in: the item holding the first block of a receiving plane sets its hist_len to
// common_len + k, and the items of the lowest receiving plane append the kept frames to hist_t.
//
// A staged form (below) serves contiguous caches of 1024 planes or more: a copy-only form for the steps in which no
// kept key turns, and a form that turns the temporal chunks through registers for the others.
//
// Paged caches (block pools addressed through block tables) use the same decomposition: a thread's source and
// destination offsets inside a plane come from the tables once per item, and a plane's base from its layer and head.
#include <type_traits>

#include "rephase_body.cuh"

namespace dcp {

namespace {

// 2 CTAs per SM (up to 128 registers) so that two planes' vectors fit in registers: the software pipeline keeps the
// next plane's loads in flight while the current plane is turned and stored (measured on the full-depth step:
// 248.5 us vs 253.2 us without the pipeline at 3 CTAs/SM; 259.2 us vs 269.9 us when every key turns; at 3 CTAs/SM
// the pipelined form spills).
// Shared memory of the gathers that turn keys: the leaving chunk's cos/sin table (F x n_t entries), then one flag per
// frame ("this frame's keys turn").
__host__ __device__ inline size_t table_smem_bytes(int n_frames, int n_t) {
  return 16 * (size_t)n_frames * n_t + (((size_t)n_frames + 15) & ~(size_t)15);
}

// After the wait for the scan: its table of the leaving chunk, into shared memory (nothing when no key turns).  A CTA
// barrier must follow before use.
__device__ __forceinline__ void table_copy(const GatherParams& p, float4* s_trig) {
  if (p.no_turn) return;
  uint8_t* s_rot = reinterpret_cast<uint8_t*>(s_trig + p.n_frames * p.n_t);
  for (int e = threadIdx.x; e < p.n_frames * p.n_t; e += kThreads) s_trig[e] = p.trig_g[e];
  for (int f = threadIdx.x; f < p.n_frames; f += kThreads) s_rot[f] = p.rot_g[f];
}

// The gather of one launch, after the predecessor's verdict (not aborted) has been read.  s_trig: shared memory for
// the leaving chunk's cos/sin table and frame flags (table_smem_bytes).  Every thread of the CTA must call it.
template <int NW, bool PAGED, bool LIST>
__device__ __forceinline__ void gather_body(const GatherParams& p, const Ctrl* c, float4* s_trig) {
  using Off = typename std::conditional<PAGED, int64_t, int>::type;
  constexpr int VB = NW * 4;                      // bytes per vector
  constexpr int SLOTS = kBytesPerThread / VB;     // vectors per thread, tensor and plane
  if (!c->has_dyn) return;
  const int k = c->k;
  if (k <= 0) return;
  // turned key vectors read their cos/sin entries from shared memory (measured with every key turning: gather
  // 249.5 vs 254.2 us reading them through L1 from the workspace)
  table_copy(p, s_trig);
  __syncthreads();
  const uint8_t* s_rot = reinterpret_cast<const uint8_t*>(s_trig + p.n_frames * p.n_t);
  const int64_t common = c->common_len;
  const int first_dyn = c->first_dyn;
  const int vpr = p.row_bytes / VB;               // vectors per row (<= kThreads: rows are at most 4 KiB)
  const int rows_per_slot = kThreads / vpr;
  const int rows_per_item = SLOTS * rows_per_slot;
  const int shift = vpr >= SLOTS ? vpr / SLOTS : 1;
  const int nblk = (k + rows_per_item - 1) / rows_per_item;
  // about four smaller items per CTA rather than one large one (measured on the full-depth step: gather 238.9 vs
  // 240.3 us, and 252.2 vs 256.9 us when every key turns)
  const int n_seq = LIST ? c->n_dyn : p.n_planes;  // planes split into ranges (all, or the receiving list)
  int ranges = (int)gridDim.x * 4 / nblk;
  if (ranges > n_seq / 4) ranges = n_seq / 4;  // at least four planes per item (small caches)
  if (ranges < 1) ranges = 1;
  const int ppr = (n_seq + ranges - 1) / ranges;
  const int items = nblk * ranges;
  const int ppv = p.dtype == DCP_BF16 ? VB / 4 : VB / 8;   // rotary pairs per vector
  const int temporal_vecs = (p.n_t + ppv - 1) / ppv;
  const int row_in_slot = threadIdx.x / vpr, lane_in_row = threadIdx.x - row_in_slot * vpr;
  const int64_t src_slot = PAGED ? 0 : p.src_row0 * (int64_t)p.row_bytes;
  auto plane_base = [&](int pl) -> int64_t {
    if (PAGED) return (int64_t)(pl / p.pg.H) * p.pg.s_layer + (int64_t)(pl % p.pg.H) * p.pg.s_head;
    return (int64_t)pl * p.plane_bytes;
  };

  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int jb = it % nblk, r = it / nblk;
    const int p0 = r * ppr, p1 = min(n_seq, p0 + ppr);  // positions in the plane sequence
    const int j0 = jb * rows_per_item, nrows = min(rows_per_item, k - j0);
    const int64_t dst_block = PAGED ? 0 : (p.dst_row0 + common + j0) * (int64_t)p.row_bytes;

    Off src_rel[SLOTS];  // source vector inside the leaving chunk's rows, -1 if the slot is unused
    Off dst_rel[SLOTS];  // destination vector inside the block's contiguous destination rows (paged: in the plane)
    int rot[SLOTS];      // (frame << 16) | vector for a key vector the frame's table turns, -1 if it is only copied
#pragma unroll
    for (int u = 0; u < SLOTS; ++u) {
      const int row = u * rows_per_slot + row_in_slot;
      const int vec = (lane_in_row + u * shift) % vpr;
      src_rel[u] = -1;
      dst_rel[u] = 0;
      rot[u] = -1;
      if (row_in_slot < rows_per_slot && row < nrows) {
        const int s = __ldg(p.idx + j0 + row);
        const int f = s / p.T;
        if (PAGED) {
          const int64_t pos = common + j0 + row;
          src_rel[u] = (int64_t)__ldg(p.pg.src_blocks + s / p.pg.bs) * p.pg.s_block +
                       (int64_t)(s % p.pg.bs) * p.pg.s_row + vec * VB;
          dst_rel[u] = (int64_t)__ldg(p.pg.hist_blocks + pos / p.pg.bs) * p.pg.s_block +
                       (pos % p.pg.bs) * p.pg.s_row + vec * VB;
        } else {
          src_rel[u] = s * p.row_bytes + vec * VB;
          dst_rel[u] = row * p.row_bytes + vec * VB;
        }
        if (vec < temporal_vecs && !p.no_turn && s_rot[f]) rot[u] = (f << 16) | vec;
        const bool writes_t = LIST ? r == 0 : first_dyn >= p0 && first_dyn < p1;  // one item per row block
        if (vec == 0 && writes_t) p.hist_t[common + j0 + row] = p.evict_first_frame + f;
      }
    }

    auto receives = [&](int j) { return LIST || !(p.head_is_static && __ldg(p.head_is_static + j)); };
    auto plane_of = [&](int j) { return LIST ? __ldg(p.dyn_list + j) : j; };
    // software pipeline over the planes: the next receiving plane's loads are in flight while this one is turned
    // and stored
    int pj = p0;
    while (pj < p1 && !receives(pj)) ++pj;
    Vec<NW> ck[SLOTS], cv[SLOTS], nk[SLOTS], nv[SLOTS];
    if (pj < p1) {
      const int pl = plane_of(pj);
#pragma unroll
      for (int u = 0; u < SLOTS; ++u)
        if (src_rel[u] >= 0) {
          ld_stream(ck[u], p.k + plane_base(pl) + src_slot + src_rel[u]);
          ld_stream(cv[u], p.v + plane_base(pl) + src_slot + src_rel[u]);
        }
    }
    while (pj < p1) {
      const int pl = plane_of(pj);
      int nj = pj + 1;
      while (nj < p1 && !receives(nj)) ++nj;
      if (nj < p1) {
        const int nx = plane_of(nj);
#pragma unroll
        for (int u = 0; u < SLOTS; ++u)
          if (src_rel[u] >= 0) {
            ld_stream(nk[u], p.k + plane_base(nx) + src_slot + src_rel[u]);
            ld_stream(nv[u], p.v + plane_base(nx) + src_slot + src_rel[u]);
          }
      }
#pragma unroll
      for (int u = 0; u < SLOTS; ++u)
        if (rot[u] >= 0)
          dev_rotate_vec(ck[u], p.dtype, (rot[u] & 0xFFFF) * ppv, p.n_t, s_trig + (rot[u] >> 16) * p.n_t);
      char* kb = p.k + plane_base(pl);
      char* vb = p.v + plane_base(pl);
#pragma unroll
      for (int u = 0; u < SLOTS; ++u) {
        if (src_rel[u] >= 0) {
          st_stream(kb + dst_block + dst_rel[u], ck[u]);
          st_stream(vb + dst_block + dst_rel[u], cv[u]);
        }
      }
      if (jb == 0 && threadIdx.x == 0) p.hist_len[pl] = (int32_t)(common + k);
#pragma unroll
      for (int u = 0; u < SLOTS; ++u) {
        ck[u] = nk[u];
        cv[u] = nv[u];
      }
      pj = nj;
    }
  }
}

template <int NW, bool PAGED, bool LIST>
__global__ void __launch_bounds__(kThreads, 2) gather_kernel(const GatherParams p) {
  extern __shared__ float4 s_trig[];               // the leaving chunk's cos/sin table and frame flags
  wait_for_predecessor();
  const Ctrl* c = p.ctrl;
  if (c->abort) return;
  gather_body<NW, PAGED, LIST>(p, c, s_trig);
}

// Re-index and gather of one prune step in one launch, for steps in which every plane receives the kept rows (no
// static heads).  The two touch disjoint rows: the gather appends rows [common_len, common_len + k) and their frames,
// the re-index turns history rows [0, common_len) of every plane (every plane's length before the step is the scan's
// common_len, so hist_len, which the gather grows, is not read).  Each CTA first takes its gather items, then
// re-indexes its equal contiguous share of the (row block, plane) units; one launch instead of two removes the second
// kernel's ramp and tail.  Measured against the two kernels (mid eviction; last ten steps of the eager minute
// rollout): 45.1 vs 48.1 us and 1114.5 vs 1122.3 us with the gather first and four planes in flight per re-index
// thread; the re-index first measured 1118.5 us, six planes in flight 1138-1150 us, and three CTAs per SM (the
// re-index kernel's own occupancy, with a gather that holds one plane at a time) 1199.8 us.  The re-index here keeps
// the next group of four planes' loads in flight while a group is turned and stored (two register sets in turn):
// rollout 1096.6-1097.8 vs 1109.9-1110.9 us without (two planes per group: 1262.6 us).
constexpr int kFusedPlanesInFlight = 4;

template <int NW, bool PAGED>
__global__ void __launch_bounds__(kThreads, 2) step_kernel(const GatherParams gp, const RephaseParams rp) {
  extern __shared__ float4 s_trig[];
  wait_for_predecessor();
  const Ctrl* c = gp.ctrl;
  if (c->abort) return;
  gather_body<NW, PAGED, false>(gp, c, s_trig);
  const int rp_max = c->rp_max;  // = common_len: every plane receives, and the scan checked they agree
  if (rp_max > 0 && rp.nvt > 0) {
    int rows_per_item = 0;
    const int64_t units = rephase_unit_count(rp, rp_max, &rows_per_item);
    rephase_units<NW, PAGED, kFusedPlanesInFlight, true>(rp, rp_max, rows_per_item, rp_max,
                                                         units * blockIdx.x / gridDim.x,
                                                         units * (blockIdx.x + 1) / gridDim.x);
  }
}

// Staged form, for caches of 1024 planes or more.  256 threads, two CTAs per SM, item = (block of up to 64 kept rows,
// range of planes) as above.  Per receiving plane, every thread copies its share of the block's K and V rows into a
// shared-memory stage with 16-byte cp.async (the LSU path: fine-grained requests for the scattered source rows, no
// registers held); when a stage has landed (cp.async groups + one CTA barrier), thread 0 writes the block's two
// destination runs, which are contiguous, with one bulk copy each (TMA).  Three planes are in flight per CTA, twice
// what registers allow in the kernel above (measured on the full-depth step: gather 236.0 vs 240.4 us).
//
// TURN = false serves steps in which no kept key turns (no_turn: the phase map is the identity on the leaving chunk,
// decided on the host from g's closed form; the scan then builds no cos/sin table for the chunk): rows move unchanged.
// TURN = true serves steps whose keys turn.  The 16-byte chunks of a row that hold temporal pairs (the first tc of
// its vpr chunks) do not go through cp.async: they are loaded into registers with the same stage's copies, turned
// with the frame's table entries and written to the stage with st.shared one iteration ahead of the stage's store,
// so the turn overlaps the other stages' memory traffic instead of sitting between a stage's landing and its store.
// A block's chunks are numbered temporal chunks first (row-major over nrows x tc), then the K chunks without temporal
// pairs, then the V chunks, and thread t takes chunks t, t + 256, ...: every thread holds at most two temporal
// chunks (the host takes this form only when 64 x tc <= 512), so the turning is spread over all threads.  (Turning
// the staged rows in shared memory after they landed measured 279 us, and a layout that left all temporal chunks
// to a third of the threads 311 us, against 249 us for the register-staged kernel above.)
constexpr int kStagedRows = 64;
constexpr int kStages = 3;
constexpr int kMaxChunksPerThread = 9;  // 2 x 64 rows of up to 288 bytes in 16-byte chunks over 256 threads
constexpr int kMaxTurnChunks = 2;       // temporal chunks per thread in the TURN form (64 x tc <= 2 x 256)

template <bool TURN>
__global__ void __launch_bounds__(kThreads) gather_staged_kernel(const GatherParams p) {
  constexpr int S = kStages, R = kStagedRows;
  extern __shared__ __align__(128) unsigned char smem[];
  wait_for_predecessor();
  const Ctrl* c = p.ctrl;
  if (c->abort || !c->has_dyn) return;
  const int k = c->k;
  if (k <= 0) return;
  const int tid = threadIdx.x;
  const int rb = p.row_bytes;
  const int stage_bytes = 2 * R * rb;
  int* s_row = reinterpret_cast<int*>(smem + S * stage_bytes);  // [R, 2R): source rows of the block
  float4* s_trig = reinterpret_cast<float4*>(smem + S * stage_bytes + 8 * R);  // TURN: table and frame flags
  const uint8_t* s_rot = reinterpret_cast<const uint8_t*>(s_trig + p.n_frames * p.n_t);
  const int ppv = p.dtype == DCP_BF16 ? 4 : 2;  // rotary pairs per 16-byte chunk
  const int tc = TURN ? (p.n_t + ppv - 1) / ppv : 0;  // chunks of a row that hold temporal pairs
  if (TURN) table_copy(p, s_trig);  // (the item loop's first barrier orders it before use)

  const int64_t common = c->common_len;
  const int first_dyn = c->first_dyn;
  const int nblk = (k + R - 1) / R;
  const int n_seq = p.dyn_list ? c->n_dyn : p.n_planes;  // planes split into ranges (all, or the receiving list)
  int ranges = (int)gridDim.x * 2 / nblk;  // longer plane ranges than above: the stages fill once per item
  if (ranges > n_seq / 4) ranges = n_seq / 4;
  if (ranges < 1) ranges = 1;
  const int ppr = (n_seq + ranges - 1) / ranges;
  const int items = nblk * ranges;
  const int vpr = rb / 16;                  // 16-byte chunks per row
  const int chunks = R * vpr;               // per tensor and stage
  const int per_thread = (2 * chunks + kThreads - 1) / kThreads;
  const int64_t src0 = p.src_row0 * (int64_t)rb;

  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int jb = it % nblk, r = it / nblk;
    const int p0 = r * ppr, p1 = min(n_seq, p0 + ppr);  // positions in the plane sequence
    const int j0 = jb * R, nrows = min(R, k - j0);
    __syncthreads();  // the previous item's stages and rows are no longer read
    if (tid < nrows) {
      const int s = __ldg(p.idx + j0 + tid);
      s_row[R + tid] = s;
      const bool writes_t = p.dyn_list ? r == 0 : first_dyn >= p0 && first_dyn < p1;  // one item per row block
      if (writes_t) p.hist_t[common + j0 + tid] = p.evict_first_frame + s / p.T;
    }
    __syncthreads();
    const int64_t dst_off = (p.dst_row0 + common + j0) * (int64_t)rb;
    const int nchunks = nrows * vpr;        // per tensor

    // this thread's 16-byte chunks of the block: the same (source, stage offset) pairs for every plane of the item
    int c_src[kMaxChunksPerThread];          // byte offset inside the leaving chunk's rows, -1 when unused
    uint32_t c_dst[kMaxChunksPerThread];     // byte offset inside a stage (V chunks past the K half)
    uint32_t c_v = 0;                        // bit u: chunk u is a V chunk
    uint32_t c_reg = 0;                      // TURN, bit u (u < kMaxTurnChunks): chunk u is a temporal K chunk
    int c_rot[kMaxTurnChunks];               // TURN: (frame << 16) | chunk column of a temporal chunk, -1 if it
                                             // stays as stored (its frame does not move)
#pragma unroll
    for (int u = 0; u < kMaxChunksPerThread; ++u) {
      const int e = tid + kThreads * u;
      c_src[u] = -1;
      c_dst[u] = 0;
      if (u < kMaxTurnChunks) c_rot[u] = -1;
      if (u >= per_thread) continue;
      if constexpr (!TURN) {
        const int t = e >= chunks;  // tensor: K, then V
        const int ci = e - t * chunks;
        if (ci < nchunks) {
          const int row = ci / vpr, col = ci - row * vpr;
          c_src[u] = s_row[R + row] * rb + col * 16;
          c_dst[u] = (uint32_t)(t * R * rb + row * rb + col * 16);
          c_v |= (uint32_t)t << u;
        }
      } else {
        const int n_tmp = nrows * tc, n_kplain = nrows * (vpr - tc);
        int row, col, t = 0;
        if (e < n_tmp) {
          row = e / tc;
          col = e - row * tc;
          if (u < kMaxTurnChunks) {
            c_reg |= 1u << u;
            const int f = s_row[R + row] / p.T;
            if (s_rot[f]) c_rot[u] = (f << 16) | col;
          }
        } else if (e < n_tmp + n_kplain) {
          const int q = e - n_tmp;
          row = q / (vpr - tc);
          col = tc + (q - row * (vpr - tc));
        } else if (e < n_tmp + n_kplain + nchunks) {
          const int q = e - n_tmp - n_kplain;
          t = 1;
          row = q / vpr;
          col = q - row * vpr;
        } else {
          continue;
        }
        c_src[u] = s_row[R + row] * rb + col * 16;
        c_dst[u] = (uint32_t)(t * R * rb + row * rb + col * 16);
        c_v |= (uint32_t)t << u;
      }
    }

    auto receives = [&](int j) { return p.dyn_list || !(p.head_is_static && __ldg(p.head_is_static + j)); };
    auto plane_of = [&](int j) { return p.dyn_list ? __ldg(p.dyn_list + j) : j; };
    auto next_plane = [&](int j) {  // next receiving position
      while (j < p1 && !receives(j)) ++j;
      return j;
    };
    // a stage's copies: cp.async for the plain chunks, register loads for the temporal ones (TURN)
    auto issue = [&](int stage, int pl, Vec<4>(&reg)[kMaxTurnChunks]) {
      const uint32_t st = smem_u32(smem + stage * stage_bytes);
      const char* kp = p.k + pl * p.plane_bytes + src0;
      const char* vp = p.v + pl * p.plane_bytes + src0;
#pragma unroll
      for (int u = 0; u < kMaxChunksPerThread; ++u) {
        if (c_src[u] < 0) continue;
        if (TURN && u < kMaxTurnChunks && ((c_reg >> u) & 1u)) ld_stream(reg[u], kp + c_src[u]);
        else cp_async16(st + c_dst[u], ((c_v >> u) & 1u ? vp : kp) + c_src[u]);
      }
    };
    // TURN: turn a stage's temporal chunks held in registers and write them into the stage
    auto turn_store = [&](int stage, Vec<4>(&reg)[kMaxTurnChunks]) {
      unsigned char* st = smem + stage * stage_bytes;
#pragma unroll
      for (int u = 0; u < kMaxTurnChunks; ++u) {
        if (!((c_reg >> u) & 1u)) continue;
        if (c_rot[u] >= 0)
          dev_rotate_vec(reg[u], p.dtype, (c_rot[u] & 0xFFFF) * ppv, p.n_t, s_trig + (c_rot[u] >> 16) * p.n_t);
        *reinterpret_cast<uint4*>(st + c_dst[u]) = make_uint4(reg[u].w[0], reg[u].w[1], reg[u].w[2], reg[u].w[3]);
      }
    };

    Vec<4> set_a[kMaxTurnChunks], set_b[kMaxTurnChunks];  // registers of the stages in flight (TURN): stage s in
                                                           // set s % 2
    int load_j = next_plane(p0);
    int queue[S];  // the plane each stage holds
    int n_issued = 0;
    for (int q = 0; q < S - 1; ++q) {
      if (load_j < p1) {
        queue[q] = plane_of(load_j);
        if (q == 0) issue(q, queue[q], set_a);
        else issue(q, queue[q], set_b);
        ++n_issued;
        load_j = next_plane(load_j + 1);
      }
      cp_async_commit();  // one group per slot, empty or not, so the group count stays uniform
    }
    if (TURN && n_issued > 0) turn_store(0, set_a);
    // iteration i stores stage i, issues stage i + S - 1 into the registers of stage i (set i % 2, free since its
    // turn) and turns stage i + 1 (set (i + 1) % 2); two calls per loop pass keep every register index static
    auto iteration = [&](int i, Vec<4>(&reg_issue)[kMaxTurnChunks], Vec<4>(&reg_turn)[kMaxTurnChunks]) {
      const int stage = i % S;
      const int pl = queue[stage];
      unsigned char* st = smem + stage * stage_bytes;
      if (tid == 0) bulk_wait_read_all();  // the store issued last iteration has finished reading its stage
      cp_async_wait<S - 2>();              // this thread's copies into stage i have landed
      fence_proxy_async_smem();            // the stage's generic-proxy writes before the bulk copy reads them
      __syncthreads();
      if (tid == 0) {
        bulk_store(p.k + pl * p.plane_bytes + dst_off, smem_u32(st), (uint32_t)(nrows * rb));
        bulk_store(p.v + pl * p.plane_bytes + dst_off, smem_u32(st + R * rb), (uint32_t)(nrows * rb));
        bulk_commit();
        if (jb == 0) p.hist_len[pl] = (int32_t)(common + k);
      }
      // refill the stage the previous store read (thread 0 waited for that store before the barrier above)
      if (load_j < p1) {
        const int rs = (i + S - 1) % S;
        queue[rs] = plane_of(load_j);
        issue(rs, queue[rs], reg_issue);
        ++n_issued;
        load_j = next_plane(load_j + 1);
      }
      cp_async_commit();
      if (TURN && i + 1 < n_issued) turn_store((i + 1) % S, reg_turn);
    };
    for (int i = 0; i < n_issued; i += 2) {
      iteration(i, set_a, set_b);
      if (i + 1 < n_issued) iteration(i + 1, set_b, set_a);
    }
    cp_async_wait<0>();
    if (tid == 0) bulk_wait_read_all();
  }
  if (tid == 0) bulk_wait_all();
}

size_t staged_smem_bytes(const GatherParams& p, bool turn) {
  return (size_t)kStages * 2 * kStagedRows * p.row_bytes + 8 * kStagedRows +
         (turn ? table_smem_bytes(p.n_frames, p.n_t) : 0);
}

// Temporal 16-byte chunks per row, and whether the TURN form's at-most-two-per-thread layout holds them.
bool staged_turn_fits(const GatherParams& p) {
  const int ppv = p.dtype == DCP_BF16 ? 4 : 2;
  const int tc = (p.n_t + ppv - 1) / ppv;
  return tc >= 1 && kStagedRows * tc <= kMaxTurnChunks * kThreads;
}

template <bool TURN>
cudaError_t launch_staged(const GatherParams& p, cudaStream_t s, bool overlap_launch) {
  const size_t smem = staged_smem_bytes(p, TURN);
  static LaunchCache lc;
  int blocks_per_sm = 1;
  const cudaError_t e = launch_setup(lc, gather_staged_kernel<TURN>, kThreads, smem, &blocks_per_sm);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_launch ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_staged_kernel<TURN>, p);
}

template <int NW, bool PAGED, bool LIST>
cudaError_t launch_gather_w(const GatherParams& p, cudaStream_t s, bool overlap_launch) {
  const size_t smem = table_smem_bytes(p.n_frames, p.n_t);
  static LaunchCache lc;
  int blocks_per_sm = 1;
  const cudaError_t e = launch_setup(lc, gather_kernel<NW, PAGED, LIST>, kThreads, smem, &blocks_per_sm);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_launch ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_kernel<NW, PAGED, LIST>, p);
}

template <int NW, bool PAGED>
cudaError_t launch_step_w(const GatherParams& gp, const RephaseParams& rp, cudaStream_t s, bool overlap_launch) {
  const size_t smem = table_smem_bytes(gp.n_frames, gp.n_t);
  static LaunchCache lc;
  int blocks_per_sm = 1;
  const cudaError_t e = launch_setup(lc, step_kernel<NW, PAGED>, kThreads, smem, &blocks_per_sm);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_launch ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, step_kernel<NW, PAGED>, gp, rp);
}

}  // namespace

cudaError_t launch_step_fused(const GatherParams& gp, const RephaseParams& rp, cudaStream_t s, bool overlap_launch,
                              bool paged) {
  if (paged)
    return gp.vb == 32 ? launch_step_w<8, true>(gp, rp, s, overlap_launch)
                       : launch_step_w<4, true>(gp, rp, s, overlap_launch);
  return gp.vb == 32 ? launch_step_w<8, false>(gp, rp, s, overlap_launch)
                     : launch_step_w<4, false>(gp, rp, s, overlap_launch);
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t s, bool overlap_launch, bool paged) {
  // the staged form when the cache has many planes and two CTAs' stages fit in shared memory (rows up to 288 bytes;
  // the turning form also needs at most two temporal chunks per thread).  Measured on the full-depth eviction (1600
  // planes): step 248.1 vs 250.5 us copy-only, 255 vs 262 us when every key turns; on the same eviction cut to 320
  // planes the register-staged kernel is faster (step 59.5 vs 64.0 us: items of a few planes spend much of their
  // time filling and draining three stages).
  if (!paged && p.n_planes >= 1024 && p.row_bytes % 16 == 0 && p.row_bytes <= 288) {
    if (p.no_turn && staged_smem_bytes(p, false) <= 110 * 1024) return launch_staged<false>(p, s, overlap_launch);
    if (!p.no_turn && staged_turn_fits(p) && staged_smem_bytes(p, true) <= 110 * 1024)
      return launch_staged<true>(p, s, overlap_launch);
  }
  // the receiving-plane list (head-specialised steps) is a compile-time choice: reading the plane sequence through
  // it in every step cost the paged full-depth gather 243 -> 264 us
  if (p.dyn_list) {
    if (paged)
      return p.vb == 32 ? launch_gather_w<8, true, true>(p, s, overlap_launch)
                        : launch_gather_w<4, true, true>(p, s, overlap_launch);
    return p.vb == 32 ? launch_gather_w<8, false, true>(p, s, overlap_launch)
                      : launch_gather_w<4, false, true>(p, s, overlap_launch);
  }
  if (paged)
    return p.vb == 32 ? launch_gather_w<8, true, false>(p, s, overlap_launch)
                      : launch_gather_w<4, true, false>(p, s, overlap_launch);
  return p.vb == 32 ? launch_gather_w<8, false, false>(p, s, overlap_launch)
                    : launch_gather_w<4, false, false>(p, s, overlap_launch);
}

}  // namespace dcp
