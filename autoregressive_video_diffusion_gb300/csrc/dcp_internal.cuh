// Internal declarations of libdcp: workspace layout, kernel parameter blocks, device helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dcp.h"

namespace dcp {

constexpr int kThreads = 256;          // every kernel of the library runs 256-thread CTAs
constexpr int kMaxTile = 256;          // tokens per scan tile (one token per thread in the mask phase)

// Control block at the start of the workspace.  The scan kernel's final CTA writes the verdict fields, which the
// re-index and gather kernels that follow it on the stream read.  The completion counter and the accumulators start
// at zero (a zeroed workspace) and the final CTA puts them back to zero at the end of every call.
struct Ctrl {
  uint32_t done;            // CTAs of the scan kernel that finished
  int32_t snap_abort;       // snapshot / restore: nonzero -> the copy kernel does nothing
  int32_t snap_hist_t_len;  // snapshot / restore: longest history of the image
  int32_t abort;            // verdict: nonzero -> the later kernels of the call do nothing
  int32_t k;                // kept tokens
  int32_t has_dyn;          // at least one plane receives the kept rows
  int32_t common_len;       // history length of the receiving planes before the step
  int32_t first_dyn;        // lowest receiving plane (its gather items also append hist_t), -1 if none
  int32_t rp_max;           // longest history of any plane before the step (re-index extent)
  // plane checks, accumulated with atomicMax by the scan CTAs (0 = nothing seen yet)
  int32_t acc_len_max1;     // max over receiving planes of hist_len + 1
  int32_t acc_len_min_inv;  // max over receiving planes of INT32_MAX - hist_len
  int32_t acc_first_inv;    // max over receiving planes of INT32_MAX - plane
  int32_t acc_rp_max;       // max over all planes of hist_len
  int32_t acc_bad;          // some plane's hist_len is outside [0, hist_cap]
  int32_t acc_all_min_inv;  // max over all planes of INT32_MAX - hist_len
  int32_t rp_min;           // shortest history of any plane before the step (rows below it exist in every plane)
  int32_t acc_n_dyn;        // receiving planes listed so far (head-specialised steps)
  int32_t n_dyn;            // receiving planes in the list
  int64_t snap_rows;        // snapshot / restore: saved rows per tensor
  int64_t snap_data_off;    // snapshot / restore: byte offset of the K block in the image
  int32_t pad[42];
};
static_assert(sizeof(Ctrl) == 256, "ctrl block is one 256-byte line");

struct Layout {           // byte offsets inside the workspace
  size_t bits, ell, mask, idx, trig_g, rot_g, trig_h, rot_h, plane_off, dyn, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline Layout make_layout(int64_t n_tok, int64_t n_planes, int64_t F, int64_t n_t, int64_t max_frames) {
  Layout L{};
  size_t off = sizeof(Ctrl);
  L.bits = off;       off = align256(off + 4 * (size_t)((n_tok + 31) / 32));
  L.ell = off;        off = align256(off + 4 * (size_t)n_tok);
  L.mask = off;       off = align256(off + (size_t)n_tok);
  L.idx = off;        off = align256(off + 4 * (size_t)n_tok);
  L.trig_g = off;     off = align256(off + 16 * (size_t)(F * n_t));
  L.rot_g = off;      off = align256(off + (size_t)F);
  L.trig_h = off;     off = align256(off + 16 * (size_t)(max_frames * n_t));
  L.rot_h = off;      off = align256(off + (size_t)max_frames);
  L.plane_off = off;  off = align256(off + 8 * (size_t)(n_planes > 0 ? n_planes + 1 : 0));
  L.dyn = off;        off = align256(off + 4 * (size_t)(n_planes > 0 ? n_planes : 0));
  L.total = off;
  return L;
}

// ------------------------------------------------------------------------------------------ kernel params
struct ScanParams {
  // score inputs (x0hat == nullptr -> the mask comes from mask_in)
  const float* x0hat;
  const float* xref;
  const uint8_t* mask_in;
  int32_t n_tok, d;
  float gamma;
  int32_t keep_rule;       // 2 (with score inputs): the Random ablation at rule 0's count
  uint64_t random_stream;  // its SplitMix64 seed
  int32_t tile, n_tiles, lpt;  // tokens per tile, tiles, lanes per token of the vector path (0 = warp path)
  float* ell_out;
  uint8_t* mask_out;
  int32_t* idx_out;
  // control
  Ctrl* ctrl;
  uint32_t* bits;          // keep mask as ballot words, one bit per token
  int32_t* status;
  int32_t* kept_dev;
  int32_t* kept_host;      // page-locked host memory reached through unified addressing (nullable)
  // plane checks (the check CTAs, after the tile and table CTAs, each check 256 planes)
  int32_t update_cache;   // a gather follows: check the receiving planes and the history capacity
  int32_t want_rephase;   // a re-index follows: find the longest history
  const int32_t* hist_len;
  const uint8_t* head_is_static;
  int32_t* dyn_list;       // head-specialised steps: the receiving planes are listed here (order not significant)
  int32_t n_planes, n_plane_slices;
  int64_t hist_cap;
  // paged caches: every block-table entry the step will use must name a block of the pools (the check CTAs each
  // check 256 entries of tbl_a followed by tbl_b)
  const int32_t* tbl_a;
  const int32_t* tbl_b;
  int32_t n_tbl_a, n_tbl_b, n_tbl_slices;
  int64_t n_blocks;
  // phase tables, built by the CTAs numbered past the tiles (tbl_per entries each, at most kTableEntries)
  int32_t n_trig_blocks, tbl_per;
  float4* trig_g;          // [F][n_t]: turn from t to t~(t; q0) for the leaving chunk's frames
  uint8_t* rot_g;          // [F]: nonzero if that frame turns at all
  int32_t g_frames;        // F, or 0 when no gather follows (read-time re-index: frames [T_s, q0))
  int32_t evict_first_frame;
  int32_t g_identity;      // read-time re-index mode: moved keys keep their phase (the trig_g turns are zero)
  float4* trig_h;          // [max_frames][n_t]: turn from t~(t; q0_prev) to t~(t; q0)
  uint8_t* rot_h;          // [max_frames]
  int32_t h_lo, h_hi;      // frames [h_lo, h_hi) of the history table (empty when no re-index follows)
  int32_t n_t;
  double base, R, S;
  int32_t g_mode;
  int32_t T_s;             // first non-sink frame
  int32_t q0, q0_prev;
  int32_t n_counted;       // CTAs that take part in the completion count (set by launch_scan)
};

// Table entries per table CTA: at most kTableEntries, at least kTableMinEntries, spread over about
// kTableTargetCTAs CTAs.  GB300 runs fp64 at a small fraction of its fp32 rate, so one entry (an exp2, the phase map's
// divisions, a sincos) takes microseconds of one SM's fp64 pipe; short tables spread thinly finish sooner.
constexpr int kTableEntries = 64;
constexpr int kTableMinEntries = 8;
constexpr int kTableTargetCTAs = 128;
// The streaming kernels move 64 bytes per thread, tensor and plane: four 16-byte vectors, or two 32-byte vectors
// when rows and base addresses are 32-byte aligned.
constexpr int kBytesPerThread = 64;

// Addressing of a paged cache (unused for the contiguous layout): plane (l, h) starts at l * s_layer + h * s_head;
// position i of a region whose block table is tbl sits at tbl[i / bs] * s_block + (i % bs) * s_row from there.
struct Paging {
  int32_t H, bs;
  int64_t s_layer, s_head, s_block, s_row;
  const int32_t* src_blocks;   // gather: the leaving ring slot's blocks
  const int32_t* hist_blocks;  // history blocks
};

struct GatherParams {
  char* k;
  char* v;
  int64_t plane_bytes;     // cap * row_bytes
  int32_t row_bytes;       // D * element size (multiple of 16, at most 16 KiB)
  int32_t vb;              // bytes per vector: 32 when rows and bases are 32-byte aligned, else 16
  int64_t src_row0;        // first row of the leaving chunk's slot
  int64_t dst_row0;        // first history row (sink_rows)
  int32_t n_planes;
  const Ctrl* ctrl;
  const int32_t* idx;
  const uint8_t* head_is_static;
  int32_t* hist_len;       // receiving planes: set to common_len + k
  int32_t* hist_t;         // positions [common_len, common_len + k) get the kept tokens' frames
  int32_t evict_first_frame;
  const float4* trig_g;
  const uint8_t* rot_g;
  int32_t T, n_t, dtype;
  Paging pg;
  int32_t n_frames;        // F (rows of trig_g)
  int32_t no_turn;         // no kept key changes phase in this step (the phase map is the identity on the chunk):
                           // the scan builds no trig_g / rot_g for it and the kernels must not read them
  int32_t* status;
  const int32_t* dyn_list; // head-specialised steps: the scan's list of receiving planes (ctrl->n_dyn of them);
                           // the planes split into ranges along it, so static planes take no share of the work
};

struct RephaseParams {
  char* k;
  int64_t plane_bytes;
  int32_t row_bytes;
  int32_t vb;              // bytes per vector (16 or 32)
  int32_t nvt;             // vectors of a row that hold temporal pairs
  int64_t hist_row0;       // sink_rows
  int32_t n_planes;
  const Ctrl* ctrl;
  const int32_t* hist_len; // read before the gather of the same step grows it
  const int32_t* hist_t;
  const float4* trig_h;
  const uint8_t* rot_h;
  int32_t n_t, dtype;
  int32_t h_lo, h_hi;      // frames the table covers
  int32_t* status;
  Paging pg;
};

// Snapshot / restore of the cache's non-derivable state to / from a host image (layout documented in dcp.h).
struct SnapParams {
  int32_t dir;             // 0: cache -> image (snapshot), 1: image -> cache (restore)
  char* k;
  char* v;
  int64_t plane_bytes;
  int32_t row_bytes;       // multiple of 16
  int32_t n_planes;
  int64_t sink_rows, hist_cap, C;
  uint32_t live_slots;     // ring slots saved (bit s = slot s)
  int32_t n_live;
  int32_t* hist_len;       // cache, device
  int32_t* hist_t;         // cache, device
  char* img;               // device address of the host image (16-byte aligned)
  int64_t img_bytes;
  int32_t L, H, D, dtype;  // header fields of a snapshot
  int64_t cap;
  int32_t window_chunks, q0;
  Ctrl* ctrl;
  int64_t* plane_off;      // workspace [n_planes + 1]: first image row of each plane inside a tensor block
  int32_t* status;
};

// Read-time re-index: history keys turned from their own frame t to t~(t; q0) into a contiguous output.
struct ReadParams {
  char* k;
  int64_t plane_bytes;
  int32_t row_bytes;
  int32_t vb;              // bytes per vector (16 or 32)
  int32_t nvt;             // vectors of a row that hold temporal pairs
  int32_t vpr;             // vectors per row
  int64_t hist_row0;       // sink_rows
  int32_t plane0, n_planes;
  int64_t hist_cap;        // output rows per plane
  char* out;               // [n_planes][hist_cap][D]
  const Ctrl* ctrl;
  const int32_t* hist_len;
  const int32_t* hist_t;
  const float4* trig;      // [frames][n_t]: turn from t to t~(t; q0), frames from f_lo
  const uint8_t* rot;
  int32_t f_lo, f_hi;
  int32_t n_t, dtype;
  int32_t* status;
  Paging pg;
};

cudaError_t launch_scan(const ScanParams& p, cudaStream_t s);
cudaError_t launch_phase_table(float4* out, int32_t frame_lo, int32_t n_entries, int32_t n_t, double base, double R,
                               double S, int32_t g_mode, int32_t T_s, int32_t q0, cudaStream_t s);
cudaError_t launch_read(const ReadParams& p, cudaStream_t s, bool paged);
cudaError_t launch_snapshot(const SnapParams& p, cudaStream_t s);
cudaError_t launch_gather(const GatherParams& p, cudaStream_t s, bool overlap_launch, bool paged);
cudaError_t launch_rephase(const RephaseParams& p, cudaStream_t s, bool overlap_launch, bool paged);
// The re-index and the gather of a step in one launch (every plane receives: no static heads; gp.vb == rp.vb).
cudaError_t launch_step_fused(const GatherParams& gp, const RephaseParams& rp, cudaStream_t s, bool overlap_launch,
                              bool paged);
int sm_count();
// dcp_prune_step that first zeroes ws[0, ws_clear_bytes) on the stream, once every host check has passed (nothing is
// launched for a refused call).
dcp_status prune_step_cleared(const dcp_cache* cache, const dcp_config* cfg, const float* x0hat, const float* xref,
                              int32_t dd, int32_t evict_slot, int32_t evict_first_frame, int32_t q0_prev, int32_t q0,
                              const uint8_t* head_is_static, int32_t* kept_dev, int32_t* kept_host_pinned, void* ws,
                              size_t ws_bytes, size_t ws_clear_bytes, void* stream);

// Per-device launch set-up of one kernel, made on first use on each device: the dynamic shared-memory opt-in (a
// per-device function attribute) and the number of CTAs that fit on an SM with that much shared memory.  Host
// threads that launch on different caches share it, so it is updated under a mutex (the opt-in must only grow).
constexpr int kMaxDevices = 64;
struct LaunchCache {
  std::mutex m;
  size_t opted[kMaxDevices];    // dynamic shared memory opted in so far (bytes)
  size_t counted[kMaxDevices];  // shared-memory size + 1 that blocks[] was computed for (0: not yet)
  int blocks[kMaxDevices];
};

template <typename Kernel>
cudaError_t launch_setup(LaunchCache& lc, Kernel kernel, int threads, size_t smem, int* blocks_per_sm) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(lc.m);
  if (smem > 48 * 1024 && smem > lc.opted[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    lc.opted[dev] = smem;
  }
  if (lc.counted[dev] != smem + 1) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
    lc.blocks[dev] = n;
    lc.counted[dev] = smem + 1;
  }
  *blocks_per_sm = lc.blocks[dev];
  return cudaSuccess;
}

// ------------------------------------------------------------------------------------------ device helpers
#ifdef __CUDACC__

// g and t~ in double with explicit round-to-nearest operations (never contracted into fma), so the decision
// "does this frame's phase change" is taken on exactly the values the definition gives.
__device__ __forceinline__ double dev_g(double delta, double delta_max, double R, double S, int mode) {
  double span_end = mode == 0 ? S : __dadd_rn(R, S);
  if (delta <= R || delta_max <= span_end) return delta;
  return __dadd_rn(__ddiv_rn(__dmul_rn(__dsub_rn(delta, R), __dsub_rn(span_end, R)), __dsub_rn(delta_max, R)), R);
}

__device__ __forceinline__ double dev_phase(double t, double q0, double T_s, double R, double S, int mode) {
  return __dsub_rn(q0, dev_g(__dsub_rn(q0, t), __dsub_rn(q0, T_s), R, S, mode));
}

// A double rounded to 16 significant bits, as a float (round half away from zero on the dropped 8 bits).
__device__ __forceinline__ float round_to_16_bits(double x) {
  const uint32_t u = __float_as_uint(__double2float_rn(x));
  if ((u & 0x7F800000u) == 0x7F800000u) return __uint_as_float(u);
  return __uint_as_float((u + 0x80u) & 0xFFFFFF00u);
}

// cos/sin of an angle as unevaluated pairs {c_hi, c_lo, s_hi, s_lo}: the high part has 16 significant bits (so its
// product with a bf16 value, 8 bits, is exact in fp32), the low part is the fp32 rounding of the rest: ~40 bits in all.
__device__ __forceinline__ float4 dev_trig_entry(double phi) {
  double s, c;
  sincos(phi, &s, &c);
  const float chi = round_to_16_bits(c), shi = round_to_16_bits(s);
  return make_float4(chi, __double2float_rn(__dsub_rn(c, (double)chi)), shi,
                     __double2float_rn(__dsub_rn(s, (double)shi)));
}

// Table entry of the turn from frame t to t~(t; q0) for rotary pair pp, with theta_pp = base^(-pp / n_t) evaluated as
// exp2(log2(base) * (-pp / n_t)) (the same value to a few ulps of fp64, far below the 2^-40 the entry carries, and
// much cheaper than pow on a part with a low fp64 rate); *moves: t~ differs from t.  Every table of the library is
// built by this function, so tables built by different kernels hold the same bits.  (Each gather CTA building the
// leaving chunk's table itself, before its wait for the scan, measured slower: 304 CTAs paying GB300's low fp64 rate
// for the same 88 entries made the rotated full-depth gather 248 instead of 238 us.)
__device__ __forceinline__ float4 dev_turn_entry(double t, int pp, int n_t, double log2_base, double q0, double T_s,
                                                 double R, double S, int mode, bool identity, bool* moves) {
  const double delta = identity ? 0.0 : __dsub_rn(dev_phase(t, q0, T_s, R, S, mode), t);
  const double theta = exp2(__dmul_rn(-(double)pp / (double)n_t, log2_base));
  *moves = delta != 0.0;
  return dev_trig_entry(__dmul_rn(theta, delta));
}

// Table entry of a history key's re-index when the query frame moves from q0_prev to q0: the turn of pair pp from
// t~(t; q0_prev) to t~(t; q0); *moves: the two phases differ.  (A step kernel whose CTAs each built the entries of
// their own frames with it, so as to re-index before the scan completes, measured slower: each CTA waited on one
// fp64 chain of GB300's low fp64 rate first; mid eviction 53.1 vs 45.4 us.)
__device__ __forceinline__ float4 dev_reindex_entry(double t, int pp, int n_t, double log2_base, double q0_prev,
                                                    double q0, double T_s, double R, double S, int mode, bool* moves) {
  const double before = dev_phase(t, q0_prev, T_s, R, S, mode);
  const double after = dev_phase(t, q0, T_s, R, S, mode);
  const double delta = __dsub_rn(after, before);
  const double theta = exp2(__dmul_rn(-(double)pp / (double)n_t, log2_base));
  *moves = after != before;
  return dev_trig_entry(__dmul_rn(theta, delta));
}

// Rotate one pair (a, b) of fp32 values by the angle whose cos/sin pairs are in t:
//   out_a = a*c - b*s, out_b = a*s + b*c.
// The rounding error of the b-products is recovered exactly with an fma and the low parts of cos/sin are added, so
// the result carries ~2^-23 relative error plus ~2^-38 (|a| + |b|) absolute error.
__device__ __forceinline__ void dev_rotate(float a, float b, const float4 t, float& oa, float& ob) {
  float q0 = __fmul_rn(b, t.z);
  float e0 = __fmaf_rn(b, t.z, -q0);
  float r0 = __fmaf_rn(a, t.x, -q0);
  float k0 = __fmaf_rn(a, t.y, -__fmul_rn(b, t.w));
  oa = __fadd_rn(r0, __fsub_rn(k0, e0));
  float q1 = __fmul_rn(b, t.x);
  float e1 = __fmaf_rn(b, t.x, -q1);
  float r1 = __fmaf_rn(a, t.z, q1);
  float k1 = __fmaf_rn(a, t.w, __fmul_rn(b, t.y));
  ob = __fadd_rn(r1, __fadd_rn(k1, e1));
}

// The same turn for a pair read from bf16 storage (8 significant bits): a * c_hi and b * s_hi are exact in fp32
// (8 + 16 bits), so one fma rounds their difference once and the low-part products complete it.  Same error bound
// as dev_rotate: rounding the result to bf16 gives the correctly rounded value or its neighbour, never further.
__device__ __forceinline__ void dev_rotate_bf16in(float a, float b, const float4 t, float& oa, float& ob) {
  oa = __fadd_rn(__fmaf_rn(a, t.x, -__fmul_rn(b, t.z)), __fmaf_rn(a, t.y, -__fmul_rn(b, t.w)));
  ob = __fadd_rn(__fmaf_rn(a, t.z, __fmul_rn(b, t.x)), __fmaf_rn(a, t.w, __fmul_rn(b, t.y)));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

// A vector of NW 32-bit words (NW = 4: 16 bytes, NW = 8: 32 bytes) moved by one load or store instruction.
template <int NW>
struct Vec {
  uint32_t w[NW];
};

// Rotate the pairs held in one vector.  p0 = index of its first pair; pairs >= n_t are left as stored.  trig points
// at the table row of the key's frame.  bf16: word i holds pair p0 + i; fp32: words 2i, 2i+1 hold pair p0 + i.
template <int NW>
__device__ __forceinline__ void dev_rotate_vec(Vec<NW>& x, int dtype, int p0, int n_t, const float4* trig) {
  if (dtype == DCP_BF16) {
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int p = p0 + i;
      if (p < n_t) {
        float oa, ob;
        dev_rotate_bf16in(bf16lo(x.w[i]), bf16hi(x.w[i]), trig[p], oa, ob);
        x.w[i] = pack_bf16x2(oa, ob);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NW / 2; ++i) {
      const int p = p0 + i;
      if (p < n_t) {
        float oa, ob;
        dev_rotate(__uint_as_float(x.w[2 * i]), __uint_as_float(x.w[2 * i + 1]), trig[p], oa, ob);
        x.w[2 * i] = __float_as_uint(oa);
        x.w[2 * i + 1] = __float_as_uint(ob);
      }
    }
  }
}

// Same turn with the vector's table entries already in registers: tr[i] belongs to pair p0 + i.
template <int NW>
__device__ __forceinline__ void dev_rotate_vec_regs(Vec<NW>& x, int dtype, int p0, int n_t, const float4 (&tr)[NW]) {
  if (dtype == DCP_BF16) {
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      if (p0 + i < n_t) {
        float oa, ob;
        dev_rotate_bf16in(bf16lo(x.w[i]), bf16hi(x.w[i]), tr[i], oa, ob);
        x.w[i] = pack_bf16x2(oa, ob);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NW / 2; ++i) {
      if (p0 + i < n_t) {
        float oa, ob;
        dev_rotate(__uint_as_float(x.w[2 * i]), __uint_as_float(x.w[2 * i + 1]), tr[i], oa, ob);
        x.w[2 * i] = __float_as_uint(oa);
        x.w[2 * i + 1] = __float_as_uint(ob);
      }
    }
  }
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may start while its
// predecessor drains; it must wait here before it reads anything the predecessor wrote.  Without that launch
// attribute the wait returns at once.
__device__ __forceinline__ void wait_for_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Streaming copies: data read once (no L1 allocation) and written once.  The 32-byte forms (sm_100 and later) also
// mark the lines evict-first in L2.
__device__ __forceinline__ void ld_stream(Vec<4>& v, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
               : "l"(p));
}

__device__ __forceinline__ void ld_stream(Vec<8>& v, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                 "=r"(v.w[6]), "=r"(v.w[7])
               : "l"(p));
}

__device__ __forceinline__ void st_stream(void* p, const Vec<4>& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]),
               "r"(v.w[3])
               : "memory");
}

__device__ __forceinline__ void st_stream(void* p, const Vec<8>& v) {
  asm volatile("st.global.L1::no_allocate.L2::evict_first.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
               "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
               : "memory");
}

// Shared-memory staging (Ampere-style per-thread async copies in, Hopper/Blackwell bulk copies out).
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Shared -> global bulk copy (TMA engine), tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy writes to shared memory before later async-proxy (bulk copy) reads of it.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// In-place (read-modify-write) accesses of the re-index kernel: plain cached loads and stores, written out as single
// vector instructions (a struct copy of Vec would be split into 32-bit accesses: one L2 request per word).
__device__ __forceinline__ void ld_plain(Vec<4>& v, const void* p) {
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
               : "l"(p));
}

__device__ __forceinline__ void ld_plain(Vec<8>& v, const void* p) {
  asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                 "=r"(v.w[6]), "=r"(v.w[7])
               : "l"(p));
}

__device__ __forceinline__ void st_plain(void* p, const Vec<4>& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
               : "memory");
}

__device__ __forceinline__ void st_plain(void* p, const Vec<8>& v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]),
               "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
               : "memory");
}

#endif  // __CUDACC__

}  // namespace dcp
