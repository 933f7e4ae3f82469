// Plain CPU oracle of the DeCoPrune history-KV prune step.  TEST INFRASTRUCTURE ONLY.
//
// Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may load this library.  It shares
// no code, header, table or constant generator with the CUDA path: every function below is written from the method's
// description on the page "DeCoPrune이 디노이징 불일치로 비디오 KV 캐시를 85% 줄인다" (onedev.kr/papers/726),
// cited per function by that page's section:
//   [how]    어떻게 동작하나 "how it works"    - the discrepancy, the threshold mask shared by all layers, the protected
//                                               sink, the dense window of w chunks, the physical K[m], V[m] gather.
//   [differs] 무엇과 다른가 "what differs"    - prefix pruning, RoPE re-indexing t~(t) = q0 - g(q0 - t), DeCoPrune-HS.
//   [use]    어떻게 쓰나 "how to use"          - the cumulative history-KV position reduction (PR) versus FullKV.
//   [limits] 전제와 한계 "premises and limits" - the 4-step schedule (999, 957, 899, 702), probe index 2, gamma 0.10.
//
// Style: one thread, plain loops, fp64 arithmetic, one rounding to the storage type at the end of each value.
// Readings of points the page leaves open (the CUDA path takes the same ones):
//   * keep rule: keep when l > gamma (strict), drop otherwise; the reverse criterion is the complement; the Random
//     ablation keeps the same number of tokens, drawn uniformly without replacement from a SplitMix64 stream.
//   * pair p of the temporal RoPE sub-vector occupies dims (2p, 2p+1); theta_p = base^(-p / n_t).
//   * g(D) = D when D <= R (recent offsets) or when no compression is needed; otherwise a linear map that sends R to
//     R and the oldest non-sink offset Dmax to the span end (mode 0: S is the total virtual span; mode 1: old offsets
//     occupy (R, R + S]).
//   * the sink keeps its phase; only history keys are re-phased; values and non-temporal dims are copied bitwise.
//   * read-time re-index (reindex_mode 1): history keys stay at their own frame's phase and are turned to
//     t~(t; q0) when read; a step then moves keys bitwise and re-indexes nothing.
// Parity: every function here is pinned by tests/test_oracle_pins.py (closed forms, invariants, brute force).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" {

struct oracle_cache {
  void* k;               // host, [L][H][cap][D], dtype 0 = bf16 bits (uint16), 1 = fp32
  void* v;
  int32_t L, H, D, dtype;
  int64_t cap;           // rows per (layer, head) plane: sink | history (hist_cap) | window ring (w + 1 slots)
  int64_t hist_cap;
  int32_t* hist_len;     // [L*H]
  int32_t* hist_t;       // [hist_cap] latent frame index of each history position
};

struct oracle_config {
  float gamma;
  int32_t keep_rule;     // 0 = keep large discrepancy (DeCoPrune), 1 = the reverse criterion, 2 = Random at the
                         // same count as rule 0
  int32_t sink_chunks, window_chunks, tokens_per_frame, frames_per_chunk;
  int32_t n_temporal_pairs;
  double rope_base;
  double g_recent_R, g_span_S;
  int32_t g_mode;        // 0: S is the total virtual span; 1: old offsets occupy (R, R + S]
  uint32_t random_seed;  // keep_rule 2: the prune step draws from the stream (random_seed << 32) | evict_first_frame
  int32_t reindex_mode;  // 0: keys re-phased when stored and re-indexed every step; 1: keys kept at their own frame
                         // and turned to t~(t; q0) when read (oracle_read_history_keys)
};

enum { ORACLE_OK = 0, ORACLE_EINVAL = 1, ORACLE_ECAPACITY = 2 };

// ------------------------------------------------------------------------------------------- constants [limits]
// The page's experiments use a 4-step noise schedule and take the zero-based index 2 as the probe timestep.
static const int32_t kSchedule[4] = {999, 957, 899, 702};
int32_t oracle_schedule(int32_t i) { return (i >= 0 && i < 4) ? kSchedule[i] : -1; }
int32_t oracle_probe_index(void) { return 2; }
float oracle_default_gamma(void) { return 0.10f; }

// ------------------------------------------------------------------------------------------- score [how]
// Per-token mean squared discrepancy between the probe-step clean prediction x0hat(tau*) and the final output:
// l[n] = (1/d) * sum_j (x0hat[n][j] - xref[n][j])^2, accumulated in double, rounded once to fp32.
// In the prefix pass [differs] xref is the clean observed chunk instead of x_final.
void oracle_score(const float* x0hat, const float* xref, int64_t n, int32_t d, float* ell) {
  for (int64_t i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int32_t j = 0; j < d; ++j) {
      double diff = (double)x0hat[i * d + j] - (double)xref[i * d + j];
      acc += diff * diff;
    }
    ell[i] = (float)(acc / (double)d);
  }
}

// ------------------------------------------------------------------------------------------- mask [how]
// One binary mask for the chunk, shared by every layer and head: keep tokens whose discrepancy is large.
void oracle_keep(const float* ell, int64_t n, float gamma, int32_t keep_rule, uint8_t* mask) {
  for (int64_t i = 0; i < n; ++i) {
    bool large = ell[i] > gamma;
    mask[i] = (uint8_t)(keep_rule == 0 ? large : !large);
  }
}

// ------------------------------------------------------------------------------------------- Random ablation [limits]
// The page's ablation compares DeCoPrune with a Random policy at the same compression ratio.  Reading: Random keeps
// as many tokens of the chunk as the discrepancy rule would (so the PR is the same chunk by chunk), drawn uniformly
// without replacement.  The draw: token n gets the n-th output of a SplitMix64 sequence (Steele, Lea & Flood, "Fast
// splittable pseudorandom number generators", OOPSLA 2014) started at the stream value, and the tokens with the
// smallest outputs are kept.  The outputs of one sequence are distinct (the state steps by an odd constant and the
// output function is a bijection of 64-bit words), so the kept set is unique.
uint64_t oracle_splitmix64(uint64_t stream, int64_t i) {
  uint64_t z = stream + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ull;  // state after i + 1 steps
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

void oracle_keep_random(const float* ell, int64_t n, float gamma, uint64_t stream, uint8_t* mask) {
  int64_t k = 0;
  for (int64_t i = 0; i < n; ++i) k += ell[i] > gamma ? 1 : 0;
  std::vector<std::pair<uint64_t, int64_t>> order((size_t)n);
  for (int64_t i = 0; i < n; ++i) order[(size_t)i] = {oracle_splitmix64(stream, i), i};
  std::sort(order.begin(), order.end());
  for (int64_t i = 0; i < n; ++i) mask[i] = 0;
  for (int64_t j = 0; j < k; ++j) mask[order[(size_t)j].second] = 1;
}

// ------------------------------------------------------------------------------------------- indices m [how]
// The kept positions in increasing order (the m of K[m], V[m]); returns how many there are.
int64_t oracle_indices(const uint8_t* mask, int64_t n, int32_t* idx) {
  int64_t k = 0;
  for (int64_t i = 0; i < n; ++i)
    if (mask[i]) idx[k++] = (int32_t)i;
  return k;
}

// ------------------------------------------------------------------------------------------- phase map [differs]
// g leaves recent offsets unchanged and compresses old ones linearly into a fixed virtual span.
double oracle_g(double delta, double delta_max, double R, double S, int32_t mode) {
  double span_end = (mode == 0) ? S : R + S;
  if (delta <= R || delta_max <= span_end) return delta;
  return ((delta - R) * (span_end - R)) / (delta_max - R) + R;
}

// t~(t) = q0 - g(q0 - t); T_s is the first non-sink frame, so the oldest re-indexed offset is q0 - T_s.
double oracle_phase(double t, double q0, double T_s, double R, double S, int32_t mode) {
  return q0 - oracle_g(q0 - t, q0 - T_s, R, S, mode);
}

double oracle_theta(int32_t p, int32_t n_t, double base) { return std::pow(base, -(double)p / (double)n_t); }

// ------------------------------------------------------------------------------------------- rounding
double oracle_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round a double straight to the nearest bfloat16 (ties to even), without passing through fp32.
uint16_t oracle_bf16_round(double x) {
  if (std::isnan(x)) return 0x7FC0;
  uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  double a = std::fabs(x);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e = 0;
  std::frexp(a, &e);                       // a = f * 2^e with f in [0.5, 1): 8 significant bits -> spacing 2^(e-8)
  int q_exp = e - 8 < -133 ? -133 : e - 8; // below 2^-126 the spacing stays at the subnormal step 2^-133
  double q = std::nearbyint(std::ldexp(a, -q_exp));  // default rounding mode: to nearest, ties to even
  double r = std::ldexp(q, q_exp);
  if (r >= 0x1.0p128) return (uint16_t)(sign | 0x7F80);
  float f = (float)r;                      // exact
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(sign | (u >> 16));
}

static double load_elem(const void* base, int32_t dtype, int64_t i) {
  return dtype == 0 ? oracle_bf16_value(((const uint16_t*)base)[i]) : (double)((const float*)base)[i];
}

static void store_elem(void* base, int32_t dtype, int64_t i, double x) {
  if (dtype == 0) ((uint16_t*)base)[i] = oracle_bf16_round(x);
  else ((float*)base)[i] = (float)x;
}

// ------------------------------------------------------------------------------------------- key re-phase [differs]
// Move a stored key's temporal phase by dphase frames: pair p of the temporal sub-vector turns by theta_p * dphase.
// Only the first n_t pairs change; every other dim is left as stored.
void oracle_rotate_key_row(void* row, int32_t dtype, int32_t D, int32_t n_t, double base, double dphase) {
  (void)D;
  for (int32_t p = 0; p < n_t; ++p) {
    double phi = oracle_theta(p, n_t, base) * dphase;
    double c = std::cos(phi), s = std::sin(phi);
    double a = load_elem(row, dtype, 2 * p), b = load_elem(row, dtype, 2 * p + 1);
    double na = a * c - b * s;
    double nb = a * s + b * c;
    store_elem(row, dtype, 2 * p, na);
    store_elem(row, dtype, 2 * p + 1, nb);
  }
}

static int64_t elem_size(int32_t dtype) { return dtype == 0 ? 2 : 4; }

static char* row_ptr(void* base, const oracle_cache* c, int64_t plane, int64_t row) {
  return (char*)base + ((plane * c->cap + row) * (int64_t)c->D) * elem_size(c->dtype);
}

// One gathered key row: copy, then rotate from its true frame t to t~(t; q0).  Used for sampled checks at full size.
void oracle_gather_key_row(const void* src, void* dst, const oracle_cache* c, const oracle_config* cfg, int32_t t,
                           int32_t q0) {
  std::memcpy(dst, src, (size_t)c->D * elem_size(c->dtype));
  double T_s = (double)cfg->sink_chunks * cfg->frames_per_chunk;
  double tt = oracle_phase(t, q0, T_s, cfg->g_recent_R, cfg->g_span_S, cfg->g_mode);
  oracle_rotate_key_row(dst, c->dtype, c->D, cfg->n_temporal_pairs, cfg->rope_base, tt - (double)t);
}

// ------------------------------------------------------------------------------------------- compaction [how]
// When a non-sink chunk leaves the dense window, each layer keeps only the selected entries K[m], V[m], appended in
// order to the history region; keys are re-phased to t~(t; q0) as they move [differs].  Static heads of the
// head-specialised variant follow the Streaming policy: they keep nothing of the leaving chunk [differs].
int32_t oracle_compact_layers(oracle_cache* c, const oracle_config* cfg, int32_t evict_slot, int32_t evict_first_frame,
                              const uint8_t* mask, const uint8_t* head_is_static, int32_t q0, int32_t* idx_out,
                              int64_t* k_out) {
  const int64_t T = cfg->tokens_per_frame, C = T * cfg->frames_per_chunk;
  const int64_t n_planes = (int64_t)c->L * c->H;
  const int64_t sink_rows = (int64_t)cfg->sink_chunks * C;
  const int64_t win_row0 = sink_rows + c->hist_cap;
  std::vector<int32_t> idx((size_t)C);
  int64_t k = oracle_indices(mask, C, idx.data());
  if (idx_out) for (int64_t j = 0; j < k; ++j) idx_out[j] = idx[(size_t)j];
  if (k_out) *k_out = k;

  int64_t common = -1;
  for (int64_t p = 0; p < n_planes; ++p) {
    if (head_is_static && head_is_static[p]) continue;
    if (common < 0) common = c->hist_len[p];
    else if (c->hist_len[p] != common) return ORACLE_EINVAL;  // the shared mask keeps dynamic heads in step
  }
  if (common < 0) return ORACLE_OK;                            // every head is static: nothing is kept
  if (common + k > c->hist_cap) return ORACLE_ECAPACITY;

  const int64_t row_bytes = (int64_t)c->D * elem_size(c->dtype);
  for (int64_t p = 0; p < n_planes; ++p) {
    if (head_is_static && head_is_static[p]) continue;
    for (int64_t j = 0; j < k; ++j) {
      int64_t src = win_row0 + (int64_t)evict_slot * C + idx[(size_t)j];
      int64_t dst = sink_rows + common + j;
      int32_t t = evict_first_frame + (int32_t)(idx[(size_t)j] / T);
      std::memcpy(row_ptr(c->v, c, p, dst), row_ptr(c->v, c, p, src), (size_t)row_bytes);
      if (cfg->reindex_mode == 1)
        std::memcpy(row_ptr(c->k, c, p, dst), row_ptr(c->k, c, p, src), (size_t)row_bytes);
      else
        oracle_gather_key_row(row_ptr(c->k, c, p, src), row_ptr(c->k, c, p, dst), c, cfg, t, q0);
    }
    c->hist_len[p] = (int32_t)(common + k);
  }
  for (int64_t j = 0; j < k; ++j) c->hist_t[common + j] = evict_first_frame + (int32_t)(idx[(size_t)j] / T);
  return ORACLE_OK;
}

// ------------------------------------------------------------------------------------------- history re-phase [differs]
// When the query frame moves from q0_prev to q0, every history key whose t~ changes turns by the phase difference.
int32_t oracle_rope_reindex(oracle_cache* c, const oracle_config* cfg, int32_t q0_prev, int32_t q0) {
  const int64_t C = (int64_t)cfg->tokens_per_frame * cfg->frames_per_chunk;
  const int64_t n_planes = (int64_t)c->L * c->H;
  const int64_t sink_rows = (int64_t)cfg->sink_chunks * C;
  const double T_s = (double)cfg->sink_chunks * cfg->frames_per_chunk;
  for (int64_t p = 0; p < n_planes; ++p) {
    for (int64_t j = 0; j < c->hist_len[p]; ++j) {
      double t = (double)c->hist_t[j];
      double before = oracle_phase(t, q0_prev, T_s, cfg->g_recent_R, cfg->g_span_S, cfg->g_mode);
      double after = oracle_phase(t, q0, T_s, cfg->g_recent_R, cfg->g_span_S, cfg->g_mode);
      if (after != before)
        oracle_rotate_key_row(row_ptr(c->k, c, p, sink_rows + j), c->dtype, c->D, cfg->n_temporal_pairs,
                              cfg->rope_base, after - before);
    }
  }
  return ORACLE_OK;
}

// ------------------------------------------------------------------------------------------- read-time re-index
// Keys kept at their own frame t (reindex_mode 1) reach attention with the phase t~(t; q0): each history row of
// each plane is read, its temporal pairs turned once from t to t~(t; q0), and written to out [planes][hist_cap][D]
// (rows past a plane's history are left as they are).  Reading from the raw key turns it once, so nothing drifts.
void oracle_read_history_keys(const oracle_cache* c, const oracle_config* cfg, int32_t q0, void* out) {
  const int64_t C = (int64_t)cfg->tokens_per_frame * cfg->frames_per_chunk;
  const int64_t n_planes = (int64_t)c->L * c->H;
  const int64_t sink_rows = (int64_t)cfg->sink_chunks * C;
  const int64_t row_bytes = (int64_t)c->D * elem_size(c->dtype);
  for (int64_t p = 0; p < n_planes; ++p)
    for (int64_t j = 0; j < c->hist_len[p]; ++j) {
      char* dst = (char*)out + (p * c->hist_cap + j) * row_bytes;
      oracle_gather_key_row(row_ptr(c->k, c, p, sink_rows + j), dst, c, cfg, c->hist_t[j], q0);
    }
}

// ------------------------------------------------------------------------------------------- one prune step
// Score the leaving chunk, threshold it, re-phase the history already present for the new q0, then compact.
int32_t oracle_prune_step(oracle_cache* c, const oracle_config* cfg, const float* x0hat, const float* xref, int32_t d,
                          int32_t evict_slot, int32_t evict_first_frame, int32_t q0_prev, int32_t q0,
                          const uint8_t* head_is_static, float* ell_out, uint8_t* mask_out, int32_t* idx_out,
                          int64_t* k_out) {
  const int64_t C = (int64_t)cfg->tokens_per_frame * cfg->frames_per_chunk;
  std::vector<float> ell((size_t)C);
  std::vector<uint8_t> mask((size_t)C);
  oracle_score(x0hat, xref, C, d, ell.data());
  if (cfg->keep_rule == 2)
    oracle_keep_random(ell.data(), C, cfg->gamma, ((uint64_t)cfg->random_seed << 32) | (uint32_t)evict_first_frame,
                       mask.data());
  else
    oracle_keep(ell.data(), C, cfg->gamma, cfg->keep_rule, mask.data());
  if (ell_out) std::memcpy(ell_out, ell.data(), sizeof(float) * (size_t)C);
  if (mask_out) std::memcpy(mask_out, mask.data(), (size_t)C);
  // the step is checked before anything moves, so a refused step leaves the cache as it was
  int64_t k = 0;
  for (int64_t i = 0; i < C; ++i) k += mask[(size_t)i];
  const int64_t n_planes = (int64_t)c->L * c->H;
  int64_t common = -1;
  for (int64_t p = 0; p < n_planes; ++p) {
    if (head_is_static && head_is_static[p]) continue;
    if (common < 0) common = c->hist_len[p];
    else if (c->hist_len[p] != common) return ORACLE_EINVAL;
  }
  if (common >= 0 && common + k > c->hist_cap) return ORACLE_ECAPACITY;
  if (cfg->reindex_mode != 1) {
    int32_t rc = oracle_rope_reindex(c, cfg, q0_prev, q0);
    if (rc != ORACLE_OK) return rc;
  }
  return oracle_compact_layers(c, cfg, evict_slot, evict_first_frame, mask.data(), head_is_static, q0, idx_out, k_out);
}

// ------------------------------------------------------------------------------------------- PR [use]
// Visible history positions for one generated chunk, summed over every (layer, head): the sink, the compacted
// history and the dense window chunks that precede it.  FullKV would show all prior tokens in every head.
void oracle_pr_chunk(const int32_t* hist_len, int64_t n_planes, int64_t sink_tokens_visible,
                     int64_t window_tokens_visible, int64_t prior_tokens, int64_t* visible, int64_t* full) {
  int64_t v = 0;
  for (int64_t p = 0; p < n_planes; ++p) v += sink_tokens_visible + hist_len[p] + window_tokens_visible;
  *visible += v;
  *full += n_planes * prior_tokens;
}

// ------------------------------------------------------------------------------------------- host snapshot
// Page "기술 요약: 생성형 월드 모델을 위한 지속적 계산 상태" (gist.science/ko/paper/2607.21686), section "PCS contract":
// a checkpoint / restore pair whose restore gives back a state equal to the original (round trip) and whose
// checkpoint holds exactly the state that cannot be re-derived (snapshot completeness).  For the pruned cache that
// state is: every plane's sink rows and its history rows [0, hist_len), the live ring slots of the dense window,
// hist_len, hist_t[0, longest history) and the query frame q0.  Rows past a plane's history and ring slots that
// are not live are free space and are not saved.
//
// Image (little-endian), all offsets in bytes:
//   [0, 128)    header: "DCPSNAP1", int32 L, H, D, dtype, int64 cap, hist_cap, sink_rows, chunk_rows,
//               int32 window_chunks, uint32 live_slots (bit s = ring slot s is live), int32 q0, int32 hist_t_len,
//               int64 row_bytes, rows_per_tensor, total_bytes, zero padding
//   [128, ...)  int32 hist_len[L*H], then int32 hist_t[hist_t_len] (hist_t_len = longest history)
//   data_off = first multiple of 256 after those: K block, then V block; each block holds, plane by plane, the
//               plane's sink rows and history rows [0, hist_len[p]) (one run: they are adjacent in the cache),
//               then its live ring slots in increasing slot order (chunk_rows rows each).
static int64_t snap_align256(int64_t x) { return (x + 255) & ~(int64_t)255; }

struct snap_geom {
  int64_t C, sink_rows, row_bytes, n_planes, rows_per_tensor, hist_t_len, data_off, total;
  int32_t n_live;
};

static int32_t snap_geometry(const oracle_cache* c, const oracle_config* cfg, uint32_t live_slots, snap_geom* g) {
  g->C = (int64_t)cfg->tokens_per_frame * cfg->frames_per_chunk;
  g->sink_rows = (int64_t)cfg->sink_chunks * g->C;
  g->row_bytes = (int64_t)c->D * elem_size(c->dtype);
  g->n_planes = (int64_t)c->L * c->H;
  if (cfg->window_chunks + 1 > 32) return ORACLE_EINVAL;
  if (cfg->window_chunks + 1 < 32 && (live_slots >> (cfg->window_chunks + 1)) != 0) return ORACLE_EINVAL;
  g->n_live = 0;
  for (int32_t s = 0; s <= cfg->window_chunks; ++s) g->n_live += (live_slots >> s) & 1u;
  g->rows_per_tensor = 0;
  g->hist_t_len = 0;
  for (int64_t p = 0; p < g->n_planes; ++p) {
    if (c->hist_len[p] < 0 || c->hist_len[p] > c->hist_cap) return ORACLE_EINVAL;
    g->rows_per_tensor += g->sink_rows + c->hist_len[p] + (int64_t)g->n_live * g->C;
    if (c->hist_len[p] > g->hist_t_len) g->hist_t_len = c->hist_len[p];
  }
  g->data_off = snap_align256(128 + 4 * g->n_planes + 4 * g->hist_t_len);
  g->total = g->data_off + 2 * g->rows_per_tensor * g->row_bytes;
  return ORACLE_OK;
}

int64_t oracle_snapshot_size(const oracle_cache* c, const oracle_config* cfg, uint32_t live_slots) {
  snap_geom g;
  return snap_geometry(c, cfg, live_slots, &g) == ORACLE_OK ? g.total : -1;
}

static void put_i32(uint8_t* b, int64_t off, int32_t x) { std::memcpy(b + off, &x, 4); }
static void put_i64(uint8_t* b, int64_t off, int64_t x) { std::memcpy(b + off, &x, 8); }
static int32_t get_i32(const uint8_t* b, int64_t off) { int32_t x; std::memcpy(&x, b + off, 4); return x; }
static int64_t get_i64(const uint8_t* b, int64_t off) { int64_t x; std::memcpy(&x, b + off, 8); return x; }

// The plane's saved rows in image order: (first cache row, row count) runs.
static int32_t snap_runs(const oracle_cache* c, const oracle_config* cfg, const snap_geom& g, uint32_t live_slots,
                         int64_t p, int64_t* first, int64_t* count) {
  int32_t n = 0;
  first[n] = 0;
  count[n++] = g.sink_rows + c->hist_len[p];
  for (int32_t s = 0; s <= cfg->window_chunks; ++s)
    if ((live_slots >> s) & 1u) {
      first[n] = g.sink_rows + c->hist_cap + (int64_t)s * g.C;
      count[n++] = g.C;
    }
  return n;
}

int32_t oracle_snapshot(const oracle_cache* c, const oracle_config* cfg, uint32_t live_slots, int32_t q0,
                        uint8_t* out, int64_t out_bytes) {
  snap_geom g;
  if (snap_geometry(c, cfg, live_slots, &g) != ORACLE_OK || out_bytes < g.total) return ORACLE_EINVAL;
  std::memset(out, 0, (size_t)g.data_off);
  std::memcpy(out, "DCPSNAP1", 8);
  put_i32(out, 8, c->L);
  put_i32(out, 12, c->H);
  put_i32(out, 16, c->D);
  put_i32(out, 20, c->dtype);
  put_i64(out, 24, c->cap);
  put_i64(out, 32, c->hist_cap);
  put_i64(out, 40, g.sink_rows);
  put_i64(out, 48, g.C);
  put_i32(out, 56, cfg->window_chunks);
  put_i32(out, 60, (int32_t)live_slots);
  put_i32(out, 64, q0);
  put_i32(out, 68, (int32_t)g.hist_t_len);
  put_i64(out, 72, g.row_bytes);
  put_i64(out, 80, g.rows_per_tensor);
  put_i64(out, 88, g.total);
  for (int64_t p = 0; p < g.n_planes; ++p) put_i32(out, 128 + 4 * p, c->hist_len[p]);
  for (int64_t j = 0; j < g.hist_t_len; ++j) put_i32(out, 128 + 4 * g.n_planes + 4 * j, c->hist_t[j]);
  int64_t first[33], count[33];
  for (int32_t tensor = 0; tensor < 2; ++tensor) {
    void* base = tensor == 0 ? c->k : c->v;
    int64_t off = g.data_off + tensor * g.rows_per_tensor * g.row_bytes;
    for (int64_t p = 0; p < g.n_planes; ++p) {
      int32_t n = snap_runs(c, cfg, g, live_slots, p, first, count);
      for (int32_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < count[r]; ++i) {
          std::memcpy(out + off, row_ptr(base, c, p, first[r] + i), (size_t)g.row_bytes);
          off += g.row_bytes;
        }
    }
  }
  return ORACLE_OK;
}

// Restore an image into a cache of the same geometry: the saved rows, hist_len and hist_t come back; free rows of
// the cache are left as they are.
int32_t oracle_restore(oracle_cache* c, const oracle_config* cfg, const uint8_t* in, int64_t in_bytes,
                       int32_t* q0_out, uint32_t* live_out) {
  if (in_bytes < 128 || std::memcmp(in, "DCPSNAP1", 8) != 0) return ORACLE_EINVAL;
  const int64_t C = (int64_t)cfg->tokens_per_frame * cfg->frames_per_chunk;
  if (get_i32(in, 8) != c->L || get_i32(in, 12) != c->H || get_i32(in, 16) != c->D || get_i32(in, 20) != c->dtype ||
      get_i64(in, 24) != c->cap || get_i64(in, 32) != c->hist_cap || get_i64(in, 40) != cfg->sink_chunks * C ||
      get_i64(in, 48) != C || get_i32(in, 56) != cfg->window_chunks)
    return ORACLE_EINVAL;
  const uint32_t live = (uint32_t)get_i32(in, 60);
  const int64_t n_planes = (int64_t)c->L * c->H;
  if (in_bytes < 128 + 4 * n_planes) return ORACLE_EINVAL;
  std::vector<int32_t> saved_len((size_t)n_planes);
  for (int64_t p = 0; p < n_planes; ++p) saved_len[(size_t)p] = get_i32(in, 128 + 4 * p);
  // geometry of the image, from its own lengths
  std::vector<int32_t> keep_len(c->hist_len, c->hist_len + n_planes);
  for (int64_t p = 0; p < n_planes; ++p) c->hist_len[p] = saved_len[(size_t)p];
  snap_geom g;
  int32_t rc = snap_geometry(c, cfg, live, &g);
  if (rc != ORACLE_OK || g.total != get_i64(in, 88) || g.total > in_bytes || g.hist_t_len != get_i32(in, 68) ||
      g.rows_per_tensor != get_i64(in, 80) || g.row_bytes != get_i64(in, 72)) {
    for (int64_t p = 0; p < n_planes; ++p) c->hist_len[p] = keep_len[(size_t)p];
    return ORACLE_EINVAL;
  }
  for (int64_t j = 0; j < g.hist_t_len; ++j) c->hist_t[j] = get_i32(in, 128 + 4 * n_planes + 4 * j);
  int64_t first[33], count[33];
  for (int32_t tensor = 0; tensor < 2; ++tensor) {
    void* base = tensor == 0 ? c->k : c->v;
    int64_t off = g.data_off + tensor * g.rows_per_tensor * g.row_bytes;
    for (int64_t p = 0; p < n_planes; ++p) {
      int32_t n = snap_runs(c, cfg, g, live, p, first, count);
      for (int32_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < count[r]; ++i) {
          std::memcpy(row_ptr(base, c, p, first[r] + i), in + off, (size_t)g.row_bytes);
          off += g.row_bytes;
        }
    }
  }
  if (q0_out) *q0_out = get_i32(in, 64);
  if (live_out) *live_out = live;
  return ORACLE_OK;
}

}  // extern "C"
