/* dcp.h - C ABI of the GB300 DeCoPrune history-KV prune step (libdcp.so).
 *
 * The method is the one described on the page "DeCoPrune이 디노이징 불일치로 비디오 KV 캐시를 85% 줄인다"
 * (onedev.kr/papers/726).  Sections of that page are cited as:
 *   [how]     어떻게 동작하나 "how it works":   per-token discrepancy l = (1/d)||x0hat(tau*) - x_final||^2, threshold
 *                                             gamma into one binary mask shared by all layers, protected sink chunk,
 *                                             dense window of the w most recent chunks, physical gather K[m], V[m]
 *                                             when a non-sink chunk leaves the window.
 *   [differs] 무엇과 다른가 "what differs":   prefix pruning (score the re-noised observed chunk against the clean
 *                                             one), RoPE re-indexing t~(t) = q0 - g(q0 - t) of key phase only, and
 *                                             the head-specialised variant (static heads: Streaming; dynamic heads:
 *                                             DeCoPrune).
 *   [use]     어떻게 쓰나 "how to use":        cumulative history-KV position reduction (PR) versus FullKV.
 *   [limits]  전제와 한계:                      schedule (999, 957, 899, 702), probe index 2 (tau* = 899), gamma 0.10.
 *
 * Conventions shared by every entry point
 *   - Pointers named *_dev, and every pointer inside dcp_cache, are DEVICE pointers owned by the caller.  Pointers
 *     named *_host are host pointers.  The library never allocates, frees or keeps any pointer past the call.
 *   - `stream` is a cudaStream_t passed as void*.  Every call is asynchronous on that stream.
 *   - Host-detectable errors (null or misaligned pointers, bad sizes, bad config) return before any launch and
 *     change nothing.  Errors only the device can see (history capacity exceeded, inconsistent head lengths or
 *     history frames) are written to the cache's device status word; nothing traps.
 *     Read it with dcp_get_status().  A step refused for capacity or inconsistent lengths leaves the cache contents
 *     and lengths as they were; a history frame outside [first non-sink frame, q0) is found while re-indexing, and
 *     only that row is left unturned.
 *   - The workspace is caller-owned device scratch of dcp_workspace_size() bytes, 256-byte aligned.  Zero it once
 *     with dcp_workspace_init() before its first use; every call leaves it ready for the next.  Calls that share a
 *     workspace or a cache must be ordered on one stream (not thread-safe per workspace or cache).  Host threads
 *     may call the library at the same time on different caches and workspaces (on one or several devices).
 *
 * KV cache layout (dcp_cache): K and V are [L][H][cap][D] arrays (bf16 or fp32), row-major, one plane of cap rows
 * per (layer, head).  Rows of a plane are laid out as
 *     [0, sink_rows)                       sink chunks (sink_chunks * C rows), never touched
 *     [sink_rows, sink_rows + hist_cap)    compacted history; hist_len[l*H + h] rows are valid
 *     [sink_rows + hist_cap, cap)          dense window ring of (window_chunks + 1) slots of C rows
 * with C = tokens_per_frame * frames_per_chunk.  Token n of a chunk (frame-major, then raster order inside a
 * frame) is row n of its slot and row n of the score inputs; its latent frame is first_frame + n / tokens_per_frame.
 * hist_t[j] is the latent frame of history position j; it is shared by every plane (all dynamic heads keep the same
 * tokens because the mask is shared; static heads keep none).  Keys are stored rotated (RoPE): the first
 * n_temporal_pairs pairs (2p, 2p+1) carry the temporal coordinate with frequency theta_p = rope_base^(-p / n_t).
 */
#ifndef DCP_H
#define DCP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t dcp_status;
#define DCP_OK 0
#define DCP_EINVAL 1    /* invalid argument, detected on the host before any launch */
#define DCP_ECAPACITY 2 /* device: history would exceed hist_cap; the step was skipped */
#define DCP_ECUDA 3     /* a CUDA runtime call failed */
#define DCP_ETIMEOUT 4  /* reserved: the kernels of this version contain no waits, so nothing times out */
#define DCP_EDEVICE 5   /* device: dynamic heads disagree on hist_len (corrupt cache state); the step was skipped */

#define DCP_BF16 0
#define DCP_F32 1

typedef struct dcp_cache {
  void* k;            /* device [L][H][cap][D], 16-byte aligned; D * element size must be a multiple of 16 */
  void* v;            /* device, same shape and type as k */
  int32_t L, H, D;    /* layers, KV heads, head_dim (D even) */
  int32_t dtype;      /* DCP_BF16 or DCP_F32 */
  int64_t cap;        /* rows per plane, >= sink_rows + hist_cap + (window_chunks + 1) * C */
  int64_t hist_cap;   /* history rows per plane */
  int32_t* hist_len;  /* device [L*H], in/out */
  int32_t* hist_t;    /* device [hist_cap], in/out */
  int32_t* status;    /* device, one int32: first device-side error of a call (0 = none) */
} dcp_cache;

typedef struct dcp_config {
  float gamma;               /* threshold on l; the page's value is 0.10 [limits] */
  int32_t keep_rule;         /* 0: keep l > gamma (DeCoPrune [how]); 1: the reverse criterion, keep !(l > gamma);
                                2: the Random ablation [limits]: keep as many tokens as rule 0 would, drawn uniformly
                                without replacement (see dcp_score_mask) */
  int32_t sink_chunks;       /* protected leading chunks [how] */
  int32_t window_chunks;     /* w: most recent chunks kept dense [how] */
  int32_t tokens_per_frame;  /* T latent tokens per latent frame */
  int32_t frames_per_chunk;  /* F latent frames per chunk (4 on the page [limits]) */
  int32_t n_temporal_pairs;  /* n_t leading rotary pairs that carry the temporal coordinate (0 <= n_t <= D/2) */
  int32_t pair_layout;       /* 0: pair p occupies dims (2p, 2p+1); no other layout is supported */
  double rope_base;          /* rotary base of the temporal ladder */
  double g_recent_R;         /* g is the identity on offsets <= R; must satisfy R >= window_chunks * F */
  double g_span_S;           /* g_mode 0: total virtual span (oldest history offset maps to S, S >= R);
                                g_mode 1: old offsets are compressed into (R, R + S] */
  int32_t g_mode;
  int32_t rephase_sink;      /* must be 0: the sink keeps its stored phase */
  int32_t max_frames;        /* largest q0 (latent frame index) the workspace is sized for */
  uint32_t random_seed;      /* keep_rule 2: a prune step draws from stream (random_seed << 32) | evict_first_frame */
  int32_t reindex_mode;      /* 0: keys take t~(t; q0) when they enter the history and the history is re-indexed at
                                every step (eager); 1: read-time re-index: history keys keep their own frame's phase,
                                move bitwise, nothing is re-indexed, and dcp_read_history_keys turns them to
                                t~(t; q0) when they are read */
  int32_t reserved;          /* must be 0 */
} dcp_config;

/* Bytes of device workspace the cache/config need (prune, compact, re-index and score calls for this cache). */
size_t dcp_workspace_size(const dcp_cache* cache, const dcp_config* cfg);

/* Bytes of device workspace a standalone dcp_score_mask over n_tok tokens needs. */
size_t dcp_score_workspace_size(int32_t n_tok);

/* Zero a workspace (stream-ordered).  Needed once per workspace, before its first use. */
dcp_status dcp_workspace_init(void* workspace_dev, size_t ws_bytes, void* stream);

/* Score + threshold + ordered index list for one chunk [how], [differs: prefix pruning uses xref = clean chunk].
 *   x0hat_dev, xref_dev : fp32 [n_tok][d] row-major (the probe-step clean prediction and the final output, or the
 *                         re-noised prediction and the clean observed chunk in the prefix pass).  Device memory, or
 *                         page-locked host memory (cudaHostAlloc / cudaHostRegister), which the scan kernel then
 *                         reads directly over the host link; other host memory is refused (DCP_EINVAL).
 *   ell_dev   (nullable): fp32 [n_tok] out, l[n] = (1/d) sum_j (x0hat[n][j] - xref[n][j])^2, fp32 arithmetic.
 *   keep_rule           : 0 keep l > gamma; 1 keep !(l > gamma); 2 the Random ablation of section "premises and
 *                         limits" (Random at the same compression ratio): keep exactly as many tokens as rule 0, the
 *                         ones with the smallest priorities z_n = n-th output (0-based) of a SplitMix64 sequence
 *                         (Steele, Lea & Flood 2014) seeded with random_stream.  The priorities of one stream are
 *                         distinct, so the kept set is unique.  Its cost grows with n_tok in one CTA (a radix
 *                         select of up to 8 passes over the chunk's priorities).
 *   random_stream       : SplitMix64 seed of rule 2 (ignored otherwise).  dcp_prune_step uses
 *                         ((uint64_t)cfg->random_seed << 32) | (uint32_t)evict_first_frame.
 *   mask_dev  (nullable): uint8 [n_tok] out, 1 = keep (rule from keep_rule).
 *   idx_dev   (nullable): int32 [n_tok] out, increasing kept positions in [0, kept).
 *   kept_dev  (nullable): int32 out, number of kept tokens.
 *   status_dev          : int32 device status word (no device error is produced by this call today).
 * Errors: DCP_EINVAL for null inputs, n_tok < 1 or > 2^30, d < 1, non-finite gamma, keep_rule outside {0, 1, 2},
 * short workspace. */
dcp_status dcp_score_mask(const float* x0hat_dev, const float* xref_dev, int32_t n_tok, int32_t d, float gamma,
                          int32_t keep_rule, uint64_t random_stream, float* ell_dev, uint8_t* mask_dev,
                          int32_t* idx_dev, int32_t* kept_dev, int32_t* status_dev, void* workspace_dev,
                          size_t ws_bytes, void* stream);

/* Physical compaction of the leaving chunk [how] with the fused key re-phase [differs].
 * The chunk in ring slot evict_slot (its first latent frame is evict_first_frame) is compacted: for every
 * dynamic plane, K and V rows idx[j] of the slot (the kept positions of mask_dev, uint8 [C]) are appended in order
 * at hist_len; each appended key's temporal pairs turn from its stored frame t to t~(t; q0); values and every other
 * key dim are copied bitwise.  hist_len of dynamic planes grows by kept, hist_t gets the kept frames.  Planes with
 * head_is_static_dev[l*H+h] != 0 (nullable: none) follow the Streaming policy and keep nothing.  The ring slot is
 * left as it was.  kept_dev (nullable) receives the kept count.
 * Device errors: DCP_ECAPACITY (hist_len + kept > hist_cap), DCP_EDEVICE (dynamic planes disagree on hist_len).
 * Host errors: DCP_EINVAL (see dcp_cache/dcp_config; evict_slot outside [0, w]; evict_first_frame < sink frames;
 * q0 < evict_first_frame + F; q0 > max_frames). */
dcp_status dcp_compact_layers(const dcp_cache* cache, const dcp_config* cfg, int32_t evict_slot,
                              int32_t evict_first_frame, const uint8_t* mask_dev, const uint8_t* head_is_static_dev,
                              int32_t q0, int32_t* kept_dev, void* workspace_dev, size_t ws_bytes, void* stream);

/* RoPE re-index of the history already present [differs]: when the query frame moves from q0_prev to q0, every
 * history key whose t~(t) changes turns its temporal pairs by theta_p * (t~(t; q0) - t~(t; q0_prev)) in place.
 * Rows whose t~ does not change are not touched.  Values are never touched.
 * Host errors: DCP_EINVAL (q0_prev > q0, q0 > max_frames, q0_prev < sink frames, bad cache/config). */
dcp_status dcp_rope_reindex(const dcp_cache* cache, const dcp_config* cfg, int32_t q0_prev, int32_t q0,
                            void* workspace_dev, size_t ws_bytes, void* stream);

/* One full prune step, the unit the library is measured on: score the leaving chunk (x0hat/xref fp32 [C][d]),
 * threshold it, build the index list, re-index the history present before the step from q0_prev to q0, and compact
 * the chunk into the history with its keys re-phased to q0.  Equivalent to dcp_score_mask + dcp_rope_reindex +
 * dcp_compact_layers on the same arguments.  x0hat_dev / xref_dev may be page-locked host memory (as for
 * dcp_score_mask: read by the scan kernel over the host link, no separate copy).  kept_dev (nullable, device) and
 * kept_host_pinned (nullable, page-locked host memory, written by the scan kernel's last CTA; valid once the stream
 * has reached the end of the step) receive the kept count; pageable host memory there is refused (DCP_EINVAL).  dcp_workspace_outputs() gives the device
 * addresses where the step leaves l, the mask and the index list. */
dcp_status dcp_prune_step(const dcp_cache* cache, const dcp_config* cfg, const float* x0hat_dev, const float* xref_dev,
                          int32_t d, int32_t evict_slot, int32_t evict_first_frame, int32_t q0_prev, int32_t q0,
                          const uint8_t* head_is_static_dev, int32_t* kept_dev, int32_t* kept_host_pinned,
                          void* workspace_dev, size_t ws_bytes, void* stream);

/* CUDA graphs: dcp_prune_step (and dcp_paged_prune_step, dcp_read_history_keys) enqueue only kernel launches on
 * `stream` (with programmatic-dependent-launch attributes, which stream capture records as programmatic edges), so a
 * call can be recorded into a CUDA graph by stream capture and replayed; the replay repeats the step with the
 * captured arguments and pointers.  Make one call with the same cache geometry outside capture first: the first call
 * on a device sets up per-kernel launch attributes (shared-memory size, occupancy), which capture does not allow.
 * Score inputs in page-locked host memory are read at replay time, so a serving loop can refill them between
 * replays. */

/* Largest workspace dcp_prune_step_noalloc can use: 4 MiB (the full-depth 40 x 40 x 128 cache with 6240-token
 * chunks and max_frames 256 needs about 190 KB). */
#define DCP_NOALLOC_WORKSPACE_BYTES (4u << 20)

/* dcp_prune_step for callers that cannot allocate device memory (for example code running inside a device
 * allocator's callback, or an engine that forbids allocation after start-up).  The paper has no counterpart: this
 * is a packaging variant of dcp_prune_step, with the same arguments minus the workspace and the same results.
 * Instead of a caller workspace it uses a scratch array of DCP_NOALLOC_WORKSPACE_BYTES compiled into the library,
 * which every GPU that loads the library holds until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   - Returns DCP_EINVAL when dcp_workspace_size(cache, cfg) is 0 (invalid) or larger than the scratch array, and
 *     for every argument dcp_prune_step rejects.
 *   - The first call made in a CUDA context (for the runtime's primary contexts: the first call with a given device
 *     current) looks up the array's device address in that context (cudaGetSymbolAddress); make that first call
 *     before any stream capture.  The address is remembered per context id, so a context created later (after
 *     cudaDeviceReset, say) is looked up afresh.
 *   - Every call shares the one array and finds the previous call's contents in it.  Only the scan's 256-byte control
 *     block must start at zero: it is cleared on `stream` once the arguments have passed every host check, right
 *     before the first kernel (a refused call launches nothing).  Calls whose work overlaps on the GPU (other streams
 *     or threads on the same device) race on the array: order them. */
dcp_status dcp_prune_step_noalloc(const dcp_cache* cache, const dcp_config* cfg, const float* x0hat_dev,
                                  const float* xref_dev, int32_t d, int32_t evict_slot, int32_t evict_first_frame,
                                  int32_t q0_prev, int32_t q0, const uint8_t* head_is_static_dev, int32_t* kept_dev,
                                  int32_t* kept_host_pinned, void* stream);

/* Read-time re-index [differs] (reindex_mode 1): the history keys of planes [plane0, plane0 + n_planes) as attention
 * at query frame q0 sees them.  Row j of plane p (j < hist_len[p]) is the stored key, which sits at its own frame
 * t = hist_t[j], with each temporal pair p' turned once by theta_p' * (t~(t; q0) - t); every other dim is copied
 * bitwise.  out_dev: [n_planes][hist_cap][D] of the cache's type (16-byte aligned); rows at or past a plane's
 * history length are not written.  Keys are turned from their raw phase at every read, so repeated reads at moving
 * q0 accumulate no rounding.  Two launches (phase table, then the read), no host synchronisation.
 * Device errors: DCP_EDEVICE (a hist_len outside [0, hist_cap]: nothing is written; a history frame outside
 * [sink frames, q0): that row is not written).
 * Host errors: DCP_EINVAL (bad cache/config, reindex_mode != 1, q0 outside [sink frames, max_frames], plane range
 * outside [0, L*H), null or misaligned out_dev, short workspace). */
dcp_status dcp_read_history_keys(const dcp_cache* cache, const dcp_config* cfg, int32_t q0, int32_t plane0,
                                 int32_t n_planes, void* out_dev, void* workspace_dev, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------------------------
 * Paged variant: the same prune step on a cache kept in block pools addressed through block tables, the layout of
 * paged serving stacks.  The method is unchanged (section "how it works": the kept K[m], V[m] are physically moved
 * into the history, shortening the real KV sequence); only where a row lives differs.
 *   pool layout DCP_PAGED_HND: k_pool, v_pool are [L][n_blocks][H][block_size][D] (one pool per layer, each block
 *               holding block_size consecutive positions of every head, head-major inside the block);
 *   pool layout DCP_PAGED_NHD: [L][n_blocks][block_size][H][D] (position-major inside the block).
 * Position i of the history of plane (l, h) is row i % block_size of block hist_blocks[i / block_size] in layer
 * l's pool, head h; position n of ring slot s is row n % block_size of block
 * window_blocks[s * C / block_size + n / block_size].  One table serves every layer and head (a block id names
 * the same block in each layer's pool).  The sink is never touched by a prune step, so its table is not needed
 * here.  The caller owns the tables and the pools and must give the history, the ring slots and the sink distinct
 * blocks.  Table entries outside [0, n_blocks) are found by the scan kernel before anything moves: the step then
 * records DCP_EDEVICE and leaves the cache as it was.
 * --------------------------------------------------------------------------------------------------------------- */
#define DCP_PAGED_HND 0
#define DCP_PAGED_NHD 1

typedef struct dcp_paged_cache {
  void* k_pool;                /* device, 16-byte aligned; D * element size a multiple of 16 */
  void* v_pool;
  int32_t L, H, D, dtype;
  int32_t block_size;          /* positions per block; C and hist_cap are multiples of it */
  int32_t layout;              /* DCP_PAGED_HND or DCP_PAGED_NHD */
  int64_t n_blocks;            /* blocks in each layer's pool */
  int64_t hist_cap;            /* history positions covered by hist_blocks */
  const int32_t* hist_blocks;  /* device [hist_cap / block_size] */
  const int32_t* window_blocks;/* device [(window_chunks + 1) * C / block_size] */
  int32_t* hist_len;           /* device [L*H], in/out */
  int32_t* hist_t;             /* device [hist_cap], in/out */
  int32_t* status;             /* device, one int32 */
} dcp_paged_cache;

/* Workspace bytes of dcp_paged_prune_step for this cache/config (0 if either is invalid). */
size_t dcp_paged_workspace_size(const dcp_paged_cache* cache, const dcp_config* cfg);

/* Phase table of read-time re-index [differs], for kernels that fuse the turn into their own reads of K (attention):
 * for frames t in [frame_lo, frame_hi) and temporal pairs p < n_t, the turn from a key's own phase t to t~(t; q0):
 *   out_dev[(t - frame_lo) * n_t + p] = {c_hi, c_lo, s_hi, s_lo}  (four floats, 16-byte aligned),
 * with cos(phi) = c_hi + c_lo and sin(phi) = s_hi + s_lo to about 40 bits, phi = theta_p * (t~(t; q0) - t) and
 * theta_p = rope_base^(-p / n_t), evaluated in double precision; c_hi and s_hi carry 16 significant bits, so their
 * products with bf16 values are exact in fp32.  Pair (a, b) turns to (a cos - b sin, a sin + b cos).  Frames that
 * keep their phase get {1, 0, 0, 0}.  dcp_read_history_keys applies exactly this table.  One stream-ordered launch.
 * Host errors: DCP_EINVAL (config fields as for dcp_workspace_size; frame_lo < sink frames, frame_hi > q0,
 * frame_lo > frame_hi, n_temporal_pairs < 1, null or misaligned out_dev). */
dcp_status dcp_phase_table(const dcp_config* cfg, int32_t q0, int32_t frame_lo, int32_t frame_hi, float* out_dev,
                           void* stream);

/* dcp_read_history_keys on a paged cache (history rows found through hist_blocks; entries are checked first). */
dcp_status dcp_paged_read_history_keys(const dcp_paged_cache* cache, const dcp_config* cfg, int32_t q0,
                                       int32_t plane0, int32_t n_planes, void* out_dev, void* workspace_dev,
                                       size_t ws_bytes, void* stream);

/* dcp_prune_step on a paged cache: same arguments, results and errors, plus DCP_EDEVICE for a table entry outside
 * [0, n_blocks) (checked before anything moves) and DCP_EINVAL for a block size that does not divide C or hist_cap
 * or an unknown layout. */
dcp_status dcp_paged_prune_step(const dcp_paged_cache* cache, const dcp_config* cfg, const float* x0hat_dev,
                                const float* xref_dev, int32_t d, int32_t evict_slot, int32_t evict_first_frame,
                                int32_t q0_prev, int32_t q0, const uint8_t* head_is_static_dev, int32_t* kept_dev,
                                int32_t* kept_host_pinned, void* workspace_dev, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------------------------
 * Host snapshot and restore of the pruned cache.
 * Page "기술 요약: 생성형 월드 모델을 위한 지속적 계산 상태" (gist.science/ko/paper/2607.21686), section "PCS contract":
 * a checkpoint / restore pair where restore gives back the state (round trip) and the checkpoint holds exactly the
 * state that cannot be re-derived (snapshot completeness).  For this cache that state is each plane's sink rows and
 * history rows [0, hist_len), the live ring slots of the dense window (bit s of live_slots = ring slot s holds a
 * chunk; window_chunks + 1 <= 32), hist_len, hist_t[0, longest history) and the query frame q0.  Rows past a
 * plane's history and ring slots that are not live are free space: never saved, never written back.
 *
 * Image layout (little-endian, byte offsets):
 *   [0, 128)   header: char magic[8] = "DCPSNAP1"; int32 L, H, D, dtype; int64 cap, hist_cap, sink_rows,
 *              chunk_rows (C); int32 window_chunks; uint32 live_slots; int32 q0; int32 hist_t_len (longest
 *              history); int64 row_bytes, rows_per_tensor, total_bytes; zero up to byte 128.
 *   [128, ..)  int32 hist_len[L*H], then int32 hist_t[hist_t_len].
 *   data_off   the first multiple of 256 at or after the end of hist_t (bytes in between are zero).  The K block
 *              then the V block (rows_per_tensor rows each): plane by plane (plane = l*H + h), the plane's sink and
 *              history rows [0, sink_rows + hist_len), then its live ring slots in increasing slot order (C rows
 *              each).  total_bytes = data_off + 2 * rows_per_tensor * row_bytes.
 * Images move between the device and page-locked host memory (cudaHostAlloc / cudaHostRegister, 16-byte aligned)
 * by a kernel pair on the caller's stream (the device reaches the host image through unified addressing).
 * --------------------------------------------------------------------------------------------------------------- */

/* Image size when every plane's history is full: an upper bound for dcp_snapshot.  0 for an invalid
 * cache/config or live_slots. */
size_t dcp_snapshot_max_bytes(const dcp_cache* cache, const dcp_config* cfg, uint32_t live_slots);

/* Write the cache's state into image_host (image_bytes long), stream-ordered, without host synchronisation: the
 * image is complete once `stream` has reached this point.  Its total_bytes field (offset 88) gives the size used.
 * Device errors: DCP_ECAPACITY (the image is too small: only the header is written, with the size needed),
 * DCP_EDEVICE (a hist_len outside [0, hist_cap]: nothing but the header is written).
 * Host errors: DCP_EINVAL (bad cache/config, live_slots with bits past the ring, image not page-locked host memory
 * or not 16-byte aligned, image_bytes < 128, short workspace). */
dcp_status dcp_snapshot(const dcp_cache* cache, const dcp_config* cfg, uint32_t live_slots, int32_t q0,
                        void* image_host, size_t image_bytes, void* workspace_dev, size_t ws_bytes, void* stream);

/* Restore an image into a cache of the same geometry (L, H, D, dtype, cap, hist_cap, sink rows, C, window_chunks).
 * The image must be complete when the call is made (any snapshot that wrote it has been synchronised): the host
 * checks its header and lengths, fills q0_out / live_slots_out (nullable), then the copy is stream-ordered.  The
 * saved rows, hist_len and hist_t come back; free rows of the cache are not touched.
 * Host errors: DCP_EINVAL (bad magic, geometry that differs from the cache, inconsistent lengths or sizes,
 * image_bytes short of total_bytes, image not page-locked, short workspace).  Nothing is launched then. */
dcp_status dcp_restore(const dcp_cache* cache, const dcp_config* cfg, const void* image_host, size_t image_bytes,
                       int32_t* q0_out, uint32_t* live_slots_out, void* workspace_dev, size_t ws_bytes,
                       void* stream);

/* Device addresses inside a prune-step workspace: l (fp32 [C]), the mask (uint8 [C]) and the index list
 * (int32 [C], first `kept` entries valid) of the last dcp_prune_step / dcp_compact_layers call. */
dcp_status dcp_workspace_outputs(const dcp_cache* cache, const dcp_config* cfg, void* workspace_dev, float** ell_dev,
                                 uint8_t** mask_dev, int32_t** idx_dev);

/* Synchronise `stream` and return the device status word (DCP_OK if no device error was recorded). */
dcp_status dcp_get_status(const int32_t* status_dev, void* stream);

/* Clear the device status word (stream-ordered). */
dcp_status dcp_reset_status(int32_t* status_dev, void* stream);

const char* dcp_status_string(dcp_status s);

/* Cumulative PR bookkeeping [use]: PR = 1 - visible / full summed over generated chunks, where a chunk that has
 * `prior_tokens` tokens before it sees, in each of n_planes planes, the sink, its hist_len rows and the dense
 * window; FullKV would see all prior tokens.  hist_len_sum is the sum of hist_len over the planes (host value). */
typedef struct dcp_pr_counter {
  int64_t visible;
  int64_t full;
} dcp_pr_counter;
void dcp_pr_add_chunk(dcp_pr_counter* acc, int64_t n_planes, int64_t hist_len_sum, int64_t sink_tokens_visible,
                      int64_t window_tokens_visible, int64_t prior_tokens);
double dcp_pr_value(const dcp_pr_counter* acc);

/* Profiling hook.  When ev_after_scan / ev_after_gather are non-null (cudaEvent_t passed as void*), every later
 * dcp_prune_step records them on its stream right after the scan kernel and right after the gather kernel, so a
 * caller can time each kernel with CUDA events inside a timed region.  Pass nulls to switch it off.  Process-wide
 * setting, not thread-safe. */
dcp_status dcp_set_phase_events(void* ev_after_scan, void* ev_after_gather);

/* ABI check for bindings: (sizeof(dcp_cache) << 16) | sizeof(dcp_config). */
uint32_t dcp_abi_struct_sizes(void);

/* ABI check for bindings: sizeof(dcp_paged_cache). */
uint32_t dcp_abi_paged_cache_size(void);


#ifdef __cplusplus
}
#endif

#endif /* DCP_H */
