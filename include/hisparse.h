/*
 * hisparse.h -- C ABI of the HiSparse RESOLVE hot path on GB300 (sm_103a).
 *
 * HiSparse keeps the authoritative KV of every decoding request in pinned host
 * memory and only a fixed B-slot hot buffer per (request, layer) in HBM.  Each
 * sparse layer, after its indexer picks k logical positions, runs RESOLVE:
 * find the selections already in the hot buffer, pick LRU victims for the
 * rest, copy the missing records from the host pool into the victims with GPU
 * threads, and publish the position -> slot vector that sparse attention reads.
 *
 * Sources (cited by page title and section):
 *   [DD]  gentlecold.top, "HiSparse 深度解析：论文、SGLang 实现与 vLLM Hybrid
 *         HiSparse" (HiSparse deep dive): §3.2 hierarchy and metadata, §3.3
 *         replacement policy, §3.4 request lifecycle and write-through, §3.5
 *         RESOLVE fused kernel, §3.6 exact cross-layer prefetch, §5.2
 *         per-request tensors and the newest slot, §5.5 swap-in kernel,
 *         §5.6 prefetch in SGLang, §5.7 --hisparse-config fields.
 *   [VD]  docs.vllm.ai, "HiSparse local KV offload architecture" (vLLM design
 *         doc): "Hot lookup and LRU" and "Performance invariants".
 *
 * Conventions
 *   - Every call returns HISPARSE_OK (0) or a negative HISPARSE_E* code.
 *     Host-side argument errors are detected before any CUDA call.
 *   - "d_" arguments are device pointers; everything else is host memory.
 *   - Launch calls (resolve, writeback, prefetch_plan) never allocate, never
 *     synchronise and never read device values on the host, so they can be
 *     captured in a CUDA graph ([VD] "Performance invariants": no scalar
 *     readback, no CPU/device round trip).
 *   - Errors in device-side inputs never trap the GPU: the kernel records them
 *     in a sticky status word (HISPARSE_ERR_* bits, read with
 *     hisparse_get_status) and in a per-(layer, request) error code, and the
 *     failing unit keeps its previous state.
 *   - A stream argument is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).
 */
#ifndef HISPARSE_H
#define HISPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define HISPARSE_OK 0
#define HISPARSE_EINVAL (-1)  /* NULL pointer, bad layer id, misaligned buffer,
                                 record size not a multiple of 16, bad stride */
#define HISPARSE_EBOUND (-2)  /* a size outside what the library supports
                                 (B < k, B > 32767, shared memory too large, ...) */
#define HISPARSE_ENOMEM (-3)  /* device or pinned host allocation failed */
#define HISPARSE_ECUDA (-4)   /* a CUDA call failed; see hisparse_last_cuda_error */
#define HISPARSE_EROLE (-5)   /* resolve on a shared-index layer, or a replay
                                 pair that is not (anchor, its follower) */

/* ---- device-detected error bits (status word and per-unit codes) ------- */
#define HISPARSE_ERR_RANGE 1u /* a selected position outside [-1, P), or a
                                 newest / write-back position outside [-1, P) */
#define HISPARSE_ERR_DUP 2u   /* one position selected twice by one request */

/* ---- resolve flags ----------------------------------------------------- */
#define HISPARSE_RECORD_PLAN 1u /* record the miss plan for shared layers ([DD] §5.5) */
#define HISPARSE_SKIP_IO 2u     /* the pages' no-IO oracle: metadata only, missed
                                   rows keep stale bytes ([DD] §4.4, §5.6) */
#define HISPARSE_FROM_MIRROR 4u /* copy missed rows from the layer's HBM mirror
                                   of the host pool instead of the host pool */
#define HISPARSE_UNION 8u       /* speculative verification ([DD] §6.5): d_sel holds a
                                   request's verify rows one after another (top_k
                                   entries in all) and RESOLVE works on their union:
                                   a position repeated anywhere is resolved at its
                                   first reference and every reference outputs the
                                   same row (no HISPARSE_ERR_DUP); misses take victims
                                   in first-reference order and are fetched, counted
                                   and planned once.  Page-table lookup only. */
#define HISPARSE_WITH_SHARED 16u /* also fill the layer's shared-index layers
                                   (anchor_of == layer; 8 at most) in the same
                                   launch: each missed record's row of every such
                                   layer is read from that layer's host pool (its
                                   mirror with FROM_MIRROR) into its hot buffer at
                                   the same slot -- the bytes hisparse_prefetch_plan
                                   would copy, without a plan replay.  Their
                                   write-backs must come first.  With SKIP_IO
                                   nothing is filled.  Page-table lookup only;
                                   more than 8 shared-index layers: EBOUND. */

/* ---- lookup strategies (hisparse_config.lookup) ------------------------- */
#define HISPARSE_LOOKUP_PAGE_TABLE 0
#define HISPARSE_LOOKUP_HASH 1

typedef struct hisparse_handle hisparse_handle;

/* Sizes of one HiSparse instance ([DD] §5.7 --hisparse-config: top_k,
 * device_buffer_size = B excluding the newest page). */
typedef struct {
  int32_t num_requests;     /* R: requests in the (graph-padded) decode batch, 1..8192 */
  int32_t num_layers;       /* L: layers with a hot buffer, 1..4096 */
  int32_t top_k;            /* k: selections per (request, layer, step), >= 1 */
  int32_t buffer_slots;     /* B: LRU slots per (request, layer), k <= B <= 32767;
                               row B of every hot buffer is the newest-token row */
  int64_t host_rows;        /* P: logical positions (host rows) per (request, layer),
                               1 <= P <= 2^31 - 1 */
  int32_t record_bytes;     /* bytes of one position's KV in one layer; a positive
                               multiple of 16 */
  int32_t ctas_per_request; /* CTAs (one thread-block cluster) per request in
                               resolve, 1..16; 0 = chosen by the library */
  int32_t replay_ctas;      /* CTAs of the plan-replay kernel; 0 = chosen by the library */
  int32_t lookup;           /* how RESOLVE finds the resident selections:
                               HISPARSE_LOOKUP_PAGE_TABLE (0, default): worker CTAs read
                               the page table, mark hits and start the missed-record
                               reads while the leader CTA chooses victims;
                               HISPARSE_LOOKUP_HASH (1): one CTA stages the selection in
                               a shared-memory hash and probes every slot ([DD] §3.5
                               stages 1-2), then the cluster fetches.  Same results. */
  const int32_t *anchor_of; /* [L] host array or NULL (= all -1): -1 if the layer runs
                               RESOLVE itself, else the id of the anchor layer whose
                               selection and slot table it shares ([DD] §3.6).  An
                               anchor must itself have anchor_of == -1. */
} hisparse_config;

/* Memory of one layer.  The caller owns it and keeps it alive until
 * hisparse_destroy.  Row (r, p) of the host pool is at
 * host_pool + r*host_req_stride + p*host_row_stride; row (r, s) of the hot
 * buffer, s in [0, B], is at hot + r*hot_req_stride + s*hot_row_stride.
 * All pointers and strides must be multiples of 16 bytes, and row strides at
 * least record_bytes. */
typedef struct {
  void *host_pool;          /* pinned, device-mapped host memory (hisparse_host_alloc or
                               cudaHostAlloc / cudaHostRegister with mapping) */
  int64_t host_req_stride;
  int64_t host_row_stride;
  void *hot;                /* device memory, R x (B+1) rows */
  int64_t hot_req_stride;
  int64_t hot_row_stride;
  void *mirror;             /* optional device copy of host_pool with the host pool's
                               strides, read instead of the pool with
                               HISPARSE_FROM_MIRROR; NULL if none.  The caller fills it;
                               the library keeps it equal to the pool: every write-back
                               (hisparse_writeback, the fused one of
                               hisparse_resolve_step) stores the row to both. */
} hisparse_layer_buffers;

/* Read-only facts about an instance (for reporting). */
typedef struct {
  int32_t ctas_per_request; /* cluster size used by resolve */
  int32_t threads_per_cta;
  int32_t smem_bytes;       /* dynamic shared memory per resolve CTA */
  int32_t hash_capacity;    /* open-addressing table entries per request */
  int32_t replay_ctas;
  int32_t sm_count;
  int64_t metadata_bytes;   /* device bytes owned by the library */
  int32_t lookup;           /* HISPARSE_LOOKUP_* in use */
} hisparse_info;

/* Create an instance.  Validates every size and buffer on the host, then
 * allocates the library-owned metadata in device memory (slot -> position,
 * LRU order, page table, miss plan, miss counts, error codes, status word;
 * [DD] §5.2 tensor table) and resets every unit to its admission state: all
 * slots empty, LRU order 0..B-1 ([DD] §5.4 request release).  Layers with
 * anchor_of != -1 get no metadata of their own.  Synchronises the device.
 * Errors: EINVAL, EBOUND, EROLE (bad anchor_of), ENOMEM, ECUDA. */
int hisparse_init(const hisparse_config *cfg, const hisparse_layer_buffers *layers /* [L] */,
                  hisparse_handle **out);

/* Free the library-owned metadata (not the caller's buffers).  Synchronises. */
int hisparse_destroy(hisparse_handle *h);

/* RESOLVE one layer for requests [0, *d_num_reqs) in one launch ([DD] §3.5;
 * [VD] "Hot lookup and LRU").  For request r:
 *   d_sel[r*k + i]  int32 logical position, or -1 for padding;
 *   d_newest[r]     int32 position of the newest token, bound to hot row B and
 *                   never fetched, or -1 (d_newest may be NULL = all -1);
 *   d_out[r*k + i]  int32 physical hot row for d_sel[r*k+i]: a slot in [0, B),
 *                   B for the newest token, -1 for padding ([DD] §3.5 stage 5,
 *                   top_k_device_locs aligned with the top-k order).
 * d_num_reqs is a device int32 read by the kernel, so a graph captured at the
 * padded batch size R serves any smaller batch ([DD] §5.5 num_real_reqs);
 * NULL means R.  Requests at or beyond it are not touched.
 * Replacement rule ([DD] §3.3, worked example §3.5): hits of this step become
 * the most recent (in ascending slot order), this step's fetches come just
 * before them (in selection-list order), and the j-th miss in list order takes
 * the j-th least recent slot that is not a hit; empty slots are ordinary LRU
 * entries.  Which slot each missed record lands in is fixed by this rule; the
 * order the records are read in is not part of the result.  On a
 * device-detected input error (HISPARSE_ERR_*) the request's out row is all
 * -1 and its state is unchanged.
 * The host pool rows fetched must be complete when this runs (order any
 * write-back before it with an event), and hot row B must already hold the
 * newest token's KV.  flags: HISPARSE_RECORD_PLAN | HISPARSE_SKIP_IO |
 * HISPARSE_FROM_MIRROR | HISPARSE_UNION | HISPARSE_WITH_SHARED (the last two
 * with the page-table lookup only; EINVAL otherwise, and EBOUND for
 * WITH_SHARED on more than 8 shared-index layers).  With the page-table lookup the kernel is launched
 * with programmatic dependent launch: it may be set up while the previous
 * kernel of `stream` finishes but reads no memory before that kernel is done,
 * and the next kernel, if launched the same way, may be set up while this one
 * runs.  Errors: EINVAL, EBOUND, EROLE (layer is a follower), ECUDA. */
int hisparse_resolve(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                     const int32_t *d_num_reqs, const int32_t *d_newest, int32_t *d_out,
                     uint32_t flags, void *stream);

/* hisparse_writeback(h, layer, d_prev_pos, d_new_rows, d_num_reqs) followed by
 * hisparse_resolve(h, layer, ...) for one layer that runs RESOLVE, in one
 * launch and with identical results: row B of each request is written to
 * host row d_prev_pos[r] (skipped for -1), d_new_rows (device [R][record_bytes],
 * may be NULL) replaces it, and then the layer is resolved -- a previous
 * token that is selected again is filled from the row B just written back
 * rather than read back over the host link.  With HISPARSE_LOOKUP_HASH this
 * is two launches (d_prev_pos must then be given).  Shared-index layers keep
 * using hisparse_writeback.  Errors: as hisparse_resolve and hisparse_writeback. */
int hisparse_resolve_step(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                          const int32_t *d_num_reqs, const int32_t *d_newest,
                          const int32_t *d_prev_pos, const void *d_new_rows, int32_t *d_out,
                          uint32_t flags, void *stream);

/* Options of hisparse_resolve_ex; zero-initialise and set what is used. */
typedef struct {
  /* fused write-through, as hisparse_resolve_step (both NULL: none) */
  const int32_t *d_prev_pos;  /* device [R] */
  const void *d_new_rows;     /* device [R][record_bytes], 16-byte aligned */
  /* resident tier, as hisparse_resolve_resident (NULL: none) */
  const int32_t *d_res_blocks; /* device [R][res_max_blocks] */
  int32_t res_max_blocks;
  int32_t res_block_tokens;
  /* Block-id selections ([DD] §5.5, TopKIsBlocks): when > 1, d_sel holds
   * top_k / sel_block_tokens block ids per request ([R][top_k /
   * sel_block_tokens]); block b stands for positions b*sel_block_tokens ..
   * b*sel_block_tokens + sel_block_tokens - 1 in that order, -1 for as many
   * paddings, and d_out stays [R][top_k], one entry per position.  The kernel
   * expands the ids in registers; no position list is written.  Other negative
   * ids, and ids whose positions reach P, fail the request with
   * HISPARSE_ERR_RANGE.  top_k must be a multiple; page-table lookup only.
   * 0 or 1: d_sel holds positions. */
  int32_t sel_block_tokens;
  /* Short requests ([DD] §5.4 short-sequence fast path and on-demand buffer
   * growth; §5.5 the swap-in kernel's early return): device int32 [R], the
   * number of positions of each request so far, the newest included; NULL:
   * every request takes the general path.  A request with d_seq_lens[r] <= B
   * skips the LRU lookup.  First its buffer grows by its previous token: when
   * d_prev_pos[r] >= 0 (the fused write-through), that token is resolved as a
   * one-entry selection -- a miss takes the least recent slot, filled from
   * the row it was just written back from (and, with HISPARSE_WITH_SHARED,
   * the shared-index layers' rows), is mapped and recorded in the plan; a hit
   * moves its slot to the recent end; without a previous token the miss
   * count and plan count are 0.  Then each selection outputs -1 for padding,
   * its resident row when d_res_blocks has one, B for d_newest[r], else the
   * slot numbered like the position; a position outside [0, seq_len) or
   * [0, P) fails the request's output (all -1, HISPARSE_ERR_RANGE; the
   * growth stays); repeats are not errors.  This is exact when slot s holds
   * position s for every position before the newest: a request admitted
   * with hisparse_admit preloading its host_len positions and decoded with
   * the fused write-through since.  The pages' early return then equals the
   * general resolve's output (all hits) without its LRU work.  Longer
   * requests in the same launch take the general path; a request that
   * outgrows B takes it from its next step on, its un-grown slot being the
   * least recent.  Page-table lookup only. */
  const int32_t *d_seq_lens;
} hisparse_resolve_options;

/* The general RESOLVE: hisparse_resolve with the options above (opt may be
 * NULL = hisparse_resolve).  hisparse_resolve_step and
 * hisparse_resolve_resident are this call with the corresponding options.
 * Errors: as hisparse_resolve_step; EINVAL for options the lookup does not
 * support or a top_k that is not a multiple of sel_block_tokens. */
int hisparse_resolve_ex(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                        const int32_t *d_num_reqs, const int32_t *d_newest,
                        const hisparse_resolve_options *opt, int32_t *d_out, uint32_t flags,
                        void *stream);

/* Three-tier RESOLVE ([VD] "Hot lookup and LRU": resident page -> resident
 * physical row, else hot row, else a copy from pinned host memory; [DD] §6.5):
 * hisparse_resolve_step with a resident tier checked first.  d_res_blocks is a
 * device int32 [R][res_max_blocks] block table shared by the layers: entry b of
 * request r is -1 when positions [b*res_block_tokens, (b+1)*res_block_tokens)
 * have no device-resident copy, else the index of their block in the caller's
 * resident store; positions past the table are not resident.  A selected
 * position p in a resident block outputs B + 1 + row, row = entry *
 * res_block_tokens + p % res_block_tokens: it touches neither the LRU, the page
 * table, the miss count nor the plan, and is not part of the duplicate check
 * (a repeated resident position outputs its row at each index).  A selected
 * position whose entry is below -1, or whose B + 1 + row exceeds INT32_MAX,
 * fails the request with HISPARSE_ERR_RANGE.  A request whose selections are
 * all resident leaves its cache state unchanged.  d_res_blocks == NULL is
 * hisparse_resolve_step.  Page-table lookup only (EINVAL with
 * HISPARSE_LOOKUP_HASH, or with res_max_blocks or res_block_tokens < 1).
 * Errors: as hisparse_resolve_step. */
int hisparse_resolve_resident(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                              const int32_t *d_num_reqs, const int32_t *d_newest,
                              const int32_t *d_prev_pos, const void *d_new_rows,
                              const int32_t *d_res_blocks, int32_t res_max_blocks,
                              int32_t res_block_tokens, int32_t *d_out, uint32_t flags,
                              void *stream);

/* Admission of requests into the cache ([DD] §5.3, direct admission: a long
 * request starts with every token absent and misses everything on its first
 * step; a short one, whose host length fits the buffer, is preloaded).  For
 * i < n, request d_reqs[i] (device int32 [n]) of `layer` (-1: every layer)
 * goes to the reset state, and, when d_preload (device int32 [n]) is given,
 * its first d_preload[i] positions are copied from the layer's host pool into
 * slots 0 .. d_preload[i]-1: slot s holds position s and the LRU order is the
 * empty slots then the preloaded ones -- the state that resolving positions
 * 0, 1, ... in order from the reset state gives.  Shared-index layers get the
 * bytes (their slots move with the anchor's).  An entry outside [0, R), or a
 * preload outside [0, min(B, P)], sets HISPARSE_ERR_RANGE and is skipped; a
 * request listed twice gives unspecified contents.  Graph-capturable; order
 * it between decode steps.  Errors: EINVAL, ECUDA. */
int hisparse_admit(hisparse_handle *h, int32_t layer, const int32_t *d_reqs, int32_t n,
                   const int32_t *d_preload, void *stream);

/* Write-through of the newest row ([DD] §3.4 step 4, §5.4 eager backup):
 * for r < *d_num_reqs with d_pos[r] >= 0, copy hot row B of (layer, r) to
 * host row d_pos[r] of (layer, r) (and of its HBM mirror, if it has one);
 * then, if d_new_rows is not NULL, place the new token's KV (d_new_rows,
 * device, [R][record_bytes] per layer, 16-byte aligned) in row B -- the old
 * row is always read before it is replaced.  d_new_rows is this library's
 * addition to the pages' write-back: the caller's new-token KV enters row B
 * in the same launch ([DD] §5.4 writes it to the newest slot separately).
 * layer == -1 does every layer in one launch (d_pos is then [L][R] and
 * d_new_rows [L][R][record_bytes]).  Positions >= P set HISPARSE_ERR_RANGE in
 * the status word and are not written back.  Make every resolve that may
 * fetch those rows wait for this launch (same stream or an event).
 * Errors: EINVAL, ECUDA. */
int hisparse_writeback(hisparse_handle *h, int32_t layer, const int32_t *d_pos,
                       const void *d_new_rows, const int32_t *d_num_reqs, void *stream);

/* Exact prefetch for a shared-index layer ([DD] §3.6, §5.6): copy, for
 * r < *d_num_reqs, every (position, slot) of the miss plan of the anchor's
 * last resolve (empty unless that resolve had HISPARSE_RECORD_PLAN) from the
 * follower's own host pool into the follower's hot buffer.  The
 * follower's slots stay in lockstep with the anchor's, so the anchor's d_out
 * rows are also the follower's.  Order it after the anchor's resolve (same
 * stream or an event) and before the anchor's next resolve.
 * follower_layer == -1 fills every shared-index layer of the anchor: one
 * launch per 8 such layers, each reading a plan record's rows for all its
 * layers back to back (with the group's layers interleaved in the host pool,
 * rows of one page).  The bytes written are the same as one call per layer.
 * An anchor without shared-index layers then launches nothing.
 * Errors: EINVAL (bad layer id), EROLE (anchor_layer is a shared-index
 * layer, or follower_layer is not one of its layers), ECUDA. */
int hisparse_prefetch_plan(hisparse_handle *h, int32_t anchor_layer, int32_t follower_layer,
                           const int32_t *d_num_reqs, void *stream);

/* (Library call, not a step of the pages' method.)
 * Copy `bytes` (a multiple of 16) from src to dst with SM threads, on
 * `stream`, after the stream's previous work (graph-capturable, no
 * synchronisation).  Either side may be device memory or pinned host memory
 * mapped for the device (hisparse_host_alloc, cudaHostAlloc); both 16-byte
 * aligned, not overlapping.  This is not part of the pages' method: it moves a
 * decode step's inputs and results between host and HBM over the coherent
 * host link with less latency than a copy engine for transfers of a few
 * hundred KB.  Errors: EINVAL (NULL, misaligned, bad size), ECUDA. */
int hisparse_copy(void *dst, const void *src, int64_t bytes, void *stream);

/* (Library call, not a step of the pages' method.)
 * Copy the per-request miss counts of one anchor layer's last resolve
 * (int32 [R]) to device memory d_dst, asynchronously on `stream` (no
 * synchronisation; graph-capturable).  Errors: EINVAL, EROLE, ECUDA. */
int hisparse_copy_miss_counts(hisparse_handle *h, int32_t layer, int32_t *d_dst, void *stream);

/* (Library call, not a step of the pages' method: how device-detected input
 * errors reach the host.)
 * Read and clear the sticky status word (bit-OR of HISPARSE_ERR_*), and copy
 * the per-unit codes of the last resolve ([L][R] int32, zero for followers)
 * if unit_err_out is not NULL.  Synchronises the device: not for use inside
 * a graph capture or a timed region. */
int hisparse_get_status(hisparse_handle *h, uint32_t *flags_out, int32_t *unit_err_out);

/* (Library call, not a step of the pages' method: checkpoint and test access
 * to the metadata of [DD] §5.2.)
 * Copy one anchor layer's state to host arrays (any may be NULL):
 * slot_pos [R][B] int32 (-1 empty), lru [R][B] int16 (least recent first),
 * page_table [R][P] int32 (slot, or -1 = host only), miss_counts [R] int32
 * (misses of the last resolve).  Synchronises.  Errors: EINVAL, EROLE, ECUDA. */
int hisparse_export_state(hisparse_handle *h, int32_t layer, int32_t *slot_pos, int16_t *lru,
                          int32_t *page_table, int32_t *miss_counts);

/* (Library call, not a step of the pages' method.)
 * Replace one anchor layer's state (checkpoint / test set-up): the arrays of
 * hisparse_export_state.  slot_pos, lru and page_table are required;
 * miss_counts may be NULL (the layer's miss counts are then left as they
 * are).  The arrays are validated first: every slot_pos in [-1, P) with no
 * position twice, lru a permutation of [0, B) per request, page_table[p] == s
 * exactly when slot_pos[s] == p, and every miss count in [0, k].  Nothing is
 * written unless all of it is valid.  Synchronises.
 * Errors: EINVAL, EROLE, ECUDA. */
int hisparse_import_state(hisparse_handle *h, int32_t layer, const int32_t *slot_pos,
                          const int16_t *lru, const int32_t *page_table,
                          const int32_t *miss_counts);

/* (Library call, not a step of the pages' method: host access to the plan of
 * [DD] §5.5.)
 * Copy one anchor layer's last miss plan to host arrays: count [R],
 * pos [R][k] int32, slot [R][k] int32 (only the first count[r] entries of a
 * row are meaningful).  Entries are the (position, slot) pairs fetched by the
 * last resolve: in list order with HISPARSE_LOOKUP_PAGE_TABLE, in ascending
 * position with HISPARSE_LOOKUP_HASH.  Synchronises.
 * Errors: EINVAL, EROLE, ECUDA. */
int hisparse_export_plan(hisparse_handle *h, int32_t layer, int32_t *count, int32_t *pos,
                         int32_t *slot);

/* Reset one anchor layer (or all layers with layer == -1) to the admission
 * state: slots empty, LRU 0..B-1, page table all host-only ([DD] §5.4
 * request release).  Asynchronous on `stream` (the stream argument is this
 * library's: a reset is ordered with the launches around it, and can be
 * captured in a graph).  Errors: EINVAL, EROLE, ECUDA. */
int hisparse_reset(hisparse_handle *h, int32_t layer, void *stream);

/* Keep the page tables of the layers that run RESOLVE in L2 between decode
 * steps (build-own call; the pages keep their slot lookup in shared memory
 * and have no counterpart).  RESOLVE with HISPARSE_LOOKUP_PAGE_TABLE gathers
 * one page-table entry per selection right after reading the selections;
 * when the rest of a decode step has evicted that table from L2 the gather
 * costs a DRAM round trip on the critical path.  With bytes > 0 this sets the
 * calling process's persisting-L2 set-aside (cudaLimitPersistingL2CacheSize,
 * a limit of this CUDA context that ends with it) to min(bytes, the device
 * maximum), and every later page-table RESOLVE launch carries an
 * access-policy window over its layer's page table whose hit ratio lets the
 * tables of all RESOLVE layers share the set-aside.  bytes == 0 turns it off:
 * persisting lines go back to normal (cudaCtxResetPersistingL2Cache) and the
 * set-aside to what it was before this handle first changed it;
 * hisparse_destroy does the same.
 * Results are unchanged either way.  Not during graph capture: launches
 * captured earlier keep the setting they were captured with.
 * Errors: EINVAL (bytes < 0), EBOUND (no persisting L2 on the device, or one
 * layer's table larger than an access-policy window), ECUDA. */
int hisparse_set_l2_persisting(hisparse_handle *h, int64_t bytes);

/* (Library call.)  Fill `out` with facts about the instance. */
int hisparse_get_info(const hisparse_handle *h, hisparse_info *out);

/* (Library calls, not steps of the pages' method: the pages assume a pinned
 * host pool, [DD] §3.2; these allocate one without rounding.)
 * Pinned, device-mapped, portable host memory for host pools: the PINNED kind
 * below (cudaHostAlloc; contents unspecified).  Free with hisparse_host_free.
 * Errors: EINVAL, ENOMEM. */
int hisparse_host_alloc(size_t bytes, void **out);
int hisparse_host_free(void *p);

/* Host-pool kinds for hisparse_host_alloc_kind. */
#define HISPARSE_HOST_HUGE 0   /* transparent-huge-page backed, cudaHostRegister'ed */
#define HISPARSE_HOST_PINNED 1 /* cudaHostAlloc: driver-pinned base pages (the default) */

/* hisparse_host_alloc with an explicit kind.
 * PINNED: driver-allocated pinned memory.  It is never split or migrated; the
 *   GPU pays one translation miss per first-touched 64 KB page, after which
 *   random record fetches run at the host-link rate.
 * HUGE: huge-page-advised memory (zero-filled, size rounded up to whole huge
 *   pages) registered with cudaHostRegister, excluded from fork() children
 *   (MADV_DONTFORK).  The GPU translates it with few, large pages.  On a host
 *   whose GPU driver migrates GPU-hot host pages (ATS access-counter
 *   migration), huge pages can be split under the pool while it is in use and
 *   GPU fetches then stall in fault service for up to milliseconds; the
 *   operator-side remedy is to disable that migration in the driver.  A
 *   request smaller than one huge page, or a refused registration, falls back
 *   to PINNED.
 * Errors: EINVAL, ENOMEM. */
int hisparse_host_alloc_kind(size_t bytes, int32_t kind, void **out);

/* Bytes of [p, p + bytes) that the host kernel backs with transparent huge
 * pages (from /proc/self/smaps; whole mappings that overlap the range are
 * counted, capped at `bytes`).  A pool with few huge pages still works but
 * costs the GPU more address-translation work per fetched record.
 * Errors: EINVAL. */
int hisparse_host_hugepage_bytes(const void *p, size_t bytes, size_t *huge_out);

/* (Library calls.)
 * The cudaError_t of the last failed CUDA call made by this thread through
 * the library (0 if none), and a static message for any return code. */
int hisparse_last_cuda_error(void);
const char *hisparse_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* HISPARSE_H */
