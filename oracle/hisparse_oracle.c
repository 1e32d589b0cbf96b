/*
 * Plain single-threaded C model of the HiSparse RESOLVE step.
 * TEST INFRASTRUCTURE ONLY: built and called by tests/, by the smoke check and
 * by the CPU-baseline leg of bench.py.  It shares no code, header or constant
 * table with the CUDA library; it defines everything it needs here.
 *
 * What it computes (one unit = one (request, layer) pair; units independent):
 *   gentlecold.top "HiSparse 深度解析" (HiSparse deep dive):
 *     §3.2  two-level hierarchy; page table pos -> slot or host-only
 *     §3.3  per-(request, layer) LRU; this step's hits rank as more recent than
 *           this step's new misses
 *     §3.4  write-through of the newest token to the host pool
 *     §3.5  the five RESOLVE stages and the worked example (B=8, k=4)
 *     §3.6  exact cross-layer prefetch: shared layers replay the anchor's plan
 *     §5.2  newest token in an extra row B outside the LRU
 *     §5.5  miss plan (pos, slot) recorded where the eviction is decided
 * Readings where the pages are open (same as the Python model in tiny.py):
 *   hits of one step ordered by ascending slot; misses take the oldest
 *   evictables in selection-list order; -1 is padding; a duplicate or
 *   out-of-range position fails the unit with its state untouched and an
 *   output row of -1; the newest-token binding is a hit, not a miss.
 *
 * The page table is a direct-address table over [0, P) (-1 = host-only), which
 * is the plainest dictionary for integer keys in a known range.
 *
 * Three-tier resolve (docs.vllm.ai "HiSparse local KV offload architecture",
 * "Hot lookup and LRU"; gentlecold.top §6.5): with a resident block table, a
 * position whose block has a device-resident copy resolves to that copy first
 * (output B + 1 + row, row = entry * block_tokens + offset in the block) and
 * is neither a hit nor a miss.  A block entry below -1, or a row whose output
 * does not fit int32, fails the unit like an out-of-range position.  The
 * duplicate check covers positions that reach the hot tier only (a resident
 * position never touches the cache; the pages exit before the hash table).
 *
 * Union mode (speculative verification, gentlecold.top §6.5: one block
 * resolves the union of all verify rows' top-k, misses in (row, top-k)
 * first-reference order): the rows come as one list; a repeated position is
 * resolved at its first reference and later references output the same row.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <limits.h>

#define HSO_ERR_RANGE 1
#define HSO_ERR_DUP 2

/* One layer's state for R requests.  Arrays are owned by the caller. */
typedef struct {
  int32_t R, k, B;
  int64_t P;                 /* host rows (logical positions) per unit */
  int32_t rec;               /* record bytes */
  int32_t *slot_pos;         /* [R][B]  logical position in each slot, -1 empty */
  int16_t *lru;              /* [R][B]  slot ids, oldest first */
  int32_t *page_table;       /* [R][P]  slot of each position, -1 host-only */
  int32_t *miss_count;       /* [R] */
  int32_t *unit_err;         /* [R] */
  uint8_t *hot;              /* [R][B+1][rec] or NULL: metadata only */
  /* host pool: rows [0, host_split) read from `host` (shared, read-only);
     rows [host_split, P) live in `host_tail`, which this model owns and
     updates on write-back. */
  const uint8_t *host;       /* row (r, p) at host + r*host_req_stride + p*host_row_stride */
  int64_t host_req_stride;
  int64_t host_split;
  uint8_t *host_tail;        /* [R][P - host_split][rec] or NULL */
  int32_t *plan_pos;         /* [R][k] */
  int32_t *plan_slot;        /* [R][k] */
  int32_t *plan_count;       /* [R] */
  int32_t *mark;             /* [P] scratch for duplicate detection */
  int32_t mark_gen;
  uint8_t *hit;              /* [B] scratch */
  int32_t *misses;           /* [k] scratch */
  int16_t *ev;               /* [B] scratch */
  int32_t *first;            /* [P] scratch: first list index of each position */
  int64_t host_row_stride;   /* bytes between consecutive host rows (0: rec) */
} hso_layer;

static const uint8_t *host_row(const hso_layer *L, int32_t r, int64_t p) {
  if (p < L->host_split)
    return L->host + (int64_t)r * L->host_req_stride +
           p * (L->host_row_stride ? L->host_row_stride : (int64_t)L->rec);
  return L->host_tail + ((int64_t)r * (L->P - L->host_split) + (p - L->host_split)) * (int64_t)L->rec;
}

/* Reset one unit to its admission state: every slot empty, LRU 0..B-1. */
void hso_reset_unit(hso_layer *L, int32_t r) {
  int32_t s;
  int64_t p;
  for (s = 0; s < L->B; s++) {
    L->slot_pos[(int64_t)r * L->B + s] = -1;
    L->lru[(int64_t)r * L->B + s] = (int16_t)s;
  }
  for (p = 0; p < L->P; p++) L->page_table[(int64_t)r * L->P + p] = -1;
  L->miss_count[r] = 0;
  L->unit_err[r] = 0;
  L->plan_count[r] = 0;
}

/* Resident row of position p for one request's block table `blk` ([nblk],
   entries -1 = not resident), -1 if not resident, -2 if the entry or the row
   is invalid. */
static int64_t resident_row(const hso_layer *L, const int32_t *blk, int32_t nblk, int32_t tok,
                            int32_t p) {
  int64_t b, e, row;
  if (!blk) return -1;
  b = p / tok;
  if (b >= nblk) return -1;
  e = blk[b];
  if (e == -1) return -1;
  if (e < -1) return -2;
  row = e * tok + p % tok;
  if ((int64_t)L->B + 1 + row > INT32_MAX) return -2;
  return row;
}

/* RESOLVE for unit (r) of this layer.  sel: [k]; out: [k].
   io: 1 = copy missed records from the host pool into the hot rows,
       0 = metadata only (the pages' no-IO mode: bytes left stale).
   blk / nblk / tok: this request's resident block table (NULL: none).
   Returns 0 or a bit-OR of HSO_ERR_*. */
int32_t hso_resolve_unit_res(hso_layer *L, int32_t r, const int32_t *sel, int32_t newest,
                             int32_t io, const int32_t *blk, int32_t nblk, int32_t tok,
                             int32_t union_mode, int32_t *out) {
  const int32_t B = L->B, k = L->k;
  const int64_t P = L->P;
  int32_t *slot_pos = L->slot_pos + (int64_t)r * B;
  int16_t *lru = L->lru + (int64_t)r * B;
  int32_t *pt = L->page_table + (int64_t)r * P;
  int32_t *plan_pos = L->plan_pos + (int64_t)r * k;
  int32_t *plan_slot = L->plan_slot + (int64_t)r * k;
  int32_t err = 0, i, j, s, M = 0, E = 0, n = 0;
  int64_t rr;

  /* validation */
  L->mark_gen++;
  for (i = 0; i < k; i++) {
    int32_t p = sel[i];
    if (p == -1) continue;
    if (p < -1 || (int64_t)p >= P) { err |= HSO_ERR_RANGE; continue; }
    rr = resident_row(L, blk, nblk, tok, p);
    if (rr == -2) { err |= HSO_ERR_RANGE; continue; }
    if (rr >= 0) continue; /* resident: never reaches the hot tier */
    if (L->mark[p] == L->mark_gen) {
      if (!union_mode) err |= HSO_ERR_DUP;
    } else {
      L->mark[p] = L->mark_gen;
      L->first[p] = i;
    }
  }
  if (newest < -1 || (int64_t)newest >= P) err |= HSO_ERR_RANGE;
  L->unit_err[r] = err;
  if (err) {
    for (i = 0; i < k; i++) out[i] = -1;
    L->miss_count[r] = 0;
    L->plan_count[r] = 0;
    return err;
  }

  /* stages 1-2: classify */
  memset(L->hit, 0, (size_t)B);
  for (i = 0; i < k; i++) {
    int32_t p = sel[i];
    if (p == -1) {
      out[i] = -1;
    } else if (resident_row(L, blk, nblk, tok, p) >= 0) {
      out[i] = (int32_t)(L->B + 1 + resident_row(L, blk, nblk, tok, p));
    } else if (union_mode && L->first[p] != i) {
      out[i] = INT32_MIN; /* a later reference: its first's row, below */
    } else if (newest >= 0 && p == newest) {
      out[i] = B;
    } else if (pt[p] >= 0) {
      out[i] = pt[p];
      L->hit[pt[p]] = 1;
    } else {
      L->misses[M++] = i;
    }
  }

  /* stage 3: evictables in LRU order */
  for (j = 0; j < B; j++)
    if (!L->hit[lru[j]]) L->ev[E++] = lru[j];
  /* B >= k guarantees M <= E (checked at set-up by the caller) */

  /* stages 4-5: victims, fetch, publish, plan */
  for (j = 0; j < M; j++) {
    int32_t p, old;
    s = L->ev[j];
    p = sel[L->misses[j]];
    old = slot_pos[s];
    if (old >= 0) pt[old] = -1;
    slot_pos[s] = p;
    pt[p] = s;
    if (io && L->hot)
      memcpy(L->hot + ((int64_t)r * (B + 1) + s) * (int64_t)L->rec, host_row(L, r, p), (size_t)L->rec);
    out[L->misses[j]] = s;
    plan_pos[j] = p;
    plan_slot[j] = s;
  }

  if (union_mode)
    for (i = 0; i < k; i++)
      if (out[i] == INT32_MIN) out[i] = out[L->first[sel[i]]];

  /* new LRU: remaining evictables, then this step's fetches, then hits */
  for (j = M; j < E; j++) lru[n++] = L->ev[j];
  for (j = 0; j < M; j++) lru[n++] = L->ev[j];
  for (s = 0; s < B; s++)
    if (L->hit[s]) lru[n++] = (int16_t)s;

  L->miss_count[r] = M;
  L->plan_count[r] = M;
  return 0;
}

int32_t hso_resolve_unit(hso_layer *L, int32_t r, const int32_t *sel, int32_t newest,
                         int32_t io, int32_t *out) {
  return hso_resolve_unit_res(L, r, sel, newest, io, NULL, 0, 1, 0, out);
}

/* One layer-step over requests [0, num_reqs): sel [R][k], newest [R] or NULL,
   res_blocks [R][nblk] or NULL, out [R][k].  Returns the bit-OR of the units'
   errors. */
int32_t hso_resolve_layer_res(hso_layer *L, const int32_t *sel, const int32_t *newest,
                              const int32_t *res_blocks, int32_t nblk, int32_t tok,
                              int32_t union_mode, int32_t num_reqs, int32_t io, int32_t *out) {
  int32_t r, e = 0;
  for (r = 0; r < num_reqs; r++)
    e |= hso_resolve_unit_res(L, r, sel + (int64_t)r * L->k, newest ? newest[r] : -1, io,
                              res_blocks ? res_blocks + (int64_t)r * nblk : NULL, nblk, tok,
                              union_mode, out + (int64_t)r * L->k);
  return e;
}

int32_t hso_resolve_layer(hso_layer *L, const int32_t *sel, const int32_t *newest,
                          int32_t num_reqs, int32_t io, int32_t *out) {
  return hso_resolve_layer_res(L, sel, newest, NULL, 0, 1, 0, num_reqs, io, out);
}

/* Short-sequence lookup (gentlecold.top §5.4 and §5.5: when a request's
   seq_len <= B its tokens sit in the buffer in order, and the kernel returns
   each selection's slot by position, with no host IO and no LRU work).
   Reading R17: for request r with seq_len <= B, a selection outputs -1 for
   padding, its resident row first when the resident table has one (as in
   the three-tier resolve), B for the newest token, else the slot numbered
   like the position.  A position outside [0, seq_len) or [0, P), a newest
   position outside [-1, P) or an invalid resident entry fails the request
   (out all -1); repeats are not checked (nothing is allocated).  Nothing of
   the unit's state changes here; the growth of the buffer by the previous
   token is a one-entry resolve the caller runs before (see tiny.py).
   Returns 0 or a bit-OR of HSO_ERR_*; sets unit_err[r]. */
int32_t hso_short_lookup_unit(hso_layer *L, int32_t r, const int32_t *sel, int32_t newest,
                              int32_t seq_len, const int32_t *blk, int32_t nblk, int32_t tok,
                              int32_t *out) {
  int32_t err = 0, i;
  int64_t rr;
  if (newest < -1 || (int64_t)newest >= L->P) err |= HSO_ERR_RANGE;
  for (i = 0; i < L->k; i++) {
    int32_t p = sel[i];
    if (p == -1) { out[i] = -1; continue; }
    if (p < -1 || (int64_t)p >= L->P) { err |= HSO_ERR_RANGE; continue; }
    rr = resident_row(L, blk, nblk, tok, p);
    if (rr == -2) { err |= HSO_ERR_RANGE; continue; }
    if (rr >= 0) { out[i] = (int32_t)(L->B + 1 + rr); continue; }
    if (newest >= 0 && p == newest) { out[i] = L->B; continue; }
    if (p >= seq_len) { err |= HSO_ERR_RANGE; continue; }
    out[i] = p;
  }
  if (err)
    for (i = 0; i < L->k; i++) out[i] = -1;
  L->unit_err[r] = err;
  return err;
}

/* The caller writes the new token's KV into row B of each request. */
void hso_set_newest_rows(hso_layer *L, const uint8_t *rows /* [R][rec] */, int32_t num_reqs) {
  int32_t r;
  for (r = 0; r < num_reqs; r++)
    memcpy(L->hot + ((int64_t)r * (L->B + 1) + L->B) * (int64_t)L->rec,
           rows + (int64_t)r * L->rec, (size_t)L->rec);
}

/* Write-through: host[r][pos[r]] <- hot[r][B] for pos[r] >= 0.
   Only rows in the model-owned tail can be written.  Returns -1 if a position
   falls outside [host_split, P), else 0. */
int32_t hso_writeback(hso_layer *L, const int32_t *pos, int32_t num_reqs) {
  int32_t r;
  for (r = 0; r < num_reqs; r++) {
    int64_t p = pos[r];
    if (p < 0) continue;
    if (p < L->host_split || p >= L->P) return -1;
    memcpy(L->host_tail + ((int64_t)r * (L->P - L->host_split) + (p - L->host_split)) * (int64_t)L->rec,
           L->hot + ((int64_t)r * (L->B + 1) + L->B) * (int64_t)L->rec, (size_t)L->rec);
  }
  return 0;
}

/* Plan replay into a shared layer: follower_hot[r][s] <- follower host row p
   for every (p, s) of the anchor's last plan.  `F` describes the follower's
   bytes (its hot rows and host pool); its metadata arrays are not used. */
void hso_replay(const hso_layer *anchor, hso_layer *F, int32_t num_reqs) {
  int32_t r, j;
  for (r = 0; r < num_reqs; r++) {
    const int32_t *pp = anchor->plan_pos + (int64_t)r * anchor->k;
    const int32_t *ps = anchor->plan_slot + (int64_t)r * anchor->k;
    for (j = 0; j < anchor->plan_count[r]; j++)
      memcpy(F->hot + ((int64_t)r * (F->B + 1) + ps[j]) * (int64_t)F->rec, host_row(F, r, pp[j]),
             (size_t)F->rec);
  }
}
