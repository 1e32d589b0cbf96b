/*
 * Seeded synthetic KV records (input generation only; no cache arithmetic).
 *
 * Record (layer, req, pos) is rec_bytes of bf16 values.  Each 8-byte word w of
 * the record is four bf16 values looked up in a 65536-entry table of standard
 * normal quantiles with four 16-bit fields of one SplitMix64 output:
 *
 *   counter c = ((((layer << 16) | req) << 24 | pos) << 12) | w
 *   x = splitmix64 output number c of the stream seeded with `seed`
 *     = mix(seed + (c + 1) * 0x9E3779B97F4A7C15)
 *   values = table[x & 0xFFFF], table[(x >> 16) & 0xFFFF], ...
 *
 * SplitMix64 is Steele, Lea and Flood's generator (OOPSLA 2014, "Fast
 * splittable pseudorandom number generators"); `mix` is its finaliser.
 * The caller builds the table (bf16 bits of the normal quantile at
 * (u + 0.5) / 65536) so the values are N(0,1) to 16-bit resolution.
 * Limits: layer < 256, req < 65536, pos < 2^24, rec_bytes <= 32768.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

typedef struct {
  uint8_t *dst;
  int64_t n_rows, row_stride, pos0;
  int32_t rec_bytes, layer, req;
  uint64_t seed;
  const uint16_t *table;
  int64_t row_begin, row_end;
} job_t;

static void fill_rows(const job_t *j) {
  int64_t i;
  const int32_t words = j->rec_bytes / 8;
  for (i = j->row_begin; i < j->row_end; i++) {
    uint16_t *out = (uint16_t *)(j->dst + i * j->row_stride);
    uint64_t pos = (uint64_t)(j->pos0 + i);
    uint64_t base = ((((uint64_t)j->layer << 16) | (uint64_t)j->req) << 24 | pos) << 12;
    int32_t w;
    for (w = 0; w < words; w++) {
      uint64_t x = sm64_mix(j->seed + (base + (uint64_t)w + 1ull) * 0x9E3779B97F4A7C15ull);
      out[4 * w + 0] = j->table[x & 0xFFFF];
      out[4 * w + 1] = j->table[(x >> 16) & 0xFFFF];
      out[4 * w + 2] = j->table[(x >> 32) & 0xFFFF];
      out[4 * w + 3] = j->table[(x >> 48) & 0xFFFF];
    }
  }
}

static void *worker(void *arg) {
  fill_rows((const job_t *)arg);
  return 0;
}

/* Fill n_rows records for positions pos0 .. pos0+n_rows-1 of unit
   (layer, req); row i starts at dst + i*row_stride.  Returns 0, or -1 on a
   bad argument. */
int32_t wl_fill_records(uint8_t *dst, int64_t n_rows, int64_t row_stride, int32_t rec_bytes,
                        uint64_t seed, int32_t layer, int32_t req, int64_t pos0,
                        const uint16_t *table, int32_t nthreads) {
  job_t jobs[64];
  pthread_t th[64];
  int32_t started[64];
  int32_t t;
  if (rec_bytes <= 0 || rec_bytes % 8 || rec_bytes > 32768 || layer < 0 || layer > 255 ||
      req < 0 || req > 65535 || pos0 < 0 || n_rows < 0 || pos0 + n_rows > (1ll << 24))
    return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n_rows < 4096) nthreads = 1;
  for (t = 0; t < nthreads; t++) {
    jobs[t].dst = dst;
    jobs[t].n_rows = n_rows;
    jobs[t].row_stride = row_stride;
    jobs[t].pos0 = pos0;
    jobs[t].rec_bytes = rec_bytes;
    jobs[t].layer = layer;
    jobs[t].req = req;
    jobs[t].seed = seed;
    jobs[t].table = table;
    jobs[t].row_begin = n_rows * t / nthreads;
    jobs[t].row_end = n_rows * (t + 1) / nthreads;
  }
  for (t = 1; t < nthreads; t++) {
    started[t] = pthread_create(&th[t], 0, worker, &jobs[t]) == 0;
    if (!started[t]) fill_rows(&jobs[t]);
  }
  fill_rows(&jobs[0]);
  for (t = 1; t < nthreads; t++)
    if (started[t]) pthread_join(th[t], 0);
  return 0;
}

/* Fill rows for an explicit list of positions (used for new-token records). */
int32_t wl_fill_positions(uint8_t *dst, int64_t row_stride, int32_t rec_bytes, uint64_t seed,
                          int32_t layer, int32_t req, const int64_t *pos, int64_t n,
                          const uint16_t *table) {
  int64_t i;
  for (i = 0; i < n; i++) {
    int32_t e = wl_fill_records(dst + i * row_stride, 1, row_stride, rec_bytes, seed, layer, req,
                                pos[i], table, 1);
    if (e) return e;
  }
  return 0;
}
