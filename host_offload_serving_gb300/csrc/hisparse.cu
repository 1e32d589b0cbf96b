// hisparse.cu -- RESOLVE, write-through and plan-replay kernels for GB300
// (sm_103a), and the C ABI declared in include/hisparse.h.
//
// Pages (cited by title and section):
//   [DD] gentlecold.top, "HiSparse 深度解析：论文、SGLang 实现与 vLLM Hybrid
//        HiSparse": §3.3 replacement policy, §3.4 write-through, §3.5 the five
//        RESOLVE stages and the worked example, §3.6 exact prefetch, §5.2
//        newest slot, §5.5 swap-in kernel (num_real_reqs, miss plan, one warp
//        per miss, 16-byte non-coherent loads), §5.6 copy-only replay kernel.
//   [VD] docs.vllm.ai, "HiSparse local KV offload architecture":
//        "Hot lookup and LRU", "Performance invariants".
//
// Kernels:
//   resolve_pt_kernel (default, HISPARSE_LOOKUP_PAGE_TABLE): one thread-block
//     CLUSTER per request.  Worker CTAs classify slices of the selection list
//     through the published page table and issue the host loads of their
//     first missed records into registers before any victim is known; the
//     leader CTA merges the slices through distributed shared memory, checks
//     duplicates, picks victims and the new LRU order, writes each worker's
//     victims into that worker's shared memory, and publishes.  Two hardware
//     cluster barriers, no spin-waits.  The write-through of the previous
//     token is fused in; the launch uses programmatic dependent launch.  A
//     second instantiation adds the resident tier, block-id selections and
//     the union of speculative verify rows.  With HISPARSE_WITH_SHARED the
//     workers also fill the anchor's shared-index layers at the same slots.
//   resolve_kernel (HISPARSE_LOOKUP_HASH): the pages' stage order (hash
//     staging, mark, scans, fetch by the whole cluster), kept as an ablation.
//   replay_kernel: plan replay into one or several shared-index layers of an
//     anchor (a record's rows for all of them back to back).
//   writeback_kernel, admit_kernel, reset_kernel, copy_kernel: the separate
//     write-through, admission with preload, the reset state, and copies by
//     SM threads between pinned host memory and HBM.
// Common to the fetches: the misses of a request are one flat run of 16-byte
// chunks (miss j, chunk o), so no lane idles on records that are not a
// multiple of 512 bytes (1152-byte records are 72 chunks), read with
// non-coherent 16-byte loads from mapped pinned host memory.
#include <cuda_runtime.h>
#include <sys/mman.h>

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "hisparse.h"

namespace {

constexpr int kThreads = 1024;            // threads per resolve CTA
constexpr int kWarps = kThreads / 32;     // == 32: one warp total per lane
constexpr int kUnroll = 4;                // 16-byte loads in flight per thread
constexpr int32_t kUnresolved = INT32_MIN;
constexpr uint32_t kAlias = 1u << 30;  // a victim entry of a repeated miss (union mode): not fetched
constexpr unsigned kFull = 0xffffffffu;
static_assert(kWarps == 32, "warp-total scan assumes 32 warps");

thread_local int g_last_cuda_error = 0;

// ---------------------------------------------------------------------------
// Shared-memory layout of a resolve CTA (identical on host and device).
// ---------------------------------------------------------------------------
struct SmemLayout {
  uint32_t key, val, sel, out, slotpos, hit, lru, newlru, missidx, victim, bkt, misc, total;
};

constexpr int kMaxBuckets = 2048;   // host-row buckets used to order the fetches

__host__ __device__ inline uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ inline SmemLayout smem_layout(int k, int B, int cap) {
  SmemLayout L;
  uint32_t o = 0;
  L.key = o;     o += align16(4u * cap);   // hash keys; later the fetch positions
  L.val = o;     o += align16(2u * cap);   // hash values (selection index); later fetch slots
  L.sel = o;     o += align16(4u * k);
  L.out = o;     o += align16(4u * k);
  L.slotpos = o; o += align16(4u * B);
  L.hit = o;     o += align16(1u * B);
  L.lru = o;     o += align16(2u * B);
  L.newlru = o;  o += align16(2u * B);
  L.missidx = o; o += align16(2u * k);
  L.victim = o;  o += align16(2u * k);
  L.bkt = o;     o += align16(4u * kMaxBuckets);
  L.misc = o;    o += align16(4u * (8 + 3 * kWarps));
  L.total = o;
  return L;
}

// misc words
enum { kMiscErr = 0, kMiscM = 1 };

// ---------------------------------------------------------------------------
// Kernel arguments
// ---------------------------------------------------------------------------
struct ResolveArgs {
  int32_t R, k, B, cap_log2, rec16, io;
  int32_t vec;                 // 1: sel, slot_pos and lru rows are 16-byte aligned
  int32_t bucket_shift, nbuckets;
  int64_t P;
  const int32_t *sel, *num_reqs, *newest;
  int32_t *out;
  int32_t *slot_pos;
  int16_t *lru;
  int32_t *page_table, *miss_count, *unit_err;
  uint32_t *status;
  int32_t *plan_pos, *plan_slot, *plan_count;
  const char *src;             // host pool (device-visible address) or HBM mirror
  int64_t src_req_stride, src_row_stride;
  char *hot;
  int64_t hot_req_stride, hot_row_stride;
};

struct LayerDev {              // one layer's buffers, device-visible addresses
  const char *host;            // host pool
  char *host_w;                // same, writable
  int64_t host_req_stride, host_row_stride;
  char *hot;
  int64_t hot_req_stride, hot_row_stride;
  char *mirror;                // HBM mirror of the host pool (same strides) or null;
                               // every write-back stores to it as well
};

struct WritebackArgs {
  const LayerDev *layers;      // device array [L]
  int32_t layer0, R, B, rec16;
  int64_t P;
  const int32_t *pos;          // [nl][R]
  const char *new_rows;        // [nl][R][rec16 * 16] or null
  const int32_t *num_reqs;
  uint32_t *status;
};

// One shared-index layer a replay fills: its host pool and hot buffer.
struct ReplayTarget {
  const char *src;
  int64_t src_req_stride, src_row_stride;
  char *hot;
  int64_t hot_req_stride, hot_row_stride;
};
constexpr int kMaxReplayTargets = 8;  // shared-index layers one replay launch fills
struct ReplayArgs {
  int32_t R, k, rec16, nf;
  const int32_t *num_reqs;
  const int32_t *plan_pos, *plan_slot, *plan_count;
  ReplayTarget f[kMaxReplayTargets];  // nf of them
};

// ---------------------------------------------------------------------------
// PTX helpers: cluster barrier, cluster rank, distributed shared memory,
// non-coherent 16-byte loads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of `p` (this CTA's shared memory) in the shared window of CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
  uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_dsmem_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// 16-byte load through the non-coherent path ([DD] §5.5: GPU threads read
// pinned host memory directly with vectorised non-coherent loads).
__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_v4(void *p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Knuth's multiplicative hash into a table of 2^cap_log2 entries ([DD] §3.5
// stage 1).
__device__ __forceinline__ uint32_t hash_pos(int32_t p, int cap_log2) {
  return (static_cast<uint32_t>(p) * 2654435761u) >> (32 - cap_log2);
}

// Exclusive prefix sum of a[0..n), n <= 2 * kThreads, in place (all threads).
__device__ __forceinline__ void block_exclusive_scan(int32_t *a, int n, int32_t *warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 2 * tid;
  const int v0 = i0 < n ? a[i0] : 0, v1 = i0 + 1 < n ? a[i0 + 1] : 0;
  const int sum = v0 + v1;
  int inc = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(kFull, inc, d);
    if (lane >= d) inc += t;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  const int wt = warp_tot[lane];
  int winc = wt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(kFull, winc, d);
    if (lane >= d) winc += t;
  }
  const int excl = __shfl_sync(kFull, winc - wt, warp) + inc - sum;
  __syncthreads();
  if (i0 < n) a[i0] = excl;
  if (i0 + 1 < n) a[i0 + 1] = excl + v0;
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Leader CTA: stages 1, 2, 3 and 5 for request r.  On return (after a block
// barrier) misc[kMiscM] holds the number of misses M and, for j < M,
// fpos[j] / fslot[j] hold the position and victim slot of miss j.
// ---------------------------------------------------------------------------
template <bool kRecordPlan>
__device__ bool leader_resolve(const ResolveArgs &a, int r, unsigned char *smem,
                               const SmemLayout &L) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, B = a.B, cap = 1 << a.cap_log2;
  const int64_t P = a.P;
  int32_t *s_key = reinterpret_cast<int32_t *>(smem + L.key);
  int16_t *s_val = reinterpret_cast<int16_t *>(smem + L.val);
  int32_t *s_sel = reinterpret_cast<int32_t *>(smem + L.sel);
  int32_t *s_out = reinterpret_cast<int32_t *>(smem + L.out);
  int32_t *s_slotpos = reinterpret_cast<int32_t *>(smem + L.slotpos);
  uint8_t *s_hit = reinterpret_cast<uint8_t *>(smem + L.hit);
  int16_t *s_lru = reinterpret_cast<int16_t *>(smem + L.lru);
  int16_t *s_newlru = reinterpret_cast<int16_t *>(smem + L.newlru);
  int16_t *s_missidx = reinterpret_cast<int16_t *>(smem + L.missidx);
  int16_t *s_victim = reinterpret_cast<int16_t *>(smem + L.victim);
  uint32_t *s_misc = reinterpret_cast<uint32_t *>(smem + L.misc);
  int32_t *s_cnt = reinterpret_cast<int32_t *>(s_misc + 8);  // [3][32]
  int32_t *s_fpos = s_key;                                   // reused after stage 2
  int16_t *s_fslot = s_val;

  const int32_t *g_sel = a.sel + static_cast<int64_t>(r) * k;
  int32_t *g_slotpos = a.slot_pos + static_cast<int64_t>(r) * B;
  int16_t *g_lru = a.lru + static_cast<int64_t>(r) * B;
  int32_t *g_pt = a.page_table + static_cast<int64_t>(r) * P;

  // ---- stage 0: issue every global load of the unit at once (one memory
  //      round trip), then stage them in shared memory ----
  const int nreq = a.num_reqs ? min(*a.num_reqs, a.R) : a.R;
  const int32_t newest = a.newest ? a.newest[r] : -1;
  constexpr int kV = 2;  // 16-byte vectors per thread and array in the batched path
  int4 vs[kV], vp[kV];
  uint4 vl[kV];
  const int nk4 = a.vec ? k / 4 : 0, nb4 = a.vec ? B / 4 : 0, nb8 = a.vec ? B / 8 : 0;
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    const int i = tid + u * kThreads;
    if (i < nk4) vs[u] = reinterpret_cast<const int4 *>(g_sel)[i];
    if (i < nb4) vp[u] = reinterpret_cast<const int4 *>(g_slotpos)[i];
    if (i < nb8) vl[u] = reinterpret_cast<const uint4 *>(g_lru)[i];
  }
  if (r >= nreq) return false;  // graph padding: the whole cluster leaves together
  for (int i = tid; i < cap; i += kThreads) s_key[i] = -1;
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    const int i = tid + u * kThreads;
    if (i < nk4) reinterpret_cast<int4 *>(s_sel)[i] = vs[u];
    if (i < nb4) reinterpret_cast<int4 *>(s_slotpos)[i] = vp[u];
    if (i < nb8) reinterpret_cast<uint4 *>(s_lru)[i] = vl[u];
  }
  // whatever the batched path did not cover (unaligned rows or large k, B)
  for (int i = 4 * min(nk4, kV * kThreads) + tid; i < k; i += kThreads) s_sel[i] = g_sel[i];
  for (int s = 4 * min(nb4, kV * kThreads) + tid; s < B; s += kThreads) s_slotpos[s] = g_slotpos[s];
  for (int s = 8 * min(nb8, kV * kThreads) + tid; s < B; s += kThreads) s_lru[s] = g_lru[s];
  if (tid == 0) s_misc[kMiscErr] = (newest < -1 || newest >= P) ? HISPARSE_ERR_RANGE : 0u;
  __syncthreads();

  // ---- stage 1: stage the selection in the hash, validate ----
  for (int i = tid; i < k; i += kThreads) {
    const int32_t p = s_sel[i];
    int32_t o = -1;
    if (p != -1) {
      if (p < -1 || p >= P) {
        atomicOr(&s_misc[kMiscErr], HISPARSE_ERR_RANGE);
      } else {
        o = (p == newest) ? B : kUnresolved;
        uint32_t h = hash_pos(p, a.cap_log2);
        for (int probe = 0; probe < cap; ++probe) {
          const int32_t prev = atomicCAS(&s_key[h], -1, p);
          if (prev == -1) {
            s_val[h] = static_cast<int16_t>(i);
            break;
          }
          if (prev == p) {
            atomicOr(&s_misc[kMiscErr], HISPARSE_ERR_DUP);
            break;
          }
          h = (h + 1) & (cap - 1);
        }
      }
    }
    s_out[i] = o;
  }
  __syncthreads();

  const uint32_t err = s_misc[kMiscErr];
  if (err) {  // uniform: the unit keeps its state, its out row is all -1
    for (int i = tid; i < k; i += kThreads) a.out[static_cast<int64_t>(r) * k + i] = -1;
    if (tid == 0) {
      a.unit_err[r] = static_cast<int32_t>(err);
      atomicOr(a.status, err);
      a.miss_count[r] = 0;
      a.plan_count[r] = 0;
      s_misc[kMiscM] = 0;
    }
    __syncthreads();
    return true;
  }

  // ---- stage 2: mark each slot hit or evictable ----
  for (int s = tid; s < B; s += kThreads) {
    const int32_t p = s_slotpos[s];
    uint8_t hit = 0;
    if (p >= 0 && p != newest) {
      uint32_t h = hash_pos(p, a.cap_log2);
      for (int probe = 0; probe < cap; ++probe) {
        const int32_t key = s_key[h];
        if (key == p) {
          s_out[s_val[h]] = s;
          hit = 1;
          break;
        }
        if (key == -1) break;
        h = (h + 1) & (cap - 1);
      }
    }
    s_hit[s] = hit;
  }
  __syncthreads();

  // ---- stage 3: three order-stable compactions ----
  //   misses     : selection indices still unresolved, in list order
  //   evictables : slots that are not hits, in LRU order (oldest first)
  //   hits       : hit slots, in ascending slot order
  const int segk = ((k + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int segb = ((B + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int k0 = warp * segk, k1 = min(k, k0 + segk);
  const int b0 = warp * segb, b1 = min(B, b0 + segb);
  int cm = 0, ce = 0, ch = 0;
  for (int i0 = k0; i0 < k1; i0 += 32) {
    const int i = i0 + lane;
    cm += __popc(__ballot_sync(kFull, i < k1 && s_out[i] == kUnresolved));
  }
  for (int j0 = b0; j0 < b1; j0 += 32) {
    const int j = j0 + lane;
    const bool in = j < b1;
    ce += __popc(__ballot_sync(kFull, in && !s_hit[in ? s_lru[j] : 0]));
    ch += __popc(__ballot_sync(kFull, in && s_hit[in ? j : 0]));
  }
  if (lane == 0) {
    s_cnt[warp] = cm;
    s_cnt[32 + warp] = ce;
    s_cnt[64 + warp] = ch;
  }
  __syncthreads();
  int vm = s_cnt[lane], ve = s_cnt[32 + lane], vh = s_cnt[64 + lane];
  int im = vm, ie = ve, ih = vh;  // inclusive scans over the 32 warps
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int tm = __shfl_up_sync(kFull, im, d), te = __shfl_up_sync(kFull, ie, d),
              th = __shfl_up_sync(kFull, ih, d);
    if (lane >= d) {
      im += tm;
      ie += te;
      ih += th;
    }
  }
  const int M = __shfl_sync(kFull, im, 31);
  const int E = __shfl_sync(kFull, ie, 31);
  int om = __shfl_sync(kFull, im - vm, warp);
  int oe = __shfl_sync(kFull, ie - ve, warp);
  int oh = __shfl_sync(kFull, ih - vh, warp);
  const uint32_t lt = lanemask_lt();
  for (int i0 = k0; i0 < k1; i0 += 32) {
    const int i = i0 + lane;
    const bool f = i < k1 && s_out[i] == kUnresolved;
    const uint32_t m = __ballot_sync(kFull, f);
    if (f) s_missidx[om + __popc(m & lt)] = static_cast<int16_t>(i);
    om += __popc(m);
  }
  for (int j0 = b0; j0 < b1; j0 += 32) {
    const int j = j0 + lane;
    const bool in = j < b1;
    const int16_t sl = in ? s_lru[j] : 0;
    const bool fe = in && !s_hit[sl];
    uint32_t m = __ballot_sync(kFull, fe);
    if (fe) {
      const int e = oe + __popc(m & lt);
      if (e < M) s_victim[e] = sl;                            // miss e takes it
      s_newlru[e >= M ? e - M : E - M + e] = sl;              // untouched, then fetched
    }
    oe += __popc(m);
    const bool fh = in && s_hit[in ? j : 0];
    m = __ballot_sync(kFull, fh);
    if (fh) s_newlru[E + oh + __popc(m & lt)] = static_cast<int16_t>(j);  // hits newest
    oh += __popc(m);
  }
  __syncthreads();

  // ---- stage 5 (metadata half): victims, page table, slot map ----
  for (int j = tid; j < M; j += kThreads) {
    const int i = s_missidx[j];
    const int16_t v = s_victim[j];
    const int32_t p = s_sel[i];
    const int32_t old = s_slotpos[v];
    s_out[i] = v;
    if (old >= 0) g_pt[old] = -1;
    g_pt[p] = v;
    g_slotpos[v] = p;
    s_fpos[j] = p;
    s_fslot[j] = v;
  }
  if (tid == 0) {
    s_misc[kMiscM] = static_cast<uint32_t>(M);
    a.miss_count[r] = M;
    a.unit_err[r] = 0;
    a.plan_count[r] = kRecordPlan ? M : 0;  // a replay follows only a recorded plan
  }
  __syncthreads();
  for (int i = tid; i < k; i += kThreads) a.out[static_cast<int64_t>(r) * k + i] = s_out[i];
  for (int s = tid; s < B; s += kThreads) g_lru[s] = s_newlru[s];

  // ---- fetch order: misses sorted by host row ----
  // Which slot a miss lands in is fixed above; the order in which the records
  // are read is free.  Reading them in ascending host-row order lets records
  // touched at the same time share GPU page-table walks, which on a large
  // pinned pool costs far less than selection order.  Counting sort into
  // buckets of 2^bucket_shift rows, then each entry's rank inside its bucket.
  if (M > 1) {
    int32_t *s_bkt = reinterpret_cast<int32_t *>(smem + L.bkt);
    int32_t *s_bpos = s_key + cap / 2;   // cap >= 2k: second half is free
    int16_t *s_bslot = s_val + cap / 2;
    const int sh = a.bucket_shift, nb = a.nbuckets;
    for (int b = tid; b < nb; b += kThreads) s_bkt[b] = 0;
    __syncthreads();
    for (int j = tid; j < M; j += kThreads) atomicAdd(&s_bkt[s_fpos[j] >> sh], 1);
    __syncthreads();
    block_exclusive_scan(s_bkt, nb, s_cnt);
    for (int j = tid; j < M; j += kThreads) {
      const int32_t p = s_fpos[j];
      const int q = atomicAdd(&s_bkt[p >> sh], 1);
      s_bpos[q] = p;
      s_bslot[q] = s_fslot[j];
    }
    __syncthreads();
    // now s_bkt[b] is the end of bucket b (and the start of bucket b + 1)
    for (int q = tid; q < M; q += kThreads) {
      const int32_t p = s_bpos[q];
      const int b = p >> sh;
      const int b0 = b ? s_bkt[b - 1] : 0, b1 = s_bkt[b];
      int rnk = 0;
      for (int x = b0; x < b1; ++x) rnk += s_bpos[x] < p;
      s_fpos[b0 + rnk] = p;
      s_fslot[b0 + rnk] = s_bslot[q];
    }
    __syncthreads();
  }
  if (kRecordPlan) {  // the plan lists the same fetches, in the same order
    for (int j = tid; j < M; j += kThreads) {
      a.plan_pos[static_cast<int64_t>(r) * k + j] = s_fpos[j];
      a.plan_slot[static_cast<int64_t>(r) * k + j] = s_fslot[j];
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// RESOLVE: grid = R clusters of `cs` CTAs; cluster c serves request c.
// ---------------------------------------------------------------------------
template <bool kRecordPlan>
__global__ void __launch_bounds__(kThreads, 1) resolve_kernel(const ResolveArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const uint32_t cs = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int r = static_cast<int>(blockIdx.x / cs);
  const SmemLayout L = smem_layout(a.k, a.B, 1 << a.cap_log2);
  int32_t *s_fpos = reinterpret_cast<int32_t *>(smem + L.key);
  int16_t *s_fslot = reinterpret_cast<int16_t *>(smem + L.val);
  uint32_t *s_misc = reinterpret_cast<uint32_t *>(smem + L.misc);

  // Requests at or beyond *num_reqs are graph padding: every CTA of the
  // cluster sees the same count and leaves before any cluster barrier.
  if (rank == 0) {
    if (!leader_resolve<kRecordPlan>(a, r, smem, L)) return;
  } else {
    const int nreq = a.num_reqs ? min(*a.num_reqs, a.R) : a.R;
    if (r >= nreq) return;
  }
  cluster_arrive_release();
  cluster_wait_acquire();

  // Every CTA takes the miss list out of the leader's shared memory.
  int M;
  if (rank == 0) {
    M = static_cast<int>(s_misc[kMiscM]);
  } else {
    M = static_cast<int>(ld_dsmem_u32(dsmem_addr(&s_misc[kMiscM], 0)));
    const int n_pos16 = (M * 4 + 15) / 16, n_slot16 = (M * 2 + 15) / 16;
    const uint32_t rp = dsmem_addr(s_fpos, 0), rs = dsmem_addr(s_fslot, 0);
    for (int c = threadIdx.x; c < n_pos16; c += kThreads)
      reinterpret_cast<uint4 *>(s_fpos)[c] = ld_dsmem_v4(rp + 16u * c);
    for (int c = threadIdx.x; c < n_slot16; c += kThreads)
      reinterpret_cast<uint4 *>(s_fslot)[c] = ld_dsmem_v4(rs + 16u * c);
    __syncthreads();
  }
  cluster_arrive_relaxed();  // this CTA is done reading the leader's memory

  // ---- stage 4: fetch, all CTAs of the cluster ----
  if (a.io && M > 0) {
    const int64_t total = static_cast<int64_t>(M) * a.rec16;
    const int64_t T = static_cast<int64_t>(cs) * kThreads;
    const char *src = a.src + static_cast<int64_t>(r) * a.src_req_stride;
    char *dst = a.hot + static_cast<int64_t>(r) * a.hot_req_stride;
    for (int64_t base = static_cast<int64_t>(rank) * kThreads + threadIdx.x; base < total;
         base += T * kUnroll) {
      uint4 v[kUnroll];
      char *d[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t c = base + u * T;
        d[u] = nullptr;
        if (c < total) {
          const uint32_t c32 = static_cast<uint32_t>(c);
          const int j = static_cast<int>(c32 / static_cast<uint32_t>(a.rec16));
          const int o = static_cast<int>(c32 - static_cast<uint32_t>(j) * a.rec16);
          v[u] = ld_nc_v4(src + static_cast<int64_t>(s_fpos[j]) * a.src_row_stride + 16 * o);
          d[u] = dst + static_cast<int64_t>(s_fslot[j]) * a.hot_row_stride + 16 * o;
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (d[u]) st_v4(d[u], v[u]);
    }
  }
  cluster_wait_acquire();  // the leader's memory must outlive every reader
}

// ===========================================================================
// RESOLVE, page-table lookup (the default).  One cluster per request.
//   workers (CTAs 1..cs-1, or CTA 0 alone when cs == 1) each take a slice of
//     the selection list, classify every entry through the page table (padding,
//     newest token, hit, miss), mark hit slots in a bitmap, list their misses
//     in list order, and -- without waiting for any decision -- start reading
//     the missed records from the host pool into registers;
//   the leader (CTA 0) merges the slices through distributed shared memory,
//     checks duplicates, runs the two order-stable compactions (hit slots in
//     slot order; evictable slots in LRU order) that give every miss its
//     victim and the new LRU order, and releases the workers, which store the
//     staged records into their victims while the leader publishes the page
//     table, slot map, LRU order and plan.
// The reads from host memory thus overlap the leader's decision instead of
// following it.  Results are identical to the hash-staged kernel above.
// ===========================================================================
constexpr int kStage = 4;        // 16-byte chunks a worker thread stages in registers
constexpr int kMaxWorkers = 15;  // cluster size 16 at most
constexpr int kGroup = 4;        // selections a worker thread classifies per load batch
constexpr int kRankSortMax = 128;  // up to this many misses a slice is ordered by direct ranking

struct PtLayout {
  uint32_t w_sel, w_out, w_mi, w_mp, w_hit, w_vict, w_misc, w_bkt, w_bidx, w_ord;  // worker
  uint32_t l_lru, l_slotpos, l_hit, l_newlru, l_ev, l_mpos, l_hkey, l_misc;     // leader
  uint32_t l_prevrow;                                                             // leader
  uint32_t l_hmin, l_alias;  // union mode: first list index per set entry, per miss its unique index
  uint32_t cnt, total;
};

__host__ __device__ inline PtLayout pt_layout(int k, int B, int ks, int hcap, int rec) {
  PtLayout L;
  uint32_t o = 0;
  const uint32_t nwords = (B + 31) / 32;
  L.w_sel = o;     o += align16(4u * ks);
  L.w_out = o;     o += align16(4u * ks);
  L.w_mi = o;      o += align16(4u * ks);
  L.w_mp = o;      o += align16(4u * ks);
  L.w_hit = o;     o += align16(4u * nwords);
  L.w_vict = o;    o += align16(4u * ks);
  L.w_misc = o;    o += align16(4u * 8);
  L.w_bkt = o;     o += align16(4u * kMaxBuckets);
  L.w_bidx = o;    o += align16(4u * ks);
  L.w_ord = o;     o += align16(4u * ks);
  L.l_lru = o;     o += align16(2u * B);
  L.l_slotpos = o; o += align16(4u * B);
  L.l_hit = o;     o += align16(4u * nwords);
  L.l_newlru = o;  o += align16(2u * B);
  L.l_ev = o;      o += align16(4u * k);
  L.l_mpos = o;    o += align16(4u * k);
  L.l_hkey = o;    o += align16(4u * hcap);
  L.l_misc = o;    o += align16(4u * (8 + kMaxWorkers + 1));
  L.l_hmin = o;    o += align16(4u * hcap);
  L.l_alias = o;   o += align16(4u * k);
  L.cnt = o;       o += align16(4u * 64);
  L.l_prevrow = o; o += align16(static_cast<uint32_t>(rec));
  L.total = o;
  return L;
}

// worker misc words / leader misc words
enum { kWErr = 0, kWNewest = 1, kWCount = 2, kWLeadErr = 3 };
enum { kLErr = 0, kLM = 1, kLHits = 2, kLAnyHit = 3, kLSame = 4, kLPrefix = 8 };

struct PtArgs {
  int32_t R, k, B, rec16, io, ks, hcap_log2;
  int32_t bucket_shift, nbuckets;  // host-row buckets for the fetch order
  // Fused write-through (hisparse_resolve_step): the previous token's row B
  // goes to host row prev_pos[r], then new_rows[r] replaces it.  With
  // prev_from_row the previous token, if selected, is filled from row B
  // (which is what the host row now holds) instead of being read back.
  const int32_t *prev_pos;
  const char *new_rows;
  char *host_w;
  char *mirror_w;  // the layer's HBM mirror (null if none): written back alongside
  int64_t host_req_stride, host_row_stride;
  int32_t prev_from_row;
  // Resident tier (three-tier resolve): per request a block table
  // [R][res_nblk] of resident block indices (-1 = not resident), res_tok
  // positions per block; NULL = no resident tier.
  const int32_t *res_blocks;
  int32_t res_nblk, res_tok;
  // Block-id selections: sel holds k / sel_bt block ids per request, each
  // standing for sel_bt consecutive positions (1 = sel holds positions).
  int32_t sel_bt;
  // Union mode (speculative verify rows resolved as one list): a repeated
  // position is resolved at its first reference and shares its row.
  int32_t union_mode;
  // Short requests (hisparse_resolve_options.d_seq_lens): a request whose
  // seq_len is at most B grows by its previous token and is looked up by
  // position; NULL = every request takes the general path.
  const int32_t *seq_lens;
  // Shared-index layers filled in the same launch (HISPARSE_WITH_SHARED):
  // every missed record's row of each, at the anchor's victim slot.
  int32_t nfl;
  ReplayTarget fl[kMaxReplayTargets];
  int64_t P;
  const int32_t *sel, *num_reqs, *newest;
  int32_t *out;
  int32_t *slot_pos;
  int16_t *lru;
  int32_t *page_table, *miss_count, *unit_err;
  uint32_t *status;
  int32_t *plan_pos, *plan_slot, *plan_count;
  const char *src;
  int64_t src_req_stride, src_row_stride;
  char *hot;
  int64_t hot_req_stride, hot_row_stride;
};

// Stable block-wide compaction of [0, n): emit(i, rank) for every i with
// flag(i), rank = number of flagged elements before i.  Each warp scans one
// contiguous segment with __ballot_sync/__popc; one barrier publishes the 32
// warp totals, which every warp prefix-sums with shuffles.  Returns the count.
template <class Flag, class Emit>
__device__ __forceinline__ int block_compact(int n, Flag flag, Emit emit, int32_t *s_cnt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = ((n + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int i0 = warp * seg, i1 = min(n, i0 + seg);
  int c = 0;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    c += __popc(__ballot_sync(kFull, i < i1 && flag(i)));
  }
  if (lane == 0) s_cnt[warp] = c;
  __syncthreads();
  const int v = s_cnt[lane];
  int inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(kFull, inc, d);
    if (lane >= d) inc += t;
  }
  const int total = __shfl_sync(kFull, inc, 31);
  int base = __shfl_sync(kFull, inc - v, warp);
  const uint32_t lt = lanemask_lt();
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const bool f = i < i1 && flag(i);
    const uint32_t m = __ballot_sync(kFull, f);
    if (f) emit(i, base + __popc(m & lt));
    base += __popc(m);
  }
  __syncthreads();
  return total;
}

// Two stable compactions of [0, n) in one pass (one barrier for both):
// emitA(i, rank) for flagA, emitB(i, rank) for flagB.  s_cnt holds 64 ints.
template <class FlagA, class EmitA, class FlagB, class EmitB>
__device__ __forceinline__ void block_compact2(int n, FlagA flagA, EmitA emitA, FlagB flagB,
                                               EmitB emitB, int32_t *s_cnt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = ((n + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int i0 = warp * seg, i1 = min(n, i0 + seg);
  int ca = 0, cb = 0;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const bool in = i < i1;
    ca += __popc(__ballot_sync(kFull, in && flagA(i)));
    cb += __popc(__ballot_sync(kFull, in && flagB(i)));
  }
  if (lane == 0) {
    s_cnt[warp] = ca;
    s_cnt[32 + warp] = cb;
  }
  __syncthreads();
  const int va = s_cnt[lane], vb = s_cnt[32 + lane];
  int ia = va, ib = vb;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int ta = __shfl_up_sync(kFull, ia, d), tb = __shfl_up_sync(kFull, ib, d);
    if (lane >= d) {
      ia += ta;
      ib += tb;
    }
  }
  int ba = __shfl_sync(kFull, ia - va, warp), bb = __shfl_sync(kFull, ib - vb, warp);
  const uint32_t lt = lanemask_lt();
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const bool in = i < i1;
    const bool fa = in && flagA(i), fb = in && flagB(i);
    const uint32_t ma = __ballot_sync(kFull, fa), mb = __ballot_sync(kFull, fb);
    if (fa) emitA(i, ba + __popc(ma & lt));
    if (fb) emitB(i, bb + __popc(mb & lt));
    ba += __popc(ma);
    bb += __popc(mb);
  }
  __syncthreads();
}

__device__ __forceinline__ bool bit_of(const uint32_t *bits, int s) {
  return (bits[s >> 5] >> (s & 31)) & 1u;
}

// Worker: classify selections [i0, i0 + n) of request r.
// Position of selection index t (0 <= t < k) of request r: the list entry
// itself, or, for block-id selections, entry t / sel_bt expanded in registers
// (gentlecold.top §5.5: block ids are expanded into token positions without a
// token list in memory).  -1 blocks give padding; other negative ids give
// negative positions, which classification rejects as out of range.
template <bool kExt>
__device__ __forceinline__ int32_t sel_position(const PtArgs &a, int r, int t) {
  if (!kExt || a.sel_bt == 1) return a.sel[static_cast<int64_t>(r) * a.k + t];
  const int kb = a.k / a.sel_bt;
  const int32_t b = a.sel[static_cast<int64_t>(r) * kb + t / a.sel_bt];
  if (b == -1) return -1;
  const int64_t q = static_cast<int64_t>(b) * a.sel_bt + t % a.sel_bt;
  return q > INT32_MAX ? INT32_MAX : (q < INT32_MIN ? INT32_MIN : static_cast<int32_t>(q));
}

template <bool kExt>
__device__ int pt_worker_classify(const PtArgs &a, int r, int i0, int n, int32_t newest,
                                  const int32_t (&first)[kGroup], unsigned char *smem,
                                  const PtLayout &L) {
  const int tid = threadIdx.x;
  const int B = a.B;
  const int64_t P = a.P;
  int32_t *w_sel = reinterpret_cast<int32_t *>(smem + L.w_sel);
  int32_t *w_out = reinterpret_cast<int32_t *>(smem + L.w_out);
  int32_t *w_mi = reinterpret_cast<int32_t *>(smem + L.w_mi);
  int32_t *w_mp = reinterpret_cast<int32_t *>(smem + L.w_mp);
  uint32_t *w_hit = reinterpret_cast<uint32_t *>(smem + L.w_hit);
  uint32_t *w_misc = reinterpret_cast<uint32_t *>(smem + L.w_misc);
  int32_t *s_cnt = reinterpret_cast<int32_t *>(smem + L.cnt);
  const int nwords = (B + 31) / 32;
  for (int x = tid; x < nwords; x += kThreads) w_hit[x] = 0;
  if (tid < 8) w_misc[tid] = 0;
  __syncthreads();
  const int32_t *g_pt = a.page_table + static_cast<int64_t>(r) * P;
  const int32_t *g_res = (kExt && a.res_blocks) ? a.res_blocks + static_cast<int64_t>(r) * a.res_nblk : nullptr;
  for (int base = 0; base < n; base += kGroup * kThreads) {
    int32_t p[kGroup], s[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int t = base + u * kThreads + tid;
      p[u] = base == 0 ? first[u] : (t < n ? sel_position<kExt>(a, r, i0 + t) : -1);
    }
    int32_t e[kGroup];  // resident block entry of each selection (-1: none)
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      s[u] = -1;
      e[u] = -1;
      if (p[u] >= 0 && p[u] < P) {
        if (kExt && g_res && p[u] / a.res_tok < a.res_nblk) e[u] = g_res[p[u] / a.res_tok];
        if (p[u] != newest) s[u] = g_pt[p[u]];
      }
    }
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int t = base + u * kThreads + tid;
      if (t >= n) continue;
      int32_t v;
      if (p[u] == -1) {
        v = -1;
      } else if (p[u] < -1 || p[u] >= P) {
        atomicOr(&w_misc[kWErr], HISPARSE_ERR_RANGE);
        v = -1;
      } else if (kExt && e[u] != -1) {
        // resident copy: B + 1 + row, no hit, no miss, no duplicate check
        // (vLLM docs "Hot lookup and LRU"; gentlecold.top §6.5)
        const int64_t row = static_cast<int64_t>(e[u]) * a.res_tok + p[u] % a.res_tok;
        if (e[u] < -1 || static_cast<int64_t>(B) + 1 + row > INT32_MAX) {
          atomicOr(&w_misc[kWErr], HISPARSE_ERR_RANGE);
          v = -1;
        } else {
          v = static_cast<int32_t>(B + 1 + row);
        }
      } else if (p[u] == newest) {
        atomicAdd(&w_misc[kWNewest], 1u);
        v = B;
      } else if (s[u] >= 0) {
        if (s[u] >= B) {  // a page-table entry outside [-1, B): treat the unit as failed
          atomicOr(&w_misc[kWErr], HISPARSE_ERR_RANGE);
          v = -1;
        } else {
          const uint32_t bit = 1u << (s[u] & 31);
          if ((atomicOr(&w_hit[s[u] >> 5], bit) & bit) && !(kExt && a.union_mode))
            atomicOr(&w_misc[kWErr], HISPARSE_ERR_DUP);
          v = s[u];
        }
      } else {
        v = kUnresolved;
      }
      w_sel[t] = p[u];
      w_out[t] = v;
    }
  }
  __syncthreads();
  const int mw = block_compact(
      n, [&](int t) { return w_out[t] == kUnresolved; },
      [&](int t, int j) {
        w_mi[j] = t;
        w_mp[j] = w_sel[t];
      },
      s_cnt);
  if (tid == 0) w_misc[kWCount] = static_cast<uint32_t>(mw);
  __syncthreads();
  return mw;
}

// Worker: order the slice's misses j0 .. mw-1 by ascending host row into
// w_ord[0 .. mw-j0).  Which slot each lands in does not depend on it; reading
// in address order lets nearby records share the GPU's address-translation
// walks, which matters whenever the GPU cannot keep the pool's translations
// cached.  Ties (equal rows) only occur in a failing unit; they are broken by
// list index, so w_ord always holds each index once.
__device__ void pt_worker_order(const PtArgs &a, int j0, int mw, unsigned char *smem,
                                const PtLayout &L) {
  const int tid = threadIdx.x;
  const int32_t *w_mp = reinterpret_cast<const int32_t *>(smem + L.w_mp);
  int32_t *w_ord = reinterpret_cast<int32_t *>(smem + L.w_ord);
  int32_t *s_cnt = reinterpret_cast<int32_t *>(smem + L.cnt);
  const int n = mw - j0;
  if (n <= 0) return;
  if (n <= 32) {
    if (tid < 32) {  // one warp: each lane ranks its miss against the others
      const int32_t key = tid < n ? w_mp[j0 + tid] : 0;
      int rnk = 0;
      for (int i = 0; i < n; ++i) {
        const int32_t ki = __shfl_sync(kFull, key, i);
        rnk += ki < key || (ki == key && i < tid);
      }
      if (tid < n) w_ord[rnk] = j0 + tid;
    }
  } else if (n <= kRankSortMax) {
    for (int i = tid; i < n; i += kThreads) {  // rank against every miss (broadcast reads)
      const int32_t key = w_mp[j0 + i];
      int rnk = 0;
      for (int x = 0; x < n; ++x) {
        const int32_t kx = w_mp[j0 + x];
        rnk += kx < key || (kx == key && x < i);
      }
      w_ord[rnk] = j0 + i;
    }
  } else {  // counting sort into row buckets, then a rank inside each bucket
    int32_t *w_bkt = reinterpret_cast<int32_t *>(smem + L.w_bkt);
    int32_t *w_bidx = reinterpret_cast<int32_t *>(smem + L.w_bidx);
    const int sh = a.bucket_shift, nb = a.nbuckets;
    for (int b = tid; b < nb; b += kThreads) w_bkt[b] = 0;
    __syncthreads();
    for (int j = j0 + tid; j < mw; j += kThreads) atomicAdd(&w_bkt[w_mp[j] >> sh], 1);
    __syncthreads();
    block_exclusive_scan(w_bkt, nb, s_cnt);
    for (int j = j0 + tid; j < mw; j += kThreads) w_bidx[atomicAdd(&w_bkt[w_mp[j] >> sh], 1)] = j;
    __syncthreads();
    // now w_bkt[b] ends bucket b; rank each entry inside its bucket
    for (int q = tid; q < n; q += kThreads) {
      const int j = w_bidx[q];
      const int32_t p = w_mp[j];
      const int b = p >> sh;
      const int b0 = b ? w_bkt[b - 1] : 0, b1 = w_bkt[b];
      int rnk = 0;
      for (int x = b0; x < b1; ++x) {
        const int32_t px = w_mp[w_bidx[x]];
        rnk += px < p || (px == p && x < q);
      }
      w_ord[b0 + rnk] = j;
    }
  }
  __syncthreads();
}

// Leader: merge the workers' slices, check duplicates, choose victims and the
// new LRU order.  Returns nothing; results live in the leader's shared memory.
template <bool kExt>
__device__ void pt_leader_decide(const PtArgs &a, int cs, int nw, int32_t newest,
                                 unsigned char *smem, const PtLayout &L) {
  const bool uni = kExt && a.union_mode;
  const int tid = threadIdx.x, lane = tid & 31;
  const int B = a.B;
  const int nwords = (B + 31) / 32;
  const int hcap = 1 << a.hcap_log2;
  int16_t *l_lru = reinterpret_cast<int16_t *>(smem + L.l_lru);
  uint32_t *l_hit = reinterpret_cast<uint32_t *>(smem + L.l_hit);
  int16_t *l_newlru = reinterpret_cast<int16_t *>(smem + L.l_newlru);
  int32_t *l_ev = reinterpret_cast<int32_t *>(smem + L.l_ev);
  int32_t *l_mpos = reinterpret_cast<int32_t *>(smem + L.l_mpos);
  int32_t *l_hkey = reinterpret_cast<int32_t *>(smem + L.l_hkey);
  int32_t *l_hmin = reinterpret_cast<int32_t *>(smem + L.l_hmin);
  int32_t *l_alias = reinterpret_cast<int32_t *>(smem + L.l_alias);
  uint32_t *l_misc = reinterpret_cast<uint32_t *>(smem + L.l_misc);
  int32_t *s_cnt = reinterpret_cast<int32_t *>(smem + L.cnt);
  const uint32_t *w_misc0 = reinterpret_cast<const uint32_t *>(smem + L.w_misc);
  const uint32_t *w_hit0 = reinterpret_cast<const uint32_t *>(smem + L.w_hit);
  const int32_t *w_mp0 = reinterpret_cast<const int32_t *>(smem + L.w_mp);
  auto wrank = [&](int w) { return static_cast<uint32_t>(cs == 1 ? 0 : w + 1); };

  // Every read of a worker's shared memory below is issued by a different
  // thread, so the cluster's distributed-shared-memory latency is paid once
  // per phase, not once per worker.
  // (1) per-worker counts -> prefix offsets in list order; error bits (warp 0)
  if (tid < 32) {
    uint32_t err = 0, seen = 0;
    int cnt = 0;
    if (lane < nw) {
      err = ld_dsmem_u32(dsmem_addr(&w_misc0[kWErr], wrank(lane)));
      seen = ld_dsmem_u32(dsmem_addr(&w_misc0[kWNewest], wrank(lane)));
      cnt = static_cast<int>(ld_dsmem_u32(dsmem_addr(&w_misc0[kWCount], wrank(lane))));
    }
    int inc = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(kFull, inc, d);
      if (lane >= d) inc += t;
      err |= __shfl_xor_sync(kFull, err, d);
      seen += __shfl_xor_sync(kFull, seen, d);
    }
    if (lane < nw) l_misc[kLPrefix + lane] = static_cast<uint32_t>(inc - cnt);
    if (lane == 31) {
      if (newest < -1 || newest >= a.P) err |= HISPARSE_ERR_RANGE;
      if (seen > 1 && !uni) err |= HISPARSE_ERR_DUP;
      l_misc[kLPrefix + nw] = static_cast<uint32_t>(inc);
      l_misc[kLErr] = err;
      l_misc[kLM] = static_cast<uint32_t>(inc);
      l_misc[kLHits] = 0;
      l_misc[kLAnyHit] = 0;
      l_misc[kLSame] = 0;
    }
  }
  for (int x = tid; x < nwords; x += kThreads) l_hit[x] = 0;
  __syncthreads();
  // (2) hit bitmap: OR of the slices (a slot hit by two slices is a duplicate),
  //     and the miss positions in list order, with duplicates among misses
  //     caught by an open-addressing set ([DD] §3.5 stage 1's hash).
  {
    uint32_t dup = 0, any = 0;
    for (int idx = tid; idx < nw * nwords; idx += kThreads) {
      const int w = idx / nwords, x = idx - w * nwords;
      const uint32_t b = ld_dsmem_u32(dsmem_addr(&w_hit0[x], wrank(w)));
      if (b) dup |= atomicOr(&l_hit[x], b) & b;
      any |= b;
    }
    if (uni) dup = 0;  // a slot hit from two slices is one shared position
    if (any) l_misc[kLAnyHit] = 1;
    const int M = static_cast<int>(l_misc[kLM]);
    for (int g = tid; g < M; g += kThreads) {
      int w = 0;
      while (w + 1 < nw && static_cast<int>(l_misc[kLPrefix + w + 1]) <= g) ++w;
      const int j = g - static_cast<int>(l_misc[kLPrefix + w]);
      const int32_t p = static_cast<int32_t>(ld_dsmem_u32(dsmem_addr(&w_mp0[j], wrank(w))));
      l_mpos[g] = p;
      uint32_t h = hash_pos(p, a.hcap_log2);
      for (int probe = 0; probe < hcap; ++probe) {
        const int32_t prev = atomicCAS(&l_hkey[h], -1, p);
        if (prev == -1 || prev == p) {
          if (uni) atomicMin(&l_hmin[h], g);  // the entry keeps its first reference
          else if (prev == p) dup = 1;
          break;
        }
        h = (h + 1) & (hcap - 1);
      }
    }
    if (dup) atomicOr(&l_misc[kLErr], HISPARSE_ERR_DUP);
  }
  __syncthreads();
  if (l_misc[kLErr]) return;  // uniform
  if (uni) {
    // Union mode ([DD] §6.5: misses in first-reference order): miss g is a
    // real miss when it is its position's first reference; its unique index
    // u is the number of first references before it.  Every miss g records in
    // l_alias the unique index of its position's first reference, negated and
    // offset (-1 - u) for a later reference.  The unique positions then
    // replace l_mpos in list order.
    const int Mall = static_cast<int>(l_misc[kLM]);
    int32_t *l_upos = l_hkey;  // the set is not needed once l_alias is known
    for (int g0 = 0; g0 < Mall; g0 += kThreads) {
      const int g = g0 + tid;
      int32_t rep = g;
      if (g < Mall) {
        const int32_t p = l_mpos[g];
        uint32_t h = hash_pos(p, a.hcap_log2);
        for (int probe = 0; probe < hcap && l_hkey[h] != p; ++probe) h = (h + 1) & (hcap - 1);
        rep = l_hmin[h];
      }
      const bool first = g < Mall && rep == g;
      const uint32_t m = __ballot_sync(kFull, first);
      if (lane == 31) s_cnt[tid >> 5] = __popc(m);
      __syncthreads();
      int before = static_cast<int>(l_misc[kLHits]);  // running count of first references
      for (int x = 0; x < (tid >> 5); ++x) before += s_cnt[x];
      const int u = before + __popc(m & lanemask_lt());
      if (first) l_alias[g] = u;
      else if (g < Mall) l_alias[g] = -1 - rep;  // resolved below, once every u is known
      __syncthreads();
      if (tid == kThreads - 1) l_misc[kLHits] = static_cast<uint32_t>(u + (first ? 1 : 0));
      __syncthreads();
    }
    for (int g = tid; g < Mall; g += kThreads) {
      const int32_t v = l_alias[g];
      if (v >= 0) l_upos[v] = l_mpos[g];
    }
    __syncthreads();
    for (int g = tid; g < Mall; g += kThreads) {
      const int32_t v = l_alias[g];
      if (v < 0) l_alias[g] = -1 - l_alias[-1 - v];  // later reference: -1 - (its first's u)
    }
    const int M = static_cast<int>(l_misc[kLHits]);
    __syncthreads();
    for (int u = tid; u < M; u += kThreads) l_mpos[u] = l_upos[u];
    if (tid == 0) {
      l_misc[kLM] = static_cast<uint32_t>(M);
      l_misc[kLHits] = 0;
    }
    __syncthreads();
  }
  // No miss and no hot hit (every selection resident, newest or padding): the
  // LRU order stays as it is ([DD] §6.5: resident hits exit before the LRU).
  if (l_misc[kLM] == 0 && l_misc[kLAnyHit] == 0) {
    __syncthreads();
    if (tid == 0) l_misc[kLSame] = 1;
    return;
  }
  // (3) one block-wide pass compacts the hits (slot order) and the evictables
  //     (LRU order) together.  Thread t owns slots and LRU positions
  //     [t*per, t*per + per); one exclusive scan of the packed per-thread
  //     counts (hits << 16 | evictables; both < 2^15) gives every thread its
  //     output ranks and every warp the hit total H.
  const int M = static_cast<int>(l_misc[kLM]);
  const int per = (B + kThreads - 1) / kThreads;  // <= 32 since B <= 32767
  const int j0 = min(B, tid * per), j1 = min(B, j0 + per);
  uint32_t ma = 0, mb = 0;  // bit i: slot j0+i is hit / LRU entry j0+i is evictable
  for (int j = j0; j < j1; ++j) {
    ma |= static_cast<uint32_t>(bit_of(l_hit, j)) << (j - j0);
    mb |= static_cast<uint32_t>(!bit_of(l_hit, l_lru[j])) << (j - j0);
  }
  const uint32_t v = (static_cast<uint32_t>(__popc(ma)) << 16) | static_cast<uint32_t>(__popc(mb));
  uint32_t inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, inc, d);
    if (lane >= d) inc += t;
  }
  if (lane == 31) s_cnt[tid >> 5] = static_cast<int32_t>(inc);
  __syncthreads();
  const uint32_t wt = static_cast<uint32_t>(s_cnt[lane]);
  uint32_t winc = wt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, winc, d);
    if (lane >= d) winc += t;
  }
  const uint32_t total = __shfl_sync(kFull, winc, 31);
  const uint32_t base = __shfl_sync(kFull, winc - wt, tid >> 5) + inc - v;
  const int H = static_cast<int>(total >> 16);
  const int E = B - H;
  int ha = static_cast<int>(base >> 16), eb = static_cast<int>(base & 0xFFFFu);
  for (int j = j0; j < j1; ++j) {
    const int i = j - j0;
    if ((ma >> i) & 1u) l_newlru[E + ha++] = static_cast<int16_t>(j);
    if ((mb >> i) & 1u) {
      const int16_t sl = l_lru[j];
      if (eb < M) l_ev[eb] = sl;
      l_newlru[eb >= M ? eb - M : E - M + eb] = sl;
      ++eb;
    }
  }
  if (tid == 0) l_misc[kLHits] = static_cast<uint32_t>(H);
  __syncthreads();
}

// Leader: hand every slice the verdict and its victims, written straight
// into the workers' shared memory, so that after the next cluster barrier a
// worker reads them locally.
template <bool kExt>
__device__ void pt_leader_push(const PtArgs &a, int cs, int nw, unsigned char *smem,
                               const PtLayout &L) {
  const int tid = threadIdx.x;
  const uint32_t *l_misc = reinterpret_cast<const uint32_t *>(smem + L.l_misc);
  const int32_t *l_ev = reinterpret_cast<const int32_t *>(smem + L.l_ev);
  const int32_t *l_alias = reinterpret_cast<const int32_t *>(smem + L.l_alias);
  const uint32_t *w_misc0 = reinterpret_cast<const uint32_t *>(smem + L.w_misc);
  const int32_t *w_vict0 = reinterpret_cast<const int32_t *>(smem + L.w_vict);
  auto wrank = [&](int w) { return static_cast<uint32_t>(cs == 1 ? 0 : w + 1); };
  const uint32_t err = l_misc[kLErr];
  for (int w = tid; w < nw; w += kThreads)
    st_dsmem_u32(dsmem_addr(&w_misc0[kWLeadErr], wrank(w)), err);
  if (err) return;
  const bool uni = kExt && a.union_mode;
  // every miss of every slice, repeats included (union mode)
  const int Mall = static_cast<int>(uni ? l_misc[kLPrefix + nw] : l_misc[kLM]);
  for (int g = tid; g < Mall; g += kThreads) {
    int w = 0;
    while (w + 1 < nw && static_cast<int>(l_misc[kLPrefix + w + 1]) <= g) ++w;
    const int j = g - static_cast<int>(l_misc[kLPrefix + w]);
    uint32_t v;
    if (uni) {  // a later reference takes its first's slot and is not fetched
      const int32_t al = l_alias[g];
      v = al >= 0 ? static_cast<uint32_t>(l_ev[al]) : (static_cast<uint32_t>(l_ev[-1 - al]) | kAlias);
    } else {
      v = static_cast<uint32_t>(l_ev[g]);
    }
    st_dsmem_u32(dsmem_addr(&w_vict0[j], wrank(w)), v);
  }
}

// Leader: publish page table, slot map, LRU order, counts, plan.
template <bool kRecordPlan>
__device__ void pt_leader_publish(const PtArgs &a, int r, int32_t prev, int32_t skip_pos,
                                  unsigned char *smem, const PtLayout &L) {
  const int tid = threadIdx.x;
  const int B = a.B, k = a.k;
  const int64_t P = a.P;
  if (a.prev_pos && prev >= 0 && prev < P) {
    // fused write-through, second half: the kept row B -> host row prev
    const uint4 *keep = reinterpret_cast<const uint4 *>(smem + L.l_prevrow);
    uint4 *hrow = reinterpret_cast<uint4 *>(a.host_w + static_cast<int64_t>(r) * a.host_req_stride +
                                            static_cast<int64_t>(prev) * a.host_row_stride);
    for (int c = tid; c < a.rec16; c += kThreads) st_v4(hrow + c, keep[c]);
    if (a.mirror_w) {  // the mirror stays a byte-for-byte copy of the host pool
      uint4 *mrow = reinterpret_cast<uint4 *>(a.mirror_w + static_cast<int64_t>(r) * a.host_req_stride +
                                              static_cast<int64_t>(prev) * a.host_row_stride);
      for (int c = tid; c < a.rec16; c += kThreads) st_v4(mrow + c, keep[c]);
    }
  }
  const int32_t *l_slotpos = reinterpret_cast<const int32_t *>(smem + L.l_slotpos);
  const int16_t *l_newlru = reinterpret_cast<const int16_t *>(smem + L.l_newlru);
  const int32_t *l_ev = reinterpret_cast<const int32_t *>(smem + L.l_ev);
  const int32_t *l_mpos = reinterpret_cast<const int32_t *>(smem + L.l_mpos);
  const uint32_t *l_misc = reinterpret_cast<const uint32_t *>(smem + L.l_misc);
  const uint32_t err = l_misc[kLErr];
  if (err) {
    if (tid == 0) {
      a.unit_err[r] = static_cast<int32_t>(err);
      atomicOr(a.status, err);
      a.miss_count[r] = 0;
      a.plan_count[r] = 0;
    }
    return;
  }
  const int M = static_cast<int>(l_misc[kLM]);
  int32_t *g_pt = a.page_table + static_cast<int64_t>(r) * P;
  int32_t *g_slotpos = a.slot_pos + static_cast<int64_t>(r) * B;
  if (skip_pos >= 0 && a.io) {  // the previous token's record, from the kept row B
    __shared__ int32_t s_prev_victim;
    if (tid == 0) s_prev_victim = -1;
    __syncthreads();
    for (int g = tid; g < M; g += kThreads)
      if (l_mpos[g] == skip_pos) s_prev_victim = l_ev[g];
    __syncthreads();
    const int32_t pv = s_prev_victim;
    if (pv >= 0) {
      const uint4 *keep = reinterpret_cast<const uint4 *>(smem + L.l_prevrow);
      uint4 *row = reinterpret_cast<uint4 *>(a.hot + static_cast<int64_t>(r) * a.hot_req_stride +
                                             static_cast<int64_t>(pv) * a.hot_row_stride);
      for (int c = tid; c < a.rec16; c += kThreads) st_v4(row + c, keep[c]);
    }
  }
  for (int g = tid; g < M; g += kThreads) {
    const int32_t v = l_ev[g], p = l_mpos[g], old = l_slotpos[v];
    if (old >= 0) g_pt[old] = -1;
    g_pt[p] = v;
    g_slotpos[v] = p;
    if (kRecordPlan) {
      a.plan_pos[static_cast<int64_t>(r) * k + g] = p;
      a.plan_slot[static_cast<int64_t>(r) * k + g] = v;
    }
  }
  int16_t *g_lru = a.lru + static_cast<int64_t>(r) * B;
  if (!l_misc[kLSame])
    for (int s = tid; s < B; s += kThreads) g_lru[s] = l_newlru[s];
  if (tid == 0) {
    a.miss_count[r] = M;
    a.unit_err[r] = 0;
    a.plan_count[r] = kRecordPlan ? M : 0;
  }
}

// Worker, after the leader's decision (its verdict and this slice's victims
// are already in this CTA's shared memory): store the `staged` records held in
// registers (the slice's first misses, in list order), read and store the rest
// in host-row order (w_ord), and write the slice's slot vector.
__device__ void pt_worker_finish(const PtArgs &a, int r, int i0, int n, int32_t skip_pos,
                                 int staged, const uint4 *v, const char *src, char *dst,
                                 unsigned char *smem, const PtLayout &L) {
  const int tid = threadIdx.x;
  const int32_t *w_vict = reinterpret_cast<const int32_t *>(smem + L.w_vict);
  const int32_t *w_out = reinterpret_cast<const int32_t *>(smem + L.w_out);
  const int32_t *w_mi = reinterpret_cast<const int32_t *>(smem + L.w_mi);
  const int32_t *w_mp = reinterpret_cast<const int32_t *>(smem + L.w_mp);
  const int32_t *w_ord = reinterpret_cast<const int32_t *>(smem + L.w_ord);
  const uint32_t *w_misc = reinterpret_cast<const uint32_t *>(smem + L.w_misc);
  const int mw = static_cast<int>(w_misc[kWCount]);
  const uint32_t err = w_misc[kWLeadErr];
  if (!err && a.io) {
    const int64_t totc = static_cast<int64_t>(staged) * a.rec16;
#pragma unroll
    for (int u = 0; u < kStage; ++u) {
      const int64_t q = tid + static_cast<int64_t>(u) * kThreads;
      if (v && q < totc) {
        const uint32_t q32 = static_cast<uint32_t>(q);
        const int f = static_cast<int>(q32 / static_cast<uint32_t>(a.rec16));
        const int o = static_cast<int>(q32 - static_cast<uint32_t>(f) * a.rec16);
        if (w_mp[f] != skip_pos && !(w_vict[f] & kAlias))
          st_v4(dst + static_cast<int64_t>(w_vict[f]) * a.hot_row_stride + 16 * o, v[u]);
      }
    }
    // the rest of the slice's misses, in host-row order
    const int64_t totr = static_cast<int64_t>(mw - staged) * a.rec16;
    for (int64_t b0 = tid; b0 < totr; b0 += static_cast<int64_t>(kThreads) * kUnroll) {
      uint4 x[kUnroll];
      char *d[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t q = b0 + static_cast<int64_t>(u) * kThreads;
        d[u] = nullptr;
        if (q < totr) {
          const uint32_t q32 = static_cast<uint32_t>(q);
          const int f = static_cast<int>(q32 / static_cast<uint32_t>(a.rec16));
          const int o = static_cast<int>(q32 - static_cast<uint32_t>(f) * a.rec16);
          const int j = w_ord[f];
          if (w_mp[j] != skip_pos && !(w_vict[j] & kAlias)) {
            x[u] = ld_nc_v4(src + static_cast<int64_t>(w_mp[j]) * a.src_row_stride + 16 * o);
            d[u] = dst + static_cast<int64_t>(w_vict[j]) * a.hot_row_stride + 16 * o;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (d[u]) st_v4(d[u], x[u]);
    }
    // the shared-index layers: a miss's rows of all of them back to back
    // (adjacent host rows when the group's rows are interleaved)
    if (a.nfl > 0) {
      const uint32_t rec16 = static_cast<uint32_t>(a.rec16);
      const uint32_t per = static_cast<uint32_t>(a.nfl) * rec16;
      const int64_t totf = static_cast<int64_t>(mw) * per;
      for (int64_t b0 = tid; b0 < totf; b0 += static_cast<int64_t>(kThreads) * kUnroll) {
        uint4 x[kUnroll];
        char *d[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t q = b0 + static_cast<int64_t>(u) * kThreads;
          d[u] = nullptr;
          if (q < totf) {
            const uint32_t q32 = static_cast<uint32_t>(q);
            const uint32_t j = q32 / per, rem = q32 - j * per;
            const uint32_t f = rem / rec16, o = rem - f * rec16;
            const int32_t vj = w_vict[j];
            if (!(vj & kAlias)) {
              const ReplayTarget &T = a.fl[f];
              x[u] = ld_nc_v4(T.src + static_cast<int64_t>(r) * T.src_req_stride +
                              static_cast<int64_t>(w_mp[j]) * T.src_row_stride + 16 * o);
              d[u] = T.hot + static_cast<int64_t>(r) * T.hot_req_stride +
                     static_cast<int64_t>(vj) * T.hot_row_stride + 16 * o;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (d[u]) st_v4(d[u], x[u]);
      }
    }
  }
  // the slice's slot vector ([DD] §3.5 stage 5: aligned with the list)
  int32_t *g_out = a.out + static_cast<int64_t>(r) * a.k + i0;
  for (int t = tid; t < n; t += kThreads) {
    const int32_t val = w_out[t];
    if (err) g_out[t] = -1;
    else if (val != kUnresolved) g_out[t] = val;
  }
  if (!err)
    for (int j = tid; j < mw; j += kThreads) g_out[w_mi[j]] = w_vict[j] & ~static_cast<int32_t>(kAlias);
}

// Leader: the unit's LRU order and slot map into shared memory, and an empty
// duplicate set.  `sp0` is this thread's first 16-byte piece of the slot map
// when it was read ahead (vector rows only).
__device__ void pt_leader_load_state(const PtArgs &a, int r, bool have_sp0, int4 sp0,
                                     unsigned char *smem, const PtLayout &L) {
  const int tid = threadIdx.x;
  int16_t *l_lru = reinterpret_cast<int16_t *>(smem + L.l_lru);
  int32_t *l_slotpos = reinterpret_cast<int32_t *>(smem + L.l_slotpos);
  int32_t *l_hkey = reinterpret_cast<int32_t *>(smem + L.l_hkey);
  const int16_t *g_lru = a.lru + static_cast<int64_t>(r) * a.B;
  const int32_t *g_slotpos = a.slot_pos + static_cast<int64_t>(r) * a.B;
  if (a.B % 8 == 0) {  // 16-byte rows: one vector per 8 LRU / 4 slot entries
    const int4 *g_lru16 = reinterpret_cast<const int4 *>(g_lru);
    const int4 *g_sp16 = reinterpret_cast<const int4 *>(g_slotpos);
    int4 *l_lru16 = reinterpret_cast<int4 *>(l_lru);
    int4 *l_sp16 = reinterpret_cast<int4 *>(l_slotpos);
    for (int c = tid; c < a.B / 4; c += kThreads)
      l_sp16[c] = (have_sp0 && c == tid) ? sp0 : g_sp16[c];
    for (int c = tid; c < a.B / 8; c += kThreads) l_lru16[c] = g_lru16[c];
  } else {
    for (int s = tid; s < a.B; s += kThreads) {
      l_lru[s] = g_lru[s];
      l_slotpos[s] = g_slotpos[s];
    }
  }
  for (int i = tid; i < (1 << a.hcap_log2); i += kThreads) l_hkey[i] = -1;
  if (a.union_mode) {
    int32_t *l_hmin = reinterpret_cast<int32_t *>(smem + L.l_hmin);
    for (int i = tid; i < (1 << a.hcap_log2); i += kThreads) l_hmin[i] = INT32_MAX;
  }
}

// Leader, fused write-through ([DD] §3.4 step 4), first half: keep the
// previous token's row B in shared memory and put the new token's KV in its
// place.  The kept row goes to host row prev in pt_leader_publish, after the
// decision, so that no release on the way there waits for host stores.
__device__ void pt_leader_write_through(const PtArgs &a, int r, int32_t prev, unsigned char *smem,
                                        const PtLayout &L) {
  if (!a.prev_pos && !a.new_rows) return;
  const int tid = threadIdx.x;
  uint4 *rowb = reinterpret_cast<uint4 *>(a.hot + static_cast<int64_t>(r) * a.hot_req_stride +
                                          static_cast<int64_t>(a.B) * a.hot_row_stride);
  const uint4 *nrow = a.new_rows ? reinterpret_cast<const uint4 *>(
                                       a.new_rows + static_cast<int64_t>(r) * a.rec16 * 16)
                                 : nullptr;
  uint4 *keep = reinterpret_cast<uint4 *>(smem + L.l_prevrow);
  if (prev >= a.P && tid == 0) atomicOr(a.status, HISPARSE_ERR_RANGE);
  for (int c = tid; c < a.rec16; c += kThreads) {
    keep[c] = rowb[c];
    if (nrow) rowb[c] = nrow[c];
  }
}

// Short request ([DD] §5.4: with seq_len <= B every token of the request sits
// in the buffer in order and RESOLVE returns slots by position, with no host
// IO; the buffer grows on demand; §5.5: the kernel's fast path returns before
// any LRU work).  Run by the leader CTA alone, the cluster's other CTAs having
// left:
//   1. the fused write-through (row B kept, new token in, kept row to the
//      host pool and its mirror);
//   2. growth: the previous token resolved as a one-entry selection -- a hit
//      moves its slot to the recent end of the LRU order; a miss takes the
//      least recent slot, filled from the kept row (and, inline, the shared
//      layers' rows), mapped, planned, and moved to the recent end;
//   3. the lookup: padding -1, a resident row first, the newest token B, a
//      position in [0, seq_len) its own slot, anything else fails the lookup.
template <bool kRecordPlan>
__device__ void pt_short_path(const PtArgs &a, int r, int32_t prev, int32_t newest,
                              int32_t seq_len, unsigned char *smem, const PtLayout &L) {
  const int tid = threadIdx.x;
  const int B = a.B, k = a.k;
  const int64_t P = a.P;
  int16_t *l_lru = reinterpret_cast<int16_t *>(smem + L.l_lru);
  int32_t *l_out = reinterpret_cast<int32_t *>(smem + L.l_ev);   // k entries
  uint32_t *l_misc = reinterpret_cast<uint32_t *>(smem + L.l_misc);
  int32_t *g_pt = a.page_table + static_cast<int64_t>(r) * P;
  int32_t *g_sp = a.slot_pos + static_cast<int64_t>(r) * B;
  int16_t *g_lru = a.lru + static_cast<int64_t>(r) * B;
  const uint4 *keep = reinterpret_cast<const uint4 *>(smem + L.l_prevrow);

  // (0) every load the three steps need goes out at once: row B and the new
  // token's row, the previous token's page-table entry, the LRU row and the
  // selections (one memory round trip instead of three)
  const bool grow = a.prev_pos && prev >= 0 && prev < P;
  const bool through = a.prev_pos || a.new_rows;
  uint4 *rowb = reinterpret_cast<uint4 *>(a.hot + static_cast<int64_t>(r) * a.hot_req_stride +
                                          static_cast<int64_t>(B) * a.hot_row_stride);
  const uint4 *nrow = a.new_rows ? reinterpret_cast<const uint4 *>(
                                       a.new_rows + static_cast<int64_t>(r) * a.rec16 * 16)
                                 : nullptr;
  uint4 kv = make_uint4(0, 0, 0, 0), nv = make_uint4(0, 0, 0, 0);
  if (through && tid < a.rec16) kv = rowb[tid];
  if (nrow && tid < a.rec16) nv = nrow[tid];
  const int32_t hs0 = (grow && tid == 0) ? g_pt[prev] : -1;
  const bool lru16 = grow && B % 8 == 0;
  int4 lv = make_int4(0, 0, 0, 0);
  if (lru16 && tid < B / 8) lv = reinterpret_cast<const int4 *>(g_lru)[tid];
  int32_t sv[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = tid + u * kThreads;
    sv[u] = i < k ? sel_position<true>(a, r, i) : -1;
  }
  // (1) write-through, first half: row B kept, the new token in its place
  uint4 *keep_w = reinterpret_cast<uint4 *>(smem + L.l_prevrow);
  if (through) {
    for (int c = tid; c < a.rec16; c += kThreads) {
      keep_w[c] = c == tid ? kv : rowb[c];
      if (nrow) rowb[c] = c == tid ? nv : nrow[c];
    }
    if (prev >= P && tid == 0) atomicOr(a.status, HISPARSE_ERR_RANGE);
  }
  if (grow) {
    if (lru16) {
      if (tid < B / 8) reinterpret_cast<int4 *>(l_lru)[tid] = lv;
      for (int c = tid + kThreads; c < B / 8; c += kThreads)
        reinterpret_cast<int4 *>(l_lru)[c] = reinterpret_cast<const int4 *>(g_lru)[c];
    } else {
      for (int j = tid; j < B; j += kThreads) l_lru[j] = g_lru[j];
    }
  }
  if (tid == 0) {
    l_misc[kLErr] = (newest < -1 || newest >= P) ? HISPARSE_ERR_RANGE : 0u;
    l_misc[kLM] = static_cast<uint32_t>(hs0);
    l_misc[kLHits] = 0;
  }
  __syncthreads();
  if (grow) {
    uint4 *hrow = reinterpret_cast<uint4 *>(a.host_w + static_cast<int64_t>(r) * a.host_req_stride +
                                            static_cast<int64_t>(prev) * a.host_row_stride);
    for (int c = tid; c < a.rec16; c += kThreads) st_v4(hrow + c, keep[c]);
    if (a.mirror_w) {
      uint4 *mrow = reinterpret_cast<uint4 *>(a.mirror_w + static_cast<int64_t>(r) * a.host_req_stride +
                                              static_cast<int64_t>(prev) * a.host_row_stride);
      for (int c = tid; c < a.rec16; c += kThreads) st_v4(mrow + c, keep[c]);
    }
    // (2) growth by the previous token
    const int32_t hslot = static_cast<int32_t>(l_misc[kLM]);
    const bool bad = hslot >= B || hslot < -1;   // a corrupt page-table entry
    if (hslot >= 0 && !bad)
      for (int j = tid; j < B; j += kThreads)
        if (l_lru[j] == hslot) l_misc[kLHits] = static_cast<uint32_t>(j);
    __syncthreads();
    if (bad) {
      if (tid == 0) l_misc[kLErr] |= HISPARSE_ERR_RANGE;
    } else {
      const int jm = hslot >= 0 ? static_cast<int>(l_misc[kLHits]) : 0;
      const int16_t moved = hslot >= 0 ? static_cast<int16_t>(hslot) : l_lru[0];
      for (int j = tid; j < B; j += kThreads) g_lru[j] = j < B - 1 ? l_lru[j + (j >= jm)] : moved;
      if (hslot < 0) {   // a miss into the least recent slot
        const int v = moved;
        if (tid == 0) {
          const int32_t old = g_sp[v];
          if (old >= 0) g_pt[old] = -1;
          g_sp[v] = prev;
          g_pt[prev] = v;
          if (kRecordPlan) {
            a.plan_pos[static_cast<int64_t>(r) * k] = prev;
            a.plan_slot[static_cast<int64_t>(r) * k] = v;
          }
        }
        if (a.io) {
          uint4 *row = reinterpret_cast<uint4 *>(a.hot + static_cast<int64_t>(r) * a.hot_req_stride +
                                                 static_cast<int64_t>(v) * a.hot_row_stride);
          for (int c = tid; c < a.rec16; c += kThreads) st_v4(row + c, keep[c]);
          for (int f = 0; f < a.nfl; ++f) {   // the shared-index layers' rows, inline
            const ReplayTarget &T = a.fl[f];
            const uint4 *src = reinterpret_cast<const uint4 *>(
                T.src + static_cast<int64_t>(r) * T.src_req_stride +
                static_cast<int64_t>(prev) * T.src_row_stride);
            uint4 *dst = reinterpret_cast<uint4 *>(T.hot + static_cast<int64_t>(r) * T.hot_req_stride +
                                                   static_cast<int64_t>(v) * T.hot_row_stride);
            for (int c = tid; c < a.rec16; c += kThreads) st_v4(dst + c, ld_nc_v4(src + c));
          }
        }
      }
      if (tid == 0) {
        a.miss_count[r] = hslot < 0 ? 1 : 0;
        a.plan_count[r] = (kRecordPlan && hslot < 0) ? 1 : 0;
      }
    }
  } else if (tid == 0) {
    a.miss_count[r] = 0;
    a.plan_count[r] = 0;
  }
  // (3) the lookup by position
  const int32_t *g_res = a.res_blocks ? a.res_blocks + static_cast<int64_t>(r) * a.res_nblk : nullptr;
  uint32_t err = 0;
  for (int i = tid; i < k; i += kThreads) {
    const int u = (i - tid) / kThreads;
    const int32_t p = u < 2 ? sv[u] : sel_position<true>(a, r, i);
    int32_t v = -1;
    if (p != -1) {
      if (p < -1 || p >= P) {
        err |= HISPARSE_ERR_RANGE;
      } else {
        const int32_t e = (g_res && p / a.res_tok < a.res_nblk) ? g_res[p / a.res_tok] : -1;
        if (e < -1) {
          err |= HISPARSE_ERR_RANGE;
        } else if (e >= 0) {
          const int64_t row = static_cast<int64_t>(e) * a.res_tok + p % a.res_tok;
          if (static_cast<int64_t>(B) + 1 + row > INT32_MAX) err |= HISPARSE_ERR_RANGE;
          else v = static_cast<int32_t>(B + 1 + row);
        } else if (p == newest) {
          v = B;
        } else if (p >= seq_len) {
          err |= HISPARSE_ERR_RANGE;
        } else {
          v = p;   // the slot numbered like the position
        }
      }
    }
    l_out[i] = v;
  }
  if (err) atomicOr(&l_misc[kLErr], err);
  __syncthreads();
  const uint32_t uerr = l_misc[kLErr];
  int32_t *g_out = a.out + static_cast<int64_t>(r) * k;
  for (int i = tid; i < k; i += kThreads) g_out[i] = uerr ? -1 : l_out[i];
  if (tid == 0) {
    a.unit_err[r] = static_cast<int32_t>(uerr);
    if (uerr) atomicOr(a.status, uerr);
  }
}

template <bool kRecordPlan, bool kExt>
__global__ void __launch_bounds__(kThreads, 1) resolve_pt_kernel(const PtArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  // Programmatic dependent launch: this grid may be set up while the previous
  // kernel of the stream finishes, but reads nothing before that kernel has
  // completed; the next kernel may be set up as soon as this one runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int cs = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int r = static_cast<int>(blockIdx.x) / cs;
  const int tid = threadIdx.x;
  const int nw = cs == 1 ? 1 : cs - 1;
  const bool leader = rank == 0;
  const bool worker = cs == 1 || rank > 0;
  const int w = cs == 1 ? 0 : rank - 1;
  const PtLayout L = pt_layout(a.k, a.B, a.ks, 1 << a.hcap_log2, a.rec16 * 16);
  const int i0 = w * a.ks;
  const int n = worker ? max(0, min(a.k, i0 + a.ks) - i0) : 0;
  // The first loads of every role go out together with the batch-size and
  // newest-position reads (all are in bounds for any r < R); the padding check
  // then costs no extra memory round trip.  Workers read their first
  // selections, the leader its first 16-byte pieces of the LRU row and the
  // slot map.
  static_assert(kGroup == 4, "a leader keeps one 16-byte slot-map piece in first[]");
  int32_t first[kGroup] = {-1, -1, -1, -1};
  const bool sp_ahead = !worker && a.B % 8 == 0 && tid < a.B / 4;
  if (worker) {
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int t = u * kThreads + tid;
      first[u] = t < n ? sel_position<kExt>(a, r, i0 + t) : -1;
    }
  } else if (sp_ahead) {
    const int4 v = reinterpret_cast<const int4 *>(a.slot_pos + static_cast<int64_t>(r) * a.B)[tid];
    first[0] = v.x; first[1] = v.y; first[2] = v.z; first[3] = v.w;
  }
  const int32_t newest = a.newest ? a.newest[r] : -1;
  const int32_t prev = a.prev_pos ? a.prev_pos[r] : -1;
  const int32_t seq_len = (kExt && a.seq_lens) ? a.seq_lens[r] : INT32_MAX;
  const int nreq = a.num_reqs ? min(*a.num_reqs, a.R) : a.R;
  if (r >= nreq) return;  // graph padding: every CTA of the cluster leaves
  if (kExt && seq_len <= a.B) {  // a short request: the leader alone, no cluster barrier
    if (leader) pt_short_path<kRecordPlan>(a, r, prev, newest, seq_len, smem, L);
    return;
  }
  // the previous token's record, when filled from row B, is not read from the host
  const int32_t skip_pos = (a.prev_from_row && prev >= 0) ? prev : -2;

  const char *src = a.src + static_cast<int64_t>(r) * a.src_req_stride;
  char *dst = a.hot + static_cast<int64_t>(r) * a.hot_req_stride;

  if (cs == 1) {
    // one CTA plays every role in order; nothing to overlap, nothing staged
    pt_leader_load_state(a, r, false, make_int4(0, 0, 0, 0), smem, L);
    pt_leader_write_through(a, r, prev, smem, L);
    const int mw = pt_worker_classify<kExt>(a, r, i0, n, newest, first, smem, L);
    pt_worker_order(a, 0, mw, smem, L);
    pt_leader_decide<kExt>(a, cs, nw, newest, smem, L);
    __syncthreads();
    pt_leader_push<kExt>(a, cs, nw, smem, L);
    pt_leader_publish<kRecordPlan>(a, r, prev, skip_pos, smem, L);
    __syncthreads();
    pt_worker_finish(a, r, i0, n, skip_pos, 0, nullptr, src, dst, smem, L);
    return;
  }
  if (leader) {
    // #0: the leader publishes nothing here, so it arrives at once and reads
    // its state while the workers classify their slices
    cluster_arrive_relaxed();
    pt_leader_load_state(a, r, sp_ahead, make_int4(first[0], first[1], first[2], first[3]), smem,
                         L);
    pt_leader_write_through(a, r, prev, smem, L);
    __syncthreads();
    cluster_wait_acquire();    //    the slices are ready
    pt_leader_decide<kExt>(a, cs, nw, newest, smem, L);
    __syncthreads();
    pt_leader_push<kExt>(a, cs, nw, smem, L);
    __syncthreads();
    cluster_arrive_release();  // #1: the verdict and victims, in the workers' memory
    pt_leader_publish<kRecordPlan>(a, r, prev, skip_pos, smem, L);
    cluster_wait_acquire();    //    (no CTA touches another's memory after #1)
    return;
  }
  // worker
  const int mw = pt_worker_classify<kExt>(a, r, i0, n, newest, first, smem, L);
  // #0: the slice, for the leader.  The block barrier that ends the
  // classification orders every thread's shared-memory writes before the last
  // warp's cluster-scope fence, which releases them all; the other warps
  // arrive without a fence, so their host loads below do not wait on one.
  if (tid >= kThreads - 32) fence_acq_rel_cluster();
  cluster_arrive_relaxed();
  // Read the slice's first missed records into registers now, in list order,
  // before any victim is known: the reads fly while the leader decides.
  const int32_t *w_mp = reinterpret_cast<const int32_t *>(smem + L.w_mp);
  const int staged = a.io ? min(mw, kStage * kThreads / a.rec16) : 0;
  const int64_t totc = static_cast<int64_t>(staged) * a.rec16;
  uint4 v[kStage];
#pragma unroll
  for (int u = 0; u < kStage; ++u) {
    const int64_t q = tid + static_cast<int64_t>(u) * kThreads;
    if (q < totc) {
      const uint32_t q32 = static_cast<uint32_t>(q);
      const int f = static_cast<int>(q32 / static_cast<uint32_t>(a.rec16));
      const int o = static_cast<int>(q32 - static_cast<uint32_t>(f) * a.rec16);
      const int32_t pm = w_mp[f];
      if (pm != skip_pos) v[u] = ld_nc_v4(src + static_cast<int64_t>(pm) * a.src_row_stride + 16 * o);
    }
  }
  pt_worker_order(a, staged, mw, smem, L);  // the rest go out in host-row order later
  cluster_wait_acquire();
  cluster_arrive_relaxed();  // #1: nothing new to publish; the staged loads stay in flight
  cluster_wait_acquire();    //    the leader's decision is visible
  pt_worker_finish(a, r, i0, n, skip_pos, staged, v, src, dst, smem, L);
}

// ---------------------------------------------------------------------------
// Write-through: grid (R, layers); copies hot row B to host row pos.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) writeback_kernel(const WritebackArgs a) {
  const int r = blockIdx.x, li = blockIdx.y;
  const int nreq = a.num_reqs ? min(*a.num_reqs, a.R) : a.R;
  if (r >= nreq) return;
  const int32_t p = a.pos[static_cast<int64_t>(li) * a.R + r];
  const LayerDev &Ld = a.layers[a.layer0 + li];
  uint4 *row = reinterpret_cast<uint4 *>(Ld.hot + static_cast<int64_t>(r) * Ld.hot_req_stride +
                                         static_cast<int64_t>(a.B) * Ld.hot_row_stride);
  const bool wb = p >= 0 && p < a.P;
  if (p >= a.P && threadIdx.x == 0) atomicOr(a.status, HISPARSE_ERR_RANGE);
  uint4 *d = reinterpret_cast<uint4 *>(Ld.host_w + static_cast<int64_t>(r) * Ld.host_req_stride +
                                       static_cast<int64_t>(wb ? p : 0) * Ld.host_row_stride);
  const uint4 *nr = a.new_rows ? reinterpret_cast<const uint4 *>(
                                     a.new_rows + (static_cast<int64_t>(li) * a.R + r) * a.rec16 * 16)
                               : nullptr;
  uint4 *m = Ld.mirror ? reinterpret_cast<uint4 *>(Ld.mirror + static_cast<int64_t>(r) * Ld.host_req_stride +
                                                   static_cast<int64_t>(wb ? p : 0) * Ld.host_row_stride)
                       : nullptr;
  // each thread moves its own chunks: old row B out first (to the host pool and
  // its HBM mirror), then the new token in
  for (int c = threadIdx.x; c < a.rec16; c += blockDim.x) {
    const uint4 v = row[c];
    if (wb) {
      st_v4(d + c, v);
      if (m) st_v4(m + c, v);
    }
    if (nr) row[c] = nr[c];
  }
}

// ---------------------------------------------------------------------------
// Plan replay for a shared-index layer ([DD] §3.6, §5.6).  The plan's records
// (every request's, back to back) are split evenly over a small grid; a CTA
// resolves a batch of its records to source and destination rows once, into
// shared memory, then streams the batch's 16-byte chunks with kReplayDepth
// host loads in flight per thread.  Nothing on the load path waits on a global
// read of the plan.  (Reading each batch in source-address order was measured
// to change nothing: a plan record's rows are on distinct 64 KB host pages in
// any order.)
// ---------------------------------------------------------------------------
constexpr int kReplayThreads = 512;
constexpr int kReplayBatch = 512;  // plan records resolved to rows per round
constexpr int kReplayDepth = 8;    // 16-byte host loads in flight per thread

__host__ __device__ inline int replay_pref_bytes(int R) { return ((R + 1) * 4 + 15) & ~15; }
__host__ __device__ inline size_t replay_smem_bytes(int R) {
  // prefix [R + 1], then source and destination rows of a batch
  return static_cast<size_t>(replay_pref_bytes(R)) + 2 * sizeof(char *) * kReplayBatch;
}

__global__ void __launch_bounds__(kReplayThreads) replay_kernel(const ReplayArgs a) {
  extern __shared__ __align__(16) unsigned char rsm[];
  int32_t *s_pref = reinterpret_cast<int32_t *>(rsm);  // [R + 1] exclusive prefix of plan counts
  const char **s_src = reinterpret_cast<const char **>(rsm + replay_pref_bytes(a.R));  // [kReplayBatch]
  char **s_dst = reinterpret_cast<char **>(rsm + replay_pref_bytes(a.R) + sizeof(char *) * kReplayBatch);
  const int tid = threadIdx.x;
  const int nreq = a.num_reqs ? min(*a.num_reqs, a.R) : a.R;
  if (tid < 32) {
    int run = 0;
    for (int r0 = 0; r0 < nreq; r0 += 32) {
      const int r = r0 + tid;
      int v = r < nreq ? a.plan_count[r] : 0, inc = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(kFull, inc, d);
        if (tid >= d) inc += t;
      }
      if (r < nreq) s_pref[r] = run + inc - v;
      run += __shfl_sync(kFull, inc, 31);
    }
    if (tid == 0) s_pref[nreq] = run;
  }
  __syncthreads();
  // Work items are (plan record, target) pairs, the targets of one record
  // next to each other: with the group's layers interleaved in the host pool,
  // consecutive items read adjacent host rows of one page.
  const int nf = a.nf;
  const int64_t W = static_cast<int64_t>(s_pref[nreq]) * nf;
  const int64_t w0 = W * blockIdx.x / gridDim.x, w1 = W * (blockIdx.x + 1) / gridDim.x;
  const uint32_t rec16 = static_cast<uint32_t>(a.rec16);
  for (int64_t b0 = w0; b0 < w1; b0 += kReplayBatch) {
    const int nb = static_cast<int>(min(static_cast<int64_t>(kReplayBatch), w1 - b0));
    for (int i = tid; i < nb; i += kReplayThreads) {
      const int64_t item = b0 + i;
      const int m = static_cast<int>(item / nf), f = static_cast<int>(item - int64_t(m) * nf);
      int lo = 0, hi = nreq - 1;  // the request: last r with s_pref[r] <= m
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pref[mid] <= m) lo = mid; else hi = mid - 1;
      }
      const int64_t pk = static_cast<int64_t>(lo) * a.k + (m - s_pref[lo]);
      const ReplayTarget &T = a.f[f];
      s_src[i] = T.src + static_cast<int64_t>(lo) * T.src_req_stride +
                 static_cast<int64_t>(a.plan_pos[pk]) * T.src_row_stride;
      s_dst[i] = T.hot + static_cast<int64_t>(lo) * T.hot_req_stride +
                 static_cast<int64_t>(a.plan_slot[pk]) * T.hot_row_stride;
    }
    __syncthreads();
    const uint32_t n = static_cast<uint32_t>(nb) * rec16;
    for (uint32_t q0 = tid; q0 < n; q0 += kReplayThreads * kReplayDepth) {
      uint4 v[kReplayDepth];
      char *d[kReplayDepth];
#pragma unroll
      for (int u = 0; u < kReplayDepth; ++u) {
        const uint32_t q = q0 + u * kReplayThreads;
        d[u] = nullptr;
        if (q < n) {
          const uint32_t i = q / rec16, o = q - i * rec16;
          v[u] = ld_nc_v4(s_src[i] + 16 * o);
          d[u] = s_dst[i] + 16 * o;
        }
      }
#pragma unroll
      for (int u = 0; u < kReplayDepth; ++u)
        if (d[u]) st_v4(d[u], v[u]);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Copy by SM threads (hisparse_copy): 16-byte loads and stores, 4 in flight
// per thread.  For the small per-step transfers between pinned host memory
// and HBM over the coherent host link, this has less latency than a copy
// engine.  Launched with programmatic dependent launch: it waits for the
// previous kernel of the stream, and lets the next one be set up at once.
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;
constexpr int kCopyMaxCtas = 128;  // 2 MB in flight at most (32 CTAs measured no better)
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint4 *dst, const uint4 *src, int64_t n) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCopyThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = ld_nc_v4(src + i), b = ld_nc_v4(src + i + stride);
    const uint4 c = ld_nc_v4(src + i + 2 * stride), d = ld_nc_v4(src + i + 3 * stride);
    st_v4(dst + i, a);
    st_v4(dst + i + stride, b);
    st_v4(dst + i + 2 * stride, c);
    st_v4(dst + i + 3 * stride, d);
  }
  for (; i < n; i += stride) st_v4(dst + i, ld_nc_v4(src + i));
}

// Reset: slot_pos = -1, lru = 0..B-1 for `n` units; page table -1 via memset.
__global__ void reset_kernel(int32_t *slot_pos, int16_t *lru, int64_t n_units, int32_t B) {
  const int64_t total = n_units * B;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    slot_pos[i] = -1;
    lru[i] = static_cast<int16_t>(i % B);
  }
}

// ---------------------------------------------------------------------------
// Admission ([DD] §5.3, direct admission): listed requests go to the reset
// state; a short request's first n positions are preloaded into slots 0..n-1
// in order, the state that resolving positions 0..n-1 in order from the reset
// state gives (slot s holds position s; LRU: empty slots, then the preloaded
// ones).  Grid (listed requests, C): block (i, c) does the c-th share of the
// request's page table and of its preload copy.
// ---------------------------------------------------------------------------
struct AdmitArgs {
  const int32_t *reqs, *preload;
  int32_t R, B, rec16;
  int64_t P;
  int32_t *slot_pos;  // metadata of a RESOLVE layer; NULL for a shared-index layer
  int16_t *lru;
  int32_t *page_table, *miss_count, *unit_err, *plan_count;
  uint32_t *status;
  const char *src;
  int64_t src_req_stride, src_row_stride;
  char *hot;
  int64_t hot_req_stride, hot_row_stride;
};
constexpr int kAdmitThreads = 256;

__global__ void __launch_bounds__(kAdmitThreads) admit_kernel(const AdmitArgs a) {
  const int i = blockIdx.x, c = blockIdx.y, C = gridDim.y, tid = threadIdx.x;
  const int r = a.reqs[i];
  const int n = a.preload ? a.preload[i] : 0;
  if (r < 0 || r >= a.R || n < 0 || n > a.B || n > a.P) {
    if (c == 0 && tid == 0) atomicOr(a.status, HISPARSE_ERR_RANGE);
    return;
  }
  if (a.slot_pos) {
    int32_t *pt = a.page_table + static_cast<int64_t>(r) * a.P;
    for (int64_t p = static_cast<int64_t>(c) * kAdmitThreads + tid; p < a.P;
         p += static_cast<int64_t>(C) * kAdmitThreads)
      pt[p] = p < n ? static_cast<int32_t>(p) : -1;
    if (c == 0) {
      int32_t *sp = a.slot_pos + static_cast<int64_t>(r) * a.B;
      int16_t *lru = a.lru + static_cast<int64_t>(r) * a.B;
      for (int s = tid; s < a.B; s += kAdmitThreads) {
        sp[s] = s < n ? s : -1;
        lru[s] = static_cast<int16_t>(s < a.B - n ? n + s : s - (a.B - n));
      }
      if (tid == 0) {
        a.miss_count[r] = 0;
        a.unit_err[r] = 0;
        a.plan_count[r] = 0;
      }
    }
  }
  const char *src = a.src + static_cast<int64_t>(r) * a.src_req_stride;
  char *dst = a.hot + static_cast<int64_t>(r) * a.hot_req_stride;
  const int64_t total = static_cast<int64_t>(n) * a.rec16;
  const int64_t T = static_cast<int64_t>(C) * kAdmitThreads;
  for (int64_t b0 = static_cast<int64_t>(c) * kAdmitThreads + tid; b0 < total; b0 += T * kUnroll) {
    uint4 v[kUnroll];
    char *d[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t q = b0 + u * T;
      d[u] = nullptr;
      if (q < total) {
        const int64_t s = q / a.rec16, o = q - s * a.rec16;
        v[u] = ld_nc_v4(src + s * a.src_row_stride + 16 * o);
        d[u] = dst + s * a.hot_row_stride + 16 * o;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (d[u]) st_v4(d[u], v[u]);
  }
}

}  // namespace

// ===========================================================================
// Host side
// ===========================================================================
struct AnchorMeta {
  int32_t *slot_pos = nullptr;
  int16_t *lru = nullptr;
  int32_t *page_table = nullptr;
  int32_t *miss_count = nullptr;
  int32_t *unit_err = nullptr;
  int32_t *plan_pos = nullptr;
  int32_t *plan_slot = nullptr;
  int32_t *plan_count = nullptr;
};

struct hisparse_handle {
  int32_t R, L, k, B, rec;
  int64_t P;
  int32_t cs, cap_log2, replay_ctas, sm_count, device, lookup, ks;
  uint32_t smem;
  float l2_hit_ratio = 0.f;   // > 0: RESOLVE launches keep the page table persisting in L2
  bool l2_limit_saved = false;
  size_t l2_prev_limit = 0;   // the persisting-L2 limit before this handle changed it
  std::vector<int32_t> anchor_of;
  std::vector<LayerDev> layers;
  std::vector<int32_t> bucket_shift, nbuckets;  // per layer: fetch-order buckets
  std::vector<AnchorMeta> meta;
  LayerDev *d_layers = nullptr;
  uint32_t *d_status = nullptr;
  int32_t *d_unit_err_all = nullptr;  // [L][R]
  void *arena = nullptr;
  int64_t arena_bytes = 0;
};

namespace {

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return HISPARSE_ECUDA;
}
#define HS_CUDA(call)                              \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_);   \
  } while (0)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int layer_ok(const hisparse_handle *h, int32_t layer) {
  if (!h || layer < 0 || layer >= h->L) return HISPARSE_EINVAL;
  return HISPARSE_OK;
}

int slice_size(int k, int cs) {
  const int nw = cs == 1 ? 1 : cs - 1;
  return (k + nw - 1) / nw;
}

uint32_t resolve_smem(const hisparse_handle *h, int cs) {
  if (h->lookup == HISPARSE_LOOKUP_HASH) return smem_layout(h->k, h->B, 1 << h->cap_log2).total;
  return pt_layout(h->k, h->B, slice_size(h->k, cs), 1 << h->cap_log2, h->rec).total;
}

// Choose the cluster size: as many CTAs per request as the GPU can run at once
// for the whole batch (one wave), at most 16.
int configure_resolve(hisparse_handle *h, int want_cs) {
  const bool hash = h->lookup == HISPARSE_LOOKUP_HASH;
  const void *fns[4];
  int nf = 2;
  if (hash) {
    fns[0] = reinterpret_cast<const void *>(&resolve_kernel<false>);
    fns[1] = reinterpret_cast<const void *>(&resolve_kernel<true>);
  } else {
    fns[0] = reinterpret_cast<const void *>(&resolve_pt_kernel<false, false>);
    fns[1] = reinterpret_cast<const void *>(&resolve_pt_kernel<true, false>);
    fns[2] = reinterpret_cast<const void *>(&resolve_pt_kernel<false, true>);
    fns[3] = reinterpret_cast<const void *>(&resolve_pt_kernel<true, true>);
    nf = 4;
  }
  // Dynamic + static shared memory must stay within the device's opt-in limit
  // per block.  The layout shrinks with the cluster size (a worker's slice is
  // k / (cs - 1) selections), so a cluster size is a candidate only if its
  // layout fits; the attribute covers the largest candidate.
  int optin = 0;
  HS_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device));
  size_t stat = 0;
  for (int i = 0; i < nf; ++i) {
    cudaFuncAttributes fa;
    HS_CUDA(cudaFuncGetAttributes(&fa, fns[i]));
    stat = std::max(stat, fa.sharedSizeBytes);
  }
  auto fits = [&](int cs) {
    return static_cast<size_t>(resolve_smem(h, cs)) + stat <= static_cast<size_t>(optin);
  };
  uint32_t smax = 0;
  for (int cs = 1; cs <= 16; ++cs)
    if (fits(cs)) smax = std::max(smax, resolve_smem(h, cs));
  if (smax == 0) return HISPARSE_EBOUND;
  for (int i = 0; i < nf; ++i) {
    HS_CUDA(cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smax));
    HS_CUDA(cudaFuncSetAttribute(fns[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
  }
  auto active_clusters = [&](int cs) -> int {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(cs) * h->R);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = resolve_smem(h, cs);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fns[1], &lc) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  };
  int cs = 0;
  if (want_cs > 0) {
    if (want_cs > 16 || !fits(want_cs)) return HISPARSE_EBOUND;
    if (active_clusters(want_cs) < 1) return HISPARSE_EBOUND;
    cs = want_cs;
  } else {
    for (int c = std::min(16, h->sm_count / h->R); c >= 2; --c) {
      if (fits(c) && active_clusters(c) >= h->R) {
        cs = c;
        break;
      }
    }
    // else one CTA per request; with a layout too large for that, the largest
    // cluster that fits and runs at all
    if (cs == 0 && fits(1)) cs = 1;
    for (int c = 16; cs == 0 && c >= 2; --c)
      if (fits(c) && active_clusters(c) >= 1) cs = c;
    if (cs == 0) return HISPARSE_EBOUND;
  }
  h->cs = cs;
  h->smem = resolve_smem(h, cs);
  h->ks = slice_size(h->k, cs);
  return HISPARSE_OK;
}

// Host pools allocated by hisparse_host_alloc through cudaHostRegister.
std::mutex g_host_mu;
std::map<void *, size_t> g_host_regs;

constexpr int kMadvCollapse = 25;  // Linux MADV_COLLAPSE (6.1+); ignored where unknown

// Size of a transparent huge page (0 if the kernel does not say).
size_t thp_bytes() {
  FILE *f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r");
  if (!f) return 0;
  unsigned long long v = 0;
  if (std::fscanf(f, "%llu", &v) != 1) v = 0;
  std::fclose(f);
  return static_cast<size_t>(v);
}

// Zero-fill with a few threads so the pages are populated after the advice.
void first_touch(void *p, size_t bytes) {
  const unsigned n = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
  std::vector<std::thread> th;
  const size_t chunk = (bytes / n + 4095) & ~size_t(4095);
  for (unsigned i = 0; i < n; ++i) {
    const size_t b = std::min(bytes, i * chunk), e = std::min(bytes, b + chunk);
    if (b >= e) break;
    th.emplace_back([=] { std::memset(static_cast<char *>(p) + b, 0, e - b); });
  }
  for (auto &t : th) t.join();
}

// Turn the handle's L2 window off: persisting lines back to normal and the
// context's set-aside back to what it was before the handle changed it.
int l2_persisting_off(hisparse_handle *h) {
  h->l2_hit_ratio = 0.f;
  if (!h->l2_limit_saved) return HISPARSE_OK;
  HS_CUDA(cudaCtxResetPersistingL2Cache());
  HS_CUDA(cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, h->l2_prev_limit));
  h->l2_limit_saved = false;
  return HISPARSE_OK;
}

}  // namespace

extern "C" {

int hisparse_last_cuda_error(void) { return g_last_cuda_error; }

const char *hisparse_strerror(int code) {
  switch (code) {
    case HISPARSE_OK: return "ok";
    case HISPARSE_EINVAL: return "invalid argument";
    case HISPARSE_EBOUND: return "size outside supported bounds";
    case HISPARSE_ENOMEM: return "out of memory";
    case HISPARSE_ECUDA: return "CUDA call failed";
    case HISPARSE_EROLE: return "layer role mismatch (anchor / shared layer)";
    default: return "unknown error";
  }
}

int hisparse_host_alloc(size_t bytes, void **out) {
  return hisparse_host_alloc_kind(bytes, HISPARSE_HOST_PINNED, out);
}

int hisparse_host_alloc_kind(size_t bytes, int32_t kind, void **out) {
  if (!out || bytes == 0) return HISPARSE_EINVAL;
  if (kind != HISPARSE_HOST_HUGE && kind != HISPARSE_HOST_PINNED) return HISPARSE_EINVAL;
  *out = nullptr;
  // Large pools: transparent-huge-page backed memory registered with the GPU.
  // The GPU then maps the pool with large pages, so random record fetches
  // miss its address-translation caches far less often than with
  // cudaHostAlloc's base-page mappings.
  const size_t hp = kind == HISPARSE_HOST_HUGE ? thp_bytes() : 0;
  if (hp && bytes >= hp) {
    const size_t sz = (bytes + hp - 1) / hp * hp;
    void *p = nullptr;
    if (posix_memalign(&p, hp, sz) == 0) {
      madvise(p, sz, MADV_HUGEPAGE);  // advice only: a refusal still leaves valid memory
      first_touch(p, sz);
      madvise(p, sz, kMadvCollapse);  // ask for huge pages now where the first touch got none
      // A fork() of this process would split every pinned huge page of the
      // pool into base pages in the parent (pinned pages cannot be shared
      // copy-on-write), and the GPU would then stall on translation misses.
      // Children never need the pool.
      madvise(p, sz, MADV_DONTFORK);
      cudaError_t e = cudaHostRegister(p, sz, cudaHostRegisterMapped | cudaHostRegisterPortable);
      if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lk(g_host_mu);
        g_host_regs[p] = sz;
        *out = p;
        return HISPARSE_OK;
      }
      cudaGetLastError();
      free(p);
    }
  }
  cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();
    *out = nullptr;
    return HISPARSE_ENOMEM;
  }
  return HISPARSE_OK;
}

int hisparse_host_hugepage_bytes(const void *p, size_t bytes, size_t *huge_out) {
  if (!p || !huge_out) return HISPARSE_EINVAL;
  *huge_out = 0;
  FILE *f = std::fopen("/proc/self/smaps", "r");
  if (!f) return HISPARSE_EINVAL;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p), hi = lo + bytes;
  char line[512];
  bool in = false;
  unsigned long long a = 0, b = 0, kb = 0;
  while (std::fgets(line, sizeof line, f)) {
    if (std::sscanf(line, "%llx-%llx", &a, &b) == 2 && std::strchr(line, '-') &&
        std::strchr(line, ' ') > std::strchr(line, '-')) {
      in = a < hi && b > lo;  // a mapping that overlaps the range
      continue;
    }
    if (in && std::sscanf(line, "AnonHugePages: %llu kB", &kb) == 1) *huge_out += kb * 1024ull;
  }
  std::fclose(f);
  if (*huge_out > bytes) *huge_out = bytes;
  return HISPARSE_OK;
}

int hisparse_host_free(void *p) {
  if (!p) return HISPARSE_EINVAL;
  bool registered = false;
  {
    std::lock_guard<std::mutex> lk(g_host_mu);
    auto it = g_host_regs.find(p);
    if (it != g_host_regs.end()) {
      registered = true;
      g_host_regs.erase(it);
    }
  }
  if (registered) {
    HS_CUDA(cudaHostUnregister(p));
    free(p);
    return HISPARSE_OK;
  }
  HS_CUDA(cudaFreeHost(p));
  return HISPARSE_OK;
}

int hisparse_init(const hisparse_config *cfg, const hisparse_layer_buffers *layers,
                  hisparse_handle **out) {
  if (!cfg || !layers || !out) return HISPARSE_EINVAL;
  *out = nullptr;
  const int32_t R = cfg->num_requests, L = cfg->num_layers, k = cfg->top_k, B = cfg->buffer_slots;
  const int64_t P = cfg->host_rows;
  const int32_t rec = cfg->record_bytes;
  if (R < 1 || L < 1 || k < 1 || P < 1) return HISPARSE_EINVAL;
  if (rec <= 0 || rec % 16) return HISPARSE_EINVAL;
  if (R > 8192 || L > 4096 || B < k || B > 32767 || P > INT32_MAX) return HISPARSE_EBOUND;
  // chunk indices of one launch's fetches stay below 2^31 (32-bit index math)
  if (static_cast<int64_t>(R) * k * (rec / 16) >= (int64_t(1) << 31)) return HISPARSE_EBOUND;
  if (cfg->ctas_per_request < 0 || cfg->ctas_per_request > 16 || cfg->replay_ctas < 0)
    return HISPARSE_EBOUND;
  if (cfg->lookup != HISPARSE_LOOKUP_PAGE_TABLE && cfg->lookup != HISPARSE_LOOKUP_HASH)
    return HISPARSE_EINVAL;
  std::vector<int32_t> anchor(L, -1);
  if (cfg->anchor_of) {
    for (int l = 0; l < L; ++l) anchor[l] = cfg->anchor_of[l];
    for (int l = 0; l < L; ++l) {
      const int a = anchor[l];
      if (a == -1) continue;
      if (a < 0 || a >= L || a == l || anchor[a] != -1) return HISPARSE_EROLE;
    }
  }
  for (int l = 0; l < L; ++l) {
    const hisparse_layer_buffers &b = layers[l];
    if (!b.host_pool || !b.hot) return HISPARSE_EINVAL;
    if (!aligned16(b.host_pool) || !aligned16(b.hot) || (b.mirror && !aligned16(b.mirror)))
      return HISPARSE_EINVAL;
    if (b.host_req_stride % 16 || b.host_row_stride % 16 || b.hot_req_stride % 16 ||
        b.hot_row_stride % 16)
      return HISPARSE_EINVAL;
    if (b.host_row_stride < rec || b.hot_row_stride < rec || b.host_req_stride < 0 ||
        b.hot_req_stride < 0)
      return HISPARSE_EINVAL;
  }

  hisparse_handle *h = new (std::nothrow) hisparse_handle();
  if (!h) return HISPARSE_ENOMEM;
  h->R = R; h->L = L; h->k = k; h->B = B; h->P = P; h->rec = rec;
  h->lookup = cfg->lookup;
  h->anchor_of = anchor;
  int cap_log2 = 1;
  while ((1 << cap_log2) < 2 * k) ++cap_log2;
  h->cap_log2 = cap_log2;
  int rc = HISPARSE_OK;
  auto fail = [&](int code) {
    hisparse_destroy(h);
    return code;
  };
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  h->replay_ctas = cfg->replay_ctas > 0 ? cfg->replay_ctas : 16;

  // device-visible addresses of the host pools
  h->layers.resize(L);
  for (int l = 0; l < L; ++l) {
    const hisparse_layer_buffers &b = layers[l];
    void *dp = nullptr;
    e = cudaHostGetDevicePointer(&dp, b.host_pool, 0);
    if (e != cudaSuccess) {
      cudaGetLastError();
      g_last_cuda_error = static_cast<int>(e);
      return fail(HISPARSE_EINVAL);  // not pinned + mapped host memory
    }
    LayerDev &d = h->layers[l];
    d.host = static_cast<const char *>(dp);
    d.host_w = static_cast<char *>(dp);
    d.host_req_stride = b.host_req_stride;
    d.host_row_stride = b.host_row_stride;
    d.hot = static_cast<char *>(b.hot);
    d.hot_req_stride = b.hot_req_stride;
    d.hot_row_stride = b.hot_row_stride;
    d.mirror = static_cast<char *>(b.mirror);
  }

  // Fetch-order buckets: about 2 MB of host rows each, at most kMaxBuckets.
  h->bucket_shift.resize(L);
  h->nbuckets.resize(L);
  for (int l = 0; l < L; ++l) {
    const int64_t rows = std::max<int64_t>(1, (int64_t(2) << 20) / layers[l].host_row_stride);
    int sh = 0;
    while ((int64_t(1) << (sh + 1)) <= rows) ++sh;
    while (((P - 1) >> sh) + 1 > kMaxBuckets) ++sh;
    h->bucket_shift[l] = sh;
    h->nbuckets[l] = static_cast<int32_t>(((P - 1) >> sh) + 1);
  }

  rc = configure_resolve(h, cfg->ctas_per_request);
  if (rc != HISPARSE_OK) return fail(rc);
  e = cudaFuncSetAttribute(replay_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(replay_smem_bytes(R)));
  if (e != cudaSuccess) return fail(cuda_fail(e));

  // one arena for all metadata
  auto al = [](int64_t x) { return (x + 255) & ~int64_t(255); };
  int64_t per_anchor = al(4LL * R * B) + al(2LL * R * B) + al(4LL * R * P) + 3 * al(4LL * R) +
                       2 * al(4LL * R * k);
  int n_anchor = 0;
  for (int l = 0; l < L; ++l) n_anchor += anchor[l] == -1;
  const int64_t bytes = per_anchor * n_anchor + al(4LL * L * R) + al(sizeof(LayerDev) * L) + 256;
  e = cudaMalloc(&h->arena, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_last_cuda_error = static_cast<int>(e);
    return fail(HISPARSE_ENOMEM);
  }
  h->arena_bytes = bytes;
  char *cur = static_cast<char *>(h->arena);
  auto take = [&](int64_t n) {
    char *p = cur;
    cur += al(n);
    return p;
  };
  h->d_status = reinterpret_cast<uint32_t *>(take(256));
  h->d_unit_err_all = reinterpret_cast<int32_t *>(take(4LL * L * R));
  h->d_layers = reinterpret_cast<LayerDev *>(take(sizeof(LayerDev) * L));
  h->meta.resize(L);
  for (int l = 0; l < L; ++l) {
    if (anchor[l] != -1) continue;
    AnchorMeta &m = h->meta[l];
    m.slot_pos = reinterpret_cast<int32_t *>(take(4LL * R * B));
    m.lru = reinterpret_cast<int16_t *>(take(2LL * R * B));
    m.page_table = reinterpret_cast<int32_t *>(take(4LL * R * P));
    m.miss_count = reinterpret_cast<int32_t *>(take(4LL * R));
    m.unit_err = h->d_unit_err_all + static_cast<int64_t>(l) * R;
    m.plan_count = reinterpret_cast<int32_t *>(take(4LL * R));
    take(4LL * R);
    m.plan_pos = reinterpret_cast<int32_t *>(take(4LL * R * k));
    m.plan_slot = reinterpret_cast<int32_t *>(take(4LL * R * k));
  }
  e = cudaMemset(h->arena, 0, bytes);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  e = cudaMemcpy(h->d_layers, h->layers.data(), sizeof(LayerDev) * L, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  rc = hisparse_reset(h, -1, nullptr);
  if (rc != HISPARSE_OK) return fail(rc);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(cuda_fail(e));
  *out = h;
  return HISPARSE_OK;
}

int hisparse_destroy(hisparse_handle *h) {
  if (!h) return HISPARSE_EINVAL;
  int rc = l2_persisting_off(h);
  if (h->arena) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaFree(h->arena);
    if (e != cudaSuccess) rc = cuda_fail(e);
  }
  delete h;
  return rc;
}

int hisparse_reset(hisparse_handle *h, int32_t layer, void *stream) {
  if (!h) return HISPARSE_EINVAL;
  if (layer != -1) {
    if (layer_ok(h, layer)) return HISPARSE_EINVAL;
    if (h->anchor_of[layer] != -1) return HISPARSE_EROLE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int l = 0; l < h->L; ++l) {
    if (h->anchor_of[l] != -1 || (layer != -1 && l != layer)) continue;
    const AnchorMeta &m = h->meta[l];
    HS_CUDA(cudaMemsetAsync(m.page_table, 0xff, sizeof(int32_t) * h->R * h->P, s));
    HS_CUDA(cudaMemsetAsync(m.miss_count, 0, sizeof(int32_t) * h->R, s));
    HS_CUDA(cudaMemsetAsync(m.plan_count, 0, sizeof(int32_t) * h->R, s));
    HS_CUDA(cudaMemsetAsync(m.unit_err, 0, sizeof(int32_t) * h->R, s));
    const int64_t n = static_cast<int64_t>(h->R) * h->B;
    const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
    reset_kernel<<<grid, 256, 0, s>>>(m.slot_pos, m.lru, h->R, h->B);
    HS_CUDA(cudaGetLastError());
  }
  return HISPARSE_OK;
}

int hisparse_admit(hisparse_handle *h, int32_t layer, const int32_t *d_reqs, int32_t n,
                   const int32_t *d_preload, void *stream) {
  if (!h || !d_reqs || n < 0) return HISPARSE_EINVAL;
  if (layer != -1 && layer_ok(h, layer)) return HISPARSE_EINVAL;
  if (n == 0) return HISPARSE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int l = 0; l < h->L; ++l) {
    if (layer != -1 && l != layer) continue;
    const LayerDev &Ld = h->layers[l];
    AdmitArgs a = {};
    a.reqs = d_reqs; a.preload = d_preload;
    a.R = h->R; a.B = h->B; a.rec16 = h->rec / 16; a.P = h->P;
    if (h->anchor_of[l] == -1) {
      const AnchorMeta &m = h->meta[l];
      a.slot_pos = m.slot_pos; a.lru = m.lru; a.page_table = m.page_table;
      a.miss_count = m.miss_count; a.unit_err = m.unit_err; a.plan_count = m.plan_count;
    }
    a.status = h->d_status;
    a.src = Ld.host; a.src_req_stride = Ld.host_req_stride; a.src_row_stride = Ld.host_row_stride;
    a.hot = Ld.hot; a.hot_req_stride = Ld.hot_req_stride; a.hot_row_stride = Ld.hot_row_stride;
    admit_kernel<<<dim3(static_cast<unsigned>(n), 16), kAdmitThreads, 0, s>>>(a);
    HS_CUDA(cudaGetLastError());
  }
  return HISPARSE_OK;
}

int hisparse_resolve(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                     const int32_t *d_num_reqs, const int32_t *d_newest, int32_t *d_out,
                     uint32_t flags, void *stream) {
  return hisparse_resolve_step(h, layer, d_sel, d_num_reqs, d_newest, nullptr, nullptr, d_out,
                               flags, stream);
}

int hisparse_resolve_step(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                          const int32_t *d_num_reqs, const int32_t *d_newest,
                          const int32_t *d_prev_pos, const void *d_new_rows, int32_t *d_out,
                          uint32_t flags, void *stream) {
  hisparse_resolve_options o = {};
  o.d_prev_pos = d_prev_pos;
  o.d_new_rows = d_new_rows;
  return hisparse_resolve_ex(h, layer, d_sel, d_num_reqs, d_newest, &o, d_out, flags, stream);
}

int hisparse_resolve_resident(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                              const int32_t *d_num_reqs, const int32_t *d_newest,
                              const int32_t *d_prev_pos, const void *d_new_rows,
                              const int32_t *d_res_blocks, int32_t res_max_blocks,
                              int32_t res_block_tokens, int32_t *d_out, uint32_t flags,
                              void *stream) {
  hisparse_resolve_options o = {};
  o.d_prev_pos = d_prev_pos;
  o.d_new_rows = d_new_rows;
  o.d_res_blocks = d_res_blocks;
  o.res_max_blocks = res_max_blocks;
  o.res_block_tokens = res_block_tokens;
  return hisparse_resolve_ex(h, layer, d_sel, d_num_reqs, d_newest, &o, d_out, flags, stream);
}

int hisparse_resolve_ex(hisparse_handle *h, int32_t layer, const int32_t *d_sel,
                        const int32_t *d_num_reqs, const int32_t *d_newest,
                        const hisparse_resolve_options *opt, int32_t *d_out, uint32_t flags,
                        void *stream) {
  static const hisparse_resolve_options kNone = {};
  if (!opt) opt = &kNone;
  const int32_t *d_prev_pos = opt->d_prev_pos;
  const void *d_new_rows = opt->d_new_rows;
  const int32_t *d_res_blocks = opt->d_res_blocks;
  const int32_t res_max_blocks = opt->res_max_blocks, res_block_tokens = opt->res_block_tokens;
  const int32_t sel_bt = opt->sel_block_tokens < 1 ? 1 : opt->sel_block_tokens;
  const int32_t *d_seq_lens = opt->d_seq_lens;
  if (layer_ok(h, layer)) return HISPARSE_EINVAL;
  if (d_seq_lens && h->lookup == HISPARSE_LOOKUP_HASH) return HISPARSE_EINVAL;
  if (d_res_blocks && (res_max_blocks < 1 || res_block_tokens < 1 ||
                       h->lookup == HISPARSE_LOOKUP_HASH))
    return HISPARSE_EINVAL;
  if (sel_bt > 1 && (h->k % sel_bt != 0 || h->lookup == HISPARSE_LOOKUP_HASH))
    return HISPARSE_EINVAL;
  if (d_new_rows && !aligned16(d_new_rows)) return HISPARSE_EINVAL;
  if (!d_sel || !d_out) return HISPARSE_EINVAL;
  if (flags & ~(HISPARSE_RECORD_PLAN | HISPARSE_SKIP_IO | HISPARSE_FROM_MIRROR | HISPARSE_UNION |
                HISPARSE_WITH_SHARED))
    return HISPARSE_EINVAL;
  if ((flags & (HISPARSE_UNION | HISPARSE_WITH_SHARED)) && h->lookup == HISPARSE_LOOKUP_HASH)
    return HISPARSE_EINVAL;
  if (h->anchor_of[layer] != -1) return HISPARSE_EROLE;
  const LayerDev &Ld = h->layers[layer];
  const AnchorMeta &m = h->meta[layer];
  if ((flags & HISPARSE_FROM_MIRROR) && !Ld.mirror) return HISPARSE_EINVAL;
  std::vector<int32_t> shared_layers;  // filled in this launch (HISPARSE_WITH_SHARED)
  if (flags & HISPARSE_WITH_SHARED) {
    for (int32_t l = 0; l < h->L; ++l)
      if (h->anchor_of[l] == layer) shared_layers.push_back(l);
    if (shared_layers.size() > static_cast<size_t>(kMaxReplayTargets)) return HISPARSE_EBOUND;
    // a slice's (miss, layer, chunk) index stays below 2^31 (32-bit index math)
    if (static_cast<int64_t>(h->k) * static_cast<int64_t>(shared_layers.size()) * (h->rec / 16) >=
        (int64_t(1) << 31))
      return HISPARSE_EBOUND;
    for (int32_t l : shared_layers)
      if ((flags & HISPARSE_FROM_MIRROR) && !h->layers[l].mirror) return HISPARSE_EINVAL;
  }
  const bool plan = flags & HISPARSE_RECORD_PLAN;

  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(h->cs) * h->R);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = h->smem;
  lc.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute at[3];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = h->cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  // hisparse_set_l2_persisting: the layer's page table, read by one gather
  // per selection, is marked persisting so it survives in L2 between steps
  at[2].id = cudaLaunchAttributeAccessPolicyWindow;
  at[2].val.accessPolicyWindow.base_ptr = m.page_table;
  at[2].val.accessPolicyWindow.num_bytes = static_cast<size_t>(h->R) * h->P * sizeof(int32_t);
  at[2].val.accessPolicyWindow.hitRatio = h->l2_hit_ratio;
  at[2].val.accessPolicyWindow.hitProp = cudaAccessPropertyPersisting;
  at[2].val.accessPolicyWindow.missProp = cudaAccessPropertyStreaming;
  lc.attrs = at;
  lc.numAttrs = 1;
  cudaError_t e;
  if (h->lookup == HISPARSE_LOOKUP_HASH) {
    if (d_prev_pos || d_new_rows) {  // the hash kernel has no fused write-through
      if (!d_prev_pos) return HISPARSE_EINVAL;
      const int rc = hisparse_writeback(h, layer, d_prev_pos, d_new_rows, d_num_reqs, stream);
      if (rc != HISPARSE_OK) return rc;
    }
    ResolveArgs a;
    a.R = h->R; a.k = h->k; a.B = h->B; a.cap_log2 = h->cap_log2; a.rec16 = h->rec / 16;
    a.io = (flags & HISPARSE_SKIP_IO) ? 0 : 1;
    a.vec = (h->k % 4 == 0 && h->B % 8 == 0 && (reinterpret_cast<uintptr_t>(d_sel) & 15u) == 0) ? 1 : 0;
    a.bucket_shift = h->bucket_shift[layer];
    a.nbuckets = h->nbuckets[layer];
    a.P = h->P;
    a.sel = d_sel; a.num_reqs = d_num_reqs; a.newest = d_newest; a.out = d_out;
    a.slot_pos = m.slot_pos; a.lru = m.lru; a.page_table = m.page_table;
    a.miss_count = m.miss_count; a.unit_err = m.unit_err; a.status = h->d_status;
    a.plan_pos = m.plan_pos; a.plan_slot = m.plan_slot; a.plan_count = m.plan_count;
    a.src = (flags & HISPARSE_FROM_MIRROR) ? Ld.mirror : Ld.host;
    a.src_req_stride = Ld.host_req_stride; a.src_row_stride = Ld.host_row_stride;
    a.hot = Ld.hot; a.hot_req_stride = Ld.hot_req_stride; a.hot_row_stride = Ld.hot_row_stride;
    e = plan ? cudaLaunchKernelEx(&lc, resolve_kernel<true>, a)
             : cudaLaunchKernelEx(&lc, resolve_kernel<false>, a);
  } else {
    PtArgs a;
    a.R = h->R; a.k = h->k; a.B = h->B; a.rec16 = h->rec / 16;
    a.io = (flags & HISPARSE_SKIP_IO) ? 0 : 1;
    a.ks = h->ks; a.hcap_log2 = h->cap_log2;
    a.bucket_shift = h->bucket_shift[layer];
    a.nbuckets = h->nbuckets[layer];
    a.prev_pos = d_prev_pos;
    a.new_rows = static_cast<const char *>(d_new_rows);
    a.host_w = Ld.host_w;
    a.mirror_w = Ld.mirror;
    a.host_req_stride = Ld.host_req_stride;
    a.host_row_stride = Ld.host_row_stride;
    // the host pool and its mirror hold the same bytes, so the kept row serves either source
    a.prev_from_row = d_prev_pos ? 1 : 0;
    a.res_blocks = d_res_blocks;
    a.res_nblk = d_res_blocks ? res_max_blocks : 0;
    a.res_tok = d_res_blocks ? res_block_tokens : 1;
    a.sel_bt = sel_bt;
    a.union_mode = (flags & HISPARSE_UNION) ? 1 : 0;
    a.seq_lens = d_seq_lens;
    a.P = h->P;
    a.sel = d_sel; a.num_reqs = d_num_reqs; a.newest = d_newest; a.out = d_out;
    a.slot_pos = m.slot_pos; a.lru = m.lru; a.page_table = m.page_table;
    a.miss_count = m.miss_count; a.unit_err = m.unit_err; a.status = h->d_status;
    a.plan_pos = m.plan_pos; a.plan_slot = m.plan_slot; a.plan_count = m.plan_count;
    a.src = (flags & HISPARSE_FROM_MIRROR) ? Ld.mirror : Ld.host;
    a.src_req_stride = Ld.host_req_stride; a.src_row_stride = Ld.host_row_stride;
    a.hot = Ld.hot; a.hot_req_stride = Ld.hot_req_stride; a.hot_row_stride = Ld.hot_row_stride;
    a.nfl = static_cast<int32_t>(shared_layers.size());
    for (int i = 0; i < a.nfl; ++i) {
      const LayerDev &Lf = h->layers[shared_layers[i]];
      a.fl[i].src = (flags & HISPARSE_FROM_MIRROR) ? Lf.mirror : Lf.host;
      a.fl[i].src_req_stride = Lf.host_req_stride;
      a.fl[i].src_row_stride = Lf.host_row_stride;
      a.fl[i].hot = Lf.hot;
      a.fl[i].hot_req_stride = Lf.hot_req_stride;
      a.fl[i].hot_row_stride = Lf.hot_row_stride;
    }
    lc.numAttrs = h->l2_hit_ratio > 0.f ? 3 : 2;  // cluster shape + programmatic dependent
                                                  // launch (+ the L2 window)
    if (d_res_blocks || sel_bt > 1 || a.union_mode || d_seq_lens)  // the extended instantiation
      e = plan ? cudaLaunchKernelEx(&lc, resolve_pt_kernel<true, true>, a)
               : cudaLaunchKernelEx(&lc, resolve_pt_kernel<false, true>, a);
    else
      e = plan ? cudaLaunchKernelEx(&lc, resolve_pt_kernel<true, false>, a)
               : cudaLaunchKernelEx(&lc, resolve_pt_kernel<false, false>, a);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return HISPARSE_OK;
}

int hisparse_writeback(hisparse_handle *h, int32_t layer, const int32_t *d_pos,
                       const void *d_new_rows, const int32_t *d_num_reqs, void *stream) {
  if (!h || !d_pos) return HISPARSE_EINVAL;
  if (layer != -1 && layer_ok(h, layer)) return HISPARSE_EINVAL;
  if (d_new_rows && !aligned16(d_new_rows)) return HISPARSE_EINVAL;
  WritebackArgs a;
  a.layers = h->d_layers;
  a.layer0 = layer == -1 ? 0 : layer;
  a.R = h->R; a.B = h->B; a.rec16 = h->rec / 16; a.P = h->P;
  a.pos = d_pos; a.num_reqs = d_num_reqs; a.status = h->d_status;
  a.new_rows = static_cast<const char *>(d_new_rows);
  const dim3 grid(h->R, layer == -1 ? h->L : 1);
  writeback_kernel<<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(a);
  HS_CUDA(cudaGetLastError());
  return HISPARSE_OK;
}

int hisparse_prefetch_plan(hisparse_handle *h, int32_t anchor_layer, int32_t follower_layer,
                           const int32_t *d_num_reqs, void *stream) {
  if (layer_ok(h, anchor_layer) || (follower_layer != -1 && layer_ok(h, follower_layer)))
    return HISPARSE_EINVAL;
  if (h->anchor_of[anchor_layer] != -1) return HISPARSE_EROLE;
  if (follower_layer != -1 && h->anchor_of[follower_layer] != anchor_layer) return HISPARSE_EROLE;
  // the layers to fill: the one named, or every shared-index layer of the anchor
  std::vector<int32_t> fl;
  if (follower_layer != -1) fl.push_back(follower_layer);
  else
    for (int32_t l = 0; l < h->L; ++l)
      if (h->anchor_of[l] == anchor_layer) fl.push_back(l);
  const AnchorMeta &m = h->meta[anchor_layer];
  const size_t smem = replay_smem_bytes(h->R);
  for (size_t f0 = 0; f0 < fl.size(); f0 += kMaxReplayTargets) {
    ReplayArgs a;
    a.R = h->R; a.k = h->k; a.rec16 = h->rec / 16; a.num_reqs = d_num_reqs;
    a.plan_pos = m.plan_pos; a.plan_slot = m.plan_slot; a.plan_count = m.plan_count;
    a.nf = static_cast<int32_t>(std::min(fl.size() - f0, static_cast<size_t>(kMaxReplayTargets)));
    for (int i = 0; i < a.nf; ++i) {
      const LayerDev &Lf = h->layers[fl[f0 + i]];
      a.f[i].src = Lf.host;
      a.f[i].src_req_stride = Lf.host_req_stride;
      a.f[i].src_row_stride = Lf.host_row_stride;
      a.f[i].hot = Lf.hot;
      a.f[i].hot_req_stride = Lf.hot_req_stride;
      a.f[i].hot_row_stride = Lf.hot_row_stride;
    }
    replay_kernel<<<h->replay_ctas, kReplayThreads, smem, static_cast<cudaStream_t>(stream)>>>(a);
    HS_CUDA(cudaGetLastError());
  }
  return HISPARSE_OK;
}

int hisparse_copy(void *dst, const void *src, int64_t bytes, void *stream) {
  if (bytes < 0 || bytes % 16) return HISPARSE_EINVAL;
  if (bytes == 0) return HISPARSE_OK;
  if (!dst || !src || !aligned16(dst) || !aligned16(src)) return HISPARSE_EINVAL;
  const int64_t n = bytes / 16;
  const int64_t per_cta = static_cast<int64_t>(kCopyThreads) * 4;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>((n + per_cta - 1) / per_cta, kCopyMaxCtas)));
  lc.blockDim = dim3(kCopyThreads);
  lc.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&lc, copy_kernel, static_cast<uint4 *>(dst),
                                           static_cast<const uint4 *>(src), n);
  if (e != cudaSuccess) return cuda_fail(e);
  return HISPARSE_OK;
}

int hisparse_copy_miss_counts(hisparse_handle *h, int32_t layer, int32_t *d_dst, void *stream) {
  if (layer_ok(h, layer) || !d_dst) return HISPARSE_EINVAL;
  if (h->anchor_of[layer] != -1) return HISPARSE_EROLE;
  HS_CUDA(cudaMemcpyAsync(d_dst, h->meta[layer].miss_count, sizeof(int32_t) * h->R,
                          cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
  return HISPARSE_OK;
}

int hisparse_get_status(hisparse_handle *h, uint32_t *flags_out, int32_t *unit_err_out) {
  if (!h || !flags_out) return HISPARSE_EINVAL;
  HS_CUDA(cudaDeviceSynchronize());
  HS_CUDA(cudaMemcpy(flags_out, h->d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  HS_CUDA(cudaMemset(h->d_status, 0, sizeof(uint32_t)));
  if (unit_err_out)
    HS_CUDA(cudaMemcpy(unit_err_out, h->d_unit_err_all, sizeof(int32_t) * h->L * h->R,
                       cudaMemcpyDeviceToHost));
  HS_CUDA(cudaDeviceSynchronize());
  return HISPARSE_OK;
}

int hisparse_export_state(hisparse_handle *h, int32_t layer, int32_t *slot_pos, int16_t *lru,
                          int32_t *page_table, int32_t *miss_counts) {
  if (layer_ok(h, layer)) return HISPARSE_EINVAL;
  if (h->anchor_of[layer] != -1) return HISPARSE_EROLE;
  const AnchorMeta &m = h->meta[layer];
  HS_CUDA(cudaDeviceSynchronize());
  const size_t RB = static_cast<size_t>(h->R) * h->B;
  if (slot_pos) HS_CUDA(cudaMemcpy(slot_pos, m.slot_pos, 4 * RB, cudaMemcpyDeviceToHost));
  if (lru) HS_CUDA(cudaMemcpy(lru, m.lru, 2 * RB, cudaMemcpyDeviceToHost));
  if (page_table)
    HS_CUDA(cudaMemcpy(page_table, m.page_table, 4 * static_cast<size_t>(h->R) * h->P,
                       cudaMemcpyDeviceToHost));
  if (miss_counts) HS_CUDA(cudaMemcpy(miss_counts, m.miss_count, 4 * h->R, cudaMemcpyDeviceToHost));
  return HISPARSE_OK;
}

int hisparse_import_state(hisparse_handle *h, int32_t layer, const int32_t *slot_pos,
                          const int16_t *lru, const int32_t *page_table,
                          const int32_t *miss_counts) {
  if (layer_ok(h, layer) || !slot_pos || !lru || !page_table) return HISPARSE_EINVAL;
  if (h->anchor_of[layer] != -1) return HISPARSE_EROLE;
  const int32_t B = h->B;
  const int64_t P = h->P;
  std::vector<uint8_t> seen(B);
  for (int r = 0; r < h->R; ++r) {
    const int32_t *sp = slot_pos + static_cast<int64_t>(r) * B;
    const int16_t *lr = lru + static_cast<int64_t>(r) * B;
    const int32_t *pt = page_table + static_cast<int64_t>(r) * P;
    std::fill(seen.begin(), seen.end(), 0);
    for (int j = 0; j < B; ++j) {
      if (lr[j] < 0 || lr[j] >= B || seen[lr[j]]) return HISPARSE_EINVAL;
      seen[lr[j]] = 1;
    }
    int64_t occupied = 0;
    for (int s = 0; s < B; ++s) {
      if (sp[s] < -1 || sp[s] >= P) return HISPARSE_EINVAL;
      if (sp[s] >= 0) {
        if (pt[sp[s]] != s) return HISPARSE_EINVAL;  // also rules out a position twice
        ++occupied;
      }
    }
    int64_t mapped = 0;
    for (int64_t p = 0; p < P; ++p) {
      if (pt[p] == -1) continue;
      if (pt[p] < 0 || pt[p] >= B || sp[pt[p]] != p) return HISPARSE_EINVAL;
      ++mapped;
    }
    if (mapped != occupied) return HISPARSE_EINVAL;
    if (miss_counts && (miss_counts[r] < 0 || miss_counts[r] > h->k)) return HISPARSE_EINVAL;
  }
  const AnchorMeta &m = h->meta[layer];
  HS_CUDA(cudaDeviceSynchronize());
  const size_t RB = static_cast<size_t>(h->R) * B;
  HS_CUDA(cudaMemcpy(m.slot_pos, slot_pos, 4 * RB, cudaMemcpyHostToDevice));
  HS_CUDA(cudaMemcpy(m.lru, lru, 2 * RB, cudaMemcpyHostToDevice));
  HS_CUDA(cudaMemcpy(m.page_table, page_table, 4 * static_cast<size_t>(h->R) * P,
                     cudaMemcpyHostToDevice));
  if (miss_counts)
    HS_CUDA(cudaMemcpy(m.miss_count, miss_counts, 4 * static_cast<size_t>(h->R),
                       cudaMemcpyHostToDevice));
  return HISPARSE_OK;
}

int hisparse_export_plan(hisparse_handle *h, int32_t layer, int32_t *count, int32_t *pos,
                         int32_t *slot) {
  if (layer_ok(h, layer) || !count || !pos || !slot) return HISPARSE_EINVAL;
  if (h->anchor_of[layer] != -1) return HISPARSE_EROLE;
  const AnchorMeta &m = h->meta[layer];
  HS_CUDA(cudaDeviceSynchronize());
  const size_t Rk = static_cast<size_t>(h->R) * h->k;
  HS_CUDA(cudaMemcpy(count, m.plan_count, 4 * h->R, cudaMemcpyDeviceToHost));
  HS_CUDA(cudaMemcpy(pos, m.plan_pos, 4 * Rk, cudaMemcpyDeviceToHost));
  HS_CUDA(cudaMemcpy(slot, m.plan_slot, 4 * Rk, cudaMemcpyDeviceToHost));
  return HISPARSE_OK;
}

int hisparse_set_l2_persisting(hisparse_handle *h, int64_t bytes) {
  if (!h || bytes < 0) return HISPARSE_EINVAL;
  if (bytes == 0) return l2_persisting_off(h);
  int max_persist = 0, max_window = 0;
  HS_CUDA(cudaDeviceGetAttribute(&max_persist, cudaDevAttrMaxPersistingL2CacheSize, h->device));
  HS_CUDA(cudaDeviceGetAttribute(&max_window, cudaDevAttrMaxAccessPolicyWindowSize, h->device));
  const int64_t table = static_cast<int64_t>(h->R) * h->P * static_cast<int64_t>(sizeof(int32_t));
  if (max_persist <= 0 || table > max_window) return HISPARSE_EBOUND;
  int64_t tables = 0;
  for (int l = 0; l < h->L; ++l)
    if (h->anchor_of[l] == -1) tables += table;
  const int64_t aside = std::min<int64_t>(bytes, max_persist);
  if (!h->l2_limit_saved) {
    HS_CUDA(cudaDeviceGetLimit(&h->l2_prev_limit, cudaLimitPersistingL2CacheSize));
    h->l2_limit_saved = true;
  }
  HS_CUDA(cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, static_cast<size_t>(aside)));
  // the share of each window's lines marked persisting, so that all layers'
  // persisting lines fit the set-aside together
  h->l2_hit_ratio = static_cast<float>(std::min<double>(1.0, double(aside) / double(tables)));
  return HISPARSE_OK;
}

int hisparse_get_info(const hisparse_handle *h, hisparse_info *out) {
  if (!h || !out) return HISPARSE_EINVAL;
  out->ctas_per_request = h->cs;
  out->threads_per_cta = kThreads;
  out->smem_bytes = static_cast<int32_t>(h->smem);
  out->hash_capacity = 1 << h->cap_log2;
  out->replay_ctas = h->replay_ctas;
  out->sm_count = h->sm_count;
  out->metadata_bytes = h->arena_bytes;
  out->lookup = h->lookup;
  return HISPARSE_OK;
}

}  // extern "C"
