// Device building blocks of the sample-guided exact Top-K selector (sm_103a).
//
// Method (web pages on "Sample-Guided Exact Top-K Selection for Long-Context
// Sparse Attention", Tencent HPC-Ops):
//   * PaperDaily "腾讯|长上下文稀疏注意力前K精确选择", section 问题二, Fig. 4:
//     stage 1, a fixed-stride view of the current row proposes a provisional
//     threshold tau0 and a wider nested tau1; stage 2, the mandatory full-row
//     pass counts C(tau0), forms the admitted candidate set and seeds the first
//     FP32 radix histogram; if C(tau0) < K the nested threshold is used, and if
//     that still underfills the row is recovered exactly from the whole row;
//     stage 3, exact radix refinement over the raw FP32 bits runs only on the
//     unresolved boundary bin, resolved high bins are emitted and never
//     revisited, output order is free.
//   * codexqa.cn "几何平均快 1.55 倍…腾讯怎么测精确 Top-K", section
//     "采样不是处处都该开": stride 128, primary target 1.5K, nested 1.75K on
//     H20 (the defaults here are wider, see the parameter notes in topk.h).
//   * arxivdaily abstract: certification and candidate formation are fused in
//     one pass; persistent, KV-split and direct-exact execution sit behind a
//     graph-capturable ragged-row dispatch.
//
// Order key: key(v) maps FP32 bits to an unsigned integer whose order is the
// IEEE order of the scores, with -0.0 mapped onto +0.0 so that the key order
// and the float comparison agree on every non-NaN value.
//
// This build differs from the pages' H20 design where GB300 pays for it: the
// full-row pass streams the row through shared memory with 1-D bulk async
// copies (TMA) into a 3-stage ring driven by mbarriers; candidates of the
// nested band are collected in the same pass (into shared memory, then a
// global spill area), so the tau1 path needs no re-read; radix rounds use
// data-relative 11-bit digits so the first histogram is not degenerate on
// concentrated scores; rows may be FP32, bfloat16 or FP8 E4M3 (widened exactly).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "score_elem.cuh"
#include "topk_launch.h"

namespace tk {

// ----------------------------------------------------------------- constants
constexpr int THREADS = 512;                // threads per CTA for every kernel
constexpr int NWARPS = THREADS / 32;
constexpr int CONSUMER_WARPS = NWARPS - 1;  // warp 0 issues the bulk copies; at most
                                            // the others consume (see Ring::cw)
constexpr int NB_BITS = 11;
constexpr int NB = 1 << NB_BITS;            // bins per radix round
static_assert(NB == 4 * THREADS, "boundary search maps 4 bins to each thread");
constexpr int STAGES = 3;                   // ring stages
constexpr int UNIT_CHUNK_BYTES = 32 * 32;    // chunk bytes per consumer warp: two 16-byte
                                            // units per consumer thread
constexpr int STAGE_BYTES = UNIT_CHUNK_BYTES * CONSUMER_WARPS;  // ring stage (15 KB)
constexpr int STAGE_FLOATS = STAGE_BYTES / 4;
constexpr int CAP = 6144;                   // on-chip candidate capacity (entries of 8 B)
constexpr int SPILL = 10240;                // further candidates kept in global memory
constexpr int CAP_ALL = CAP + SPILL;        // candidates one full-row pass can keep
constexpr int TIE_CAP = 4096;               // indices of scores equal to tau1 kept (>= any K)
constexpr int SMALL = 32;                   // frontier size finished by one warp
constexpr int SAMPLE_SMEM = 2 * CAP;        // sample keys kept on chip (they alias the candidates)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // bounded waits give up after 2 s

// Row paths and status bits (same values as the public header).
constexpr int32_t PATH_SENTINEL = 0, PATH_DIRECT = 1, PATH_TAU0 = 2, PATH_TAU1 = 3,
                  PATH_RECOVERY = 4;
constexpr uint32_t F_LEN_CLAMPED = 0x1u, F_OVERFLOW = 0x2u, F_RECOVERY = 0x4u,
                   F_INTERNAL = 0x8u, F_TIMEOUT = 0x10u, F_K_CLAMPED = 0x20u;

constexpr unsigned FULL_MASK = 0xffffffffu;

// --------------------------------------------------------------- order key
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return k + (k == 0x7fffffffu);  // -0.0 joins +0.0
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// ----------------------------------------------------------------- PTX glue
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Slow path of mbar_wait: polls until the phase completes, giving up after
// limit_ns (WAIT_LIMIT_NS in the kernels) so that no wait can hang the GPU.
// `abort` is the fail-fast flag of the work the waiting CTA belongs to (a
// persistent launch's workspace header, a KV-split row's header; nullptr for
// a CTA that works alone): the first wait that gives up sets it, and every
// later wait on that work then fails at once, so a launch that lost a copy
// ends quickly (its rows flagged) instead of timing out wait after wait.  The
// flag lives in memory that belongs to one launch and is reset by it (the
// last CTA of a persistent launch, the prepare kernel of a KV-split launch),
// so an abort never reaches another launch.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, uint32_t* abort,
                                            uint64_t limit_ns = WAIT_LIMIT_NS) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort != nullptr && *reinterpret_cast<volatile uint32_t*>(abort) != 0u) return false;
      if (globaltimer() - t0 > limit_ns) {
        if (abort != nullptr) atomicExch(abort, 1u);
        return false;
      }
    }
  }
}

// Polls until the phase completes or limit_ns passes, whatever the fail-fast
// flag says (used to let copies in flight land before a CTA exits).
static __device__ __noinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > limit_ns) return false;
  return true;
}

// Waits for the phase of `bar` with the given parity (false after a timeout
// or once `abort` is set).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort);
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 prefetch of the line holding `p` (no data returned to the thread),
// marked evict-last.
__device__ __forceinline__ void prefetch_l2_keep(const void* p) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

// Bulk prefetch of [src, src + bytes) into L2 (no data to the CTA; src
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------ warp / block
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(FULL_MASK, x, o);
    if (lane >= (uint32_t)o) x += y;
  }
  return x;
}

// Shared scratch of every kernel.  Lives at the start of dynamic shared memory.
struct __align__(16) Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint2 small[SMALL];            // (idx, key) of a small frontier
  uint32_t wtmp[NWARPS + 2];
  uint32_t wtmp2[NWARPS + 2];
  uint32_t row;
  uint32_t ncand;                // admitted candidates (counts past CAP)
  uint32_t nout;                 // indices emitted for the current row
  uint32_t c0;                   // C(tau0)
  uint32_t small_n;
  uint32_t take;
  uint32_t b, above, ok;
  uint32_t flags;
  uint32_t kmin, kmax, res;
  uint32_t key0, key1;
  uint32_t last;
  uint32_t next, next_ok;        // a row claimed ahead of time (persistent kernel)
  uint32_t nx_row, nx_ok;        // the claimed row, and whether nx_key holds its stage 1
  uint32_t nx_key[4];            // key(tau0), key(tau1), smallest and largest sample key
  uint32_t neq;                  // scores equal to tau1 (counts past the tie list)
#ifdef TOPK_PHASE_TIMING
  unsigned long long ph[12];     // cycles per phase of the persistent kernel (thread 0's clock)
  long long ph_t;                // thread 0's clock at the last mark
#endif
};

// Phase timing, compiled only with -DTOPK_PHASE_TIMING: thread 0 adds the
// cycles since its previous mark to phase i.  Marks sit right after a block
// barrier, so thread 0's clock stands for the whole block there.
__device__ __forceinline__ void phase_mark(Shared& S, int i) {
#ifdef TOPK_PHASE_TIMING
  if (threadIdx.x == 0) {
    const long long t = clock64();
    S.ph[i] += (unsigned long long)(t - S.ph_t);
    S.ph_t = t;
  }
#else
  (void)S;
  (void)i;
#endif
}

// Phase timing builds only: counts an event (slot i then holds a count).
__device__ __forceinline__ void phase_count(Shared& S, int i) {
#ifdef TOPK_PHASE_TIMING
  if (threadIdx.x == 0) S.ph[i] += 1;
#else
  (void)S;
  (void)i;
#endif
}

// Exclusive prefix sum over all THREADS threads (every thread must call).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Shared& S, uint32_t* total) {
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(v);
  if (lane == 31) S.wtmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = lane < (uint32_t)NWARPS ? S.wtmp[lane] : 0u;
    const uint32_t wi = warp_incl_scan(w);
    if (lane < (uint32_t)NWARPS) S.wtmp[lane] = wi - w;
    if (lane == NWARPS - 1) S.wtmp[NWARPS] = wi;
  }
  __syncthreads();
  const uint32_t r = S.wtmp[warp] + incl - v;
  *total = S.wtmp[NWARPS];
  __syncthreads();
  return r;
}

// Block-wide min and max of u32 values (every thread must call).
__device__ __forceinline__ void block_minmax(uint32_t mn, uint32_t mx, Shared& S, uint32_t* omn,
                                             uint32_t* omx) {
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(FULL_MASK, mn, o));
    mx = max(mx, __shfl_xor_sync(FULL_MASK, mx, o));
  }
  if (lane == 0) {
    S.wtmp[warp] = mn;
    S.wtmp2[warp] = mx;
  }
  __syncthreads();
  if (warp == 0) {
    mn = lane < (uint32_t)NWARPS ? S.wtmp[lane] : 0xffffffffu;
    mx = lane < (uint32_t)NWARPS ? S.wtmp2[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = min(mn, __shfl_xor_sync(FULL_MASK, mn, o));
      mx = max(mx, __shfl_xor_sync(FULL_MASK, mx, o));
    }
    if (lane == 0) {
      S.wtmp[NWARPS] = mn;
      S.wtmp2[NWARPS] = mx;
    }
  }
  __syncthreads();
  *omn = S.wtmp[NWARPS];
  *omx = S.wtmp2[NWARPS];
  __syncthreads();
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, Shared& S) {
  uint32_t total;
  block_excl_scan(v, S, &total);
  return total;
}

// ------------------------------------------------------------------ binning
// One radix round over the key interval [lo, hi].  Keys below `base` fall in
// bin 0, bins 1..NB-2 are 2^shift keys wide starting at base, and bin NB-1
// also takes every key above its start up to hi.
struct Bins {
  uint32_t lo, hi, base, shift;

  __device__ __forceinline__ uint32_t digit(uint32_t k) const {
    if (k < base) return 0;
    const uint32_t d = (k - base) >> shift;
    return d < (uint32_t)(NB - 1) ? d : (uint32_t)(NB - 1);
  }
  __device__ __forceinline__ uint32_t bin_lo(uint32_t b) const {
    if (b == 0) return lo;
    const uint64_t x = (uint64_t)base + ((uint64_t)b << shift);
    return x > hi ? hi : (uint32_t)x;
  }
  __device__ __forceinline__ uint32_t bin_hi(uint32_t b) const {
    if (b == (uint32_t)(NB - 1)) return hi;
    const uint64_t x = (uint64_t)base + ((uint64_t)(b + 1) << shift) - 1;
    return x > hi ? hi : (uint32_t)x;
  }
};

__device__ __forceinline__ uint32_t shift_for_span(uint32_t span, uint32_t max_digit) {
  uint32_t s = 0;
  while ((span >> s) > max_digit) ++s;
  return s;
}

// Plain bins over [lo, hi]: base = lo and the narrowest shift that fits.
__device__ __forceinline__ Bins make_bins(uint32_t lo, uint32_t hi) {
  Bins b;
  b.lo = lo;
  b.hi = hi;
  b.base = lo;
  b.shift = shift_for_span(hi - lo, NB - 1);
  return b;
}

// Bins whose regular range is [base, top] inside a wider frontier [lo, hi].
__device__ __forceinline__ Bins make_bins_focus(uint32_t lo, uint32_t hi, uint32_t base,
                                                uint32_t top) {
  Bins b;
  b.lo = lo;
  b.hi = hi;
  b.base = base < lo ? lo : (base > hi ? hi : base);
  if (top < b.base) top = b.base;
  if (top > hi) top = hi;
  b.shift = shift_for_span(top - b.base, NB - 2);
  return b;
}

// Boundary search: the largest bin b whose suffix count (bins >= b) reaches
// Kp.  Writes S.b, S.above (count in bins > b) and S.ok (0 when the histogram
// holds fewer than Kp keys).  Every thread must call.
__device__ __forceinline__ void find_boundary(const uint32_t* hist, uint32_t Kp, Shared& S) {
  const uint32_t t = threadIdx.x;
  if (t == 0) S.ok = 0;
  const int top = NB - 1 - 4 * (int)t;
  const uint32_t h0 = hist[top], h1 = hist[top - 1], h2 = hist[top - 2], h3 = hist[top - 3];
  const uint32_t s = h0 + h1 + h2 + h3;
  uint32_t total;
  const uint32_t pre = block_excl_scan(s, S, &total);
  if (pre < Kp && pre + s >= Kp) {
    uint32_t acc = pre, b = (uint32_t)top;
    const uint32_t hh[4] = {h0, h1, h2, h3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (acc + hh[j] >= Kp) {
        b = (uint32_t)(top - j);
        break;
      }
      acc += hh[j];
    }
    S.b = b;
    S.above = acc;
    S.ok = 1;
  }
  __syncthreads();
}

__device__ __forceinline__ void clear_hist(uint32_t* hist) {
  for (int i = threadIdx.x; i < NB; i += THREADS) hist[i] = 0;
}

// Descending bitonic sort of one (idx, key) pair per lane by key.
// Invalid lanes carry key 0 and idx 0xffffffff and sort last among equals.
__device__ __forceinline__ void warp_sort_desc(uint32_t& key, uint32_t& idx) {
  const uint32_t lane = lane_id();
  uint64_t v = ((uint64_t)key << 32) | (uint64_t)(~idx);
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(FULL_MASK, v, j);
      const bool asc = (lane & (uint32_t)k) == 0;
      const bool lower = (lane & (uint32_t)j) == 0;
      // an ascending network with every choice flipped sorts descending
      const bool take_max = (lower == asc);
      v = take_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  key = (uint32_t)(v >> 32);
  idx = ~(uint32_t)v;
}

// --------------------------------------------------------------- emission
// Warp-aggregated append of one index per flagged lane to the row's output.
// Every lane of the warp must call.
__device__ __forceinline__ void warp_emit(int32_t* out, int32_t K, uint32_t idx, bool flag,
                                          Shared& S, uint32_t& lflags) {
  const uint32_t m = __ballot_sync(FULL_MASK, flag);
  if (m == 0) return;
  const uint32_t lane = lane_id();
  const uint32_t leader = __ffs(m) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(&S.nout, (uint32_t)__popc(m));
  base = __shfl_sync(FULL_MASK, base, leader);
  if (flag) {
    const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
    if (pos < (uint32_t)K) out[pos] = (int32_t)idx;
    else lflags |= F_INTERNAL;
  }
}

// ------------------------------------------------------------- the TMA ring
// A 3-stage ring of 15 KB shared-memory stages filled by 1-D bulk copies.
// Warp 0, lane 0 produces; warps 1..cw consume, and a chunk is 1 KB per
// consumer warp.  With cw = 14 the last warp, instead of consuming, samples
// the next row during a certify pass (and sits the other passes out).  Every thread keeps the same
// chunk sequence number, so passes can follow one another without resetting
// the barriers.
struct Ring {
  float* buf;
  uint64_t* full;
  uint64_t* empty;
  uint32_t seq;
  uint64_t policy;
  uint32_t* abort;  // fail-fast flag of the launch's work (see mbar_wait_slow)
  uint32_t pf_ahead;  // chunks ahead of the ring a certify pass prefetches into L2
  uint32_t cw;        // consumer warps (warps 1..cw)
  uint32_t chunk;     // bytes per chunk: UNIT_CHUNK_BYTES * cw
};

__device__ __forceinline__ void ring_init(Ring& R, Shared& S, float* buf, uint32_t* abort,
                                          uint32_t cw = (uint32_t)CONSUMER_WARPS) {
  R.buf = buf;
  R.full = S.full;
  R.empty = S.empty;
  R.seq = 0;
  R.policy = l2_policy_evict_first();
  R.abort = abort;
  R.pf_ahead = 0;
  R.cw = cw;
  R.chunk = (uint32_t)UNIT_CHUNK_BYTES * cw;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], cw);
    }
    fence_mbar_init();
  }
  __syncthreads();
}

// Producer side of one chunk: wait for stage q % STAGES to be free, then
// start the bulk copy of chunk c of the 16-byte aligned body [a0, a1).
template <class E>
__device__ __forceinline__ void ring_issue(Ring& R, const E* __restrict__ row, int64_t a0,
                                           int64_t a1, uint32_t c, uint32_t& lflags,
                                           uint32_t chunk) {
  const int64_t CE = chunk / Elem<E>::kSize;
  const uint32_t q = R.seq + c, s = q % STAGES, use = q / STAGES;
  if (!mbar_wait(&R.empty[s], (use & 1u) ^ 1u, R.abort)) lflags |= F_TIMEOUT;
  const int64_t off = a0 + (int64_t)c * CE;
  const int64_t n = (a1 - off) < CE ? (a1 - off) : CE;
  const uint32_t bytes = (uint32_t)(n * Elem<E>::kSize);
  fence_proxy_async();
  mbar_arrive_expect_tx(&R.full[s], bytes);
  bulk_load(R.buf + (size_t)s * STAGE_FLOATS, row + off, bytes, &R.full[s], R.policy);
}

// The 16-byte aligned body [a0, a1) of [start, end) and its chunk count.
template <class E>
__device__ __forceinline__ uint32_t ring_span(const E* row, int64_t start, int64_t end,
                                              uint32_t chunk, int64_t* a0, int64_t* a1);

// L2 prefetch of the first max_bytes of the 16-byte aligned body of row
// [0, len) (one bulk prefetch; nothing past len is touched).
template <class E>
__device__ __forceinline__ void prefetch_row_head(const E* row, int64_t len, uint32_t max_bytes) {
  int64_t a0, a1;
  ring_span(row, 0, len, (uint32_t)STAGE_BYTES, &a0, &a1);
  int64_t n = a1 - a0;
  if (n > (int64_t)(max_bytes / Elem<E>::kSize)) n = (int64_t)(max_bytes / Elem<E>::kSize);
  const uint32_t bytes = (uint32_t)(n * Elem<E>::kSize) & ~15u;
  if (bytes) bulk_prefetch_l2(row + a0, bytes);
}

// The 16-byte aligned body [a0, a1) of [start, end) and its count of chunks
// of `chunk` bytes.
template <class E>
__device__ __forceinline__ uint32_t ring_span(const E* row, int64_t start, int64_t end,
                                              uint32_t chunk, int64_t* a0, int64_t* a1) {
  constexpr int P16 = Elem<E>::kPer16;
  const int64_t CE = chunk / Elem<E>::kSize;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + start);
  int64_t b0 = start + (int64_t)(((16u - (uint32_t)(addr & 15u)) & 15u) / Elem<E>::kSize);
  if (b0 > end) b0 = end;
  *a0 = b0;
  *a1 = b0 + ((end - b0) & ~(int64_t)(P16 - 1));
  return (uint32_t)((*a1 - b0 + CE - 1) / CE);
}

// Starts the first chunks (up to STAGES) of a later scan_pass over
// [start, end) while the ring is idle, so that they load during the row's
// sampling.  Every thread calls; returns the number started, which that
// scan_pass must be given.
template <class E>
__device__ __forceinline__ uint32_t ring_prime(Ring& R, const E* __restrict__ row,
                                               int64_t start, int64_t end, uint32_t& lflags) {
  if (end <= start) return 0;
  int64_t a0, a1;
  const uint32_t nchunks = ring_span(row, start, end, R.chunk, &a0, &a1);
  const uint32_t n = nchunks < (uint32_t)STAGES ? nchunks : (uint32_t)STAGES;
  if (threadIdx.x == 0) {
    for (uint32_t c = 0; c < n; ++c) ring_issue(R, row, a0, a1, c, lflags, R.chunk);
    // and the next pf_ahead chunks into L2, which the pass would ask for
    // first (scan_pass then starts its own prefetches past them)
    const int64_t CE = R.chunk / Elem<E>::kSize;
    if (R.pf_ahead > 0 && n < nchunks) {
      const int64_t p0 = a0 + (int64_t)n * CE;
      const int64_t p1 = min(a1, a0 + (int64_t)(n + R.pf_ahead) * CE);
      bulk_prefetch_l2(row + p0, (uint32_t)((p1 - p0) * Elem<E>::kSize));
    }
  }
  return n;
}

// Before a CTA exits: waits (bounded, even after an abort) for the copies of
// the last STAGES chunks, so that no bulk copy is still in flight into this
// CTA's shared memory.  On the normal path every one of them has long landed.
__device__ __forceinline__ void ring_drain(Ring& R) {
  if (threadIdx.x != 0) return;
  const uint32_t n = R.seq < (uint32_t)STAGES ? R.seq : (uint32_t)STAGES;
  for (uint32_t k = 0; k < n; ++k) {
    const uint32_t q = R.seq - 1u - k, s = q % STAGES, use = q / STAGES;
    mbar_wait_drain(&R.full[s], use & 1u, 100000000ull);
  }
}

// Streams elements [start, end) of `row` through the ring and calls
// f.quad(i0, float4, valid_mask) on the consumer warps, warp-uniformly, for
// every group of up to four consecutive elements, widened to FP32 (element
// i0 + e is lane e of the float4, valid when bit e of the mask is set).  The
// 16-byte aligned body goes through bulk copies; the unaligned head and tail
// (fewer than 16 bytes each) are read directly.  The caller synchronises the
// block afterwards.
template <class E, class F>
__device__ __forceinline__ void ring_pass(Ring& R, const E* __restrict__ row, int64_t start,
                                          int64_t end, F& f, uint32_t& lflags) {
  constexpr int P16 = Elem<E>::kPer16, NG = P16 / 4;
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  if (end <= start) return;
  int64_t a0, a1;
  const uint32_t nchunks = ring_span(row, start, end, R.chunk, &a0, &a1);
  if (warp == 0) {
    if (lane == 0)
      for (uint32_t c = 0; c < nchunks; ++c) ring_issue(R, row, a0, a1, c, lflags, R.chunk);
  } else if (warp <= R.cw) {
    if (warp == 1) {
      // head [start, a0) on lanes 0.., tail [a1, end) on lanes 16..
      const int64_t nh = a0 - start, nt = end - a1;
      int64_t i = -1;
      if ((int64_t)lane < nh) i = start + lane;
      else if (lane >= 16 && (int64_t)lane - 16 < nt) i = a1 + (lane - 16);
      const float v = (i >= 0) ? Elem<E>::load(row + i) : 0.0f;
      f.quad(i >= 0 ? i : 0, make_float4(v, 0.f, 0.f, 0.f), i >= 0 ? 1u : 0u);
    }
    const uint32_t ct = tid - 32;
    const int C = 32 * (int)R.cw;  // consumer threads
    const int64_t CE = R.chunk / Elem<E>::kSize;
    for (uint32_t c = 0; c < nchunks; ++c) {
      const uint32_t q = R.seq + c, s = q % STAGES, use = q / STAGES;
      if (!mbar_wait(&R.full[s], use & 1u, R.abort)) lflags |= F_TIMEOUT;
      const int64_t off = a0 + (int64_t)c * CE;
      const int64_t n = (a1 - off) < CE ? (a1 - off) : CE;
      const int nu = (int)(n / P16);
      const uint4* sm = reinterpret_cast<const uint4*>(R.buf + (size_t)s * STAGE_FLOATS);
      const int iters = (nu + C - 1) / C;
      for (int it = 0; it < iters; ++it) {
        const int j = (int)ct + it * C;
        const bool ok = j < nu;
        const uint4 u = ok ? sm[j] : make_uint4(0u, 0u, 0u, 0u);
        // one group of four widened scores at a time (the functor's work is
        // inlined per group; more would only add live registers)
#pragma unroll 1
        for (int k = 0; k < NG; ++k)
          f.quad(off + (int64_t)P16 * j + 4 * k, Elem<E>::group(u, k), ok ? 0xfu : 0u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&R.empty[s]);
    }
  }
  R.seq += nchunks;
}

// Candidate j of a row: entries [0, CAP) live in shared memory, the rest in a
// global spill area written earlier in the same kernel (read through L2).
__device__ __forceinline__ uint2 cand_at(const uint2* cand, const uint2* spill, uint32_t j) {
  if (j < (uint32_t)CAP) return cand[j];
  const uint2* p = spill + (j - (uint32_t)CAP);
  return make_uint2(__ldcg(&p->x), __ldcg(&p->y));
}

// ------------------------------------------------- certify + collect (stage 2)
// Admission: key(v) >= key(tau1).  When tau1 > +0 the signed comparison of
// the raw bits gives the same answer in one instruction (POS = true).
// An admitted score above tau1 is appended, as (index, key), to the shared
// candidate array; C(tau0) and the seeded histogram are taken from the array
// once the pass is over (tally_candidates), which keeps the histogram atomics
// out of the streaming loop.  A score equal to tau1 is only counted, and its
// index kept while the tie list has room: when the K-th largest score is
// tau1 the answer takes every score above it and any of the ties (the
// contract lets boundary ties go either way), so the first K ties suffice.
// E4M3 rows (8 values per octave) put long runs of ties at tau1, which would
// otherwise overflow the candidate buffers (with tau1 > +0 their units are
// tested byte-wise, put_e4m3_words); for FP32 and bfloat16 rows
// (TIES = false) ties are ordinary candidates, which keeps their scan loop
// leaner (measured 13 % and 5 % faster), and a rare long tie run takes the
// overflow path.
// SWAR lane tests against a positive threshold t, exact per lane: the bytes
// (E4M3) or 16-bit halves (bfloat16) of w read as signed integers.  A lane
// >= t has its top bit clear, and then its low bits plus (top - t) reach the
// top bit without a carry into the next lane (the sum stays below 2^8 or
// 2^16).  k8 = (0x80 - t) * 0x01010101, g8 = (0x7F - t) * 0x01010101,
// t4 = t * 0x01010101, k16 = (0x8000 - t) * 0x00010001.  The result has the
// top bit of every passing lane set and nothing else.
__device__ __forceinline__ uint32_t swar_ge8(uint32_t w, uint32_t k8) {
  return ((w & 0x7F7F7F7Fu) + k8) & ~w & 0x80808080u;
}
__device__ __forceinline__ uint32_t swar_gt8(uint32_t w, uint32_t g8) {
  return ((w & 0x7F7F7F7Fu) + g8) & ~w & 0x80808080u;
}
__device__ __forceinline__ uint32_t swar_ge16(uint32_t w, uint32_t k16) {
  return ((w & 0x7FFF7FFFu) + k16) & ~w & 0x80008000u;
}

template <bool POS, bool TIES>
struct ScanCollect {
  uint32_t t1;  // POS: bits of tau1; otherwise key(tau1)
  uint2* cand;  // CAP entries in shared memory
  uint2* spill; // entries CAP.. in global memory (nullptr: none)
  uint32_t cap; // CAP_ALL with a spill area, else CAP
  uint32_t* ncand;    // scores above tau1 (counts past the capacity)
  uint32_t* ties;     // indices of scores equal to tau1, at most tie_cap of them
  uint32_t tie_cap;   // the row's K (at most the list's capacity)
  uint32_t* neq;      // scores equal to tau1 (counts past tie_cap)
  uint32_t xeq;       // ties this thread counted in a register once it saw the tie list full
  bool full;          // this thread saw the tie list full

  __device__ __forceinline__ bool admit(float x) const {
    if (POS) return (int32_t)__float_as_uint(x) >= (int32_t)t1;
    return fkey(x) >= t1;
  }
  __device__ __forceinline__ bool tie(float x) const {
    if (POS) return __float_as_uint(x) == t1;
    return fkey(x) == t1;
  }
  __device__ __forceinline__ uint32_t admit_mask(const float4& v) const {
    return (admit(v.x) ? 1u : 0u) | (admit(v.y) ? 2u : 0u) | (admit(v.z) ? 4u : 0u) |
           (admit(v.w) ? 8u : 0u);
  }
  __device__ __forceinline__ uint32_t tie_mask(const float4& v) const {
    return (tie(v.x) ? 1u : 0u) | (tie(v.y) ? 2u : 0u) | (tie(v.z) ? 4u : 0u) |
           (tie(v.w) ? 8u : 0u);
  }
  // Candidates appended so far (a lower bound of the final count while the
  // pass runs).
  __device__ __forceinline__ uint32_t cands_so_far() const {
    return *reinterpret_cast<const volatile uint32_t*>(ncand);
  }
  // A thread stops listing ties (and only counts them) once the list holds
  // tie_cap - (candidates so far) of them.  The answer takes ties only when
  // the K-th largest score is tau1, and then K - C(>tau1) of them; C(>tau1)
  // only grows, so the list already covers it, while a row whose admitted
  // scores number fewer than K (recovery: every tie is needed) never reaches
  // the limit.  With tie_cap = K most ties are counted in registers instead of
  // taking an atomic and a global store.
  // Counts the ties of mask q (element e of group a for bits 0-3, of group b
  // for bits 4-7) and keeps their indices while the tie list has room.
  __device__ __forceinline__ void put_ties(uint32_t q, uint32_t ia, uint32_t ib) {
    const uint32_t c = (uint32_t)__popc(q);
    if (full) {  // the list has its first tie_cap indices: only count
      xeq += c;
      return;
    }
    uint32_t t = atomicAdd(neq, c);
    if (t + c + cands_so_far() >= tie_cap) full = true;
    while (q && t < tie_cap) {
      const uint32_t e = (uint32_t)__ffs(q) - 1u;
      q &= q - 1u;
      ties[t++] = (uint32_t)((e < 4u ? ia : ib) + (e & 3u));
    }
  }
  // Appends the admitted scores of two groups of four (elements ia.. of va
  // when ha, ib.. of vb when hb) with one shared-memory atomic, visiting only
  // the admitted elements.
  __device__ __forceinline__ void lane_put2(uint32_t ia, const float4& va, bool ha, uint32_t ib,
                                            const float4& vb, bool hb) {
    const uint32_t m = (ha ? admit_mask(va) : 0u) | ((hb ? admit_mask(vb) : 0u) << 4);
    if (!m) return;
    const uint32_t q =
        TIES ? ((ha ? tie_mask(va) : 0u) | ((hb ? tie_mask(vb) : 0u) << 4)) : 0u;
    put_masked(m & ~q, q, ia, va, ib, vb);
  }
  // Candidates of mask m and ties of mask q (bits 0-3: elements ia.. of va,
  // bits 4-7: elements ib.. of vb).
  __device__ __forceinline__ void put_masked(uint32_t m, uint32_t q, uint32_t ia, const float4& va,
                                             uint32_t ib, const float4& vb) {
    if (TIES && q) put_ties(q, ia, ib);
    if (!m) return;
    uint32_t pos = atomicAdd(ncand, (uint32_t)__popc(m));
    do {
      const uint32_t e = (uint32_t)__ffs(m) - 1u;
      m &= m - 1u;
      const float4 v = e < 4u ? va : vb;
      const uint32_t k = e & 3u;
      const float x = k == 0u ? v.x : (k == 1u ? v.y : (k == 2u ? v.z : v.w));
      // an admitted score above a positive tau1 is positive: its key is its
      // bits with the sign bit set
      const uint2 ent = make_uint2((e < 4u ? ia : ib) + k,
                                   POS ? (__float_as_uint(x) | 0x80000000u) : fkey(x));
      if (pos < (uint32_t)CAP) cand[pos] = ent;
      else if (pos < cap) spill[pos - (uint32_t)CAP] = ent;
      ++pos;
    } while (m);
  }
  // Two E4M3 units, u0 from index i0 on and u1 from i1 on, tau1 > +0 with
  // byte pattern t (repeated in the four bytes of t4), and the SWAR test
  // words ge[0..7] of their 32-bit words (bit 7 of a byte set where that
  // score is >= tau1; see swar_ge8).  The strict test of the same words
  // splits them: a byte >= tau1 but not > tau1 is a tie.  Ties are counted
  // with one popc per word (and listed while the list has room), scores above
  // tau1 are appended with one atomic for both units, and only those are
  // widened.
  __device__ __forceinline__ void put_e4m3_words(uint32_t i0, const uint4& u0, uint32_t i1,
                                                 const uint4& u1, const uint32_t (&ge)[8],
                                                 uint32_t t4) {
    const uint32_t g8 = 0x7F7F7F7Fu - t4;  // (0x7F - t) in every byte
    const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t gt[8], eq[8];
    uint32_t anygt = 0, c = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      gt[k] = swar_gt8(uw[k], g8);
      eq[k] = ge[k] & ~gt[k];
      anygt |= gt[k];
      c += (uint32_t)__popc(eq[k]);
    }
    if (c) {
      if (full) {
        xeq += c;  // the list holds enough: only count
      } else {
        uint32_t t = atomicAdd(neq, c);
        if (t + c + cands_so_far() >= tie_cap) full = true;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t q = eq[k];
          while (q && t < tie_cap) {
            const uint32_t b = (uint32_t)__ffs(q) - 1u;  // bit 7 of byte b >> 3
            q &= q - 1u;
            ties[t++] = (k < 4 ? i0 : i1) + 4u * (uint32_t)(k & 3) + (b >> 3);
          }
        }
      }
    }
    if (!anygt) return;
    uint32_t n = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) n += (uint32_t)__popc(gt[k]);
    uint32_t pos = atomicAdd(ncand, n);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t q = gt[k];
      while (q) {
        const uint32_t b = (uint32_t)__ffs(q) - 1u;
        q &= q - 1u;
        const uint32_t byte = (uw[k] >> (b - 7u)) & 0xFFu;
        const uint2 ent = make_uint2((k < 4 ? i0 : i1) + 4u * (uint32_t)(k & 3) + (b >> 3),
                                     fkey(Elem<uint8_t>::widen(byte)));
        if (pos < (uint32_t)CAP) cand[pos] = ent;
        else if (pos < cap) spill[pos - (uint32_t)CAP] = ent;
        ++pos;
      }
    }
  }
  // Two bfloat16 units, u0 from index i0 on and u1 from i1 on, tau1 > +0,
  // with the SWAR test words w[0..7] of their 32-bit words (the top bit of a
  // 16-bit half set where that pattern is admitted; see swar_ge16): patterns
  // compare as signed 16-bit integers in the order of the values, so only
  // the admitted ones become keys (a positive bfloat16 widens to bits << 16,
  // whose order key is those bits with the sign bit set), and both units take
  // one shared-memory atomic.
  __device__ __forceinline__ void put_bf16_words(uint32_t i0, const uint4& u0, uint32_t i1,
                                                 const uint4& u1, const uint32_t (&w)[8]) {
    // bit e of m: element e (0-7 of u0, 8-15 of u1); the flags sit in bytes 1
    // and 3 of each word, which byte_perm gathers four at a time
    uint32_t m = flags4(__byte_perm(w[0], w[1], 0x7531u)) |
                 (flags4(__byte_perm(w[2], w[3], 0x7531u)) << 4) |
                 (flags4(__byte_perm(w[4], w[5], 0x7531u)) << 8) |
                 (flags4(__byte_perm(w[6], w[7], 0x7531u)) << 12);
    uint32_t pos = atomicAdd(ncand, (uint32_t)__popc(m));
    do {
      const uint32_t e = (uint32_t)__ffs(m) - 1u;
      m &= m - 1u;
      const uint4 u = e < 8u ? u0 : u1;
      const uint32_t k = e & 7u;
      const uint32_t wd = k < 4u ? (k < 2u ? u.x : u.y) : (k < 6u ? u.z : u.w);
      const uint32_t b = (wd >> (16u * (k & 1u))) & 0xFFFFu;
      const uint2 ent = make_uint2((e < 8u ? i0 : i1) + k, (b << 16) | 0x80000000u);
      if (pos < (uint32_t)CAP) cand[pos] = ent;
      else if (pos < cap) spill[pos - (uint32_t)CAP] = ent;
      ++pos;
    } while (m);
  }
  // 4-bit mask of the bytes of p whose top bit is set (the only bits p may
  // hold): one multiply moves bit 7 of byte j to bit 24 + j, and no two
  // partial products share a bit below 32, so nothing carries
  __device__ static __forceinline__ uint32_t flags4(uint32_t p) {
    return (((p >> 7) & 0x01010101u) * 0x01020408u) >> 24;
  }
  // Candidates of a 16-bit mask over four groups of four scores (bits 4j..4j+3:
  // elements ij.. of vj), scores without ties (FP32 rows), one atomic.
  __device__ __forceinline__ void put_masked16(uint32_t m, uint32_t ia, const float4& va,
                                               uint32_t ib, const float4& vb, uint32_t ic,
                                               const float4& vc, uint32_t id, const float4& vd) {
    uint32_t pos = atomicAdd(ncand, (uint32_t)__popc(m));
    do {
      const uint32_t e = (uint32_t)__ffs(m) - 1u;
      m &= m - 1u;
      const uint32_t j = e >> 2, k = e & 3u;
      const float4 v = j < 2u ? (j == 0u ? va : vb) : (j == 2u ? vc : vd);
      const uint32_t i = j < 2u ? (j == 0u ? ia : ib) : (j == 2u ? ic : id);
      const float x = k == 0u ? v.x : (k == 1u ? v.y : (k == 2u ? v.z : v.w));
      const uint2 ent = make_uint2(i + k, POS ? (__float_as_uint(x) | 0x80000000u) : fkey(x));
      if (pos < (uint32_t)CAP) cand[pos] = ent;
      else if (pos < cap) spill[pos - (uint32_t)CAP] = ent;
      ++pos;
    } while (m);
  }
  // Appends the admitted scores among the elements of v selected by vm
  // (element i0 + e is lane e).
  __device__ __forceinline__ void lane_put(uint32_t i0, const float4& v, uint32_t vm) {
    const uint32_t m = admit_mask(v) & vm;
    if (!m) return;
    const uint32_t q = TIES ? (tie_mask(v) & vm) : 0u;
    put_masked(m & ~q, q, i0, v, i0, v);
  }
};

// C(tau0) and the seeded histogram of the full-row pass, from candidates
// [0, n).  Returns this thread's share of C(tau0).
__device__ __forceinline__ uint32_t tally_candidates(const uint2* cand, const uint2* spill,
                                                     uint32_t n, uint32_t key0, const Bins& sb,
                                                     uint32_t* hist) {
  uint32_t c0 = 0;
  for (uint32_t j = threadIdx.x; j < n; j += THREADS) {
    const uint32_t k = cand_at(cand, spill, j).y;
    c0 += (k >= key0) ? 1u : 0u;
    atomicAdd(&hist[sb.digit(k)], 1u);
  }
  return c0;
}

// The largest admission operand of four scores (raw bits as signed integers
// when tau1 > +0; keys mapped to signed order otherwise).
template <bool POS>
__device__ __forceinline__ int32_t max_operand(const float4& v) {
  if (POS) {
    const int32_t a = (int32_t)__float_as_uint(v.x), b = (int32_t)__float_as_uint(v.y);
    const int32_t c = (int32_t)__float_as_uint(v.z), d = (int32_t)__float_as_uint(v.w);
    return max(max(a, b), max(c, d));
  }
  return (int32_t)(max(max(fkey(v.x), fkey(v.y)), max(fkey(v.z), fkey(v.w))) ^ 0x80000000u);
}

// The certify+collect pass over [start, end) of `row`, whose first `primed`
// chunks ring_prime already started.  Same ring protocol as ring_pass, with
// the consumer side shaped for the common case: a full chunk is exactly two
// 16-byte units per consumer thread, all of their scores (8 FP32, 16
// bfloat16 or 32 E4M3) are tested with one integer max, the stage is handed back as
// soon as the loads have fed that test, and only lanes holding an admitted
// score (rare) append.
// The sampler warp runs `job` meanwhile (the next row's claim and stage 1 in
// the persistent kernel; nothing elsewhere).
// CW: the ring's consumer warps (R.cw), fixed at compile time here so that
// the chunk geometry folds into the loop.
template <class E, bool POS, bool TIES, int CW, class J>
__device__ __forceinline__ void scan_pass(Ring& R, const E* __restrict__ row, int64_t start,
                                          int64_t end, ScanCollect<POS, TIES>& f,
                                          uint32_t& lflags, uint32_t primed, const J& job) {
  constexpr int P16 = Elem<E>::kPer16, NG = P16 / 4;
  constexpr uint32_t CHUNK = (uint32_t)UNIT_CHUNK_BYTES * CW;  // two units per consumer thread
  constexpr int64_t CE = CHUNK / Elem<E>::kSize;
  constexpr uint32_t C = 32u * CW;  // consumer threads
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  if (end <= start) return;
  int64_t a0, a1;
  const uint32_t nchunks = ring_span(row, start, end, CHUNK, &a0, &a1);
  if (warp == 0) {
    if (lane == 0) {
      // chunks [primed, primed + D) in one L2 prefetch, then chunk c + D as
      // chunk c is issued: D chunks of the row stay requested beyond the ring
      const uint32_t D = R.pf_ahead;
      if (D > 0 && primed == 0 && primed < nchunks) {
        const int64_t p0 = a0 + (int64_t)primed * CE;
        const int64_t p1 = min(a1, a0 + (int64_t)(primed + D) * CE);
        bulk_prefetch_l2(row + p0, (uint32_t)((p1 - p0) * Elem<E>::kSize));
      }
      for (uint32_t c = primed; c < nchunks; ++c) {
        if (D > 0 && c + D < nchunks) {
          const int64_t p0 = a0 + (int64_t)(c + D) * CE;
          const int64_t p1 = min(a1, p0 + CE);
          bulk_prefetch_l2(row + p0, (uint32_t)((p1 - p0) * Elem<E>::kSize));
        }
        ring_issue(R, row, a0, a1, c, lflags, CHUNK);
      }
    }
  } else if (warp <= (uint32_t)CW) {
    if (warp == 1) {
      // head [start, a0) on lanes 0.., tail [a1, end) on lanes 16..
      const int64_t nh = a0 - start, nt = end - a1;
      int64_t i = -1;
      if ((int64_t)lane < nh) i = start + lane;
      else if (lane >= 16 && (int64_t)lane - 16 < nt) i = a1 + (lane - 16);
      const float v = (i >= 0) ? Elem<E>::load(row + i) : 0.0f;
      if (i >= 0) f.lane_put(i, make_float4(v, 0.f, 0.f, 0.f), 1u);
    }
    const uint32_t ct = tid - 32;
    // the admission operand's threshold (for bfloat16 with tau1 > +0: the
    // upper half of tau1's FP32 bits, as a signed 16-bit value; for E4M3:
    // tau1's byte pattern)
    int32_t thr;
    if constexpr (NG == 2 && POS) thr = (int32_t)(int16_t)(f.t1 >> 16);
    else if constexpr (NG == 4 && POS)
      thr = Elem<uint8_t>::pattern_of_positive(__uint_as_float(f.t1));
    else thr = POS ? (int32_t)f.t1 : (int32_t)(f.t1 ^ 0x80000000u);
    // SWAR constant of the narrow positive thresholds: (top - t) in every lane
    const uint32_t kk = NG == 2 ? (0x8000u - (uint32_t)thr) * 0x00010001u
                                : (0x80u - (uint32_t)thr) * 0x01010101u;
    // stage and phase of the pass's first chunk, advanced per chunk; only the
    // last chunk can be short, so the others load without bounds tests.
    // Indices fit in 32 bits (N_alloc <= INT32_MAX).
    uint32_t s = R.seq % STAGES, ph = (R.seq / STAGES) & 1u;
    const uint32_t nfull = (uint32_t)((a1 - a0) / CE);
    const uint4* const sm0 = reinterpret_cast<const uint4*>(R.buf) + ct;
    uint32_t off = (uint32_t)a0;
    uint32_t c = 0;
    if constexpr (NG == 1) {
      // FP32 rows: full chunks are taken in pairs, so that one 16-score mask,
      // one atomic and one append loop serve two chunks (a warp's append
      // loop runs as long as its busiest lane, which matters less over more
      // scores); each stage is handed back as soon as its mask is formed, so
      // the ring keeps its depth.
      for (; c + 1u < nfull; c += 2u) {
        const uint32_t s1 = (s + 1u == (uint32_t)STAGES) ? 0u : s + 1u;
        const uint32_t ph1 = ph ^ ((s1 == 0u) ? 1u : 0u);
        if (!mbar_wait(&R.full[s], ph, R.abort)) lflags |= F_TIMEOUT;
        const uint4* sa = sm0 + s * (uint32_t)(STAGE_BYTES / 16);
        const uint4 u0 = sa[0], u1 = sa[C];
        uint32_t m = f.admit_mask(Elem<E>::group(u0, 0)) |
                     (f.admit_mask(Elem<E>::group(u1, 0)) << 4);
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.empty[s]);
        if (!mbar_wait(&R.full[s1], ph1, R.abort)) lflags |= F_TIMEOUT;
        const uint4* sb = sm0 + s1 * (uint32_t)(STAGE_BYTES / 16);
        const uint4 u2 = sb[0], u3 = sb[C];
        m |= (f.admit_mask(Elem<E>::group(u2, 0)) << 8) |
             (f.admit_mask(Elem<E>::group(u3, 0)) << 12);
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.empty[s1]);
        if (m) {
          const uint32_t i0 = off + (uint32_t)P16 * ct, i2 = i0 + (uint32_t)CE;
          f.put_masked16(m, i0, Elem<E>::group(u0, 0), i0 + (uint32_t)P16 * C,
                         Elem<E>::group(u1, 0), i2, Elem<E>::group(u2, 0),
                         i2 + (uint32_t)P16 * C, Elem<E>::group(u3, 0));
        }
        s = (s1 + 1u == (uint32_t)STAGES) ? 0u : s1 + 1u;
        ph = ph1 ^ ((s == 0u) ? 1u : 0u);
        off += 2u * (uint32_t)CE;
      }
    }
    for (; c < nchunks; ++c) {
      if (!mbar_wait(&R.full[s], ph, R.abort)) lflags |= F_TIMEOUT;
      const uint4* sm = sm0 + s * (uint32_t)(STAGE_BYTES / 16);
      uint4 u0, u1;
      bool ok0 = true, ok1 = true;
      if (c < nfull) {
        u0 = sm[0];
        u1 = sm[C];
      } else {
        const int nu = (int)(((uint32_t)a1 - off) / (uint32_t)P16);
        ok0 = (int)ct < nu;
        ok1 = (int)(ct + C) < nu;
        u0 = ok0 ? sm[0] : make_uint4(0u, 0u, 0u, 0u);
        u1 = ok1 ? sm[C] : make_uint4(0u, 0u, 0u, 0u);
      }
      const uint32_t i0 = off + (uint32_t)P16 * ct, i1 = i0 + (uint32_t)P16 * C;
      if constexpr (NG == 1) {
        // FP32: the admission mask of all eight scores, kept for the append
        uint32_t m = f.admit_mask(Elem<E>::group(u0, 0)) | (f.admit_mask(Elem<E>::group(u1, 0)) << 4);
        if (!ok0) m &= 0xF0u;
        if (!ok1) m &= 0x0Fu;
        // the loads have fed the mask: hand the stage back before any appends
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.empty[s]);
        if (m) f.put_masked(m, 0u, i0, Elem<E>::group(u0, 0), i1, Elem<E>::group(u1, 0));
      } else if constexpr (NG == 2 && POS && !TIES) {
        // bfloat16 with tau1 > +0: the raw 16-bit patterns compare as signed
        // integers in the order of the values; two per SWAR lane test, and
        // the test words are kept for the append
        uint32_t w[8] = {swar_ge16(u0.x, kk), swar_ge16(u0.y, kk), swar_ge16(u0.z, kk),
                         swar_ge16(u0.w, kk), swar_ge16(u1.x, kk), swar_ge16(u1.y, kk),
                         swar_ge16(u1.z, kk), swar_ge16(u1.w, kk)};
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.empty[s]);
        // a short chunk's missing units were loaded as zero, which no
        // positive threshold admits
        if ((w[0] | w[1] | w[2] | w[3] | w[4] | w[5] | w[6] | w[7]) != 0u)
          f.put_bf16_words(i0, u0, i1, u1, w);
      } else if constexpr (NG == 4 && POS) {
        // E4M3 with tau1 > +0: the raw bytes compare as signed integers in the
        // order of the values, four per SWAR lane test; the test words are
        // kept for the tie and candidate split
        uint32_t w[8] = {swar_ge8(u0.x, kk), swar_ge8(u0.y, kk), swar_ge8(u0.z, kk),
                         swar_ge8(u0.w, kk), swar_ge8(u1.x, kk), swar_ge8(u1.y, kk),
                         swar_ge8(u1.z, kk), swar_ge8(u1.w, kk)};
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.empty[s]);
        // missing units of a short chunk were loaded as zero: never admitted
        if ((w[0] | w[1] | w[2] | w[3] | w[4] | w[5] | w[6] | w[7]) != 0u)
          f.put_e4m3_words(i0, u0, i1, u1, w, (uint32_t)thr * 0x01010101u);
      } else {
        int32_t m0 = max_operand<POS>(Elem<E>::group(u0, 0));
        int32_t m1 = max_operand<POS>(Elem<E>::group(u1, 0));
#pragma unroll
        for (int k = 1; k < NG; ++k) {
          m0 = max(m0, max_operand<POS>(Elem<E>::group(u0, k)));
          m1 = max(m1, max_operand<POS>(Elem<E>::group(u1, k)));
        }
        if (!ok0) m0 = INT32_MIN;
        if (!ok1) m1 = INT32_MIN;
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.empty[s]);
        const bool h0 = m0 >= thr, h1 = m1 >= thr;
        if (h0 || h1) {
          if constexpr (NG == 2) {
            if (h0) f.lane_put2(i0, Elem<E>::group(u0, 0), true, i0 + 4, Elem<E>::group(u0, 1), true);
            if (h1) f.lane_put2(i1, Elem<E>::group(u1, 0), true, i1 + 4, Elem<E>::group(u1, 1), true);
          } else {
            // one unit and a pair of groups (eight scores) at a time: a single
            // inlined append keeps few values live
#pragma unroll 1
            for (int t = 0; t < NG; ++t) {
              const int v = t / (NG / 2), k = 2 * (t % (NG / 2));
              if (!(v ? h1 : h0)) continue;
              const uint4& u = v ? u1 : u0;
              const uint32_t ib = (v ? i1 : i0) + 4u * (uint32_t)k;
              f.lane_put2(ib, Elem<E>::group(u, k), true, ib + 4, Elem<E>::group(u, k + 1), true);
            }
          }
        }
      }
      s = (s + 1u == (uint32_t)STAGES) ? 0u : s + 1u;
      ph ^= (s == 0u) ? 1u : 0u;
      off += (uint32_t)CE;
    }
  } else {
    job();
  }
  R.seq += nchunks;
}

// The job of a sampler warp with nothing to sample.
struct NoJob {
  __device__ __forceinline__ void operator()() const {}
};

// ------------------------------------------------ frontier refinement engine
enum PassMode : uint32_t { TAKE_ALL = 0, TAKE_SOME = 1, SMALL_SORT = 2, COLLECT = 3, NEXT_HIST = 4 };

// Per-element work of one refinement pass.  The frontier is the keys in
// [bins.lo, bins.hi]; keys above the boundary bin [nlo, nhi] are emitted, keys
// inside it are handled by the mode.
struct PassF {
  Bins bins;
  uint32_t nlo, nhi;
  uint32_t mode;
  Bins nb;
  uint32_t Kr;
  Shared* S;
  uint32_t* hist;
  uint2* cand;
  int32_t* out;
  int32_t K;
  uint32_t fl;

  __device__ __forceinline__ void elem(uint32_t idx, uint32_t key, bool valid) {
    const bool inF = valid && key >= bins.lo && key <= bins.hi;
    const bool up = inF && key > nhi;
    const bool inb = inF && !up && key >= nlo;
    bool em = up;
    if (inb) {
      if (mode == TAKE_ALL) {
        em = true;
      } else if (mode == TAKE_SOME) {
        em = atomicAdd(&S->take, 1u) < Kr;
      } else if (mode == SMALL_SORT) {
        const uint32_t t = atomicAdd(&S->small_n, 1u);
        if (t < (uint32_t)SMALL) S->small[t] = make_uint2(idx, key);
      } else if (mode == COLLECT) {
        const uint32_t t = atomicAdd(&S->ncand, 1u);
        if (t < (uint32_t)CAP) cand[t] = make_uint2(idx, key);
        atomicAdd(&hist[nb.digit(key)], 1u);
      } else {
        atomicAdd(&hist[nb.digit(key)], 1u);
      }
    }
    warp_emit(out, K, idx, em, *S, fl);
  }

  __device__ __forceinline__ void quad(int64_t i0, float4 v, uint32_t vm) {
    elem((uint32_t)i0, fkey(v.x), (vm & 1u) != 0);
    elem((uint32_t)(i0 + 1), fkey(v.y), (vm & 2u) != 0);
    elem((uint32_t)(i0 + 2), fkey(v.z), (vm & 4u) != 0);
    elem((uint32_t)(i0 + 3), fkey(v.w), (vm & 8u) != 0);
  }
};

// Histogram of the keys in [bins.lo, bins.hi] (no emission).
struct HistF {
  Bins bins;
  uint32_t* hist;
  __device__ __forceinline__ void elem(uint32_t, uint32_t key, bool valid) {
    if (valid && key >= bins.lo && key <= bins.hi) atomicAdd(&hist[bins.digit(key)], 1u);
  }
  __device__ __forceinline__ void quad(int64_t i0, float4 v, uint32_t vm) {
    elem(0, fkey(v.x), (vm & 1u) != 0);
    elem(0, fkey(v.y), (vm & 2u) != 0);
    elem(0, fkey(v.z), (vm & 4u) != 0);
    elem(0, fkey(v.w), (vm & 8u) != 0);
  }
};

// Admits the keys in [lo, hi) and appends (index, key) to the candidate
// array (shared memory, then the spill area), one shared atomic per lane.
struct BandCollect {
  uint32_t lo, hi;
  uint2* cand;
  uint2* spill;
  uint32_t cap;
  uint32_t* ncand;
  __device__ __forceinline__ void quad(int64_t i0, float4 v, uint32_t vm) {
    const uint32_t k[4] = {fkey(v.x), fkey(v.y), fkey(v.z), fkey(v.w)};
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (((vm >> e) & 1u) && k[e] >= lo && k[e] < hi) m |= 1u << e;
    if (m) {
      uint32_t pos = atomicAdd(ncand, (uint32_t)__popc(m));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((m >> e) & 1u) {
          const uint2 ent = make_uint2((uint32_t)(i0 + e), k[e]);
          if (pos < (uint32_t)CAP) cand[pos] = ent;
          else if (pos < cap) spill[pos - (uint32_t)CAP] = ent;
          ++pos;
        }
      }
    }
  }
};

// Histogram of candidates [0, n) under `bins`.
__device__ __forceinline__ void hist_candidates(const uint2* cand, const uint2* spill, uint32_t n,
                                                const Bins& bins, uint32_t* hist) {
  for (uint32_t j = threadIdx.x; j < n; j += THREADS)
    atomicAdd(&hist[bins.digit(cand_at(cand, spill, j).y)], 1u);
}

// Seeded histogram of the full-row pass rebuilt from the row (keys >= bins.lo)
// together with C(tau0).
struct SeedF {
  Bins bins;
  uint32_t key0;
  uint32_t* hist;
  uint32_t c0;
  __device__ __forceinline__ void elem(uint32_t, uint32_t key, bool valid) {
    if (valid && key >= bins.lo) {
      atomicAdd(&hist[bins.digit(key)], 1u);
      c0 += (key >= key0) ? 1u : 0u;
    }
  }
  __device__ __forceinline__ void quad(int64_t, float4 v, uint32_t vm) {
    elem(0, fkey(v.x), (vm & 1u) != 0);
    elem(0, fkey(v.y), (vm & 2u) != 0);
    elem(0, fkey(v.z), (vm & 4u) != 0);
    elem(0, fkey(v.w), (vm & 8u) != 0);
  }
};

// Sources the refinement loop can iterate.  for_each() calls f.elem (or
// f.quad) warp-uniformly; the caller synchronises the block afterwards.
struct CandSrc {  // (idx, key) entries: shared memory, then the spill area
  static constexpr bool kRow = false;
  const uint2* cand;
  const uint2* spill;
  uint32_t n;
  template <class F>
  __device__ __forceinline__ void for_each(F& f, uint32_t&) const {
    const uint32_t iters = (n + THREADS - 1) / THREADS;
    for (uint32_t it = 0; it < iters; ++it) {
      const uint32_t j = threadIdx.x + it * THREADS;
      const bool ok = j < n;
      const uint2 e = ok ? cand_at(cand, spill, j) : make_uint2(0u, 0u);
      f.elem(e.x, e.y, ok);
    }
  }
};

template <class E>
struct StagedSrc {  // a whole row staged in shared memory; element i at buf[i]
  static constexpr bool kRow = false;
  const E* buf;
  uint32_t n;
  template <class F>
  __device__ __forceinline__ void for_each(F& f, uint32_t&) const {
    const uint32_t iters = (n + THREADS - 1) / THREADS;
    for (uint32_t it = 0; it < iters; ++it) {
      const uint32_t j = threadIdx.x + it * THREADS;
      const bool ok = j < n;
      const uint32_t k = ok ? fkey(Elem<E>::load(buf + j)) : 0u;
      f.elem(j, k, ok);
    }
  }
};

template <class E>
struct RowSrc {  // a row in global memory, streamed through the ring
  static constexpr bool kRow = true;
  Ring* R;
  const E* row;
  int64_t len;
  template <class F>
  __device__ __forceinline__ void for_each(F& f, uint32_t& lflags) const {
    ring_pass(*R, row, 0, len, f, lflags);
  }
};

// Exact selection of Kp keys from the frontier of `src` (keys in
// [bins.lo, bins.hi]), given `hist`, the complete histogram of that frontier
// under `bins`.  Emits into out[] through S.nout.  Every thread must call.
// QL: the source's scores have QL zero low bits in their FP32 patterns
// (narrow types), so a boundary bin narrower than 2^QL keys on one side of
// zero holds a single score value, and any Kr of its keys finish the row.
template <int QL, class Src>
__device__ void refine(const Src& src, Bins bins, uint32_t Kp, uint32_t* hist, uint2* cand,
                       int32_t* out, int32_t K, Shared& S, uint32_t& lflags) {
  for (int guard = 0; guard < 40; ++guard) {
    __syncthreads();
    phase_count(S, 9);  // refinement rounds
    find_boundary(hist, Kp, S);
    if (!S.ok) {
      lflags |= F_INTERNAL;
      return;
    }
    const uint32_t b = S.b, above = S.above, hb = hist[b];
    const uint32_t Kr = Kp - above;
    const uint32_t nlo = bins.bin_lo(b), nhi = bins.bin_hi(b);
    uint32_t mode;
    const bool one_value =
        nlo == nhi || (QL > 0 && nhi - nlo < (1u << QL) &&
                       (nlo >= 0x80000000u || nhi < 0x80000000u));
    if (hb == Kr) mode = TAKE_ALL;
    else if (one_value) mode = TAKE_SOME;
    else if (hb <= (uint32_t)SMALL) mode = SMALL_SORT;
    else if (Src::kRow && hb <= (uint32_t)CAP) mode = COLLECT;
    else mode = NEXT_HIST;
    const Bins nb = make_bins(nlo, nhi);
    __syncthreads();  // every thread has read hist[b]
    if (mode == NEXT_HIST || mode == COLLECT) clear_hist(hist);
    if (threadIdx.x == 0) {
      S.take = 0;
      S.small_n = 0;
      S.ncand = 0;
    }
    __syncthreads();
    PassF f{bins, nlo, nhi, mode, nb, Kr, &S, hist, cand, out, K, 0u};
    src.for_each(f, lflags);
    lflags |= f.fl;
    __syncthreads();
    if (mode == TAKE_ALL || mode == TAKE_SOME) return;
    if (mode == SMALL_SORT) {
      if ((threadIdx.x >> 5) == 0) {
        const uint32_t n = min(S.small_n, (uint32_t)SMALL);
        const uint32_t lane = lane_id();
        uint32_t key = 0, idx = 0xffffffffu;
        if (lane < n) {
          key = S.small[lane].y;
          idx = S.small[lane].x;
        }
        warp_sort_desc(key, idx);
        const bool em = lane < Kr && idx != 0xffffffffu;
        warp_emit(out, K, idx, em, S, lflags);
      }
      __syncthreads();
      return;
    }
    if constexpr (Src::kRow) {
      if (mode == COLLECT) {
        const CandSrc cs{cand, nullptr, min(S.ncand, (uint32_t)CAP)};
        refine<QL>(cs, nb, Kr, hist, cand, out, K, S, lflags);
        return;
      }
    }
    bins = nb;
    Kp = Kr;
  }
  lflags |= F_INTERNAL;
}

// ------------------------------------------------------------ sampler (stage 1)
struct SampleSmem {
  const uint32_t* keys;
  __device__ __forceinline__ uint32_t operator()(int64_t i) const { return keys[i]; }
};
template <class E>
struct SampleGlobal {
  const E* row;
  int64_t stride;
  uint64_t policy;
  __device__ __forceinline__ uint32_t operator()(int64_t i) const {
    return fkey(Elem<E>::load_keep(row + i * stride, policy));
  }
};

// r-th largest key (1-based) among get(0..n-1), known to lie in [lo, hi]
// with at least r keys >= lo.  Every thread must call.
template <class G>
__device__ uint32_t select_rank(const G& get, int64_t n, uint32_t r, uint32_t lo, uint32_t hi,
                                uint32_t* hist, Shared& S) {
  uint32_t rem = r;
  for (int round = 0; round < 6; ++round) {
    if (lo == hi) return lo;
    const Bins bn = make_bins(lo, hi);
    __syncthreads();
    clear_hist(hist);
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += THREADS) {
      const uint32_t k = get(i);
      if (k >= lo && k <= hi) atomicAdd(&hist[bn.digit(k)], 1u);
    }
    __syncthreads();
    find_boundary(hist, rem, S);
    if (!S.ok) return lo;  // cannot happen for a consistent source
    const uint32_t b = S.b, hb = hist[b];
    rem -= S.above;
    const uint32_t nlo = bn.bin_lo(b), nhi = bn.bin_hi(b);
    if (hb <= (uint32_t)SMALL && nlo != nhi) {
      __syncthreads();
      if (threadIdx.x == 0) S.small_n = 0;
      __syncthreads();
      for (int64_t i = threadIdx.x; i < n; i += THREADS) {
        const uint32_t k = get(i);
        if (k >= nlo && k <= nhi) {
          const uint32_t t = atomicAdd(&S.small_n, 1u);
          if (t < (uint32_t)SMALL) S.small[t] = make_uint2(0u, k);
        }
      }
      __syncthreads();
      if ((threadIdx.x >> 5) == 0) {
        const uint32_t lane = lane_id();
        const uint32_t m = min(S.small_n, (uint32_t)SMALL);
        uint32_t key = lane < m ? S.small[lane].y : 0u, idx = lane;
        warp_sort_desc(key, idx);
        if (lane == rem - 1) S.res = key;
      }
      __syncthreads();
      return S.res;
    }
    lo = nlo;
    hi = nhi;
  }
  return lo;
}

// The r0-th and r1-th largest (r0 <= r1) of keys[0..n) held in shared memory,
// whose range is [kmin, kmax].  One histogram round finds the bin holding
// the r1-th largest; when the keys from that bin up number at most THREADS
// they are gathered into `list` and ranked by counting, which yields both
// answers at once.  Otherwise two general rank selections run.  Every thread
// must call.
static __device__ void select_two_ranks(const uint32_t* keys, uint32_t n, uint32_t r0, uint32_t r1,
                                 uint32_t kmin, uint32_t kmax, uint32_t* hist, uint32_t* list,
                                 Shared& S, uint32_t* key0, uint32_t* key1) {
  if (kmin == kmax) {
    *key0 = *key1 = kmin;
    return;
  }
  const Bins bn = make_bins(kmin, kmax);
  __syncthreads();
  clear_hist(hist);
  if (threadIdx.x == 0) S.small_n = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < n; i += THREADS) atomicAdd(&hist[bn.digit(keys[i])], 1u);
  __syncthreads();
  find_boundary(hist, r1, S);
  const uint32_t lo1 = bn.bin_lo(S.b);
  const uint32_t L = S.above + hist[S.b];
  if (S.ok && L <= (uint32_t)THREADS) {
    for (uint32_t i = threadIdx.x; i < n; i += THREADS) {
      const uint32_t k = keys[i];
      if (k >= lo1) {
        const uint32_t t = atomicAdd(&S.small_n, 1u);
        if (t < (uint32_t)THREADS) list[t] = k;
      }
    }
    __syncthreads();
    const uint32_t m = min(S.small_n, (uint32_t)THREADS);
    if (threadIdx.x < m) {
      const uint32_t k = list[threadIdx.x];
      uint32_t rank = 0;
      for (uint32_t j = 0; j < m; ++j) {
        const uint32_t kj = list[j];
        rank += (kj > k || (kj == k && j < threadIdx.x)) ? 1u : 0u;
      }
      if (rank == r0 - 1) S.key0 = k;
      if (rank == r1 - 1) S.key1 = k;
    }
    __syncthreads();
    *key0 = S.key0;
    *key1 = S.key1;
    __syncthreads();
    return;
  }
  const SampleSmem g{keys};
  *key1 = select_rank(g, n, r1, kmin, kmax, hist, S);
  *key0 = select_rank(g, n, r0, *key1, kmax, hist, S);
}

// The r0-th and r1-th largest (r0 <= r1, both in [1, ns]) of the ns values
// row[0], row[stride], ... (read with an L2 evict-last hint); leaves key0/key1
// and the range [kmin, kmax] of the values' keys in S.  Every thread must
// call.
template <class E>
__device__ void thresholds_at_ranks(const E* __restrict__ row, int64_t ns, int32_t stride,
                                    uint32_t r0, uint32_t r1, uint32_t* skeys, uint32_t* hist,
                                    uint32_t* list, Shared& S) {
  const uint64_t pol = l2_policy_evict_last();
  const bool on_chip = ns <= SAMPLE_SMEM;
  uint32_t mn = 0xffffffffu, mx = 0u;
  constexpr int U = 16;  // one round trip for up to 8192 samples
  for (int64_t i0 = threadIdx.x; i0 < ns; i0 += (int64_t)THREADS * U) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + (int64_t)u * THREADS;
      v[u] = (i < ns) ? Elem<E>::load_keep(row + i * stride, pol) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + (int64_t)u * THREADS;
      if (i < ns) {
        const uint32_t k = fkey(v[u]);
        if (on_chip) skeys[i] = k;
        mn = min(mn, k);
        mx = max(mx, k);
      }
    }
  }
  uint32_t kmin, kmax;
  block_minmax(mn, mx, S, &kmin, &kmax);
  phase_mark(S, 8);
  uint32_t key1, key0;
  if (on_chip) {
    select_two_ranks(skeys, (uint32_t)ns, r0, r1, kmin, kmax, hist, list, S, &key0, &key1);
  } else {
    const SampleGlobal<E> g{row, stride, pol};
    key1 = select_rank(g, ns, r1, kmin, kmax, hist, S);
    key0 = select_rank(g, ns, r0, key1, kmax, hist, S);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    S.key0 = key0;
    S.key1 = key1;
    S.kmin = kmin;
    S.kmax = kmax;
  }
  __syncthreads();
}

// Sample rank of candidate target T for a row of len elements viewed through
// ns samples: r = clamp(ceil(T * ns / len), 1, ns).
__device__ __forceinline__ uint32_t sample_rank(uint32_t T, int64_t ns, int64_t len) {
  int64_t r = ((int64_t)T * ns + len - 1) / len;
  r = r < 1 ? 1 : (r > ns ? ns : r);
  return (uint32_t)r;
}

// Stage 1.  Samples at 0, s, 2s, ... < len; tau_j = r_j-th largest sample
// with r_j = clamp(ceil(T_j * n_s / len), 1, n_s).  Leaves key0/key1 and the
// sample key range in S.  Every thread must call.
template <class E>
__device__ void sample_thresholds(const E* __restrict__ row, int64_t len, int32_t stride,
                                  uint32_t T0, uint32_t T1, uint32_t* skeys, uint32_t* hist,
                                  uint32_t* list, Shared& S) {
  const int64_t ns = (len + stride - 1) / stride;
  thresholds_at_ranks(row, ns, stride, sample_rank(T0, ns, len), sample_rank(T1, ns, len), skeys,
                      hist, list, S);
}

// ------------------------------------------ stage 1 on one warp, ahead of time
// The same thresholds as sample_thresholds, taken by a single warp with no
// block barrier and no shared memory, so that the sampler warp can prepare
// the next row while the consumer warps stream the current one.  The ranks
// r0 <= r1 are small in every sampling tier (about rho * K / s: 12 to 18 with
// the default tiers), so the warp keeps the r1 largest sample keys seen so
// far, sorted across lanes 0..r1-1, and inserts each later key that beats the
// smallest of them; the r-th largest is then lane r-1's key.  With samples in
// no particular order a key enters with probability about r1 / (keys seen),
// so a row of n_s samples costs about r1 * (1 + ln(n_s / r1)) insertions.
constexpr uint32_t WARP_RANK_MAX = 32;  // ranks the sampler warp can take

// Returns false (nothing computed) when r1 > WARP_RANK_MAX; the row is then
// sampled at its own start.  Otherwise out = {key(tau0), key(tau1), smallest
// and largest sample key}, exactly as sample_thresholds leaves them.  Every
// lane of the warp must call.
template <class E>
__device__ __noinline__ bool warp_sample_thresholds(const E* __restrict__ row, int64_t len,
                                                   int32_t stride, uint32_t T0, uint32_t T1,
                                                   uint32_t* out) {
  const uint32_t lane = lane_id();
  const int64_t ns = (len + stride - 1) / stride;
  const uint32_t r0 = sample_rank(T0, ns, len), r1 = sample_rank(T1, ns, len);
  if (r1 > WARP_RANK_MAX || r0 > r1) return false;
  const uint64_t pol = l2_policy_evict_last();
  const uint32_t live = (r1 == 32u) ? FULL_MASK : ((1u << r1) - 1u);  // lanes of the list
  // the list: key 0 marks an empty place (only a NaN pattern has key 0, and
  // NaN is not a supported score; every valid sample has a larger key)
  uint32_t top = 0u, floor = 0u;  // floor: the list's smallest key (lane r1 - 1)
  uint32_t mn = 0xffffffffu, mx = 0u;
  constexpr int U = 8;  // 256 samples per round trip
  for (int64_t i0 = 0; i0 < ns; i0 += 32 * U) {
    uint32_t k[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + 32 * u + lane;
      k[u] = (i < ns) ? fkey(Elem<E>::load_keep(row + i * stride, pol)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + 32 * u + lane;
      if (i < ns) {
        mn = min(mn, k[u]);
        mx = max(mx, k[u]);
      }
      uint32_t m = __ballot_sync(FULL_MASK, k[u] > floor);
      while (m) {
        const uint32_t src = (uint32_t)__ffs(m) - 1u;
        m &= m - 1u;
        const uint32_t x = __shfl_sync(FULL_MASK, k[u], src);
        if (x <= floor) continue;  // the list moved past it
        // x goes after every listed key >= x; the keys below it move down
        const uint32_t pos = (uint32_t)__popc(__ballot_sync(FULL_MASK, top >= x) & live);
        const uint32_t up = __shfl_up_sync(FULL_MASK, top, 1);
        if (lane > pos) top = up;
        else if (lane == pos) top = x;
        floor = __shfl_sync(FULL_MASK, top, r1 - 1u);
      }
    }
  }
  out[0] = __shfl_sync(FULL_MASK, top, r0 - 1u);
  out[1] = floor;
  out[2] = __reduce_min_sync(FULL_MASK, mn);
  out[3] = __reduce_max_sync(FULL_MASK, mx);
  return true;
}

// Seeded bins of the full-row pass: the candidates' keys start at key(tau1);
// the regular bins span up to the largest sample, the top bin takes the rest.
__device__ __forceinline__ Bins scan_bins(uint32_t key1, uint32_t kmax) {
  return make_bins_focus(key1, 0xffffffffu, key1, kmax);
}

// Bins of the first recovery pass: the frontier is every key below key(tau1);
// the regular bins start at the smallest sample.
__device__ __forceinline__ Bins recovery_bins(uint32_t key1, uint32_t kmin) {
  const uint32_t hi = key1 - 1u;
  return make_bins_focus(0u, hi, kmin, hi);
}

__device__ __forceinline__ void write_sentinel_row(int32_t* out, int32_t K, int64_t len) {
  for (int32_t i = threadIdx.x; i < K; i += THREADS) out[i] = (i < len) ? i : -1;
}

}  // namespace tk
