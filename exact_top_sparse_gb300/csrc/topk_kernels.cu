// Kernels of the sample-guided exact Top-K selector and their launchers.
//
// Three execution paths (arxivdaily abstract of "Sample-Guided Exact Top-K
// Selection for Long-Context Sparse Attention"; PaperDaily walkthrough,
// section 问题二, last paragraphs):
//   * direct     -- one CTA per row; the whole row is staged on chip with bulk
//                   copies and selected exactly there (short rows, where the
//                   codexqa.cn width sweep found an exact boundary beats
//                   sampling);
//   * persistent -- long-lived CTAs pull whole rows from a queue and run
//                   sample -> certify+collect -> refine / recover per row;
//   * KV-split   -- few very long rows: a prepare kernel samples each row, then
//                   several CTAs scan disjoint segments of one score row and
//                   merge counts, candidates and histograms in global memory;
//                   the last CTA of a row to finish (an atomic ticket, nobody
//                   waits) runs the exact refinement.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "topk_device.cuh"
#include "topk_launch.h"

namespace tk {

__device__ uint32_t g_status;  // OR of row flags since the last read

#ifdef TOPK_PHASE_TIMING
// Cycles per phase of k_persistent summed over its CTAs (thread 0's clock):
// 0 row claim, 8 first chunks and sample loads, 1 rank selection of the
// sample, 2 certify+collect pass, 3 tally, 4 next-row claim and prefetches,
// 5 selection after the pass, 6 closing the row, 7 rows served without
// sampling.
constexpr int NPHASE = 12;
__device__ unsigned long long g_phase[NPHASE];
#endif

// Per-CTA timeline of a k_persistent launch (a build with -DTOPK_PHASE_TIMING
// only; global timer, ns): slot 0 the CTA's start, 1 its exit, then for each
// of its first TL_ROWS rows five slots: row + 1, the claim, the start and the
// end of the full-row pass (0 for a row served without sampling) and the
// row's close.
constexpr int TL_CTAS = 1024, TL_ROWS = 4, TL_SLOTS = 2 + 5 * TL_ROWS;
#ifdef TOPK_PHASE_TIMING
__device__ unsigned long long g_timeline[TL_CTAS * TL_SLOTS];
#endif
__device__ __forceinline__ unsigned long long tl_now() {
#ifdef TOPK_PHASE_TIMING
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
#else
  return 0;
#endif
}
// Thread 0 writes slot `slot` of its CTA's record (no-op without the flag).
__device__ __forceinline__ void tl_put(int slot, unsigned long long v) {
#ifdef TOPK_PHASE_TIMING
  if (threadIdx.x == 0 && blockIdx.x < (unsigned)TL_CTAS && slot < TL_SLOTS)
    g_timeline[(size_t)blockIdx.x * TL_SLOTS + slot] = v;
#else
  (void)slot;
  (void)v;
#endif
}
// Field f (0..4) of the CTA's n-th row.
__device__ __forceinline__ void tl_row(int n, int f, unsigned long long v) {
  if (n < TL_ROWS) tl_put(2 + 5 * n + f, v);
}

// Sampling stride and targets of a row of `len` elements.
struct SampleSpec {
  int32_t stride;
  uint32_t target0, target1;
};
__device__ __forceinline__ uint32_t target_of(float rho, int32_t k) {
  return (uint32_t)ceil((double)rho * (double)k);
}
// `k` is the row's own K (the call's K unless per-row K values were given).
__device__ __forceinline__ SampleSpec sample_spec(const Params& P, int64_t len, int32_t k) {
  const bool lg = P.long_len > 0 && len >= P.long_len;
  if (k == P.K) {
    if (lg) return {P.long_stride, P.long_target0, P.long_target1};
    return {P.stride, P.target0, P.target1};
  }
  const uint32_t t0 = target_of(lg ? P.long_rho0 : P.rho0, k);
  const uint32_t t1 = target_of(lg ? P.long_rho1 : P.rho1, k);
  return {lg ? P.long_stride : P.stride, t0, t1 < t0 ? t0 : t1};
}

// The row's own K: the call's K, or clamp(row_k[r], 0, K) when per-row
// values were given (a value outside that range is flagged).
__device__ __forceinline__ int32_t row_k_of(const Params& P, int64_t r, uint32_t& fl) {
  if (P.row_k == nullptr) return P.K;
  int32_t k = P.row_k[r];
  if (k < 0) {
    k = 0;
    fl |= F_K_CLAMPED;
  }
  if (k > P.K) {
    k = P.K;
    fl |= F_K_CLAMPED;
  }
  return k;
}

// ------------------------------------------------------- shared-memory plan
constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
constexpr size_t SH_HDR = align_up(sizeof(Shared), 128);
constexpr size_t SH_RING = SH_HDR;
constexpr size_t SH_CAND = SH_RING + (size_t)STAGES * STAGE_BYTES;
constexpr size_t SH_HIST = SH_CAND + (size_t)CAP * sizeof(uint2);
constexpr size_t SH_LIST = SH_HIST + (size_t)NB * sizeof(uint32_t);
constexpr size_t SH_ROW_TOTAL = SH_LIST + (size_t)THREADS * sizeof(uint32_t);

// KV-split per-row state in the workspace.
struct KvHdr {
  uint32_t mode;  // 0 sentinel, 1 exact without sampling, 2 sampled
  uint32_t len;
  uint32_t key0, key1, kmin, kmax;
  uint32_t c0, ncand, ticket, ovf, flags;
  float tau0, tau1;
  int32_t k;     // the row's own K
  uint32_t neq;  // scores equal to tau1 over all segments
  uint32_t abort;  // fail-fast flag of the row's CTAs (reset by k_kv_prepare)
};
constexpr size_t KV_HIST_OFF = 256;
constexpr size_t KV_CAND_OFF = KV_HIST_OFF + (size_t)NB * sizeof(uint32_t);
constexpr size_t KV_TIE_OFF = KV_CAND_OFF + (size_t)CAP_ALL * sizeof(uint2);
constexpr size_t KV_ROW_BYTES = align_up(KV_TIE_OFF + (size_t)TIE_CAP * sizeof(uint32_t), 256);
// persistent CTA's global area: candidate spill, then the tie list
constexpr size_t CTA_AREA_BYTES = (size_t)SPILL * sizeof(uint2) + (size_t)TIE_CAP * sizeof(uint32_t);
static_assert(CTA_AREA_BYTES % 256 == 0, "CTA areas keep 256-byte alignment");
static_assert(sizeof(KvHdr) <= KV_HIST_OFF, "KV row header too large");
static_assert(KV_ROW_BYTES == kKvRowBytes, "kKvRowBytes must match the KV-split row layout");
static_assert(offsetof(KvHdr, ncand) == kKvNcandOff && offsetof(KvHdr, tau1) == kKvTau1Off &&
                  offsetof(KvHdr, ovf) == kKvOvfOff &&
                  KV_CAND_OFF == kKvCandOff && (size_t)CAP_ALL == kKvCandCap &&
                  align_up(KV_CAND_OFF + (size_t)CAP_ALL * sizeof(uint2), 256) == kFusedRowBytes,
              "fused row state must follow the KV-split row layout");

struct RowCarve {
  Shared* S;
  float* ring;
  uint2* cand;
  uint32_t* hist;
  uint32_t* list;
};

__device__ __forceinline__ RowCarve carve(uint8_t* smem) {
  RowCarve c;
  c.S = reinterpret_cast<Shared*>(smem);
  c.ring = reinterpret_cast<float*>(smem + SH_RING);
  c.cand = reinterpret_cast<uint2*>(smem + SH_CAND);
  c.hist = reinterpret_cast<uint32_t*>(smem + SH_HIST);
  c.list = reinterpret_cast<uint32_t*>(smem + SH_LIST);
  return c;
}

__device__ __forceinline__ int64_t clamp_len(int32_t raw, int64_t n_alloc, uint32_t& fl) {
  int64_t v = raw;
  if (v < 0) {
    v = 0;
    fl |= F_LEN_CLAMPED;
  }
  if (v > n_alloc) {
    v = n_alloc;
    fl |= F_LEN_CLAMPED;
  }
  return v;
}

// Closes a row of K selected slots in an output row of Kout >= K slots: pads
// a short selection (only after an internal failure) and the slots past K
// with -1, folds the per-thread flags and writes the diagnostics.  Every
// thread must call.
__device__ void finish_row(Shared& S, int32_t* out, int32_t K, int32_t Kout, uint32_t lflags,
                           RowDiag* diag, int64_t r, int32_t path, float tau0, float tau1,
                           uint32_t c0, uint32_t c1) {
  __syncthreads();
  const uint32_t nout = S.nout;
  if (nout != (uint32_t)K) {
    lflags |= F_INTERNAL;
    for (uint32_t i = min(nout, (uint32_t)K) + threadIdx.x; i < (uint32_t)K; i += THREADS)
      out[i] = -1;
  }
  for (int32_t i = K + (int32_t)threadIdx.x; i < Kout; i += THREADS) out[i] = -1;
  if (lflags) atomicOr(&S.flags, lflags);
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t fl = S.flags;
    if (fl) atomicOr(&g_status, fl);
    if (diag) {
      RowDiag d;
      d.tau0 = tau0;
      d.tau1 = tau1;
      d.count0 = c0;
      d.count1 = c1;
      d.path = path;
      d.flags = fl;
      diag[r] = d;
    }
    S.flags = 0;
  }
  __syncthreads();
}

// Exact selection without sampling, streaming the row from global memory:
// one histogram pass over the whole key range, then refinement passes.
template <class E>
__device__ void exact_row_stream(const E* row, int64_t len, int32_t* out, int32_t K, Ring& R,
                                 const RowCarve& c, uint32_t& lflags) {
  Shared& S = *c.S;
  const Bins bins = make_bins(0u, 0xffffffffu);
  __syncthreads();
  clear_hist(c.hist);
  __syncthreads();
  HistF hf{bins, c.hist};
  ring_pass(R, row, 0, len, hf, lflags);
  __syncthreads();
  refine<Elem<E>::kKeyQuantum>(RowSrc<E>{&R, row, len}, bins, (uint32_t)K, c.hist, c.cand, out, K,
                               S, lflags);
}

// Exact selection of a row staged in shared memory (element i at buf[i]):
// data-relative bins over the keys' [min, max], one histogram pass, then
// refinement rounds on chip.
template <class E>
__device__ void select_staged(const E* buf, int64_t len, int32_t* out, int32_t K, uint32_t* hist,
                              Shared& S, uint32_t& lflags) {
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int64_t i = threadIdx.x; i < len; i += THREADS) {
    const uint32_t k = fkey(Elem<E>::load(buf + i));
    mn = min(mn, k);
    mx = max(mx, k);
  }
  uint32_t kmin, kmax;
  block_minmax(mn, mx, S, &kmin, &kmax);
  const Bins bins = make_bins(kmin, kmax);
  clear_hist(hist);
  __syncthreads();
  const StagedSrc<E> src{buf, (uint32_t)len};
  HistF hf{bins, hist};
  src.for_each(hf, lflags);
  __syncthreads();
  refine<Elem<E>::kKeyQuantum>(src, bins, (uint32_t)K, hist, nullptr, out, K, S, lflags);
}

// Rows an unsampled row can be staged for in the candidate buffer (which
// such a row does not otherwise use).
template <class E>
__device__ __forceinline__ bool fits_stage(int64_t len) {
  return len * (int64_t)Elem<E>::kSize <= (int64_t)CAP * (int64_t)sizeof(uint2);
}

// Exact selection of a short row: one read of the row into the candidate
// buffer, then the on-chip selection.
template <class E>
__device__ void exact_row_staged(const E* row, int64_t len, int32_t* out, int32_t K,
                                 const RowCarve& c, uint32_t& lflags) {
  E* buf = reinterpret_cast<E*>(c.cand);
  __syncthreads();  // earlier users of the candidate buffer are done
  int64_t i = threadIdx.x;
#pragma unroll 1
  for (; i + 7 * THREADS < len; i += 8 * THREADS) {
    E v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcs(row + i + u * THREADS);
#pragma unroll
    for (int u = 0; u < 8; ++u) buf[i + u * THREADS] = v[u];
  }
  for (; i < len; i += THREADS) buf[i] = __ldcs(row + i);
  __syncthreads();
  select_staged(buf, len, out, K, c.hist, *c.S, lflags);
}

// Where the scores equal to tau1 go: their indices (the first `cap` of
// them, in global memory) and their count (shared or global memory).
struct TieList {
  uint32_t* idx;
  uint32_t cap;
  uint32_t* n;
};

// The full-row certify+collect pass over [s0, s1): candidates above tau1 in
// c.cand and past CAP in `spill` (nullptr: none), their count in S.ncand
// (past the capacity when they did not fit), the scores equal to tau1 in
// `tl` (E4M3 rows; for the other types they are candidates and the tie count
// stays 0), the seeded histogram of the kept candidates in c.hist.  Returns
// C(tau0) over the kept candidates (without the ties, which the caller adds
// when tau0 == tau1); exact unless the candidates overflowed.
template <int CW, class E, class J>
__device__ uint32_t scan_collect(const E* row, int64_t s0, int64_t s1, Ring& R,
                                 const RowCarve& c, uint2* spill, const TieList& tl,
                                 uint32_t key0, uint32_t key1, const Bins& sb, uint32_t& lflags,
                                 uint32_t primed, const J& job) {
  Shared& S = *c.S;
  const float tau1 = key_to_float(key1);
  const uint32_t cap = spill ? (uint32_t)CAP_ALL : (uint32_t)CAP;
  constexpr bool TIES = sizeof(E) == 1;  // a tie list for E4M3 rows only
  uint32_t xeq = 0;
  if (tau1 > 0.0f) {
    ScanCollect<true, TIES> f{__float_as_uint(tau1), c.cand, spill, cap, &S.ncand,
                              tl.idx, tl.cap, tl.n, 0u, false};
    scan_pass<E, true, TIES, CW>(R, row, s0, s1, f, lflags, primed, job);
    xeq = f.xeq;
  } else {
    ScanCollect<false, TIES> f{key1, c.cand, spill, cap, &S.ncand, tl.idx, tl.cap, tl.n, 0u,
                               false};
    scan_pass<E, false, TIES, CW>(R, row, s0, s1, f, lflags, primed, job);
    xeq = f.xeq;
  }
  __syncthreads();
  if constexpr (TIES) {
    // the ties counted in registers once the list was full join the count
    const uint32_t x = block_sum(xeq, S);
    if (threadIdx.x == 0 && x) atomicAdd(tl.n, x);
    __syncthreads();
  }
  phase_mark(S, 2);
  const uint32_t c0 = tally_candidates(c.cand, spill, min(S.ncand, cap), key0, sb, c.hist);
  const uint32_t total = block_sum(c0, S);
  phase_mark(S, 3);
  return total;
}

// Emits out[] entries for indices src(j), j < n (every thread calls).
template <class G>
__device__ __forceinline__ void emit_all(const G& src, uint32_t n, int32_t* out, int32_t K,
                                         Shared& S, uint32_t& lflags) {
  const uint32_t iters = (n + THREADS - 1) / THREADS;
  for (uint32_t it = 0; it < iters; ++it) {
    const uint32_t j = threadIdx.x + it * THREADS;
    const bool ok = j < n;
    warp_emit(out, K, ok ? src(j) : 0u, ok, S, lflags);
  }
}
struct CandIdx {  // candidate j's index (j < CAP: shared memory)
  const uint2* cand;
  __device__ __forceinline__ uint32_t operator()(uint32_t j) const { return cand[j].x; }
};
struct TieIdx {  // tie j's index (global memory written earlier in this kernel)
  const uint32_t* idx;
  __device__ __forceinline__ uint32_t operator()(uint32_t j) const { return __ldcg(idx + j); }
};

// Everything after the full-row pass of a sampled row whose candidates
// (c.cand, then `spill`), histogram and counts are ready: refine, or re-read
// on overflow, or recover.  Returns the row path.
// Cgt: scores above tau1 (the candidates), Ceq: scores equal to tau1 (the
// first TIE_CAP of them in `ties`); C(tau1) = Cgt + Ceq.
template <class E>
__device__ int32_t select_after_scan(const E* row, int64_t len, int32_t* out, int32_t K,
                                     Ring& R, const RowCarve& c, uint2* spill,
                                     const uint32_t* ties, const SampleSpec& sp, uint32_t& C0,
                                     uint32_t Cgt, uint32_t Ceq, bool overflow, uint32_t key0,
                                     uint32_t key1, uint32_t kmin, const Bins& sb,
                                     uint32_t& lflags) {
  Shared& S = *c.S;
  constexpr bool TIES = sizeof(E) == 1;  // only E4M3 rows keep ties apart (Ceq = 0 otherwise)
  const uint32_t C1 = Cgt + Ceq;
  int32_t path = (C0 >= (uint32_t)K) ? PATH_TAU0 : (C1 >= (uint32_t)K ? PATH_TAU1 : PATH_RECOVERY);
  if (C1 >= (uint32_t)K && !overflow) {
    if (!TIES || Cgt >= (uint32_t)K) {
      // the K-th largest score is above tau1: the ties cannot be selected
      refine<Elem<E>::kKeyQuantum>(CandSrc{c.cand, spill, Cgt}, sb, (uint32_t)K, c.hist, c.cand,
                                   out, K, S, lflags);
    } else {
      // the K-th largest score is tau1: every score above it, then any
      // K - Cgt of the ties (Cgt < K <= CAP: every candidate is on chip)
      emit_all(CandIdx{c.cand}, Cgt, out, K, S, lflags);
      emit_all(TieIdx{ties}, (uint32_t)K - Cgt, out, K, S, lflags);
    }
  } else if (C1 >= (uint32_t)K) {
    // More admitted scores than the candidate buffers hold.  The ones past
    // them were not kept, so one pass over the row rebuilds the seeded
    // histogram and C(tau0); the refinement then re-reads the row for the
    // boundary bin only.
    lflags |= F_OVERFLOW;
    __syncthreads();
    clear_hist(c.hist);
    __syncthreads();
    SeedF sf{sb, key0, c.hist, 0u};
    ring_pass(R, row, 0, len, sf, lflags);
    __syncthreads();
    C0 = block_sum(sf.c0, S);
    path = (C0 >= (uint32_t)K) ? PATH_TAU0 : PATH_TAU1;
    refine<Elem<E>::kKeyQuantum>(RowSrc<E>{&R, row, len}, sb, (uint32_t)K, c.hist, c.cand, out, K,
                                 S, lflags);
  } else {
    // C(tau1) < K: every admitted score belongs to the answer; the remaining
    // K - C(tau1) come from the scores below tau1, selected exactly from the
    // whole row.
    lflags |= F_RECOVERY;
    if (key1 == 0u) {
      lflags |= F_INTERNAL;
      return path;
    }
    // C(tau1) < K <= CAP, TIE_CAP: every admitted score was kept
    emit_all(CandIdx{c.cand}, Cgt, out, K, S, lflags);
    if constexpr (TIES) emit_all(TieIdx{ties}, Ceq, out, K, S, lflags);
    __syncthreads();
    // One pass when it suffices: a lower threshold tau2 from the same view
    // (rank of the target 2 * T1) admits the band [tau2, tau1); if the band
    // holds the K - C(tau1) still missing and fits the candidate buffers, it
    // is refined on chip.  Otherwise the two-pass selection below runs.
    const uint32_t need = (uint32_t)K - C1;
    const uint32_t cap = spill ? (uint32_t)CAP_ALL : (uint32_t)CAP;
    sample_thresholds(row, len, sp.stride, 2u * sp.target1, 2u * sp.target1,
                      reinterpret_cast<uint32_t*>(c.cand), c.hist, c.list, S);
    const uint32_t key2 = S.key1;
    if (key2 < key1) {
      if (threadIdx.x == 0) S.ncand = 0;
      __syncthreads();
      BandCollect bf{key2, key1, c.cand, spill, cap, &S.ncand};
      ring_pass(R, row, 0, len, bf, lflags);
      __syncthreads();
      const uint32_t n2 = S.ncand;
      if (n2 >= need && n2 <= cap) {
        const Bins bb = make_bins(key2, key1 - 1u);
        clear_hist(c.hist);
        __syncthreads();
        hist_candidates(c.cand, spill, n2, bb, c.hist);
        refine<Elem<E>::kKeyQuantum>(CandSrc{c.cand, spill, n2}, bb, need, c.hist, c.cand, out, K,
                                     S, lflags);
        return path;
      }
    }
    const Bins rb = recovery_bins(key1, kmin);
    __syncthreads();
    clear_hist(c.hist);
    __syncthreads();
    HistF hf{rb, c.hist};
    ring_pass(R, row, 0, len, hf, lflags);
    __syncthreads();
    refine<Elem<E>::kKeyQuantum>(RowSrc<E>{&R, row, len}, rb, (uint32_t)K - C1, c.hist, c.cand,
                                 out, K, S, lflags);
  }
  return path;
}

// The sampler warp's job while a persistent CTA streams a sampled row:
// claim the next row and, when that row is sampled, take its stage 1
// (warp_sample_thresholds, the same thresholds sample_thresholds gives), so
// that the row starts its full-row pass as soon as this one is done.  The
// results reach the other warps through S after the block barrier that ends
// the pass.
template <class E>
struct NextRowJob {
  const E* scores;
  const int32_t* row_lens;
  const Params* P;
  uint32_t* queue;
  Shared* S;
  __device__ __forceinline__ void operator()() const {
    const uint32_t lane = lane_id();
    uint32_t rn = 0;
    if (lane == 0) rn = atomicAdd(queue, 1u);
    rn = __shfl_sync(FULL_MASK, rn, 0);
    uint32_t key[4] = {0u, 0u, 0u, 0u};
    bool sampled = false;
    if ((int64_t)rn < P->M) {
      uint32_t fl = 0;
      const int64_t ln = clamp_len(row_lens[rn], P->N_alloc, fl);
      const int32_t kn = row_k_of(*P, rn, fl);
      if (ln > kn && kn > 0 && ln >= P->sample_min_len) {
        const E* row = scores + (int64_t)rn * P->N_alloc;
        if (lane == 0 && P->pf_next_bytes) prefetch_row_head(row, ln, P->pf_next_bytes);
        const SampleSpec sp = sample_spec(*P, ln, kn);
        sampled = warp_sample_thresholds(row, ln, sp.stride, sp.target0, sp.target1, key);
      }
    }
    if (lane == 0) {
      S->next = rn;
      S->next_ok = 1u;
      S->nx_row = rn;
      S->nx_ok = sampled ? 1u : 0u;
      for (int j = 0; j < 4; ++j) S->nx_key[j] = key[j];
    }
  }
};

// Warms L2 with the sample points of a row the CTA takes next (evict-last,
// as the sampler's own loads), so that its sampling, latency-bound DRAM
// loads otherwise, reads L2 instead.  Issued while the current row is
// refined (persistent kernel without a sampler warp).  Every address lies
// inside the row's valid prefix.  Every thread may call.
template <class E>
__device__ void warm_samples(const E* row, int64_t len, int32_t stride) {
  const int64_t ns = (len + stride - 1) / stride;
  for (int64_t i = threadIdx.x; i < ns; i += THREADS) prefetch_l2_keep(row + i * stride);
}

// ------------------------------------------------------------ persistent path
// CW: consumer warps, CONSUMER_WARPS, or one fewer with the last warp as
// the sampler warp (Params::sampler_warp says which instance is launched).
template <class E, int CW>
__global__ void __launch_bounds__(THREADS, 2)
    k_persistent(const E* __restrict__ scores, const int32_t* __restrict__ row_lens,
                 int32_t* __restrict__ out_idx, RowDiag* __restrict__ diag, uint32_t* hdr,
                 uint2* __restrict__ spill_all, const __grid_constant__ Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const RowCarve c = carve(smem);
  // this CTA's global area: candidate spill, then the tie list
  uint8_t* area = reinterpret_cast<uint8_t*>(spill_all) + (size_t)blockIdx.x * CTA_AREA_BYTES;
  uint2* spill = reinterpret_cast<uint2*>(area);
  uint32_t* ties = reinterpret_cast<uint32_t*>(area + (size_t)SPILL * sizeof(uint2));
  Shared& S = *c.S;
  tl_put(0, tl_now());
  int nrow = 0;  // rows this CTA has taken (timeline only)
  if (threadIdx.x == 0) {
    S.flags = 0;
    S.next_ok = 0;
    S.nx_ok = 0;
#ifdef TOPK_PHASE_TIMING
    for (int i = 0; i < NPHASE; ++i) S.ph[i] = 0;
    S.ph_t = clock64();
#endif
  }
  Ring R;
  // hdr[2]: this launch's fail-fast flag; with CW = 14, warp 15 samples
  ring_init(R, S, c.ring, hdr + 2, (uint32_t)CW);
  R.pf_ahead = P.pf_ahead;
  const int32_t K = P.K;
  for (;;) {
    if (threadIdx.x == 0) {
      S.row = S.next_ok ? S.next : atomicAdd(&hdr[0], 1u);
      S.next_ok = 0;
    }
    __syncthreads();
    const int64_t r = S.row;
    // stage 1 of this row, when the sampler warp took it during the last pass
    const bool pre = CW < CONSUMER_WARPS && S.nx_ok != 0u && (int64_t)S.nx_row == r;
    const uint32_t pk0 = S.nx_key[0], pk1 = S.nx_key[1], pk2 = S.nx_key[2], pk3 = S.nx_key[3];
    __syncthreads();
    phase_mark(S, 0);
    if (r >= P.M) break;
    tl_row(nrow, 0, (unsigned long long)r + 1u);
    tl_row(nrow, 1, tl_now());
    uint32_t lflags = 0;
    const int64_t len = clamp_len(row_lens[r], P.N_alloc, lflags);
    const E* row = scores + r * P.N_alloc;
    int32_t* out = out_idx + r * (int64_t)K;
    if (threadIdx.x == 0) {
      S.nout = 0;
      S.nx_ok = 0;
    }
    __syncthreads();
    const float qnan = __int_as_float(0x7fc00000);
    const int32_t K0 = row_k_of(P, r, lflags);
    if (len <= K0 || K0 == 0) {
      write_sentinel_row(out, K0, len);
      if (threadIdx.x == 0) S.nout = (uint32_t)K0;
      finish_row(S, out, K0, K, lflags, diag, r, PATH_SENTINEL, qnan, qnan, 0, 0);
      phase_mark(S, 7);
      tl_row(nrow++, 4, tl_now());
      continue;
    }
    if (len < P.sample_min_len) {
      if (fits_stage<E>(len)) exact_row_staged(row, len, out, K0, c, lflags);
      else exact_row_stream(row, len, out, K0, R, c, lflags);
      finish_row(S, out, K0, K, lflags, diag, r, PATH_DIRECT, qnan, qnan, 0, 0);
      phase_mark(S, 7);
      tl_row(nrow++, 4, tl_now());
      continue;
    }
    // the ring is idle: start the row's first chunks before sampling it
    const uint32_t primed = ring_prime(R, row, 0, len, lflags);
    uint32_t key0 = pk0, key1 = pk1, kmin = pk2, kmax = pk3;
    if (!pre) {
      const SampleSpec sp = sample_spec(P, len, K0);
      sample_thresholds(row, len, sp.stride, sp.target0, sp.target1,
                        reinterpret_cast<uint32_t*>(c.cand), c.hist, c.list, S);
      key0 = S.key0;
      key1 = S.key1;
      kmin = S.kmin;
      kmax = S.kmax;
    }
    phase_mark(S, 1);
    tl_row(nrow, 2, tl_now());
    const Bins sb = scan_bins(key1, kmax);
    __syncthreads();
    clear_hist(c.hist);
    if (threadIdx.x == 0) {
      S.ncand = 0;
      S.neq = 0;
    }
    __syncthreads();
    // a sampler warp claims the next row and takes its stage 1 meanwhile
    const TieList tl{ties, (uint32_t)min(K0, (int32_t)TIE_CAP), &S.neq};
    uint32_t C0;
    if constexpr (CW == CONSUMER_WARPS)
      C0 = scan_collect<CW>(row, 0, len, R, c, spill, tl, key0, key1, sb, lflags, primed, NoJob{});
    else
      C0 = scan_collect<CW>(row, 0, len, R, c, spill, tl, key0, key1, sb, lflags, primed,
                            NextRowJob<E>{scores, row_lens, &P, hdr, &S});
    const uint32_t Cgt = S.ncand, Ceq = S.neq;
    tl_row(nrow, 3, tl_now());
    if (key0 == key1) C0 += Ceq;
    if (CW == CONSUMER_WARPS) {
      // claim the next row now and warm L2 with its sample points while
      // this one is refined
      if (threadIdx.x == 0) {
        S.next = atomicAdd(&hdr[0], 1u);
        S.next_ok = 1u;
      }
      __syncthreads();
      const int64_t rn = S.next;
      if (rn < P.M) {
        uint32_t fl = 0;
        const int64_t ln = clamp_len(row_lens[rn], P.N_alloc, fl);
        const int32_t kn = row_k_of(P, rn, fl);
        if (ln > kn && kn > 0 && ln >= P.sample_min_len) {
          warm_samples(scores + rn * P.N_alloc, ln, sample_spec(P, ln, kn).stride);
          if (threadIdx.x == 0 && P.pf_next_bytes)
            prefetch_row_head(scores + rn * P.N_alloc, ln, P.pf_next_bytes);
        }
      }
    }
    phase_mark(S, 4);
    // the row's K and sampling spec again, rather than held in registers
    // over the scan
    const int32_t Kr = row_k_of(P, r, lflags);
    const int32_t path =
        select_after_scan(row, len, out, Kr, R, c, spill, ties, sample_spec(P, len, Kr), C0, Cgt,
                          Ceq, Cgt > (uint32_t)CAP_ALL, key0, key1, kmin, sb, lflags);
    phase_mark(S, 5);
    finish_row(S, out, Kr, K, lflags, diag, r, path, key_to_float(key0), key_to_float(key1), C0,
               Cgt + Ceq);
    phase_mark(S, 6);
    tl_row(nrow++, 4, tl_now());
  }
  tl_put(1, tl_now());
#ifdef TOPK_PHASE_TIMING
  if (threadIdx.x == 0)
    for (int i = 0; i < NPHASE; ++i) atomicAdd(&g_phase[i], S.ph[i]);
#endif
  ring_drain(R);
  // The last CTA to leave resets the queue and the fail-fast flag, so the
  // next launch (or graph replay) on this workspace starts from zero without
  // a separate memset.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&hdr[1], 1u) == gridDim.x - 1) {
      atomicExch(&hdr[0], 0u);
      atomicExch(&hdr[1], 0u);
      atomicExch(&hdr[2], 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------- direct path
template <class E>
__global__ void __launch_bounds__(THREADS, 1)
    k_direct(const E* __restrict__ scores, const int32_t* __restrict__ row_lens,
             int32_t* __restrict__ out_idx, RowDiag* __restrict__ diag, Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  Shared& S = *reinterpret_cast<Shared*>(smem);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + SH_HDR);
  E* stage = reinterpret_cast<E*>(smem + SH_HDR + (size_t)NB * sizeof(uint32_t));
  const int64_t r = blockIdx.x;
  const int32_t K = P.K;
  uint32_t lflags = 0;
  const int64_t len = clamp_len(row_lens[r], P.N_alloc, lflags);
  const int32_t Kr = row_k_of(P, r, lflags);
  const E* row = scores + r * P.N_alloc;
  int32_t* out = out_idx + r * (int64_t)K;
  const float qnan = __int_as_float(0x7fc00000);
  if (threadIdx.x == 0) {
    S.flags = 0;
    S.nout = 0;
  }
  __syncthreads();
  if (len <= Kr || Kr == 0) {
    write_sentinel_row(out, Kr, len);
    if (threadIdx.x == 0) S.nout = (uint32_t)Kr;
    finish_row(S, out, Kr, K, lflags, diag, r, PATH_SENTINEL, qnan, qnan, 0, 0);
    return;
  }
  // Stage the row: the 16-byte aligned body by bulk copies, head and tail
  // singly.  Element i lives at buf[i] with buf = stage + sh, where sh makes
  // the body's first element land on a 16-byte boundary.
  constexpr int P16 = Elem<E>::kPer16;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  int64_t a0 = (int64_t)(((16u - (uint32_t)(addr & 15u)) & 15u) / Elem<E>::kSize);
  if (a0 > len) a0 = len;
  const int64_t a1 = a0 + ((len - a0) & ~(int64_t)(P16 - 1));
  const int64_t sh = (P16 - (a0 % P16)) % P16;
  E* buf = stage + sh;
  if (threadIdx.x == 0) {
    mbar_init(&S.full[0], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t pol = l2_policy_evict_first();
    const uint32_t bytes = (uint32_t)((a1 - a0) * Elem<E>::kSize);
    mbar_arrive_expect_tx(&S.full[0], bytes);
    constexpr uint32_t PIECE = 32768;
    for (uint32_t o = 0; o < bytes; o += PIECE) {
      const uint32_t nb = (bytes - o) < PIECE ? (bytes - o) : PIECE;
      bulk_load(reinterpret_cast<uint8_t*>(buf + a0) + o,
                reinterpret_cast<const uint8_t*>(row + a0) + o, nb, &S.full[0], pol);
    }
  }
  for (int64_t i = threadIdx.x; i < a0; i += THREADS) buf[i] = row[i];
  for (int64_t i = a1 + threadIdx.x; i < len; i += THREADS) buf[i] = row[i];
  if (!mbar_wait(&S.full[0], 0, nullptr)) {  // one wait per CTA: nothing to fail fast
    lflags |= F_TIMEOUT;
    // gave up: still let the copies land (bounded) before this CTA moves on
    if (threadIdx.x == 0) mbar_wait_drain(&S.full[0], 0, 100000000ull);
  }
  __syncthreads();
  select_staged(buf, len, out, Kr, hist, S, lflags);
  finish_row(S, out, Kr, K, lflags, diag, r, PATH_DIRECT, qnan, qnan, 0, 0);
}

// --------------------------------------------------------------- KV-split path
__device__ __forceinline__ KvHdr* kv_hdr(uint8_t* ws_rows, int64_t r) {
  return reinterpret_cast<KvHdr*>(ws_rows + (size_t)r * KV_ROW_BYTES);
}

// One CTA per row: lengths, thresholds, and a fresh merge state.
template <class E>
__global__ void __launch_bounds__(THREADS, 1)
    k_kv_prepare(const E* __restrict__ scores, const int32_t* __restrict__ row_lens,
                 uint8_t* __restrict__ ws_rows, Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  Shared& S = *reinterpret_cast<Shared*>(smem);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + SH_HDR);
  uint32_t* list = hist + NB;
  uint32_t* skeys = list + THREADS;
  const int64_t r = blockIdx.x;
  uint32_t lflags = 0;
  const int64_t len = clamp_len(row_lens[r], P.N_alloc, lflags);
  const int32_t Kr = row_k_of(P, r, lflags);
  const E* row = scores + r * P.N_alloc;
  uint8_t* base = ws_rows + (size_t)r * KV_ROW_BYTES;
  KvHdr* h = reinterpret_cast<KvHdr*>(base);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(base + KV_HIST_OFF);
  for (int i = threadIdx.x; i < NB; i += THREADS) ghist[i] = 0;
  uint32_t mode = 2;
  if (len <= Kr || Kr == 0) mode = 0;
  else if (len < P.sample_min_len) mode = 1;
  uint32_t key0 = 0, key1 = 0, kmin = 0, kmax = 0;
  if (mode == 2) {
    const SampleSpec sp = sample_spec(P, len, Kr);
    sample_thresholds(row, len, sp.stride, sp.target0, sp.target1, skeys, hist, list, S);
    key0 = S.key0;
    key1 = S.key1;
    kmin = S.kmin;
    kmax = S.kmax;
  }
  if (threadIdx.x == 0) {
    h->mode = mode;
    h->len = (uint32_t)len;
    h->key0 = key0;
    h->key1 = key1;
    h->kmin = kmin;
    h->kmax = kmax;
    h->c0 = 0;
    h->ncand = 0;
    h->neq = 0;
    h->ticket = 0;
    h->ovf = 0;
    h->flags = lflags;
    h->tau0 = key_to_float(key0);
    h->tau1 = key_to_float(key1);
    h->k = Kr;
    h->abort = 0;
  }
}

template <class E>
__global__ void __launch_bounds__(THREADS, 2)
    k_kv_segment(const E* __restrict__ scores, int32_t* __restrict__ out_idx,
                 RowDiag* __restrict__ diag, uint8_t* __restrict__ ws_rows, Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const RowCarve c = carve(smem);
  Shared& S = *c.S;
  const int64_t item = blockIdx.x;
  const int64_t r = item / P.segments;
  const int32_t seg = (int32_t)(item % P.segments);
  uint8_t* base = ws_rows + (size_t)r * KV_ROW_BYTES;
  KvHdr* h = reinterpret_cast<KvHdr*>(base);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(base + KV_HIST_OFF);
  uint2* gcand = reinterpret_cast<uint2*>(base + KV_CAND_OFF);
  uint32_t* gties = reinterpret_cast<uint32_t*>(base + KV_TIE_OFF);
  const uint32_t mode = h->mode;
  const int64_t len = h->len;
  const uint32_t key0 = h->key0, key1 = h->key1, kmin = h->kmin, kmax = h->kmax;
  const E* row = scores + r * P.N_alloc;
  const int32_t K = P.K;
  const int32_t Kr = h->k;
  if (threadIdx.x == 0) {
    S.flags = 0;
    S.nout = 0;
  }
  Ring R;
  ring_init(R, S, c.ring, &h->abort);
  R.pf_ahead = P.pf_ahead;
  uint32_t lflags = 0;
  const Bins sb = scan_bins(key1, kmax);
  if (mode == 2) {
    const int64_t s0 = len * seg / P.segments, s1 = len * (seg + 1) / P.segments;
    clear_hist(c.hist);
    if (threadIdx.x == 0) S.ncand = 0;
    __syncthreads();
    const uint32_t C0 = scan_collect<CONSUMER_WARPS>(row, s0, s1, R, c, nullptr,
                                     TieList{gties, (uint32_t)TIE_CAP, &h->neq}, key0, key1, sb,
                                     lflags, 0u, NoJob{});
    const uint32_t nloc = S.ncand;
    if (threadIdx.x == 0) {
      atomicAdd(&h->c0, C0);
      S.res = atomicAdd(&h->ncand, nloc);
      if (nloc > (uint32_t)CAP) atomicOr(&h->ovf, 1u);
    }
    __syncthreads();
    const uint32_t gbase = S.res;
    const uint32_t ncopy = min(nloc, (uint32_t)CAP);
    for (uint32_t j = threadIdx.x; j < ncopy; j += THREADS) {
      if (gbase + j < (uint32_t)CAP_ALL) gcand[gbase + j] = c.cand[j];
    }
    for (int i = threadIdx.x; i < NB; i += THREADS) {
      const uint32_t v = c.hist[i];
      if (v) atomicAdd(&ghist[i], v);
    }
  }
  // Ticket: the CTA that completes the row's last segment selects it.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t t = atomicAdd(&h->ticket, 1u);
    S.last = (t == (uint32_t)P.segments - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!S.last) {
    ring_drain(R);
    return;
  }
  __threadfence();
  int32_t* out = out_idx + r * (int64_t)K;
  const float qnan = __int_as_float(0x7fc00000);
  lflags |= __ldcg(&h->flags);
  if (mode == 0) {
    write_sentinel_row(out, Kr, len);
    if (threadIdx.x == 0) S.nout = (uint32_t)Kr;
    finish_row(S, out, Kr, K, lflags, diag, r, PATH_SENTINEL, qnan, qnan, 0, 0);
    ring_drain(R);
    return;
  }
  if (mode == 1) {
    if (fits_stage<E>(len)) exact_row_staged(row, len, out, Kr, c, lflags);
    else exact_row_stream(row, len, out, Kr, R, c, lflags);
    finish_row(S, out, Kr, K, lflags, diag, r, PATH_DIRECT, qnan, qnan, 0, 0);
    ring_drain(R);
    return;
  }
  uint32_t C0 = __ldcg(&h->c0);
  const uint32_t Cgt = __ldcg(&h->ncand), Ceq = __ldcg(&h->neq);
  if (key0 == key1) C0 += Ceq;
  const bool overflow = __ldcg(&h->ovf) != 0u || Cgt > (uint32_t)CAP_ALL;
  for (int i = threadIdx.x; i < NB; i += THREADS) c.hist[i] = __ldcg(&ghist[i]);
  const uint32_t nload = min(Cgt, (uint32_t)CAP);
  for (uint32_t j = threadIdx.x; j < nload; j += THREADS) {
    const uint2* p = gcand + j;
    c.cand[j] = make_uint2(__ldcg(&p->x), __ldcg(&p->y));
  }
  __syncthreads();
  const int32_t path =
      select_after_scan(row, len, out, Kr, R, c, gcand + CAP, gties, sample_spec(P, len, Kr), C0,
                        Cgt, Ceq, overflow, key0, key1, kmin, sb, lflags);
  finish_row(S, out, Kr, K, lflags, diag, r, path, key_to_float(key0), key_to_float(key1), C0,
             Cgt + Ceq);
  ring_drain(R);
}

// ------------------------------------------------------ fused score -> select
// The fused path applies the method one stage earlier: the sample view of a
// row is the score kernel's own output at keys 0, s, 2s, ... < len (computed
// first, from those keys alone), its thresholds follow the same rank rule,
// and the full-row pass is the score kernel itself, whose epilogue admits
// every score >= tau1 into the row's candidate area while it writes the row.
// The selection then certifies C(tau0) >= K from the candidates and refines
// them; a row the candidates cannot serve (C(tau1) < K, or more candidates
// than the area holds) is served from the materialised row by the same
// recovery and re-read paths as every other row.

// One CTA per row: the row's mode and thresholds from its sample scores.
__global__ void __launch_bounds__(THREADS, 1)
    k_fused_prepare(const float* __restrict__ sscores, int64_t ld_s,
                    const int32_t* __restrict__ row_lens, uint8_t* __restrict__ rows, Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  Shared& S = *reinterpret_cast<Shared*>(smem);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + SH_HDR);
  uint32_t* list = hist + NB;
  uint32_t* skeys = list + THREADS;
  const int64_t r = blockIdx.x;
  uint32_t lflags = 0;
  const int64_t len = clamp_len(row_lens[r], P.N_alloc, lflags);
  const int32_t Kr = row_k_of(P, r, lflags);
  KvHdr* h = reinterpret_cast<KvHdr*>(rows + (size_t)r * kFusedRowBytes);
  uint32_t mode = 2;
  if (len <= Kr || Kr == 0) mode = 0;
  else if (len < P.sample_min_len) mode = 1;
  uint32_t key0 = 0, key1 = 0, kmin = 0, kmax = 0;
  if (mode == 2) {
    const SampleSpec sp = sample_spec(P, len, Kr);
    const int64_t ns = (len + sp.stride - 1) / sp.stride;
    thresholds_at_ranks(sscores + r * ld_s, ns, 1, sample_rank(sp.target0, ns, len),
                        sample_rank(sp.target1, ns, len), skeys, hist, list, S);
    key0 = S.key0;
    key1 = S.key1;
    kmin = S.kmin;
    kmax = S.kmax;
  }
  if (threadIdx.x == 0) {
    h->mode = mode;
    h->len = (uint32_t)len;
    h->key0 = key0;
    h->key1 = key1;
    h->kmin = kmin;
    h->kmax = kmax;
    h->c0 = 0;
    h->ncand = 0;
    h->neq = 0;
    h->ticket = 0;
    h->ovf = 0;
    h->flags = lflags;
    h->tau0 = key_to_float(key0);
    h->tau1 = mode == 2 ? key_to_float(key1) : __int_as_float(0x7f800000);  // +inf: admit none
    h->k = Kr;
    h->abort = 0;
  }
}

// One CTA per row: C(tau0) and the seeded histogram from the candidates the
// score kernel appended, then the selection (refinement, or the recovery and
// re-read paths over the materialised row).
__global__ void __launch_bounds__(THREADS, 2)
    k_fused_finish(const float* __restrict__ scores, int64_t ld, int32_t* __restrict__ out_idx,
                   RowDiag* __restrict__ diag, uint8_t* __restrict__ rows, Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const RowCarve c = carve(smem);
  Shared& S = *c.S;
  const int64_t r = blockIdx.x;
  uint8_t* base = rows + (size_t)r * kFusedRowBytes;
  KvHdr* h = reinterpret_cast<KvHdr*>(base);
  uint2* gcand = reinterpret_cast<uint2*>(base + KV_CAND_OFF);
  if (threadIdx.x == 0) {
    S.flags = 0;
    S.nout = 0;
  }
  Ring R;
  ring_init(R, S, c.ring, &h->abort);
  R.pf_ahead = P.pf_ahead;
  const uint32_t mode = __ldcg(&h->mode);
  const int64_t len = __ldcg(&h->len);
  const uint32_t key0 = __ldcg(&h->key0), key1 = __ldcg(&h->key1), kmin = __ldcg(&h->kmin),
                 kmax = __ldcg(&h->kmax);
  const int32_t K = P.K;
  const int32_t Kr = __ldcg(&h->k);
  uint32_t lflags = __ldcg(&h->flags);
  const float* row = scores + r * ld;
  int32_t* out = out_idx + r * (int64_t)K;
  const float qnan = __int_as_float(0x7fc00000);
  if (mode == 0) {
    write_sentinel_row(out, Kr, len);
    if (threadIdx.x == 0) S.nout = (uint32_t)Kr;
    finish_row(S, out, Kr, K, lflags, diag, r, PATH_SENTINEL, qnan, qnan, 0, 0);
    ring_drain(R);
    return;
  }
  if (mode == 1) {
    if (fits_stage<float>(len)) exact_row_staged(row, len, out, Kr, c, lflags);
    else exact_row_stream(row, len, out, Kr, R, c, lflags);
    finish_row(S, out, Kr, K, lflags, diag, r, PATH_DIRECT, qnan, qnan, 0, 0);
    ring_drain(R);
    return;
  }
  const uint32_t Cgt = __ldcg(&h->ncand);
  // some admitted scores were not kept (the score kernel's staging of a unit
  // overflowed): the count C(tau1) is still exact, the candidates are not
  const bool lost = __ldcg(&h->ovf) != 0u;
  if (lost && Cgt < (uint32_t)Kr) {
    // fewer than K admitted, and not all of them at hand: the exact
    // selection over the whole written row
    lflags |= F_OVERFLOW | F_RECOVERY;
    exact_row_stream(row, len, out, Kr, R, c, lflags);
    finish_row(S, out, Kr, K, lflags, diag, r, PATH_RECOVERY, key_to_float(key0),
               key_to_float(key1), 0, Cgt);
    ring_drain(R);
    return;
  }
  const bool overflow = lost || Cgt > (uint32_t)CAP_ALL;
  const uint32_t nkeep = min(Cgt, (uint32_t)CAP_ALL), nload = min(Cgt, (uint32_t)CAP);
  for (uint32_t j = threadIdx.x; j < nload; j += THREADS) {
    const uint2* p = gcand + j;
    c.cand[j] = make_uint2(__ldcg(&p->x), __ldcg(&p->y));
  }
  const Bins sb = scan_bins(key1, kmax);
  clear_hist(c.hist);
  __syncthreads();
  const uint32_t c0 = tally_candidates(c.cand, gcand + CAP, nkeep, key0, sb, c.hist);
  uint32_t C0 = block_sum(c0, S);
  const int32_t path =
      select_after_scan(row, len, out, Kr, R, c, gcand + CAP, nullptr, sample_spec(P, len, Kr), C0,
                        Cgt, 0u, overflow, key0, key1, kmin, sb, lflags);
  finish_row(S, out, Kr, K, lflags, diag, r, path, key_to_float(key0), key_to_float(key1), C0,
             Cgt);
  ring_drain(R);
}

// ------------------------------------------------------------------ launchers
size_t persistent_smem_bytes() { return SH_ROW_TOTAL; }
size_t kv_segment_smem_bytes() { return SH_ROW_TOTAL; }
size_t kv_prepare_smem_bytes() {
  return SH_HDR + (size_t)(NB + THREADS + SAMPLE_SMEM) * sizeof(uint32_t);
}
size_t direct_smem_bytes(int64_t n_alloc, int elem_bytes) {
  // the row plus up to one 16-byte unit of alignment shift
  return SH_HDR + (size_t)NB * sizeof(uint32_t) +
         align_up((size_t)n_alloc * elem_bytes + 16, 16);
}
size_t kv_row_bytes() { return KV_ROW_BYTES; }
size_t fused_prepare_smem_bytes() { return kv_prepare_smem_bytes(); }
size_t persistent_spill_bytes() { return CTA_AREA_BYTES; }

static cudaError_t set_smem(const void* fn, size_t bytes) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t prepare_device() {
  cudaError_t e;
  int dev = 0, optin = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
      cudaSuccess)
    return e;
  const void* row_kernels[] = {
      (const void*)k_persistent<float, CONSUMER_WARPS>,
      (const void*)k_persistent<uint16_t, CONSUMER_WARPS>,
      (const void*)k_persistent<uint8_t, CONSUMER_WARPS>,
      (const void*)k_persistent<float, CONSUMER_WARPS - 1>,
      (const void*)k_persistent<uint16_t, CONSUMER_WARPS - 1>,
      (const void*)k_persistent<uint8_t, CONSUMER_WARPS - 1>, (const void*)k_kv_segment<float>,
      (const void*)k_kv_segment<uint16_t>, (const void*)k_kv_segment<uint8_t>};
  for (const void* fn : row_kernels)
    if ((e = set_smem(fn, persistent_smem_bytes())) != cudaSuccess) return e;
  const void* prep_kernels[] = {(const void*)k_kv_prepare<float>,
                                (const void*)k_kv_prepare<uint16_t>,
                                (const void*)k_kv_prepare<uint8_t>};
  for (const void* fn : prep_kernels)
    if ((e = set_smem(fn, kv_prepare_smem_bytes())) != cudaSuccess) return e;
  if ((e = set_smem((const void*)k_fused_prepare, kv_prepare_smem_bytes())) != cudaSuccess) return e;
  if ((e = set_smem((const void*)k_fused_finish, persistent_smem_bytes())) != cudaSuccess) return e;
  const void* direct_kernels[] = {(const void*)k_direct<float>, (const void*)k_direct<uint16_t>,
                                  (const void*)k_direct<uint8_t>};
  for (const void* fn : direct_kernels)
    if ((e = set_smem(fn, (size_t)optin)) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t persistent_occupancy(int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_persistent<float, CONSUMER_WARPS>, THREADS,
                                                       persistent_smem_bytes());
}

template <class E>
static cudaError_t launch_direct_t(const E* scores, const int32_t* row_lens, int32_t* out,
                                   RowDiag* diag, const Params& P, cudaStream_t st) {
  k_direct<E><<<(unsigned)P.M, THREADS, direct_smem_bytes(P.N_alloc, Elem<E>::kSize), st>>>(
      scores, row_lens, out, diag, P);
  return cudaGetLastError();
}

template <class E>
static cudaError_t launch_persistent_t(const E* scores, const int32_t* row_lens, int32_t* out,
                                       RowDiag* diag, uint32_t* hdr, void* spill, int grid,
                                       const Params& P, cudaStream_t st) {
  if (P.sampler_warp)
    k_persistent<E, CONSUMER_WARPS - 1><<<grid, THREADS, persistent_smem_bytes(), st>>>(
      scores, row_lens, out, diag, hdr, static_cast<uint2*>(spill), P);
  else
    k_persistent<E, CONSUMER_WARPS><<<grid, THREADS, persistent_smem_bytes(), st>>>(
      scores, row_lens, out, diag, hdr, static_cast<uint2*>(spill), P);
  return cudaGetLastError();
}

template <class E>
static cudaError_t launch_kvsplit_t(const E* scores, const int32_t* row_lens, int32_t* out,
                                    RowDiag* diag, uint8_t* ws_rows, const Params& P,
                                    cudaStream_t st) {
  k_kv_prepare<E><<<(unsigned)P.M, THREADS, kv_prepare_smem_bytes(), st>>>(scores, row_lens,
                                                                           ws_rows, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t items = P.M * (int64_t)P.segments;
  k_kv_segment<E><<<(unsigned)items, THREADS, kv_segment_smem_bytes(), st>>>(scores, out, diag,
                                                                            ws_rows, P);
  return cudaGetLastError();
}

cudaError_t launch_direct(const void* scores, const int32_t* row_lens, int32_t* out,
                          RowDiag* diag, const Params& P, cudaStream_t st) {
  if (P.elem_bytes == 2)
    return launch_direct_t(static_cast<const uint16_t*>(scores), row_lens, out, diag, P, st);
  if (P.elem_bytes == 1)
    return launch_direct_t(static_cast<const uint8_t*>(scores), row_lens, out, diag, P, st);
  return launch_direct_t(static_cast<const float*>(scores), row_lens, out, diag, P, st);
}

cudaError_t launch_persistent(const void* scores, const int32_t* row_lens, int32_t* out,
                              RowDiag* diag, uint32_t* hdr, void* spill, int grid, const Params& P,
                              cudaStream_t st) {
  if (P.elem_bytes == 2)
    return launch_persistent_t(static_cast<const uint16_t*>(scores), row_lens, out, diag, hdr,
                               spill, grid, P, st);
  if (P.elem_bytes == 1)
    return launch_persistent_t(static_cast<const uint8_t*>(scores), row_lens, out, diag, hdr,
                               spill, grid, P, st);
  return launch_persistent_t(static_cast<const float*>(scores), row_lens, out, diag, hdr, spill,
                             grid, P, st);
}

cudaError_t launch_kvsplit(const void* scores, const int32_t* row_lens, int32_t* out,
                           RowDiag* diag, uint8_t* ws_rows, const Params& P, cudaStream_t st) {
  if (P.elem_bytes == 2)
    return launch_kvsplit_t(static_cast<const uint16_t*>(scores), row_lens, out, diag, ws_rows, P,
                            st);
  if (P.elem_bytes == 1)
    return launch_kvsplit_t(static_cast<const uint8_t*>(scores), row_lens, out, diag, ws_rows, P,
                            st);
  return launch_kvsplit_t(static_cast<const float*>(scores), row_lens, out, diag, ws_rows, P, st);
}

cudaError_t launch_fused_prepare(const float* sscores, int64_t ld_s, const int32_t* row_lens,
                                 uint8_t* rows, const Params& P, cudaStream_t st) {
  k_fused_prepare<<<(unsigned)P.M, THREADS, kv_prepare_smem_bytes(), st>>>(sscores, ld_s, row_lens,
                                                                          rows, P);
  return cudaGetLastError();
}

cudaError_t launch_fused_finish(const float* scores, int64_t ld, int32_t* out, RowDiag* diag,
                                uint8_t* rows, const Params& P, cudaStream_t st) {
  k_fused_finish<<<(unsigned)P.M, THREADS, persistent_smem_bytes(), st>>>(scores, ld, out, diag,
                                                                         rows, P);
  return cudaGetLastError();
}

// Self-test of the bounded wait: one thread waits on a barrier that nothing
// completes, with the kernels' own wait routine and a short limit; giving up
// sets F_TIMEOUT in the status word.  The probe's fail-fast flag is its own
// (a local), so no later launch sees it.  No copy or other memory operation
// is pending meanwhile.
__global__ void k_wait_probe(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort;
  if (threadIdx.x == 0) {
    abort = 0u;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_slow(&bar, 0u, &abort, limit_ns)) atomicOr(&g_status, F_TIMEOUT);
  }
}

cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t st) {
  k_wait_probe<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_and_clear_status(cudaStream_t st, uint32_t* flags) {
  uint32_t h = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_status, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(st);
  *flags = h;
  return e;
}

}  // namespace tk

#ifdef TOPK_PHASE_TIMING
// Reads (and with reset != 0 clears) the phase cycle sums of k_persistent on
// the current device.  Exported only by a build with -DTOPK_PHASE_TIMING.
extern "C" int topk_debug_phase_cycles(unsigned long long* out, int reset) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -4;
  if (cudaMemcpyFromSymbol(out, tk::g_phase, sizeof(tk::g_phase)) != cudaSuccess) return -4;
  if (reset) {
    static const unsigned long long zero[tk::NPHASE] = {};
    if (cudaMemcpyToSymbol(tk::g_phase, zero, sizeof(zero)) != cudaSuccess) return -4;
  }
  return 0;
}

// Copies the timeline records of CTAs [0, ctas) of the last k_persistent
// launches into out (ctas * slots values; with reset != 0 clears them first
// instead) and returns the slots per CTA (negative on a CUDA error).
// Exported only by a build with -DTOPK_PHASE_TIMING.
extern "C" int topk_debug_timeline(unsigned long long* out, int ctas, int reset) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -4;
  if (reset) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, tk::g_timeline) != cudaSuccess) return -4;
    if (cudaMemset(p, 0, sizeof(tk::g_timeline)) != cudaSuccess) return -4;
    if (cudaDeviceSynchronize() != cudaSuccess) return -4;
  } else if (out && ctas > 0) {
    const int n = ctas < tk::TL_CTAS ? ctas : tk::TL_CTAS;
    if (cudaMemcpyFromSymbol(out, tk::g_timeline,
                             (size_t)n * tk::TL_SLOTS * sizeof(unsigned long long)) != cudaSuccess)
      return -4;
  }
  return tk::TL_SLOTS;
}
#endif
