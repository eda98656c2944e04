// Indexer scores on the 5th-generation tensor cores (sm_103a), the stage that
// produces the rows the selector reads.
//
// Definition (xllm-io review of LiteTopK, section "核心公式", eq. (1)):
//   I[t][s] = sum over heads j of w[t][j] * ReLU( q[t][j] . k[s] )
// with q [T][H][D] and k [S][D] in bfloat16 and w [T][H] in float; the output
// is FP32 [T][ld] with row t's scores at columns 0..S-1.
//
// GB300 design.  The contraction over D runs as tcgen05 MMAs with the KEYS on
// the M side and the QUERY HEADS on the N side: one MMA tile is 128 keys x
// (4 queries x 64 heads) x 128 dims, accumulated in FP32 in tensor memory.
// With the heads along N, a thread that reads TMEM lane m holds all 64 head
// values of key m for a query in its own registers, so the ReLU-weighted sum
// over heads is a plain per-thread FMA chain (no cross-lane reduction), and a
// warp's 32 consecutive keys store 128 contiguous bytes of an output row.
//
// One CTA per SM, persistent over work units (4 queries x a chunk of key
// tiles).  Warp roles:
//   warp 0        TMA producer: the unit's query block (64 KB, stays in shared
//                 memory for the unit) and a 4-stage ring of 32 KB key tiles,
//                 both in the 128-byte swizzled K-major layout;
//   warp 1        tensor-memory owner and MMA issuer (one thread): 8 MMAs of
//                 K = 16 per tile into one of two 256-column accumulators;
//   warps 2..5    epilogue: tcgen05.ld of the accumulator, ReLU, times w,
//                 sum over heads, masked causal suffix, coalesced stores.
// Every wait is bounded; a timeout sets an abort flag that all roles honour,
// and tensor memory is always released.
//
// Optionally the epilogue also gates every score against its query's
// threshold tau1 and appends the admitted (key, order key) pairs to that
// query's candidate area (the fused score -> select path; the thresholds come
// from a first pass of this kernel over a fixed-stride sample of the keys).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "topk.h"
#include "topk_device.cuh"
#include "topk_launch.h"

namespace tki {

constexpr int HEADS = 64;
constexpr int DIM = 128;
constexpr int QB = 4;                   // queries per work unit
constexpr int NCOL = QB * HEADS;        // MMA N = 256
constexpr int KT = 128;                 // keys per tile (MMA M)
constexpr int STAGES = 4;               // key-tile ring
constexpr int CHUNK_TILES = 256;        // key tiles per work unit
constexpr int THREADS = 192;            // 6 warps
constexpr uint32_t A_HALF = KT * 64 * 2;        // 16 KB: 128 keys x 64 dims
constexpr uint32_t A_BYTES = 2 * A_HALF;        // 32 KB
constexpr uint32_t B_HALF = NCOL * 64 * 2;      // 32 KB: 256 rows x 64 dims
constexpr uint32_t B_BYTES = 2 * B_HALF;        // 64 KB
constexpr uint32_t TMEM_COLS = 2 * NCOL;        // two accumulators
constexpr uint64_t WAIT_NS = 2000000000ull;

// shared-memory plan, offsets from a 1024-byte aligned base
constexpr uint32_t OFF_B = 0;
constexpr uint32_t OFF_A = OFF_B + B_BYTES;
constexpr uint32_t OFF_W = OFF_A + STAGES * A_BYTES;       // QB * HEADS floats
constexpr uint32_t OFF_BAR = OFF_W + QB * HEADS * 4;
constexpr uint32_t NBAR = 2 * STAGES + 2 + 4 + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
// Gated scores of the fused path are staged in shared memory, per query of
// the unit and per epilogue warp (no atomics while scoring), and flushed to
// the query's candidate area once per unit.
constexpr uint32_t STG_W = 256;                             // entries per query, warp and unit
constexpr uint32_t OFF_STG = OFF_MISC + 128;
constexpr uint32_t SMEM_BYTES = OFF_STG + QB * 4 * STG_W * 8 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory plan exceeds the opt-in limit");

__device__ uint32_t g_idx_status;  // OR of error bits since the last read

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Bounded parity wait; false (and the abort flag set) after WAIT_NS, or at
// once when another role already aborted.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (it == 0) t0 = gtime();
    else if ((it & 255u) == 0 && gtime() - t0 > WAIT_NS) {
      *abort = 1u;
      atomicOr(&g_idx_status, TOPK_FLAG_TIMEOUT);
      return false;
    }
  }
}
// Bounded wait that ignores the abort flag: lets copies and MMAs already in
// flight finish before the CTA releases its tensor memory and exits.
__device__ __forceinline__ void bar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = gtime();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok || gtime() - t0 > 100000000ull) return;
  }
}

// Two-lane FP32 fused multiply-add (fma.rn.f32x2, sm_100 family): lanes are
// the low and high halves of each 64-bit operand.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float sum2(uint64_t x) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
  return lo + hi;
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart; the tile base is 1024-byte aligned, so stepping K by 16
// elements inside a swizzle row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                   // leading offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;        // stride between 8-row groups
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}
// Instruction descriptor: BF16 x BF16 -> F32, both operands K-major.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NCOL >> 3) << 17) |
                            ((uint32_t)(KT >> 4) << 24);

struct Args {
  const float* w;          // [T][HEADS]
  const int32_t* lens;     // [T] valid prefix per query, or nullptr
  float* out;              // [T][ld]
  int64_t ld;
  int32_t T, S;
  int32_t n_tiles;         // S / KT
  int32_t n_chunks;        // ceil(n_tiles / CHUNK_TILES)
  int32_t n_units;         // (T / QB) * n_chunks
  uint8_t* rows;           // fused path: row states (tau1, candidate count and area); or nullptr
};

__device__ __forceinline__ void unit_coords(const Args& a, int32_t u, int32_t* qb, int32_t* t0,
                                            int32_t* t1) {
  *qb = u / a.n_chunks;
  const int32_t c = u % a.n_chunks;
  *t0 = c * CHUNK_TILES;
  *t1 = min(*t0 + CHUNK_TILES, a.n_tiles);
}

// End of the key tiles a unit must compute: tiles that start at or past every
// one of its queries' valid length hold only -inf and skip the MMA.
__device__ __forceinline__ int32_t unit_end(const Args& a, int32_t qb, int32_t t0, int32_t t1) {
  if (!a.lens) return t1;
  int64_t mx = 0;
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    int64_t l = a.lens[qb * QB + q];
    l = l < 0 ? 0 : (l > a.S ? a.S : l);
    mx = l > mx ? l : mx;
  }
  const int32_t te = (int32_t)((mx + KT - 1) / KT);
  return te < t0 ? t0 : (te > t1 ? t1 : te);
}

__global__ void __launch_bounds__(THREADS, 1)
    k_index_scores(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_q,
                   Args a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  float* w_s = reinterpret_cast<float*>(sm + OFF_W);
  const uint32_t bars = base + OFF_BAR;
  auto a_full = [&](uint32_t s) { return bars + 8u * s; };
  auto a_empty = [&](uint32_t s) { return bars + 8u * (STAGES + s); };
  const uint32_t b_full = bars + 8u * (2 * STAGES), b_empty = bars + 8u * (2 * STAGES + 1);
  auto acc_full = [&](uint32_t b) { return bars + 8u * (2 * STAGES + 2 + b); };
  auto acc_empty = [&](uint32_t b) { return bars + 8u * (2 * STAGES + 4 + b); };
  const uint32_t drain = bars + 8u * (2 * STAGES + 6);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  uint32_t* stg_n = misc + 2;      // [QB][4] scores each epilogue warp admitted in this unit
  uint32_t* stg_base = misc + 18;  // [QB] where the unit's go in the query's candidate area
  uint2* stg = reinterpret_cast<uint2*>(sm + OFF_STG);  // [QB][4][STG_W]
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      bar_init(a_full(s), 1);
      bar_init(a_empty(s), 1);
    }
    bar_init(b_full, 1);
    bar_init(b_empty, 1);
    for (int b = 0; b < 2; ++b) {
      bar_init(acc_full(b), 1);
      bar_init(acc_empty(b), 4);  // one arrival per epilogue warp
    }
    bar_init(drain, 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(misc)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t aseq = 0, ui = 0;  // ui counts the units that compute
      for (int32_t u = blockIdx.x; u < a.n_units && !*abort_flag; u += gridDim.x) {
        int32_t qb, t0, t1;
        unit_coords(a, u, &qb, &t0, &t1);
        const int32_t te = unit_end(a, qb, t0, t1);
        if (te == t0) continue;
        if (ui > 0 && !bar_wait(b_empty, (ui - 1) & 1u, abort_flag)) break;
        ++ui;
        bar_expect(b_full, B_BYTES);
        tma_2d(base + OFF_B, &map_q, 0, qb * NCOL, b_full);
        tma_2d(base + OFF_B + B_HALF, &map_q, 64, qb * NCOL, b_full);
        for (int32_t t = t0; t < te; ++t, ++aseq) {
          const uint32_t s = aseq % STAGES, use = aseq / STAGES;
          if (!bar_wait(a_empty(s), (use & 1u) ^ 1u, abort_flag)) break;
          const uint32_t dst = base + OFF_A + s * A_BYTES;
          bar_expect(a_full(s), A_BYTES);
          tma_2d(dst, &map_k, 0, t * KT, a_full(s));
          tma_2d(dst + A_HALF, &map_k, 64, t * KT, a_full(s));
        }
      }
      // the last copies of each kind have landed before the CTA exits
      for (uint32_t k = 0; k < aseq && k < (uint32_t)STAGES; ++k) {
        const uint32_t q = aseq - 1u - k;
        bar_drain(a_full(q % STAGES), (q / STAGES) & 1u);
      }
      if (ui > 0) bar_drain(b_full, (ui - 1u) & 1u);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t aseq = 0, accseq = 0, ui = 0;
      bool issued = false;
      for (int32_t u = blockIdx.x; u < a.n_units && !*abort_flag; u += gridDim.x) {
        int32_t qb, t0, t1;
        unit_coords(a, u, &qb, &t0, &t1);
        const int32_t te = unit_end(a, qb, t0, t1);
        if (te == t0) continue;
        if (!bar_wait(b_full, ui & 1u, abort_flag)) break;
        ++ui;
        bool ok = true;
        for (int32_t t = t0; t < te; ++t, ++aseq, ++accseq) {
          const uint32_t s = aseq % STAGES, buf = accseq & 1u;
          if (!bar_wait(a_full(s), (aseq / STAGES) & 1u, abort_flag) ||
              !bar_wait(acc_empty(buf), ((accseq >> 1) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          issued = true;
          const uint32_t a_base = base + OFF_A + s * A_BYTES, b_base = base + OFF_B;
          const uint32_t d_tmem = tmem + buf * NCOL;
#pragma unroll
          for (uint32_t kk = 0; kk < DIM / 16; ++kk) {
            const uint32_t half = kk >> 2, off = (kk & 3u) * 32u;
            const uint64_t ad = sw128_desc(a_base + half * A_HALF + off);
            const uint64_t bd = sw128_desc(b_base + half * B_HALF + off);
            const uint32_t accum = kk > 0 ? 1u : 0u;
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
                "l"(ad), "l"(bd), "r"(kIdesc), "r"(accum)
                : "memory");
          }
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                  a_empty(s))
              : "memory");
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                  acc_full(buf))
              : "memory");
        }
        if (!ok) break;
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                b_empty)
            : "memory");
      }
      // every MMA this thread issued has completed before tensor memory is
      // released
      if (issued) {
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                drain)
            : "memory");
        bar_drain(drain, 0u);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const uint32_t quarter = warp & 3u;          // TMEM lanes this warp may read
    const uint32_t row = quarter * 32u + lane;   // key within the tile
    const uint32_t etid = tid - 64u;             // 0..127
    uint32_t accseq = 0;
    bool ok = true;
    for (int32_t u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
      int32_t qb, t0, t1;
      unit_coords(a, u, &qb, &t0, &t1);
      // this unit's weights: every epilogue thread has finished the last unit
      asm volatile("bar.sync 1, 128;" ::: "memory");
      for (uint32_t i = etid; i < (uint32_t)(QB * HEADS); i += 128u)
        w_s[i] = a.w[(int64_t)qb * QB * HEADS + i];
      asm volatile("bar.sync 1, 128;" ::: "memory");
      uint32_t cnt[QB];  // this warp's admitted scores per query in the unit (warp-uniform)
#pragma unroll
      for (int q = 0; q < QB; ++q) cnt[q] = 0u;
      int32_t lenq[QB];
      float tau1q[QB];
#pragma unroll
      for (int q = 0; q < QB; ++q) {
        lenq[q] = a.lens ? a.lens[qb * QB + q] : a.S;
        const uint8_t* rs = a.rows + (size_t)(qb * QB + q) * tk::kFusedRowBytes;
        tau1q[q] = a.rows ? __ldcg(reinterpret_cast<const float*>(rs + tk::kKvTau1Off)) : 0.0f;
      }
      const int32_t te = unit_end(a, qb, t0, t1);
      // tiles past every query's valid length: -inf, no accumulator
      for (int32_t t = te; t < t1; ++t) {
        const int64_t key = (int64_t)t * KT + row;
#pragma unroll
        for (int q = 0; q < QB; ++q) a.out[((int64_t)qb * QB + q) * a.ld + key] = -INFINITY;
      }
      for (int32_t t = t0; t < te; ++t, ++accseq) {
        const uint32_t buf = accseq & 1u;
        const bool got = bar_wait(acc_full(buf), (accseq >> 1) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {  // keep the warp converged for tcgen05.ld
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int64_t key = (int64_t)t * KT + row;
        float res[QB];
#pragma unroll
        for (int q = 0; q < QB; ++q) {
          uint32_t v[32];
          uint64_t acc = 0ull;  // partial sums of the even and of the odd heads
#pragma unroll
          for (int h0 = 0; h0 < HEADS; h0 += 32) {
            const uint32_t taddr = tmem + ((quarter * 32u) << 16) + buf * NCOL + q * HEADS + h0;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31},"
                " [%32];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                  "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                  "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),
                  "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
                  "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
                  "=r"(v[30]), "=r"(v[31])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            // the weights of heads h0+j, h0+j+1 as one 64-bit pair
            const uint64_t* w2 = reinterpret_cast<const uint64_t*>(w_s + q * HEADS + h0);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const uint64_t r2 = pack2(fmaxf(__uint_as_float(v[j]), 0.0f),
                                        fmaxf(__uint_as_float(v[j + 1]), 0.0f));
              acc = ffma2(r2, w2[j >> 1], acc);
            }
          }
          res[q] = sum2(acc);
        }
        // the accumulator is in registers: hand the buffer back to the MMA
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) bar_arrive(acc_empty(buf));
        if (key < a.S) {
#pragma unroll
          for (int q = 0; q < QB; ++q) {
            const int64_t tq = (int64_t)qb * QB + q;
            a.out[tq * a.ld + key] = key < lenq[q] ? res[q] : -INFINITY;
          }
        }
        if (a.rows) {
          // the gate: scores >= tau1 of the query are staged in this warp's
          // region (positions from the ballot, no atomics)
#pragma unroll
          for (int q = 0; q < QB; ++q) {
            const bool adm = key < a.S && key < lenq[q] && res[q] >= tau1q[q];
            const uint32_t m = __ballot_sync(0xffffffffu, adm);
            const uint32_t pos = cnt[q] + (uint32_t)__popc(m & ((1u << lane) - 1u));
            if (adm && pos < STG_W)
              stg[(q * 4 + quarter) * STG_W + pos] = make_uint2((uint32_t)key, tk::fkey(res[q]));
            cnt[q] += (uint32_t)__popc(m);
          }
        }
      }
      if (a.rows) {
        // flush the unit's staged candidates: one global atomic per query
        // reserves their place (and counts C(tau1) exactly, kept or not); a
        // query whose staging overflowed is marked, and its row is then
        // served from the written scores
        if (lane == 0)
#pragma unroll
          for (int q = 0; q < QB; ++q) stg_n[q * 4 + quarter] = cnt[q];
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (etid < (uint32_t)QB) {
          uint8_t* rs = a.rows + (size_t)(qb * QB + etid) * tk::kFusedRowBytes;
          uint32_t n = 0u;
          bool lost = false;
#pragma unroll
          for (int wq = 0; wq < 4; ++wq) {
            n += stg_n[etid * 4 + wq];
            lost = lost || stg_n[etid * 4 + wq] > STG_W;
          }
          if (lost) atomicOr(reinterpret_cast<uint32_t*>(rs + tk::kKvOvfOff), 1u);
          uint32_t* count = reinterpret_cast<uint32_t*>(rs + tk::kKvNcandOff);
          stg_base[etid] = n ? atomicAdd(count, n) : 0u;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
        for (int q = 0; q < QB; ++q) {
          uint2* dst = reinterpret_cast<uint2*>(a.rows + (size_t)(qb * QB + q) * tk::kFusedRowBytes +
                                                tk::kKvCandOff);
          uint32_t g = stg_base[q];
#pragma unroll
          for (int wq = 0; wq < 4; ++wq) {
            const uint32_t n = min(stg_n[q * 4 + wq], STG_W);
            for (uint32_t j = etid; j < n; j += 128u)
              if (g + j < tk::kKvCandCap) dst[g + j] = stg[(q * 4 + wq) * STG_W + j];
            g += n;
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bfloat16 map over rows x 128 dims (row stride 256 B), box 64 dims x
// box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)DIM, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)DIM * 2};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Sample keys of the fused path and the samples' valid counts (one thread
// per 16-byte piece of a key row; then one thread per query).
__global__ void k_gather_sample_keys(const uint4* __restrict__ k, int64_t S, int32_t stride,
                                     int64_t S_s, uint4* __restrict__ ks,
                                     const int32_t* __restrict__ row_lens, int64_t T,
                                     int32_t* __restrict__ lens_s) {
  constexpr int PIECES = DIM * 2 / 16;  // 16 uint4 per key row
  const int64_t n = S_s * PIECES;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n + T;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < n) {
      const int64_t j = i / PIECES, p = i % PIECES, src = j * stride;
      ks[i] = src < S ? k[src * PIECES + p] : make_uint4(0u, 0u, 0u, 0u);
    } else {
      const int64_t t = i - n;
      int64_t l = row_lens[t];
      l = l < 0 ? 0 : (l > S ? S : l);
      lens_s[t] = (int32_t)((l + stride - 1) / stride);
    }
  }
}

cudaError_t launch_gather_sample_keys(const uint16_t* k, int64_t S, int32_t stride, int64_t S_s,
                                      uint16_t* ks, const int32_t* row_lens, int64_t T,
                                      int32_t* lens_s, cudaStream_t stream) {
  const int64_t work = S_s * (DIM * 2 / 16) + T;
  const int blocks = (int)((work + 255) / 256 < 1024 ? (work + 255) / 256 : 1024);
  k_gather_sample_keys<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(k), S, stride,
                                                   S_s, reinterpret_cast<uint4*>(ks), row_lens, T,
                                                   lens_s);
  return cudaGetLastError();
}

// Argument checks of the score stage (shapes the kernel tiles, alignment).
int check_index_args(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                     int32_t H, int32_t D, const int32_t* row_lens, const float* scores,
                     int64_t ld_scores) {
  if (T < 0 || S < 0 || ld_scores < S) return TOPK_ERR_ARG;
  if (H != HEADS || D != DIM) return TOPK_ERR_UNSUPPORTED_SHAPE;
  if (T % QB != 0 || S % KT != 0) return TOPK_ERR_UNSUPPORTED_SHAPE;
  if (T > INT32_MAX || S > INT32_MAX || T * (int64_t)HEADS > INT32_MAX) return TOPK_ERR_ARG;
  if (T == 0 || S == 0) return TOPK_OK;
  if (!q || !k || !w || !scores) return TOPK_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(k) & 15u) ||
      (reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(scores) & 3u) ||
      (row_lens && (reinterpret_cast<uintptr_t>(row_lens) & 3u)))
    return TOPK_ERR_ALIGN;
  return TOPK_OK;
}

int launch_index_scores(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                        const int32_t* row_lens, float* scores, int64_t ld_scores, uint8_t* rows,
                        cudaStream_t stream) {
  if (T == 0 || S == 0) return TOPK_OK;
  int dev = 0, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return TOPK_ERR_CUDA;
  if (major != 10 || minor != 3) return TOPK_ERR_NO_DEVICE;
  CUtensorMap mk, mq;
  if (!make_map(&mk, k, (uint64_t)S, KT) || !make_map(&mq, q, (uint64_t)T * HEADS, NCOL))
    return TOPK_ERR_CUDA;
  Args a;
  a.w = w;
  a.lens = row_lens;
  a.out = scores;
  a.ld = ld_scores;
  a.T = (int32_t)T;
  a.S = (int32_t)S;
  a.n_tiles = (int32_t)(S / KT);
  a.n_chunks = (a.n_tiles + CHUNK_TILES - 1) / CHUNK_TILES;
  const int64_t units = (T / QB) * (int64_t)a.n_chunks;
  if (units > INT32_MAX) return TOPK_ERR_ARG;
  a.n_units = (int32_t)units;
  a.rows = rows;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(k_index_scores, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return TOPK_ERR_CUDA;
  const int grid = (int)(units < sms ? units : sms);
  k_index_scores<<<grid, THREADS, SMEM_BYTES, stream>>>(mk, mq, a);
  return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

}  // namespace tki

extern "C" {

int topk_index_scores(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                      int32_t H, int32_t D, const int32_t* row_lens, float* scores,
                      int64_t ld_scores, struct CUstream_st* stream) {
  const int rc = tki::check_index_args(q, k, w, T, S, H, D, row_lens, scores, ld_scores);
  if (rc != TOPK_OK) return rc;
  return tki::launch_index_scores(q, k, w, T, S, row_lens, scores, ld_scores, nullptr,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int topk_index_topk(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                    int32_t H, int32_t D, const int32_t* row_lens, float* scores,
                    int64_t ld_scores, int32_t K, int32_t* out_idx, struct CUstream_st* stream) {
  if (!row_lens || K < 1) return TOPK_ERR_ARG;
  if (K > TOPK_K_MAX) return TOPK_ERR_UNSUPPORTED_K;
  if (T > 0 && !out_idx) return TOPK_ERR_ARG;
  const int rc = topk_index_scores(q, k, w, T, S, H, D, row_lens, scores, ld_scores, stream);
  if (rc != TOPK_OK) return rc;
  return topk_ragged(scores, row_lens, T, ld_scores, K, out_idx, stream);
}

int topk_index_read_status(struct CUstream_st* stream, uint32_t* flags) {
  if (!flags) return TOPK_ERR_ARG;
  uint32_t h = 0, zero = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyFromSymbolAsync(&h, tki::g_idx_status, sizeof h, 0, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(tki::g_idx_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                              st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return TOPK_ERR_CUDA;
  *flags = h;
  return TOPK_OK;
}

}  // extern "C"
