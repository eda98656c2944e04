// Optional ordering of a Top-K result: each row's K indices sorted by score,
// largest first, ties by index; -1 sentinels last.  The selector's contract
// leaves the order free (codexqa.cn, section "什么叫精确，时间怎么量"), so
// this is a separate, opt-in pass over the result.
//
// One CTA per row: the K (key, index) pairs are gathered from the row into
// shared memory as 64-bit words (inverted key above, index below, so that an
// ascending sort gives the wanted order and a sentinel, all ones, sorts last)
// and sorted with a bitonic network over the next power of two >= K.
#include <cuda_runtime.h>

#include <cstdint>

#include "topk.h"
#include "score_elem.cuh"

namespace tks {

constexpr int THREADS = 512;

__device__ __forceinline__ uint32_t key_of(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;  // -0.0 sorts with +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float load_score(const float* row, int64_t i) { return row[i]; }
__device__ __forceinline__ float load_score(const uint16_t* row, int64_t i) {
  return __uint_as_float((uint32_t)row[i] << 16);
}
__device__ __forceinline__ float load_score(const uint8_t* row, int64_t i) {
  return tk::Elem<uint8_t>::widen(row[i]);
}

template <class E>
__global__ void __launch_bounds__(THREADS)
    k_sort_rows(const E* __restrict__ scores, int64_t N_alloc, int32_t K, int32_t* out_idx,
                int32_t P2) {
  extern __shared__ unsigned long long w[];
  const E* row = scores + blockIdx.x * N_alloc;
  int32_t* out = out_idx + blockIdx.x * (int64_t)K;
  for (int32_t j = threadIdx.x; j < P2; j += THREADS) {
    unsigned long long v = ~0ull;
    if (j < K) {
      const int32_t idx = out[j];
      if (idx >= 0 && idx < N_alloc)
        v = ((unsigned long long)(~key_of(load_score(row, idx))) << 32) | (uint32_t)idx;
    }
    w[j] = v;
  }
  __syncthreads();
  for (int32_t size = 2; size <= P2; size <<= 1) {
    for (int32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (int32_t t = threadIdx.x; t < (P2 >> 1); t += THREADS) {
        const int32_t lo = 2 * t - (t & (stride - 1));
        const int32_t hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long a = w[lo], b = w[hi];
        if ((a > b) == up) {
          w[lo] = b;
          w[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int32_t j = threadIdx.x; j < K; j += THREADS) {
    const unsigned long long v = w[j];
    out[j] = v == ~0ull ? -1 : (int32_t)(uint32_t)v;
  }
}

template <class E>
int sort_rows(const E* scores, int64_t N_alloc, int64_t M, int32_t K, int32_t* out_idx,
              cudaStream_t st) {
  if (M < 0 || N_alloc < 0 || K < 1) return TOPK_ERR_ARG;
  if (K > TOPK_K_MAX) return TOPK_ERR_UNSUPPORTED_K;
  if (M == 0) return TOPK_OK;
  if (M > INT32_MAX || !out_idx || (N_alloc > 0 && !scores)) return TOPK_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(out_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(scores) & (sizeof(E) - 1)))
    return TOPK_ERR_ALIGN;
  int32_t P2 = 1;
  while (P2 < K) P2 <<= 1;
  const size_t smem = (size_t)P2 * sizeof(unsigned long long);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(k_sort_rows<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return TOPK_ERR_CUDA;
  k_sort_rows<E><<<(unsigned)M, THREADS, smem, st>>>(scores, N_alloc, K, out_idx, P2);
  return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

}  // namespace tks

extern "C" {

int topk_sort_rows(const float* scores, int64_t M, int64_t N_alloc, int32_t K, int32_t* out_idx,
                   struct CUstream_st* stream) {
  return tks::sort_rows(scores, N_alloc, M, K, out_idx, reinterpret_cast<cudaStream_t>(stream));
}

int topk_sort_rows_bf16(const uint16_t* scores, int64_t M, int64_t N_alloc, int32_t K,
                        int32_t* out_idx, struct CUstream_st* stream) {
  return tks::sort_rows(scores, N_alloc, M, K, out_idx, reinterpret_cast<cudaStream_t>(stream));
}

int topk_sort_rows_e4m3(const uint8_t* scores, int64_t M, int64_t N_alloc, int32_t K,
                        int32_t* out_idx, struct CUstream_st* stream) {
  return tks::sort_rows(scores, N_alloc, M, K, out_idx, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
