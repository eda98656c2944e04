// Internal interface between the C-ABI layer and the kernels (not installed).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace tk {

// Per-call parameters passed by value to every kernel.
struct Params {
  int64_t M;
  int64_t N_alloc;
  int32_t K;
  int32_t stride;
  uint32_t target0;  // ceil(rho0 * K)
  uint32_t target1;  // ceil(rho1 * K)
  int64_t sample_min_len;
  int32_t segments;  // KV-split segments per row
  int32_t elem_bytes;  // 4: FP32 scores, 2: bfloat16 scores, 1: FP8 E4M3 scores
  int64_t long_len;  // rows this long or longer sample with the long_* values (0: none)
  int32_t long_stride;
  uint32_t long_target0;
  uint32_t long_target1;
  // Per-row K (nullptr: every row takes K).  Row r then selects
  // clamp(row_k[r], 0, K) and its targets are ceil(rho * that) with the rho
  // of its sampling tier; the output row stride stays K.
  const int32_t* row_k;
  float rho0, rho1, long_rho0, long_rho1;
  // L2 prefetch of the row a full-row pass streams: the producer keeps
  // pf_ahead chunks ahead of its shared-memory ring prefetched into L2 (0:
  // none), and a persistent CTA prefetches the first pf_next_bytes of the
  // row it takes next as soon as its current row's pass ends (0: none).
  uint32_t pf_ahead;
  uint32_t pf_next_bytes;
  // Persistent kernel: 1 when its last warp, instead of consuming chunks,
  // claims the next row and takes its stage 1 during each certify pass (14
  // consumer warps, 14 KB chunks); 0 for 15 consumer warps, the next row then
  // claimed after the pass and sampled at its own start.
  uint32_t sampler_warp;
};

// Same layout as topk_row_diag in the public header.
struct RowDiag {
  float tau0, tau1;
  int64_t count0, count1;
  int32_t path;
  uint32_t flags;
};

size_t persistent_smem_bytes();
size_t kv_segment_smem_bytes();
size_t kv_prepare_smem_bytes();
size_t direct_smem_bytes(int64_t n_alloc, int elem_bytes);
size_t kv_row_bytes();
// Bytes of KV-split merge state per row (equals kv_row_bytes()).
constexpr size_t kKvRowBytes = 155904;

// Row state of the fused score -> select path: the KV-split row header and
// candidate area (no tie list), which the score kernel's epilogue fills.
// Offsets inside a row state (checked against the KV-split layout where it
// is defined):
constexpr size_t kKvNcandOff = 28;      // uint32: admitted scores (counts past the capacity)
constexpr size_t kKvOvfOff = 36;        // uint32: nonzero when admitted scores were not kept
constexpr size_t kKvTau1Off = 48;       // float: tau1 (+inf: the row admits nothing)
constexpr size_t kKvCandOff = 8448;     // uint2 (index, order key) entries
constexpr uint32_t kKvCandCap = 16384;  // entries kept
constexpr size_t kFusedRowBytes = 139520;
// Bytes of global memory per persistent CTA (candidate spill area and tie list).
size_t persistent_spill_bytes();

// Sets the kernels' shared-memory limits on the current device.
cudaError_t prepare_device();
cudaError_t persistent_occupancy(int* blocks_per_sm);

cudaError_t launch_direct(const void* scores, const int32_t* row_lens, int32_t* out,
                          RowDiag* diag, const Params& P, cudaStream_t st);
cudaError_t launch_persistent(const void* scores, const int32_t* row_lens, int32_t* out,
                              RowDiag* diag, uint32_t* hdr, void* spill, int grid, const Params& P,
                              cudaStream_t st);
cudaError_t launch_kvsplit(const void* scores, const int32_t* row_lens, int32_t* out,
                           RowDiag* diag, uint8_t* ws_rows, const Params& P, cudaStream_t st);

cudaError_t read_and_clear_status(cudaStream_t st, uint32_t* flags);
cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t st);

// Fused score -> select.  After the sample scores exist: k_fused_prepare
// (one CTA per row) writes each row state's thresholds from its sample
// scores sscores[r][0 .. ceil(len_r / P.stride)); after the score kernel has
// appended the scores >= tau1 of every row: k_fused_finish (one CTA per row)
// selects from the candidates, or from the materialised row `scores` when
// the candidates do not certify the row.
size_t fused_prepare_smem_bytes();
cudaError_t launch_fused_prepare(const float* sscores, int64_t ld_s, const int32_t* row_lens,
                                 uint8_t* rows, const Params& P, cudaStream_t st);
cudaError_t launch_fused_finish(const float* scores, int64_t ld, int32_t* out, RowDiag* diag,
                                uint8_t* rows, const Params& P, cudaStream_t st);

}  // namespace tk

namespace tki {

// Argument checks of topk_index_scores(): TOPK_OK or the status it returns.
int check_index_args(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                     int32_t H, int32_t D, const int32_t* row_lens, const float* scores,
                     int64_t ld_scores);

// Indexer scores of topk_index_scores() (shapes and pointers already
// checked), optionally gating them: with `rows` non-null, every score at
// key s < row_lens[t] that is >= the row state's tau1 is also appended to row
// t's candidate area (row states kFusedRowBytes apart).
int launch_index_scores(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                        const int32_t* row_lens, float* scores, int64_t ld_scores, uint8_t* rows,
                        cudaStream_t stream);

// Sample keys of the fused path: ks[j] = k[j * stride] for j * stride < S,
// zero rows up to S_s; lens_s[t] = ceil(clamp(row_lens[t], 0, S) / stride).
cudaError_t launch_gather_sample_keys(const uint16_t* k, int64_t S, int32_t stride, int64_t S_s,
                                      uint16_t* ks, const int32_t* row_lens, int64_t T,
                                      int32_t* lens_s, cudaStream_t stream);

}  // namespace tki
