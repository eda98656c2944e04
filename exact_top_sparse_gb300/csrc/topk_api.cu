// C ABI of the exact Top-K selector: argument checks, the host planner that
// picks the execution path, the per-(device, stream) workspace cache and the
// host-buffer pipeline.  The planner reads only sizes and device properties,
// never device memory, so every call can be captured in a CUDA graph once its
// workspace exists (the pages' timings are CUDA-graph replays: codexqa.cn
// article, section "什么叫精确，时间怎么量"; graph-capturable ragged-row dispatch:
// arxivdaily abstract).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/topk.h"
#include "topk_launch.h"

namespace {

constexpr int kVersion = 10300;  // 1.3.0: FP8 E4M3 rows (1.2.0: per-row K; 1.1.0: bfloat16
                                 // rows, ordered output, indexer scores)
constexpr size_t kHdrBytes = 256;
constexpr int64_t kMinSegment = 32768;  // floats per KV-split segment, at least
// Planner crossovers, measured on GB300 over 128K-1M columns and M = 64-2048:
// with at least two rows per resident CTA the persistent queue balances
// well; below that, rows of 768K+ elements leave a long tail on the
// persistent path and are split, and shorter rows are split only when they
// would leave half the CTAs idle (512K x 256 / x 512: persistent 0.121 /
// 0.224 ms, split 0.134 / 0.231; 768K x 512: 0.320 against 0.307; 1M x 512:
// 0.397 against 0.381).  KV-split cuts rows into segments of about 256K
// floats, and into more when that gives fewer CTAs than resident.
constexpr int kPersistentRowsPerCta = 2;
constexpr int64_t kKvLongRow = 786432;
constexpr int64_t kKvSegmentTarget = 262144;

std::mutex g_mu;
topk_params g_params;
bool g_params_init = false;
// L2 prefetch distances of the full-row pass (see tk::Params): four chunks
// (60 KB) kept requested beyond the ring measured 3.7 % faster on 1M-column
// rows (5.35 -> 5.15 ms at 8192 rows) and neutral below 512K; eight gave
// less, sixteen or more lost (the lines left L2 before the ring read them).
// Prefetching the next row's head during the current row's selection gave
// nothing on any width.
uint32_t g_knob_pf_ahead = 4;
uint32_t g_knob_pf_next_bytes = 0;
// The persistent kernel's sampler warp (see tk::Params::sampler_warp): -1
// chooses by row width and element size, 0 and 1 force it (tuning builds).
int g_knob_sampler = -1;

// Whether a persistent launch over rows of N_alloc elements of elem_bytes
// each gives its last warp to sampling the next row.  The certify pass is
// bound by its consumer warps' instructions, so one warp fewer streams about
// 1/15 slower, while the next row's stage 1 (about 6 us per row on the whole
// CTA) leaves the critical path.  Measured (8192 causal rows, ms per call,
// without / with): FP32 128K 1.029 / 0.936, 256K 1.566 / 1.496, 512K 2.737 /
// 2.750, 1M 5.073 / 5.125; bfloat16 1M 3.197 / 3.047; E4M3 1M 2.600 / 2.524.
// FP32 rows of 512K elements and more stream without it.
bool use_sampler_warp(int64_t N, int elem_bytes) {
  if (g_knob_sampler >= 0) return g_knob_sampler != 0;
  return elem_bytes < 4 || N < ((int64_t)1 << 19);
}

struct DevInfo {
  bool ready = false;
  int sm_count = 0;
  int occ = 0;
  size_t optin = 0;
};
std::map<int, DevInfo> g_dev;

struct Buf {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, uintptr_t>, Buf> g_ws;  // (device, stream) -> workspace
// Workspaces a stream has grown out of.  A CUDA graph captured earlier on
// that stream still holds their addresses, so they stay allocated until
// topk_release_workspaces().
std::vector<std::pair<int, void*>> g_retired;

struct HostPipe {
  std::mutex mu;  // one host-buffer call at a time per device
  float* scores[2] = {nullptr, nullptr};
  int32_t* lens[2] = {nullptr, nullptr};
  int32_t* out[2] = {nullptr, nullptr};
  size_t score_bytes = 0, lens_bytes = 0, out_bytes = 0;
  cudaStream_t st[2] = {nullptr, nullptr};
};
std::map<int, HostPipe> g_pipe;

void defaults(topk_params* p) {
  p->stride = 256;
  p->rho0 = 2.0f;
  p->rho1 = 2.25f;
  p->sample_min_len = 12288;
  p->direct_max = 16384;
  p->force_kind = TOPK_KIND_AUTO;
  p->kv_segments = 0;
  p->long_len = 786432;
  p->long_stride = 512;
  p->long_rho0 = 2.75f;
  p->long_rho1 = 3.0f;
}

topk_params params_snapshot() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_params_init) {
    defaults(&g_params);
    g_params_init = true;
  }
  return g_params;
}

int device_info(DevInfo* out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return TOPK_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return TOPK_ERR_NO_DEVICE;  // built for sm_103a only
    if (tk::prepare_device() != cudaSuccess) return TOPK_ERR_CUDA;
    int occ = 0;
    if (tk::persistent_occupancy(&occ) != cudaSuccess || occ < 1) return TOPK_ERR_CUDA;
    d.sm_count = prop.multiProcessorCount;
    d.occ = occ;
    d.optin = prop.sharedMemPerBlockOptin;
    d.ready = true;
  }
  *out = d;
  if (dev_out) *dev_out = dev;
  return TOPK_OK;
}

struct Plan {
  int kind = TOPK_KIND_AUTO;
  int grid = 0;
  int segments = 1;
  size_t ws = 0;
  size_t smem = 0;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

int check_sizes(int64_t M, int64_t N, int32_t K) {
  if (M < 0 || N < 0 || N > INT32_MAX || M > INT32_MAX) return TOPK_ERR_ARG;
  if (K < 1) return TOPK_ERR_ARG;
  if (K > TOPK_K_MAX) return TOPK_ERR_UNSUPPORTED_K;
  if (M > 0 && N > 0 && M > INT64_MAX / N) return TOPK_ERR_ARG;
  return TOPK_OK;
}

int make_plan(int64_t M, int64_t N, int32_t K, const topk_params& p, const DevInfo& d, Plan* pl,
              int elem_bytes = 4) {
  (void)K;
  const int resident = d.sm_count * d.occ;
  const bool direct_fits = tk::direct_smem_bytes(N, elem_bytes) <= d.optin;
  int kind = p.force_kind;
  if (kind == TOPK_KIND_DIRECT && !direct_fits) return TOPK_ERR_ARG;
  if (kind == TOPK_KIND_AUTO) {
    if (N <= p.direct_max && direct_fits) kind = TOPK_KIND_DIRECT;
    else if (M >= (int64_t)kPersistentRowsPerCta * resident) kind = TOPK_KIND_PERSISTENT;
    else if (N >= kKvLongRow || 2 * M < (int64_t)resident) kind = TOPK_KIND_KVSPLIT;
    else kind = TOPK_KIND_PERSISTENT;
  }
  int segments = 1;
  if (kind == TOPK_KIND_KVSPLIT) {
    int64_t P = p.kv_segments;
    if (P <= 0) {
      const int64_t by_len = (N + kKvSegmentTarget - 1) / kKvSegmentTarget;
      const int64_t by_fill = ((int64_t)resident + M - 1) / (M > 0 ? M : 1);
      P = by_len > by_fill ? by_len : by_fill;
      int64_t pmax = N / kMinSegment;
      if (pmax < 1) pmax = 1;
      if (P > pmax) P = pmax;
    }
    if (P < 1) P = 1;
    if (P > 4096) P = 4096;
    if (M * P > INT32_MAX) return TOPK_ERR_ARG;
    if (P == 1 && p.force_kind != TOPK_KIND_KVSPLIT) kind = TOPK_KIND_PERSISTENT;
    segments = (int)P;
  }
  pl->kind = kind;
  pl->segments = (kind == TOPK_KIND_KVSPLIT) ? segments : 1;
  pl->ws = kHdrBytes;
  if (kind == TOPK_KIND_DIRECT) {
    pl->grid = (int)M;
    pl->smem = tk::direct_smem_bytes(N, elem_bytes);
  } else if (kind == TOPK_KIND_PERSISTENT) {
    pl->grid = (int)(M < resident ? M : resident);
    pl->smem = tk::persistent_smem_bytes();
    pl->ws += (size_t)pl->grid * tk::persistent_spill_bytes();
  } else {
    pl->grid = (int)(M * pl->segments);
    pl->smem = tk::kv_segment_smem_bytes();
    pl->ws += (size_t)M * tk::kv_row_bytes();
  }
  return TOPK_OK;
}

int validate_ptrs(const void* scores, const int32_t* row_lens, int64_t M, int64_t N,
                  int32_t* out_idx, int elem_bytes = 4) {
  if (M == 0) return TOPK_OK;
  if (!row_lens || !out_idx) return TOPK_ERR_ARG;
  if (N > 0 && !scores) return TOPK_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(scores) & (uintptr_t)(elem_bytes - 1)) ||
      (reinterpret_cast<uintptr_t>(out_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(row_lens) & 3u))
    return TOPK_ERR_ALIGN;
  return TOPK_OK;
}

tk::Params kernel_params(int64_t M, int64_t N, int32_t K, const topk_params& p, const Plan& pl,
                         int elem_bytes = 4) {
  tk::Params P;
  P.elem_bytes = elem_bytes;
  P.M = M;
  P.N_alloc = N;
  P.K = K;
  P.stride = p.stride;
  P.target0 = (uint32_t)std::ceil((double)p.rho0 * (double)K);
  P.target1 = (uint32_t)std::ceil((double)p.rho1 * (double)K);
  if (P.target1 < P.target0) P.target1 = P.target0;
  P.long_len = p.long_len;
  P.long_stride = p.long_stride;
  P.long_target0 = (uint32_t)std::ceil((double)p.long_rho0 * (double)K);
  P.long_target1 = (uint32_t)std::ceil((double)p.long_rho1 * (double)K);
  if (P.long_target1 < P.long_target0) P.long_target1 = P.long_target0;
  P.sample_min_len = p.sample_min_len;
  P.segments = pl.segments;
  P.row_k = nullptr;
  P.rho0 = p.rho0;
  P.rho1 = p.rho1;
  P.long_rho0 = p.long_rho0;
  P.long_rho1 = p.long_rho1;
  P.pf_ahead = g_knob_pf_ahead;
  P.pf_next_bytes = g_knob_pf_next_bytes;
  P.sampler_warp = use_sampler_warp(N, elem_bytes) ? 1u : 0u;
  return P;
}

int launch(const Plan& pl, const tk::Params& P, const void* scores, const int32_t* row_lens,
           int32_t* out_idx, topk_row_diag* diag, void* ws, cudaStream_t st) {
  tk::RowDiag* d = reinterpret_cast<tk::RowDiag*>(diag);
  cudaError_t e;
  if (pl.kind == TOPK_KIND_DIRECT) {
    e = tk::launch_direct(scores, row_lens, out_idx, d, P, st);
  } else if (pl.kind == TOPK_KIND_PERSISTENT) {
    e = tk::launch_persistent(scores, row_lens, out_idx, d, static_cast<uint32_t*>(ws),
                              static_cast<uint8_t*>(ws) + kHdrBytes, pl.grid, P, st);
  } else {
    e = tk::launch_kvsplit(scores, row_lens, out_idx, d,
                           static_cast<uint8_t*>(ws) + kHdrBytes, P, st);
  }
  return e == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

// Workspace for (current device, stream), grown on demand (at least doubling,
// so a stream retires few buffers).  The buffer it replaces is never freed
// here: a graph captured on this stream may still use it, so it moves to
// g_retired.  A new buffer is zero-filled on the call's own stream, ahead of
// the kernels that read it (the persistent queue counters and the fail-fast
// flag must start at zero).
int cached_workspace(int dev, cudaStream_t st, size_t need, void** ptr) {
  std::lock_guard<std::mutex> lk(g_mu);
  Buf& b = g_ws[{dev, reinterpret_cast<uintptr_t>(st)}];
  if (b.bytes >= need && b.ptr) {
    *ptr = b.ptr;
    return TOPK_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return TOPK_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return TOPK_ERR_CAPTURE_ALLOC;
  size_t bytes = need < (1u << 20) ? (1u << 20) : need;
  if (b.ptr && bytes < 2 * b.bytes) bytes = 2 * b.bytes;
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  if (cudaMemsetAsync(p, 0, bytes, st) != cudaSuccess) {
    cudaFree(p);
    return TOPK_ERR_CUDA;
  }
  if (b.ptr) g_retired.emplace_back(dev, b.ptr);
  b.ptr = p;
  b.bytes = bytes;
  *ptr = p;
  return TOPK_OK;
}

int run(const void* scores, const int32_t* row_lens, int64_t M, int64_t N, int32_t K,
        int32_t* out_idx, topk_row_diag* diag, void* ws, size_t ws_bytes, bool explicit_ws,
        cudaStream_t st, int elem_bytes = 4, const int32_t* row_k = nullptr) {
  int rc = check_sizes(M, N, K);
  if (rc) return rc;
  rc = validate_ptrs(scores, row_lens, M, N, out_idx, elem_bytes);
  if (rc) return rc;
  if (M == 0) return TOPK_OK;
  if (row_k && (reinterpret_cast<uintptr_t>(row_k) & 3u)) return TOPK_ERR_ALIGN;
  if (explicit_ws) {
    if (!ws) return TOPK_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return TOPK_ERR_ALIGN;
  }
  DevInfo d;
  int dev = 0;
  rc = device_info(&d, &dev);
  if (rc) return rc;
  const topk_params p = params_snapshot();
  Plan pl;
  rc = make_plan(M, N, K, p, d, &pl, elem_bytes);
  if (rc) return rc;
  if (explicit_ws) {
    if (ws_bytes < pl.ws) return TOPK_ERR_WORKSPACE;
  } else {
    rc = cached_workspace(dev, st, pl.ws, &ws);
    if (rc) return rc;
  }
  tk::Params P = kernel_params(M, N, K, p, pl, elem_bytes);
  P.row_k = row_k;
  return launch(pl, P, scores, row_lens, out_idx, diag, ws, st);
}

}  // namespace

extern "C" {

int topk_ragged(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                int32_t K, int32_t* out_idx, struct CUstream_st* stream) {
  return run(scores, row_lens, M, N_alloc, K, out_idx, nullptr, nullptr, 0, false, stream);
}

int topk_ragged_diag(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* out_idx, topk_row_diag* diag,
                     struct CUstream_st* stream) {
  if (M > 0 && !diag) return TOPK_ERR_ARG;
  return run(scores, row_lens, M, N_alloc, K, out_idx, diag, nullptr, 0, false, stream);
}

int topk_ragged_bf16(const uint16_t* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* out_idx, struct CUstream_st* stream) {
  return run(scores, row_lens, M, N_alloc, K, out_idx, nullptr, nullptr, 0, false, stream, 2);
}

int topk_ragged_bf16_diag(const uint16_t* scores, const int32_t* row_lens, int64_t M,
                          int64_t N_alloc, int32_t K, int32_t* out_idx, topk_row_diag* diag,
                          struct CUstream_st* stream) {
  if (M > 0 && !diag) return TOPK_ERR_ARG;
  return run(scores, row_lens, M, N_alloc, K, out_idx, diag, nullptr, 0, false, stream, 2);
}

int topk_ragged_e4m3(const uint8_t* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* out_idx, struct CUstream_st* stream) {
  return run(scores, row_lens, M, N_alloc, K, out_idx, nullptr, nullptr, 0, false, stream, 1);
}

int topk_ragged_e4m3_diag(const uint8_t* scores, const int32_t* row_lens, int64_t M,
                          int64_t N_alloc, int32_t K, int32_t* out_idx, topk_row_diag* diag,
                          struct CUstream_st* stream) {
  if (M > 0 && !diag) return TOPK_ERR_ARG;
  return run(scores, row_lens, M, N_alloc, K, out_idx, diag, nullptr, 0, false, stream, 1);
}

int topk_ragged_ws(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                   int32_t K, int32_t* out_idx, void* workspace, size_t workspace_bytes,
                   struct CUstream_st* stream) {
  return run(scores, row_lens, M, N_alloc, K, out_idx, nullptr, workspace, workspace_bytes, true,
             stream);
}

int topk_ragged_k(const float* scores, const int32_t* row_lens, const int32_t* row_k, int64_t M,
                  int64_t N_alloc, int32_t K_max, int32_t* out_idx, struct CUstream_st* stream) {
  if (M > 0 && !row_k) return TOPK_ERR_ARG;
  return run(scores, row_lens, M, N_alloc, K_max, out_idx, nullptr, nullptr, 0, false, stream, 4,
             row_k);
}

int topk_ragged_k_bf16(const uint16_t* scores, const int32_t* row_lens, const int32_t* row_k,
                       int64_t M, int64_t N_alloc, int32_t K_max, int32_t* out_idx,
                       struct CUstream_st* stream) {
  if (M > 0 && !row_k) return TOPK_ERR_ARG;
  return run(scores, row_lens, M, N_alloc, K_max, out_idx, nullptr, nullptr, 0, false, stream, 2,
             row_k);
}

int topk_ragged_k_e4m3(const uint8_t* scores, const int32_t* row_lens, const int32_t* row_k,
                       int64_t M, int64_t N_alloc, int32_t K_max, int32_t* out_idx,
                       struct CUstream_st* stream) {
  if (M > 0 && !row_k) return TOPK_ERR_ARG;
  return run(scores, row_lens, M, N_alloc, K_max, out_idx, nullptr, nullptr, 0, false, stream, 1,
             row_k);
}

int topk_ragged_k_diag(const float* scores, const int32_t* row_lens, const int32_t* row_k,
                       int64_t M, int64_t N_alloc, int32_t K_max, int32_t* out_idx,
                       topk_row_diag* diag, struct CUstream_st* stream) {
  if (M > 0 && (!row_k || !diag)) return TOPK_ERR_ARG;
  return run(scores, row_lens, M, N_alloc, K_max, out_idx, diag, nullptr, 0, false, stream, 4,
             row_k);
}

}  // extern "C"

namespace {

// Scratch of topk_ragged_noalloc(): the KV-split merge state of up to
// TOPK_NOALLOC_MAX_ROWS rows.  In host code this name is only a stand-in for
// the device object; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[(size_t)TOPK_NOALLOC_MAX_ROWS *
                                                           tk::kKvRowBytes];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoallocMaxDevices] = {};  // per device, found on its first call

}  // namespace

extern "C" {

int topk_ragged_noalloc(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                        int32_t K, int32_t* out_idx, struct CUstream_st* stream) {
  int rc = check_sizes(M, N_alloc, K);
  if (rc) return rc;
  rc = validate_ptrs(scores, row_lens, M, N_alloc, out_idx);
  if (rc) return rc;
  if (M == 0) return TOPK_OK;
  if (M > TOPK_NOALLOC_MAX_ROWS) return TOPK_ERR_WORKSPACE;
  DevInfo d;
  int dev = 0;
  rc = device_info(&d, &dev);
  if (rc) return rc;
  if (dev < 0 || dev >= kNoallocMaxDevices) return TOPK_ERR_NO_DEVICE;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
      }
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  topk_params p = params_snapshot();
  p.force_kind = TOPK_KIND_KVSPLIT;
  Plan pl;
  rc = make_plan(M, N_alloc, K, p, d, &pl);
  if (rc) return rc;
  if (pl.kind != TOPK_KIND_KVSPLIT ||
      (size_t)M * tk::kv_row_bytes() > sizeof(g_noalloc_scratch))
    return TOPK_ERR_WORKSPACE;
  const cudaError_t e =
      tk::launch_kvsplit(scores, row_lens, out_idx, nullptr, static_cast<uint8_t*>(scratch),
                         kernel_params(M, N_alloc, K, p, pl), stream);
  return e == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

size_t topk_workspace_bytes(int64_t M, int64_t N_alloc, int32_t K) {
  if (check_sizes(M, N_alloc, K) || M == 0) return 0;
  DevInfo d;
  if (device_info(&d, nullptr)) return 0;
  Plan pl;
  if (make_plan(M, N_alloc, K, params_snapshot(), d, &pl)) return 0;
  return pl.ws;
}

int topk_index_topk_fused(const uint16_t* q, const uint16_t* k, const float* w, int64_t T,
                          int64_t S, int32_t H, int32_t D, const int32_t* row_lens, float* scores,
                          int64_t ld_scores, int32_t K, int32_t* out_idx, topk_row_diag* diag,
                          struct CUstream_st* stream) {
  if (!row_lens || K < 1) return TOPK_ERR_ARG;
  if (K > TOPK_K_MAX) return TOPK_ERR_UNSUPPORTED_K;
  int rc = tki::check_index_args(q, k, w, T, S, H, D, row_lens, scores, ld_scores);
  if (rc) return rc;
  if (T == 0) return TOPK_OK;
  if (!out_idx) return TOPK_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(out_idx) & 3u) return TOPK_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S == 0) {  // every row is empty: K sentinels, through the selector
    return topk_ragged(scores, row_lens, T, ld_scores, K, out_idx, stream);
  }
  DevInfo d;
  int dev = 0;
  rc = device_info(&d, &dev);
  if (rc) return rc;
  // one sampling tier for the whole call, the one rows of S keys would take
  topk_params p = params_snapshot();
  const bool lg = p.long_len > 0 && S >= p.long_len;
  p.stride = lg ? p.long_stride : p.stride;
  p.rho0 = lg ? p.long_rho0 : p.rho0;
  p.rho1 = lg ? p.long_rho1 : p.rho1;
  p.long_len = 0;
  const int64_t s = p.stride;
  const int64_t ns_max = (S + s - 1) / s;
  const int64_t S_s = (ns_max + 127) / 128 * 128;  // the score kernel tiles 128 keys
  // workspace: row states, sample keys, sample lengths, sample scores
  const size_t rows_b = (size_t)T * tk::kFusedRowBytes;
  const size_t ks_b = align256((size_t)S_s * 128 * 2);
  const size_t ls_b = align256((size_t)T * 4);
  const size_t ss_b = align256((size_t)T * S_s * 4);
  const size_t need = kHdrBytes + rows_b + ks_b + ls_b + ss_b;
  void* ws = nullptr;
  rc = cached_workspace(dev, st, need, &ws);
  if (rc) return rc;
  uint8_t* rows = static_cast<uint8_t*>(ws) + kHdrBytes;
  uint16_t* ks = reinterpret_cast<uint16_t*>(rows + rows_b);
  int32_t* lens_s = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ks) + ks_b);
  float* ss = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(lens_s) + ls_b);
  Plan pl;
  pl.kind = TOPK_KIND_KVSPLIT;
  pl.segments = 1;
  tk::Params P = kernel_params(T, S, K, p, pl);
  if (tki::launch_gather_sample_keys(k, S, (int32_t)s, S_s, ks, row_lens, T, lens_s, st) !=
      cudaSuccess)
    return TOPK_ERR_CUDA;
  rc = tki::launch_index_scores(q, ks, w, T, S_s, lens_s, ss, S_s, nullptr, st);
  if (rc) return rc;
  if (tk::launch_fused_prepare(ss, S_s, row_lens, rows, P, st) != cudaSuccess) return TOPK_ERR_CUDA;
  rc = tki::launch_index_scores(q, k, w, T, S, row_lens, scores, ld_scores, rows, st);
  if (rc) return rc;
  return tk::launch_fused_finish(scores, ld_scores, out_idx,
                                 reinterpret_cast<tk::RowDiag*>(diag), rows, P, st) == cudaSuccess
             ? TOPK_OK
             : TOPK_ERR_CUDA;
}

int topk_cached_workspace(struct CUstream_st* stream, void** ptr, size_t* bytes) {
  if (!ptr || !bytes) return TOPK_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  const auto it = g_ws.find({dev, reinterpret_cast<uintptr_t>(stream)});
  *ptr = it == g_ws.end() ? nullptr : it->second.ptr;
  *bytes = it == g_ws.end() ? 0 : it->second.bytes;
  return TOPK_OK;
}

int topk_plan(int64_t M, int64_t N_alloc, int32_t K, topk_plan_info* info) {
  if (!info) return TOPK_ERR_ARG;
  int rc = check_sizes(M, N_alloc, K);
  if (rc) return rc;
  DevInfo d;
  rc = device_info(&d, nullptr);
  if (rc) return rc;
  Plan pl;
  rc = make_plan(M, N_alloc, K, params_snapshot(), d, &pl);
  if (rc) return rc;
  info->kind = pl.kind;
  info->grid = pl.grid;
  info->segments = pl.segments;
  info->sm_count = d.sm_count;
  info->workspace_bytes = pl.ws;
  info->smem_bytes = pl.smem;
  return TOPK_OK;
}

void topk_default_params(topk_params* p) {
  if (p) defaults(p);
}

int topk_set_params(const topk_params* p) {
  if (!p) return TOPK_ERR_ARG;
  if (p->stride < 1 || !(p->rho0 >= 1.0f) || !(p->rho1 >= p->rho0) || !(p->rho1 <= 64.0f) ||
      p->long_stride < 1 || !(p->long_rho0 >= 1.0f) || !(p->long_rho1 >= p->long_rho0) ||
      !(p->long_rho1 <= 64.0f) || p->long_len < 0 ||
      p->sample_min_len < 0 || p->direct_max < 0 || p->kv_segments < 0 ||
      p->kv_segments > 4096 || p->force_kind < TOPK_KIND_AUTO || p->force_kind > TOPK_KIND_KVSPLIT)
    return TOPK_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_params = *p;
  g_params_init = true;
  return TOPK_OK;
}

int topk_get_params(topk_params* p) {
  if (!p) return TOPK_ERR_ARG;
  *p = params_snapshot();
  return TOPK_OK;
}

int topk_read_status(struct CUstream_st* stream, uint32_t* flags) {
  if (!flags) return TOPK_ERR_ARG;
  DevInfo d;
  int rc = device_info(&d, nullptr);
  if (rc) return rc;
  return tk::read_and_clear_status(stream, flags) == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

int topk_ragged_host(const float* h_scores, const int32_t* h_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* h_out, int64_t rows_per_chunk) {
  int rc = check_sizes(M, N_alloc, K);
  if (rc) return rc;
  if (M == 0) return TOPK_OK;
  if (!h_lens || !h_out || (N_alloc > 0 && !h_scores) || rows_per_chunk < 0) return TOPK_ERR_ARG;
  DevInfo d;
  int dev = 0;
  rc = device_info(&d, &dev);
  if (rc) return rc;
  const size_t row_bytes = (size_t)N_alloc * sizeof(float);
  int64_t rows = rows_per_chunk;
  if (rows == 0) rows = row_bytes ? (int64_t)((1ull << 30) / row_bytes) : M;
  if (rows < 1) rows = 1;
  if (rows > M) rows = M;
  HostPipe* hp;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    hp = &g_pipe[dev];  // map nodes stay put; only topk_release_workspaces removes them
  }
  // Calls from several host threads on one device take turns on its buffers
  // and streams.
  std::lock_guard<std::mutex> pipe_lock(hp->mu);
  const size_t need_s = (size_t)rows * row_bytes, need_l = (size_t)M * 4,
               need_o = (size_t)rows * K * 4;
  for (int i = 0; i < 2; ++i) {
    if (!hp->st[i] && cudaStreamCreateWithFlags(&hp->st[i], cudaStreamNonBlocking) != cudaSuccess)
      return TOPK_ERR_CUDA;
  }
  if (hp->score_bytes < need_s || hp->lens_bytes < need_l || hp->out_bytes < need_o) {
    for (int i = 0; i < 2; ++i) {
      cudaStreamSynchronize(hp->st[i]);
      cudaFree(hp->scores[i]);
      cudaFree(hp->lens[i]);
      cudaFree(hp->out[i]);
      hp->scores[i] = nullptr;
      hp->lens[i] = nullptr;
      hp->out[i] = nullptr;
    }
    hp->score_bytes = hp->lens_bytes = hp->out_bytes = 0;
    for (int i = 0; i < 2; ++i) {
      if (cudaMalloc(&hp->scores[i], need_s ? need_s : 16) != cudaSuccess ||
          cudaMalloc(&hp->lens[i], need_l) != cudaSuccess ||
          cudaMalloc(&hp->out[i], need_o) != cudaSuccess) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
      }
    }
    hp->score_bytes = need_s;
    hp->lens_bytes = need_l;
    hp->out_bytes = need_o;
  }
  // Every row length in one copy (a few KB; the caller's array may be
  // pageable, which would make a copy per chunk hold the host thread).
  if (cudaMemcpy(hp->lens[0], h_lens, (size_t)M * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return TOPK_ERR_CUDA;
  // Chunk c's result is read back only after chunk c + 1's copy and
  // selection are queued: a read into pageable memory holds the host thread
  // until it is done, and the copy engine then still has chunk c + 1's rows
  // to move.  Each buffer pair is reused two chunks later on the same stream,
  // after its result was read.
  int64_t prev_r0 = -1, prev_n = 0;
  int prev_s = 0;
  for (int64_t r0 = 0, c = 0; r0 < M; r0 += rows, ++c) {
    const int64_t n = (M - r0) < rows ? (M - r0) : rows;
    const int s = (int)(c & 1);
    cudaStream_t st = hp->st[s];
    if (row_bytes &&
        cudaMemcpyAsync(hp->scores[s], h_scores + r0 * N_alloc, (size_t)n * row_bytes,
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
      return TOPK_ERR_CUDA;
    rc = topk_ragged(hp->scores[s], hp->lens[0] + r0, n, N_alloc, K, hp->out[s], st);
    if (rc) return rc;
    if (prev_r0 >= 0 &&
        cudaMemcpyAsync(h_out + prev_r0 * K, hp->out[prev_s], (size_t)prev_n * K * 4,
                        cudaMemcpyDeviceToHost, hp->st[prev_s]) != cudaSuccess)
      return TOPK_ERR_CUDA;
    prev_r0 = r0;
    prev_n = n;
    prev_s = s;
  }
  if (prev_r0 >= 0 &&
      cudaMemcpyAsync(h_out + prev_r0 * K, hp->out[prev_s], (size_t)prev_n * K * 4,
                      cudaMemcpyDeviceToHost, hp->st[prev_s]) != cudaSuccess)
    return TOPK_ERR_CUDA;
  for (int i = 0; i < 2; ++i)
    if (cudaStreamSynchronize(hp->st[i]) != cudaSuccess) return TOPK_ERR_CUDA;
  return TOPK_OK;
}

int topk_check_wait_timeout(uint64_t limit_ns, struct CUstream_st* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return TOPK_ERR_ARG;
  DevInfo d;
  int rc = device_info(&d, nullptr);
  if (rc) return rc;
  return tk::launch_wait_probe(limit_ns, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TOPK_OK
             : TOPK_ERR_CUDA;
}

void topk_release_workspaces(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_ws) {
    if (!kv.second.ptr) continue;
    cudaSetDevice(kv.first.first);
    cudaDeviceSynchronize();
    cudaFree(kv.second.ptr);
  }
  g_ws.clear();
  for (auto& r : g_retired) {
    cudaSetDevice(r.first);
    cudaDeviceSynchronize();
    cudaFree(r.second);
  }
  g_retired.clear();
  for (auto& kv : g_pipe) {
    cudaSetDevice(kv.first);
    cudaDeviceSynchronize();
    for (int i = 0; i < 2; ++i) {
      cudaFree(kv.second.scores[i]);
      cudaFree(kv.second.lens[i]);
      cudaFree(kv.second.out[i]);
      if (kv.second.st[i]) cudaStreamDestroy(kv.second.st[i]);
    }
  }
  g_pipe.clear();
  cudaSetDevice(cur);
}

const char* topk_status_string(int code) {
  switch (code) {
    case TOPK_OK: return "ok";
    case TOPK_ERR_ARG: return "invalid argument";
    case TOPK_ERR_ALIGN: return "misaligned pointer";
    case TOPK_ERR_WORKSPACE: return "workspace too small";
    case TOPK_ERR_CUDA: return "CUDA runtime error";
    case TOPK_ERR_CAPTURE_ALLOC: return "workspace allocation needed during stream capture";
    case TOPK_ERR_UNSUPPORTED_K: return "K larger than TOPK_K_MAX";
    case TOPK_ERR_NO_DEVICE: return "no usable sm_103 device";
    case TOPK_ERR_UNSUPPORTED_SHAPE: return "indexer-score shape not supported";
    default: return "unknown status";
  }
}

int topk_version(void) { return kVersion; }

#ifdef TOPK_PHASE_TIMING
// Tuning hook of a build with -DTOPK_PHASE_TIMING: sets the L2 prefetch
// distances of the full-row pass (chunks ahead of the ring, bytes of the next
// row).  Not thread-safe with calls in flight.
int topk_debug_set_prefetch(uint32_t ahead_chunks, uint32_t next_bytes) {
  g_knob_pf_ahead = ahead_chunks;
  g_knob_pf_next_bytes = next_bytes & ~15u;
  return TOPK_OK;
}
// Forces the persistent kernel's sampler warp on (1) or off (0), or leaves
// the choice to the width rule (-1).
int topk_debug_set_sampler(int mode) {
  g_knob_sampler = mode < 0 ? -1 : (mode ? 1 : 0);
  return TOPK_OK;
}
#endif

}  // extern "C"
