/*
 * topk.h -- sample-guided exact Top-K over ragged FP32 score rows (GB300, sm_103a).
 *
 * The operation: for every row r of a row-major FP32 matrix scores[M][N_alloc]
 * with valid prefix length len_r = clamp(row_lens[r], 0, N_alloc), return the
 * indices of the K largest scores of that prefix.  The result follows the set
 * contract of "Sample-Guided Exact Top-K Selection for Long-Context Sparse
 * Attention" as summarised in the codexqa.cn article "几何平均快 1.55 倍，但短行
 * 采样会输：腾讯怎么测精确 Top-K", section "什么叫精确，时间怎么量":
 *   - indices are distinct and lie inside [0, len_r);
 *   - len_r > K: exactly K indices, min(selected scores) >= max(scores left
 *     out); equal scores at the boundary may go either way; order is free;
 *     no floating-point tolerance;
 *   - len_r <= K: every valid index 0..len_r-1, followed by K - len_r
 *     sentinels of value -1.
 * The method (PaperDaily "腾讯|长上下文稀疏注意力前K精确选择", section 问题二,
 * Fig. 4; arxivdaily abstract of the same paper): a fixed-stride sample of the
 * current row proposes a coarse threshold tau0 and a nested, wider tau1; one
 * mandatory full-row pass certifies C(tau0) >= K, collects the admitted
 * candidates and seeds an FP32 radix histogram; exact radix refinement runs
 * only over the unresolved boundary bin; the nested threshold and an exact
 * whole-row recovery serve rows the proposal underfills.  Short rows use an
 * exact boundary directly, long rows with few rows per call are split across
 * CTAs (KV-split), and many rows run on persistent CTAs.
 *
 * Scores are compared by their IEEE order with -0.0 equal to +0.0.  NaN is not
 * a supported score value (the library stays in bounds but the result is not
 * specified).
 *
 * Conventions for every entry point below:
 *   - "device" pointers are CUDA device (or managed) memory owned by the
 *     caller; the library never frees or keeps them past the call's work;
 *   - scores must be 4-byte aligned; rows start at scores + r * N_alloc and
 *     need not be 16-byte aligned (unaligned heads/tails are read singly);
 *   - a call never reads a score at or beyond len_r in its row;
 *   - work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and the call returns without waiting for it, so device
 *     memory errors surface at the caller's next synchronisation;
 *   - the calls do no host synchronisation and read no device memory from the
 *     host, so they can be captured in a CUDA graph once the library's
 *     workspace for that stream exists (a call that would have to allocate
 *     during capture returns TOPK_ERR_CAPTURE_ALLOC);
 *   - the library's workspace for a (device, stream) only grows; when a
 *     larger call replaces it, the old buffer is kept allocated (a graph
 *     captured earlier may still use it) until topk_release_workspaces(), so
 *     a captured graph stays valid until then, whatever eager calls run on
 *     its stream in between;
 *   - a bounded wait inside a kernel that gives up flags its rows
 *     (TOPK_FLAG_TIMEOUT) and makes the other waits of the same launch give
 *     up at once; that state belongs to the launch and never reaches a
 *     later call, whether or not the status word is read;
 *   - on an error code nothing has been enqueued.
 */
#ifndef EXACT_TOPK_GB300_TOPK_H
#define EXACT_TOPK_GB300_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

typedef enum topk_status {
  TOPK_OK = 0,
  TOPK_ERR_ARG = -1,            /* null pointer, negative size, K < 1, size overflow */
  TOPK_ERR_ALIGN = -2,          /* scores or out_idx not 4-byte aligned, workspace not 256-byte aligned */
  TOPK_ERR_WORKSPACE = -3,      /* explicit workspace smaller than topk_workspace_bytes() */
  TOPK_ERR_CUDA = -4,           /* a CUDA runtime call failed (allocation, launch, copy) */
  TOPK_ERR_CAPTURE_ALLOC = -5,  /* the call would allocate while `stream` is capturing */
  TOPK_ERR_UNSUPPORTED_K = -6,  /* K > TOPK_K_MAX */
  TOPK_ERR_NO_DEVICE = -7,      /* no usable sm_103 device is current */
  TOPK_ERR_UNSUPPORTED_SHAPE = -8 /* indexer-score shape outside what the kernel tiles (see below) */
} topk_status;

/* Largest supported K.  The sampled path is tuned for K = 2048. */
#define TOPK_K_MAX 4096

/* Per-row path identifiers reported by topk_ragged_diag(). */
#define TOPK_PATH_SENTINEL 0 /* len <= K: 0..len-1 then -1 */
#define TOPK_PATH_DIRECT 1   /* exact boundary without sampling (short rows) */
#define TOPK_PATH_TAU0 2     /* C(tau0) >= K: refinement over the certified candidates */
#define TOPK_PATH_TAU1 3     /* C(tau0) < K <= C(tau1): the nested threshold serves the row */
#define TOPK_PATH_RECOVERY 4 /* C(tau1) < K: exact whole-row recovery */

/* Bits of topk_row_diag.flags and of the device status word. */
#define TOPK_FLAG_LEN_CLAMPED 0x1u /* row_lens[r] was outside [0, N_alloc] and was clamped */
#define TOPK_FLAG_OVERFLOW 0x2u    /* admitted candidates exceeded the on-chip buffer; served by re-reading the row */
#define TOPK_FLAG_RECOVERY 0x4u    /* exact whole-row recovery ran */
#define TOPK_FLAG_INTERNAL 0x8u    /* an internal invariant failed (a library bug; the row is not valid) */
#define TOPK_FLAG_TIMEOUT 0x10u    /* a bounded wait on an asynchronous copy gave up (the row is not valid) */
#define TOPK_FLAG_K_CLAMPED 0x20u  /* row_k[r] was outside [0, K_max] and was clamped (per-row K calls) */

/* Execution paths of the host planner (topk_plan_info.kind, topk_params.force_kind). */
#define TOPK_KIND_AUTO 0
#define TOPK_KIND_DIRECT 1     /* one CTA per row, the row staged on chip */
#define TOPK_KIND_PERSISTENT 2 /* persistent CTAs pull whole rows from a queue */
#define TOPK_KIND_KVSPLIT 3    /* several CTAs per row scan disjoint segments; the last one to finish selects */

/* Per-row diagnostics written by topk_ragged_diag() (device array of M). */
typedef struct topk_row_diag {
  float tau0;      /* primary sampled threshold (NaN when the row was not sampled) */
  float tau1;      /* nested secondary threshold (NaN when the row was not sampled) */
  int64_t count0;  /* C(tau0): scores of the valid prefix >= tau0 (0 when not sampled) */
  int64_t count1;  /* C(tau1) (0 when not sampled) */
  int32_t path;    /* TOPK_PATH_* */
  uint32_t flags;  /* TOPK_FLAG_* for this row */
} topk_row_diag;

/* Process-wide tuning knobs.  A sampled row is viewed at a fixed stride s
 * (positions 0, s, 2s, ... below len, n_s = ceil(len / s) samples); its
 * thresholds are the samples of rank r = ceil(T * n_s / len), clamped to
 * [1, n_s], with targets T = ceil(rho * K) (codexqa.cn section
 * "采样不是处处都该开", which uses s = 128, T = 1.5K and 1.75K on H20).
 * Every sampled element costs one DRAM access on GB300, so the defaults
 * take a wider stride with proportionally larger targets (the same sample
 * ranks), and rows of at least long_len elements a wider one still:
 *   len <  long_len: s = stride,      T = rho0 * K,      rho1 * K
 *   len >= long_len: s = long_stride, T = long_rho0 * K, long_rho1 * K */
typedef struct topk_params {
  int32_t stride;          /* sample stride s >= 1 (default 256) */
  float rho0;              /* primary target as a multiple of K (default 2.0) */
  float rho1;              /* secondary target, >= rho0 (default 2.25) */
  int64_t sample_min_len;  /* rows shorter than this skip sampling (exact boundary; default 12288) */
  int64_t direct_max;      /* N_alloc at or below which the on-chip direct kernel serves every row
                              (default 16384) */
  int32_t force_kind;      /* TOPK_KIND_*; AUTO lets the planner choose */
  int32_t kv_segments;     /* KV-split segments per row; 0 = planner's choice */
  int64_t long_len;        /* rows this long or longer use the long_* knobs; 0 = never (default 786432) */
  int32_t long_stride;     /* default 512 */
  float long_rho0;         /* default 2.75 */
  float long_rho1;         /* >= long_rho0, default 3.0 */
} topk_params;

typedef struct topk_plan_info {
  int32_t kind;            /* TOPK_KIND_* chosen for (M, N_alloc, K) on the current device */
  int32_t grid;            /* CTAs of the main kernel */
  int32_t segments;        /* KV-split segments per row (1 otherwise) */
  int32_t sm_count;        /* SMs on the current device */
  size_t workspace_bytes;  /* device workspace the call needs */
  size_t smem_bytes;       /* dynamic shared memory per CTA of the main kernel */
} topk_plan_info;

/* Exact Top-K of every row (the spec call).
 *   scores   device, [M][N_alloc] FP32, row-major, row stride N_alloc
 *   row_lens device, [M] int32; values outside [0, N_alloc] are clamped and
 *            flagged in the device status word (TOPK_FLAG_LEN_CLAMPED)
 *   M >= 0, 0 <= N_alloc <= INT32_MAX, 1 <= K <= TOPK_K_MAX
 *   out_idx  device, [M][K] int32, written completely
 * Uses a workspace the library allocates on first use per (device, stream)
 * and keeps until topk_release_workspaces().  M == 0 is a no-op.
 * Returns TOPK_OK or a topk_status error. */
int topk_ragged(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                int32_t K, int32_t* out_idx, struct CUstream_st* stream);

/* Same as topk_ragged, and also writes diag[M] (device) with each row's
 * thresholds, counts, path and flags. */
int topk_ragged_diag(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* out_idx, topk_row_diag* diag,
                     struct CUstream_st* stream);

/* Same as topk_ragged / topk_ragged_diag for bfloat16 score rows: `scores`
 * holds raw bfloat16 bit patterns [M][N_alloc] (2-byte aligned).  A bfloat16
 * widens exactly to FP32, and the selection is the exact Top-K of the
 * widened values (same contract, same thresholds and paths), reading half the
 * bytes.  This is an extension beyond the pages, which measure FP32 rows only
 * (PaperDaily, section 问题四, lists lower-precision scores as untested). */
int topk_ragged_bf16(const uint16_t* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* out_idx, struct CUstream_st* stream);
int topk_ragged_bf16_diag(const uint16_t* scores, const int32_t* row_lens, int64_t M,
                          int64_t N_alloc, int32_t K, int32_t* out_idx, topk_row_diag* diag,
                          struct CUstream_st* stream);

/* Same for FP8 E4M3 score rows (the OCP 8-bit format without infinities:
 * sign, 4 exponent bits with bias 7, 3 mantissa bits), given as raw bytes
 * [M][N_alloc] with no alignment requirement.  Every E4M3 value widens
 * exactly to FP32 and the selection is the exact Top-K of the widened values,
 * reading a quarter of the FP32 bytes.  With 8 values per octave, rows hold
 * long runs of equal scores; ties at the boundary are broken freely as the
 * contract allows.  The NaN pattern S.1111.111 is not a supported score.  An
 * extension beyond the pages, as the bfloat16 form. */
int topk_ragged_e4m3(const uint8_t* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* out_idx, struct CUstream_st* stream);
int topk_ragged_e4m3_diag(const uint8_t* scores, const int32_t* row_lens, int64_t M,
                          int64_t N_alloc, int32_t K, int32_t* out_idx, topk_row_diag* diag,
                          struct CUstream_st* stream);

/* Device workspace bytes a call with these sizes needs under the current
 * parameters (0 is a valid answer only for M == 0).  The workspace is
 * O(M) (KV-split merge state per row) or O(CTAs) (persistent spill areas),
 * never O(M * N_alloc): the codexqa.cn article, section "20 个形状都最快",
 * contrasts the method with a spill strategy that reserves 2 * M * N 32-bit
 * entries and runs out of memory at long widths.  The size depends on the
 * plan (topk_plan) and the parameters (topk_set_params). */
size_t topk_workspace_bytes(int64_t M, int64_t N_alloc, int32_t K);

/* Explicit-workspace form of topk_ragged() (same contract and errors), for
 * callers that manage device memory themselves; the workspace is the only
 * memory the call uses beyond its inputs and outputs, and it is bounded as
 * topk_workspace_bytes() states (codexqa.cn, section "20 个形状都最快").
 *   workspace        device memory of at least topk_workspace_bytes(M,
 *                    N_alloc, K) bytes, 256-byte aligned (else
 *                    TOPK_ERR_ALIGN), zero-filled before its first use; every
 *                    call leaves it ready for the next; owned by the caller
 *   workspace_bytes  its size; smaller than needed -> TOPK_ERR_WORKSPACE
 * Calls that share one workspace must be ordered (same stream, or
 * synchronised).  Never allocates, so it can be captured in a CUDA graph
 * whenever the workspace outlives the graph. */
int topk_ragged_ws(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                   int32_t K, int32_t* out_idx, void* workspace, size_t workspace_bytes,
                   struct CUstream_st* stream);

/* Per-row K.  Row r takes its own k_r = clamp(row_k[r], 0, K_max) (a value
 * outside that range sets TOPK_FLAG_K_CLAMPED) and gets the result of
 * topk_ragged() with K = k_r in slots [0, k_r) of an output row of K_max
 * slots; slots [k_r, K_max) hold -1.  So k_r = 0 gives a row of -1, and
 * len_r <= k_r gives 0..len_r-1 followed by -1.  A sampled row's targets are
 * ceil(rho * k_r) with the rho of its sampling tier (topk_params).  The
 * pages use one K for every row (PaperDaily, section 问题四: K = 2048
 * throughout); per-row K is an extension for callers whose rows need
 * different budgets.
 *   row_k    device, [M] int32
 *   K_max    1 <= K_max <= TOPK_K_MAX: the output row stride
 *   out_idx  device, [M][K_max] int32, written completely
 * Other arguments, workspace and errors as topk_ragged() (and
 * topk_ragged_bf16(), topk_ragged_e4m3() and topk_ragged_diag() for the _bf16,
 * _e4m3 and _diag forms). */
int topk_ragged_k(const float* scores, const int32_t* row_lens, const int32_t* row_k, int64_t M,
                  int64_t N_alloc, int32_t K_max, int32_t* out_idx, struct CUstream_st* stream);
int topk_ragged_k_bf16(const uint16_t* scores, const int32_t* row_lens, const int32_t* row_k,
                       int64_t M, int64_t N_alloc, int32_t K_max, int32_t* out_idx,
                       struct CUstream_st* stream);
int topk_ragged_k_e4m3(const uint8_t* scores, const int32_t* row_lens, const int32_t* row_k,
                       int64_t M, int64_t N_alloc, int32_t K_max, int32_t* out_idx,
                       struct CUstream_st* stream);
int topk_ragged_k_diag(const float* scores, const int32_t* row_lens, const int32_t* row_k,
                       int64_t M, int64_t N_alloc, int32_t K_max, int32_t* out_idx,
                       topk_row_diag* diag, struct CUstream_st* stream);

/* Rows topk_ragged_noalloc() accepts in one call. */
#define TOPK_NOALLOC_MAX_ROWS 64

/* Fixed-scratch form, for callers that may not allocate device memory.  The
 * paper has no counterpart; this exists because some callers cannot call
 * cudaMalloc: serving processes whose allocator owns every byte of the GPU,
 * plugin hosts that forbid allocation while they execute, and code that must
 * not risk the device-wide synchronisation or out-of-memory failure an
 * allocation can bring.  It runs the KV-split path with its per-row merge
 * state in one statically sized device array (TOPK_NOALLOC_MAX_ROWS rows,
 * about 9.5 MiB) that every GPU loading this library holds until the process
 * exits.  Arguments and results are those of topk_ragged(); M above
 * TOPK_NOALLOC_MAX_ROWS returns TOPK_ERR_WORKSPACE.  The first call on a
 * device looks up the array's device address (make that first call before
 * any stream capture).  Every call shares the one array and the kernels
 * re-initialise it, so calls that overlap on the GPU (different streams, or
 * other host threads) race and must be serialised by the caller.  It never
 * calls cudaMalloc or cudaFree. */
int topk_ragged_noalloc(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                        int32_t K, int32_t* out_idx, struct CUstream_st* stream);

/* Host-buffer form: copies the rows in chunks to the device, selects and
 * copies the indices back, overlapping copies with selection on two streams.
 *   h_scores  host [M][N_alloc] FP32 (page-locked memory gives full copy speed)
 *   h_lens    host [M] int32
 *   h_out     host [M][K] int32
 *   rows_per_chunk  rows per device chunk; 0 picks about 1 GiB of scores per chunk
 * Synchronous: returns after h_out is written.  Device buffers and the two
 * streams are cached per device until topk_release_workspaces(); calls from
 * several host threads on one device take turns on them (a lock held for the
 * whole call). */
int topk_ragged_host(const float* h_scores, const int32_t* h_lens, int64_t M, int64_t N_alloc,
                     int32_t K, int32_t* h_out, int64_t rows_per_chunk);

/* The library's cached workspace for (current device, `stream`): its device
 * address and size in *ptr and *bytes (NULL and 0 when none exists yet).
 * Read-only; for callers that check what a captured graph refers to. */
int topk_cached_workspace(struct CUstream_st* stream, void** ptr, size_t* bytes);

/* Read-only planning: what a call with these sizes would launch. */
int topk_plan(int64_t M, int64_t N_alloc, int32_t K, topk_plan_info* info);

/* Set / get the process-wide parameters (host memory structs).  Invalid
 * values (stride < 1, rho0 < 1, rho1 < rho0, negative lengths, unknown kind)
 * return TOPK_ERR_ARG and change nothing.  Not thread-safe with calls in
 * flight on other host threads. */
int topk_set_params(const topk_params* p);
int topk_get_params(topk_params* p);
void topk_default_params(topk_params* p);

/* Read and clear the current device's status word: the OR of TOPK_FLAG_* over
 * every row selected since the last read (host memory *flags).  The set
 * contract treats failures as their own outcome, never as a slower correct
 * run (codexqa.cn, sections "什么叫精确，时间怎么量" and "这组数字不能外推的
 * 地方": illegal results, illegal accesses and out-of-memory are reported
 * apart); this word is where a call reports rows it could not serve
 * exactly (TOPK_FLAG_INTERNAL, TOPK_FLAG_TIMEOUT) apart from informational
 * bits (clamped lengths or K, overflow and recovery paths taken).  Enqueues a
 * copy on `stream` and synchronises it; TOPK_ERR_ARG for a null `flags`,
 * TOPK_ERR_CUDA if the copy or the synchronisation fails. */
int topk_read_status(struct CUstream_st* stream, uint32_t* flags);

/* Free every cached workspace (including those a stream has grown out of)
 * and host-path buffer of this process (synchronises the devices that own
 * them).  Graphs captured over the library's workspaces must not be replayed
 * afterwards, and no call may be in flight on another host thread. */
void topk_release_workspaces(void);

/* Human-readable name of a topk_status code (static string). */
const char* topk_status_string(int code);

/* Self-test of failure detection: one thread on `stream` waits, with the
 * kernels' own bounded-wait routine, on a barrier that nothing completes;
 * after limit_ns (1 ns .. 10 s) it gives up and sets TOPK_FLAG_TIMEOUT in the
 * status word, which topk_read_status() returns (and clears).  Its fail-fast
 * flag is its own, so later calls run normally whether or not the status is
 * read.  No memory operation is pending meanwhile and the context stays
 * usable.  TOPK_ERR_ARG for a limit outside that range. */
int topk_check_wait_timeout(uint64_t limit_ns, struct CUstream_st* stream);

/* Library version as major * 10000 + minor * 100 + patch. */
int topk_version(void);

/* Optional order for a Top-K result (the contract leaves it free): sorts each
 * of the M rows of out_idx [M][K] (device, as written by topk_ragged) in
 * place by score, largest first, equal scores by index, -1 sentinels last.
 * `scores` are the rows the indices refer to (device, row stride N_alloc);
 * topk_sort_rows_bf16 takes bfloat16 patterns, topk_sort_rows_e4m3 FP8 E4M3
 * bytes.  One launch on `stream`, no
 * allocation.  Errors as topk_ragged. */
int topk_sort_rows(const float* scores, int64_t M, int64_t N_alloc, int32_t K, int32_t* out_idx,
                   struct CUstream_st* stream);
int topk_sort_rows_bf16(const uint16_t* scores, int64_t M, int64_t N_alloc, int32_t K,
                        int32_t* out_idx, struct CUstream_st* stream);
int topk_sort_rows_e4m3(const uint8_t* scores, int64_t M, int64_t N_alloc, int32_t K,
                        int32_t* out_idx, struct CUstream_st* stream);

/* ---------------------------------------------------------------------------
 * Indexer scores: the stage that produces the selector's rows (eq. (1) of the
 * xllm-io review of LiteTopK, section "核心公式"):
 *   scores[t][s] = sum over heads j of w[t][j] * ReLU( q[t][j] . k[s] )
 * computed with tcgen05 tensor-core MMAs (bf16 inputs, FP32 accumulation,
 * FP32 ReLU/weight/head-sum epilogue).
 *   q        device, bfloat16 bit patterns [T][H][D], 16-byte aligned
 *   k        device, bfloat16 bit patterns [S][D], 16-byte aligned
 *   w        device, float [T][H], 16-byte aligned
 *   row_lens device int32 [T] or NULL: scores[t][s] for s >= row_lens[t]
 *            (causal suffix) are written as -inf; values must lie in [0, S]
 *   scores   device, float [T][ld_scores], ld_scores >= S; columns S.. are
 *            not written
 * Supported shapes: H == 64, D == 128, T a multiple of 4, S a multiple of
 * 128 (else TOPK_ERR_UNSUPPORTED_SHAPE); the pointers' alignment is checked
 * (TOPK_ERR_ALIGN).  Asynchronous on `stream`, no allocation, graph-
 * capturable.  A bounded internal wait that gives up sets TOPK_FLAG_TIMEOUT
 * in the status word topk_index_read_status() returns. */
int topk_index_scores(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                      int32_t H, int32_t D, const int32_t* row_lens, float* scores,
                      int64_t ld_scores, struct CUstream_st* stream);

/* Scores and exact Top-K in one call: topk_index_scores() into `scores`,
 * then topk_ragged(scores, row_lens, T, ld_scores, K, out_idx, stream) on the
 * same stream (two launches; capturable into one CUDA graph after a first
 * uncaptured call has created the selector's workspace).  row_lens is
 * required. */
int topk_index_topk(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                    int32_t H, int32_t D, const int32_t* row_lens, float* scores,
                    int64_t ld_scores, int32_t K, int32_t* out_idx, struct CUstream_st* stream);

/* Scores and exact Top-K with the selection's proposal and certification
 * moved into the score stage (the fused score -> filter step of the xllm-io
 * review of LiteTopK, sections "核心思想" and "详细方法": scores are gated
 * against a threshold while they are produced, and survivors go to a
 * candidate buffer).  The threshold is this method's own (PaperDaily section
 * 问题二): the score kernel first scores a fixed-stride sample of the keys
 * (k[0], k[s], k[2s], ...; s and the targets those of the sampling tier that
 * rows of S keys take under topk_params), each row's tau0 and tau1 are its
 * samples of rank ceil(T * n_s / len); then the full score pass writes
 * `scores` as topk_index_scores() does and also appends every score >= tau1
 * of a row to that row's candidate area, counting C(tau1).  The selection
 * certifies C(tau0) >= K from the candidates and refines them exactly; a row
 * whose candidates do not certify it (C(tau1) < K, or more than 16384
 * candidates) is served from its materialised row in `scores` by the same
 * recovery and re-read paths as topk_ragged(), so the result is always the
 * exact Top-K of the scores written (same set contract).
 * Arguments as topk_index_topk(); diag (device, [T] topk_row_diag) may be
 * NULL.  Uses the library's workspace for the stream: about
 * T * 140 KB + T * ceil(S / s) * 4 B (+ the sample keys); TOPK_ERR_CAPTURE_ALLOC
 * if that must grow during stream capture.  Five launches on `stream`,
 * capturable into one CUDA graph after a first uncaptured call. */
int topk_index_topk_fused(const uint16_t* q, const uint16_t* k, const float* w, int64_t T,
                          int64_t S, int32_t H, int32_t D, const int32_t* row_lens, float* scores,
                          int64_t ld_scores, int32_t K, int32_t* out_idx, topk_row_diag* diag,
                          struct CUstream_st* stream);

/* Read and clear the score kernel's status word (TOPK_FLAG_TIMEOUT); syncs
 * the stream. */
int topk_index_read_status(struct CUstream_st* stream, uint32_t* flags);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_TOPK_GB300_TOPK_H */
