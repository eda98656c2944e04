"""Sample-guided exact Top-K over ragged FP32 score rows (CUDA, sm_103a).

A thin ctypes binding of the C ABI in include/topk.h.  It only marshals
arguments: every step of the selection runs in the CUDA kernels of
``lib/libtopk.so``.  PyTorch provides device memory and the current stream.
There is no CPU fallback: if the library has not been built, every call
raises.

    import torch, exact_top_sparse_gb300 as ets
    idx = ets.topk_ragged(scores, row_lens, K=2048)   # [M, K] int32, -1 padded
"""
import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libtopk.so")

TOPK_OK = 0
STATUS_NAMES = {
    0: "TOPK_OK", -1: "TOPK_ERR_ARG", -2: "TOPK_ERR_ALIGN", -3: "TOPK_ERR_WORKSPACE",
    -4: "TOPK_ERR_CUDA", -5: "TOPK_ERR_CAPTURE_ALLOC", -6: "TOPK_ERR_UNSUPPORTED_K",
    -7: "TOPK_ERR_NO_DEVICE", -8: "TOPK_ERR_UNSUPPORTED_SHAPE",
}
K_MAX = 4096

PATH_SENTINEL, PATH_DIRECT, PATH_TAU0, PATH_TAU1, PATH_RECOVERY = 0, 1, 2, 3, 4
FLAG_LEN_CLAMPED, FLAG_OVERFLOW, FLAG_RECOVERY, FLAG_INTERNAL, FLAG_TIMEOUT = 1, 2, 4, 8, 16
FLAG_K_CLAMPED = 32
KIND_AUTO, KIND_DIRECT, KIND_PERSISTENT, KIND_KVSPLIT = 0, 1, 2, 3
KIND_NAMES = {0: "auto", 1: "direct", 2: "persistent", 3: "kvsplit"}


class TopKError(RuntimeError):
    def __init__(self, code, where):
        super().__init__("%s: %s (%d)" % (where, STATUS_NAMES.get(code, "unknown"), code))
        self.code = code


class RowDiag(ctypes.Structure):
    _fields_ = [("tau0", ctypes.c_float), ("tau1", ctypes.c_float),
                ("count0", ctypes.c_int64), ("count1", ctypes.c_int64),
                ("path", ctypes.c_int32), ("flags", ctypes.c_uint32)]


DIAG_DTYPE = np.dtype([("tau0", "<f4"), ("tau1", "<f4"), ("count0", "<i8"), ("count1", "<i8"),
                       ("path", "<i4"), ("flags", "<u4")])
assert DIAG_DTYPE.itemsize == ctypes.sizeof(RowDiag)


class Params(ctypes.Structure):
    _fields_ = [("stride", ctypes.c_int32), ("rho0", ctypes.c_float), ("rho1", ctypes.c_float),
                ("sample_min_len", ctypes.c_int64), ("direct_max", ctypes.c_int64),
                ("force_kind", ctypes.c_int32), ("kv_segments", ctypes.c_int32),
                ("long_len", ctypes.c_int64), ("long_stride", ctypes.c_int32),
                ("long_rho0", ctypes.c_float), ("long_rho1", ctypes.c_float)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("grid", ctypes.c_int32), ("segments", ctypes.c_int32),
                ("sm_count", ctypes.c_int32), ("workspace_bytes", ctypes.c_size_t),
                ("smem_bytes", ctypes.c_size_t)]


EXPORTS = ("topk_ragged", "topk_ragged_diag", "topk_ragged_ws", "topk_workspace_bytes",
           "topk_ragged_host", "topk_plan", "topk_set_params", "topk_get_params",
           "topk_default_params", "topk_read_status", "topk_release_workspaces",
           "topk_status_string", "topk_version", "topk_ragged_noalloc",
           "topk_index_scores", "topk_index_topk", "topk_index_read_status",
           "topk_ragged_bf16", "topk_ragged_bf16_diag", "topk_sort_rows", "topk_sort_rows_bf16",
           "topk_check_wait_timeout", "topk_ragged_k", "topk_ragged_k_bf16", "topk_ragged_k_diag",
           "topk_ragged_e4m3", "topk_ragged_e4m3_diag", "topk_ragged_k_e4m3", "topk_sort_rows_e4m3",
           "topk_cached_workspace", "topk_index_topk_fused")
NOALLOC_MAX_ROWS = 64

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and return the CUDA library; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            "CUDA selector library not found at %s; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no CPU fallback)" % path)
    lib = ctypes.CDLL(path)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    lib.topk_ragged.argtypes = [vp, vp, i64, i64, i32, vp, vp]
    lib.topk_ragged_diag.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp]
    lib.topk_ragged_ws.argtypes = [vp, vp, i64, i64, i32, vp, vp, sz, vp]
    lib.topk_ragged_noalloc.argtypes = [vp, vp, i64, i64, i32, vp, vp]
    lib.topk_ragged_bf16.argtypes = [vp, vp, i64, i64, i32, vp, vp]
    lib.topk_ragged_k.argtypes = [vp, vp, vp, i64, i64, i32, vp, vp]
    lib.topk_ragged_k_bf16.argtypes = [vp, vp, vp, i64, i64, i32, vp, vp]
    lib.topk_ragged_k_diag.argtypes = [vp, vp, vp, i64, i64, i32, vp, vp, vp]
    lib.topk_ragged_e4m3.argtypes = [vp, vp, i64, i64, i32, vp, vp]
    lib.topk_ragged_e4m3_diag.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp]
    lib.topk_ragged_k_e4m3.argtypes = [vp, vp, vp, i64, i64, i32, vp, vp]
    lib.topk_sort_rows_e4m3.argtypes = [vp, i64, i64, i32, vp, vp]
    lib.topk_sort_rows.argtypes = [vp, i64, i64, i32, vp, vp]
    lib.topk_check_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.topk_check_wait_timeout.restype = ctypes.c_int
    lib.topk_sort_rows_bf16.argtypes = [vp, i64, i64, i32, vp, vp]
    lib.topk_ragged_bf16_diag.argtypes = [vp, vp, i64, i64, i32, vp, vp, vp]
    lib.topk_index_scores.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, vp, i64, vp]
    lib.topk_index_topk.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, vp, i64, i32, vp, vp]
    lib.topk_index_topk_fused.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, vp, i64, i32, vp,
                                          vp, vp]
    lib.topk_index_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.topk_workspace_bytes.argtypes = [i64, i64, i32]
    lib.topk_workspace_bytes.restype = sz
    lib.topk_ragged_host.argtypes = [vp, vp, i64, i64, i32, vp, i64]
    lib.topk_plan.argtypes = [i64, i64, i32, ctypes.POINTER(PlanInfo)]
    lib.topk_cached_workspace.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(sz)]
    lib.topk_set_params.argtypes = [ctypes.POINTER(Params)]
    lib.topk_get_params.argtypes = [ctypes.POINTER(Params)]
    lib.topk_default_params.argtypes = [ctypes.POINTER(Params)]
    lib.topk_default_params.restype = None
    lib.topk_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.topk_release_workspaces.argtypes = []
    lib.topk_release_workspaces.restype = None
    lib.topk_status_string.argtypes = [ctypes.c_int]
    lib.topk_status_string.restype = ctypes.c_char_p
    lib.topk_version.argtypes = []
    for name in ("topk_ragged", "topk_ragged_diag", "topk_ragged_ws", "topk_ragged_host",
                 "topk_ragged_noalloc", "topk_index_scores", "topk_index_topk",
                 "topk_ragged_bf16", "topk_ragged_bf16_diag", "topk_sort_rows",
                 "topk_sort_rows_bf16", "topk_ragged_k", "topk_ragged_k_bf16",
                 "topk_ragged_k_diag", "topk_ragged_e4m3", "topk_ragged_e4m3_diag",
                 "topk_ragged_k_e4m3", "topk_sort_rows_e4m3", "topk_index_read_status",
                 "topk_plan", "topk_set_params", "topk_get_params", "topk_read_status",
                 "topk_version", "topk_cached_workspace", "topk_index_topk_fused"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(code, where):
    if code != TOPK_OK:
        raise TopKError(code, where)


def _stream_handle(device, stream):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


E4M3 = getattr(torch, "float8_e4m3fn", None)
NARROW = tuple(t for t in (torch.bfloat16, E4M3) if t is not None)


def _pick(lib, scores, name):
    """The entry point for the scores' element type: name, name_bf16 / _e4m3
    (a _diag suffix goes after the type, as in the C header)."""
    base, diag = (name[:-5], "_diag") if name.endswith("_diag") else (name, "")
    if scores.dtype == torch.bfloat16:
        return getattr(lib, base + "_bf16" + diag)
    if E4M3 is not None and scores.dtype == E4M3:
        return getattr(lib, base + "_e4m3" + diag)
    return getattr(lib, name)


def _inputs(scores, row_lens, K, out, allow_bf16=False):
    if not (isinstance(scores, torch.Tensor) and scores.is_cuda):
        raise TypeError("scores must be a CUDA tensor")
    ok_types = (torch.float32,) + NARROW if allow_bf16 else (torch.float32,)
    if scores.dtype not in ok_types or scores.dim() != 2:
        raise TypeError("scores must be a 2-D %s tensor [M, N_alloc]"
                        % " or ".join(str(t).replace("torch.", "") for t in ok_types))
    if not scores.is_contiguous():
        raise ValueError("scores must be contiguous (row stride N_alloc)")
    if not (isinstance(row_lens, torch.Tensor) and row_lens.device == scores.device
            and row_lens.dtype == torch.int32 and row_lens.dim() == 1
            and row_lens.shape[0] == scores.shape[0] and row_lens.is_contiguous()):
        raise TypeError("row_lens must be a contiguous int32 [M] tensor on the scores' device")
    M, N = scores.shape
    if out is None:
        out = torch.empty((M, K), dtype=torch.int32, device=scores.device)
    elif not (out.device == scores.device and out.dtype == torch.int32
              and tuple(out.shape) == (M, K) and out.is_contiguous()):
        raise TypeError("out must be a contiguous int32 [M, K] tensor on the scores' device")
    return M, N, out


def topk_ragged(scores: torch.Tensor, row_lens: torch.Tensor, K: int = 2048,
                out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Exact Top-K of every row's valid prefix; [M, K] int32, unsorted, -1 padded.
    Scores are float32, bfloat16 or float8_e4m3fn (the narrow types selected as
    their exact float32 values)."""
    lib = load_library()
    M, N, out = _inputs(scores, row_lens, K, out, allow_bf16=True)
    fn = _pick(lib, scores, "topk_ragged")
    with torch.cuda.device(scores.device):
        rc = fn(scores.data_ptr(), row_lens.data_ptr(), M, N, K, out.data_ptr(),
                _stream_handle(scores.device, stream))
    _check(rc, "topk_ragged")
    return out


def _row_k(row_k, scores):
    if not (isinstance(row_k, torch.Tensor) and row_k.device == scores.device
            and row_k.dtype == torch.int32 and row_k.dim() == 1
            and row_k.shape[0] == scores.shape[0] and row_k.is_contiguous()):
        raise TypeError("row_k must be a contiguous int32 [M] tensor on the scores' device")
    return row_k


def topk_ragged_k(scores: torch.Tensor, row_lens: torch.Tensor, row_k: torch.Tensor,
                  K_max: int = 2048, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """Per-row K: row r gets its Top-k_r, k_r = clamp(row_k[r], 0, K_max), in
    slots [0, k_r) of an [M, K_max] int32 result; the other slots hold -1."""
    lib = load_library()
    M, N, out = _inputs(scores, row_lens, K_max, out, allow_bf16=True)
    row_k = _row_k(row_k, scores)
    fn = _pick(lib, scores, "topk_ragged_k")
    with torch.cuda.device(scores.device):
        rc = fn(scores.data_ptr(), row_lens.data_ptr(), row_k.data_ptr(), M, N, K_max,
                out.data_ptr(), _stream_handle(scores.device, stream))
    _check(rc, "topk_ragged_k")
    return out


def topk_ragged_k_diag(scores, row_lens, row_k, K_max: int = 2048, out=None, stream=None):
    """topk_ragged_k (float32 rows) plus per-row diagnostics (host copy)."""
    lib = load_library()
    M, N, out = _inputs(scores, row_lens, K_max, out)
    row_k = _row_k(row_k, scores)
    diag = torch.empty(M * DIAG_DTYPE.itemsize, dtype=torch.uint8, device=scores.device)
    with torch.cuda.device(scores.device):
        rc = lib.topk_ragged_k_diag(scores.data_ptr(), row_lens.data_ptr(), row_k.data_ptr(), M,
                                    N, K_max, out.data_ptr(), diag.data_ptr(),
                                    _stream_handle(scores.device, stream))
    _check(rc, "topk_ragged_k_diag")
    return out, diag.cpu().numpy().view(DIAG_DTYPE)


def topk_sort_rows(scores, out, stream=None):
    """Sort each row of a Top-K result in place: score descending, equal
    scores by index, -1 sentinels last (the selection itself is unordered)."""
    lib = load_library()
    if not (isinstance(scores, torch.Tensor) and scores.is_cuda and scores.dim() == 2
            and scores.dtype in (torch.float32,) + NARROW and scores.is_contiguous()):
        raise TypeError("scores must be a contiguous 2-D float32, bfloat16 or float8_e4m3fn "
                        "CUDA tensor")
    if not (isinstance(out, torch.Tensor) and out.device == scores.device
            and out.dtype == torch.int32 and out.dim() == 2 and out.shape[0] == scores.shape[0]
            and out.is_contiguous()):
        raise TypeError("out must be a contiguous int32 [M, K] tensor on the scores' device")
    M, N = scores.shape
    fn = _pick(lib, scores, "topk_sort_rows")
    with torch.cuda.device(scores.device):
        rc = fn(scores.data_ptr(), M, N, out.shape[1], out.data_ptr(),
                _stream_handle(scores.device, stream))
    _check(rc, "topk_sort_rows")
    return out


def topk_ragged_diag(scores, row_lens, K: int = 2048, out=None, stream=None):
    """topk_ragged plus per-row diagnostics (numpy structured array, host copy)."""
    lib = load_library()
    M, N, out = _inputs(scores, row_lens, K, out, allow_bf16=True)
    diag = torch.empty(M * DIAG_DTYPE.itemsize, dtype=torch.uint8, device=scores.device)
    fn = _pick(lib, scores, "topk_ragged_diag")
    with torch.cuda.device(scores.device):
        rc = fn(scores.data_ptr(), row_lens.data_ptr(), M, N, K, out.data_ptr(), diag.data_ptr(),
                _stream_handle(scores.device, stream))
    _check(rc, "topk_ragged_diag")
    return out, diag.cpu().numpy().view(DIAG_DTYPE)


def workspace_bytes(M: int, N_alloc: int, K: int = 2048) -> int:
    return int(load_library().topk_workspace_bytes(M, N_alloc, K))


def topk_ragged_ws(scores, row_lens, K, workspace: torch.Tensor, out=None, stream=None):
    """Explicit-workspace form; `workspace` is a zero-initialised CUDA byte tensor."""
    lib = load_library()
    M, N, out = _inputs(scores, row_lens, K, out)
    with torch.cuda.device(scores.device):
        rc = lib.topk_ragged_ws(scores.data_ptr(), row_lens.data_ptr(), M, N, K, out.data_ptr(),
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream_handle(scores.device, stream))
    _check(rc, "topk_ragged_ws")
    return out


def topk_ragged_noalloc(scores, row_lens, K: int = 2048, out=None, stream=None):
    """Fixed-scratch form: allocates no device memory in the library.

    For callers that may not allocate (an allocator that owns the whole GPU,
    a plugin host that forbids allocation while it runs).  At most
    NOALLOC_MAX_ROWS rows per call; calls that overlap on the GPU race on the
    shared scratch.  Pass `out` to avoid the one allocation this wrapper would
    otherwise make for the result tensor.
    """
    lib = load_library()
    M, N, out = _inputs(scores, row_lens, K, out)
    with torch.cuda.device(scores.device):
        rc = lib.topk_ragged_noalloc(scores.data_ptr(), row_lens.data_ptr(), M, N, K,
                                     out.data_ptr(), _stream_handle(scores.device, stream))
    _check(rc, "topk_ragged_noalloc")
    return out


def topk_ragged_host(scores: np.ndarray, row_lens: np.ndarray, K: int = 2048,
                     out: np.ndarray = None, rows_per_chunk: int = 0) -> np.ndarray:
    """Host-buffer form: host arrays in, host indices out (copies inside the call)."""
    lib = load_library()
    if not (isinstance(scores, np.ndarray) and scores.dtype == np.float32 and scores.ndim == 2
            and scores.flags.c_contiguous):
        raise TypeError("scores must be a C-contiguous float32 [M, N_alloc] array")
    row_lens = np.ascontiguousarray(row_lens, dtype=np.int32)
    M, N = scores.shape
    if out is None:
        out = np.empty((M, K), dtype=np.int32)
    rc = lib.topk_ragged_host(scores.ctypes.data, row_lens.ctypes.data, M, N, K, out.ctypes.data,
                              rows_per_chunk)
    _check(rc, "topk_ragged_host")
    return out


def plan(M: int, N_alloc: int, K: int = 2048) -> dict:
    info = PlanInfo()
    _check(load_library().topk_plan(M, N_alloc, K, ctypes.byref(info)), "topk_plan")
    return {"kind": KIND_NAMES[info.kind], "grid": info.grid, "segments": info.segments,
            "sm_count": info.sm_count, "workspace_bytes": info.workspace_bytes,
            "smem_bytes": info.smem_bytes}


def get_params() -> dict:
    p = Params()
    _check(load_library().topk_get_params(ctypes.byref(p)), "topk_get_params")
    return {f: getattr(p, f) for f, _ in Params._fields_}


def default_params() -> dict:
    p = Params()
    load_library().topk_default_params(ctypes.byref(p))
    return {f: getattr(p, f) for f, _ in Params._fields_}


def set_params(**kw) -> dict:
    """Update process-wide parameters; returns the previous values."""
    old = get_params()
    new = dict(old)
    for k, v in kw.items():
        if k not in new:
            raise KeyError(k)
        new[k] = v
    p = Params(**new)
    _check(load_library().topk_set_params(ctypes.byref(p)), "topk_set_params")
    return old


def read_status(device=None, stream=None) -> int:
    """Read and clear the device status word (OR of FLAG_* since the last read)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        _check(load_library().topk_read_status(_stream_handle(dev, stream), ctypes.byref(flags)),
               "topk_read_status")
    return int(flags.value)


def cached_workspace(device=None, stream=None):
    """(device address, bytes) of the library's workspace for (device, stream);
    (0, 0) when the stream has none yet."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    ptr, nbytes = ctypes.c_void_p(0), ctypes.c_size_t(0)
    with torch.cuda.device(dev):
        _check(load_library().topk_cached_workspace(_stream_handle(dev, stream),
                                                    ctypes.byref(ptr), ctypes.byref(nbytes)),
               "topk_cached_workspace")
    return int(ptr.value or 0), int(nbytes.value)


def release_workspaces() -> None:
    load_library().topk_release_workspaces()


def version() -> int:
    return int(load_library().topk_version())


def _index_inputs(q, k, w, row_lens, scores):
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("w", w, torch.float32)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dt and t.is_contiguous()):
            raise TypeError("%s must be a contiguous CUDA %s tensor" % (name, dt))
    if q.dim() != 3 or k.dim() != 2 or w.dim() != 2:
        raise TypeError("need q [T, H, D], k [S, D], w [T, H]")
    T, H, D = q.shape
    S = k.shape[0]
    if k.shape[1] != D or tuple(w.shape) != (T, H):
        raise TypeError("q, k and w disagree on H or D")
    if not (k.device == q.device == w.device):
        raise TypeError("q, k and w must be on one device")
    if row_lens is not None and not (row_lens.device == q.device and row_lens.dtype == torch.int32
                                     and tuple(row_lens.shape) == (T,)
                                     and row_lens.is_contiguous()):
        raise TypeError("row_lens must be a contiguous int32 [T] tensor on q's device")
    if scores is None:
        scores = torch.empty((T, S), dtype=torch.float32, device=q.device)
    elif not (scores.device == q.device and scores.dtype == torch.float32 and scores.dim() == 2
              and scores.shape[0] == T and scores.shape[1] >= S and scores.stride(1) == 1
              and scores.stride(0) == scores.shape[1]):
        raise TypeError("scores must be a contiguous float32 [T, >= S] tensor on q's device")
    return T, S, H, D, scores


def topk_index_scores(q, k, w, row_lens=None, scores=None, stream=None):
    """Indexer scores scores[t, s] = sum_j w[t, j] * ReLU(q[t, j] . k[s]) on the
    tensor cores; q [T, 64, 128] and k [S, 128] bfloat16, w [T, 64] float32.
    Scores at s >= row_lens[t] are -inf when row_lens is given."""
    lib = load_library()
    T, S, H, D, scores = _index_inputs(q, k, w, row_lens, scores)
    with torch.cuda.device(q.device):
        rc = lib.topk_index_scores(q.data_ptr(), k.data_ptr(), w.data_ptr(), T, S, H, D,
                                   row_lens.data_ptr() if row_lens is not None else None,
                                   scores.data_ptr(), scores.shape[1],
                                   _stream_handle(q.device, stream))
    _check(rc, "topk_index_scores")
    return scores


def topk_index_topk(q, k, w, row_lens, K: int = 2048, scores=None, out=None, stream=None):
    """Scores (as topk_index_scores) then the exact Top-K of every row's valid
    prefix; returns (scores, out_idx [T, K] int32)."""
    lib = load_library()
    if row_lens is None:
        raise TypeError("row_lens is required")
    T, S, H, D, scores = _index_inputs(q, k, w, row_lens, scores)
    if out is None:
        out = torch.empty((T, K), dtype=torch.int32, device=q.device)
    elif not (out.device == q.device and out.dtype == torch.int32 and tuple(out.shape) == (T, K)
              and out.is_contiguous()):
        raise TypeError("out must be a contiguous int32 [T, K] tensor on q's device")
    with torch.cuda.device(q.device):
        rc = lib.topk_index_topk(q.data_ptr(), k.data_ptr(), w.data_ptr(), T, S, H, D,
                                 row_lens.data_ptr(), scores.data_ptr(), scores.shape[1], K,
                                 out.data_ptr(), _stream_handle(q.device, stream))
    _check(rc, "topk_index_topk")
    return scores, out


def topk_index_topk_fused(q, k, w, row_lens, K: int = 2048, scores=None, out=None, diag=False,
                          stream=None):
    """Scores with the Top-K's threshold and candidate collection moved into
    the score kernel (see topk_index_topk_fused in include/topk.h): returns
    (scores, out_idx [T, K] int32) or, with diag=True, (scores, out_idx, diag
    as a numpy structured array).  The result is the exact Top-K of the
    scores written."""
    lib = load_library()
    if row_lens is None:
        raise TypeError("row_lens is required")
    T, S, H, D, scores = _index_inputs(q, k, w, row_lens, scores)
    if out is None:
        out = torch.empty((T, K), dtype=torch.int32, device=q.device)
    elif not (out.device == q.device and out.dtype == torch.int32 and tuple(out.shape) == (T, K)
              and out.is_contiguous()):
        raise TypeError("out must be a contiguous int32 [T, K] tensor on q's device")
    dg = torch.empty(T * DIAG_DTYPE.itemsize, dtype=torch.uint8, device=q.device) if diag else None
    with torch.cuda.device(q.device):
        rc = lib.topk_index_topk_fused(q.data_ptr(), k.data_ptr(), w.data_ptr(), T, S, H, D,
                                       row_lens.data_ptr(), scores.data_ptr(), scores.shape[1], K,
                                       out.data_ptr(), dg.data_ptr() if diag else None,
                                       _stream_handle(q.device, stream))
    _check(rc, "topk_index_topk_fused")
    if diag:
        return scores, out, dg.cpu().numpy().view(DIAG_DTYPE)
    return scores, out


def index_read_status(device=None, stream=None) -> int:
    """Read and clear the score kernel's status word (syncs the stream)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        _check(lib.topk_index_read_status(_stream_handle(dev, stream), ctypes.byref(flags)),
               "topk_index_read_status")
    return int(flags.value)

