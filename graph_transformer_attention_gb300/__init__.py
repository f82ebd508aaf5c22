"""Topology-biased graph attention on one GB300 (thin Python binding of libgt).

Every step of the computation runs in the CUDA kernels of libgt.so; this module
only marshals torch tensors into the C ABI declared in include/gt_attn.h (raw
device pointers, sizes, the current CUDA stream) and allocates outputs and
workspace with torch.  There is no CPU path: if libgt.so is missing or cannot
be loaded the calls raise.

Functions (same names as the C entry points):
    gt_spd_build(indptr, indices, n, D)                       -> spd int8 [n][ld]
    gt_bias_attn_fwd(q, k, v, spd, T, scale=None, kv_block=0) -> (o, lse)
    gt_bias_attn_bwd(q, k, v, o, dO, lse, spd, T, scale=None) -> (dq, dk, dv, dT)
The operation follows MegaGraph (abstract: attention scores plus a
topology-aware bias matrix; Fig. 4: blockwise KV streaming with the bias column
slice formed per block) with the Graphormer bias b[h][i][j] = T[h][spd[i][j]].
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = [
    "GtError", "load_library", "library_path", "gt_spd_build", "gt_bias_attn_fwd",
    "gt_bias_attn_bwd", "gt_spd_workspace_size", "gt_bias_attn_workspace_size",
    "gt_check_device_status", "gt_status_string", "spd_ld", "GT_F32", "GT_BF16",
    "GT_SPD_AUTO", "GT_SPD_SCAN32", "GT_SPD_SCAN16", "GT_SPD_QUEUE32", "GT_SPD_GLOBAL64",
]

GT_F32 = 0
GT_BF16 = 1
# search algorithms of gt_spd_build (include/gt_attn.h)
GT_SPD_AUTO, GT_SPD_SCAN32, GT_SPD_SCAN16, GT_SPD_QUEUE32, GT_SPD_GLOBAL64 = 0, 1, 2, 3, 4
GT_OK = 0
_STATUS = {0: "GT_OK", -1: "GT_ERR_INVALID_ARG", -2: "GT_ERR_UNSUPPORTED", -3: "GT_ERR_CUDA",
           -4: "GT_ERR_TIMEOUT", -5: "GT_ERR_WORKSPACE"}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgt.so")
_lock = threading.Lock()
_lib = None


class GtError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        text = _lib.gt_status_string(status).decode() if _lib is not None else ""
        super().__init__(f"{call} returned {_STATUS.get(status, status)}: {text}")


def library_path() -> str:
    return _LIB_PATH


class KernelStat(ctypes.Structure):
    """gt_kernel_stat of the C ABI."""
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


def load_library():
    """Load libgt.so (build it with graph_transformer_attention_gb300.build first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libgt.so not found at {_LIB_PATH}; run "
                               "`python -m graph_transformer_attention_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                                ctypes.c_float)
        lib.gt_status_string.argtypes = [ctypes.c_int]
        lib.gt_status_string.restype = ctypes.c_char_p
        lib.gt_spd_workspace_size.argtypes = [i32, i64, i32]
        lib.gt_spd_workspace_size.restype = sz
        lib.gt_spd_build.argtypes = [P, P, i32, i64, i32, P, i64, P, sz, P]
        lib.gt_spd_build.restype = ctypes.c_int
        lib.gt_spd_workspace_size_algo.argtypes = [i32, i32, i64, i32]
        lib.gt_spd_workspace_size_algo.restype = sz
        lib.gt_spd_build_algo.argtypes = [i32, P, P, i32, i64, i32, P, i64, P, sz, P]
        lib.gt_spd_build_algo.restype = ctypes.c_int
        lib.gt_bias_attn_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.gt_bias_attn_workspace_size.restype = sz
        lib.gt_bias_attn_fwd_kv_block.argtypes = [i32, i32, i32, i32, i32]
        lib.gt_bias_attn_fwd_kv_block.restype = i32
        lib.gt_bias_attn_fwd_ctas.argtypes = [i32, i32, i32, i32, i32]
        lib.gt_bias_attn_fwd_ctas.restype = i32
        lib.gt_bias_attn_launches.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.gt_bias_attn_launches.restype = ctypes.c_int
        lib.gt_bias_attn_bwd_split.argtypes = [i32, i32, i32, i32, i32]
        lib.gt_bias_attn_bwd_split.restype = i32
        lib.gt_bias_attn_fwd.argtypes = [i32, i32, i32, i32, P, P, P, P, i64, P, i32, f32, i32,
                                         P, P, P, sz, P]
        lib.gt_bias_attn_fwd.restype = ctypes.c_int
        lib.gt_bias_attn_bwd.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, i64, P, i32, f32,
                                         P, P, P, P, P, sz, P]
        lib.gt_bias_attn_bwd.restype = ctypes.c_int
        lib.gt_check_device_status.argtypes = [P]
        lib.gt_check_device_status.restype = ctypes.c_int
        lib.gt_selftest_wait_timeout.argtypes = [i64, P]
        lib.gt_selftest_wait_timeout.restype = ctypes.c_int
        lib.gt_layer_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.gt_layer_workspace_size.restype = sz
        lib.gt_layer_fwd.argtypes = [i32, i32, i32, i32, P, P, P, i64, P, i32, P, P, P, P, P, P, P, sz, P]
        lib.gt_layer_fwd.restype = ctypes.c_int
        lib.gt_layer_bwd.argtypes = [i32, i32, i32, i32, P, P, P, i64, P, i32, P, P, P, P, P, P, P, P, P,
                                     P, sz, P]
        lib.gt_layer_bwd.restype = ctypes.c_int
        lib.gt_bias_attn_fwd_partial.argtypes = [i32, i32, i32, i32, P, P, P, P, i64, P, i32, f32, i32,
                                                 i32, P, P, P]
        lib.gt_bias_attn_fwd_partial.restype = ctypes.c_int
        lib.gt_bias_attn_merge.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P]
        lib.gt_bias_attn_merge.restype = ctypes.c_int
        lib.gt_kernel_stats_reset.argtypes = [i32]
        lib.gt_kernel_stats_reset.restype = ctypes.c_int
        lib.gt_kernel_stats_read.argtypes = [ctypes.POINTER(KernelStat), i32, ctypes.POINTER(i32)]
        lib.gt_kernel_stats_read.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(call: str, rc: int):
    if rc != GT_OK:
        raise GtError(call, rc)


def _stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GT_F32
    if t.dtype == torch.bfloat16:
        return GT_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("libgt works on CUDA tensors only")
            if not t.is_contiguous():
                raise ValueError("libgt needs contiguous tensors")


def spd_ld(n: int) -> int:
    """Row stride of the SPD matrix: n rounded up to a multiple of 16 bytes."""
    return (n + 15) // 16 * 16


def launches_per_call(dtype: str, h: int, d: int, n: int, kv_block: int = 0, nb: int = 18) -> dict:
    """Number of libgt kernels gt_bias_attn_fwd and gt_bias_attn_bwd launch for
    these sizes on the current device (memsets not counted)."""
    code = GT_F32 if dtype == "f32" else GT_BF16
    fwd, bwd = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("gt_bias_attn_launches",
           load_library().gt_bias_attn_launches(code, n, h, d, nb, kv_block, ctypes.byref(fwd), ctypes.byref(bwd)))
    return {"fwd": int(fwd.value), "bwd": int(bwd.value)}


def gt_status_string(status: int) -> str:
    return load_library().gt_status_string(status).decode()


def gt_spd_workspace_size(n: int, nnz: int, D: int, algo: int = 0) -> int:
    """Workspace bytes of gt_spd_build (0 when `algo` cannot take n vertices here)."""
    return int(load_library().gt_spd_workspace_size_algo(algo, n, nnz, D))


def gt_bias_attn_workspace_size(dtype: int, n: int, h: int, d: int, kv_block: int = 0) -> int:
    return int(load_library().gt_bias_attn_workspace_size(dtype, n, h, d, kv_block))


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def gt_spd_build(indptr: torch.Tensor, indices: torch.Tensor, n: int, D: int,
                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                 stream=None, algo: int = 0) -> torch.Tensor:
    """Clipped shortest-path bucket matrix, int8 [n][spd_ld(n)] (columns >= n unspecified).

    `algo` picks the search (GT_SPD_*; 0 = the first that fits the device)."""
    lib = load_library()
    _need_cuda(indptr, indices)
    if indptr.dtype != torch.int64 or indices.dtype != torch.int32:
        raise TypeError("indptr must be int64 and indices int32")
    if out is None:
        out = torch.empty((n, spd_ld(n)), dtype=torch.int8, device=indptr.device)
    if workspace is None:
        need = lib.gt_spd_workspace_size_algo(algo, n, indices.numel(), D)
        if need == 0:
            raise GtError("gt_spd_build", -2)      # the algorithm cannot take n vertices here
        workspace = _workspace(need, indptr.device)
    rc = lib.gt_spd_build_algo(algo, _ptr(indptr), _ptr(indices), n, indices.numel(), D, _ptr(out),
                               out.stride(0), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check("gt_spd_build", rc)
    return out


def gt_bias_attn_fwd(q, k, v, spd, T, scale: float | None = None, kv_block: int = 0,
                     out=None, lse=None, workspace=None, stream=None):
    """Biased attention forward; q, k, v [n][h][d] (fp32 or bf16), spd int8 [n][ld], T fp32 [h][nb]."""
    lib = load_library()
    _need_cuda(q, k, v, spd, T)
    n, h, d = q.shape
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((h, n), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(lib.gt_bias_attn_workspace_size(dt, n, h, d, kv_block), q.device)
    rc = lib.gt_bias_attn_fwd(dt, n, h, d, _ptr(q), _ptr(k), _ptr(v), _ptr(spd), spd.stride(0),
                              _ptr(T), T.shape[1], float(scale), kv_block, _ptr(out), _ptr(lse),
                              _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check("gt_bias_attn_fwd", rc)
    return out, lse


def gt_bias_attn_fwd_partial(q, k, v, spd, T, kv_begin: int, kv_end: int, scale: float | None = None,
                             o_part=None, lse_part=None, stream=None):
    """Forward over the KV columns [kv_begin, kv_end) only: fp32 o_part [n][h][d]
    (normalised over those columns) and lse_part [h][n]."""
    lib = load_library()
    _need_cuda(q, k, v, spd, T)
    n, h, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o_part is None:
        o_part = torch.empty((n, h, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((h, n), dtype=torch.float32, device=q.device)
    _need_cuda(o_part, lse_part)
    rc = lib.gt_bias_attn_fwd_partial(_dtype_code(q), n, h, d, _ptr(q), _ptr(k), _ptr(v), _ptr(spd),
                                      spd.stride(0), _ptr(T), T.shape[1], float(scale), kv_begin, kv_end,
                                      _ptr(o_part), _ptr(lse_part), _stream_handle(stream))
    _check("gt_bias_attn_fwd_partial", rc)
    return o_part, lse_part


def gt_bias_attn_merge(o_parts, lse_parts, dtype=torch.bfloat16, out=None, lse=None, stream=None):
    """Exact merge of partials: o_parts fp32 [p][n][h][d], lse_parts fp32 [p][h][n]."""
    lib = load_library()
    _need_cuda(o_parts, lse_parts)
    nparts, n, h, d = o_parts.shape
    if out is None:
        out = torch.empty((n, h, d), dtype=dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty((h, n), dtype=torch.float32, device=o_parts.device)
    _need_cuda(out, lse)
    rc = lib.gt_bias_attn_merge(_dtype_code(out), n, h, d, nparts, _ptr(o_parts), _ptr(lse_parts),
                                _ptr(out), _ptr(lse), _stream_handle(stream))
    _check("gt_bias_attn_merge", rc)
    return out, lse


def gt_bias_attn_bwd(q, k, v, o, dO, lse, spd, T, scale: float | None = None,
                     dq=None, dk=None, dv=None, dT=None, workspace=None, stream=None):
    """Gradients of sum(o * dO): returns (dq, dk, dv, dT)."""
    lib = load_library()
    _need_cuda(q, k, v, o, dO, lse, spd, T)
    n, h, d = q.shape
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dT = torch.empty_like(T) if dT is None else dT
    if workspace is None:
        workspace = _workspace(lib.gt_bias_attn_workspace_size(dt, n, h, d, 0), q.device)
    rc = lib.gt_bias_attn_bwd(dt, n, h, d, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                              _ptr(spd), spd.stride(0), _ptr(T), T.shape[1], float(scale),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dT), _ptr(workspace),
                              workspace.numel(), _stream_handle(stream))
    _check("gt_bias_attn_bwd", rc)
    return dq, dk, dv, dT


LAYER_PARAMS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_1", "b_1", "w_2", "b_2")


class _LayerPtrs(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in LAYER_PARAMS]


def _layer_ptrs(tensors: dict) -> _LayerPtrs:
    for name in LAYER_PARAMS:
        t = tensors[name]
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"layer tensor {name} must be contiguous fp32 on the GPU")
    return _LayerPtrs(*[_ptr(tensors[name]) for name in LAYER_PARAMS])


def gt_layer_workspace_size(n: int, h: int = 8, d: int = 8, f: int = 64) -> int:
    return int(load_library().gt_layer_workspace_size(n, h, d, f))


def gt_layer_fwd(x, params: dict, spd, T, workspace=None, stream=None):
    """GT encoder layer forward: y fp32 [n][64] from x fp32 [n][64], and the saved
    tensors of the backward {q, k, v, o (bf16 [n][8][8]), lse}."""
    lib = load_library()
    _need_cuda(x, spd, T)
    n = x.shape[0]
    dev = x.device
    saved = {name: torch.empty((n, 8, 8), dtype=torch.bfloat16, device=dev) for name in ("q", "k", "v", "o")}
    saved["lse"] = torch.empty((8, n), dtype=torch.float32, device=dev)
    y = torch.empty_like(x)
    if workspace is None:
        workspace = _workspace(lib.gt_layer_workspace_size(n, 8, 8, 64), dev)
    w = _layer_ptrs(params)
    rc = lib.gt_layer_fwd(n, 8, 8, 64, _ptr(x), ctypes.byref(w), _ptr(spd), spd.stride(0), _ptr(T), T.shape[1],
                          _ptr(saved["q"]), _ptr(saved["k"]), _ptr(saved["v"]), _ptr(saved["o"]),
                          _ptr(saved["lse"]), _ptr(y), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check("gt_layer_fwd", rc)
    return y, saved


def gt_layer_bwd(x, params: dict, spd, T, saved: dict, dy, workspace=None, stream=None):
    """GT encoder layer backward: (dx, {weight name: gradient}, dT)."""
    lib = load_library()
    _need_cuda(x, spd, T, dy)
    n = x.shape[0]
    dev = x.device
    grads = {name: torch.empty_like(params[name]) for name in LAYER_PARAMS}
    dx = torch.empty_like(x)
    dT = torch.empty_like(T)
    if workspace is None:
        workspace = _workspace(lib.gt_layer_workspace_size(n, 8, 8, 64), dev)
    w = _layer_ptrs(params)
    g = _layer_ptrs(grads)
    rc = lib.gt_layer_bwd(n, 8, 8, 64, _ptr(x), ctypes.byref(w), _ptr(spd), spd.stride(0), _ptr(T), T.shape[1],
                          _ptr(saved["q"]), _ptr(saved["k"]), _ptr(saved["v"]), _ptr(saved["o"]),
                          _ptr(saved["lse"]), _ptr(dy), _ptr(dx), ctypes.byref(g), _ptr(dT), _ptr(workspace),
                          workspace.numel(), _stream_handle(stream))
    _check("gt_layer_bwd", rc)
    return dx, grads, dT


def gt_check_device_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel gave up a bounded wait."""
    _check("gt_check_device_status", load_library().gt_check_device_status(_stream_handle(stream)))


def gt_selftest_wait_timeout(limit_ns: int = 50_000_000, stream=None) -> None:
    """Launch the library's bounded-wait self-test: a wait that nothing ends, which
    gives up after limit_ns; the next gt_check_device_status reports GT_ERR_TIMEOUT."""
    _check("gt_selftest_wait_timeout",
           load_library().gt_selftest_wait_timeout(int(limit_ns), _stream_handle(stream)))


def gt_kernel_stats_reset(timing: bool = False) -> None:
    """Clear the library's launch table; with timing, bracket every launch with
    CUDA events on its stream from now on."""
    _check("gt_kernel_stats_reset", load_library().gt_kernel_stats_reset(1 if timing else 0))


def gt_kernel_stats() -> dict:
    """{kernel name: (launches, total device ms or -1 without timing)} since the
    last reset, in first-launch order."""
    lib = load_library()
    count = ctypes.c_int32(0)
    _check("gt_kernel_stats_read", lib.gt_kernel_stats_read(None, 0, ctypes.byref(count)))
    arr = (KernelStat * max(1, count.value))()
    _check("gt_kernel_stats_read", lib.gt_kernel_stats_read(arr, count.value, ctypes.byref(count)))
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms))
            for i in range(count.value)}
