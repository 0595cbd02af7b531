"""Fused hidden-state projection for GB300 (sm_103a): Python binding.

The work happens in ``_lib/libhsp_proj.so`` (hand-written CUDA behind the C ABI
declared in ``include/proj.h``).  This module only marshals arguments: device
pointers from torch tensors, the current CUDA stream, host arrays of split sizes
and output pointers.  There is no CPU path; if the library is missing, importing
the functions raises.

    y = x @ w_cat.T            (x [M, K], w_cat [sum(splits), K])
    outs[i] = y[:, off_i : off_i + splits[i]]   as separate dense tensors

TensorRT-LLM PR #20636 (DeepSeek-V4.1 wq_a/wkv via tinygemm2), Description.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libhsp_proj.so")

PROJ_BF16, PROJ_FP32, PROJ_TF32 = 0, 1, 2
STATUS_NAMES = {0: "PROJ_OK", 1: "PROJ_ERR_INVALID_ARG", 2: "PROJ_ERR_UNSUPPORTED_SHAPE",
                3: "PROJ_ERR_MISALIGNED", 4: "PROJ_ERR_UNSUPPORTED_DTYPE", 5: "PROJ_ERR_DEVICE",
                6: "PROJ_ERR_CUDA", 7: "PROJ_ERR_TIMEOUT"}
STATUS = {v: k for k, v in STATUS_NAMES.items()}
MAX_SPLITS = 8
MAX_M = 64

EXPORTED = ("proj_fused_gemm", "proj_fused_gemm_prefetch", "proj_fused_gemm_host",
            "proj_host_plan_create", "proj_host_plan_launch", "proj_host_plan_destroy", "proj_fused_gemm_rmsnorm", "proj_rmsnorm_workspace_bytes",
            "proj_fused_gemm_rmsnorm_static",
            "proj_separate_gemm", "proj_pack_weights", "proj_pack_check",
            "proj_supported", "proj_describe_plan", "proj_set_options", "proj_get_options",
            "proj_check_device_error", "proj_launch_count", "proj_last_error_string", "proj_version")


class ProjError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


class Options(ctypes.Structure):
    _fields_ = [("pdl", ctypes.c_int32), ("wait_limit_us", ctypes.c_int32),
                ("skip_stage_plus1", ctypes.c_int32), ("large_m_path", ctypes.c_int32),
                ("l2_prefetch", ctypes.c_int32), ("trigger_early", ctypes.c_int32),
                ("small_m_path", ctypes.c_int32), ("reg_path", ctypes.c_int32)]


class PrefetchRange(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_uint64)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "bucket", "compute", "rows_per_cta", "row_ctas", "slices", "k_warps", "row_warps",
        "row_tiles", "token_tiles", "ring_stages", "stage_bytes", "smem_bytes", "k_per_stage",
        "stages_total", "threads", "units_per_slice", "engine", "tensor_copies")] + [("reserved", ctypes.c_int32 * 2)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_ if n != "reserved"}


_lib = None


def lib() -> ctypes.CDLL:
    """Load libhsp_proj.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                           "(python -m hidden_state_projection_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    gemm_args = [vp, vp, ctypes.POINTER(i32), i32, ctypes.POINTER(vp), i32, i32, ctypes.c_int, vp]
    for name in ("proj_fused_gemm", "proj_separate_gemm"):
        getattr(L, name).argtypes = gemm_args
        getattr(L, name).restype = ctypes.c_int
    L.proj_fused_gemm_host.argtypes = gemm_args[:8] + [vp, ctypes.POINTER(vp), vp]
    L.proj_fused_gemm_host.restype = ctypes.c_int
    L.proj_host_plan_create.argtypes = gemm_args[:8] + [vp, ctypes.POINTER(vp), ctypes.POINTER(vp)]
    L.proj_host_plan_create.restype = ctypes.c_int
    L.proj_host_plan_launch.argtypes = [vp, vp]
    L.proj_host_plan_launch.restype = ctypes.c_int
    L.proj_host_plan_destroy.argtypes = [vp]
    L.proj_host_plan_destroy.restype = ctypes.c_int
    L.proj_fused_gemm_prefetch.argtypes = gemm_args[:8] + [ctypes.POINTER(PrefetchRange), i32, vp]
    L.proj_fused_gemm_prefetch.restype = ctypes.c_int
    L.proj_pack_weights.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(i32), i32, i32, ctypes.c_int, vp, vp]
    L.proj_pack_weights.restype = ctypes.c_int
    L.proj_fused_gemm_rmsnorm.argtypes = [vp, vp, ctypes.POINTER(i32), i32, ctypes.POINTER(i32), ctypes.POINTER(vp),
                                          ctypes.c_float, ctypes.POINTER(vp), i32, i32, ctypes.c_int, vp,
                                          ctypes.c_size_t, vp]
    L.proj_fused_gemm_rmsnorm.restype = ctypes.c_int
    L.proj_fused_gemm_rmsnorm_static.argtypes = [vp, vp, ctypes.POINTER(i32), i32, ctypes.POINTER(i32),
                                                 ctypes.POINTER(vp), ctypes.c_float, ctypes.POINTER(vp), i32, i32,
                                                 ctypes.c_int, vp]
    L.proj_fused_gemm_rmsnorm_static.restype = ctypes.c_int
    L.proj_rmsnorm_workspace_bytes.argtypes = [i32, i32, ctypes.POINTER(i32), i32, ctypes.POINTER(i32), ctypes.c_int]
    L.proj_rmsnorm_workspace_bytes.restype = ctypes.c_size_t
    L.proj_pack_check.argtypes = [vp, vp, i64, i32, i32, i32, ctypes.c_int]
    L.proj_pack_check.restype = ctypes.c_int
    L.proj_supported.argtypes = [i32, i32, i32, ctypes.c_int]
    L.proj_supported.restype = ctypes.c_int
    L.proj_describe_plan.argtypes = [i32, i32, i32, ctypes.c_int, ctypes.POINTER(PlanInfo)]
    L.proj_describe_plan.restype = ctypes.c_int
    L.proj_set_options.argtypes = [ctypes.POINTER(Options)]
    L.proj_set_options.restype = ctypes.c_int
    L.proj_get_options.argtypes = [ctypes.POINTER(Options)]
    L.proj_get_options.restype = ctypes.c_int
    L.proj_check_device_error.argtypes = [vp]
    L.proj_check_device_error.restype = ctypes.c_int
    L.proj_launch_count.argtypes = []
    L.proj_launch_count.restype = ctypes.c_uint64
    L.proj_last_error_string.argtypes = []
    L.proj_last_error_string.restype = ctypes.c_char_p
    L.proj_version.argtypes = []
    L.proj_version.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int) -> None:
    if status != 0:
        msg = lib().proj_last_error_string().decode(errors="replace")
        raise ProjError(status, msg)


def dtype_code(t: torch.Tensor, tf32: bool = False) -> int:
    if t.dtype == torch.bfloat16:
        return PROJ_BF16
    if t.dtype == torch.float32:
        return PROJ_TF32 if tf32 else PROJ_FP32
    raise ProjError(4, f"unsupported tensor dtype {t.dtype}")


def _stream_ptr(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- pointer-level calls (exactly the C ABI) -----------------------------------

def fused_gemm_ptr(x_ptr: int, w_ptr: int, splits: Sequence[int], out_ptrs: Sequence[int],
                   M: int, K: int, dtype: int, stream_ptr: int = 0) -> None:
    ns = (ctypes.c_int32 * len(splits))(*[int(s) for s in splits])
    po = (ctypes.c_void_p * len(out_ptrs))(*[int(p) for p in out_ptrs])
    _check(lib().proj_fused_gemm(x_ptr, w_ptr, ns, len(splits), po, M, K, dtype, stream_ptr))


def fused_gemm_prefetch_ptr(x_ptr: int, w_ptr: int, splits: Sequence[int], out_ptrs: Sequence[int],
                            M: int, K: int, dtype: int, prefetch: Sequence[tuple], stream_ptr: int = 0) -> None:
    ns = (ctypes.c_int32 * len(splits))(*[int(s) for s in splits])
    po = (ctypes.c_void_p * len(out_ptrs))(*[int(p) for p in out_ptrs])
    pr = (PrefetchRange * max(1, len(prefetch)))(*[PrefetchRange(int(p), int(b)) for p, b in prefetch])
    _check(lib().proj_fused_gemm_prefetch(x_ptr, w_ptr, ns, len(splits), po, M, K, dtype, pr, len(prefetch),
                                          stream_ptr))


def separate_gemm_ptr(x_ptr: int, w_ptr: int, splits: Sequence[int], out_ptrs: Sequence[int],
                      M: int, K: int, dtype: int, stream_ptr: int = 0) -> None:
    ns = (ctypes.c_int32 * len(splits))(*[int(s) for s in splits])
    po = (ctypes.c_void_p * len(out_ptrs))(*[int(p) for p in out_ptrs])
    _check(lib().proj_separate_gemm(x_ptr, w_ptr, ns, len(splits), po, M, K, dtype, stream_ptr))


# ---- tensor-level calls ---------------------------------------------------------

def _outs(x: torch.Tensor, splits: Sequence[int], outs: Optional[List[torch.Tensor]]):
    M = x.shape[0]
    if outs is None:
        return [torch.empty((M, int(n)), dtype=x.dtype, device=x.device) for n in splits]
    if len(outs) != len(splits):
        raise ProjError(1, "one output per split is required")
    for o, n in zip(outs, splits):
        if o.shape != (M, int(n)) or o.dtype != x.dtype or not o.is_contiguous():
            raise ProjError(1, f"output must be a dense [{M}, {n}] {x.dtype} tensor")
    return outs


def _gemm(fn, x, w_cat, splits, outs, tf32, stream):
    if x.dim() != 2 or w_cat.dim() != 2 or not x.is_contiguous() or not w_cat.is_contiguous():
        raise ProjError(1, "x and w_cat must be dense 2-D tensors")
    if x.dtype != w_cat.dtype:
        raise ProjError(4, "x and w_cat must have the same dtype")
    if x.shape[1] != w_cat.shape[1] or w_cat.shape[0] != sum(int(s) for s in splits):
        raise ProjError(2, "shapes do not match: x [M, K], w_cat [sum(splits), K]")
    outs = _outs(x, splits, outs)
    fn(x.data_ptr(), w_cat.data_ptr(), splits, [o.data_ptr() for o in outs], x.shape[0], x.shape[1],
       dtype_code(x, tf32), _stream_ptr(stream))
    return outs


def fused_gemm(x: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int],
               outs: Optional[List[torch.Tensor]] = None, tf32: bool = False, stream=None):
    """One launch over all of w_cat; returns one dense [M, N_i] tensor per split."""
    return _gemm(fused_gemm_ptr, x, w_cat, splits, outs, tf32, stream)


def fused_gemm_prefetch(x: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int],
                        prefetch: Sequence[torch.Tensor], outs: Optional[List[torch.Tensor]] = None,
                        tf32: bool = False, stream=None):
    """fused_gemm that also prefetches the given tensors (e.g. the next layer's weights) into L2."""
    ranges = [(t.data_ptr(), t.numel() * t.element_size()) for t in prefetch]

    def fn(xp, wp, sp, op, M, K, dt, st):
        fused_gemm_prefetch_ptr(xp, wp, sp, op, M, K, dt, ranges, st)
    return _gemm(fn, x, w_cat, splits, outs, tf32, stream)


class HostCall:
    """A fused call bound once to fixed buffers, for a loop that repeats it (a decode
    step): proj_fused_gemm_host with its ctypes arguments built here, so each call is one
    foreign-function call.  x_host / outs_host are pinned CPU tensors, x_dev / outs_dev
    device staging tensors of the same shapes; w_cat stays on the device.  Calling the
    object enqueues the token copy (a staging kernel when x_host is pinned, else a
    copy-engine copy), the projection and, for outputs not in pinned memory, D2H copies on
    the stream; synchronise before reading outs_host."""

    def __init__(self, x_host: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int],
                 outs_host: Sequence[torch.Tensor], x_dev: torch.Tensor, outs_dev: Sequence[torch.Tensor],
                 tf32: bool = False, stream=None):
        M, K = x_dev.shape
        if x_host.shape != x_dev.shape or x_host.dtype != x_dev.dtype or not x_host.is_contiguous():
            raise ProjError(1, "x_host must be a dense tensor shaped and typed like x_dev")
        if len(outs_host) != len(splits) or len(outs_dev) != len(splits):
            raise ProjError(1, "one host and one device output per split")
        _outs(x_dev, splits, list(outs_dev))
        for h, n in zip(outs_host, splits):
            if h.shape != (M, int(n)) or h.dtype != x_dev.dtype or not h.is_contiguous():
                raise ProjError(1, f"host output must be a dense [{M}, {n}] {x_dev.dtype} tensor")
        self._keep = (x_host, w_cat, list(outs_host), x_dev, list(outs_dev))
        vp = ctypes.c_void_p
        self._args = (x_host.data_ptr(), w_cat.data_ptr(),
                      (ctypes.c_int32 * len(splits))(*[int(s) for s in splits]), len(splits),
                      (vp * len(splits))(*[h.data_ptr() for h in outs_host]), M, K, dtype_code(x_dev, tf32),
                      x_dev.data_ptr(), (vp * len(splits))(*[o.data_ptr() for o in outs_dev]), _stream_ptr(stream))
        self._fn = lib().proj_fused_gemm_host

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != 0:
            _check(rc)


class HostPlan:
    """proj_host_plan_*: the host step of HostCall recorded once as a CUDA graph inside the
    library; each call is one graph launch (H2D copy, projection, D2H copies) on the
    stream.  x_host and outs_host must be pinned; all buffers are kept alive by the plan."""

    def __init__(self, x_host: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int],
                 outs_host: Sequence[torch.Tensor], x_dev: torch.Tensor, outs_dev: Sequence[torch.Tensor],
                 tf32: bool = False, stream=None):
        bound = HostCall(x_host, w_cat, splits, outs_host, x_dev, outs_dev, tf32, stream)
        self._keep = bound._keep
        a = bound._args
        self._handle = ctypes.c_void_p()
        _check(lib().proj_host_plan_create(*a[:10], ctypes.byref(self._handle)))
        self._stream = _stream_ptr(stream)
        self._launch = lib().proj_host_plan_launch

    def __call__(self) -> None:
        rc = self._launch(self._handle, self._stream)
        if rc != 0:
            _check(rc)

    def close(self) -> None:
        if self._handle:
            _check(lib().proj_host_plan_destroy(self._handle))
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            if self._handle and _lib is not None:
                _lib.proj_host_plan_destroy(self._handle)
        except Exception:
            pass


def fused_gemm_host(x_host: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int],
                    outs_host: Sequence[torch.Tensor], x_dev: torch.Tensor, outs_dev: Sequence[torch.Tensor],
                    tf32: bool = False, stream=None) -> None:
    """One proj_fused_gemm_host call (see HostCall for a loop of them)."""
    HostCall(x_host, w_cat, splits, outs_host, x_dev, outs_dev, tf32, stream)()


def rmsnorm_workspace_bytes(M: int, K: int, splits: Sequence[int], norm_cols: Sequence[int], dtype: int = 0) -> int:
    """Workspace bytes of proj_fused_gemm_rmsnorm for this shape (raises if unsupported)."""
    ns = (ctypes.c_int32 * len(splits))(*[int(v) for v in splits])
    nc = (ctypes.c_int32 * len(norm_cols))(*[int(v) for v in norm_cols])
    n = int(lib().proj_rmsnorm_workspace_bytes(int(M), int(K), ns, len(splits), nc, int(dtype)))
    if n == 0:
        raise ProjError(2, lib().proj_last_error_string().decode())
    return n


def fused_gemm_rmsnorm_ptr(x_ptr: int, w_ptr: int, splits: Sequence[int], norm_cols: Sequence[int],
                           gamma_ptrs: Sequence[int], eps: float, out_ptrs: Sequence[int], M: int, K: int, dtype: int,
                           ws_ptr: int, ws_bytes: int, stream_ptr: int = 0) -> None:
    ns = (ctypes.c_int32 * len(splits))(*[int(v) for v in splits])
    nc = (ctypes.c_int32 * len(norm_cols))(*[int(v) for v in norm_cols])
    gp = (ctypes.c_void_p * len(gamma_ptrs))(*[int(p) if p else None for p in gamma_ptrs])
    po = (ctypes.c_void_p * len(out_ptrs))(*[int(p) for p in out_ptrs])
    _check(lib().proj_fused_gemm_rmsnorm(x_ptr, w_ptr, ns, len(splits), nc, gp, float(eps), po, M, K, dtype,
                                         ws_ptr, int(ws_bytes), stream_ptr))


def fused_gemm_rmsnorm(x: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int], norm_cols: Sequence[int],
                       gammas: Sequence[Optional[torch.Tensor]], eps: float, workspace: torch.Tensor,
                       outs: Optional[List[torch.Tensor]] = None, stream=None):
    """fused_gemm with the RMSNorm epilogue on the first norm_cols[i] columns of split i.
    `workspace` is a device byte tensor of at least rmsnorm_workspace_bytes(...) bytes,
    zeroed once before its first use (each call leaves it ready for the next)."""
    if len(norm_cols) != len(splits) or len(gammas) != len(splits):
        raise ProjError(1, "one norm_cols entry and one gamma per split")
    for g, c in zip(gammas, norm_cols):
        if c and (g is None or g.dtype != x.dtype or g.numel() < int(c) or not g.is_contiguous()):
            raise ProjError(1, "gamma of a normalized split must be a dense tensor of the data type")
    gp = [g.data_ptr() if (g is not None and c) else 0 for g, c in zip(gammas, norm_cols)]
    ws_bytes = workspace.numel() * workspace.element_size()

    def fn(xp, wp, sp, op, M, K, dt, st):
        fused_gemm_rmsnorm_ptr(xp, wp, sp, norm_cols, gp, eps, op, M, K, dt, workspace.data_ptr(), ws_bytes, st)
    return _gemm(fn, x, w_cat, splits, outs, False, stream)


def fused_gemm_rmsnorm_static(x: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int],
                              norm_cols: Sequence[int], gammas: Sequence[Optional[torch.Tensor]], eps: float,
                              outs: Optional[List[torch.Tensor]] = None, stream=None):
    """fused_gemm_rmsnorm without a workspace argument: proj_fused_gemm_rmsnorm_static uses
    the library's own fixed device array (for callers that cannot allocate).  Calls that
    overlap on the GPU race on that array."""
    if len(norm_cols) != len(splits) or len(gammas) != len(splits):
        raise ProjError(1, "one norm_cols entry and one gamma per split")
    for g, c in zip(gammas, norm_cols):
        if c and (g is None or g.dtype != x.dtype or g.numel() < int(c) or not g.is_contiguous()):
            raise ProjError(1, "gamma of a normalized split must be a dense tensor of the data type")
    gp = [g.data_ptr() if (g is not None and c) else 0 for g, c in zip(gammas, norm_cols)]

    def fn(xp, wp, sp, op, M, K, dt, st):
        ns = (ctypes.c_int32 * len(sp))(*[int(v) for v in sp])
        nc = (ctypes.c_int32 * len(norm_cols))(*[int(v) for v in norm_cols])
        gpa = (ctypes.c_void_p * len(gp))(*[int(p) if p else None for p in gp])
        po = (ctypes.c_void_p * len(op))(*[int(p) for p in op])
        _check(lib().proj_fused_gemm_rmsnorm_static(xp, wp, ns, len(sp), nc, gpa, float(eps), po, M, K, dt, st))
    return _gemm(fn, x, w_cat, splits, outs, False, stream)


def separate_gemm(x: torch.Tensor, w_cat: torch.Tensor, splits: Sequence[int],
                  outs: Optional[List[torch.Tensor]] = None, tf32: bool = False, stream=None):
    """One launch per split over its rows of w_cat; bitwise equal to fused_gemm."""
    return _gemm(separate_gemm_ptr, x, w_cat, splits, outs, tf32, stream)


def pack_weights(ws: Sequence[torch.Tensor], w_cat: Optional[torch.Tensor] = None, stream=None):
    """Row-concatenate weights into w_cat on the device (one copy kernel; parts that
    already are their own rows of w_cat are skipped); returns (w_cat, views of it).
    Passing the same w_cat again refreshes it in place, e.g. after a reload."""
    if not ws:
        raise ProjError(1, "at least one weight is required")
    K = ws[0].shape[1]
    dt = ws[0].dtype
    for w in ws:
        if w.dim() != 2 or w.shape[1] != K or w.dtype != dt or not w.is_contiguous():
            raise ProjError(1, "weights must be dense 2-D tensors with the same K and dtype")
    n_rows = [int(w.shape[0]) for w in ws]
    if w_cat is None:
        w_cat = torch.empty((sum(n_rows), K), dtype=dt, device=ws[0].device)
    elif w_cat.shape != (sum(n_rows), K) or w_cat.dtype != dt or not w_cat.is_contiguous():
        raise ProjError(1, f"w_cat must be a dense [{sum(n_rows)}, {K}] {dt} tensor")
    code = dtype_code(w_cat)
    ptrs = (ctypes.c_void_p * len(ws))(*[w.data_ptr() for w in ws])
    ns = (ctypes.c_int32 * len(ws))(*n_rows)
    _check(lib().proj_pack_weights(ptrs, ns, len(ws), K, code, w_cat.data_ptr(), _stream_ptr(stream)))
    views, off = [], 0
    for n in n_rows:
        views.append(w_cat[off:off + n])
        off += n
    return w_cat, views


def pack_check(w: torch.Tensor, w_cat: torch.Tensor, row_off: int) -> bool:
    """True if w is still the view of rows [row_off, row_off + len(w)) of w_cat."""
    return bool(lib().proj_pack_check(w.data_ptr(), w_cat.data_ptr(), row_off, w.shape[0],
                                      w_cat.shape[0], w_cat.shape[1], dtype_code(w_cat)))


def supported(M: int, K: int, n_total: int, dtype: int) -> bool:
    return bool(lib().proj_supported(M, K, n_total, dtype))


def describe_plan(M: int, K: int, n_rows: int, dtype: int) -> dict:
    info = PlanInfo()
    _check(lib().proj_describe_plan(M, K, n_rows, dtype, ctypes.byref(info)))
    return info.as_dict()


def set_options(pdl: Optional[bool] = None, wait_limit_us: int = 0, skip_stage: Optional[int] = None,
                large_m_path: int = 0, l2_prefetch: bool = False, trigger_early: bool = False,
                small_m_path: int = 0, reg_path: int = 0):
    o = Options()
    o.pdl = -1 if pdl is None else int(bool(pdl))
    o.wait_limit_us = int(wait_limit_us)
    o.skip_stage_plus1 = 0 if skip_stage is None else int(skip_stage) + 1
    o.large_m_path = int(large_m_path)
    o.l2_prefetch = 1 if l2_prefetch else 0
    o.trigger_early = 1 if trigger_early else 0
    o.small_m_path = int(small_m_path)
    o.reg_path = int(reg_path)
    _check(lib().proj_set_options(ctypes.byref(o)))


def get_options() -> dict:
    o = Options()
    _check(lib().proj_get_options(ctypes.byref(o)))
    return {"pdl": o.pdl, "wait_limit_us": o.wait_limit_us, "skip_stage_plus1": o.skip_stage_plus1,
            "large_m_path": o.large_m_path, "l2_prefetch": o.l2_prefetch, "trigger_early": o.trigger_early,
            "small_m_path": o.small_m_path, "reg_path": o.reg_path}


def check_device_error(stream=None) -> None:
    """Synchronise the stream and raise ProjError(PROJ_ERR_TIMEOUT) if a kernel gave up a wait."""
    _check(lib().proj_check_device_error(_stream_ptr(stream)))


def launch_count() -> int:
    return int(lib().proj_launch_count())


def version() -> str:
    return lib().proj_version().decode()
