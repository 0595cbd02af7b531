"""CPU oracle for the fused hidden-state projection (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it: the arithmetic lives in ``oracle.c`` (fp64 accumulate
in index order, one rounding to the output dtype), and this module only builds
that file with the host C compiler and marshals numpy arrays into it.

    y[m, n]   = sum_k x[m, k] * w_cat[n, k]         (fp64, increasing k)
    out_i     = round_out(y[:, off_i : off_i + N_i])  (bf16 RNE or fp32 RNE)

Passages: TensorRT-LLM PR #20636 (DeepSeek-V4.1 wq_a/wkv via tinygemm2),
Description -- row-concatenated weight, one GEMM, per-projection dense outputs;
TensorRT-LLM PR #12055 (indexer wk + weights_proj in one TF32 GEMM),
Description -- the FP32 indexer variant; TensorRT-LLM PR #20502 (GLM-5.2
decode target), glmFusedAGemm commit message -- FP32 sums rounded once.

Parity pins (tests/test_oracle.py): brute force with exact integer arithmetic,
one-hot activations, linearity in X, the concatenation invariant, a float64
library matmul, a brute-force nearest-value search for the bf16 rounding, and
hand-derived values in tests/golden/.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

BF16 = 0
FP32 = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared object with the host C compiler.

    Plain -O2 without fast-math and without FMA contraction, so every fp64
    operation is the IEEE one written in the source."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.oracle_fused.argtypes = [vp, vp, ctypes.POINTER(i32), i32, ctypes.POINTER(vp),
                                 i64, i64, ctypes.c_int, ctypes.c_int]
    lib.oracle_fused.restype = ctypes.c_int
    lib.oracle_separate.argtypes = lib.oracle_fused.argtypes
    lib.oracle_separate.restype = ctypes.c_int
    lib.oracle_accumulate.argtypes = [vp, vp, i64, i64, i64, ctypes.c_int, vp]
    lib.oracle_accumulate.restype = None
    lib.oracle_round.argtypes = [vp, i64, ctypes.c_int, vp]
    lib.oracle_round.restype = None
    lib.oracle_fused_rmsnorm.argtypes = [vp, vp, ctypes.POINTER(i32), i32, ctypes.POINTER(i32),
                                         ctypes.POINTER(vp), ctypes.c_double, ctypes.POINTER(vp), i64, i64,
                                         ctypes.c_int]
    lib.oracle_fused_rmsnorm.restype = ctypes.c_int
    lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    _lib = lib
    return lib


def _in_array(a: np.ndarray, dtype: int) -> np.ndarray:
    """bf16 data travels as uint16 bit patterns, fp32 as float32."""
    want = np.uint16 if dtype == BF16 else np.float32
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"oracle expects {want.__name__} arrays for dtype {dtype}, got {a.dtype}")
    return a


def accumulate(x: np.ndarray, w: np.ndarray, dtype: int) -> np.ndarray:
    """fp64 sums y[m, n] = sum_k x[m, k] w[n, k], before any rounding."""
    lib = _load()
    x = _in_array(x, dtype)
    w = _in_array(w, dtype)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2
    y = np.zeros((M, N), dtype=np.float64)
    lib.oracle_accumulate(x.ctypes.data, w.ctypes.data, M, N, K, dtype, y.ctypes.data)
    return y


def round_out(y: np.ndarray, dtype: int) -> np.ndarray:
    """Round fp64 values once to the output dtype (bf16 bits as uint16, or fp32)."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.empty(y.shape, dtype=np.uint16 if dtype == BF16 else np.float32)
    lib.oracle_round(y.ctypes.data, y.size, dtype, out.ctypes.data)
    return out


def double_to_bf16(v: float) -> int:
    return int(_load().oracle_double_to_bf16(float(v)))


def _run(fn_name: str, x, w_cat, n_splits: Sequence[int], dtype: int, threads: int):
    lib = _load()
    x = _in_array(x, dtype)
    w_cat = _in_array(w_cat, dtype)
    M, K = x.shape
    if w_cat.shape != (sum(n_splits), K):
        raise ValueError("w_cat shape does not match the splits")
    odt = np.uint16 if dtype == BF16 else np.float32
    outs = [np.empty((M, int(n)), dtype=odt) for n in n_splits]
    ns = (ctypes.c_int32 * len(n_splits))(*[int(n) for n in n_splits])
    ptrs = (ctypes.c_void_p * len(outs))(*[o.ctypes.data for o in outs])
    rc = getattr(lib, fn_name)(x.ctypes.data, w_cat.ctypes.data, ns, len(n_splits), ptrs,
                               M, K, dtype, int(threads))
    if rc != 0:
        raise RuntimeError(f"{fn_name} failed ({rc})")
    return outs


def fused(x, w_cat, n_splits: Sequence[int], dtype: int, threads: int = 1):
    """Fused projection: list of per-split outputs [M, N_i]."""
    return _run("oracle_fused", x, w_cat, n_splits, dtype, threads)


def separate(x, w_cat, n_splits: Sequence[int], dtype: int, threads: int = 1):
    """One projection per split over its row range of w_cat."""
    return _run("oracle_separate", x, w_cat, n_splits, dtype, threads)


def fused_rmsnorm(x, w_cat, n_splits: Sequence[int], norm_cols: Sequence[int], gammas, eps: float, dtype: int):
    """Fused projection with the RMSNorm epilogue: split i's first norm_cols[i] columns
    are normalized per token and scaled by gammas[i] (an array of the data type, or
    None when norm_cols[i] is 0)."""
    lib = _load()
    x = _in_array(x, dtype)
    w_cat = _in_array(w_cat, dtype)
    M, K = x.shape
    if w_cat.shape != (sum(n_splits), K):
        raise ValueError("w_cat shape does not match the splits")
    odt = np.uint16 if dtype == BF16 else np.float32
    outs = [np.empty((M, int(n)), dtype=odt) for n in n_splits]
    gs = [None if g is None else _in_array(np.asarray(g), dtype) for g in gammas]
    ns = (ctypes.c_int32 * len(n_splits))(*[int(n) for n in n_splits])
    nc = (ctypes.c_int32 * len(n_splits))(*[int(c) for c in norm_cols])
    gp = (ctypes.c_void_p * len(n_splits))(*[None if g is None else g.ctypes.data for g in gs])
    ptrs = (ctypes.c_void_p * len(outs))(*[o.ctypes.data for o in outs])
    rc = lib.oracle_fused_rmsnorm(x.ctypes.data, w_cat.ctypes.data, ns, len(n_splits), nc, gp, float(eps),
                                  ptrs, M, K, dtype)
    if rc != 0:
        raise RuntimeError(f"oracle_fused_rmsnorm failed ({rc})")
    return outs


def cpu_count() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# Arm main-ID part numbers of server cores (Arm's technical reference manuals)
_ARM_PARTS = {"0xd0c": "Neoverse N1", "0xd40": "Neoverse V1", "0xd49": "Neoverse N2",
              "0xd4f": "Neoverse V2", "0xd84": "Neoverse V3", "0xd8e": "Neoverse N3"}


def host_description() -> str:
    """CPU model of the host: the x86 model name, or for Arm the core named by its part number."""
    model, implementer, part = "", "", ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model") and not model:
                    model = line.split(":", 1)[1].strip()
                elif key == "cpu implementer" and not implementer:
                    implementer = line.split(":", 1)[1].strip().lower()
                elif key == "cpu part" and not part:
                    part = line.split(":", 1)[1].strip().lower()
    except OSError:
        pass
    if model:
        return model
    if implementer == "0x41" and part:
        return f"{platform.machine()} {_ARM_PARTS.get(part, 'Arm part ' + part)}"
    return platform.machine()
