"""The C ABI without a GPU: the library builds, loads and exports every function
include/proj.h declares; host-side validation returns the documented status
codes; the planner keeps the K-split independent of the row count (the
precondition of bitwise fused == separate); and with no device the library
fails loudly instead of computing on the CPU."""
import ctypes
import os
import re
import subprocess

import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hsp():
    from hidden_state_projection_gb300 import build
    build.build()
    import hidden_state_projection_gb300 as m
    m.lib()
    return m


def _declared():
    text = open(os.path.join(ROOT, "include", "proj.h")).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(proj_\w+)\s*\(", text, re.M)))


def test_header_declarations_are_exported(hsp):
    names = _declared()
    assert "proj_fused_gemm" in names and "proj_separate_gemm" in names
    lib = hsp.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", hsp.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (proj_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    assert set(hsp.EXPORTED) == set(names)


def _call(hsp, x=0x10000, w=0x20000, splits=(16, 8), outs=None, M=1, K=64, dtype=0, n=None):
    outs = outs if outs is not None else [0x30000 + 0x1000 * i for i in range(len(splits))]
    ns = (ctypes.c_int32 * max(1, len(splits)))(*splits)
    po = (ctypes.c_void_p * max(1, len(outs)))(*outs)
    return hsp.lib().proj_fused_gemm(x, w, ns, len(splits) if n is None else n, po, M, K, dtype, None)


def test_validation_codes(hsp):
    S = hsp.STATUS
    assert _call(hsp, dtype=9) == S["PROJ_ERR_UNSUPPORTED_DTYPE"]
    assert _call(hsp, M=65) == S["PROJ_ERR_UNSUPPORTED_SHAPE"]
    assert _call(hsp, M=-1) == S["PROJ_ERR_INVALID_ARG"]
    assert _call(hsp, K=0) == S["PROJ_ERR_UNSUPPORTED_SHAPE"]
    assert _call(hsp, K=60) == S["PROJ_ERR_MISALIGNED"]           # 120-byte rows
    assert _call(hsp, K=62, dtype=1) == S["PROJ_ERR_MISALIGNED"]  # 248-byte rows
    assert _call(hsp, x=0x10008) == S["PROJ_ERR_MISALIGNED"]
    assert _call(hsp, w=0x20004) == S["PROJ_ERR_MISALIGNED"]
    assert _call(hsp, outs=[0x30001, 0x31000]) == S["PROJ_ERR_MISALIGNED"]
    assert _call(hsp, x=0) == S["PROJ_ERR_INVALID_ARG"]
    assert _call(hsp, outs=[0x30000, 0]) == S["PROJ_ERR_INVALID_ARG"]
    assert _call(hsp, splits=(16, 0)) == S["PROJ_ERR_INVALID_ARG"]
    assert _call(hsp, splits=tuple([1] * 9)) == S["PROJ_ERR_UNSUPPORTED_SHAPE"]
    assert _call(hsp, splits=(), outs=[]) == S["PROJ_ERR_INVALID_ARG"]
    assert "exceeds" in hsp.lib().proj_last_error_string().decode() or True
    # an empty batch touches nothing and needs no device
    assert _call(hsp, M=0) == S["PROJ_OK"]


def test_no_device_fails_loudly(hsp):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    st = _call(hsp)
    assert st in (hsp.STATUS["PROJ_ERR_CUDA"], hsp.STATUS["PROJ_ERR_DEVICE"])
    assert hsp.lib().proj_last_error_string().decode()


def test_supported(hsp):
    assert hsp.supported(1, 5120, 1792, 0)
    assert hsp.supported(64, 7168, 2304, 0)
    assert hsp.supported(64, 7168, 192, 2)
    assert not hsp.supported(65, 5120, 1792, 0)
    assert not hsp.supported(0, 5120, 1792, 0)
    assert not hsp.supported(1, 5121, 1792, 0)
    assert not hsp.supported(1, 5120, 1792, 7)


def _plan_dtype(dtype, tf32):
    return 0 if dtype == "bf16" else (2 if tf32 else 1)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_k_split_independent_of_rows(hsp, name):
    wl = W.WORKLOADS[name]
    for tf32 in ([False, True] if wl.dtype == "fp32" else [False]):
        dt = _plan_dtype(wl.dtype, tf32)
        for M in range(1, 65):
            full = hsp.describe_plan(M, wl.K, wl.n_total, dt)
            for n in list(wl.splits) + [1, 3, 17, 5000]:
                part = hsp.describe_plan(M, wl.K, n, dt)
                for key in ("bucket", "k_warps", "slices", "units_per_slice", "compute"):
                    assert part[key] == full[key], (name, M, n, key)


def test_plan_fits_the_hardware(hsp):
    for name, wl in W.WORKLOADS.items():
        for dt in ([0] if wl.dtype == "bf16" else [1, 2]):
            for M in (1, 8, 9, 16, 17, 32, 33, 64):
                for n in (wl.n_total, *wl.splits):
                    p = hsp.describe_plan(M, wl.K, n, dt)
                    assert p["smem_bytes"] <= 232448
                    assert p["row_ctas"] * p["rows_per_cta"] >= n
                    assert p["slices"] in (1, 2, 4, 8, 16)
                    if p["engine"] == 3:     # fp32 register GEMV: all of K per CTA, one token group
                        assert dt == 1 and p["slices"] == 1 and p["threads"] == 512
                        cap = min(8, 192 * 1024 // (wl.K * 4))
                        groups = -(-M // cap)
                        assert p["token_tiles"] == groups
                        assert p["smem_bytes"] == -(-M // groups) * wl.K * 4 <= 192 * 1024
                        assert (groups - 1) * -(-M // groups) < M          # no empty group
                        assert p["row_ctas"] * groups <= 152
                    elif p["engine"] == 2:   # register-ring kernel: bf16, M <= 8, 16 warps split K
                        assert M <= 8 and dt == 0 and wl.K * 2 % 128 == 0
                        assert p["rows_per_cta"] <= 16 and p["threads"] == 512 and p["slices"] == 1
                        assert p["smem_bytes"] == wl.K * 2 * M + 1024
                    elif p["engine"] == 0:   # bulk-copy + mma.sync / FMA kernel
                        assert p["rows_per_cta"] <= p["row_warps"] * p["row_tiles"] * 16
                        assert p["ring_stages"] >= 1
                        assert (p["row_warps"] * p["row_tiles"] * 16) % p["slices"] == 0
                        assert p["threads"] == 288
                    else:                    # tensor-memory kernel: 64- or 128-row tiles, 2 CTAs per SM
                        assert (M > 8 and dt == 0) or dt == 2      # bf16 above 8 tokens; tf32 at every M
                        assert p["rows_per_cta"] in (64, 128) and p["threads"] == 128
                        assert p["smem_bytes"] <= 113 * 1024
                        assert p["ring_stages"] >= 2 and p["rows_per_cta"] % p["slices"] == 0
                        # 64-row tiles when all of them fit one wave at 2 per SM, or at 3 per SM
                        # where their shared memory allows (16 or 32 tokens)
                        tiles64 = -(-n // 64) * p["slices"]
                        fits2 = tiles64 <= {1: 304, 2: 304, 4: 296, 8: 288, 16: 224}[p["slices"]]
                        fits3 = tiles64 <= {1: 456, 2: 456, 4: 448, 8: 432, 16: 336}[p["slices"]]
                        if p["rows_per_cta"] == 64:
                            assert fits2 or (fits3 and p["smem_bytes"] <= 74 * 1024)
                        else:
                            assert not fits2 and (M > 32 or not fits3)
                        # two k-blocks per stage only where no stage reaches past its slice
                        # or adds a zero-filled k-block (so the bits are those of one)
                        esz = 2 if dt == 0 else 4
                        kb_total = -(-wl.K * esz // 128)
                        if p["k_per_stage"] == 2 * 128 // esz:
                            assert p["rows_per_cta"] == 64 and wl.K * esz % 128 == 0
                            assert kb_total % 2 == 0 and p["units_per_slice"] % 2 == 0
                            assert p["stages_total"] * 2 == p["units_per_slice"]
                        else:
                            assert p["k_per_stage"] == 128 // esz



def test_pack_check_and_options(hsp):
    lib = hsp.lib()
    base = 0x7F0000000000
    K = 5120
    assert lib.proj_pack_check(base + 1280 * K * 2, base, 1280, 512, 1792, K, 0) == 1
    assert lib.proj_pack_check(base + 1280 * K * 2 + 2, base, 1280, 512, 1792, K, 0) == 0
    assert lib.proj_pack_check(base, base, 1280, 513, 1792, K, 0) == 0
    hsp.set_options(pdl=False, wait_limit_us=5, skip_stage=3)
    assert hsp.get_options() == {"pdl": 0, "wait_limit_us": 5, "skip_stage_plus1": 4,
                                 "large_m_path": 0, "l2_prefetch": 0, "trigger_early": 0, "small_m_path": 0,
                                 "reg_path": 0}
    hsp.set_options(pdl=True, wait_limit_us=0, skip_stage=None, large_m_path=1, l2_prefetch=True)
    assert hsp.get_options()["large_m_path"] == 1 and hsp.get_options()["l2_prefetch"] == 1
    hsp.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    assert hsp.get_options() == {"pdl": 1, "wait_limit_us": 0, "skip_stage_plus1": 0,
                                 "large_m_path": 0, "l2_prefetch": 0, "trigger_early": 0, "small_m_path": 0,
                                 "reg_path": 0}
    with pytest.raises(hsp.ProjError):
        hsp.set_options(wait_limit_us=-1)
    with pytest.raises(hsp.ProjError):
        hsp.set_options(large_m_path=3)
    # the default engine for bf16: streaming (or the register ring) up to 8 tokens, tensor memory above
    assert [hsp.describe_plan(M, 7168, 2304, 0)["engine"] for M in (1, 8, 9, 16, 17, 64)] == [0, 0, 1, 1, 1, 1]
    hsp.set_options(large_m_path=2)
    assert [hsp.describe_plan(M, 7168, 2304, 0)["engine"] for M in (8, 9, 16, 17)] == [0, 1, 1, 1]
    # bf16 rows of at most 80 k-units (K <= 5120) at M <= 8: the register-ring kernel
    hsp.set_options(pdl=True)
    assert [hsp.describe_plan(M, 5120, 1792, 0)["engine"] for M in (1, 4, 8, 9)] == [2, 2, 2, 1]
    assert hsp.describe_plan(8, 5120, 1792, 0)["rows_per_cta"] <= 16
    assert hsp.describe_plan(8, 5112, 1792, 0)["engine"] == 0        # rows not a whole number of k-units
    assert hsp.describe_plan(1, 5120, 1792, 1)["engine"] == 3        # fp32: the register GEMV
    hsp.set_options(reg_path=1)
    assert hsp.describe_plan(8, 5120, 1792, 0)["engine"] == 0
    hsp.set_options(reg_path=2)
    assert hsp.describe_plan(8, 7168, 2304, 0)["engine"] == 2
    assert hsp.describe_plan(8, 8256, 2304, 0)["engine"] == 0        # 129 k-units: past the forced limit
    # fp32 at M <= 8 with the tokens within 192 KB: the register GEMV; tf32 keeps the tensor cores
    hsp.set_options(pdl=True)
    assert [hsp.describe_plan(M, 7168, 192, 1)["engine"] for M in (1, 4, 6, 7, 9)] == [3, 3, 3, 0, 0]
    assert [hsp.describe_plan(M, 6144, 256, 1)["engine"] for M in (8, 9)] == [3, 0]
    # forced: more tokens than one CTA holds (6 rows of 7168 floats within 192 KB) go in groups
    hsp.set_options(reg_path=2)
    assert [hsp.describe_plan(M, 7168, 192, 1)["engine"] for M in (1, 7, 16, 64)] == [3] * 4
    assert [hsp.describe_plan(M, 7168, 192, 1)["token_tiles"] for M in (6, 7, 16, 64)] == [1, 2, 3, 11]
    assert hsp.describe_plan(64, 7168, 192, 1)["smem_bytes"] == 6 * 7168 * 4
    hsp.set_options(reg_path=0)
    assert [hsp.describe_plan(M, 6144, 256, 1)["engine"] for M in (1, 8)] == [3, 3]
    # tf32: the streaming mma.sync kernel by default; large_m_path 2: the tensor-memory kernel (kind::tf32)
    assert [hsp.describe_plan(M, 7168, 192, 2)["engine"] for M in (1, 8, 9, 64)] == [0, 0, 0, 0]
    hsp.set_options(large_m_path=2)
    assert [hsp.describe_plan(M, 7168, 192, 2)["engine"] for M in (1, 8, 9, 64)] == [1, 1, 1, 1]
    assert hsp.describe_plan(64, 7168, 192, 2)["slices"] == 16
    hsp.set_options(large_m_path=0)
    assert hsp.describe_plan(1, 8196, 192, 1)["engine"] == 0            # K past 8192
    hsp.set_options(reg_path=1)
    assert hsp.describe_plan(1, 7168, 192, 1)["engine"] == 0
    with pytest.raises(hsp.ProjError):
        hsp.set_options(reg_path=3)
    hsp.set_options(pdl=True)


def _pack(hsp, ws, n_rows, K=64, dtype=0, w_cat=0x7F0000000000, num=None):
    ptrs = (ctypes.c_void_p * max(1, len(ws)))(*ws)
    ns = (ctypes.c_int32 * max(1, len(n_rows)))(*n_rows)
    return hsp.lib().proj_pack_weights(ptrs, ns, len(ws) if num is None else num, K, dtype, w_cat, None)


def test_pack_refusals(hsp):
    """proj_pack_weights checks its arguments on the host before anything is enqueued
    (TensorRT-LLM PR #20636, Description: the packed tensor is the weights' row
    concatenation, so a source inside W_cat other than its own rows cannot be copied)."""
    S = hsp.STATUS
    base, K = 0x7F0000000000, 64
    pitch = K * 2
    a, b = 0x7E0000000000, 0x7E0000100000
    before = hsp.launch_count()
    assert _pack(hsp, [a, b], [16, 8], dtype=9) == S["PROJ_ERR_UNSUPPORTED_DTYPE"]
    assert _pack(hsp, [a, b], [16, 8], K=60) == S["PROJ_ERR_MISALIGNED"]           # 120-byte rows
    assert _pack(hsp, [a, b], [16, 8], K=62, dtype=1) == S["PROJ_ERR_MISALIGNED"]  # 248-byte rows
    assert _pack(hsp, [a, b], [16, 8], w_cat=base + 8) == S["PROJ_ERR_MISALIGNED"]
    assert _pack(hsp, [a + 4, b], [16, 8]) == S["PROJ_ERR_MISALIGNED"]
    assert _pack(hsp, [a, 0], [16, 8]) == S["PROJ_ERR_INVALID_ARG"]
    assert _pack(hsp, [a, b], [16, -1]) == S["PROJ_ERR_INVALID_ARG"]
    assert _pack(hsp, [a, b], [16, 8], K=0) == S["PROJ_ERR_INVALID_ARG"]
    assert _pack(hsp, [a] * 9, [1] * 9) == S["PROJ_ERR_INVALID_ARG"]
    assert _pack(hsp, [], [], num=0) == S["PROJ_ERR_INVALID_ARG"]
    assert _pack(hsp, [a, b], [16, 8], w_cat=0) == S["PROJ_ERR_INVALID_ARG"]
    # sources inside W_cat that are not their own rows: refused, whatever the overlap
    assert _pack(hsp, [base + 16 * pitch, b], [16, 8]) == S["PROJ_ERR_INVALID_ARG"]   # ws[0] on ws[1]'s rows
    assert _pack(hsp, [a, base + 8 * pitch], [16, 8]) == S["PROJ_ERR_INVALID_ARG"]    # ws[1] straddles both
    assert _pack(hsp, [base - 8 * pitch, b], [16, 8]) == S["PROJ_ERR_INVALID_ARG"]    # ends inside W_cat
    assert "overlaps w_cat" in hsp.lib().proj_last_error_string().decode()
    # just below and just past W_cat: no overlap; every part its own rows: nothing to do
    assert _pack(hsp, [base, base + 16 * pitch], [16, 8]) == S["PROJ_OK"]
    assert _pack(hsp, [base, b], [16, 0]) == S["PROJ_OK"]                              # empty part skipped
    assert _pack(hsp, [base, 0], [16, 0]) == S["PROJ_OK"]                              # ... even as NULL
    assert hsp.launch_count() == before


def test_prefetch_entry_validation(hsp):
    import ctypes
    S = hsp.STATUS
    lib = hsp.lib()
    ns = (ctypes.c_int32 * 2)(16, 8)
    po = (ctypes.c_void_p * 2)(0x30000, 0x31000)
    def call(ranges, n):
        arr = (hsp.PrefetchRange * max(1, len(ranges)))(*[hsp.PrefetchRange(p, b) for p, b in ranges])
        return lib.proj_fused_gemm_prefetch(0x10000, 0x20000, ns, 2, po, 1, 64, 0, arr, n, None)
    assert call([], 5) == S["PROJ_ERR_INVALID_ARG"]
    assert call([(0, 64)], 1) == S["PROJ_ERR_INVALID_ARG"]
    assert call([(0x40008, 64)], 1) == S["PROJ_ERR_MISALIGNED"]
    assert call([(0x40000, 60)], 1) == S["PROJ_ERR_MISALIGNED"]
    assert call([(0x40000, 0)], 1) == S["PROJ_ERR_INVALID_ARG"]


def test_rmsnorm_workspace_size(hsp):
    """Workspace sizing is host-only: counters, parked fp32 values [M][cols] per split
    and per-CTA sums; 0 (with a reason) for shapes the epilogue does not run."""
    n = hsp.rmsnorm_workspace_bytes(1, 5120, (1280, 512), (1280, 512))
    assert n >= 256 + (1280 + 512) * 4 and n % 256 == 0
    assert hsp.rmsnorm_workspace_bytes(8, 5120, (1280, 512), (1280, 512)) >= 256 + 8 * (1280 + 512) * 4
    assert hsp.rmsnorm_workspace_bytes(1, 5120, (1280, 512), (0, 0)) == 256
    for bad in ((9, 5120, (1280, 512), (1280, 512), 0), (1, 5120, (1280, 512), (1281, 512), 0),
                (1, 5120, (1280, 512), (1280, 512), 1)):
        with pytest.raises(hsp.ProjError):
            hsp.rmsnorm_workspace_bytes(*bad)
