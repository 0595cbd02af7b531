"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Every workload of the pages at its full size and every token count it names
(all outputs compared), plus ragged and edge shapes: K not a multiple of the
box width, splits of 1 / 3 / 17 rows, a single row, more rows than one wave,
every M from 1 to 64, small-integer inputs that must match bit for bit, and
one-hot activations that must reproduce weight columns exactly.
"""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import as_f64, check_close, mode_of, oracle_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    return m


def _run_both(hsp, x, w_cat, splits, tf32=False):
    dev = torch.device("cuda")
    xd, wd = x.to(dev), w_cat.to(dev)
    fused = hsp.fused_gemm(xd, wd, splits, tf32=tf32)
    sep = hsp.separate_gemm(xd, wd, splits, tf32=tf32)
    hsp.check_device_error()
    for a, b in zip(fused, sep):
        assert torch.equal(a, b), "fused and separate outputs differ"
    return fused


CASES = []
for name, wl in W.WORKLOADS.items():
    modes = [False, True] if wl.dtype == "fp32" else [False]
    for M in wl.Ms:
        for tf32 in modes:
            CASES.append(pytest.param(name, M, tf32, id=f"{name}-M{M}{'-tf32' if tf32 else ''}"))


@pytest.mark.parametrize("name,M,tf32", CASES)
def test_workload_full_size(hsp, name, M, tf32):
    wl = W.WORKLOADS[name]
    x = W.activation(wl, M)
    w_cat = W.weight_cat(wl)
    outs = _run_both(hsp, x, w_cat, wl.splits, tf32)
    check_close(outs, oracle_outputs(x, w_cat, wl.splits), mode_of(wl.dtype, tf32), f"{name} M{M}")


EDGE = [
    # (K, splits, M)
    (72, (1, 3, 17), 1),          # K one box plus a ragged tail, tiny splits
    (520, (33, 7), 3),            # K = 8 boxes + 8
    (64, (1,), 1),                # one row, one box
    (4096, (5000,), 2),           # more rows than one wave of CTAs
    (5120, (1536, 576, 128, 64), 5),
    (1024, (16, 16, 16, 16, 16, 16, 16, 16), 8),   # eight splits
    (6144, (2048, 576, 128), 7),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("K,splits,M", EDGE)
def test_edge_shapes(hsp, dtype, K, splits, M):
    x, ws = W.random_case(K, splits, M, dtype, seed=K + M + len(splits))
    w_cat = torch.cat(ws, 0)
    for tf32 in ([False, True] if dtype == "fp32" else [False]):
        outs = _run_both(hsp, x, w_cat, splits, tf32)
        check_close(outs, oracle_outputs(x, w_cat, splits), mode_of(dtype, tf32), f"K{K}")


@pytest.mark.parametrize("K,splits,M,row_tiles,token_tiles,slices", [
    (4096, (300, 100), 12, 4, 2, 16),   # 58 rows per CTA: four 16-row tiles, 4 x 2 lane tiles
    (4096, (300, 100), 24, 4, 4, 16),   # four tiles, 4 x 8 lane tiles
    (4096, (200, 100), 20, 3, 4, 16),   # 43 rows per CTA: three tiles
    (4096, (300, 100), 40, 3, 8, 16),   # 33-64 tokens: at most three tiles (12 x 8)
    (4096, (150, 50), 40, 2, 8, 16),    # 29 rows per CTA: two tiles (8 x 8)
    (4096, (60, 40), 48, 1, 8, 16),     # 15 rows per CTA: one tile (4 x 8)
    (2048, (60, 40), 10, 1, 2, 2),      # one tile, two K slices
])
def test_fp32_chunk_layout_tiles(hsp, K, splits, M, row_tiles, token_tiles, slices):
    """fp32 above 8 tokens: eight K warps, each on one 16-byte chunk of every unit, over
    one to four 16-row tiles (three at most from 33 tokens).  Every instance the planner can
    pick, against the oracle, fused and separate."""
    plan = hsp.describe_plan(M, K, sum(splits), 1)
    assert (plan["engine"], plan["k_warps"], plan["row_warps"]) == (0, 8, 1), plan
    assert (plan["row_tiles"], plan["token_tiles"], plan["slices"]) == (row_tiles, token_tiles, slices), plan
    x, ws = W.random_case(K, splits, M, "fp32", seed=3300 + K + M)
    w_cat = torch.cat(ws, 0)
    outs = _run_both(hsp, x, w_cat, splits)
    check_close(outs, oracle_outputs(x, w_cat, splits), "fp32", f"chunk K{K} M{M} RT{row_tiles}")


@pytest.mark.parametrize("dtype,tf32", [("bf16", False), ("fp32", False), ("fp32", True)])
def test_every_token_count(hsp, dtype, tf32):
    K, splits = 1536, (200, 56)
    for M in range(1, 65):
        x, ws = W.random_case(K, splits, M, dtype, seed=500 + M)
        w_cat = torch.cat(ws, 0)
        outs = _run_both(hsp, x, w_cat, splits, tf32)
        check_close(outs, oracle_outputs(x, w_cat, splits), mode_of(dtype, tf32), f"M{M}")


@pytest.mark.parametrize("name,tf32", [("wq_a_wkv", False), ("qk_indexer", False), ("glm_fused_a", False),
                                       ("indexer_fp32", False), ("indexer_fp32", True)])
def test_every_token_count_full_size(hsp, name, tf32):
    """Every M from 1 to 64 on a full-size weight of the pages' workloads, so that each
    switch of the dispatcher is crossed at real K and N: the register ring / streaming /
    tensor-memory engines at M = 8 | 9, the tcgen05 tile height at 32 | 33 (where it fits
    one wave), the fp32 GEMV's one-CTA token limit at 6 | 7, the token tiles of every
    bucket.  All outputs against the oracle, fused and separate bitwise equal."""
    wl = W.WORKLOADS[name]
    w_cat = W.weight_cat(wl)
    wd = w_cat.cuda()
    for M in range(1, 65):
        x = W.activation(wl, M, 2)
        xd = x.cuda()
        fused = hsp.fused_gemm(xd, wd, wl.splits, tf32=tf32)
        sep = hsp.separate_gemm(xd, wd, wl.splits, tf32=tf32)
        hsp.check_device_error()
        for a, b in zip(fused, sep):
            assert torch.equal(a, b), (name, M)
        check_close(fused, oracle_outputs(x, w_cat, wl.splits, threads=16), mode_of(wl.dtype, tf32), f"{name} M{M}")


@pytest.mark.parametrize("dtype,tf32", [("bf16", False), ("fp32", False), ("fp32", True)])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 33, 64])
def test_small_integers_bit_exact(hsp, dtype, tf32, M):
    # Every partial sum is an integer below 2^11: exact in fp32 and tf32 products,
    # results within bf16's exact integer range.
    K, splits = 64, (3, 16, 17)
    x, ws = W.small_int_case(K, splits, M, dtype, seed=77 + M)
    w_cat = torch.cat(ws, 0)
    outs = _run_both(hsp, x, w_cat, splits, tf32)
    ref = oracle_outputs(x, w_cat, splits)
    for g, r in zip(outs, ref):
        assert np.array_equal(as_f64(g), r)


@pytest.mark.parametrize("dtype,tf32", [("bf16", False), ("fp32", False)])
def test_one_hot_reproduces_columns(hsp, dtype, tf32):
    K, splits = 5120, (1280, 512)
    _, ws = W.random_case(K, splits, 1, dtype, seed=99)
    w_cat = torch.cat(ws, 0)
    cols = [0, 1, 63, 64, 511, 512, 2047, 4095, K - 2, K - 1]
    x = torch.zeros(len(cols), K, dtype=w_cat.dtype)
    for m, c in enumerate(cols):
        x[m, c] = 1
    outs = _run_both(hsp, x, w_cat, splits, tf32)
    for wi, oi in zip(ws, outs):
        for m, c in enumerate(cols):
            assert torch.equal(oi[m].cpu(), wi[:, c]), (dtype, c)


def test_zero_weights_and_negation(hsp):
    K, splits = 7168, (1536, 576)
    x, ws = W.random_case(K, splits, 8, "bf16", seed=5)
    w_cat = torch.cat(ws, 0)
    z = _run_both(hsp, x, torch.zeros_like(w_cat), splits)
    assert all(torch.count_nonzero(o) == 0 for o in z)
    pos = _run_both(hsp, x, w_cat, splits)
    neg = _run_both(hsp, -x, w_cat, splits)
    for p, n in zip(pos, neg):
        assert torch.equal(p, -n)


def test_empty_batch_is_a_no_op(hsp):
    K, splits = 512, (16, 8)
    w = torch.randn(24, K, device="cuda").to(torch.bfloat16)
    x = torch.empty(0, K, device="cuda", dtype=torch.bfloat16)
    before = hsp.launch_count()
    outs = hsp.fused_gemm(x, w, splits)
    assert [tuple(o.shape) for o in outs] == [(0, 16), (0, 8)]
    assert hsp.launch_count() == before


@pytest.mark.parametrize("M", [9, 16, 17, 32, 33, 64])
@pytest.mark.parametrize("forced", [1, 2])
def test_large_m_engines_match_oracle(hsp, M, forced):
    """bf16 at M > 8 runs the tensor-memory kernel; the streaming kernel can be forced for
    every M, and each must agree with the oracle."""
    K, splits = 7168, (1536, 576, 128, 64)
    x, ws = W.random_case(K, splits, M, "bf16", seed=900 + M)
    w_cat = torch.cat(ws, 0)
    hsp.set_options(pdl=True, large_m_path=forced)
    try:
        assert hsp.describe_plan(M, K, sum(splits), 0)["engine"] == (0 if forced == 1 else 1)
        outs = _run_both(hsp, x, w_cat, splits)
    finally:
        hsp.set_options(pdl=True, large_m_path=0)
    assert hsp.describe_plan(M, K, sum(splits), 0)["engine"] == 1
    check_close(outs, oracle_outputs(x, w_cat, splits), "bf16", f"engine {forced} M{M}")


@pytest.mark.parametrize("M", [33, 48, 64])
def test_tensor_memory_tile_height_keeps_the_bits(hsp, M):
    """At 33-64 tokens glm_fused_a's 2752 rows run as 128-row tiles when fused (43 tiles of
    64 over eight K slices would not fit one wave at two CTAs per SM) and each of its
    splits alone as 64-row tiles: the tile height is the MMA's M, and the stage shape (one
    k-block per stage at 128 rows, two at 64) is the copy granularity; neither may change
    a single output bit (fused = separate), and both agree with the oracle."""
    wl = W.WORKLOADS["glm_fused_a"]
    x = W.activation(wl, M)
    w_cat = W.weight_cat(wl)
    assert hsp.describe_plan(M, wl.K, wl.n_total, 0)["rows_per_cta"] == 128
    assert [hsp.describe_plan(M, wl.K, n, 0)["rows_per_cta"] for n in wl.splits] == [64] * len(wl.splits)
    outs = _run_both(hsp, x, w_cat, wl.splits)
    check_close(outs, oracle_outputs(x, w_cat, wl.splits), "bf16", f"glm_fused_a M{M}")


@pytest.mark.parametrize("M", [9, 16, 32])
def test_tensor_memory_stage_shape_keeps_the_bits(hsp, M):
    """9-32 tokens: 4096 rows of K = 6144 run fused as 128-row tiles with one k-block per
    stage (64 tiles of 64 rows over eight K slices would not fit one wave even at three
    CTAs per SM), each 2048-row split alone as 64-row tiles with two k-blocks per stage
    (one 3-D box of each).  The outputs must be bitwise equal and agree with the oracle."""
    K, splits = 6144, (2048, 2048)
    fused_plan = hsp.describe_plan(M, K, sum(splits), 0)
    split_plan = hsp.describe_plan(M, K, splits[0], 0)
    assert (fused_plan["rows_per_cta"], fused_plan["k_per_stage"]) == (128, 64), fused_plan
    assert (split_plan["rows_per_cta"], split_plan["k_per_stage"]) == (64, 128), split_plan
    x, ws = W.random_case(K, splits, M, "bf16", seed=5100 + M)
    w_cat = torch.cat(ws, 0)
    outs = _run_both(hsp, x, w_cat, splits)
    check_close(outs, oracle_outputs(x, w_cat, splits), "bf16", f"stage shape M{M}")


@pytest.mark.parametrize("M", [1, 2])
def test_bf16_fma_small_m_path_matches_oracle(hsp, M):
    """The opt-in CUDA-core path for bf16 with one or two tokens."""
    K, splits = 5120, (1280, 512)
    x, ws = W.random_case(K, splits, M, "bf16", seed=700 + M)
    w_cat = torch.cat(ws, 0)
    hsp.set_options(pdl=True, small_m_path=1)
    try:
        assert hsp.describe_plan(M, K, sum(splits), 0)["compute"] == 3
        outs = _run_both(hsp, x, w_cat, splits)
    finally:
        hsp.set_options(pdl=True, small_m_path=0)
    check_close(outs, oracle_outputs(x, w_cat, splits), "bf16", f"bf16 fma M{M}")


@pytest.mark.parametrize("K,splits", [(5120, (1280, 512)), (1536, (200, 56)), (7168, (1536, 576, 128, 64))])
@pytest.mark.parametrize("reg_path", [0, 1, 2])
def test_register_ring_and_streaming_engines_match_oracle(hsp, K, splits, reg_path):
    """bf16 at M <= 8: the register-ring kernel (default for K <= 5120, forced up to
    K = 8192 with reg_path 2, where its ring of five k-units is refilled) and the
    streaming kernel (reg_path 1) both agree with the oracle, fused and separate."""
    hsp.set_options(pdl=True, reg_path=reg_path)
    try:
        for M in (1, 2, 5, 8):
            x, ws = W.random_case(K, splits, M, "bf16", seed=1300 + M + K)
            w_cat = torch.cat(ws, 0)
            want = 2 if (reg_path == 2 or (reg_path == 0 and K <= 5120)) else 0
            assert hsp.describe_plan(M, K, sum(splits), 0)["engine"] == want
            outs = _run_both(hsp, x, w_cat, splits)
            check_close(outs, oracle_outputs(x, w_cat, splits), "bf16", f"reg_path {reg_path} K{K} M{M}")
    finally:
        hsp.set_options(pdl=True, reg_path=0)


@pytest.mark.parametrize("K,splits", [(7168, (128, 64)), (6144, (256,)), (1536, (200, 56)), (4096, (5000,))])
@pytest.mark.parametrize("reg_path", [0, 1, 2])
def test_fp32_register_gemv_and_streaming_match_oracle(hsp, K, splits, reg_path):
    """fp32: the register GEMV kernel (default while the tokens fit one CTA; rows in
    blocks of two, all of K per CTA, 5000 rows = 33 or more rows per CTA exercises the
    block loop; forced with reg_path 2, tokens past what one CTA holds go in groups
    along grid.y, the last one ragged: M = 7 at K = 7168 is 4 + 3, M = 17 is 6 + 6 + 5,
    M = 40 at K = 6144 is 8 x 5) and the streaming kernel (reg_path 1) all meet the
    fp32 tolerance, fused and separate."""
    hsp.set_options(pdl=True, reg_path=reg_path)
    try:
        for M in (1, 3, 4, 7, 8, 17, 40, 64):
            x, ws = W.random_case(K, splits, M, "fp32", seed=1700 + M + K)
            w_cat = torch.cat(ws, 0)
            plan = hsp.describe_plan(M, K, sum(splits), 1)
            cap = min(8, 192 * 1024 // (K * 4))
            gemv = reg_path == 2 or (reg_path == 0 and M <= cap)
            assert plan["engine"] == (3 if gemv else 0)
            if gemv:
                assert plan["token_tiles"] == -(-M // cap)
            outs = _run_both(hsp, x, w_cat, splits)
            check_close(outs, oracle_outputs(x, w_cat, splits), "fp32", f"reg_path {reg_path} K{K} M{M}")
    finally:
        hsp.set_options(pdl=True, reg_path=0)


@pytest.mark.parametrize("name", ["indexer_fp32", "glm_router_fp32"])
@pytest.mark.parametrize("forced", [1, 2])
def test_tf32_engines_match_oracle(hsp, name, forced):
    """PROJ_TF32 runs the streaming mma.sync kernel by default (large_m_path 1 too);
    large_m_path 2 takes the tensor-memory kernel (kind::tf32, sixteen K slices of these
    long fp32 rows).  Both meet the tf32 tolerance at the workload's full size, fused
    and separate."""
    wl = W.WORKLOADS[name]
    w_cat = W.weight_cat(wl)
    hsp.set_options(pdl=True, large_m_path=forced)
    try:
        for M in (1, 5, 16, 40, 64):
            assert hsp.describe_plan(M, wl.K, wl.n_total, 2)["engine"] == (0 if forced == 1 else 1)
            x = W.activation(wl, M, 5)
            outs = _run_both(hsp, x, w_cat, wl.splits, tf32=True)
            check_close(outs, oracle_outputs(x, w_cat, wl.splits), "tf32", f"{name} engine {forced} M{M}")
    finally:
        hsp.set_options(pdl=True, large_m_path=0)


@pytest.mark.parametrize("K,splits,dtype,tf32,forced", [
    (4100, (40, 24), "fp32", False, 0),     # 16400-byte rows: bulk copies, 8 K slices at M > 8
    (2056, (17, 47), "fp32", True, 0),      # tf32, 4 K slices
    (1544, (200, 100), "bf16", False, 1),   # bf16 forced onto the streaming kernel, 2 K slices
])
def test_ragged_k_with_k_slices(hsp, K, splits, dtype, tf32, forced):
    """Rows that are not a whole number of 128-byte units take the bulk-copy layout; with
    more than 8 tokens they are also cut into K slices whose partials meet through
    cluster shared memory.  Every M bucket against the oracle, fused and separate."""
    dt = {"bf16": 0, "fp32": 2 if tf32 else 1}[dtype]
    hsp.set_options(pdl=True, large_m_path=forced)
    try:
        for M in (9, 20, 33, 64):
            plan = hsp.describe_plan(M, K, sum(splits), dt)
            assert plan["engine"] == 0 and plan["tensor_copies"] == 0 and plan["slices"] > 1, plan
            x, ws = W.random_case(K, splits, M, dtype, seed=2100 + M + K)
            w_cat = torch.cat(ws, 0)
            outs = _run_both(hsp, x, w_cat, splits, tf32)
            check_close(outs, oracle_outputs(x, w_cat, splits), mode_of(dtype, tf32), f"ragged K{K} M{M}")
    finally:
        hsp.set_options(pdl=True, large_m_path=0)
