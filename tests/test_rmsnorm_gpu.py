"""The RMSNorm epilogue (q_norm / kv_norm fused into the projection) against the oracle.

TensorRT-LLM PR #20636, Description: the consumers of wq_a / wkv are the q_norm /
kv_norm RMSNorms; PR #20502, glm_mla_kv_half_append commit message: of the kv_a_proj
output only the 512 latent columns are normalised (its 64 RoPE columns are left
alone).  Checked here: every normalized output within the bf16 tolerance of the
oracle's fp64 RMSNorm; the columns and splits left alone bitwise equal to the plain
fused call; two calls in a row and CUDA-graph replay bitwise equal to eager (the
workspace's counters are left at zero by every call); argument checks.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import check_close

pytestmark = pytest.mark.gpu

EPS = 1e-6
CASES = [("wq_a_wkv_m1", 1, (1280, 512)), ("wq_a_wkv", 4, (1280, 512)), ("wq_a_wkv", 8, (1280, 512)),
         ("qk_indexer", 1, (1536, 512, 0, 0)), ("qk_indexer", 8, (1536, 512, 0, 0)),
         ("glm_fused_a", 5, (2048, 512, 0))]


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    return m


def _gammas(norm_cols, seed):
    g = torch.Generator().manual_seed(seed)
    return [None if c == 0 else (1.0 + 0.1 * torch.randn(c, generator=g)).to(torch.bfloat16) for c in norm_cols]


def _run(hsp, x, w, splits, norm_cols, gammas, ws=None, outs=None, stream=None):
    if ws is None:
        ws = torch.zeros(hsp.rmsnorm_workspace_bytes(x.shape[0], x.shape[1], splits, norm_cols), dtype=torch.uint8,
                         device="cuda")
    gd = [None if g is None else g.cuda() for g in gammas]
    return hsp.fused_gemm_rmsnorm(x, w, splits, norm_cols, gd, EPS, ws, outs=outs, stream=stream), ws


@pytest.mark.parametrize("name,M,norm_cols", CASES)
def test_rmsnorm_matches_oracle(hsp, name, M, norm_cols):
    wl = W.WORKLOADS[name]
    x, w = W.activation(wl, M), W.weight_cat(wl)
    gam = _gammas(norm_cols, 100 + M)
    outs, _ = _run(hsp, x.cuda(), w.cuda(), wl.splits, norm_cols, gam)
    hsp.check_device_error()
    ref = oracle.fused_rmsnorm(W.to_numpy_bits(x), W.to_numpy_bits(w), wl.splits, norm_cols,
                               [None if g is None else W.to_numpy_bits(g) for g in gam], EPS, oracle.BF16)
    ref = [W.from_numpy_bits(r).to(torch.float64).numpy() for r in ref]
    check_close(outs, ref, "bf16", f"{name} M{M} rmsnorm")


@pytest.mark.parametrize("name,M,norm_cols", CASES)
def test_rmsnorm_leaves_other_columns_bitwise(hsp, name, M, norm_cols):
    wl = W.WORKLOADS[name]
    x, w = W.activation(wl, M, 1).cuda(), W.weight_cat(wl).cuda()
    outs, _ = _run(hsp, x, w, wl.splits, norm_cols, _gammas(norm_cols, 7))
    plain = hsp.fused_gemm(x, w, wl.splits)
    for o, p, c in zip(outs, plain, norm_cols):
        assert torch.equal(o[:, c:], p[:, c:])
        if c:
            assert not torch.equal(o[:, :c], p[:, :c])


@pytest.mark.parametrize("name,M,norm_cols", [CASES[0], CASES[2], CASES[4]])
def test_rmsnorm_repeat_and_graph_bitwise(hsp, name, M, norm_cols):
    wl = W.WORKLOADS[name]
    w = W.weight_cat(wl).cuda()
    gam = _gammas(norm_cols, 11)
    x0 = W.activation(wl, M, 2).cuda()
    first, ws = _run(hsp, x0, w, wl.splits, norm_cols, gam)
    again, _ = _run(hsp, x0, w, wl.splits, norm_cols, gam, ws=ws)        # the same workspace, next call
    assert all(torch.equal(a, b) for a, b in zip(first, again))
    x_static = x0.clone()
    outs = [torch.empty((M, n), dtype=x0.dtype, device="cuda") for n in wl.splits]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(hsp, x_static, w, wl.splits, norm_cols, gam, ws=ws, outs=outs, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    gd = [None if g is None else g.cuda() for g in gam]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        hsp.fused_gemm_rmsnorm(x_static, w, wl.splits, norm_cols, gd, EPS, ws, outs=outs)
    for copy in (3, 4):
        xn = W.activation(wl, M, copy).cuda()
        x_static.copy_(xn)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        eager, _ = _run(hsp, xn, w, wl.splits, norm_cols, gam)
        assert all(torch.equal(a, b) for a, b in zip(outs, eager)), copy
    hsp.check_device_error()


def test_rmsnorm_argument_checks(hsp):
    wl = W.WORKLOADS["wq_a_wkv"]
    x, w = W.activation(wl, 2).cuda(), W.weight_cat(wl).cuda()
    gam = [g.cuda() for g in _gammas((1280, 512), 3)]
    need = hsp.rmsnorm_workspace_bytes(2, wl.K, wl.splits, (1280, 512))
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(hsp.ProjError) as ei:
        hsp.fused_gemm_rmsnorm(x, w, wl.splits, (1280, 512), gam, EPS, small)
    assert ei.value.status_name == "PROJ_ERR_INVALID_ARG"
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(hsp.ProjError) as ei:
        hsp.fused_gemm_rmsnorm(x, w, wl.splits, (1281, 512), gam, EPS, ws)
    assert ei.value.status_name == "PROJ_ERR_INVALID_ARG"
    with pytest.raises(hsp.ProjError) as ei:
        hsp.fused_gemm_rmsnorm(x, w, wl.splits, (1280, 512), gam, -1.0, ws)
    assert ei.value.status_name == "PROJ_ERR_INVALID_ARG"
    x9 = W.activation(wl, 9).cuda()
    with pytest.raises(hsp.ProjError) as ei:
        hsp.fused_gemm_rmsnorm(x9, w, wl.splits, (1280, 512), gam, EPS, ws)
    assert ei.value.status_name == "PROJ_ERR_UNSUPPORTED_SHAPE"
    xf, wf = x.float(), w.float()
    with pytest.raises(hsp.ProjError) as ei:
        hsp.fused_gemm_rmsnorm(xf, wf, wl.splits, (1280, 512), [g.float() for g in gam], EPS, ws)
    assert ei.value.status_name == "PROJ_ERR_UNSUPPORTED_DTYPE"
    # a failed check launches nothing and leaves the workspace usable
    outs = hsp.fused_gemm_rmsnorm(x, w, wl.splits, (1280, 512), gam, EPS, ws)
    hsp.check_device_error()
    assert all(torch.isfinite(o.float()).all() for o in outs)


@pytest.mark.parametrize("name,M,norm_cols", [CASES[2], CASES[4]])
def test_rmsnorm_workspace_reusable_after_timeout(hsp, name, M, norm_cols):
    """A call whose waits run out (the test hook leaves one stage unloaded in every CTA)
    reports PROJ_ERR_TIMEOUT; every CTA still arrives on its split's counter, so the
    same workspace, not zeroed again, gives the bits of a fresh workspace next."""
    import hidden_state_projection_gb300 as m
    wl = W.WORKLOADS[name]
    x, w = W.activation(wl, M, 6).cuda(), W.weight_cat(wl).cuda()
    gam = _gammas(norm_cols, 19)
    fresh, _ = _run(hsp, x, w, wl.splits, norm_cols, gam)
    hsp.check_device_error()
    ws = torch.zeros(hsp.rmsnorm_workspace_bytes(M, wl.K, wl.splits, norm_cols), dtype=torch.uint8, device="cuda")
    hsp.set_options(pdl=True, wait_limit_us=20000, skip_stage=0)
    try:
        _run(hsp, x, w, wl.splits, norm_cols, gam, ws=ws)
        with pytest.raises(m.ProjError) as ei:
            hsp.check_device_error()
        assert ei.value.status_name == "PROJ_ERR_TIMEOUT"
    finally:
        hsp.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    assert int(torch.count_nonzero(ws[:256])) == 0          # counters and abort flags back at zero
    for _ in range(2):
        again, _ = _run(hsp, x, w, wl.splits, norm_cols, gam, ws=ws)
        hsp.check_device_error()
        assert all(torch.equal(a, b) for a, b in zip(again, fresh))
