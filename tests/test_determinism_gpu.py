"""Bitwise reproducibility of the CUDA path, its launch counting and its bounded waits.

TensorRT-LLM PR #20636, Test Coverage: which path runs is checked by counting
launches; CUDA-graph capture and replay of the fused call must be bitwise equal
to eager execution over three new inputs.  Here also: repeated runs, PDL on vs
off, and the timeout path of the in-kernel waits (a stage that is never loaded
makes the consumers' bounded waits run out; the host reads PROJ_ERR_TIMEOUT and
the context stays usable).
"""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

# register ring (wq_a_wkv), tensor memory with 64- and 128-row tiles (qk_indexer 64 / 32),
# streaming bf16 / fp32 / tf32 (glm_fused_a 5, indexer 16, indexer 64 tf32), fp32 GEMV
# (indexer 4, router 1)
CFGS = [("wq_a_wkv_m1", 1, False), ("wq_a_wkv", 8, False), ("qk_indexer", 64, False),
        ("qk_indexer", 32, False), ("glm_fused_a", 5, False), ("indexer_fp32", 16, False),
        ("indexer_fp32", 64, True), ("indexer_fp32", 4, False), ("glm_router_fp32", 1, False)]


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    yield m
    m.set_options(pdl=True, wait_limit_us=0, skip_stage=None)


def _inputs(name, M, copy):
    wl = W.WORKLOADS[name]
    return wl, W.activation(wl, M, copy).cuda(), W.weight_cat(wl).cuda()


@pytest.mark.parametrize("name,M,tf32", CFGS)
def test_repeat_runs_bitwise(hsp, name, M, tf32):
    wl, x, w = _inputs(name, M, 0)
    first = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)
    for _ in range(3):
        again = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)
        assert all(torch.equal(a, b) for a, b in zip(first, again))
    hsp.check_device_error()


@pytest.mark.parametrize("name,M,tf32", CFGS)
def test_pdl_on_off_bitwise(hsp, name, M, tf32):
    wl, x, w = _inputs(name, M, 1)
    hsp.set_options(pdl=True)
    a = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)
    hsp.set_options(pdl=False)
    b = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)
    hsp.set_options(pdl=True)
    assert all(torch.equal(p, q) for p, q in zip(a, b))


@pytest.mark.parametrize("name,M,tf32", CFGS)
def test_trigger_order_bitwise(hsp, name, M, tf32):
    """The trigger_early option moves only the dependent-launch trigger: same bits."""
    wl, x, w = _inputs(name, M, 3)
    a = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)
    hsp.set_options(pdl=True, trigger_early=True)
    try:
        b = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)
        c = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)   # after an early-triggering call
    finally:
        hsp.set_options(pdl=True, trigger_early=False)
    hsp.check_device_error()
    assert all(torch.equal(p, q) and torch.equal(p, r) for p, q, r in zip(a, b, c))


@pytest.mark.parametrize("separate", [False, True])
@pytest.mark.parametrize("name,M,tf32", CFGS)
def test_graph_replay_matches_eager(hsp, name, M, tf32, separate):
    wl, x0, w = _inputs(name, M, 2)
    fn = hsp.separate_gemm if separate else hsp.fused_gemm
    x_static = x0.clone()
    outs = [torch.empty((M, n), dtype=x0.dtype, device="cuda") for n in wl.splits]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(x_static, w, wl.splits, outs=outs, tf32=tf32, stream=s)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(x_static, w, wl.splits, outs=outs, tf32=tf32)
    for copy in (3, 4, 5):                      # three new inputs
        xn = W.activation(wl, M, copy).cuda()
        x_static.copy_(xn)
        g.replay()
        torch.cuda.synchronize()
        eager = fn(xn, w, wl.splits, tf32=tf32)
        assert all(torch.equal(a, b) for a, b in zip(outs, eager)), copy
    hsp.check_device_error()


@pytest.mark.parametrize("reg_path,M", [(0, 4), (2, 7), (2, 17)])
def test_register_gemv_token_bits_do_not_depend_on_the_group(hsp, reg_path, M):
    """The register GEMV adds each (row, token) over all of K in one CTA, by a reduction
    tree that does not depend on how many tokens the CTA holds: every token of a call
    with M tokens (reg_path 2: in groups of up to 6 at K = 7168) has the bits of a call
    with that token alone."""
    wl, x, w = _inputs("indexer_fp32", M, 2)
    hsp.set_options(pdl=True, reg_path=reg_path)
    try:
        assert hsp.describe_plan(M, wl.K, wl.n_total, 1)["engine"] == 3
        full = hsp.fused_gemm(x, w, wl.splits)
        for t in range(M):
            one = hsp.fused_gemm(x[t:t + 1].contiguous(), w, wl.splits)
            for a, b in zip(full, one):
                assert torch.equal(a[t:t + 1], b), (M, t)
        hsp.check_device_error()
    finally:
        hsp.set_options(pdl=True, reg_path=0)


def test_launch_counting(hsp):
    wl, x, w = _inputs("qk_indexer", 8, 0)
    n0 = hsp.launch_count()
    hsp.fused_gemm(x, w, wl.splits)
    assert hsp.launch_count() == n0 + 1
    hsp.separate_gemm(x, w, wl.splits)
    assert hsp.launch_count() == n0 + 1 + len(wl.splits)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,M", [("wq_a_wkv_m1", 1), ("qk_indexer", 8), ("qk_indexer", 64), ("indexer_fp32", 1),
                                    ("indexer_fp32", 64)])
def test_bounded_wait_reports_timeout(hsp, name, M):
    import hidden_state_projection_gb300 as m
    wl, x, w = _inputs(name, M, 0)
    good = hsp.fused_gemm(x, w, wl.splits)
    hsp.check_device_error()
    # Stage 0 is never loaded: every consumer's wait on it runs out after 20 ms.
    hsp.set_options(pdl=True, wait_limit_us=20000, skip_stage=0)
    try:
        hsp.fused_gemm(x, w, wl.splits)
        with pytest.raises(m.ProjError) as ei:
            hsp.check_device_error()
        assert ei.value.status_name == "PROJ_ERR_TIMEOUT"
    finally:
        hsp.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    # The context is still usable and the next call is correct.
    again = hsp.fused_gemm(x, w, wl.splits)
    hsp.check_device_error()
    assert all(torch.equal(a, b) for a, b in zip(good, again))


@pytest.mark.parametrize("name,M,tf32", CFGS)
def test_prefetch_variant_is_bitwise_equal(hsp, name, M, tf32):
    wl, x, w = _inputs(name, M, 3)
    other = W.weight_cat(wl, 1).cuda()
    a = hsp.fused_gemm(x, w, wl.splits, tf32=tf32)
    b = hsp.fused_gemm_prefetch(x, w, wl.splits, [other, x], tf32=tf32)
    hsp.check_device_error()
    assert all(torch.equal(p, q) for p, q in zip(a, b))
