"""proj_fused_gemm_rmsnorm_static, the RMSNorm-epilogue call that allocates nothing.

Callers that cannot hand the library a workspace -- an inference runtime that owns all
device memory through its own pool and forbids side allocations, a plugin that is
given only the tensors of one operation, a latency-critical path that cannot afford
cudaMalloc's implicit synchronisation -- use this entry point: its workspace is a
fixed 1 MiB array compiled into the library.  Checked here, through the C ABI:

  * two calls in a row give exactly the bits of proj_fused_gemm_rmsnorm (same kernel,
    same workspace layout, a workspace of our own there), and both are within the
    bf16 tolerance of the oracle's fp64 RMSNorm;
  * a call launches one kernel and leaves the device's free memory where it was;
  * a call whose bounded wait runs out (the test hook that leaves a stage unloaded)
    reports PROJ_ERR_TIMEOUT, and the next static calls are correct again (the
    timed-out call left the array's counters at zero);
  * the documented pattern -- one eager call, then stream capture -- replays the
    kernel with the eager call's bits;
  * a shape whose workspace exceeds the array is refused before anything runs.

This file is collected last.
"""
import ctypes

import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import check_close

pytestmark = pytest.mark.gpu

EPS = 1e-6
CASES = [("wq_a_wkv", 8, (1280, 512)), ("qk_indexer", 1, (1536, 512, 0, 0))]


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
    return [None if c == 0 else (1.0 + 0.1 * torch.randn(c, generator=g)).to(torch.bfloat16).cuda()
            for c in norm_cols]


def _static_call(hsp, x, w, splits, norm_cols, gammas, outs, stream=None):
    i32 = ctypes.c_int32
    ns = (i32 * len(splits))(*splits)
    nc = (i32 * len(splits))(*norm_cols)
    gp = (ctypes.c_void_p * len(splits))(*[g.data_ptr() if g is not None else None for g in gammas])
    po = (ctypes.c_void_p * len(splits))(*[o.data_ptr() for o in outs])
    st = (stream or torch.cuda.current_stream()).cuda_stream
    return hsp.lib().proj_fused_gemm_rmsnorm_static(x.data_ptr(), w.data_ptr(), ns, len(splits), nc, gp,
                                                    ctypes.c_float(EPS), po, x.shape[0], x.shape[1], 0, st)


def _nan_outs(M, splits):
    return [torch.full((M, n), float("nan"), dtype=torch.bfloat16, device="cuda") for n in splits]


def _oracle(x, w, splits, norm_cols, gammas):
    ref = oracle.fused_rmsnorm(W.to_numpy_bits(x), W.to_numpy_bits(w), splits, norm_cols,
                               [None if g is None else W.to_numpy_bits(g) for g in gammas], EPS, oracle.BF16)
    return [W.from_numpy_bits(r).to(torch.float64).numpy() for r in ref]


@pytest.mark.parametrize("name,M,norm_cols", CASES)
def test_static_workspace_matches_caller_workspace(hsp, name, M, norm_cols):
    wl = W.WORKLOADS[name]
    w = W.weight_cat(wl).cuda()
    gammas = _gammas(norm_cols, 21)
    ws = torch.zeros(hsp.rmsnorm_workspace_bytes(M, wl.K, wl.splits, norm_cols), dtype=torch.uint8, device="cuda")
    for call in range(2):                                   # two calls in a row on the shared array
        x = W.activation(wl, M, call).cuda()
        ref = hsp.fused_gemm_rmsnorm(x, w, wl.splits, norm_cols, gammas, EPS, ws)
        outs = _nan_outs(M, wl.splits)
        assert _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs) == 0, hsp.lib().proj_last_error_string()
        hsp.check_device_error()
        for o, r in zip(outs, ref):
            assert torch.equal(o, r), (name, M, call)
        check_close(outs, _oracle(x.cpu(), w.cpu(), wl.splits, norm_cols, gammas), "bf16", f"{name} M{M} static")


def test_static_call_allocates_nothing(hsp):
    wl, M, norm_cols = W.WORKLOADS["wq_a_wkv"], 4, (1280, 512)
    x, w = W.activation(wl, M).cuda(), W.weight_cat(wl).cuda()
    gammas = _gammas(norm_cols, 5)
    outs = _nan_outs(M, wl.splits)
    assert _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs) == 0   # modules loaded, address looked up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    n0 = hsp.launch_count()
    for _ in range(3):
        assert _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs) == 0
    torch.cuda.synchronize()
    assert hsp.launch_count() == n0 + 3                     # one kernel per call, nothing else of ours
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_reserved() == reserved0
    hsp.check_device_error()


def test_static_call_after_a_timeout(hsp):
    """Every CTA's token copy is left out by the test hook: the bounded waits run out,
    the call reports PROJ_ERR_TIMEOUT through the device error word, and the next
    static calls give the caller-workspace bits (every CTA still arrived, so the
    timed-out call left the counters at zero)."""
    import hidden_state_projection_gb300 as m
    wl, M, norm_cols = W.WORKLOADS["wq_a_wkv"], 8, (1280, 512)
    x, w = W.activation(wl, M, 3).cuda(), W.weight_cat(wl).cuda()
    gammas = _gammas(norm_cols, 9)
    ws = torch.zeros(hsp.rmsnorm_workspace_bytes(M, wl.K, wl.splits, norm_cols), dtype=torch.uint8, device="cuda")
    ref = hsp.fused_gemm_rmsnorm(x, w, wl.splits, norm_cols, gammas, EPS, ws)
    hsp.check_device_error()
    hsp.set_options(pdl=True, wait_limit_us=20000, skip_stage=0)
    try:
        outs = _nan_outs(M, wl.splits)
        assert _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs) == 0
        with pytest.raises(m.ProjError) as ei:
            hsp.check_device_error()
        assert ei.value.status_name == "PROJ_ERR_TIMEOUT"
    finally:
        hsp.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    for _ in range(2):
        outs = _nan_outs(M, wl.splits)
        assert _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs) == 0
        hsp.check_device_error()
        assert all(torch.equal(o, r) for o, r in zip(outs, ref))


def test_static_call_captured_after_an_eager_call(hsp):
    """One eager call first (it looks up the array's address), then the call captured
    on a side stream: each replay runs the kernel, with the bits of the eager call on
    the same tokens."""
    wl, M, norm_cols = W.WORKLOADS["wq_a_wkv"], 8, (1280, 512)
    w = W.weight_cat(wl).cuda()
    gammas = _gammas(norm_cols, 13)
    x_static = W.activation(wl, M, 4).cuda()
    outs = _nan_outs(M, wl.splits)
    assert _static_call(hsp, x_static, w, wl.splits, norm_cols, gammas, outs) == 0
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        rc = _static_call(hsp, x_static, w, wl.splits, norm_cols, gammas, outs, stream=s)
    assert rc == 0, hsp.lib().proj_last_error_string()
    for copy in (5, 6):
        xn = W.activation(wl, M, copy).cuda()
        x_static.copy_(xn)
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        eager = _nan_outs(M, wl.splits)
        assert _static_call(hsp, xn, w, wl.splits, norm_cols, gammas, eager) == 0
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(outs, eager)), copy
    hsp.check_device_error()


def test_static_workspace_refuses_shapes_past_its_size(hsp):
    splits, norm_cols, M, K = (20000, 20000), (20000, 20000), 8, 64
    need = hsp.rmsnorm_workspace_bytes(M, K, splits, norm_cols)
    assert need > (1 << 20)
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(sum(splits), K, dtype=torch.bfloat16, device="cuda")
    gammas = [torch.ones(n, dtype=torch.bfloat16, device="cuda") for n in splits]
    outs = [torch.zeros(M, n, dtype=torch.bfloat16, device="cuda") for n in splits]
    before = hsp.launch_count()
    rc = _static_call(hsp, x, w, splits, norm_cols, gammas, outs)
    assert hsp.STATUS_NAMES[rc] == "PROJ_ERR_UNSUPPORTED_SHAPE"
    msg = hsp.lib().proj_last_error_string().decode()
    assert str(need) in msg and str(1 << 20) in msg, msg
    assert hsp.launch_count() == before
    assert all(int(torch.count_nonzero(o)) == 0 for o in outs)


def _captured_nodes(fn, stream):
    """Nodes of the graph that stream capture (relaxed mode) records around fn()."""
    import os
    rt = ctypes.CDLL(os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcudart.so"))
    sp = ctypes.c_void_p(stream.cuda_stream)
    assert rt.cudaStreamBeginCapture(sp, ctypes.c_int(2)) == 0           # cudaStreamCaptureModeRelaxed
    try:
        rc = fn()
    finally:
        graph = ctypes.c_void_p()
        end = rt.cudaStreamEndCapture(sp, ctypes.byref(graph))
    assert end == 0
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    rt.cudaGraphDestroy(graph)
    return rc, n.value


def test_static_call_refuses_bad_arguments_and_enqueues_nothing(hsp):
    """Argument errors found after the size check (a NULL gamma) are refused like the
    caller-workspace call's, and the refused call enqueues nothing: captured, it
    records no node, where an accepted call records exactly one (its kernel; nothing
    is cleared per call)."""
    wl, M, norm_cols = W.WORKLOADS["wq_a_wkv"], 2, (1280, 512)
    x, w = W.activation(wl, M).cuda(), W.weight_cat(wl).cuda()
    gammas = _gammas(norm_cols, 17)
    outs = _nan_outs(M, wl.splits)
    assert _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs) == 0   # address looked up, eagerly
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    before = hsp.launch_count()
    rc, nodes = _captured_nodes(lambda: _static_call(hsp, x, w, wl.splits, norm_cols, [None, None], outs, s), s)
    assert hsp.STATUS_NAMES[rc] == "PROJ_ERR_INVALID_ARG"
    assert nodes == 0
    assert hsp.launch_count() == before
    rc, nodes = _captured_nodes(lambda: _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs, s), s)
    assert rc == 0 and nodes == 1
