"""proj_fused_gemm_rmsnorm_static, the RMSNorm-epilogue call that allocates nothing.

Callers that cannot hand the library a workspace -- an inference runtime that owns all
device memory through its own pool and forbids side allocations, a plugin that is
given only the tensors of one operation, a latency-critical path that cannot afford
cudaMalloc's implicit synchronisation -- use this entry point: its workspace is a
fixed 1 MiB array compiled into the library.  Checked here, through the C ABI: two
calls in a row give the outputs of proj_fused_gemm_rmsnorm (with a workspace of our
own) within the bf16 tolerance of the other tests, and a shape whose workspace
exceeds the array is refused before anything runs.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import BF16_ATOL, BF16_RTOL

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    return m


def _static_call(hsp, x, w, splits, norm_cols, gammas, outs):
    i32 = ctypes.c_int32
    ns = (i32 * len(splits))(*splits)
    nc = (i32 * len(splits))(*norm_cols)
    gp = (ctypes.c_void_p * len(splits))(*[g.data_ptr() if g is not None else None for g in gammas])
    po = (ctypes.c_void_p * len(splits))(*[o.data_ptr() for o in outs])
    stream = torch.cuda.current_stream().cuda_stream
    return hsp.lib().proj_fused_gemm_rmsnorm_static(x.data_ptr(), w.data_ptr(), ns, len(splits), nc, gp,
                                                    ctypes.c_float(EPS), po, x.shape[0], x.shape[1], 0, stream)


@pytest.mark.parametrize("name,M,norm_cols", [("wq_a_wkv", 8, (1280, 512)), ("qk_indexer", 1, (1536, 512, 0, 0))])
def test_static_workspace_matches_caller_workspace(hsp, name, M, norm_cols):
    wl = W.WORKLOADS[name]
    w = W.weight_cat(wl).cuda()
    g = torch.Generator().manual_seed(21)
    gammas = [None if c == 0 else (1.0 + 0.1 * torch.randn(c, generator=g)).to(torch.bfloat16).cuda()
              for c in norm_cols]
    ws = torch.zeros(hsp.rmsnorm_workspace_bytes(M, wl.K, wl.splits, norm_cols), dtype=torch.uint8, device="cuda")
    for call in range(2):                                   # two calls in a row on the shared array
        x = W.activation(wl, M, call).cuda()
        ref = hsp.fused_gemm_rmsnorm(x, w, wl.splits, norm_cols, gammas, EPS, ws)
        outs = [torch.full((M, n), float("nan"), dtype=torch.bfloat16, device="cuda") for n in wl.splits]
        assert _static_call(hsp, x, w, wl.splits, norm_cols, gammas, outs) == 0, hsp.lib().proj_last_error_string()
        hsp.check_device_error()
        for o, r in zip(outs, ref):
            a, b = o.double().cpu().numpy(), r.double().cpu().numpy()
            assert np.all(np.isfinite(a))
            assert np.all(np.abs(a - b) <= BF16_ATOL + BF16_RTOL * np.abs(b)), (name, M, call)


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
