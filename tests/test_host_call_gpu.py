"""proj_fused_gemm_host through the C ABI: tokens from pinned host memory (the staging
kernel) or pageable memory (a copy-engine copy), outputs back to host memory, the
projection in between bitwise that of proj_fused_gemm; a bound call (HostCall) repeated
over several inputs; NULL host pointers refused before anything is enqueued."""
import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True)
    return m


@pytest.mark.parametrize("name,M,tf32", [("wq_a_wkv", 8, False), ("wq_a_wkv_m1", 1, False), ("qk_indexer", 64, False),
                                         ("indexer_fp32", 4, False), ("indexer_fp32", 4, True)])
def test_host_call_matches_device_call(hsp, name, M, tf32):
    wl = W.WORKLOADS[name]
    w = W.weight_cat(wl).cuda()
    x_dev = torch.empty((M, wl.K), dtype=w.dtype, device="cuda")
    outs_dev = [torch.empty((M, n), dtype=w.dtype, device="cuda") for n in wl.splits]
    outs_host = [torch.full((M, n), float("nan"), dtype=w.dtype).pin_memory() for n in wl.splits]
    xs = [W.activation(wl, M, c).pin_memory() for c in range(3)]
    calls = [hsp.HostCall(xh, w, wl.splits, outs_host, x_dev, outs_dev, tf32=tf32) for xh in xs]
    for rep in range(2):                      # every bound call twice, in a row
        for xh, call in zip(xs, calls):
            before = hsp.launch_count()
            call()
            torch.cuda.synchronize()
            assert hsp.launch_count() == before + 2      # token staging kernel + projection
            assert torch.equal(x_dev.cpu(), xh)          # the staged tokens, bit for bit
            ref = hsp.fused_gemm(xh.cuda(), w, wl.splits, tf32=tf32)
            hsp.check_device_error()
            for h, r in zip(outs_host, ref):
                assert torch.equal(h, r.cpu()), (name, M, rep)


def test_host_call_with_ragged_mapped_outputs(hsp):
    """Mapped outputs whose sizes are not whole 16-byte chunks (a 1 x 1022-byte split) are
    stored by the projection straight into host memory: two launches, same bits."""
    K, splits, M = 5120, (1280, 511), 1
    x, ws = W.random_case(K, splits, M, "bf16", seed=6100)
    w = torch.cat(ws, 0).cuda()
    x_dev = torch.empty((M, K), dtype=w.dtype, device="cuda")
    outs_dev = [torch.empty((M, n), dtype=w.dtype, device="cuda") for n in splits]
    outs_host = [torch.full((M, n), float("nan"), dtype=w.dtype).pin_memory() for n in splits]
    call = hsp.HostCall(x.pin_memory(), w, splits, outs_host, x_dev, outs_dev)
    before = hsp.launch_count()
    call()
    torch.cuda.synchronize()
    assert hsp.launch_count() == before + 2
    ref = hsp.fused_gemm(x.cuda(), w, splits)
    hsp.check_device_error()
    for h, r in zip(outs_host, ref):
        assert torch.equal(h, r.cpu())


@pytest.mark.parametrize("name,M", [("wq_a_wkv", 8), ("indexer_fp32", 64)])
def test_host_call_with_pageable_tokens(hsp, name, M):
    """Tokens in pageable memory go through a copy-engine copy; outputs in pageable memory
    come back through the device staging buffers and copies."""
    wl = W.WORKLOADS[name]
    w = W.weight_cat(wl).cuda()
    x_dev = torch.full((M, wl.K), float("nan"), dtype=w.dtype, device="cuda")
    outs_dev = [torch.empty((M, n), dtype=w.dtype, device="cuda") for n in wl.splits]
    for pinned_out in (False, True):
        outs_host = [torch.full((M, n), float("nan"), dtype=w.dtype) for n in wl.splits]
        if pinned_out:
            outs_host = [o.pin_memory() for o in outs_host]
        xh = W.activation(wl, M, 1)
        assert not xh.is_pinned()
        before = hsp.launch_count()
        hsp.HostCall(xh, w, wl.splits, outs_host, x_dev, outs_dev)()
        torch.cuda.synchronize()
        assert hsp.launch_count() == before + 1          # the projection only
        assert torch.equal(x_dev.cpu(), xh)
        ref = hsp.fused_gemm(xh.cuda(), w, wl.splits)
        hsp.check_device_error()
        for h, r in zip(outs_host, ref):
            assert torch.equal(h, r.cpu()), (name, M, pinned_out)


def test_host_call_refuses_null_host_pointers(hsp):
    S = hsp.STATUS
    lib = hsp.lib()
    x_dev = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((24, 64), dtype=torch.bfloat16, device="cuda")
    outs_dev = [torch.zeros((1, 16), dtype=torch.bfloat16, device="cuda"),
                torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda")]
    host = [torch.zeros((1, 16), dtype=torch.bfloat16).pin_memory(), torch.zeros((1, 8), dtype=torch.bfloat16).pin_memory()]
    ns = (ctypes.c_int32 * 2)(16, 8)
    od = (ctypes.c_void_p * 2)(*[o.data_ptr() for o in outs_dev])
    oh = (ctypes.c_void_p * 2)(host[0].data_ptr(), None)
    xh = torch.zeros((1, 64), dtype=torch.bfloat16).pin_memory()
    before = hsp.launch_count()
    assert lib.proj_fused_gemm_host(None, w.data_ptr(), ns, 2, oh, 1, 64, 0, x_dev.data_ptr(), od, None) == \
        S["PROJ_ERR_INVALID_ARG"]
    assert lib.proj_fused_gemm_host(xh.data_ptr(), w.data_ptr(), ns, 2, oh, 1, 64, 0, x_dev.data_ptr(), od, None) == \
        S["PROJ_ERR_INVALID_ARG"]
    assert b"outs_host[1]" in lib.proj_last_error_string()
    assert hsp.launch_count() == before


@pytest.mark.parametrize("name,M", [("wq_a_wkv", 8), ("qk_indexer", 64), ("indexer_fp32", 4)])
def test_host_plan_replays_match_device_call(hsp, name, M):
    """A host plan (one recorded graph per bound step) gives the bits of fused_gemm on
    every launch; two plans over the same staging buffers interleave correctly."""
    wl = W.WORKLOADS[name]
    ws = [W.weight_cat(wl, c).cuda() for c in range(2)]
    x_dev = torch.empty((M, wl.K), dtype=ws[0].dtype, device="cuda")
    outs_dev = [torch.empty((M, n), dtype=ws[0].dtype, device="cuda") for n in wl.splits]
    outs_host = [torch.full((M, n), float("nan"), dtype=ws[0].dtype).pin_memory() for n in wl.splits]
    xs = [W.activation(wl, M, c).pin_memory() for c in range(2)]
    plans = [hsp.HostPlan(xs[c], ws[c], wl.splits, outs_host, x_dev, outs_dev) for c in range(2)]
    try:
        for rep in range(3):
            for c in (0, 1):
                plans[c]()
                torch.cuda.synchronize()
                ref = hsp.fused_gemm(xs[c].cuda(), ws[c], wl.splits)
                hsp.check_device_error()
                for h, r in zip(outs_host, ref):
                    assert torch.equal(h, r.cpu()), (name, M, rep, c)
    finally:
        for p in plans:
            p.close()


def test_host_plan_argument_checks(hsp):
    S = hsp.STATUS
    lib = hsp.lib()
    assert lib.proj_host_plan_launch(None, None) == S["PROJ_ERR_INVALID_ARG"]
    assert lib.proj_host_plan_destroy(None) == 0
    x_dev = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((24, 64), dtype=torch.bfloat16, device="cuda")
    ns = (ctypes.c_int32 * 2)(16, 8)
    od = (ctypes.c_void_p * 2)(*[torch.zeros((1, n), dtype=torch.bfloat16, device="cuda").data_ptr() for n in (16, 8)])
    oh = (ctypes.c_void_p * 2)(None, None)
    h = ctypes.c_void_p()
    assert lib.proj_host_plan_create(None, w.data_ptr(), ns, 2, oh, 1, 64, 0, x_dev.data_ptr(), od,
                                     ctypes.byref(h)) == S["PROJ_ERR_INVALID_ARG"]
    assert not h.value


def test_host_plan_as_the_first_call_of_a_process():
    """A plan recorded before anything else ran in the process (the library's per-device
    set-up and first kernel configuration happen while the graph is being recorded)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = r'''
import sys, torch
sys.path.insert(0, %r)
import workloads as W
import hidden_state_projection_gb300 as hsp
wl = W.WORKLOADS["wq_a_wkv"]
M = 8
w = W.weight_cat(wl).cuda()
x_dev = torch.empty((M, wl.K), dtype=w.dtype, device="cuda")
outs_dev = [torch.empty((M, n), dtype=w.dtype, device="cuda") for n in wl.splits]
outs_host = [torch.zeros((M, n), dtype=w.dtype).pin_memory() for n in wl.splits]
xh = W.activation(wl, M).pin_memory()
plan = hsp.HostPlan(xh, w, wl.splits, outs_host, x_dev, outs_dev)
plan(); plan()
torch.cuda.synchronize()
ref = hsp.fused_gemm(xh.cuda(), w, wl.splits)
assert all(torch.equal(h, r.cpu()) for h, r in zip(outs_host, ref))
plan.close()
print("ok")
''' % root
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
