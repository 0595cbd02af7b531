"""Programmatic-dependent-launch ordering: the completion trigger follows the stores.

TensorRT-LLM PR #20636, Description and Test Coverage: tinygemm2 triggers its
dependents before its output stores; that is safe only for consumers that wait with
griddepcontrol.wait, and the page's stress test of the pattern (20,000 replays per
case, 0 mismatches) had no positive control.  Here, in a CUDA graph, every replay:

    poison the outputs (NaN) -> projection (PDL launch) -> consumer (PDL launch)

and the consumer counts outputs that differ from an eagerly computed reference at the
moment it reads them.  With the library's order (release fence in every storing
thread, then the trigger) a consumer that does not wait must see no mismatch in
20,000 replays.  Positive control: the test hook that triggers at kernel start (the
tinygemm2 order) must let the same non-waiting consumer see mismatches -- otherwise
the test could not detect the hazard -- while a waiting consumer stays clean.
"""
import ctypes
import os
import subprocess

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
REPLAYS = 20000
PER_GRAPH = 100


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True)
    yield m
    m.set_options(pdl=True, trigger_early=False)


@pytest.fixture(scope="module")
def consumer():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libpdl_consumer.so")
    src = os.path.join(HERE, "csrc", "pdl_consumer.cu")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                        "-Xcompiler", "-fPIC", src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.pdl_consumer_launch.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_void_p]
    lib.pdl_consumer_launch.restype = ctypes.c_int
    return lib


def _stress(hsp, consumer, name, M, separate, wait, early, replays=REPLAYS):
    wl = W.WORKLOADS[name]
    x = W.activation(wl, M).cuda()
    w = W.weight_cat(wl).cuda()
    total = M * wl.n_total
    dt = x.dtype                             # bf16, or fp32 for the indexer / router
    assert (total * x.element_size()) % 4 == 0
    flat = torch.empty(total, dtype=dt, device="cuda")
    views, off = [], 0
    for n in wl.splits:                      # dense [M, N_i] outputs inside one buffer
        views.append(flat[off:off + M * n].view(M, n))
        off += M * n
    fn = hsp.separate_gemm if separate else hsp.fused_gemm
    ref = torch.cat([o.reshape(-1) for o in hsp.fused_gemm(x, w, wl.splits)])
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    n_words = total * x.element_size() // 4
    hsp.set_options(pdl=True, trigger_early=early)
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn(x, w, wl.splits, outs=views, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            stream = torch.cuda.current_stream().cuda_stream
            for _ in range(PER_GRAPH):
                flat.view(torch.int32).fill_(-1)          # all ones: NaN in bf16 and fp32
                fn(x, w, wl.splits, outs=views)
                rc = consumer.pdl_consumer_launch(flat.data_ptr(), ref.data_ptr(), n_words, int(wait),
                                                  counter.data_ptr(), stream)
                assert rc == 0
        for _ in range(replays // PER_GRAPH):
            g.replay()
        torch.cuda.synchronize()
        hsp.check_device_error()
    finally:
        hsp.set_options(pdl=True, trigger_early=False)
    # after the last replay the outputs themselves are final and correct
    assert torch.equal(flat, ref)
    return int(counter.item())


# one case per engine: the register ring (wq_a++wkv), the streaming ring (qk_indexer M = 8),
# the tensor-memory kernel (qk_indexer M = 64), the fp32 register GEMV (indexer fp32 M = 4),
# the streaming kernel's fp32 FMA path (indexer fp32 M = 64)
CASES = [("wq_a_wkv_m1", 1, False), ("wq_a_wkv", 8, False), ("wq_a_wkv", 4, True), ("qk_indexer", 8, False),
         ("qk_indexer", 64, False), ("indexer_fp32", 4, False), ("indexer_fp32", 64, False)]


@pytest.mark.parametrize("name,M,separate", CASES)
def test_trigger_after_stores_needs_no_wait(hsp, consumer, name, M, separate):
    assert _stress(hsp, consumer, name, M, separate, wait=False, early=False) == 0


@pytest.mark.parametrize("name,M,separate", CASES[:2])
def test_waiting_consumer_is_always_safe(hsp, consumer, name, M, separate):
    assert _stress(hsp, consumer, name, M, separate, wait=True, early=False, replays=2000) == 0
    assert _stress(hsp, consumer, name, M, separate, wait=True, early=True, replays=2000) == 0


@pytest.mark.parametrize("name,M,separate", CASES[:2])
def test_positive_control_early_trigger_is_detected(hsp, consumer, name, M, separate):
    # The early trigger lets a consumer that does not wait read the outputs before the
    # projection stores them: the test must see it, or it could not see the hazard.
    assert _stress(hsp, consumer, name, M, separate, wait=False, early=True, replays=2000) > 0
