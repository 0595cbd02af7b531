"""Calls from several host threads at once, each on its own stream.

The library keeps per-process state that concurrent callers share: the per-device set-up,
the tensor-map cache, the launch counter and the per-thread error text.  Four threads,
each on its own CUDA stream and its own engine (register ring, streaming, tensor memory,
register GEMV), repeat their fused call while the others run; every result must have the
bits of the same call made alone, and no thread may see another's error or a refused call.
"""
import threading

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

JOBS = [("wq_a_wkv", 4), ("qk_indexer", 8), ("qk_indexer", 64), ("indexer_fp32", 4)]
REPEATS = 40


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True)
    return m


def test_threads_on_their_own_streams_match_serial_calls(hsp):
    inputs, expect = [], []
    for k, (name, M) in enumerate(JOBS):
        wl = W.WORKLOADS[name]
        x, w = W.activation(wl, M, 30 + k).cuda(), W.weight_cat(wl).cuda()
        inputs.append((wl, x, w))
        expect.append([o.clone() for o in hsp.fused_gemm(x, w, wl.splits)])
    torch.cuda.synchronize()
    hsp.check_device_error()

    errors = []
    barrier = threading.Barrier(len(JOBS))

    def run(k):
        try:
            wl, x, w = inputs[k]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                barrier.wait()
                for _ in range(REPEATS):
                    outs = hsp.fused_gemm(x, w, wl.splits)
                    stream.synchronize()
                    for got, ref in zip(outs, expect[k]):
                        if not torch.equal(got, ref):
                            errors.append((JOBS[k], "bits differ"))
                            return
        except Exception as e:  # noqa: BLE001 -- reported below with the job
            errors.append((JOBS[k], repr(e)))

    threads = [threading.Thread(target=run, args=(k,)) for k in range(len(JOBS))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
    hsp.check_device_error()
