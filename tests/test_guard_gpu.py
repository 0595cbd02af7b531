"""No kernel writes outside its outputs: every output [M, N_i] sits in the middle of a
larger buffer whose bytes before and after it hold a sentinel pattern, and after the call
(fused and separate) the sentinels must be intact while the outputs equal those of a
plain call.  One case per engine and layout, at ragged shapes (rows not a multiple of the
tile, a one-row split, token counts between tiles)."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

PAD = 4096  # elements of sentinel before and after each output


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True)
    return m


def _guarded(M, splits, dtype):
    """Outputs as views into sentinel-filled buffers; returns (outs, buffers)."""
    bufs, outs = [], []
    for n in splits:
        b = torch.empty(PAD + M * n + PAD, dtype=dtype, device="cuda")
        bits = b.view(torch.int16) if dtype == torch.bfloat16 else b.view(torch.int32)
        bits.fill_(0x5A5A if dtype == torch.bfloat16 else 0x5A5A5A5A)
        bufs.append(b)
        outs.append(b[PAD:PAD + M * n].view(M, n))
    return outs, bufs


def _sentinels_intact(bufs, M, splits):
    for b, n in zip(bufs, splits):
        bits = b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)
        want = 0x5A5A if b.dtype == torch.bfloat16 else 0x5A5A5A5A
        head, tail = bits[:PAD], bits[PAD + M * n:]
        assert bool((head == want).all()) and bool((tail == want).all()), f"write outside a [{M}, {n}] output"


# (K, splits, M, dtype, tf32, options): register ring, fp32 GEMV (one group and token
# groups), streaming ring (bf16, fp32 FMA, tf32; tensor and bulk copy layouts),
# tensor-memory kernel (128- and 64-row tiles, 8 and 2 K slices)
CASES = [
    (5120, (1280, 511, 1), 5, "bf16", False, {}),
    (7168, (128, 63, 1), 3, "fp32", False, {}),
    (7168, (128, 63, 1), 17, "fp32", False, {"reg_path": 2}),
    (7168, (1536, 575, 1), 7, "bf16", False, {}),
    (5112, (700, 13), 6, "bf16", False, {}),
    (7168, (128, 63, 1), 40, "fp32", False, {}),
    (7168, (128, 63, 1), 9, "fp32", True, {}),
    (7168, (1536, 575, 1), 23, "bf16", False, {}),
    (7168, (1536, 575, 1), 50, "bf16", False, {}),
    (1536, (200, 55, 1), 64, "bf16", False, {}),
]


@pytest.mark.parametrize("K,splits,M,dtype,tf32,opt", CASES)
def test_no_write_outside_the_outputs(hsp, K, splits, M, dtype, tf32, opt):
    x, ws = W.random_case(K, splits, M, dtype, seed=4242 + K + M)
    x, w = x.cuda(), torch.cat(ws, 0).cuda()
    hsp.set_options(pdl=True, **opt)
    try:
        ref = hsp.fused_gemm(x, w, splits, tf32=tf32)
        for fn in (hsp.fused_gemm, hsp.separate_gemm):
            outs, bufs = _guarded(M, splits, w.dtype)
            fn(x, w, splits, outs=outs, tf32=tf32)
            hsp.check_device_error()
            torch.cuda.synchronize()
            _sentinels_intact(bufs, M, splits)
            for o, r in zip(outs, ref):
                assert torch.equal(o, r)
    finally:
        hsp.set_options(pdl=True)


def test_host_call_writes_only_its_buffers(hsp):
    """The host entry point: the device staging buffer and the pinned host outputs sit
    inside sentinel-filled buffers too."""
    K, splits, M = 5120, (1280, 511, 1), 5
    x, ws = W.random_case(K, splits, M, "bf16", seed=4343)
    w = torch.cat(ws, 0).cuda()
    xbuf = torch.empty(PAD + M * K + PAD, dtype=torch.bfloat16, device="cuda")
    xbuf.view(torch.int16).fill_(0x5A5A)
    x_dev = xbuf[PAD:PAD + M * K].view(M, K)
    outs_dev, dbufs = _guarded(M, splits, torch.bfloat16)
    hbufs = [torch.empty(PAD + M * n + PAD, dtype=torch.bfloat16).pin_memory() for n in splits]
    for b in hbufs:
        b.view(torch.int16).fill_(0x5A5A)
    outs_host = [b[PAD:PAD + M * n].view(M, n) for b, n in zip(hbufs, splits)]
    hsp.HostCall(x.pin_memory(), w, splits, outs_host, x_dev, outs_dev)()
    torch.cuda.synchronize()
    bits = xbuf.view(torch.int16)
    assert bool((bits[:PAD] == 0x5A5A).all()) and bool((bits[PAD + M * K:] == 0x5A5A).all())
    assert torch.equal(x_dev.cpu(), x)
    _sentinels_intact(dbufs, M, splits)      # outputs went straight to the pinned host buffers
    _sentinels_intact(hbufs, M, splits)
    ref = hsp.fused_gemm(x.cuda(), w, splits)
    for h, r in zip(outs_host, ref):
        assert torch.equal(h, r.cpu())
