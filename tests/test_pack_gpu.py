"""The weight packer on the GPU, through the C ABI (proj_pack_weights, proj_pack_check).

TensorRT-LLM PR #20636, Description: after loading, the projection weights that read
the same hidden state are copied into one row-concatenated tensor and the
per-projection weights are rebound as views of it; a checkpoint reload then writes
through the views, and a parameter replaced by a new tensor is no longer a view.
Test Coverage of the same page lists weight aliasing, the reload writing through the
views and the fallback for a replaced parameter.  Checked here for every workload:

  * the packed W_cat is byte for byte the row concatenation of the separate weights;
  * a fused call on it matches the oracle run on the separate weights (concatenated
    on the host);
  * packing other weights into the same W_cat (a reload) changes the next fused call's
    outputs to the oracle's for the new weights;
  * every view passes proj_pack_check, a replaced tensor does not;
  * parts that already are their own rows of W_cat are skipped: all of them, no launch;
    some of them, one launch that leaves those rows alone.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import check_close, mode_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True, wait_limit_us=0, skip_stage=None)
    return m


def _oracle(x, parts, splits):
    """Oracle outputs for tokens x and separate weights `parts` (concatenated here, on the host)."""
    dt = oracle.BF16 if x.dtype == torch.bfloat16 else oracle.FP32
    w_bits = np.concatenate([W.to_numpy_bits(p) for p in parts], axis=0)
    outs = oracle.fused(W.to_numpy_bits(x), w_bits, splits, dt, threads=8)
    return [W.from_numpy_bits(o).to(torch.float64).numpy() for o in outs]


PACK_CASES = [("wq_a_wkv", 8), ("indexer_fp32", 4), ("qk_indexer", 1), ("glm_fused_a_2784", 4)]


@pytest.mark.parametrize("name,M", PACK_CASES)
def test_pack_then_reload(hsp, name, M):
    wl = W.WORKLOADS[name]
    dev = torch.device("cuda")
    parts = W.weight_parts(wl)
    ws = [p.to(dev) for p in parts]
    before = hsp.launch_count()
    w_cat, views = hsp.pack_weights(ws)
    torch.cuda.synchronize()
    assert hsp.launch_count() == before + 1                    # one copy kernel for all parts
    assert torch.equal(w_cat.cpu().view(torch.uint8), torch.cat(parts, 0).view(torch.uint8))
    for i, v in enumerate(views):
        assert hsp.pack_check(v, w_cat, sum(wl.splits[:i]))
    mode = mode_of(wl.dtype, False)
    x = W.activation(wl, M)
    outs = hsp.fused_gemm(x.to(dev), w_cat, wl.splits)
    hsp.check_device_error()
    check_close(outs, _oracle(x, parts, wl.splits), mode, f"{name} packed")

    # reload: other weights packed into the same W_cat; the next call sees them
    new_parts = W.weight_parts(wl, copy=7)
    hsp.pack_weights([p.to(dev) for p in new_parts], w_cat=w_cat)
    outs = hsp.fused_gemm(x.to(dev), w_cat, wl.splits)
    hsp.check_device_error()
    assert torch.equal(w_cat.cpu().view(torch.uint8), torch.cat(new_parts, 0).view(torch.uint8))
    check_close(outs, _oracle(x, new_parts, wl.splits), mode, f"{name} reloaded")

    # a reload written through the views needs no pack: the views are skipped
    for v, p in zip(views, parts):
        v.copy_(p.to(dev))
    n0 = hsp.launch_count()
    hsp.pack_weights(views, w_cat=w_cat)
    assert hsp.launch_count() == n0
    outs = hsp.fused_gemm(x.to(dev), w_cat, wl.splits)
    hsp.check_device_error()
    check_close(outs, _oracle(x, parts, wl.splits), mode, f"{name} written through the views")

    # a parameter replaced by a new tensor is no longer a view
    replaced = views[0].clone()
    assert not hsp.pack_check(replaced, w_cat, 0)
    assert not hsp.pack_check(views[-1], w_cat, 0)              # right tensor, wrong rows


def test_pack_skips_parts_already_in_place(hsp):
    """One part already is its own rows of W_cat (holding a marker), the other is a new
    tensor: one launch, the marker rows stay as they were and the new part's rows are
    copied."""
    dev = torch.device("cuda")
    K, splits = 512, (48, 80)
    _, parts = W.random_case(K, splits, 1, "bf16", seed=77)
    w_cat = torch.empty((sum(splits), K), dtype=torch.bfloat16, device=dev)
    w_cat[:48] = 3.0
    n0 = hsp.launch_count()
    hsp.pack_weights([w_cat[:48], parts[1].to(dev)], w_cat=w_cat)
    torch.cuda.synchronize()
    assert hsp.launch_count() == n0 + 1
    assert bool((w_cat[:48] == 3.0).all())
    assert torch.equal(w_cat[48:].cpu(), parts[1])


def test_pack_ragged_parts_and_empty_part(hsp):
    """Parts of 1, 0, 17 and 130 rows at a K of 8 bf16 (16-byte rows): the chunk-to-part
    lookup at every boundary, and a part with no rows."""
    dev = torch.device("cuda")
    K, rows = 8, (1, 0, 17, 130)
    g = torch.Generator().manual_seed(5)
    parts = [torch.randn(n, K, generator=g).to(torch.bfloat16) for n in rows]
    w_cat, views = hsp.pack_weights([p.to(dev) if p.numel() else torch.empty(0, K, dtype=torch.bfloat16, device=dev)
                                     for p in parts])
    assert torch.equal(w_cat.cpu().view(torch.int16), torch.cat(parts, 0).view(torch.int16))
    assert [v.shape[0] for v in views] == list(rows)


def test_pack_refuses_overlap_on_device_tensors(hsp):
    """A source that overlaps W_cat other than as its own rows is refused and nothing runs."""
    dev = torch.device("cuda")
    w_cat = torch.zeros((56, 64), dtype=torch.bfloat16, device=dev)
    n0 = hsp.launch_count()
    with pytest.raises(hsp.ProjError) as e:                     # rows 8..40 are not part 0's rows 0..32
        hsp.pack_weights([w_cat[8:40], torch.ones((24, 64), dtype=torch.bfloat16, device=dev)], w_cat=w_cat)
    assert e.value.status_name == "PROJ_ERR_INVALID_ARG"
    assert hsp.launch_count() == n0
    assert int(torch.count_nonzero(w_cat)) == 0
