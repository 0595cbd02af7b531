"""Seeded synthetic workloads for the fused hidden-state projection.

This module only draws numbers and names shapes; it holds none of the
projection's arithmetic.  Both the CPU oracle (through the tests and the
benchmark's CPU leg) and the CUDA library are fed from it, so that the two
sides see the same bytes.

The shapes are those of the projections the pages fuse (the weights themselves
are real checkpoints that are not available here, so every value is drawn):

  wq_a_wkv      TensorRT-LLM PR #20636 (DeepSeek-V4.1 wq_a/wkv via tinygemm2),
                Description: wq_a 5120 -> 1280 and wkv 5120 -> 512, W_cat [1792, 5120].
  indexer_fp32  TensorRT-LLM PR #12055 (indexer wk + weights_proj in one TF32
                GEMM), Description: wk 128 + weights_proj 64 rows, hidden 7168, FP32.
  qk_indexer    TensorRT-LLM PR #8771 (QK down_proj + indexer K + weights_proj),
                Walkthrough: q_a 1536 ++ kv_a 576 ++ indexer wk 128 ++ weights_proj 64.
  glm_fused_a   TensorRT-LLM PR #20502 (GLM-5.2 decode target), glmFusedAGemm
                commit message: hidden 6144, q_a 2048 ++ kv_a 576 ++ indexer wk 128.
  glm_fused_a_2784
                the same commit message's wider cell: 2624 rows (q_a 2048,
                compressed KV 512, k_pe 64) plus the indexer's wk 128 and
                weights_proj 32 rows appended to the same weight, up to 8 tokens.
  glm_router_fp32
                the same page, glmRouterGemm commit message: the router's logits in
                FP32, 256 experts, hidden size 6144, 1-16 tokens.

Recipe: X ~ N(0, 1) and W ~ N(0, 0.02), drawn in fp32 with a CPU
torch.Generator and rounded once to bf16 (torch's round-to-nearest-even) when
the workload is bf16.  Seeds: weight part p of copy c of workload number i uses
1000*i + 100*p + c; the activation of copy c uses 1000*i + 500 + c.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import numpy as np
import torch

BF16 = "bf16"
FP32 = "fp32"


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int                 # 1-based workload number (seed base)
    name: str
    K: int
    splits: Tuple[int, ...]    # rows of each projection, in W_cat order
    split_names: Tuple[str, ...]
    dtype: str                 # element type of x, w and the outputs
    Ms: Tuple[int, ...]        # token counts exercised

    @property
    def n_total(self) -> int:
        return int(sum(self.splits))

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4

    def weight_bytes(self) -> int:
        return self.n_total * self.K * self.elem_bytes

    def algorithmic_bytes(self, M: int) -> int:
        """N*K*w + M*K*x + M*N*y: every weight and activation read once, every output written once."""
        e = self.elem_bytes
        return self.n_total * self.K * e + M * self.K * e + M * self.n_total * e


WORKLOADS = {
    "wq_a_wkv_m1": Workload(1, "wq_a_wkv_m1", 5120, (1280, 512), ("wq_a", "wkv"), BF16, (1,)),
    "wq_a_wkv": Workload(2, "wq_a_wkv", 5120, (1280, 512), ("wq_a", "wkv"), BF16, (2, 4, 8)),
    "indexer_fp32": Workload(3, "indexer_fp32", 7168, (128, 64), ("wk", "weights_proj"), FP32,
                             (1, 4, 16, 64)),
    "qk_indexer": Workload(4, "qk_indexer", 7168, (1536, 576, 128, 64),
                           ("q_a", "kv_a", "idx_wk", "idx_wp"), BF16, (1, 8, 32, 64)),
    "glm_fused_a": Workload(5, "glm_fused_a", 6144, (2048, 576, 128),
                            ("q_a", "kv_a", "idx_wk"), BF16, tuple(range(1, 9))),
    "glm_fused_a_2784": Workload(6, "glm_fused_a_2784", 6144, (2048, 512, 64, 128, 32),
                                 ("q_a", "compressed_kv", "k_pe", "idx_wk", "idx_wp"), BF16, (1, 4, 8)),
    "glm_router_fp32": Workload(7, "glm_router_fp32", 6144, (256,), ("router",), FP32, (1, 4, 16)),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _draw(shape, std: float, seed: int, dtype: str) -> torch.Tensor:
    t = torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        t = t * std
    if dtype == BF16:
        t = t.to(torch.bfloat16)
    return t.contiguous()


def weight_parts(wl: Workload, copy: int = 0) -> List[torch.Tensor]:
    """The separate projection weights W_i [N_i, K] (CPU tensors)."""
    return [_draw((n, wl.K), 0.02, 1000 * wl.index + 100 * p + copy, wl.dtype)
            for p, n in enumerate(wl.splits)]


def weight_cat(wl: Workload, copy: int = 0) -> torch.Tensor:
    """The parts stacked in W_cat row order (a plain concatenation of the drawn bytes)."""
    return torch.cat(weight_parts(wl, copy), dim=0).contiguous()


def activation(wl: Workload, M: int, copy: int = 0) -> torch.Tensor:
    """X [M, K] ~ N(0, 1) in the workload's dtype (CPU tensor)."""
    return _draw((M, wl.K), 1.0, 1000 * wl.index + 500 + copy, wl.dtype)


def random_case(K: int, splits: Sequence[int], M: int, dtype: str, seed: int,
                x_std: float = 1.0, w_std: float = 0.02):
    """A free-form seeded case for tests: (x, [W_i])."""
    x = _draw((M, K), x_std, seed, dtype)
    ws = [_draw((n, K), w_std, seed + 1 + i, dtype) for i, n in enumerate(splits)]
    return x, ws


def small_int_case(K: int, splits: Sequence[int], M: int, dtype: str, seed: int,
                   xmax: int = 2, wmax: int = 3):
    """Small-integer inputs: x in [-xmax, xmax], w in [-wmax, wmax].

    With K small enough every partial sum is an exactly representable integer
    in fp32, and a result of magnitude <= 256 is exact in bf16."""
    g = _gen(seed)
    tdt = torch.bfloat16 if dtype == BF16 else torch.float32
    x = torch.randint(-xmax, xmax + 1, (M, K), generator=g).to(tdt)
    ws = [torch.randint(-wmax, wmax + 1, (n, K), generator=g).to(tdt) for n in splits]
    return x.contiguous(), [w.contiguous() for w in ws]


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensors as uint16 bit patterns, fp32 tensors as float32 arrays."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")


def from_numpy_bits(a: np.ndarray) -> torch.Tensor:
    """Inverse of to_numpy_bits."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32).copy())
