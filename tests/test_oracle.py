"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test is chosen so that a plausible mistake in the oracle fails it:
  - exact integer brute force (dropped term, wrong index, transposed operand,
    wrong split offset);
  - one-hot activations (column indexing, which operand is which);
  - linearity in X (a non-linear slip such as squaring or abs);
  - the concatenation invariant (fused == per-projection calls);
  - a float64 library matmul (a summation bug that integers would not show);
  - brute-force nearest-value search for the bf16 rounding (tie rule,
    subnormals, overflow, double rounding through fp32);
  - hand-derived golden values (tests/golden/).
"""
import bisect
import json
import os
import re
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return W.to_numpy_bits(t)


def _bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- rounding

_BF16_TABLE = None


def _all_bf16_finite_sorted():
    """Every non-negative finite bf16 value (decoded by torch), sorted, with its bits."""
    global _BF16_TABLE
    if _BF16_TABLE is None:
        bits = np.arange(0, 0x7F80, dtype=np.int64)  # +0 .. largest finite
        vals = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        order = np.argsort(vals, kind="stable")
        _BF16_TABLE = ([Fraction(float(v)) for v in vals[order]], bits[order])
    return _BF16_TABLE


def _nearest_bf16_bruteforce(v: float) -> int:
    """Nearest representable value by search; ties -> even fraction; past the
    largest finite, 2^128 plays the role of the next value (infinity)."""
    vals, bits = _all_bf16_finite_sorted()
    sign = 0x8000 if np.signbit(v) else 0
    a = Fraction(abs(v))
    cand_vals = vals + [Fraction(2) ** 128]
    cand_bits = list(bits) + [0x7F80]
    i = bisect.bisect_left(cand_vals, a)
    if i < len(cand_vals) and cand_vals[i] == a:
        return sign | int(cand_bits[i])
    if i >= len(cand_vals):
        return sign | 0x7F80
    lo, hi = i - 1, i
    dlo, dhi = a - cand_vals[lo], cand_vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if (int(cand_bits[lo]) & 1) == 0 else hi
    return sign | int(cand_bits[pick])


def test_bf16_rounding_against_bruteforce_search(oracle_mod):
    rng = np.random.default_rng(1)
    values = []
    # random magnitudes over the whole range, including subnormals
    values += list(rng.standard_normal(300) * np.exp2(rng.integers(-140, 128, 300)))
    # exact midpoints between neighbours and one fp64 ulp either side
    vals, _ = _all_bf16_finite_sorted()
    for i in rng.integers(0, len(vals) - 1, 300):
        mid = float((vals[i] + vals[i + 1]) / 2)
        values += [mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)]
    values += [0.0, -0.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 2.0 ** -126,
               float(vals[-1]), 2.0 ** 128 - 2.0 ** 119, np.nextafter(2.0 ** 128 - 2.0 ** 119, 0),
               1e300, -1e300, 1e-300]
    for v in values:
        v = float(v)
        got = oracle_mod.double_to_bf16(v)
        want = _nearest_bf16_bruteforce(v)
        assert got == want, f"{v!r}: oracle {got:#06x} brute force {want:#06x}"


def test_bf16_rounding_matches_library_on_fp32_values(oracle_mod):
    # For values that are exactly fp32, torch's fp32 -> bf16 cast is a single RNE.
    rng = np.random.default_rng(2)
    f = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    f = np.concatenate([f, np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875], np.float32)])
    lib = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.round_out(f.astype(np.float64), oracle_mod.BF16)
    assert np.array_equal(got, lib)


def test_fp32_rounding_matches_library(oracle_mod):
    rng = np.random.default_rng(3)
    d = rng.standard_normal(5000) * np.exp2(rng.integers(-100, 100, 5000))
    assert np.array_equal(oracle_mod.round_out(d, oracle_mod.FP32), d.astype(np.float32))


def _pow2_expr(s: str) -> float:
    """Exact value of "1", "-1", "2^a", "2^a - 2^b" (terms are integers or powers of two)."""
    total = Fraction(0)
    for sign, term in re.findall(r"([+-]?)\s*(2\^-?\d+|\d+)", s):
        val = Fraction(2) ** int(term[2:]) if term.startswith("2^") else Fraction(int(term))
        total += -val if sign == "-" else val
    return float(total)


def test_golden_rounding_cases(oracle_mod):
    """Hand-derived bit patterns at rounding boundaries, bf16 and fp32 outputs: ties to
    even in both directions, no double rounding, signs, subnormals, overflow."""
    cases = json.load(open(os.path.join(GOLDEN, "rounding_cases.json")))["cases"]
    assert sum(c.get("dtype", "bf16") == "fp32" for c in cases) >= 6
    for c in cases:
        fp32 = c.get("dtype", "bf16") == "fp32"
        x = torch.tensor([[_pow2_expr(s) for s in c["x"]]], dtype=torch.float64)
        w = torch.tensor([[_pow2_expr(s) for s in c["w"]]], dtype=torch.float64)
        tdt = torch.float32 if fp32 else torch.bfloat16
        xb, wb = x.to(tdt), w.to(tdt)
        # the inputs must be exact in the dtype for the case to mean what it says
        assert torch.equal(xb.to(torch.float64), x) and torch.equal(wb.to(torch.float64), w), c["name"]
        (out,) = oracle_mod.fused(_bits(xb), _bits(wb), [1], oracle_mod.FP32 if fp32 else oracle_mod.BF16)
        got = int(np.asarray(out).view(np.uint32)[0, 0]) if fp32 else int(out[0, 0])
        assert got == int(c["expect_bits"], 16), (c["name"], hex(got))


# ---------------------------------------------------------------- closed forms

def _formula(expr: str, m, n, k):
    return {"1": np.ones_like(k), "k": k, "(-1)^k": np.where(k % 2 == 0, 1, -1),
            "m+1": m + 1 + 0 * k, "n+1": n + 1 + 0 * k}[expr]


def test_golden_closed_forms(oracle_mod):
    cases = json.load(open(os.path.join(GOLDEN, "closed_forms.json")))["cases"]
    for c in cases:
        M, K, rows = c["M"], c["K"], c["rows"]
        N = sum(rows)
        mm = np.arange(M)[:, None]
        kk = np.arange(K)[None, :]
        nn = np.arange(N)[:, None]
        x = np.broadcast_to(_formula(c["x"], mm, 0, kk), (M, K)).astype(np.float64)
        w = np.broadcast_to(_formula(c["w"], 0, nn, kk), (N, K)).astype(np.float64)
        tdt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
        xt, wt = torch.from_numpy(x).to(tdt), torch.from_numpy(w).to(tdt)
        assert torch.equal(xt.double(), torch.from_numpy(x)), c["name"]
        assert torch.equal(wt.double(), torch.from_numpy(w)), c["name"]
        dt = oracle_mod.BF16 if c["dtype"] == "bf16" else oracle_mod.FP32
        outs = oracle_mod.fused(_bits(xt), _bits(wt), rows, dt)
        got = np.concatenate([_bf16_bits_to_float(o) if dt == oracle_mod.BF16 else o.astype(np.float64)
                              for o in outs], axis=1)
        exp = c["expect"]
        if "all" in exp:
            want = np.full((M, N), float(exp["all"]))
        else:
            want = np.array([[eval(exp["per_mn"], {}, {"m": m, "n": n}) for n in range(N)]
                             for m in range(M)], dtype=np.float64)
        assert np.array_equal(got, want), c["name"]


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("M,K,splits", [(1, 8, (1,)), (2, 64, (3, 16)), (3, 72, (17, 1, 3)),
                                         (8, 64, (16, 17)), (5, 40, (2, 2, 2, 2))])
def test_integer_bruteforce_exact(oracle_mod, dtype, M, K, splits):
    x, ws = W.small_int_case(K, splits, M, dtype, seed=11 + M + K)
    dt = oracle_mod.BF16 if dtype == "bf16" else oracle_mod.FP32
    wcat = torch.cat(ws, 0)
    outs = oracle_mod.fused(_bits(x), _bits(wcat), splits, dt)
    xi = [[int(v) for v in row] for row in x.to(torch.float64).tolist()]
    for i, (wi, oi) in enumerate(zip(ws, outs)):
        wl = [[int(v) for v in row] for row in wi.to(torch.float64).tolist()]
        got = _bf16_bits_to_float(oi) if dt == oracle_mod.BF16 else oi.astype(np.float64)
        for m in range(M):
            for n in range(len(wl)):
                want = sum(xi[m][k] * wl[n][k] for k in range(K))   # exact integers
                assert abs(want) <= 256 or dtype == "fp32"
                assert got[m, n] == want, (i, m, n)


def test_one_hot_reproduces_weight_columns(oracle_mod):
    K, splits = 520, (33, 7)
    for dtype, dt in (("bf16", oracle_mod.BF16), ("fp32", oracle_mod.FP32)):
        _, ws = W.random_case(K, splits, 1, dtype, seed=77)
        wcat = torch.cat(ws, 0)
        cols = [0, 1, 63, 64, 255, 256, K - 2, K - 1]
        x = torch.zeros(len(cols), K, dtype=wcat.dtype)
        for m, c in enumerate(cols):
            x[m, c] = 1
        outs = oracle_mod.fused(_bits(x), _bits(wcat), splits, dt)
        for wi, oi in zip(ws, outs):
            for m, c in enumerate(cols):
                assert np.array_equal(oi[m], _bits(wi[:, c].contiguous())), (dtype, c)


def test_linearity_in_x(oracle_mod):
    rng = np.random.default_rng(5)
    K, N, M = 1000, 40, 3
    # multiples of 2^-8 in [-4, 4]: 3*x1 - 2*x2 stays exact in fp32
    x1 = (rng.integers(-1024, 1025, (M, K)) / 256.0).astype(np.float32)
    x2 = (rng.integers(-1024, 1025, (M, K)) / 256.0).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x3 = (3 * x1.astype(np.float64) - 2 * x2.astype(np.float64)).astype(np.float32)
    assert np.array_equal(x3.astype(np.float64), 3 * x1.astype(np.float64) - 2 * x2.astype(np.float64))
    y1 = oracle_mod.accumulate(x1, w, oracle_mod.FP32)
    y2 = oracle_mod.accumulate(x2, w, oracle_mod.FP32)
    y3 = oracle_mod.accumulate(x3, w, oracle_mod.FP32)
    scale = np.abs(x3.astype(np.float64)) @ np.abs(w.astype(np.float64)).T
    assert np.all(np.abs(y3 - (3 * y1 - 2 * y2)) <= 1e-12 * scale)


def test_concatenation_invariant_and_separate(oracle_mod):
    wl = W.WORKLOADS["qk_indexer"]
    x, ws = W.random_case(wl.K, wl.splits, 3, "bf16", seed=123)
    wcat = torch.cat(ws, 0)
    fused = oracle_mod.fused(_bits(x), _bits(wcat), wl.splits, oracle_mod.BF16, threads=4)
    sep = oracle_mod.separate(_bits(x), _bits(wcat), wl.splits, oracle_mod.BF16)
    for i, wi in enumerate(ws):
        (alone,) = oracle_mod.fused(_bits(x), _bits(wi), [wi.shape[0]], oracle_mod.BF16)
        assert np.array_equal(fused[i], alone)
        assert np.array_equal(sep[i], alone)


def test_against_float64_library_matmul(oracle_mod):
    for dtype, dt in (("bf16", oracle_mod.BF16), ("fp32", oracle_mod.FP32)):
        x, ws = W.random_case(7168, (128, 64), 4, dtype, seed=9)
        wcat = torch.cat(ws, 0)
        y = oracle_mod.accumulate(_bits(x), _bits(wcat), dt)
        ref = (x.double() @ wcat.double().T).numpy()
        scale = (x.double().abs() @ wcat.double().abs().T).numpy()
        assert np.all(np.abs(y - ref) <= 1e-13 * scale)
        outs = oracle_mod.fused(_bits(x), _bits(wcat), (128, 64), dt)
        got = np.concatenate([_bf16_bits_to_float(o) if dt == oracle_mod.BF16 else o.astype(np.float64)
                              for o in outs], 1)
        tgt = torch.from_numpy(ref).to(torch.bfloat16 if dtype == "bf16" else torch.float32).double().numpy()
        # torch's fp64 -> bf16 goes through fp32 (double rounding): rare 1-ulp disagreements only
        assert np.mean(got != tgt) < 1e-3
        ulp = np.abs(tgt) * (2.0 ** -7 if dtype == "bf16" else 2.0 ** -23)
        assert np.all(np.abs(got - tgt) <= ulp)


def test_zero_weights_and_sign_symmetry(oracle_mod):
    x, ws = W.random_case(512, (24, 8), 5, "bf16", seed=31)
    wcat = torch.cat(ws, 0)
    z = oracle_mod.fused(_bits(x), _bits(torch.zeros_like(wcat)), (24, 8), oracle_mod.BF16)
    assert all(np.all(o == 0) for o in z)
    pos = oracle_mod.fused(_bits(x), _bits(wcat), (24, 8), oracle_mod.BF16)
    neg = oracle_mod.fused(_bits(-x), _bits(wcat), (24, 8), oracle_mod.BF16)
    for p, q in zip(pos, neg):
        nz = (p & 0x7FFF) != 0
        assert np.array_equal(p[nz] ^ 0x8000, q[nz])


def test_thread_count_does_not_change_result(oracle_mod):
    wl = W.WORKLOADS["wq_a_wkv"]
    x, ws = W.random_case(wl.K, (300, 45), 2, "bf16", seed=4)
    wcat = torch.cat(ws, 0)
    a = oracle_mod.fused(_bits(x), _bits(wcat), (300, 45), oracle_mod.BF16, threads=1)
    b = oracle_mod.fused(_bits(x), _bits(wcat), (300, 45), oracle_mod.BF16, threads=7)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))


def test_pins_reject_planted_mistakes(oracle_mod):
    """The integer brute force must tell a right projection from plausible wrong
    ones (dropped term, wrong split offset, reversed k of one operand)."""
    x, ws = W.small_int_case(16, (3, 5), 2, "fp32", seed=5)
    wcat = torch.cat(ws, 0).double()
    xd = x.double()
    exact = np.array([[sum(int(xd[m, k]) * int(wcat[n, k]) for k in range(16)) for n in range(8)]
                      for m in range(2)], dtype=np.float64)
    dropped = (xd[:, 1:] @ wcat[:, 1:].T).numpy()
    shifted = np.roll((xd @ wcat.T).numpy(), 1, axis=1)
    flipped = (xd @ wcat.flip(1).T).numpy()
    for wrong in (dropped, shifted, flipped):
        assert not np.array_equal(wrong, exact)
    good = np.concatenate([o.astype(np.float64) for o in
                           oracle_mod.fused(_bits(x), _bits(torch.cat(ws, 0)), (3, 5), oracle_mod.FP32)], 1)
    assert np.array_equal(good, exact)


# ---------------------------------------------------------------- RMSNorm epilogue

def _f32(a):
    return np.asarray(a, dtype=np.float32)


def test_rmsnorm_golden_closed_forms(oracle_mod):
    with open(os.path.join(GOLDEN, "rmsnorm_closed_forms.json")) as f:
        spec = json.load(f)
    x = _f32([[1.0, 1.0]])
    w = _f32([[3.0, 0.0], [0.0, 4.0]])
    for case in spec["cases"]:
        (out,) = oracle_mod.fused_rmsnorm(x, w, (2,), (2,), [_f32(case["gamma"])], case["eps"], oracle_mod.FP32)
        if "expect_sqrt2_times" in case:
            exact = [c * np.sqrt(np.float64(2.0)) for c in case["expect_sqrt2_times"]]
        else:
            exact = [c / np.sqrt(np.float64(13.0)) for c in case["expect_over_sqrt13"]]
        assert np.array_equal(out[0], _f32(exact)), (case["name"], out[0], exact)


def test_rmsnorm_unit_mean_square(oracle_mod):
    """gamma = 1, eps = 0: every token's normalized columns have mean square 1."""
    x, ws = W.random_case(512, (96, 40), 3, "fp32", seed=31)
    wcat = torch.cat(ws, 0)
    g = [np.ones(96, np.float32), np.ones(24, np.float32)]
    a, b = oracle_mod.fused_rmsnorm(_bits(x), _bits(wcat), (96, 40), (96, 24), g, 0.0, oracle_mod.FP32)
    for out, c in ((a, 96), (b, 24)):
        ms = np.mean(out[:, :c].astype(np.float64) ** 2, axis=1)
        assert np.allclose(ms, 1.0, rtol=0, atol=1e-6), ms


def test_rmsnorm_scale_invariance_and_gamma_linearity(oracle_mod):
    """eps = 0: doubling x leaves the normalized columns unchanged bit for bit and
    doubles the others; doubling gamma doubles the normalized columns."""
    x, ws = W.random_case(256, (48, 20), 2, "bf16", seed=32)
    wcat = torch.cat(ws, 0)
    gam = torch.randn(48, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    g1 = [_bits(gam), None]
    g2 = [_bits(gam * 2), None]
    base = oracle_mod.fused_rmsnorm(_bits(x), _bits(wcat), (48, 20), (48, 0), g1, 0.0, oracle_mod.BF16)
    twice_x = oracle_mod.fused_rmsnorm(_bits(x * 2), _bits(wcat), (48, 20), (48, 0), g1, 0.0, oracle_mod.BF16)
    twice_g = oracle_mod.fused_rmsnorm(_bits(x), _bits(wcat), (48, 20), (48, 0), g2, 0.0, oracle_mod.BF16)
    assert np.array_equal(base[0], twice_x[0])
    assert np.array_equal(_bf16_bits_to_float(twice_x[1]), 2 * _bf16_bits_to_float(base[1]))
    assert np.array_equal(_bf16_bits_to_float(twice_g[0]), 2 * _bf16_bits_to_float(base[0]))


def test_rmsnorm_leaves_other_columns_as_the_projection(oracle_mod):
    """Columns past norm_cols, and splits with norm_cols 0, are the plain projection."""
    x, ws = W.random_case(576, (64, 36, 16), 4, "bf16", seed=33)
    wcat = torch.cat(ws, 0)
    gam = [_bits(torch.ones(64, dtype=torch.bfloat16)), _bits(torch.ones(32, dtype=torch.bfloat16)), None]
    normed = oracle_mod.fused_rmsnorm(_bits(x), _bits(wcat), (64, 36, 16), (64, 32, 0), gam, 1e-6, oracle_mod.BF16)
    plain = oracle_mod.fused(_bits(x), _bits(wcat), (64, 36, 16), oracle_mod.BF16)
    assert np.array_equal(normed[1][:, 32:], plain[1][:, 32:])
    assert np.array_equal(normed[2], plain[2])
    none = oracle_mod.fused_rmsnorm(_bits(x), _bits(wcat), (64, 36, 16), (0, 0, 0), [None] * 3, 1e-6, oracle_mod.BF16)
    assert all(np.array_equal(p, q) for p, q in zip(none, plain))
    assert not np.array_equal(normed[0], plain[0])


def test_rmsnorm_pins_reject_planted_mistakes(oracle_mod):
    """The closed form tells the right normalization from plausible wrong ones:
    the sum instead of the mean, the norm without the square root, eps outside it."""
    y = np.array([3.0, 4.0])
    right = y / np.sqrt(np.mean(y ** 2) + 0.5)
    for wrong in (y / np.sqrt(np.sum(y ** 2) + 0.5), y / (np.mean(y ** 2) + 0.5),
                  y / (np.sqrt(np.mean(y ** 2)) + 0.5)):
        assert not np.allclose(wrong, right, rtol=1e-3)
    assert np.allclose(right, np.array([3.0, 4.0]) / np.sqrt(13.0), rtol=0, atol=1e-15)
