"""The tf32 tensor-core path's operand rounding, bit for bit.

PROJ_TF32 on the streaming kernel rounds both mma.sync operands to tf32 (cvt.rna: round
to nearest, ties away from zero, on the 10-bit mantissa; the tensor-memory kernel's
kind::tf32 instead ignores the low mantissa bits).  With an identity weight matrix every
output is one token value times 1.0 plus exact zeros, so each output is that value's
tf32 rounding, which must equal the rule written out here on the host: ties away from
zero at bit 12 of the fp32 pattern, denormals included, and infinity past the largest
finite tf32 value.  The sum starts from +0, so a -0 input gives +0.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

K = 64


def rna_tf32_bits(bits: np.ndarray) -> np.ndarray:
    """Round fp32 bit patterns to tf32 (10 explicit mantissa bits), ties away from zero."""
    b = bits.astype(np.uint64)
    mag = b & 0x7FFFFFFF
    sign = b & 0x80000000
    # a finite magnitude rounds up when its 13 low bits are at least half of bit 13's weight
    low = mag & 0x1FFF
    up = (mag >> 13) + (low >= 0x1000)
    out = sign | ((up << 13) & 0xFFFFFFFF)
    special = (mag & 0x7F800000) == 0x7F800000
    return np.where(special, b, out).astype(np.uint32)


def _cases(seed: int) -> np.ndarray:
    one = 0x3F800000
    edge = [
        one | 0x1000,            # 1 + 2^-11: a tie, away from zero -> 1 + 2^-10
        one | 0x0FFF,            # just below the tie -> 1
        one | 0x1001,            # just above -> 1 + 2^-10
        0x80000000 | one | 0x1000,  # -(1 + 2^-11) -> -(1 + 2^-10)
        one | 0x3000,            # 1 + 3 * 2^-11: a tie above an odd mantissa -> 1 + 2^-9
        0x3FFFF000,              # 1.99951...: rounds up into the next binade -> 2.0
        0x00001000,              # a denormal tie -> 0x00002000
        0x00000FFF,              # a denormal below the tie -> 0
        0x80001000,              # its negative
        0x7F7FE000,              # already a tf32 value
        0x7F7FEFFF,              # below the tie under the largest tf32 value
        0x00000000, 0x80000000,  # zeros
    ]
    rng = np.random.default_rng(seed)
    rest = rng.integers(0, 1 << 32, size=4 * K - len(edge), dtype=np.uint64).astype(np.uint32)
    rest = rest[(rest & 0x7F800000) != 0x7F800000][: 4 * K - len(edge)]   # finite only
    rest = np.concatenate([rest, np.full(4 * K - len(edge) - rest.size, one, np.uint32)])
    return np.concatenate([np.array(edge, np.uint32), rest]).reshape(4, K)


@pytest.fixture(scope="module")
def hsp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import hidden_state_projection_gb300 as m
    m.lib()
    m.set_options(pdl=True)
    return m


def _outputs(hsp, x_bits: np.ndarray) -> np.ndarray:
    # tf32 at these token counts runs the streaming mma.sync kernel unless forced elsewhere
    M = x_bits.shape[0]
    assert hsp.describe_plan(M, K, K, 2)["engine"] == 0
    x = torch.from_numpy(x_bits.view(np.float32).copy()).cuda()
    w = torch.eye(K, dtype=torch.float32, device="cuda")
    (y,) = hsp.fused_gemm(x, w, (K,), tf32=True)
    hsp.check_device_error()
    return y.cpu().numpy().view(np.uint32)


def test_tensor_core_operands_round_to_nearest_ties_away(hsp):
    for seed in (1, 2):
        x = _cases(seed)
        expect = rna_tf32_bits(x)
        expect[expect == 0x80000000] = 0                    # -0 + (+0) = +0
        got = _outputs(hsp, x)
        assert np.array_equal(got, expect), np.argwhere(got != expect)[:5]


def test_rounding_past_the_largest_tf32_value_gives_infinity(hsp):
    # one token holding the largest finite fp32 value at k = 0 and zeros elsewhere: output 0
    # is its rounding (the other outputs are 0 * inf)
    x = np.zeros((1, K), np.uint32)
    x[0, 0] = 0x7F7FFFFF
    assert _outputs(hsp, x)[0, 0] == 0x7F800000
