"""The seeded input generators shared by the oracle and the CUDA path (CPU only)."""
import math

import numpy as np

import moe_inputs


def test_gumbel_draws_match_the_standard_gumbel_law():
    g = moe_inputs.gumbel(5, 4096, 64).astype(np.float64)
    assert g.dtype == np.float64 and np.isfinite(g).all()
    # mean = Euler-Mascheroni constant, variance = pi^2 / 6, CDF exp(-exp(-x))
    n = g.size
    assert abs(g.mean() - 0.5772156649) < 4 * math.sqrt(math.pi ** 2 / 6 / n)
    assert abs(g.var() - math.pi ** 2 / 6) < 0.02
    for x in (-1.0, 0.0, 1.0, 3.0):
        assert abs((g <= x).mean() - math.exp(-math.exp(-x))) < 3e-3
    assert np.array_equal(g, moe_inputs.gumbel(5, 4096, 64))
    assert not np.array_equal(g, moe_inputs.gumbel(6, 4096, 64))


def test_padding_mask_is_right_padded_sequences():
    T, S = 1100, 128
    m = moe_inputs.padding_mask(3, T, S)
    assert m.dtype == np.uint8 and set(np.unique(m)) <= {0, 1}
    nseq = T // S
    for s in range(nseq - 1):
        seg = m[s * S:(s + 1) * S]
        n = int(seg.sum())
        assert S // 2 <= n <= S and (seg[:n] == 1).all() and (seg[n:] == 0).all()
    assert (m[(nseq - 1) * S:] == 0).all()
    assert np.array_equal(m, moe_inputs.padding_mask(3, T, S))


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)
    b = moe_inputs.bf16_bits(v)
    back = moe_inputs.as_f64(b, "bf16")
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 0.0]
