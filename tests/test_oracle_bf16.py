"""Pins of the oracle's bf16 rounding: torch's float32 -> bfloat16 conversion (a library
routine, round-to-nearest-even) and hand-worked ties."""
import numpy as np
import torch

from oracle.bf16 import round_bf16, BF16_MAX


def _torch_bf16(a32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a32).to(torch.bfloat16).to(torch.float64).numpy()


def test_matches_torch_on_random_float32():
    rng = np.random.default_rng(0)
    a = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    want = _torch_bf16(a)
    assert np.array_equal(round_bf16(a.astype(np.float64)), want)
    assert np.array_equal(round_bf16(a).astype(np.float64), want)


def test_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7
    cases = {
        one + ulp / 2: one,                    # halfway, 1.0 has an even mantissa
        one + 3 * ulp / 2: one + 2 * ulp,      # halfway, rounds up to the even neighbour
        one + ulp / 2 + 2.0 ** -30: one + ulp,  # just above halfway
        -(one + ulp / 2): -one,
    }
    for x, want in cases.items():
        assert round_bf16(np.array([x]))[0] == want


def test_halfway_float32_ties_match_torch():
    # every bf16 value + half an ulp: exact float32 ties
    base = np.arange(0x3F00, 0x4100, dtype=np.uint32) << 16
    ties = (base | (1 << 15)).view(np.float32)
    assert np.array_equal(round_bf16(ties.astype(np.float64)), _torch_bf16(ties))


def test_specials_and_range():
    a = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 3.4e38, -3.4e38, 1e-40, 2.0 ** -133 * 0.75])
    r = round_bf16(a)
    assert r[0] == np.inf and r[1] == -np.inf and np.isnan(r[2])
    assert r[3] == 0 and np.signbit(r[4])
    assert r[5] == np.inf and r[6] == -np.inf          # above the largest finite bf16
    assert r[7] == _torch_bf16(np.array([1e-40], dtype=np.float32))[0]
    assert r[8] == 2.0 ** -133
    assert round_bf16(np.array([BF16_MAX]))[0] == BF16_MAX
