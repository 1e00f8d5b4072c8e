"""CPU: the exactness claim behind the tensor-core path's two-term split of bf16
activations (DESIGN reading c19), checked from its definition with the oracle's E4M3
encoder (pinned on its own in test_oracle_mxfp8.py), independently of the GPU.

Per 32-element group: hi = E4M3(x / 2^(s_hi - 127)) with s_hi the smallest scale byte
that keeps the group's largest magnitude within 448; lo = E4M3((x - hi) / 2^(s_lo - 127))
with s_lo = s_hi - 4 (0 below 4).  Claimed: hi + lo == x for every element within 2^14
of its group's largest, within 2^-21 of the largest for the rest."""
import numpy as np
import pytest

import oracle
from tests._harness import smallest_scale_within_448


def test_scale_rule_is_the_smallest_byte_within_448():
    rng = np.random.default_rng(0)
    amax = np.concatenate([np.exp2(rng.uniform(-120, 120, 4000)),
                           448.0 * np.exp2(np.arange(-20, 21, dtype=np.float64)),  # exact boundaries
                           np.nextafter(448.0 * np.exp2(np.arange(-20, 21, dtype=np.float64)), np.inf),
                           [0.0]])
    s = smallest_scale_within_448(amax)
    nz = amax > 0
    lim = lambda b: 448.0 * np.exp2(b.astype(np.float64) - 127)
    assert np.all(amax[nz] <= lim(s[nz]))
    above = nz & (s > 0)  # byte 0 (2^-127) is the smallest there is
    assert np.all(amax[above] > lim(s[above] - 1))
    assert np.all(amax[nz & (s == 0)] <= lim(np.zeros(1, np.int64)))
    assert s[~nz].tolist() == [0]
    # the boundaries: 448 * 2^k itself fits at byte 127 + k, the next float up needs one more
    b = 448.0 * np.exp2(np.arange(-20, 21, dtype=np.float64))
    assert np.array_equal(smallest_scale_within_448(b), 127 + np.arange(-20, 21))
    assert np.array_equal(smallest_scale_within_448(np.nextafter(b, np.inf)), 128 + np.arange(-20, 21))


def _bf16(v):
    return oracle.round_bf16(v)


def _split(x):
    """The two terms of one group per the definition above (values, not codes)."""
    amax = np.abs(x).max()
    s_hi = int(smallest_scale_within_448(np.array([amax]))[0])
    s_lo = max(s_hi - 4, 0)
    sh, sl = 2.0 ** (s_hi - 127), 2.0 ** (s_lo - 127)
    hi = np.array([oracle.e4m3(oracle.e4m3_encode(v / sh)) * sh for v in x])
    lo = np.array([oracle.e4m3(oracle.e4m3_encode(v / sl)) * sl for v in x - hi])
    return hi, lo


@pytest.mark.parametrize("spread", [4, 14, 30])
def test_two_terms_hold_bf16_within_2_14_of_the_largest(spread):
    """Random bf16 groups whose magnitudes span 2^spread (log-uniform, random signs, some
    exact zeros): the terms sum to x exactly inside 2^14 of the group's largest and to
    within 2^-21 of the largest outside; neither term saturates."""
    rng = np.random.default_rng(spread)
    for _ in range(60):
        mag = np.exp2(rng.uniform(-spread, 0, 32) + rng.uniform(-40, 40))
        x = _bf16(mag * rng.choice([-1.0, 1.0], 32))
        x[rng.integers(0, 32, 2)] = 0.0
        hi, lo = _split(x)
        amax = np.abs(x).max()
        inside = np.abs(x) >= amax * 2.0 ** -14
        assert np.array_equal((hi + lo)[inside], x[inside])
        assert np.all(np.abs(hi + lo - x)[~inside] <= amax * 2.0 ** -21)
        assert np.all(np.isfinite(hi)) and np.all(np.isfinite(lo))


def test_two_terms_of_a_group_of_zeros():
    hi, lo = _split(np.zeros(32))
    assert not hi.any() and not lo.any()
