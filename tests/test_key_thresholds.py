"""CPU check of the reading behind the division-free key codes of the append.

The key code of a rotated key k' in a group with stored minimum mn and range rng
(both fp16 values) is the number of fp32 midpoint thresholds t_j with
fl32(fl32(k' - mn) / rng) > t_j ("OmniKVQuant: KV Cache Quantization for Omni-LLMs",
section 2 METHOD, first OmniKVQuant bullet: min-max scaling against a shared fixed
codebook; the division in fp32 is the reading the oracle fixes). The quotient is
non-decreasing in d = fl32(k' - mn), so for each t_j there is a smallest fp32 d_j with
fl32(d_j / rng) > t_j, and the code equals the number of j with d >= d_j. The append
finds d_j by walking fp32 neighbours from fl32(t_j * rng). This test repeats that
search in numpy float32 (IEEE division, round to nearest even) and checks the two
decisions agree around every boundary and on random points, for the codebooks'
actual key thresholds and ranges across the fp16 range (subnormal ranges included).
"""
import numpy as np
import pytest

import oracle.okvq_oracle as o

F32 = np.float32


def next_up(x):
    return np.nextafter(F32(x), F32(np.inf), dtype=F32)


def next_down(x):
    return np.nextafter(F32(x), F32(-np.inf), dtype=F32)


def above(d, rng, t):
    """The division-based decision: fl32(d / rng) > t."""
    return bool(F32(F32(d) / F32(rng)) > F32(t))


def key_threshold(t, rng):
    """Smallest fp32 d >= 0 with fl32(d / rng) > t, walked from fl32(t * rng)."""
    if not (rng > 0) or np.isinf(rng):
        return F32(np.inf)
    d = max(F32(F32(t) * F32(rng)), F32(0))
    for _ in range(64):
        if above(d, rng, t):
            break
        d = next_up(d)
    for _ in range(64):
        if d <= 0:
            break
        dp = next_down(d)
        if not above(dp, rng, t):
            break
        d = dp
    return F32(d)


def ranges(rs):
    """fp16 ranges: subnormal, small, unit-scale and large values."""
    raw = np.concatenate([rs.integers(1, 1024, 40),                     # subnormal fp16 bit patterns
                          rs.integers(0x0400, 0x7BFF, 400)]).astype(np.uint16)
    return np.unique(raw.view(np.float16).astype(F32))


@pytest.mark.parametrize("bits", [2, 4])
def test_walk_gives_the_exact_decision_boundary(bits):
    cb = o.make_codebook(bits)
    rs = np.random.default_rng(1234 + bits)
    for rng in ranges(rs):
        for t in cb.kthr.astype(F32):
            d = key_threshold(t, rng)
            assert np.isfinite(d)
            assert above(d, rng, t)                          # d qualifies
            if d > 0:
                assert not above(next_down(d), rng, t)       # its predecessor does not


@pytest.mark.parametrize("bits", [2, 4])
def test_threshold_count_equals_division_code(bits):
    cb = o.make_codebook(bits)
    thr = cb.kthr.astype(F32)
    rs = np.random.default_rng(99 + bits)
    for rng in ranges(rs)[::7]:
        ds = np.array([key_threshold(t, rng) for t in thr], F32)
        # points: each boundary and its neighbours, plus random d in [0, 1.1 rng]
        pts = np.concatenate([ds, [next_up(x) for x in ds], [next_down(x) for x in ds if x > 0],
                              (rs.random(64) * 1.1 * rng).astype(F32), [F32(0)]])
        for d in pts:
            code_div = sum(above(d, rng, t) for t in thr)
            code_thr = int(np.sum(d >= ds))
            assert code_div == code_thr, (rng, d, code_div, code_thr)


def test_zero_and_infinite_range_give_code_zero():
    for t in o.make_codebook(2).kthr.astype(F32):
        assert key_threshold(t, F32(0)) == np.inf
        assert key_threshold(t, F32(np.inf)) == np.inf
