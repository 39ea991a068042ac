"""The decode's split of the work over CTAs (okvq_plan_decode, host only): every
page covered once and in order, segments cut at unit boundaries, and the largest
CTA cost (pages + segment_cost per segment) minimal, checked by brute force over
all contiguous splits on small inputs."""
import itertools

import numpy as np
import pytest

import parity_util as pu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pu.ensure_built()


def _okvq():
    from bit_kv_cache_rht_gb300 import okvq
    return okvq


def plan(pages, ctas, sc):
    okvq = _okvq()
    st, seg, first = okvq.okvq_plan_decode(pages, ctas, sc)
    assert st == okvq.OKVQ_OK
    return seg, first


def cta_costs(seg, first, sc):
    return [sum(int(e - b) + sc for _, b, e in seg[first[c]:first[c + 1]]) for c in range(len(first) - 1)]


def check_cover(pages, seg, first, ctas):
    P = int(sum(pages))
    nc = len(first) - 1
    assert nc <= ctas and (nc >= 1) == (P > 0)
    assert first[0] == 0 and first[-1] == len(seg) and np.all(np.diff(first) >= 1)
    # segments in order over the flattened (unit, page) list, none empty, cut at unit ends
    flat = [(u, p) for u in range(len(pages)) for p in range(pages[u])]
    got = [(int(u), p) for u, b, e in seg for p in range(b, e)]
    assert got == flat
    assert all(e > b for _, b, e in seg)
    for c in range(nc):
        units = [int(u) for u, _, _ in seg[first[c]:first[c + 1]]]
        assert units == sorted(set(units))          # one segment per unit inside a CTA


def brute_best(pages, ctas, sc):
    """Smallest largest-CTA cost over every split of the flattened page list into
    at most `ctas` non-empty contiguous ranges."""
    flat_unit = [u for u in range(len(pages)) for _ in range(pages[u])]
    P = len(flat_unit)
    if P == 0:
        return 0
    best = None
    for k in range(1, min(ctas, P) + 1):
        for cuts in itertools.combinations(range(1, P), k - 1):
            edges = (0,) + cuts + (P,)
            worst = max((edges[i + 1] - edges[i]) + sc * len(set(flat_unit[edges[i]:edges[i + 1]]))
                        for i in range(k))
            best = worst if best is None else min(best, worst)
    return best


@pytest.mark.parametrize("seed", range(40))
def test_split_is_minimal_against_brute_force(seed):
    rng = np.random.default_rng(1000 + seed)
    U = int(rng.integers(1, 5))
    pages = [int(x) for x in rng.integers(0, 5, U)]
    ctas = int(rng.integers(1, 5))
    sc = int(rng.integers(0, 4))
    seg, first = plan(pages, ctas, sc)
    check_cover(pages, seg, first, ctas)
    if sum(pages):
        assert max(cta_costs(seg, first, sc)) == brute_best(pages, ctas, sc)


@pytest.mark.parametrize("seed", range(12))
def test_split_covers_large_random_lists(seed):
    rng = np.random.default_rng(2000 + seed)
    U = int(rng.integers(1, 600))
    pages = [int(x) for x in rng.integers(0, 1100, U)]
    pages[int(rng.integers(0, U))] = 0                  # an empty unit somewhere
    ctas = int(rng.choice([1, 7, 152]))
    sc = int(rng.choice([0, 16, 48]))
    seg, first = plan(pages, ctas, sc)
    check_cover(pages, seg, first, ctas)
    costs = cta_costs(seg, first, sc)
    # no CTA is worse than an even split of the pages plus the segments a CTA
    # cannot avoid (one more than its share of unit boundaries)
    P = sum(pages)
    nonempty = sum(1 for p in pages if p)
    assert max(costs) <= -(-P // ctas) + sc * (-(-nonempty // ctas) + 2) + sc + 1


def test_zero_segment_cost_is_an_even_page_split():
    pages = [512] * 72                                   # 3B shape: 36 layers x 2 kv heads x 32 K tokens
    seg, first = plan(pages, 152, 0)
    costs = cta_costs(seg, first, 0)
    assert max(costs) == -(-sum(pages) // 152)


def test_segment_cost_beats_the_even_page_split_under_its_own_model():
    """Priced with segment cost 48, the plan made with that cost is no worse than the
    even page split; on the 3B shape (72 units of 512 pages, 152 CTAs) it is two
    one-segment CTAs per unit (144 CTAs of 256 pages, cost 304) instead of 152
    CTAs of 242-243 pages, 71 of them with two segments (cost 339)."""
    rng = np.random.default_rng(7)
    for pages in ([512] * 72, [1280] * 112, [int(x) for x in rng.integers(64, 1025, 300)]):
        seg48, first48 = plan(pages, 152, 48)
        seg0, first0 = plan(pages, 152, 0)
        assert max(cta_costs(seg48, first48, 48)) <= max(cta_costs(seg0, first0, 48))
    seg, first = plan([512] * 72, 152, 48)
    assert len(first) - 1 == 144 and np.all(np.diff(first) == 1)
    assert all(int(e - b) == 256 for _, b, e in seg)
    seg0, first0 = plan([512] * 72, 152, 0)
    assert max(cta_costs(seg0, first0, 48)) == 243 + 2 * 48


def test_empty_and_invalid_inputs():
    okvq = _okvq()
    st, seg, first = okvq.okvq_plan_decode([0, 0, 0], 152, 48)
    assert st == okvq.OKVQ_OK and len(seg) == 0 and list(first) == [0]
    st, seg, first = okvq.okvq_plan_decode([], 4, 0)
    assert st == okvq.OKVQ_OK and len(seg) == 0
    assert okvq.okvq_plan_decode([3, 4], 0, 0)[0] == okvq.OKVQ_EINVAL
    assert okvq.okvq_plan_decode([3, 4], 2, -1)[0] == okvq.OKVQ_EINVAL
    assert okvq.okvq_plan_decode([3, -4], 2, 0)[0] == okvq.OKVQ_EINVAL
