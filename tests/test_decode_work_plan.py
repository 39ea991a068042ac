"""The split okvq_decode itself uses (okvq_plan_decode_work, host only): the
contiguous split, or the row-aligned one when whole rows of pages make it at least
one row cheaper. Checked: every page of every unit covered exactly once, segments
inside their unit and never empty, a unit's partial slots consecutive in page order,
the chosen split never costlier than the contiguous one under the row model, and the
3B shape's expected layout (pieces of 21 rows, remainders on the idle CTAs)."""
import numpy as np
import pytest

import parity_util as pu

ROW_SEG = 12


@pytest.fixture(scope="module", autouse=True)
def _built():
    pu.ensure_built()


def _okvq():
    from bit_kv_cache_rht_gb300 import okvq
    return okvq


def work(pages, ctas, bits):
    okvq = _okvq()
    st, seg, first, ufirst = okvq.okvq_plan_decode_work(pages, ctas, bits)
    assert st == okvq.OKVQ_OK
    return seg, first, ufirst


def row_cost(seg, first, W):
    """Costliest CTA: a segment of n pages costs ROW_SEG + W * ceil(n / W)."""
    worst = 0
    for c in range(len(first) - 1):
        t = sum(ROW_SEG + W * -(-int(e - b) // W) for _, b, e, *_ in seg[first[c]:first[c + 1]])
        worst = max(worst, t)
    return worst


def check_work(pages, ctas, bits, seg, first, ufirst):
    U = len(pages)
    P = int(sum(pages))
    nc, ns = len(first) - 1, len(seg)
    assert nc <= ctas and (nc >= 1) == (P > 0)
    assert first[0] == 0 and first[-1] == ns and np.all(np.diff(first) >= 1)
    # every page once
    seen = [np.zeros(p, np.int32) for p in pages]
    for u, b, e, _ in seg:
        assert 0 <= u < U and 0 <= b < e <= pages[u]
        seen[u][b:e] += 1
    assert all(np.all(x == 1) for x in seen)
    # partial slots: a permutation, consecutive per unit in page order, unit_first = CSR
    slots = seg[:, 3]
    assert sorted(slots.tolist()) == list(range(ns))
    by_slot = seg[np.argsort(slots)]
    assert np.all(np.diff(by_slot[:, 0]) >= 0)
    for u in range(U):
        rows = by_slot[ufirst[u]:ufirst[u + 1]]
        assert np.all(rows[:, 0] == u)
        assert int(np.sum(rows[:, 2] - rows[:, 1])) == pages[u]
        if len(rows):
            assert rows[0, 1] == 0 and np.all(rows[1:, 1] == rows[:-1, 2])
    assert ufirst[U] == ns


def test_3b_shape_takes_whole_rows_and_the_idle_ctas():
    pages = [512] * 72                          # 36 layers x 2 kv heads, 32,768 tokens
    seg, first, ufirst = work(pages, 152, 2)
    check_work(pages, 152, 2, seg, first, ufirst)
    assert len(first) - 1 == 152
    counts = np.diff(first)
    assert np.all(counts[:144] == 1) and np.all(counts[144:] == 9)
    assert np.all(seg[:144, 2] - seg[:144, 1] == 252)             # 21 rows of 12 pages
    rest = seg[144:]
    assert np.all(rest[:, 1] == 504) and np.all(rest[:, 2] == 512)
    assert sorted(rest[:, 0].tolist()) == list(range(72))
    okvq = _okvq()
    st, cseg, cfirst = okvq.okvq_plan_decode(pages, 152, 48)
    assert row_cost(seg, first, 12) + 12 <= row_cost(cseg, cfirst, 12)


def test_contiguous_split_kept_when_rows_do_not_pay():
    okvq = _okvq()
    # whole rows already, units shorter than a row, and halves whose rows a
    # row-aligned split cannot beat: the contiguous split stays, slots in order
    for pages, ctas in (([240] * 8, 8), ([5, 7, 3], 152), ([100] * 4, 8)):
        seg, first, ufirst = work(pages, ctas, 2)
        check_work(pages, ctas, 2, seg, first, ufirst)
        st, cseg, cfirst = okvq.okvq_plan_decode(pages, ctas, 48)
        assert np.array_equal(seg[:, :3], cseg) and np.array_equal(first, cfirst)
        assert np.array_equal(seg[:, 3], np.arange(len(seg)))


@pytest.mark.parametrize("bits", [2, 4])
def test_random_shapes_cover_every_page_and_never_cost_more(bits):
    okvq = _okvq()
    W = 12 if bits == 2 else 8
    rs = np.random.default_rng(77 + bits)
    for _ in range(60):
        U = int(rs.integers(1, 90))
        mode = rs.integers(0, 3)
        if mode == 0:
            pages = [int(rs.integers(0, 1500))] * U
        elif mode == 1:
            pages = rs.integers(0, 1500, U).tolist()
        else:
            pages = (rs.integers(1, 40, U) * W + rs.integers(0, W, U)).tolist()
        ctas = int(rs.integers(1, 200))
        seg, first, ufirst = work(pages, ctas, bits)
        check_work(pages, ctas, bits, seg, first, ufirst)
        if sum(pages):
            st, cseg, cfirst = okvq.okvq_plan_decode(pages, ctas, 48)
            assert row_cost(seg, first, W) <= row_cost(cseg, cfirst, W)


def test_empty_and_bad_arguments():
    okvq = _okvq()
    seg, first, ufirst = work([0, 0, 0], 152, 2)
    assert len(seg) == 0 and len(first) == 1 and np.all(ufirst == 0)
    seg, first, ufirst = work([], 4, 4)
    assert len(seg) == 0
    E = okvq.OKVQ_EINVAL
    assert okvq.okvq_plan_decode_work([3, 4], 0, 2)[0] == E
    assert okvq.okvq_plan_decode_work([3, 4], 2, 3)[0] == E
    assert okvq.okvq_plan_decode_work([3, -4], 2, 2)[0] == E
