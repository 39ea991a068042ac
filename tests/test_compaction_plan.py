"""The library's host-side compaction planner (okvq_plan_compaction, no GPU)
against the oracle's plan_suffix_compaction on random deletion patterns."""
import numpy as np
import pytest

from oracle import okvq_oracle as o
import parity_util as pu


def _lib():
    pu.ensure_built()
    from bit_kv_cache_rht_gb300 import okvq
    return okvq


def test_planner_matches_oracle_on_random_deletions():
    okvq = _lib()
    r = np.random.default_rng(17)
    hits = 0
    for trial in range(600):
        gran = int(r.choice([16, 32, 64]))
        T = int(r.integers(0, 1500))
        dead = np.zeros(T, bool)
        for _ in range(int(r.integers(0, 10))):
            if T == 0:
                break
            a = int(r.integers(0, T))
            dead[a:a + int(r.integers(1, 300))] = True
        if trial % 11 == 0:
            dead[:] = True
        mp = int(r.integers(1, 6))
        st, sb, nl, nm = okvq.okvq_plan_compaction(dead.astype(np.uint8), T, gran, mp)
        assert st == okvq.OKVQ_OK
        plan = o.plan_suffix_compaction(dead, T, gran, mp) if T else None
        if plan is None:
            assert (sb, nl, nm) == (-1, T, 0)
        else:
            hits += 1
            assert (sb, nl, nm) == (plan[0] * gran, plan[1], len(plan[2]))
    assert hits > 100


def test_planner_rejects_bad_arguments():
    okvq = _lib()
    E = okvq.OKVQ_EINVAL
    d = np.zeros(10, np.uint8)
    assert okvq.okvq_plan_compaction(d, 10, 48, 1)[0] == E          # granule not 16/32/64
    assert okvq.okvq_plan_compaction(d, 10, 32, 0)[0] == E          # must save at least one page
    assert okvq.okvq_plan_compaction(d, -1, 32, 1)[0] == E
    assert okvq.okvq_plan_compaction(d, 0, 32, 1)[0] == okvq.OKVQ_OK


def test_eviction_entry_points_reject_a_null_handle():
    okvq = _lib()
    E = okvq.OKVQ_EINVAL
    assert okvq.okvq_evict(None, 0, [(0, 1)]) == E
    assert okvq.okvq_compact(None, 0, 1)[0] == E
    assert okvq.okvq_live_length(None, 0)[0] == E
    assert okvq.okvq_compaction_granule(None)[0] == E
