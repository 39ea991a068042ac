"""GPU parity of eviction and ordered-suffix compaction ("OmniTide" sections 5.2
and 6.2): the CUDA path through the C ABI against the oracle on the same seeded
streams and the same deletion ranges. The stored state (codes, statistics, fp16
tail, norms, modality ids, every unit's deletion mask) must match bit for bit
(boundary codes counted, as everywhere); decode outputs within the usual
tolerance; the compaction plan (new length, moved granules) must be identical."""
import numpy as np
import pytest

from bit_kv_cache_rht_gb300 import synth
from oracle import okvq_oracle as o
import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pu.ensure_built()


def _build(w, key_codec="omni", layers=None):
    from bit_kv_cache_rht_gb300.okvq import OKVQ_KEYS_TURBOQUANT, OKVQ_KEYS_GROUP_RANGE
    oc, R = pu.oracle_cache(w, layers=layers, key_codec=key_codec)
    pu.feed_oracle(oc, w)
    c = pu.gpu_cache(w, R=R, key_codec=OKVQ_KEYS_TURBOQUANT if key_codec == "turbo" else OKVQ_KEYS_GROUP_RANGE)
    assert c.check_errors() == 0
    return c, oc


def _check(c, oc, w, steps=(0,), what=""):
    import torch
    for s in range(len(w.sessions)):
        st = c.export_state(s)
        pu.assert_state_matches(pu.compare_state(st, oc, s, oc.layers, w.shape.bits))
        pu.adopt_boundary_choices(st, oc, s, oc.layers)
        u = oc.units[(s, oc.layers[0], 0)]
        assert c.length(s) == u.T
        assert c.live_length(s) == int((~u.dead[:u.T]).sum())
    for step in steps:
        Q = w.queries(step)
        out = c.decode(torch.from_numpy(Q).cuda()).cpu().numpy()
        pu.assert_outputs_close(out[:, oc.layers], oc.decode(Q), "%s step %d" % (what, step))
    assert c.check_errors() == 0


def _max_saving(u, gran):
    """Pages saved by packing every granule that holds a live token (the whole-cache
    suffix, the largest saving any plan can reach)."""
    T = u.T
    live_tokens = sum(min(gran, T - a) for a in range(0, T, gran) if not u.dead[a:min(a + gran, T)].all())
    return -(-T // 64) - (-(-live_tokens // 64))


def _evict_both(c, oc, s, ranges):
    c.evict(s, ranges)
    for a, b in ranges:
        oc.evict(s, a, b)


def _compact_both(c, oc, s, min_pages):
    nl, nm = c.compact(s, min_pages)
    plan = oc.compact(s, min_pages)
    if plan is None:
        assert nm == 0 and nl == oc.units[(s, oc.layers[0], 0)].T
    else:
        assert (nl, nm) == (plan[1], len(plan[2]))
    return plan


@pytest.mark.parametrize("key_codec,bits,G", [("omni", 2, 32), ("omni", 4, 64), ("omni", 2, 64), ("turbo", 2, 32)])
def test_eviction_then_compaction_then_appends(key_codec, bits, G):
    """Random ranges (sinks, whole groups, group interiors, tail tokens), decode;
    compaction; then the rest of the stream appended, decode again."""
    import torch
    w = synth.tiny(seed=80 + bits + G, bits=bits, group_size=G)
    T = 2048
    cut = 1700 + 13                                     # an open group at the compaction
    from bit_kv_cache_rht_gb300.okvq import OKVQ_KEYS_TURBOQUANT, OKVQ_KEYS_GROUP_RANGE
    oc, R = pu.oracle_cache(w, key_codec=key_codec)
    pu.feed_oracle(oc, w, bounds=[[(0, 900), (900, cut)]])
    c = pu.gpu_cache(w, R=R, bounds=[[(0, 900), (900, cut)]],
                     key_codec=OKVQ_KEYS_TURBOQUANT if key_codec == "turbo" else OKVQ_KEYS_GROUP_RANGE)
    r = np.random.default_rng(bits * 7 + G)
    ranges = [(0, 4), (100, 420), (431, 433), (640, 1100), (1705, cut)]
    ranges += [(int(a), int(a) + int(r.integers(1, 40))) for a in r.integers(1150, 1650, 8)]
    _evict_both(c, oc, 0, ranges)
    _check(c, oc, w, steps=(0,), what="evicted")
    plan = _compact_both(c, oc, 0, 3)
    assert plan is not None and len(plan[2]) > 0
    _check(c, oc, w, steps=(1,), what="compacted")
    K, V = w.session_kv(0)
    mod = w.sessions[0].modality()
    n0 = c.length(0)
    c.append(0, torch.from_numpy(K[cut:]).cuda(), torch.from_numpy(V[cut:]).cuda(), torch.from_numpy(mod[cut:]).cuda())
    oc.append(0, K[cut:], V[cut:], mod[cut:])
    assert c.length(0) == n0 + T - cut
    _check(c, oc, w, steps=(2,), what="appended")


def test_evicting_everything_decodes_to_zero_and_compacts_to_nothing():
    import torch
    w = synth.tiny(seed=90, tokens=300)
    c, oc = _build(w)
    _evict_both(c, oc, 0, [(0, 150), (150, 300), (10, 20)])
    out = c.decode(torch.from_numpy(w.queries(0)).cuda()).cpu().numpy()
    assert np.all(out == 0)
    assert c.live_length(0) == 0
    _compact_both(c, oc, 0, 1)                          # the shortest suffix saving a page: the last one
    assert c.length(0) == 256
    _compact_both(c, oc, 0, 4)                          # all four remaining pages
    assert c.length(0) == 0
    _check(c, oc, w)


def test_no_plan_leaves_the_cache_untouched():
    w = synth.tiny(seed=91, tokens=700)
    c, oc = _build(w)
    _evict_both(c, oc, 0, [(3, 9), (200, 230)])        # no whole empty group: nothing can shrink
    before = c.export_state(0)
    assert c.compact(0, 1) == (700, 0)
    after = c.export_state(0)
    for k in before:
        assert np.array_equal(before[k].view(np.uint8), after[k].view(np.uint8)), k


def test_argument_errors():
    from bit_kv_cache_rht_gb300 import okvq
    w = synth.tiny(seed=92, tokens=100)
    c, _ = _build(w)
    for bad in ([(5, 4)], [(-1, 3)], [(90, 101)]):
        assert okvq.okvq_evict(c._h, 0, bad) == okvq.OKVQ_EINVAL
    assert okvq.okvq_evict(c._h, 1, [(0, 1)]) == okvq.OKVQ_EINVAL      # no such session
    assert okvq.okvq_compact(c._h, 0, 0)[0] == okvq.OKVQ_EINVAL
    assert c.live_length(0) == 100                                      # nothing changed
    assert okvq.okvq_evict(c._h, 0, []) == okvq.OKVQ_OK
    assert c.compaction_granule() == 32


def test_multisession_retention_in_one_session():
    w = synth.multisession(seed=93, sessions=3, lo=500, hi=2500, layers=2)
    c, oc = _build(w)
    ranges = synth.retention_ranges(w.sessions[1], keep_recent=1, sinks=(16, 4, None))
    assert ranges
    _evict_both(c, oc, 1, ranges)
    _check(c, oc, w, what="evicted")
    _compact_both(c, oc, 1, 1)
    _check(c, oc, w, steps=(1,), what="compacted")


def test_qwen3b_shape_retention_and_full_compaction():
    """The 1-s chunk stream of the 3B shape, retention-shaped deletions, and the
    largest compaction (the whole-cache suffix's saving as the threshold)."""
    w = synth.qwen3b(seed=94, tokens=6000, layers=3)
    c, oc = _build(w)
    ranges = synth.retention_ranges(w.sessions[0], keep_recent=2)
    _evict_both(c, oc, 0, ranges)
    _check(c, oc, w, what="evicted")
    plan = _compact_both(c, oc, 0, _max_saving(oc.units[(0, 0, 0)], 32))
    assert plan[0] < 40                                   # nearly the whole cache moves
    _check(c, oc, w, steps=(1, 2), what="compacted")


def test_bench_workload_full_size_compaction_in_batches():
    """The bench workload (36 layers, 32,768 tokens): retention-shaped deletions and
    a compaction over most of the cache, which needs several scratch batches (each
    move carries 73 slots of ~2.6 KB). The oracle recomputes the first and last
    layer."""
    w = synth.qwen3b()
    c, oc = _build(w, layers=[0, w.shape.num_layers - 1])
    ranges = synth.retention_ranges(w.sessions[0], keep_recent=4, sinks=(384, 12, None))
    _evict_both(c, oc, 0, ranges)
    plan = _compact_both(c, oc, 0, _max_saving(oc.units[(0, 0, 0)], 32))
    assert plan is not None and len(plan[2]) > 348       # more moves than one 64 MB batch holds
    _check(c, oc, w, steps=(0,), what="full size compacted")
