"""GPU parity of the pseudo-token decode ("ProtoKV" section 3.3 Eq. (2),
Algorithm 4): okvq_decode_pseudo through the C ABI against the oracle's
decode_with_pseudo on the same seeded near windows and far-memory pseudo tokens,
within the usual output tolerance."""
import numpy as np
import pytest

from bit_kv_cache_rht_gb300 import synth
import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pu.ensure_built()


def _check(w, P, S, key_codec="omni", bounds=None, evict=None, steps=(0,), inactive=0.1, mass_fn=None):
    import torch
    from bit_kv_cache_rht_gb300.okvq import OKVQ_KEYS_TURBOQUANT, OKVQ_KEYS_GROUP_RANGE
    oc, R = pu.oracle_cache(w, key_codec=key_codec)
    pu.feed_oracle(oc, w, bounds=bounds)
    c = pu.gpu_cache(w, R=R, bounds=bounds,
                     key_codec=OKVQ_KEYS_TURBOQUANT if key_codec == "turbo" else OKVQ_KEYS_GROUP_RANGE)
    for s, ranges in (evict or {}).items():
        c.evict(s, ranges)
        for a, b in ranges:
            oc.evict(s, a, b)
    for s in range(len(w.sessions)):
        st = c.export_state(s)
        pu.assert_state_matches(pu.compare_state(st, oc, s, oc.layers, w.shape.bits))
        pu.adopt_boundary_choices(st, oc, s, oc.layers)
    KF, VF, MASS = w.pseudo_tokens(P, S, inactive=inactive)
    if mass_fn is not None:
        MASS = mass_fn(MASS)
    kf, vf, mf = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (KF, VF, MASS))
    errs = []
    for step in steps:
        Q = w.queries(step)
        out = c.decode_pseudo(torch.from_numpy(Q).cuda(), kf, vf, mf, S).cpu().numpy()
        ref = oc.decode_with_pseudo(Q, KF, VF, MASS, S)
        errs.append(pu.assert_outputs_close(out[:, oc.layers], ref, "pseudo step %d" % step))
    assert c.check_errors() == 0
    return c, errs


@pytest.mark.parametrize("P,S", [(64, 8), (5, 3), (1, 1), (300, 8)])
def test_tiny_near_window_with_far_memory(P, S):
    """Ragged far sizes: 512, 15, 1 and 2400 pseudo tokens per unit."""
    _check(synth.tiny(seed=100 + P), P, S, steps=(0, 1))


def test_far_memory_dominates_and_inactive_prototypes():
    """Large masses put most of the weight on the far memory; half the
    prototypes inactive."""
    _check(synth.tiny(seed=111, tokens=600), 40, 8, inactive=0.5, mass_fn=lambda m: m * 50.0)


def test_all_prototypes_inactive_equals_plain_decode():
    import torch
    w = synth.tiny(seed=112, tokens=900)
    c, _ = _check(w, 16, 8, mass_fn=lambda m: np.zeros_like(m))
    Q = torch.from_numpy(w.queries(0)).cuda()
    KF, VF, MASS = w.pseudo_tokens(16, 8)
    a = c.decode_pseudo(Q, torch.from_numpy(KF).cuda(), torch.from_numpy(VF).cuda(),
                        torch.zeros(MASS.shape, dtype=torch.float32).cuda(), 8).cpu().numpy()
    b = c.decode(Q).cpu().numpy()
    pu.assert_outputs_close(a, b.astype(np.float64), "inactive far memory vs plain decode")


def test_empty_near_window_and_evicted_near_tokens():
    w = synth.multisession(seed=113, sessions=3, lo=200, hi=1500, layers=2)
    w.sessions[1] = synth.Session([])                      # far memory only
    _check(w, 24, 8, evict={0: [(0, 100), (150, 190)]})


def test_turbo_keys_and_4bit_near_window():
    _check(synth.tiny(seed=114, bits=4, group_size=64), 32, 8)
    _check(synth.tiny(seed=115), 32, 8, key_codec="turbo")


def test_qwen3b_shape_near_and_far():
    """The 3B head shape with a 1:3 near:far budget (2,048 near tokens, 256
    prototypes x 8 pseudo tokens), two layers."""
    _check(synth.qwen3b(seed=116, tokens=2048, layers=2), 256, 8, steps=(0, 1))


def test_argument_errors():
    import torch
    from bit_kv_cache_rht_gb300 import okvq
    w = synth.tiny(seed=117, tokens=64)
    c = pu.gpu_cache(w)
    q = torch.from_numpy(w.queries(0)).cuda()
    out = torch.empty_like(q)
    kf = torch.zeros((1, 1, 2, 16, 128), dtype=torch.float16, device="cuda")
    mf = torch.ones((1, 1, 2, 2), dtype=torch.float32, device="cuda")
    E = okvq.OKVQ_EINVAL
    assert okvq.okvq_decode_pseudo(c._h, q.data_ptr(), kf.data_ptr(), kf.data_ptr(), mf.data_ptr(), 2, 0,
                                   out.data_ptr()) == E          # S < 1
    assert okvq.okvq_decode_pseudo(c._h, q.data_ptr(), 0, kf.data_ptr(), mf.data_ptr(), 2, 8,
                                   out.data_ptr()) == E          # no far keys
    assert okvq.okvq_decode_pseudo(c._h, q.data_ptr(), kf.data_ptr() + 2, kf.data_ptr(), mf.data_ptr(), 2, 8,
                                   out.data_ptr()) == E          # misaligned
    assert okvq.okvq_decode_pseudo(c._h, q.data_ptr(), 0, 0, 0, 0, 8, out.data_ptr()) == okvq.OKVQ_OK
    torch.cuda.synchronize()
    pu.assert_outputs_close(out.cpu().numpy(), c.decode(q).cpu().numpy().astype(np.float64), "no far memory")
