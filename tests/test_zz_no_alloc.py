"""okvq_decode_static_scratch, the decode variant whose split-K partials live in
the library's one static device array, against okvq_decode on the same cache.

The file name sorts last so that the comparison also runs after every other
test of the session (the array then holds whatever earlier calls left there);
it passes alone in a fresh process as well."""
import numpy as np
import pytest

from bit_kv_cache_rht_gb300 import synth
import parity_util as pu


def test_static_scratch_rejects_null_arguments_before_cuda():
    pu.ensure_built()
    from bit_kv_cache_rht_gb300 import okvq
    assert okvq.okvq_decode_static_scratch(None, 0, 0) == okvq.OKVQ_EINVAL
    assert okvq.okvq_status_string(okvq.OKVQ_ESCRATCH) == "decode work list exceeds the static scratch array"


def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pu.ensure_built()
    return torch


def _both(torch, c, Q):
    """okvq_decode's output, then okvq_decode_static_scratch's, for the same query."""
    Qd = torch.from_numpy(Q).cuda()
    ref = c.decode(Qd)
    out = torch.full_like(Qd, float("nan"))
    c.decode_static_scratch(Qd, out)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), out.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("bits,G", [(2, 32), (4, 64)])
def test_static_scratch_matches_decode_on_two_calls_in_a_row(bits, G):
    torch = _gpu()
    w = synth.tiny(seed=70 + bits + G, bits=bits, group_size=G)
    c = pu.gpu_cache(w, bounds=[[(0, 2048)]])
    Q0, Q1 = w.queries(0), w.queries(1)
    Q0d, Q1d = torch.from_numpy(Q0).cuda(), torch.from_numpy(Q1).cuda()
    ref0, ref1 = c.decode(Q0d), c.decode(Q1d)
    out0 = torch.full_like(Q0d, float("nan"))
    out1 = torch.full_like(Q1d, float("nan"))
    c.decode_static_scratch(Q0d, out0)           # two calls in a row on the shared array
    c.decode_static_scratch(Q1d, out1)
    torch.cuda.synchronize()
    assert c.check_errors() == 0
    pu.assert_outputs_close(out0.cpu().numpy(), ref0.cpu().numpy(), "static scratch, call 1")
    pu.assert_outputs_close(out1.cpu().numpy(), ref1.cpu().numpy(), "static scratch, call 2")


@pytest.mark.gpu
def test_static_scratch_follows_appends_and_other_handles():
    """The work list changes between the calls (appends, a second cache with more
    sessions); the array keeps the previous call's partials, which must not leak."""
    torch = _gpu()
    w = synth.tiny(seed=91)
    c = pu.gpu_cache(w, bounds=[[(0, 1500)]])
    ref, out = _both(torch, c, w.queries(0))
    pu.assert_outputs_close(out, ref, "before append")
    K, V = w.session_kv(0)
    mod = w.sessions[0].modality()
    c.append(0, torch.from_numpy(K[1500:]).cuda(), torch.from_numpy(V[1500:]).cuda(),
             torch.from_numpy(mod[1500:]).cuda())
    ref, out = _both(torch, c, w.queries(1))
    pu.assert_outputs_close(out, ref, "after append")
    w2 = synth.multisession(seed=44, sessions=4, lo=40, hi=3000, layers=2)
    c2 = pu.gpu_cache(w2)
    ref, out = _both(torch, c2, w2.queries(0))
    pu.assert_outputs_close(out, ref, "second handle")
    assert c2.check_errors() == 0
    ref, out = _both(torch, c, w.queries(2))
    pu.assert_outputs_close(out, ref, "first handle again")
    assert c.check_errors() == 0


@pytest.mark.gpu
def test_static_scratch_rejects_work_beyond_the_array():
    """More non-empty (session, layer, kv head) units than the array has segments:
    OKVQ_ESCRATCH with nothing launched; okvq_decode still serves the cache."""
    torch = _gpu()
    from bit_kv_cache_rht_gb300 import okvq
    L, Hkv, M = 288, 2, 1
    assert L * Hkv > okvq.OKVQ_STATIC_SCRATCH_SEGMENTS
    R = np.ascontiguousarray(np.broadcast_to(np.eye(128, dtype=np.float32), (L, Hkv, M, 128, 128)))
    c = okvq.Cache(1, L, Hkv, Hkv, 64, R, group_size=32, bits=2, num_modalities=M)
    g = torch.Generator().manual_seed(3)
    k = torch.randn(1, L, Hkv, 128, generator=g).half().cuda()
    v = torch.randn(1, L, Hkv, 128, generator=g).half().cuda()
    c.append(0, k, v, torch.zeros(1, dtype=torch.uint8).cuda())
    q = torch.randn(1, L, Hkv, 128, generator=g).half().cuda()
    out = torch.zeros_like(q)
    with pytest.raises(okvq.OkvqError) as e:
        c.decode_static_scratch(q, out)
    assert e.value.status == okvq.OKVQ_ESCRATCH
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0        # nothing was launched
    ref = c.decode(q)
    torch.cuda.synchronize()
    assert torch.isfinite(ref.float()).all() and torch.count_nonzero(ref).item() > 0
    assert c.check_errors() == 0
