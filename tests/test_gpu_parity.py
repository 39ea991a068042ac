"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. Codes and statistics must match bit for bit except counted
boundary codes; decode outputs within |gpu - ref| <= 2e-3 + 1e-2 |ref|."""
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


def _full_check(w, bounds=None, layers_check=None, steps=(0,)):
    import torch
    oc, R = pu.oracle_cache(w, layers=layers_check)
    pu.feed_oracle(oc, w, bounds=bounds)
    c = pu.gpu_cache(w, R=R, bounds=bounds)
    assert c.check_errors() == 0
    li = oc.layers
    for s in range(len(w.sessions)):
        st = c.export_state(s)
        pu.assert_state_matches(pu.compare_state(st, oc, s, li, w.shape.bits))
        pu.adopt_boundary_choices(st, oc, s, li)
    errs = []
    for step in steps:
        Q = w.queries(step)
        out = c.decode(torch.from_numpy(Q).cuda()).cpu().numpy()
        ref = oc.decode(Q)
        errs.append(pu.assert_outputs_close(out[:, li], ref, "step %d" % step))
    return c, oc, errs


@pytest.mark.parametrize("bits,G", [(2, 32), (2, 64), (4, 32), (4, 64)])
def test_tiny_one_chunk(bits, G):
    w = synth.tiny(seed=10 + bits + G, bits=bits, group_size=G)
    _full_check(w, bounds=[[(0, 2048)]], steps=(0, 1))


def test_tiny_streamed_in_odd_chunks_matches_oracle_and_single_chunk():
    w = synth.tiny(seed=21)
    T = 2048
    r = np.random.default_rng(3)
    cuts = sorted(r.choice(np.arange(1, T), 30, replace=False).tolist())
    bounds = [list(zip([0, *cuts], [*cuts, T]))]
    c1, _, _ = _full_check(w, bounds=bounds)
    c2 = pu.gpu_cache(w, bounds=[[(0, T)]])
    s1, s2 = c1.export_state(0), c2.export_state(0)
    for k in s1:
        assert np.array_equal(s1[k].view(np.uint8), s2[k].view(np.uint8)), k


def test_tiny_97_token_chunks():
    w = synth.tiny(seed=22)
    _full_check(w, bounds=[[(a, min(a + 97, 2048)) for a in range(0, 2048, 97)]])


@pytest.mark.parametrize("T", [1, 5, 16, 31, 32, 33, 63, 64, 65, 100, 130])
def test_short_sessions_and_tails(T):
    w = synth.tiny(seed=30 + T, tokens=T)
    _full_check(w, bounds=[[(0, T)]], steps=(0,))


def test_qwen3b_shape_streamed_chunks():
    w = synth.qwen3b(seed=40, tokens=5000, layers=3)
    _full_check(w, steps=(0, 1))


def test_bench_workload_full_size_sampled_layers():
    """The bench workload at full size (Qwen2.5-Omni-3B shape: 36 layers, 16 q / 2 kv
    heads, 32,768 tokens in 1-s chunks, 2-bit, G 32) through the same cache build and
    decode launch configuration bench.py times; the oracle recomputes the first and
    the last layer (both kv heads, all 16 query heads) and their stored state."""
    w = synth.qwen3b()
    _full_check(w, layers_check=[0, w.shape.num_layers - 1], steps=(0,))


def test_qwen7b_full_size_sampled_layer():
    """The 7B-shaped long stream at full size (28 layers, 28 q / 4 kv heads, 81,920
    tokens in 1-s chunks) through the same cache build and decode launch the
    benchmark times; the oracle recomputes the first layer (all 4 kv heads, all 28
    query heads) and its stored state."""
    w = synth.qwen7b()
    _full_check(w, layers_check=[0], steps=(0,))


def test_multisession_full_length_mix_sampled_sessions():
    """64 sessions with the full 4 K-64 K length mix and per-session interleaves (2
    layers): the multi-session work partition of the decode; the oracle recomputes
    the shortest and the longest session and one in between."""
    import torch
    w = synth.multisession(layers=2)
    lens = [x.length for x in w.sessions]
    pick = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 17})
    oc, R = pu.oracle_cache(w, sessions=pick)
    pu.feed_oracle(oc, w, sessions=pick)
    c = pu.gpu_cache(w, R=R)
    assert c.check_errors() == 0
    for s in pick:
        st = c.export_state(s)
        pu.assert_state_matches(pu.compare_state(st, oc, s, oc.layers, w.shape.bits))
        pu.adopt_boundary_choices(st, oc, s, oc.layers)
    Q = w.queries(0)
    out = c.decode(torch.from_numpy(Q).cuda()).cpu().numpy()
    ref = oc.decode(Q)
    pu.assert_outputs_close(out[pick], ref[pick], "sampled sessions")
    assert c.check_errors() == 0


@pytest.mark.parametrize("bits,G", [(2, 64), (4, 32), (4, 64)])
def test_multisession_full_length_mix_variants(bits, G):
    """The 64-session configuration's other code widths and group sizes with the full
    4 K-64 K length mix (1 layer): the oracle recomputes the shortest and the longest
    session and one in between, state bit for bit and outputs within tolerance."""
    import torch
    w = synth.multisession(layers=1, bits=bits, group_size=G)
    lens = [x.length for x in w.sessions]
    pick = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 17})
    oc, R = pu.oracle_cache(w, sessions=pick)
    pu.feed_oracle(oc, w, sessions=pick)
    c = pu.gpu_cache(w, R=R)
    assert c.check_errors() == 0
    for s in pick:
        st = c.export_state(s)
        pu.assert_state_matches(pu.compare_state(st, oc, s, oc.layers, w.shape.bits))
        pu.adopt_boundary_choices(st, oc, s, oc.layers)
    for step in (0, 1):
        Q = w.queries(step)
        out = c.decode(torch.from_numpy(Q).cuda()).cpu().numpy()
        ref = oc.decode(Q)
        pu.assert_outputs_close(out[pick], ref[pick], "sampled sessions, step %d" % step)
    assert c.check_errors() == 0


def test_qwen7b_shape_seven_heads_per_kv():
    w = synth.qwen7b(seed=41, tokens=3000, layers=2)
    _full_check(w, steps=(0,))


def test_multisession_mixed_lengths_and_empty():
    w = synth.multisession(seed=42, sessions=5, lo=40, hi=3000, layers=2)
    w.sessions[2] = synth.Session([])          # an empty session decodes to zeros
    c, oc, _ = _full_check(w, steps=(0,))
    import torch
    out = c.decode(torch.from_numpy(w.queries(0)).cuda()).cpu().numpy()
    assert np.all(out[2] == 0)


@pytest.mark.parametrize("bits,G", [(2, 64), (4, 32)])
def test_multisession_variants(bits, G):
    w = synth.multisession(seed=43, sessions=3, lo=500, hi=2500, layers=2, bits=bits, group_size=G)
    _full_check(w, steps=(0,))


def test_capacity_and_argument_errors():
    import torch
    from bit_kv_cache_rht_gb300 import okvq
    w = synth.tiny(seed=50, tokens=100)
    c = pu.gpu_cache(w, max_tokens=128)
    K = torch.zeros((40, 1, 2, 128), dtype=torch.float16, device="cuda")
    M = torch.zeros(40, dtype=torch.uint8, device="cuda")
    with pytest.raises(okvq.OkvqError) as e:
        c.append(0, K, K, M)
    assert e.value.status == okvq.OKVQ_ECAPACITY
    assert c.length(0) == 100                   # unchanged
    st = okvq.okvq_append_chunk(c._h, 1, K.data_ptr(), K.data_ptr(), M.data_ptr(), 4)
    assert st == okvq.OKVQ_EINVAL               # no such session
    # keys or values not 16-byte aligned (the value rows are copied in 16-byte pieces)
    B = torch.zeros(4 * 2 * 2 * 128 * 2 + 16, dtype=torch.uint8, device="cuda")   # room for 4 tokens either way
    for koff, voff in ((2, 0), (0, 8)):
        st = okvq.okvq_append_chunk(c._h, 0, B.data_ptr() + koff, B.data_ptr() + voff, M.data_ptr(), 4)
        assert st == okvq.OKVQ_EINVAL
    assert c.length(0) == 100                   # nothing appended
    assert c.check_errors() == 0


def test_bad_modality_sets_error_word():
    import torch
    w = synth.tiny(seed=51, tokens=64)
    c = pu.gpu_cache(w, max_tokens=256)
    K = torch.randn((8, 1, 2, 128), device="cuda").half()
    M = torch.full((8,), 7, dtype=torch.uint8, device="cuda")
    c.append(0, K, K, M)
    assert c.check_errors() & 1
    assert c.check_errors() == 0                # cleared by the read


def test_codebook_matches_oracle():
    w = synth.tiny(seed=52, tokens=16)
    for bits in (2, 4):
        w2 = synth.tiny(seed=52, tokens=16, bits=bits)
        c = pu.gpu_cache(w2)
        lv, kl = c.codebook()
        cb = o.make_codebook(bits)
        assert np.array_equal(lv.astype(np.float16), cb.levels16)
        assert np.array_equal(kl.astype(np.float16), cb.ktab16)


def test_decode_is_repeatable_and_query_dependent():
    import torch
    w = synth.tiny(seed=53)
    c = pu.gpu_cache(w)
    q = torch.from_numpy(w.queries(0)).cuda()
    a = c.decode(q).cpu().numpy()
    b = c.decode(q).cpu().numpy()
    assert np.array_equal(a, b)
    q2 = torch.from_numpy(w.queries(1)).cuda()
    assert not np.array_equal(a, c.decode(q2).cpu().numpy())


# ---------------------------------------------------------------- TurboQuant key codec

def _turbo_check(w, bounds=None, steps=(0,), shared_rotation=False):
    import torch
    from bit_kv_cache_rht_gb300.okvq import OKVQ_KEYS_TURBOQUANT
    R = None
    if shared_rotation:      # TurboQuant's one value rotation: the Hadamard rotation for every modality
        sh = w.shape
        Rh = o.hadamard_rotation(o.hadamard_signs(w.hadamard_seed, sh.head_dim)).astype(np.float32)
        R = np.ascontiguousarray(np.broadcast_to(Rh, (sh.num_layers, sh.num_kv_heads, sh.num_modalities,
                                                      sh.head_dim, sh.head_dim)))
    oc, R = pu.oracle_cache(w, key_codec="turbo", R=R)
    pu.feed_oracle(oc, w, bounds=bounds)
    c = pu.gpu_cache(w, R=R, bounds=bounds, key_codec=OKVQ_KEYS_TURBOQUANT)
    assert c.check_errors() == 0
    for s in range(len(w.sessions)):
        st = c.export_state(s)
        pu.assert_state_matches(pu.compare_state(st, oc, s, oc.layers, w.shape.bits))
        pu.adopt_boundary_choices(st, oc, s, oc.layers)
    for step in steps:
        Q = w.queries(step)
        out = c.decode(torch.from_numpy(Q).cuda()).cpu().numpy()
        pu.assert_outputs_close(out[:, oc.layers], oc.decode(Q), "turbo step %d" % step)


@pytest.mark.parametrize("bits", [2, 4])
def test_turbo_keys_tiny_one_chunk(bits):
    _turbo_check(synth.tiny(seed=60 + bits, bits=bits), bounds=[[(0, 2048)]], steps=(0, 1))


def test_turbo_keys_odd_chunks_and_shared_value_rotation():
    w = synth.tiny(seed=63)
    _turbo_check(w, bounds=[[(a, min(a + 97, 2048)) for a in range(0, 2048, 97)]], shared_rotation=True)


@pytest.mark.parametrize("T", [1, 17, 64, 130])
def test_turbo_keys_short_sessions(T):
    _turbo_check(synth.tiny(seed=64 + T, tokens=T), bounds=[[(0, T)]])


def test_turbo_keys_qwen3b_shape_and_multisession():
    _turbo_check(synth.qwen3b(seed=66, tokens=3000, layers=2), steps=(0, 1))
    _turbo_check(synth.multisession(seed=67, sessions=3, lo=100, hi=2000, layers=2))


def test_decode_host_equals_decode_on_device_buffers():
    """okvq_decode_host with pinned host queries and outputs (the queries read by the
    staging kernel on the decode's stream, the outputs stored by the merge kernel)
    gives okvq_decode's outputs bit for bit, with four calls queued before any
    synchronisation."""
    import torch
    w = synth.multisession(seed=45, sessions=3, lo=100, hi=2500, layers=2)
    c = pu.gpu_cache(w)
    Qs = [w.queries(step) for step in range(4)]
    refs = [c.decode(torch.from_numpy(Q).cuda()).cpu() for Q in Qs]
    qh = [torch.from_numpy(Q).pin_memory() for Q in Qs]
    oh = [torch.full(Q.shape, float("nan"), dtype=torch.float16).pin_memory() for Q in Qs]
    for q, o in zip(qh, oh):
        c.decode_host(q, o)
    torch.cuda.synchronize()
    for o, ref in zip(oh, refs):
        assert torch.equal(o, ref)


def test_decode_host_pageable_and_pinned_outputs_agree():
    """Pinned outputs are stored by the merge kernel itself; pageable outputs go
    through device staging and a copy. Both give okvq_decode's outputs bit for
    bit, also when the two kinds alternate on one handle."""
    import torch
    w = synth.qwen3b(seed=46, tokens=1500, layers=2)
    c = pu.gpu_cache(w)
    Qs = [w.queries(step) for step in range(4)]
    refs = [c.decode(torch.from_numpy(Q).cuda()).cpu() for Q in Qs]
    outs = []
    for i, Q in enumerate(Qs):
        o = torch.full(Q.shape, float("nan"), dtype=torch.float16)
        if i % 2:
            o = o.pin_memory()
        c.decode_host(torch.from_numpy(Q), o)          # pageable queries: a synchronous upload
        outs.append(o)
    torch.cuda.synchronize()
    for o, ref in zip(outs, refs):
        assert torch.equal(o, ref)


def test_decode_host_pinned_pageable_and_unaligned_queries_alternate():
    """The three query paths of okvq_decode_host on one handle, six calls queued
    before any synchronisation: pinned (the staging kernel), pageable (the copy
    stream into alternating slots) and pinned but off a 16-byte boundary (also the
    copy stream). Every call gives okvq_decode's outputs bit for bit."""
    import torch
    w = synth.qwen3b(seed=47, tokens=1800, layers=2)
    c = pu.gpu_cache(w)
    Qs = [w.queries(step) for step in range(6)]
    refs = [c.decode(torch.from_numpy(Q).cuda()).cpu() for Q in Qs]
    keep, outs = [], []
    for i, Q in enumerate(Qs):
        kind = i % 3
        if kind == 0:
            q = torch.from_numpy(Q).pin_memory()
        elif kind == 1:
            q = torch.from_numpy(Q.copy())
        else:
            buf = torch.empty(Q.size + 4, dtype=torch.float16).pin_memory()
            q = buf[4:].view(Q.shape)                  # 8 bytes past a 16-byte boundary
            q.copy_(torch.from_numpy(Q))
            assert q.data_ptr() % 16 == 8
            keep.append(buf)
        o = torch.full(Q.shape, float("nan"), dtype=torch.float16).pin_memory()
        c.decode_host(q, o)
        keep.append(q)
        outs.append(o)
    torch.cuda.synchronize()
    for o, ref in zip(outs, refs):
        assert torch.equal(o, ref)
    assert c.check_errors() == 0


def test_host_and_foreign_pointers_are_rejected_before_any_launch():
    """Pageable and pinned host memory passed where device memory is expected, and
    queries off a 16-byte boundary: OKVQ_EINVAL, nothing launched, the cache
    unchanged."""
    import torch
    from bit_kv_cache_rht_gb300 import okvq
    w = synth.tiny(seed=51, tokens=64)
    c = pu.gpu_cache(w)
    before = c.export_state(0)
    K = torch.zeros((8, 1, 2, 128), dtype=torch.float16)
    Kp = K.pin_memory()
    M = torch.zeros(8, dtype=torch.uint8)
    Kd = K.cuda()
    Md = M.cuda()
    E = okvq.OKVQ_EINVAL
    assert okvq.okvq_append_chunk(c._h, 0, K.data_ptr(), Kd.data_ptr(), Md.data_ptr(), 8) == E
    assert okvq.okvq_append_chunk(c._h, 0, Kd.data_ptr(), Kp.data_ptr(), Md.data_ptr(), 8) == E
    assert okvq.okvq_append_chunk(c._h, 0, Kd.data_ptr(), Kd.data_ptr(), M.data_ptr(), 8) == E
    q = torch.from_numpy(w.queries(0))
    qd, od = q.cuda(), torch.empty_like(q).cuda()
    assert okvq.okvq_decode(c._h, q.data_ptr(), od.data_ptr()) == E
    assert okvq.okvq_decode(c._h, qd.data_ptr(), q.pin_memory().data_ptr()) == E
    # queries off a 16-byte boundary (the decode stages them by bulk copy)
    qbuf = torch.zeros(qd.numel() + 8, dtype=torch.float16, device="cuda")
    assert okvq.okvq_decode(c._h, qbuf[1:].data_ptr(), od.data_ptr()) == E
    assert okvq.okvq_decode_static_scratch(c._h, qbuf[1:].data_ptr(), od.data_ptr()) == E
    torch.cuda.synchronize()
    assert c.length(0) == 64 and c.check_errors() == 0
    after = c.export_state(0)
    for k in before:
        assert np.array_equal(before[k].view(np.uint8), after[k].view(np.uint8)), k
    assert okvq.okvq_decode(c._h, qd.data_ptr(), od.data_ptr()) == okvq.OKVQ_OK


def test_injected_allocation_failures_give_enomem_without_leaks():
    """okvq_test_fail_alloc(k) makes the k-th device allocation of okvq_create fail:
    the call returns OKVQ_ENOMEM, frees what it had allocated and leaves no handle;
    past the last allocation the create succeeds."""
    import torch
    from bit_kv_cache_rht_gb300 import okvq
    w = synth.tiny(seed=52, tokens=64)
    R = pu.rotations(w)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    try:
        for k in range(40):
            okvq.okvq_test_fail_alloc(k)
            try:
                c = okvq.Cache(1, 1, 8, 2, 4096, R, group_size=32, bits=2)
            except okvq.OkvqError as e:
                assert e.status == okvq.OKVQ_ENOMEM
                failures += 1
                continue
            okvq.okvq_test_fail_alloc(-1)
            c.close()
            break
    finally:
        okvq.okvq_test_fail_alloc(-1)
    assert 10 <= failures < 40                   # every allocation of create was made to fail once
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info()[0] - free0) < (64 << 20)
