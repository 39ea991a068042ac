"""GPU parity for the streaming configuration: the Qwen2.5-Omni-3B head shape fed
1-s chunks of [2,304 video, 25 audio] tokens through okvq_append_chunk, with one
decode query after every chunk (each decode after an append rebuilds the decode
work split), every output compared with the CPU oracle fed the same chunks, and the
stored state compared bit for bit at several points of the stream ("OmniKVQuant:
KV Cache Quantization for Omni-LLMs", section 2 METHOD, first OmniKVQuant bullet:
groups of consecutive tokens quantized as they arrive)."""
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


def _stream(w, check_state_after, decode_every=1, static_scratch=False):
    import torch
    sh = w.shape
    oc, R = pu.oracle_cache(w)
    c = pu.gpu_cache(w, R=R, bounds=[[]])              # created empty, fed below
    K, V = w.session_kv(0)
    mod = w.sessions[0].modality()
    Kd, Vd, Md = (torch.from_numpy(x).cuda() for x in (K, V, mod))
    errs, n_dec = [], 0
    for i, (a, b) in enumerate(w.sessions[0].chunk_bounds()):
        c.append(0, Kd[a:b], Vd[a:b], Md[a:b])
        oc.append(0, K[a:b], V[a:b], mod[a:b])
        if i in check_state_after:
            st = c.export_state(0)
            pu.assert_state_matches(pu.compare_state(st, oc, 0, oc.layers, sh.bits))
            pu.adopt_boundary_choices(st, oc, 0, oc.layers)
        if i % decode_every:
            continue
        Q = w.queries(i)
        Qd = torch.from_numpy(Q).cuda()
        if static_scratch:
            out = torch.empty_like(Qd)
            c.decode_static_scratch(Qd, out)
            out = out.cpu().numpy()
        else:
            out = c.decode(Qd).cpu().numpy()
        errs.append(pu.assert_outputs_close(out, oc.decode(Q), "after chunk %d (T = %d)" % (i, b)))
        n_dec += 1
    assert c.check_errors() == 0
    return errs, n_dec


def test_streaming_2329_token_chunks_decode_after_every_chunk():
    """2 layers of the streaming configuration, 9 chunks to 20,961 tokens: a decode
    after every append (9 work-split rebuilds), the state compared after every chunk."""
    w = synth.streaming(tokens=20961, layers=2)
    assert [b - a for a, b in w.sessions[0].chunk_bounds()] == [2329] * 9
    _, n = _stream(w, check_state_after=set(range(9)))
    assert n == 9


def test_streaming_ragged_last_chunk_and_g64():
    """A stream that ends 13 tokens into its fourth chunk, key groups of 64: the
    open group's fp16 keys and a partial last page are attended after every append."""
    w = synth.streaming(tokens=7000, layers=1, group_size=64)
    assert [b - a for a, b in w.sessions[0].chunk_bounds()] == [2329, 2329, 2329, 13]
    _, n = _stream(w, check_state_after={0, 1, 2, 3})
    assert n == 4


def test_streaming_static_scratch_decode():
    """The same stream decoded through the entry point that allocates nothing."""
    w = synth.streaming(tokens=4658, layers=1)
    _, n = _stream(w, check_state_after={0, 1}, static_scratch=True)
    assert n == 2
