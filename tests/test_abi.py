"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/okvq.h declares, and rejects bad configurations
and arguments before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

from parity_util import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return ensure_built()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "okvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(okvq_[a-z_]+)\s*\(", src)))


def test_every_declared_function_is_exported(lib):
    from bit_kv_cache_rht_gb300 import okvq
    names = _header_functions()
    assert "okvq_create" in names and "okvq_decode" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(okvq.EXPORTS) == names


def test_status_strings(lib):
    from bit_kv_cache_rht_gb300 import okvq
    assert okvq.okvq_status_string(0) == "ok"
    assert okvq.okvq_status_string(3) == "capacity exceeded"
    assert okvq.okvq_status_string(99) == "unknown status"


def _cfg(**kw):
    from bit_kv_cache_rht_gb300.okvq import OkvqConfig
    R = np.zeros((1, 2, 3, 128, 128), np.float32)
    base = dict(num_sessions=1, num_layers=1, num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=32, bits=2,
                num_modalities=3, max_tokens=64, hadamard_seed=1)
    base.update(kw)
    c = OkvqConfig(base["num_sessions"], base["num_layers"], base["num_q_heads"], base["num_kv_heads"],
                   base["head_dim"], base["group_size"], base["bits"], base["num_modalities"], base["max_tokens"],
                   base["hadamard_seed"], None, R.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return c, R


@pytest.mark.parametrize("bad", [
    dict(head_dim=64), dict(group_size=16), dict(group_size=48), dict(bits=3), dict(bits=8),
    dict(num_q_heads=7), dict(num_q_heads=18), dict(num_modalities=0), dict(num_modalities=4),
    dict(max_tokens=0), dict(num_sessions=0), dict(num_layers=0),
])
def test_create_rejects_bad_configs_before_cuda(lib, bad):
    from bit_kv_cache_rht_gb300 import okvq
    cfg, _keep = _cfg(**bad)
    st, h = okvq.okvq_create(cfg)
    assert st == okvq.OKVQ_EINVAL and not h.value


def test_create_rejects_unknown_key_codec(lib):
    from bit_kv_cache_rht_gb300 import okvq
    cfg, _keep = _cfg()
    cfg.key_codec = 2
    st, h = okvq.okvq_create(cfg)
    assert st == okvq.OKVQ_EINVAL and not h.value


def test_create_rejects_non_ascending_codebook(lib):
    from bit_kv_cache_rht_gb300 import okvq
    cfg, _keep = _cfg()
    cb = np.array([-1.0, 0.5, 0.2, 1.0], np.float32)
    cfg.codebook = cb.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    st, _ = okvq.okvq_create(cfg)
    assert st == okvq.OKVQ_EINVAL


def test_null_arguments(lib):
    from bit_kv_cache_rht_gb300 import okvq
    assert lib.okvq_create(None, None, None) == okvq.OKVQ_EINVAL
    okvq.okvq_free(None)                                    # no-op
    st, _ = okvq.okvq_length(None, 0)
    assert st == okvq.OKVQ_EINVAL
    assert okvq.okvq_decode(None, 0, 0) == okvq.OKVQ_EINVAL
    assert okvq.okvq_append_chunk(None, 0, 0, 0, 0, 1) == okvq.OKVQ_EINVAL
    n = ctypes.c_size_t()
    assert lib.okvq_export_state(None, 0, None, ctypes.byref(n)) == okvq.OKVQ_EINVAL
    assert lib.okvq_profile_enable(None, 1) == okvq.OKVQ_EINVAL


def test_binding_refuses_to_run_without_the_library(tmp_path, monkeypatch):
    from bit_kv_cache_rht_gb300 import okvq
    monkeypatch.setattr(okvq, "_lib", None)
    monkeypatch.setattr(okvq, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        okvq.load()


def test_layout_tables_are_bijections():
    """The lane-chunk code placement used by the kernels covers every (token, channel) of a tile once."""
    def kcoord(lane, j, e):
        blk, reg = j >> 2, j & 3
        return (lane >> 2) + 8 * (reg & 1), 16 * blk + 2 * (lane & 3) + 8 * (reg >> 1) + e

    def vcoord(lane, j, e):
        blk, reg = j >> 2, j & 3
        return 2 * (lane & 3) + 8 * (reg >> 1) + e, 16 * blk + (lane >> 2) + 8 * (reg & 1)

    for f in (kcoord, vcoord):
        seen = {f(l, j, e) for l in range(32) for j in range(32) for e in range(2)}
        assert seen == {(t, c) for t in range(16) for c in range(128)}
