"""Python binding of libokvq (ctypes): argument marshalling only.

The functions carry the C ABI's names (okvq_create, okvq_append_chunk,
okvq_decode, okvq_free, ...); ``Cache`` wraps them for torch tensors. All
compute runs in the library's CUDA kernels; there is no fallback: if
libokvq.so is missing or fails to load, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libokvq.so")

OKVQ_OK, OKVQ_EINVAL, OKVQ_ENOMEM, OKVQ_ECAPACITY, OKVQ_ECUDA, OKVQ_ESTATE, OKVQ_ESCRATCH = range(7)
OKVQ_STATIC_SCRATCH_SEGMENTS = 512
OKVQ_KEYS_GROUP_RANGE, OKVQ_KEYS_TURBOQUANT = 0, 1   # key codecs (okvq_config.key_codec)   # work-list segments held by okvq_decode_static_scratch's array

# every function the header declares (checked against include/okvq.h by the tests)
EXPORTS = (
    "okvq_create", "okvq_free", "okvq_append_chunk", "okvq_decode", "okvq_length", "okvq_export_state",
    "okvq_codebook", "okvq_check_errors", "okvq_profile_enable", "okvq_profile_read", "okvq_status_string",
    "okvq_decode_static_scratch", "okvq_calibrate_rotations", "okvq_live_length", "okvq_evict",
    "okvq_compaction_granule", "okvq_plan_compaction", "okvq_compact", "okvq_decode_pseudo", "okvq_decode_host",
    "okvq_test_fail_alloc", "okvq_plan_decode", "okvq_plan_decode_work",
)


class OkvqConfig(ctypes.Structure):
    _fields_ = [
        ("num_sessions", ctypes.c_int32),
        ("num_layers", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("num_modalities", ctypes.c_int32),
        ("max_tokens", ctypes.c_int64),
        ("hadamard_seed", ctypes.c_uint64),
        ("codebook", ctypes.POINTER(ctypes.c_float)),
        ("value_rot", ctypes.POINTER(ctypes.c_float)),
        ("key_codec", ctypes.c_int32),
    ]


class OkvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (%d)" % (what, status_string(status), status))


_lib = None


def load() -> ctypes.CDLL:
    """Load libokvq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libokvq.so is not built (run bit_kv_cache_rht_gb300.build.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    L.okvq_create.argtypes = [ctypes.POINTER(OkvqConfig), vp, ctypes.POINTER(vp)]
    L.okvq_free.argtypes = [vp]
    L.okvq_free.restype = None
    L.okvq_append_chunk.argtypes = [vp, i32, vp, vp, vp, i32, vp]
    L.okvq_decode.argtypes = [vp, vp, vp, vp]
    L.okvq_decode_static_scratch.argtypes = [vp, vp, vp, vp]
    L.okvq_calibrate_rotations.argtypes = [i32, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp]
    L.okvq_decode_pseudo.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, vp]
    L.okvq_decode_host.argtypes = [vp, vp, vp, vp]
    L.okvq_test_fail_alloc.argtypes = [ctypes.c_int64]
    L.okvq_live_length.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64)]
    L.okvq_evict.argtypes = [vp, i32, vp, i32, vp]
    L.okvq_compaction_granule.argtypes = [vp, ctypes.POINTER(i32)]
    L.okvq_plan_compaction.argtypes = [vp, ctypes.c_int64, i32, i32, ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(i32)]
    L.okvq_compact.argtypes = [vp, i32, i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(i32), vp]
    L.okvq_plan_decode.argtypes = [vp, ctypes.c_int64, i32, i32, vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.okvq_plan_decode_work.argtypes = [vp, ctypes.c_int64, i32, i32, vp, vp, vp, ctypes.POINTER(i32),
                                        ctypes.POINTER(i32)]
    L.okvq_length.argtypes = [vp, i32, ctypes.POINTER(i64)]
    L.okvq_export_state.argtypes = [vp, i32, vp, ctypes.POINTER(ctypes.c_size_t)]
    L.okvq_codebook.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    L.okvq_check_errors.argtypes = [vp, vp, ctypes.POINTER(u32)]
    L.okvq_profile_enable.argtypes = [vp, ctypes.c_int]
    L.okvq_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float), i32,
                                    ctypes.POINTER(i32)]
    L.okvq_status_string.argtypes = [ctypes.c_int]
    L.okvq_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("okvq_free", "okvq_status_string"):
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def status_string(s: int) -> str:
    return load().okvq_status_string(int(s)).decode()


def _check(status: int, what: str):
    if status != OKVQ_OK:
        raise OkvqError(status, what)


# ---- the C entry points, same names (status codes returned, not raised) ----

def okvq_create(cfg: OkvqConfig, stream: int = 0):
    h = ctypes.c_void_p()
    st = load().okvq_create(ctypes.byref(cfg), ctypes.c_void_p(stream), ctypes.byref(h))
    return st, h


def okvq_free(h) -> None:
    load().okvq_free(h)


def okvq_append_chunk(h, session: int, k_ptr: int, v_ptr: int, mod_ptr: int, num_tokens: int, stream: int = 0) -> int:
    return load().okvq_append_chunk(h, session, ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                    ctypes.c_void_p(mod_ptr), num_tokens, ctypes.c_void_p(stream))


def okvq_decode(h, q_ptr: int, out_ptr: int, stream: int = 0) -> int:
    return load().okvq_decode(h, ctypes.c_void_p(q_ptr), ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream))


def okvq_decode_host(h, q_host_ptr: int, out_host_ptr: int, stream: int = 0) -> int:
    return load().okvq_decode_host(h, ctypes.c_void_p(q_host_ptr), ctypes.c_void_p(out_host_ptr),
                                   ctypes.c_void_p(stream))


def okvq_decode_static_scratch(h, q_ptr: int, out_ptr: int, stream: int = 0) -> int:
    return load().okvq_decode_static_scratch(h, ctypes.c_void_p(q_ptr), ctypes.c_void_p(out_ptr),
                                             ctypes.c_void_p(stream))


def okvq_calibrate_rotations(num_layers: int, num_kv_heads: int, num_modalities: int, v_ptr: int, mod_ptr: int,
                             weight_ptr: int, num_tokens: int, rot_ptr: int, eig_ptr: int, sweeps_ptr: int = 0,
                             stream: int = 0) -> int:
    return load().okvq_calibrate_rotations(num_layers, num_kv_heads, num_modalities, ctypes.c_void_p(v_ptr),
                                           ctypes.c_void_p(mod_ptr), ctypes.c_void_p(weight_ptr), num_tokens,
                                           ctypes.c_void_p(rot_ptr), ctypes.c_void_p(eig_ptr),
                                           ctypes.c_void_p(sweeps_ptr), ctypes.c_void_p(stream))


def calibrate_rotations(v, modality, num_modalities: int = 3, weight=None, stream=None, return_sweeps=False):
    """v: cuda fp16 [n][L][Hkv][128]; modality: cuda uint8 [n]; weight: cuda fp32 [n][L][Hkv] or None.
    Returns (rot [L][Hkv][M][128][128], eig [L][Hkv][M][128]) as cuda fp32 tensors, plus the
    int32 sweep counts [L][Hkv][M] when return_sweeps."""
    import torch
    n, L, Hkv, d = (int(x) for x in v.shape)
    if d != 128 or v.dtype != torch.float16 or not v.is_cuda or not v.is_contiguous():
        raise ValueError("v must be a contiguous cuda fp16 tensor [n][L][Hkv][128]")
    if modality.dtype != torch.uint8 or tuple(modality.shape) != (n,) or not modality.is_cuda:
        raise ValueError("modality must be a cuda uint8 tensor [n]")
    if weight is not None and (weight.dtype != torch.float32 or tuple(weight.shape) != (n, L, Hkv)
                               or not weight.is_cuda or not weight.is_contiguous()):
        raise ValueError("weight must be a contiguous cuda fp32 tensor [n][L][Hkv]")
    rot = torch.empty((L, Hkv, num_modalities, d, d), dtype=torch.float32, device=v.device)
    eig = torch.empty((L, Hkv, num_modalities, d), dtype=torch.float32, device=v.device)
    sweeps = torch.empty((L, Hkv, num_modalities), dtype=torch.int32, device=v.device)
    st = okvq_calibrate_rotations(L, Hkv, num_modalities, v.data_ptr(), modality.data_ptr(),
                                  weight.data_ptr() if weight is not None else 0, n, rot.data_ptr(), eig.data_ptr(),
                                  sweeps.data_ptr(), _stream_handle(stream))
    _check(st, "okvq_calibrate_rotations")
    return (rot, eig, sweeps) if return_sweeps else (rot, eig)


def okvq_length(h, session: int):
    n = ctypes.c_int64()
    st = load().okvq_length(h, session, ctypes.byref(n))
    return st, n.value


def okvq_decode_pseudo(h, q_ptr: int, k_ptr: int, v_ptr: int, mass_ptr: int, num_prototypes: int,
                       tokens_per_prototype: int, out_ptr: int, stream: int = 0) -> int:
    return load().okvq_decode_pseudo(h, ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                     ctypes.c_void_p(mass_ptr), num_prototypes, tokens_per_prototype,
                                     ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream))


def okvq_live_length(h, session: int):
    n = ctypes.c_int64()
    st = load().okvq_live_length(h, session, ctypes.byref(n))
    return st, n.value


def okvq_evict(h, session: int, ranges, stream: int = 0) -> int:
    """ranges: sequence of (begin, end) slot pairs (host)."""
    arr = np.ascontiguousarray(np.asarray(ranges, np.int64).reshape(-1, 2))
    return load().okvq_evict(h, session, arr.ctypes.data_as(ctypes.c_void_p) if len(arr) else None, len(arr),
                             ctypes.c_void_p(stream))


def okvq_compaction_granule(h):
    n = ctypes.c_int32()
    st = load().okvq_compaction_granule(h, ctypes.byref(n))
    return st, n.value


def okvq_plan_compaction(dead, length: int, granule: int, min_pages_saved: int):
    """dead: host bytes [length] (nonzero = deleted). Returns (status, suffix_begin, new_length, num_moves)."""
    d = np.ascontiguousarray(np.asarray(dead, np.uint8))
    sb, nl, nm = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    st = load().okvq_plan_compaction(d.ctypes.data_as(ctypes.c_void_p) if length > 0 else None, length, granule,
                                     min_pages_saved, ctypes.byref(sb), ctypes.byref(nl), ctypes.byref(nm))
    return st, sb.value, nl.value, nm.value


def okvq_plan_decode(unit_pages, max_ctas: int, segment_cost: int):
    """Host split of the decode work. Returns (status, segments [n][3] = (unit, first page,
    end page), cta_first [ctas + 1])."""
    p = np.ascontiguousarray(np.asarray(unit_pages, np.int64))
    units = p.shape[0]
    seg = np.zeros((units + max(max_ctas, 1), 3), np.int32)
    first = np.zeros(max(max_ctas, 1) + 1, np.int32)
    nc, ns = ctypes.c_int32(), ctypes.c_int32()
    st = load().okvq_plan_decode(p.ctypes.data_as(ctypes.c_void_p) if units else None, units, max_ctas, segment_cost,
                                 seg.ctypes.data_as(ctypes.c_void_p), first.ctypes.data_as(ctypes.c_void_p),
                                 ctypes.byref(nc), ctypes.byref(ns))
    return st, seg[:ns.value].copy(), first[:nc.value + 1].copy()


def okvq_plan_decode_work(unit_pages, max_ctas: int, bits: int):
    """The split okvq_decode uses. Returns (status, segments [n][4] = (unit, first page,
    end page, partial slot), cta_first [ctas + 1], unit_first [units + 1])."""
    p = np.ascontiguousarray(np.asarray(unit_pages, np.int64))
    units = p.shape[0]
    seg = np.zeros((units + max(max_ctas, 1) + 1, 4), np.int32)
    first = np.zeros(max(max_ctas, 1) + 1, np.int32)
    ufirst = np.zeros(units + 1, np.int32)
    nc, ns = ctypes.c_int32(), ctypes.c_int32()
    st = load().okvq_plan_decode_work(p.ctypes.data_as(ctypes.c_void_p) if units else None, units, max_ctas, bits,
                                      seg.ctypes.data_as(ctypes.c_void_p), first.ctypes.data_as(ctypes.c_void_p),
                                      ufirst.ctypes.data_as(ctypes.c_void_p), ctypes.byref(nc), ctypes.byref(ns))
    return st, seg[:ns.value].copy(), first[:nc.value + 1].copy(), ufirst


def okvq_compact(h, session: int, min_pages_saved: int, stream: int = 0):
    """Returns (status, new_length, moved_granules)."""
    nl, nm = ctypes.c_int64(), ctypes.c_int32()
    st = load().okvq_compact(h, session, min_pages_saved, ctypes.byref(nl), ctypes.byref(nm), ctypes.c_void_p(stream))
    return st, nl.value, nm.value


def okvq_test_fail_alloc(n: int) -> int:
    return load().okvq_test_fail_alloc(n)


def okvq_status_string(s: int) -> str:
    return status_string(s)


# ---- torch-facing wrapper ----

def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class Cache:
    """A multi-session 2/4-bit omni KV cache on the current CUDA device."""

    def __init__(self, num_sessions: int, num_layers: int, num_q_heads: int, num_kv_heads: int, max_tokens: int,
                 value_rot: np.ndarray, head_dim: int = 128, group_size: int = 32, bits: int = 2,
                 num_modalities: int = 3, hadamard_seed: int = 0, codebook: Optional[np.ndarray] = None,
                 stream=None, key_codec: int = OKVQ_KEYS_GROUP_RANGE):
        self._h = None
        R = np.ascontiguousarray(value_rot, dtype=np.float32)
        expect = (num_layers, num_kv_heads, num_modalities, head_dim, head_dim)
        if R.shape != expect:
            raise ValueError("value_rot must have shape %s, got %s" % (expect, R.shape))
        self._R = R
        cb = None
        if codebook is not None:
            cb = np.ascontiguousarray(codebook, dtype=np.float32)
            self._cb = cb
        cfg = OkvqConfig(num_sessions, num_layers, num_q_heads, num_kv_heads, head_dim, group_size, bits,
                         num_modalities, max_tokens, hadamard_seed & ((1 << 64) - 1),
                         cb.ctypes.data_as(ctypes.POINTER(ctypes.c_float)) if cb is not None else None,
                         R.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), int(key_codec))
        st, h = okvq_create(cfg, _stream_handle(stream))
        _check(st, "okvq_create")
        self._h = h
        self.num_sessions, self.num_layers = num_sessions, num_layers
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, num_kv_heads, head_dim
        self.group_size, self.bits, self.num_modalities, self.max_tokens = group_size, bits, num_modalities, max_tokens
        self.key_codec = int(key_codec)

    def close(self):
        if self._h is not None:
            okvq_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, session: int, k, v, modality, stream=None):
        """k, v: cuda fp16 [T][L][Hkv][128]; modality: cuda uint8 [T]."""
        import torch
        T = int(modality.shape[0])
        shp = (T, self.num_layers, self.num_kv_heads, self.head_dim)
        for name, x, dt in (("k", k, torch.float16), ("v", v, torch.float16)):
            if tuple(x.shape) != shp or x.dtype != dt or not x.is_cuda or not x.is_contiguous():
                raise ValueError("%s must be a contiguous cuda fp16 tensor of shape %s" % (name, shp))
        if modality.dtype != torch.uint8 or not modality.is_cuda or not modality.is_contiguous():
            raise ValueError("modality must be a contiguous cuda uint8 tensor")
        st = okvq_append_chunk(self._h, session, k.data_ptr(), v.data_ptr(), modality.data_ptr(), T,
                               _stream_handle(stream))
        _check(st, "okvq_append_chunk")

    def decode(self, q, out=None, stream=None):
        """q: cuda fp16 [S][L][Hq][128] -> out (same shape, fp16)."""
        import torch
        shp = (self.num_sessions, self.num_layers, self.num_q_heads, self.head_dim)
        if tuple(q.shape) != shp or q.dtype != torch.float16 or not q.is_cuda or not q.is_contiguous():
            raise ValueError("q must be a contiguous cuda fp16 tensor of shape %s" % (shp,))
        if out is None:
            out = torch.empty_like(q)
        st = okvq_decode(self._h, q.data_ptr(), out.data_ptr(), _stream_handle(stream))
        _check(st, "okvq_decode")
        return out

    def decode_host(self, q_host, out_host, stream=None):
        """okvq_decode_host: q_host, out_host are CPU fp16 tensors [S][L][Hq][128]
        (pinned for asynchronous copies); the call returns before the copies finish."""
        import torch
        shp = (self.num_sessions, self.num_layers, self.num_q_heads, self.head_dim)
        for name, x in (("q_host", q_host), ("out_host", out_host)):
            if tuple(x.shape) != shp or x.dtype != torch.float16 or x.is_cuda or not x.is_contiguous():
                raise ValueError("%s must be a contiguous CPU fp16 tensor of shape %s" % (name, shp))
        _check(okvq_decode_host(self._h, q_host.data_ptr(), out_host.data_ptr(), _stream_handle(stream)),
               "okvq_decode_host")
        return out_host

    def decode_static_scratch(self, q, out, stream=None):
        """okvq_decode_static_scratch: as decode, with the split-K partials in the
        library's one static device array (shared by all calls; see include/okvq.h).
        `out` must be given: the call allocates nothing."""
        import torch
        shp = (self.num_sessions, self.num_layers, self.num_q_heads, self.head_dim)
        for name, x in (("q", q), ("out", out)):
            if tuple(x.shape) != shp or x.dtype != torch.float16 or not x.is_cuda or not x.is_contiguous():
                raise ValueError("%s must be a contiguous cuda fp16 tensor of shape %s" % (name, shp))
        st = okvq_decode_static_scratch(self._h, q.data_ptr(), out.data_ptr(), _stream_handle(stream))
        _check(st, "okvq_decode_static_scratch")
        return out

    def length(self, session: int) -> int:
        st, n = okvq_length(self._h, session)
        _check(st, "okvq_length")
        return n

    def decode_pseudo(self, q, far_k, far_v, far_mass, tokens_per_prototype: int, out=None, stream=None):
        """Decode with far-memory pseudo tokens: far_k, far_v cuda fp16 [S][L][Hkv][P*Sp][128],
        far_mass cuda fp32 [S][L][Hkv][P] (Sp = tokens_per_prototype)."""
        import torch
        qs = (self.num_sessions, self.num_layers, self.num_q_heads, self.head_dim)
        if tuple(q.shape) != qs or q.dtype != torch.float16 or not q.is_cuda or not q.is_contiguous():
            raise ValueError("q must be a contiguous cuda fp16 tensor of shape %s" % (qs,))
        shp = (self.num_sessions, self.num_layers, self.num_kv_heads)
        P = int(far_mass.shape[-1])
        for t, dt, shape in ((far_k, torch.float16, shp + (P * tokens_per_prototype, self.head_dim)),
                             (far_v, torch.float16, shp + (P * tokens_per_prototype, self.head_dim)),
                             (far_mass, torch.float32, shp + (P,))):
            if not t.is_cuda or t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError("pseudo-token tensor must be a contiguous cuda %s tensor %s" % (dt, shape))
        if out is None:
            out = torch.empty_like(q)
        _check(okvq_decode_pseudo(self._h, q.data_ptr(), far_k.data_ptr(), far_v.data_ptr(), far_mass.data_ptr(), P,
                                  tokens_per_prototype, out.data_ptr(), _stream_handle(stream)), "okvq_decode_pseudo")
        return out

    def live_length(self, session: int) -> int:
        st, n = okvq_live_length(self._h, session)
        _check(st, "okvq_live_length")
        return n

    def evict(self, session: int, ranges, stream=None) -> None:
        """Delete [begin, end) slot ranges of a session (holes that decode skips)."""
        _check(okvq_evict(self._h, session, ranges, _stream_handle(stream)), "okvq_evict")

    def compaction_granule(self) -> int:
        st, n = okvq_compaction_granule(self._h)
        _check(st, "okvq_compaction_granule")
        return n

    def compact(self, session: int, min_pages_saved: int = 1, stream=None):
        """Ordered-suffix compaction; returns (new_length, moved_granules)."""
        st, nl, nm = okvq_compact(self._h, session, min_pages_saved, _stream_handle(stream))
        _check(st, "okvq_compact")
        return nl, nm

    def codebook(self):
        n = 1 << self.bits
        lv = (ctypes.c_float * n)()
        kl = (ctypes.c_float * n)()
        _check(load().okvq_codebook(self._h, lv, kl), "okvq_codebook")
        return np.array(lv[:], np.float32), np.array(kl[:], np.float32)

    def check_errors(self, stream=None) -> int:
        w = ctypes.c_uint32()
        st = load().okvq_check_errors(self._h, ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(w))
        if st not in (OKVQ_OK, OKVQ_ESTATE):
            _check(st, "okvq_check_errors")
        return int(w.value)

    def profile_enable(self, on: bool = True):
        _check(load().okvq_profile_enable(self._h, int(on)), "okvq_profile_enable")

    def profile_read(self, cap: int = 4096):
        a = (ctypes.c_float * cap)()
        b = (ctypes.c_float * cap)()
        n = ctypes.c_int32()
        _check(load().okvq_profile_read(self._h, a, b, cap, ctypes.byref(n)), "okvq_profile_read")
        return np.array(a[:n.value]), np.array(b[:n.value])

    def export_state(self, session: int) -> dict:
        """Canonical state of one session (layout documented in include/okvq.h)."""
        L = load()
        nbytes = ctypes.c_size_t(0)
        _check(L.okvq_export_state(self._h, session, None, ctypes.byref(nbytes)), "okvq_export_state")
        buf = np.zeros(nbytes.value, np.uint8)
        _check(L.okvq_export_state(self._h, session, buf.ctypes.data_as(ctypes.c_void_p), ctypes.byref(nbytes)),
               "okvq_export_state")
        T = self.length(session)
        G, d = self.group_size, self.head_dim
        turbo = self.key_codec == OKVQ_KEYS_TURBOQUANT
        Tf = T if turbo else (T // G) * G
        B = d * self.bits // 8
        LH = (self.num_layers, self.num_kv_heads)
        out, off = {}, 0

        def take(name, count, dtype, shape):
            nonlocal off
            nb = count * np.dtype(dtype).itemsize
            out[name] = buf[off:off + nb].view(dtype).reshape(shape)
            off += nb

        n = LH[0] * LH[1]
        take("kcodes", n * Tf * B, np.uint8, (*LH, Tf, B))
        if turbo:
            take("knorm", n * T, np.float16, (*LH, T))
        else:
            take("kstats", n * (Tf // G) * 2 * d, np.float16, (*LH, Tf // G, 2, d))
            take("ktail", n * (T - Tf) * d, np.float16, (*LH, T - Tf, d))
        take("vcodes", n * T * B, np.uint8, (*LH, T, B))
        take("vnorm", n * T, np.float16, (*LH, T))
        take("mod", T, np.uint8, (T,))
        take("dead", n * T, np.uint8, (*LH, T))
        out["dead"] = out["dead"].astype(bool)
        return out
