"""Seeded synthetic omni-modal KV streams.

This module only draws inputs: fp16 keys/values shaped like a streaming
omni-modal model's per-chunk KV, per-token modality ids, decode queries and
the per-modality value rotations that the codec takes as a parameter.  It
holds none of the codec's arithmetic (no Hadamard transform, no codebook, no
quantization, no attention); both the CUDA path and the CPU oracle consume
what it returns.

Modality ids: 0 video, 1 audio, 2 text (the unit layout of an omni stream,
OmniTide section 4, puts the image/video span, then the audio span, then text
inside each unit).

Recipe (every draw comes from a PCG64 stream keyed by (seed, purpose, ...)
through ``numpy.random.SeedSequence``, so any session/layer can be rebuilt
alone and the result does not depend on generation order):

* per (layer, kv head): per-channel key and value scales, log-uniform in
  [0.5, 4]; per-modality value means ~ N(0, 1) per channel;
* keys   K[t] = kscale * z + drift[t],  z ~ N(0, 1), drift a per-channel
  Gaussian random walk with step 0.02 per token (temporal key drift);
* values V[t] = vscale * z + mu[mod[t]];
* queries ~ N(0, 1);
* calibration slice: a separate 512-token stream of values drawn the same
  way (interleave 64 video / 25 audio / 8 text, its own PCG64 stream per
  layer).  The per-modality value rotations are calibrated from it (by the
  library's calibration kernel, or by the CPU oracle in the tests); this
  module computes no rotation itself.

Everything is cast to fp16 once (the values the codec reads).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

MOD_VIDEO, MOD_AUDIO, MOD_TEXT = 0, 1, 2
NUM_MODALITIES = 3
CALIB_TOKENS = 512
DRIFT_STEP = 0.02
SCALE_LO, SCALE_HI = 0.5, 4.0

_PURPOSE = {"params": 1, "kv": 2, "calib": 3, "query": 4, "plan": 5, "far": 6}


def _rng(seed: int, purpose: str, *ids: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), _PURPOSE[purpose], *map(int, ids)])))


@dataclass(frozen=True)
class Shape:
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int = 128
    group_size: int = 32
    bits: int = 2
    num_modalities: int = NUM_MODALITIES

    @property
    def q_per_kv(self) -> int:
        return self.num_q_heads // self.num_kv_heads


@dataclass
class Session:
    """One stream: the chunks it is appended in and their modality ids."""
    chunks: List[np.ndarray]          # each a uint8 modality array (one append call)

    @property
    def length(self) -> int:
        return int(sum(len(c) for c in self.chunks))

    def modality(self) -> np.ndarray:
        if not self.chunks:
            return np.zeros(0, np.uint8)
        return np.concatenate(self.chunks).astype(np.uint8)

    def chunk_bounds(self) -> List[tuple]:
        out, t = [], 0
        for c in self.chunks:
            out.append((t, t + len(c)))
            t += len(c)
        return out


def retention_ranges(session: "Session", keep_recent: int = 4, sinks=(64, 8, None)) -> List[tuple]:
    """Token ranges a unit-aware retention policy would delete (the shape of
    OmniPick's plans, "OmniTide" section 5.1; the policy itself is not part of
    this library): every chunk but the last ``keep_recent`` keeps, of each run of
    one modality, only its first sinks[m] tokens (None: the whole run); the rest
    of the run is one deletion range."""
    out = []
    mod = session.modality()
    bounds = session.chunk_bounds()
    for a, b in bounds[:max(0, len(bounds) - keep_recent)]:
        t = a
        while t < b:
            e = t
            while e < b and mod[e] == mod[t]:
                e += 1
            k = sinks[mod[t]]
            if k is not None and t + k < e:
                out.append((t + k, e))
            t = e
    return out


def interleave_pattern(period: Sequence[tuple], total: int) -> np.ndarray:
    """Repeat blocks [(modality, count), ...] until ``total`` tokens."""
    block = np.concatenate([np.full(n, m, np.uint8) for m, n in period])
    reps = -(-total // len(block))
    return np.tile(block, reps)[:total]


def chunked_stream(video: int, audio: int, text: int, text_every: int, total: int) -> List[np.ndarray]:
    """1-s chunks of [video, audio]; a text turn joins every ``text_every``-th chunk."""
    chunks, t, i = [], 0, 0
    while t < total:
        parts = [np.full(video, MOD_VIDEO, np.uint8), np.full(audio, MOD_AUDIO, np.uint8)]
        i += 1
        if text and text_every and i % text_every == 0:
            parts.append(np.full(text, MOD_TEXT, np.uint8))
        c = np.concatenate(parts)[: total - t]
        chunks.append(c)
        t += len(c)
    return chunks


@dataclass
class Workload:
    name: str
    shape: Shape
    sessions: List[Session]
    seed: int
    hadamard_seed: int
    max_tokens: int
    _param_cache: dict = field(default_factory=dict, repr=False)

    # ---- model-level parameters (shared by all sessions) ----
    def layer_params(self, layer: int):
        if layer not in self._param_cache:
            sh = self.shape
            r = _rng(self.seed, "params", layer)
            lo, hi = math.log(SCALE_LO), math.log(SCALE_HI)
            kscale = np.exp(r.uniform(lo, hi, (sh.num_kv_heads, sh.head_dim))).astype(np.float32)
            vscale = np.exp(r.uniform(lo, hi, (sh.num_kv_heads, sh.head_dim))).astype(np.float32)
            mu = r.standard_normal((sh.num_modalities, sh.num_kv_heads, sh.head_dim), dtype=np.float32)
            self._param_cache[layer] = (kscale, vscale, mu)
        return self._param_cache[layer]

    # ---- per-session KV ----
    def layer_kv(self, session: int, layer: int):
        """fp16 K, V of one layer for the whole session: [T][Hkv][d] each."""
        sh = self.shape
        mod = self.sessions[session].modality()
        T = len(mod)
        kscale, vscale, mu = self.layer_params(layer)
        r = _rng(self.seed, "kv", session, layer)
        shp = (T, sh.num_kv_heads, sh.head_dim)
        zk = r.standard_normal(shp, dtype=np.float32)
        steps = r.standard_normal(shp, dtype=np.float32)
        zv = r.standard_normal(shp, dtype=np.float32)
        drift = np.cumsum(steps * np.float32(DRIFT_STEP), axis=0, dtype=np.float32)
        K = (kscale[None] * zk + drift).astype(np.float16)
        V = (vscale[None] * zv + mu[mod]).astype(np.float16)
        return K, V

    def session_kv(self, session: int, layers: Optional[Sequence[int]] = None):
        """fp16 K, V [T][L'][Hkv][d] for the listed layers (default: all)."""
        layers = list(range(self.shape.num_layers)) if layers is None else list(layers)
        T = self.sessions[session].length
        sh = self.shape
        K = np.empty((T, len(layers), sh.num_kv_heads, sh.head_dim), np.float16)
        V = np.empty_like(K)
        for i, l in enumerate(layers):
            K[:, i], V[:, i] = self.layer_kv(session, l)
        return K, V

    # ---- decode queries ----
    def queries(self, step: int = 0) -> np.ndarray:
        sh = self.shape
        r = _rng(self.seed, "query", step)
        q = r.standard_normal((len(self.sessions), sh.num_layers, sh.num_q_heads, sh.head_dim), dtype=np.float32)
        return q.astype(np.float16)

    # ---- far-memory pseudo tokens (input of the pseudo-token decode) ----
    def pseudo_tokens(self, num_prototypes: int, per_proto: int, inactive: float = 0.1):
        """Pseudo tokens shaped like a prototype bank's: for every (session, layer,
        kv head), prototype centres drawn like the layer's keys and values, and
        per_proto tokens per prototype = centre + small residual modes (0.25 of
        the channel scale). Masses log-uniform in [1, 300], rounded, with about
        ``inactive`` of the prototypes at 0. Returns fp16 K, V
        [S][L][Hkv][P*per_proto][d] and fp32 masses [S][L][Hkv][P]."""
        sh = self.shape
        S, P = len(self.sessions), num_prototypes
        shp = (S, sh.num_layers, sh.num_kv_heads)
        K = np.empty(shp + (P * per_proto, sh.head_dim), np.float16)
        V = np.empty_like(K)
        mass = np.empty(shp + (P,), np.float32)
        for s in range(S):
            for l in range(sh.num_layers):
                kscale, vscale, _ = self.layer_params(l)
                r = _rng(self.seed, "far", s, l)
                for h in range(sh.num_kv_heads):
                    ck = kscale[h] * r.standard_normal((P, sh.head_dim), dtype=np.float32)
                    cv = vscale[h] * r.standard_normal((P, sh.head_dim), dtype=np.float32)
                    rk = 0.25 * kscale[h] * r.standard_normal((P * per_proto, sh.head_dim), dtype=np.float32)
                    rv = 0.25 * vscale[h] * r.standard_normal((P * per_proto, sh.head_dim), dtype=np.float32)
                    K[s, l, h] = (np.repeat(ck, per_proto, axis=0) + rk).astype(np.float16)
                    V[s, l, h] = (np.repeat(cv, per_proto, axis=0) + rv).astype(np.float16)
                    n = np.round(np.exp(r.uniform(0.0, math.log(300.0), P)))
                    n[r.random(P) < inactive] = 0.0
                    mass[s, l, h] = n
        return K, V, mass

    # ---- calibration slice (input of the value-rotation calibration) ----
    def calibration_slice(self, layers: Optional[Sequence[int]] = None):
        """fp16 values [CALIB_TOKENS][L'][Hkv][d] of the calibration slice and its
        modality ids [CALIB_TOKENS] (interleave 64 video / 25 audio / 8 text)."""
        sh = self.shape
        layers = list(range(sh.num_layers)) if layers is None else list(layers)
        mod = interleave_pattern([(MOD_VIDEO, 64), (MOD_AUDIO, 25), (MOD_TEXT, 8)], CALIB_TOKENS)
        V = np.empty((CALIB_TOKENS, len(layers), sh.num_kv_heads, sh.head_dim), np.float16)
        for i, l in enumerate(layers):
            _, vscale, mu = self.layer_params(l)
            r = _rng(self.seed, "calib", l)
            z = r.standard_normal((CALIB_TOKENS, sh.num_kv_heads, sh.head_dim), dtype=np.float32)
            V[:, i] = (vscale[None] * z + mu[mod]).astype(np.float16)
        return V, mod


# ---------------------------------------------------------------------------
# the workloads (shapes and token streams)
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, tokens: int = 2048, bits: int = 2, group_size: int = 32) -> Workload:
    """1 layer, 8 q / 2 kv heads, d 128, 2,048 tokens of [64 v, 25 a, 8 t]."""
    sh = Shape(1, 8, 2, 128, group_size, bits)
    mod = interleave_pattern([(MOD_VIDEO, 64), (MOD_AUDIO, 25), (MOD_TEXT, 8)], tokens)
    return Workload("tiny", sh, [Session([mod])], seed, 0x5EED0000 + seed, tokens)


def qwen3b(seed: int = 1, tokens: int = 32768, layers: int = 36, bits: int = 2, group_size: int = 32) -> Workload:
    """Qwen2.5-Omni-3B-shaped decode: 36 L, 16 q / 2 kv heads, 1-s chunks [640 v, 25 a] + 32 t every 30 chunks."""
    sh = Shape(layers, 16, 2, 128, group_size, bits)
    chunks = chunked_stream(640, 25, 32, 30, tokens)
    return Workload("qwen2.5-omni-3b", sh, [Session(chunks)], seed, 0x5EED0000 + seed, tokens)


def qwen7b(seed: int = 2, tokens: int = 81920, layers: int = 28, bits: int = 2, group_size: int = 32) -> Workload:
    """Qwen2.5-Omni-7B-shaped long stream: 28 L, 28 q / 4 kv heads, [1280 v, 25 a] + 16 t every 30 chunks."""
    sh = Shape(layers, 28, 4, 128, group_size, bits)
    chunks = chunked_stream(1280, 25, 16, 30, tokens)
    return Workload("qwen2.5-omni-7b", sh, [Session(chunks)], seed, 0x5EED0000 + seed, tokens)


def streaming(seed: int = 3, tokens: int = 131072, layers: int = 36, bits: int = 2, group_size: int = 32) -> Workload:
    """Config-1 shape; 1-s chunks of [2304 v, 25 a] appended up to 131,072 tokens."""
    sh = Shape(layers, 16, 2, 128, group_size, bits)
    chunks = chunked_stream(2304, 25, 0, 0, tokens)
    return Workload("streaming", sh, [Session(chunks)], seed, 0x5EED0000 + seed, tokens)


def multisession(seed: int = 4, sessions: int = 64, lo: int = 4096, hi: int = 65536, layers: int = 36,
                 bits: int = 2, group_size: int = 32) -> Workload:
    """64 independent sessions, config-1 heads, lengths U[4096, 65536], per-session interleave."""
    sh = Shape(layers, 16, 2, 128, group_size, bits)
    plan = _rng(seed, "plan")
    out = []
    for s in range(sessions):
        T = int(plan.integers(lo, hi + 1))
        r = _rng(seed, "plan", s + 1)
        video = int(r.choice([640, 1280, 2304]))
        every = int(r.integers(10, 51))
        chunks, t, i = [], 0, 0
        while t < T:
            parts = [np.full(video, MOD_VIDEO, np.uint8), np.full(25, MOD_AUDIO, np.uint8)]
            i += 1
            if i % every == 0:
                parts.append(np.full(int(r.integers(16, 33)), MOD_TEXT, np.uint8))
            c = np.concatenate(parts)[: T - t]
            chunks.append(c)
            t += len(c)
        out.append(Session(chunks))
    return Workload("multisession", sh, out, seed, 0x5EED0000 + seed, hi)


WORKLOADS = {"tiny": tiny, "qwen3b": qwen3b, "qwen7b": qwen7b, "streaming": streaming, "multisession": multisession}
