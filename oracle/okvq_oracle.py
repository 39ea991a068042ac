"""CPU oracle for the OmniKVQuant-style 2/4-bit omni KV cache (TEST INFRASTRUCTURE).

This module is the slow, plain reference that the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` may import it; the library and its
binding never do, and it shares no code with them.

Source: "OmniKVQuant: KV Cache Quantization for Omni-LLMs" (paperlayer.ai
summary), section 2 METHOD (TurboQuant bullet: magnitude/direction split,
randomized Hadamard transform, fixed codebook; OmniKVQuant bullets: min-max
scaling of rotated keys over short consecutive-token groups with stored group
statistics, shared fixed codebook; per-modality eigenbasis rotation of values)
and section 1 INTRODUCTION, Implementation bullet (rotate the query once per
head, unpack the 2-bit cache inside attention, batch the inverse value
rotations after aggregation).

Arithmetic is fp64 except where the method's decisions are fixed in a
narrower precision so that both sides decide identically:

* the key Hadamard rotation is the canonical fp32 butterfly (stride 1, 2, ...,
  d/2; a+b / a-b, round-to-nearest, no fused multiply-add) followed by one
  fp32 multiply by fp32(1/sqrt(d));
* key group statistics are the group minimum and range, both fp16: the minimum
  rounded toward -inf, the range (max - stored min, exact) rounded toward +inf,
  so the stored interval [mn, mn + rg] contains every member;
* the key code decision is u = (k' - mn) / rg in fp32, compared with fp32
  midpoint thresholds (ties go to the lower code);
* the value code decision compares fp32(w) with fp32 thresholds, w computed
  in fp64; codes whose fp64 w lies within 1e-5 of a threshold are flagged as
  boundary codes (another correct implementation may round them the other way).

Eviction and compaction ("OmniTide: Co-Designing Algorithms and Systems for
Efficient On-Device Omni-LLM Streaming", section 5.2 Applying the retention
plan, section 6.2 Selective and efficient KV migration): deleted token ranges
stay in their slots as holes that attention skips; the ordered-suffix mode
packs the surviving entries of the shortest suffix that shortens the
page-rounded span by enough pages, preserving their order.  Here the unit that
moves is a key group (its statistics serve all its members) or, for TurboQuant
keys, a 16-token tile.

Far memory ("ProtoKV: Streaming Video Understanding under Delayed Query with
Summary-State Memory", section 3.3 Eq. (2) and Algorithm 4): pseudo tokens
synthesized by the caller join the softmax with the additive log-mass bias
log n_k of their prototype; the near window is this cache.

TurboQuant key codec (the pages' comparison point, ``key_codec="turbo"``):
every key is coded on arrival like a value, with the shared randomized Hadamard
rotation instead of a modality eigenbasis (norm, direction rotated, fixed
codebook, one global scale); no group statistics and no fp16 tail.  Value
rotations are whatever the caller passes (the Hadamard rotation for every
modality reproduces TurboQuant's single shared value rotation).

Readings where the page is silent (codebook = Lloyd-Max levels for N(0,1)
rounded once to fp16; keys use those levels renormalised to [0, 1]; values
quantize sqrt(d) * R_m * v/|v| against the levels directly; groups aligned to
absolute token index, an incomplete trailing key group kept in fp16 and
attended exactly; one shared softmax over all tokens with per-modality value
accumulators) are the ones listed with each function below.

Parity pins: every function here is pinned by tests/test_oracle_pins.py to
closed forms, textbook values (Max 1960), the published SplitMix64 output,
brute force on tiny inputs and invariants; none is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

F16, F32, F64 = np.float16, np.float32, np.float64
BOUNDARY_BAND = 1e-5          # codes whose pre-quantization value is this close to a threshold
NORM_BAND_REL = 4e-6          # fp16 norms whose fp64 value is this close (relative) to a rounding midpoint

# ---------------------------------------------------------------------------
# randomized Hadamard transform (section 2, TurboQuant bullet)
# ---------------------------------------------------------------------------

_M64 = (1 << 64) - 1


def splitmix64(seed: int, n: int) -> list:
    """SplitMix64 (Steele, Lea, Flood 2014; Vigna's reference form): n outputs."""
    x = seed & _M64
    out = []
    for _ in range(n):
        x = (x + 0x9E3779B97F4A7C15) & _M64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        out.append(z ^ (z >> 31))
    return out


def hadamard_signs(seed: int, d: int) -> np.ndarray:
    """Random +-1 diagonal D of the RHT: bit c of the SplitMix64 stream, 1 -> -1."""
    words = splitmix64(seed, (d + 63) // 64)
    bits = [(words[c // 64] >> (c % 64)) & 1 for c in range(d)]
    return np.array([-1 if b else 1 for b in bits], dtype=np.int8)


def sylvester_hadamard(d: int) -> np.ndarray:
    """Unnormalised Sylvester Hadamard matrix, H[i, j] = (-1)^popcount(i & j)."""
    i = np.arange(d)
    pc = np.vectorize(lambda x: bin(x).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def fwht(x: np.ndarray, dtype=F64) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform along the last axis.

    Butterfly stages with stride 1, 2, 4, ..., d/2 in that order; at each stage
    the pair (i, i+stride) with bit ``stride`` of i clear becomes
    (x_i + x_{i+stride}, x_i - x_{i+stride}) in ``dtype`` arithmetic.  With
    dtype=float32 this is the canonical fp32 key rotation order.
    """
    x = np.array(x, dtype=dtype, copy=True)
    d = x.shape[-1]
    lead = x.shape[:-1]
    s = 1
    while s < d:
        y = x.reshape(*lead, d // (2 * s), 2, s)
        a = y[..., 0, :].copy()
        b = y[..., 1, :]
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        x = y.reshape(*lead, d)
        s *= 2
    return x


def rotate_keys_f32(k16: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """k' = fp32(1/sqrt(d)) * FWHT_fp32(s o k) for fp16 keys [..., d]."""
    d = k16.shape[-1]
    x = k16.astype(F32) * signs.astype(F32)          # exact sign flips
    y = fwht(x, F32)
    return (y * F32(1.0 / math.sqrt(d))).astype(F32)


def rotate_f64(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """(1/sqrt(d)) H D x in fp64 (used for the query, D1)."""
    d = x.shape[-1]
    return fwht(np.asarray(x, F64) * signs.astype(F64), F64) / math.sqrt(d)


def hadamard_rotation(signs: np.ndarray) -> np.ndarray:
    """The randomized Hadamard rotation (1/sqrt d) H D as an orthogonal matrix (rows = basis)."""
    d = len(signs)
    return sylvester_hadamard(d).astype(F64) * signs.astype(F64)[None, :] / math.sqrt(d)


# ---------------------------------------------------------------------------
# fixed shared codebook (section 2; reading: Lloyd-Max quantizer of N(0,1))
# ---------------------------------------------------------------------------

def _phi(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi) if math.isfinite(x) else 0.0


def _Phi(x):
    if x == math.inf:
        return 1.0
    if x == -math.inf:
        return 0.0
    return 0.5 * math.erfc(-x / math.sqrt(2.0))


def gaussian_cell_mean(a: float, b: float) -> float:
    """E[X | a < X <= b] for X ~ N(0, 1) (closed form (phi(a) - phi(b)) / (Phi(b) - Phi(a)))."""
    return (_phi(a) - _phi(b)) / (_Phi(b) - _Phi(a))


def lloyd_max_gaussian(n_levels: int, iters: int = 200000, tol: float = 1e-15) -> np.ndarray:
    """Lloyd-Max (Max 1960) levels for N(0,1): alternate midpoint thresholds and cell means."""
    lv = np.linspace(-2.0, 2.0, n_levels) * (1.0 if n_levels > 2 else 0.8)
    for _ in range(iters):
        th = [-math.inf] + [0.5 * (lv[j] + lv[j + 1]) for j in range(n_levels - 1)] + [math.inf]
        new = np.array([gaussian_cell_mean(th[j], th[j + 1]) for j in range(n_levels)])
        if np.max(np.abs(new - lv)) < tol:
            lv = new
            break
        lv = new
    return lv


@dataclass
class Codebook:
    bits: int
    levels16: np.ndarray      # fp16 value levels l_j (ascending) - these define the codebook
    levels: np.ndarray        # the same as fp64
    vthr: np.ndarray          # fp32 value thresholds: midpoints of adjacent fp16 levels
    ktab16: np.ndarray        # fp16 key levels lambda_j = (l_j - l_0) / (l_last - l_0), in [0, 1]
    ktab: np.ndarray          # the same as fp64
    kthr: np.ndarray          # fp32 key thresholds: midpoints of adjacent fp16 lambda_j


def make_codebook(bits: int, levels: Optional[np.ndarray] = None) -> Codebook:
    """Round the levels once to fp16; everything else is derived from those fp16 values."""
    n = 1 << bits
    lv = lloyd_max_gaussian(n) if levels is None else np.asarray(levels, F64)
    l16 = lv.astype(F16)
    l64 = l16.astype(F64)
    vthr = ((l64[:-1] + l64[1:]) / 2).astype(F32)
    lam = ((l64 - l64[0]) / (l64[-1] - l64[0])).astype(F16)
    lam64 = lam.astype(F64)
    kthr = ((lam64[:-1] + lam64[1:]) / 2).astype(F32)
    return Codebook(bits, l16, l64, vthr, lam, lam64, kthr)


def nearest_code(x32: np.ndarray, thr32: np.ndarray) -> np.ndarray:
    """Index of the nearest level: number of thresholds strictly below x (ties -> lower)."""
    x32 = np.asarray(x32, F32)
    c = np.zeros(x32.shape, np.uint8)
    for t in thr32:
        c += (x32 > t).astype(np.uint8)
    return c


def near_threshold(x64: np.ndarray, thr32: np.ndarray, band: float = BOUNDARY_BAND) -> np.ndarray:
    x64 = np.asarray(x64, F64)
    m = np.zeros(x64.shape, bool)
    for t in thr32.astype(F64):
        m |= np.abs(x64 - t) < band
    return m


# ---------------------------------------------------------------------------
# fp16 storage roundings
# ---------------------------------------------------------------------------

def f16_round_down(x32: np.ndarray) -> np.ndarray:
    h = np.asarray(x32, F32).astype(F16)
    over = h.astype(F32) > x32
    return np.where(over, np.nextafter(h, F16(-np.inf)), h).astype(F16)


def f16_round_up(x32: np.ndarray) -> np.ndarray:
    h = np.asarray(x32, F32).astype(F16)
    under = h.astype(F32) < x32
    return np.where(under, np.nextafter(h, F16(np.inf)), h).astype(F16)


def f16_near_midpoint(x64: np.ndarray, rel: float = NORM_BAND_REL) -> np.ndarray:
    """True where x is within ``rel`` (relative) of a midpoint between two fp16 values."""
    x64 = np.asarray(x64, F64)
    h = x64.astype(F16)
    lo = np.where(h.astype(F64) > x64, np.nextafter(h, F16(-np.inf)), h)
    hi = np.nextafter(lo, F16(np.inf))
    mid = (lo.astype(F64) + hi.astype(F64)) / 2
    return np.abs(x64 - mid) <= rel * np.maximum(np.abs(x64), 1e-30)


# ---------------------------------------------------------------------------
# append-time quantization (section 2, OmniKVQuant bullets)
# ---------------------------------------------------------------------------

def f16_round_up_f64(x64: np.ndarray) -> np.ndarray:
    """Smallest fp16 >= x (x given exactly in fp64)."""
    x64 = np.asarray(x64, F64)
    h = x64.astype(F16)
    return np.where(h.astype(F64) < x64, np.nextafter(h, F16(np.inf)), h).astype(F16)


def quantize_key_group(kp32: np.ndarray, cb: Codebook):
    """One group of G consecutive rotated keys kp32 [G][d] (fp32).

    Per channel the group statistics are mn = min over the group rounded down
    to fp16 and rg = (max - mn) rounded up to fp16, so [mn, mn + rg] contains
    every member; u = (k' - mn) / rg in fp32; code = nearest normalized key
    level.  rg == 0 gives code 0.
    Returns mn16 [d], rg16 [d], codes [G][d], boundary mask [G][d].
    """
    mn = f16_round_down(kp32.min(axis=0))
    rg = f16_round_up_f64(kp32.max(axis=0).astype(F64) - mn.astype(F64))
    mn32, rg32 = mn.astype(F32), rg.astype(F32)
    flat = rg32 == 0
    safe = np.where(flat, F32(1), rg32).astype(F32)
    u = ((kp32 - mn32[None]).astype(F32) / safe[None]).astype(F32)
    codes = nearest_code(u, cb.kthr)
    codes[:, flat] = 0
    bnd = near_threshold(u, cb.kthr)
    bnd[:, flat] = False
    return mn, rg, codes, bnd


def quantize_values(v16: np.ndarray, R: np.ndarray, cb: Codebook):
    """Values v16 [n][d] of ONE modality with its rotation R [d][d] (rows = basis).

    n = |v| (fp64) stored fp16 round-to-nearest-even; u = v/n (0 when n = 0);
    w = sqrt(d) * R u; code_c = nearest level of the value table for w_c.
    Returns norm16 [n], codes [n][d], code boundary mask [n][d], norm boundary mask [n].
    """
    d = v16.shape[-1]
    v = v16.astype(F64)
    n = np.sqrt(np.sum(v * v, axis=-1))
    u = np.where(n[:, None] > 0, v / np.where(n > 0, n, 1.0)[:, None], 0.0)
    w = math.sqrt(d) * (u @ np.asarray(R, F64).T)
    codes = nearest_code(w.astype(F32), cb.vthr)
    bnd = near_threshold(w, cb.vthr)
    return n.astype(F16), codes, bnd, f16_near_midpoint(n)


def quantize_keys_turbo(k16: np.ndarray, signs: np.ndarray, cb: Codebook):
    """TurboQuant keys (section 2 METHOD, TurboQuant bullet): the magnitude n = |k|
    is split from the direction, the direction is rotated by the randomized Hadamard
    transform toward Gaussian-like coordinates and coded with the fixed codebook, one
    global scale for every token (no per-window ranges).  Reading: exactly the value
    codec with the shared rotation R = (1/sqrt d) H D, so w = sqrt(d) R k/|k| is
    coded against the same levels.  Returns norm16, codes, code boundary mask, norm
    boundary mask, like quantize_values.
    """
    return quantize_values(k16, hadamard_rotation(signs), cb)


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Canonical packing along the last axis: 2-bit channel c at byte c//4 bits 2(c%4); 4-bit low nibble = even."""
    codes = np.asarray(codes, np.uint8)
    per = 8 // bits
    d = codes.shape[-1]
    c = codes.reshape(*codes.shape[:-1], d // per, per).astype(np.uint16)
    out = np.zeros(c.shape[:-1], np.uint16)
    for j in range(per):
        out |= c[..., j] << (bits * j)
    return out.astype(np.uint8)


def unpack_codes(packed: np.ndarray, bits: int) -> np.ndarray:
    per = 8 // bits
    p = np.asarray(packed, np.uint8)
    mask = (1 << bits) - 1
    parts = [(p >> (bits * j)) & mask for j in range(per)]
    return np.stack(parts, axis=-1).reshape(*p.shape[:-1], p.shape[-1] * per).astype(np.uint8)


class OracleUnit:
    """The cache of one (session, layer, kv head): append and decode, step by step."""

    def __init__(self, d: int, group_size: int, cb: Codebook, signs: np.ndarray, R: np.ndarray,
                 q_per_kv: int, capacity: int, key_codec: str = "omni"):
        if key_codec not in ("omni", "turbo"):
            raise ValueError("key_codec must be 'omni' (group min-max) or 'turbo' (norm + fixed scale)")
        self.key_codec = key_codec
        self.d, self.G, self.cb, self.signs = d, group_size, cb, signs
        self.R = np.asarray(R, F32)                  # [M][d][d] as given to the codec
        self.q_per_kv = q_per_kv
        cap = capacity
        self.T = 0
        self.kcodes = np.zeros((cap, d), np.uint8)
        self.kbnd = np.zeros((cap, d), bool)
        self.kmn = np.zeros((-(-cap // group_size), d), F16)
        self.krg = np.zeros_like(self.kmn)
        self.keys16 = np.zeros((cap, d), F16)          # fp16 inputs kept for the trailing (tail) group
        self.knorm = np.zeros(cap, F16)                # turbo keys: |k|
        self.knbnd = np.zeros(cap, bool)
        self.vcodes = np.zeros((cap, d), np.uint8)
        self.vbnd = np.zeros((cap, d), bool)
        self.vnorm = np.zeros(cap, F16)
        self.nbnd = np.zeros(cap, bool)
        self.mod = np.zeros(cap, np.uint8)
        self.dead = np.zeros(cap, bool)                # deleted tokens (holes left in place)

    @property
    def T_full(self) -> int:
        """Tokens whose keys are quantized (turbo keys are quantized on arrival)."""
        return self.T if self.key_codec == "turbo" else (self.T // self.G) * self.G

    def append(self, K16: np.ndarray, V16: np.ndarray, mod: np.ndarray):
        """Append n tokens: values quantized now; each key group once it is complete."""
        n = len(mod)
        t0, t1 = self.T, self.T + n
        if t1 > len(self.mod):
            raise ValueError("capacity exceeded")
        self.keys16[t0:t1] = K16
        self.mod[t0:t1] = mod
        for m in np.unique(mod):
            sel = np.nonzero(mod == m)[0]
            nrm, codes, bnd, nb = quantize_values(V16[sel], self.R[m], self.cb)
            self.vnorm[t0 + sel] = nrm
            self.vcodes[t0 + sel] = codes
            self.vbnd[t0 + sel] = bnd
            self.nbnd[t0 + sel] = nb
        if self.key_codec == "turbo":
            nrm, codes, bnd, nb = quantize_keys_turbo(K16, self.signs, self.cb)
            self.knorm[t0:t1], self.kcodes[t0:t1], self.kbnd[t0:t1], self.knbnd[t0:t1] = nrm, codes, bnd, nb
            self.T = t1
            return
        G = self.G
        for g in range(t0 // G, t1 // G):
            kp = rotate_keys_f32(self.keys16[g * G:(g + 1) * G], self.signs)
            mn, rg, codes, bnd = quantize_key_group(kp, self.cb)
            self.kmn[g], self.krg[g] = mn, rg
            self.kcodes[g * G:(g + 1) * G] = codes
            self.kbnd[g * G:(g + 1) * G] = bnd
        self.T = t1

    # ---- canonical state ----
    def export(self) -> dict:
        T, Tf, G = self.T, self.T_full, self.G
        b = self.cb.bits
        if self.key_codec == "turbo":
            return {
                "kcodes": pack_codes(self.kcodes[:T], b),
                "knorm": self.knorm[:T].copy(),
                "vcodes": pack_codes(self.vcodes[:T], b),
                "vnorm": self.vnorm[:T].copy(),
                "kbnd": self.kbnd[:T].copy(),
                "knbnd": self.knbnd[:T].copy(),
                "vbnd": self.vbnd[:T].copy(),
                "nbnd": self.nbnd[:T].copy(),
                "dead": self.dead[:T].copy(),
            }
        return {
            "kcodes": pack_codes(self.kcodes[:Tf], b),
            "kstats": np.stack([self.kmn[:Tf // G], self.krg[:Tf // G]], axis=1),   # [T/G][2][d] (min, range)
            "ktail": self.keys16[Tf:T].copy(),
            "vcodes": pack_codes(self.vcodes[:T], b),
            "vnorm": self.vnorm[:T].copy(),
            "kbnd": self.kbnd[:Tf].copy(),
            "vbnd": self.vbnd[:T].copy(),
            "nbnd": self.nbnd[:T].copy(),
            "dead": self.dead[:T].copy(),
        }

    # ---- decode (section 1 Implementation bullet) ----
    def decode(self, q16: np.ndarray) -> np.ndarray:
        """Fused-score decode of the q_per_kv heads [Gq][d] -> fp64 [Gq][d].

        q' = (1/sqrt d) H D q, scaled by the softmax factor 1/sqrt d.  A quantized
        token t in group g scores beta_g + sum_c (q'_c * rg_{g,c}) lambda(code);
        beta_g = sum_c q'_c mn_{g,c}.  A tail token scores q.k/sqrt d from its fp16 key.
        One softmax over all tokens; o_m accumulates p_t * n_t * l(vcode)/sqrt d in the
        rotated value domain of modality m; O = (sum_m R_m^T o_m) / sum p.
        """
        d, G, T, Tf = self.d, self.G, self.T, self.T_full
        Gq = q16.shape[0]
        out = np.zeros((Gq, d), F64)
        if T == 0:
            return out
        q = q16.astype(F64)
        qr = rotate_f64(q, self.signs) / math.sqrt(d)                       # [Gq][d]
        s = np.empty((Gq, T), F64)
        if self.key_codec == "turbo":
            # k' = (n / sqrt d) l(code) in the rotated domain: s_t = (n_t / sqrt d) q' . l(code_t)
            s[:] = (qr @ self.cb.levels[self.kcodes[:T]].T) * (self.knorm[:T].astype(F64) / math.sqrt(d))[None]
        elif Tf:
            ng = Tf // G
            mn = self.kmn[:ng].astype(F64)
            dl = self.krg[:ng].astype(F64)
            lam = self.cb.ktab[self.kcodes[:Tf]].reshape(ng, G, d)           # [g][t][c]
            beta = qr @ mn.T                                                 # [Gq][g]
            a = qr[:, None, :] * dl[None]                                    # [Gq][g][c]
            s[:, :Tf] = (beta[:, :, None] + np.einsum("hgc,gtc->hgt", a, lam)).reshape(Gq, Tf)
        if T > Tf:
            s[:, Tf:] = q @ self.keys16[Tf:T].astype(F64).T / math.sqrt(d)
        live = ~self.dead[:T]
        if not live.any():
            return out                                                      # nothing left to attend
        s[:, ~live] = -np.inf                                               # deleted tokens take no part
        mmax = s.max(axis=1, keepdims=True)
        p = np.exp(s - mmax)
        l = p.sum(axis=1)
        lv = self.cb.levels[self.vcodes[:T]] / math.sqrt(d)                  # [T][d]
        wv = lv * self.vnorm[:T].astype(F64)[:, None]
        R64 = self.R.astype(F64)
        for m in range(self.R.shape[0]):
            sel = self.mod[:T] == m
            if not sel.any():
                continue
            o_m = p[:, sel] @ wv[sel]                                        # [Gq][d] rotated domain
            out += o_m @ R64[m]                                              # R_m^T o_m for each head
        return out / l[:, None]

    # ---- pseudo-token far memory ("ProtoKV: Streaming Video Understanding under
    # Delayed Query with Summary-State Memory", section 3.3 Eq. (2), Appendix A.3
    # Eq. (4) and Algorithm 4) ----
    def decode_with_pseudo(self, q16: np.ndarray, kf16: np.ndarray, vf16: np.ndarray, mass: np.ndarray,
                           per_proto: int) -> np.ndarray:
        """One softmax over this unit's cache (the near window, bias 0, deleted
        tokens skipped) and far pseudo tokens kf16, vf16 [n_far][d] (fp16, the
        original key / value bases): pseudo token j belongs to prototype
        j // per_proto, whose mass n = mass[j // per_proto] adds log n to its
        logit q.k/sqrt d; prototypes with n = 0 are inactive and skipped.
        Returns fp64 [Gq][d] (zeros when nothing is attended)."""
        d, G, T, Tf = self.d, self.G, self.T, self.T_full
        Gq = q16.shape[0]
        q = q16.astype(F64)
        nf = len(kf16)
        n = np.asarray(mass, F64)[np.arange(nf) // per_proto] if nf else np.zeros(0)
        sf = q @ np.asarray(kf16, F64).T / math.sqrt(d)                    # [Gq][n_far]
        with np.errstate(divide="ignore"):
            sf = sf + np.log(n)[None]                                       # log 0 = -inf: inactive
        s = np.full((Gq, T), -np.inf)
        if T:
            qr = rotate_f64(q, self.signs) / math.sqrt(d)
            if self.key_codec == "turbo":
                s[:] = (qr @ self.cb.levels[self.kcodes[:T]].T) * (self.knorm[:T].astype(F64) / math.sqrt(d))[None]
            elif Tf:
                ng = Tf // G
                lam = self.cb.ktab[self.kcodes[:Tf]].reshape(ng, G, d)
                beta = qr @ self.kmn[:ng].astype(F64).T
                a = qr[:, None, :] * self.krg[:ng].astype(F64)[None]
                s[:, :Tf] = (beta[:, :, None] + np.einsum("hgc,gtc->hgt", a, lam)).reshape(Gq, Tf)
            if T > Tf:
                s[:, Tf:] = q @ self.keys16[Tf:T].astype(F64).T / math.sqrt(d)
            s[:, self.dead[:T]] = -np.inf
        mmax = max(s.max() if T else -np.inf, sf.max() if nf else -np.inf)
        out = np.zeros((Gq, d), F64)
        if mmax == -np.inf:
            return out
        mrow = np.maximum(s.max(axis=1) if T else -np.inf, sf.max(axis=1) if nf else -np.inf)[:, None]
        p = np.exp(s - mrow)
        pf = np.exp(sf - mrow)
        l = p.sum(axis=1) + pf.sum(axis=1)
        if T:
            lv = self.cb.levels[self.vcodes[:T]] / math.sqrt(d)
            wv = lv * self.vnorm[:T].astype(F64)[:, None]
            R64 = self.R.astype(F64)
            for m in range(self.R.shape[0]):
                sel = self.mod[:T] == m
                if sel.any():
                    out += (p[:, sel] @ wv[sel]) @ R64[m]
        out += pf @ np.asarray(vf16, F64)
        return out / l[:, None]

    def dequantized(self):
        """Explicit K-hat, V-hat [T][d] in the original bases (for brute-force attention)."""
        d, G, T, Tf = self.d, self.G, self.T, self.T_full
        H = sylvester_hadamard(d).astype(F64)
        Kh = np.empty((T, d), F64)
        if self.key_codec == "turbo":
            Rh = hadamard_rotation(self.signs)
            lk = self.cb.levels[self.kcodes[:T]] / math.sqrt(d)
            Kh[:] = (lk @ Rh) * self.knorm[:T].astype(F64)[:, None]               # n R^T l / sqrt d
            Tf = T
        elif Tf:
            g = np.arange(Tf) // G
            mn = self.kmn[g].astype(F64)
            rg = self.krg[g].astype(F64)
            kp = mn + self.cb.ktab[self.kcodes[:Tf]] * rg                    # rotated domain
            Kh[:Tf] = (kp @ H.T) * self.signs.astype(F64)[None] / math.sqrt(d)   # D H^T k'/sqrt d
        Kh[Tf:] = self.keys16[Tf:T].astype(F64)
        R64 = self.R.astype(F64)
        Vh = np.empty((T, d), F64)
        lv = self.cb.levels[self.vcodes[:T]] / math.sqrt(d)
        for t in range(T):
            Vh[t] = self.vnorm[t].astype(F64) * (R64[self.mod[t]].T @ lv[t])
        return Kh, Vh

    def decode_bruteforce(self, q16: np.ndarray) -> np.ndarray:
        """softmax(q K-hat^T / sqrt d) V-hat over the explicitly dequantized cache."""
        Gq, d = q16.shape
        if self.T == 0:
            return np.zeros((Gq, d), F64)
        Kh, Vh = self.dequantized()
        live = ~self.dead[:self.T]
        if not live.any():
            return np.zeros((Gq, d), F64)
        Kh, Vh = Kh[live], Vh[live]
        s = q16.astype(F64) @ Kh.T / math.sqrt(d)
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        return p @ Vh

    # ---- eviction and compaction ("OmniTide", sections 5.2 and 6.2) ----
    def evict(self, begin: int, end: int):
        """Delete tokens [begin, end): they stay in their slots as holes."""
        if not 0 <= begin <= end <= self.T:
            raise ValueError("eviction range outside the cache")
        self.dead[begin:end] = True

    def move_granules(self, moves, granule: int, new_T: int):
        """Apply an order-preserving move list [(src granule, dst granule)]: every
        per-token array moves with its tokens, every key group with its granule
        (granule = G for grouped keys); the cache then ends at new_T."""
        for src, dst in moves:
            a, b = src * granule, min((src + 1) * granule, self.T)
            c = dst * granule
            for arr in (self.kcodes, self.kbnd, self.keys16, self.knorm, self.knbnd, self.vcodes, self.vbnd,
                        self.vnorm, self.nbnd, self.mod, self.dead):
                arr[c:c + (b - a)] = arr[a:b]
            if self.key_codec == "omni":
                self.kmn[dst], self.krg[dst] = self.kmn[src], self.krg[src]
        self.dead[new_T:self.T] = False
        self.T = new_T


def compaction_granule(key_codec: str, group_size: int) -> int:
    """Tokens moved as one unit: a key group (its statistics belong to all its
    members), or one 16-token tile for TurboQuant keys (per-token scales)."""
    return group_size if key_codec == "omni" else 16


def plan_suffix_compaction(dead: np.ndarray, T: int, granule: int, min_pages: int, page: int = 64):
    """Ordered-suffix migration plan ("OmniTide", section 6.2, ordered-suffix
    mode), at granule granularity.  Scanning suffix starts s (granule-aligned)
    from the end of the cache backward, packing the suffix's granules that still
    hold a live token to s, s + granule, ... in their order shortens the
    page-rounded span from ceil(T/page) to ceil(T'/page); the first (shortest)
    suffix that saves at least min_pages pages is the plan.  Returns None (no
    migration) or (s_granule, T', moves) with moves [(src, dst)] for the
    granules whose slot changes."""
    if min_pages < 1:
        raise ValueError("min_pages must be >= 1")
    dead = np.asarray(dead[:T], bool)
    ng = -(-T // granule)
    lens = [min(granule, T - j * granule) for j in range(ng)]
    empty = [bool(dead[j * granule:j * granule + lens[j]].all()) for j in range(ng)]
    pages0 = -(-T // page)
    for sg in range(ng - 1, -1, -1):
        kept = [j for j in range(sg, ng) if not empty[j]]
        T2 = sg * granule + sum(lens[j] for j in kept)      # only the last granule can be partial
        if pages0 - (-(-T2 // page)) >= min_pages:
            moves = [(j, sg + i) for i, j in enumerate(kept) if j != sg + i]
            return sg, T2, moves
    return None


class OracleCache:
    """All units of a multi-session cache; mirrors the library's create/append/decode/export."""

    def __init__(self, num_sessions, num_layers, num_q_heads, num_kv_heads, head_dim, group_size, bits,
                 max_tokens, hadamard_seed, value_rot, codebook_levels=None, layers=None, num_modalities=3,
                 key_codec="omni", sessions=None):
        self.S, self.L, self.Hq, self.Hkv, self.d = num_sessions, num_layers, num_q_heads, num_kv_heads, head_dim
        self.G, self.bits, self.M = group_size, bits, num_modalities
        self.cb = make_codebook(bits, codebook_levels)
        self.signs = hadamard_signs(hadamard_seed, head_dim)
        self.layers = list(range(num_layers)) if layers is None else list(layers)
        R = np.asarray(value_rot, F32)
        self.units = {}
        self.sessions = list(range(num_sessions)) if sessions is None else list(sessions)   # the ones modelled
        for s in self.sessions:
            for l in self.layers:
                for h in range(num_kv_heads):
                    self.units[(s, l, h)] = OracleUnit(head_dim, group_size, self.cb, self.signs, R[l, h],
                                                       num_q_heads // num_kv_heads, max_tokens, key_codec)

    def append(self, session, K16, V16, mod, layers_in=None):
        """K16, V16 [T][L'][Hkv][d] where L' indexes ``layers_in`` (default: self.layers)."""
        layers_in = self.layers if layers_in is None else list(layers_in)
        for i, l in enumerate(layers_in):
            for h in range(self.Hkv):
                self.units[(session, l, h)].append(K16[:, i, h], V16[:, i, h], mod)

    def evict(self, session, begin, end):
        """Delete tokens [begin, end) of a session in every (layer, kv head)."""
        for (s, _, _), u in self.units.items():
            if s == session:
                u.evict(begin, end)

    def compact(self, session, min_pages):
        """Plan and apply the ordered-suffix compaction of a session; returns the
        plan (see plan_suffix_compaction) or None."""
        units = [u for (s, _, _), u in self.units.items() if s == session]
        u0 = units[0]
        gran = compaction_granule(u0.key_codec, self.G)
        plan = plan_suffix_compaction(u0.dead, u0.T, gran, min_pages)
        if plan is not None:
            for u in units:
                u.move_granules(plan[2], gran, plan[1])
        return plan

    def decode_with_pseudo(self, Q16, KF, VF, MASS, per_proto):
        """Q16 [S][L][Hq][d]; KF, VF [S][L][Hkv][n_far][d] fp16; MASS [S][L][Hkv][n_far / per_proto]
        -> fp64 [S][L'][Hq][d] for the oracle's layers."""
        gq = self.Hq // self.Hkv
        out = np.zeros((self.S, len(self.layers), self.Hq, self.d), F64)
        for s in self.sessions:
            for i, l in enumerate(self.layers):
                for h in range(self.Hkv):
                    u = self.units[(s, l, h)]
                    out[s, i, h * gq:(h + 1) * gq] = u.decode_with_pseudo(
                        Q16[s, l, h * gq:(h + 1) * gq], KF[s, l, h], VF[s, l, h], MASS[s, l, h], per_proto)
        return out

    def decode(self, Q16, brute=False):
        """Q16 [S][L][Hq][d] -> fp64 [S][L'][Hq][d] for the oracle's layers."""
        gq = self.Hq // self.Hkv
        out = np.zeros((self.S, len(self.layers), self.Hq, self.d), F64)
        for s in self.sessions:
            for i, l in enumerate(self.layers):
                for h in range(self.Hkv):
                    u = self.units[(s, l, h)]
                    q = Q16[s, l, h * gq:(h + 1) * gq]
                    out[s, i, h * gq:(h + 1) * gq] = u.decode_bruteforce(q) if brute else u.decode(q)
        return out


# ---------------------------------------------------------------------------
# value-rotation calibration (section 2, second OmniKVQuant bullet)
# ---------------------------------------------------------------------------

def calibrate_rotation(v16: np.ndarray, weight: Optional[np.ndarray] = None):
    """Eigenbasis of the attention-contribution-weighted covariance of ONE modality's
    calibration values v16 [n][d]: the directions are weighted by the tokens'
    contributions a_t >= 0 (``weight``; None = all 1), the covariance is
    C = sum_t a_t (v_t - mu)(v_t - mu)^T / sum_t a_t with mu the weighted mean, and
    the rotation's rows are C's eigenvectors, in descending eigenvalue order, each
    signed so that its largest-magnitude entry is positive.  Fewer than two tokens
    or zero total weight give the identity (and zero eigenvalues).
    Returns R [d][d] (fp64, rows = basis) and the eigenvalues [d] (descending).
    """
    v = np.asarray(v16, F64)
    n, d = v.shape
    a = np.ones(n, F64) if weight is None else np.asarray(weight, F64)
    W = a.sum()
    if n < 2 or W <= 0:
        return np.eye(d), np.zeros(d)
    mu = (a[:, None] * v).sum(0) / W
    x = v - mu[None]
    C = (x.T * a[None]) @ x / W
    lam, U = np.linalg.eigh(C)
    order = np.argsort(-lam, kind="stable")
    R = U[:, order].T.copy()
    idx = np.argmax(np.abs(R), axis=1)
    R *= np.sign(R[np.arange(d), idx])[:, None]
    return R, lam[order]


def calibrate_rotations(v16: np.ndarray, modality: np.ndarray, num_modalities: int,
                        weight: Optional[np.ndarray] = None):
    """calibrate_rotation for every (layer, kv head) and modality of a calibration
    stream: v16 [n][L][Hkv][d], modality ids [n] (ids >= num_modalities are
    ignored), weight [n][L][Hkv] or None.  Returns R [L][Hkv][M][d][d] and the
    eigenvalues [L][Hkv][M][d]."""
    v = np.asarray(v16)
    n, L, H, d = v.shape
    mod = np.asarray(modality)
    R = np.empty((L, H, num_modalities, d, d))
    lam = np.empty((L, H, num_modalities, d))
    for l in range(L):
        for h in range(H):
            for m in range(num_modalities):
                sel = mod == m
                a = None if weight is None else np.asarray(weight)[sel, l, h]
                R[l, h, m], lam[l, h, m] = calibrate_rotation(v[sel, l, h], a)
    return R, lam
