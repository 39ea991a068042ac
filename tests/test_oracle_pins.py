"""Pins of the CPU oracle to facts fixed outside itself (closed forms, textbook
tables, published generator output, brute force on tiny inputs, invariants).

Each test would fail on a plausible slip in the oracle: a dropped term, a
wrong sign or index, a transposed operand, a wrong stage order or rounding.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import okvq_oracle as o
from bit_kv_cache_rht_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F16, F32, F64 = np.float16, np.float32, np.float64


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- RHT

def test_splitmix64_published_sequence():
    g = _golden("splitmix64.json")
    got = o.splitmix64(g["seed"], len(g["outputs_hex"]))
    assert got == [int(h, 16) for h in g["outputs_hex"]]


def test_hadamard_signs_are_the_stream_bits():
    w0, w1 = o.splitmix64(7, 2)
    s = o.hadamard_signs(7, 128)
    assert set(np.unique(s)) <= {-1, 1}
    for c in (0, 5, 63, 64, 100, 127):
        bit = ((w0 if c < 64 else w1) >> (c % 64)) & 1
        assert s[c] == (-1 if bit else 1)


@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128])
def test_sylvester_hadamard_orthogonality_exact(d):
    H = o.sylvester_hadamard(d)
    assert np.array_equal(H @ H.T, d * np.eye(d, dtype=np.int64))
    assert np.array_equal(H, H.T)
    assert H[0].tolist() == [1] * d and H[:, 0].tolist() == [1] * d


def test_fwht_equals_matrix_product():
    r = np.random.default_rng(0)
    x = r.standard_normal((5, 128))
    H = o.sylvester_hadamard(128).astype(F64)
    assert np.allclose(o.fwht(x, F64), x @ H.T, atol=1e-11, rtol=0)


def test_fwht_fp32_exact_on_integers_and_order_matters_only_by_rounding():
    # small integers: every butterfly sum is exact, so the fp32 canonical order
    # must give exactly the fp64 (exact) transform
    r = np.random.default_rng(1)
    x = r.integers(-1000, 1000, (7, 128)).astype(F32)
    assert np.array_equal(o.fwht(x, F32).astype(F64), o.fwht(x.astype(F64), F64))


def test_rotate_keys_f32_close_to_fp64_and_norm_preserving():
    r = np.random.default_rng(2)
    k = (r.standard_normal((64, 128)) * 3).astype(F16)
    s = o.hadamard_signs(11, 128)
    k32 = o.rotate_keys_f32(k, s)
    k64 = o.rotate_f64(k.astype(F64), s)
    assert k32.dtype == F32
    assert np.max(np.abs(k32 - k64)) < 2e-5
    assert np.allclose(np.linalg.norm(k64, axis=1), np.linalg.norm(k.astype(F64), axis=1), rtol=1e-12)
    # a sign slip (D after H instead of before) is a different transform
    wrong = o.fwht(k.astype(F64), F64) * s / math.sqrt(128)
    assert np.max(np.abs(wrong - k64)) > 0.1


# ---------------------------------------------------------------- codebook

@pytest.mark.parametrize("n", [2, 4, 8, 16])
def test_lloyd_max_textbook(n):
    g = _golden("lloyd_max_gaussian.json")
    lv = o.lloyd_max_gaussian(n)
    pos = lv[n // 2:]
    ref = np.array(g["levels"][str(n)])
    ulp = 10.0 ** (np.floor(np.log10(np.abs(ref))) - 3)      # 4 significant digits printed
    assert np.all(np.abs(pos - ref) <= 0.6 * ulp)
    assert np.allclose(lv, -lv[::-1], atol=1e-13)
    # fixed point: each level is the Gaussian mean of its cell (closed form)
    th = [-math.inf] + [0.5 * (lv[j] + lv[j + 1]) for j in range(n - 1)] + [math.inf]
    for j in range(n):
        assert abs(lv[j] - o.gaussian_cell_mean(th[j], th[j + 1])) < 1e-12
    # mean-squared error of the quantizer, integrated in closed form per cell:
    # E[(X-y)^2; a<X<b] = (P + a phi(a) - b phi(b)) - 2y(phi(a)-phi(b)) + y^2 P
    mse = 0.0
    for j in range(n):
        a, b, y = th[j], th[j + 1], lv[j]
        P = o._Phi(b) - o._Phi(a)
        ta = a * o._phi(a) if math.isfinite(a) else 0.0
        tb = b * o._phi(b) if math.isfinite(b) else 0.0
        mse += (P + ta - tb) - 2 * y * (o._phi(a) - o._phi(b)) + y * y * P
    if str(n) in g["mse"]:
        ref_mse = g["mse"][str(n)]
        assert abs(mse - ref_mse) <= 0.6 * 10.0 ** (math.floor(math.log10(ref_mse)) - 3)
    # the closed form agrees with direct numerical integration of (x - y)^2 phi(x)
    from scipy.integrate import quad
    num = sum(quad(lambda x, y=lv[j]: (x - y) ** 2 * o._phi(x), max(th[j], -40.0), min(th[j + 1], 40.0),
                   epsabs=1e-15, epsrel=1e-13)[0] for j in range(n))
    assert abs(num - mse) < 1e-12


def test_lloyd_max_two_level_closed_form():
    assert abs(o.lloyd_max_gaussian(2)[1] - math.sqrt(2 / math.pi)) < 1e-13


def test_four_level_thresholds_textbook():
    g = _golden("lloyd_max_gaussian.json")
    cb = o.make_codebook(2)
    assert np.allclose(cb.vthr[1:], g["thresholds"]["4"], atol=2e-3)


@pytest.mark.parametrize("bits", [2, 4])
def test_codebook_derivation(bits):
    cb = o.make_codebook(bits)
    n = 1 << bits
    assert cb.levels16.dtype == F16 and len(cb.levels16) == n
    assert np.all(np.diff(cb.levels) > 0)
    assert np.array_equal(cb.vthr.astype(F64), (cb.levels[:-1] + cb.levels[1:]) / 2)   # exact midpoints
    assert cb.ktab[0] == 0.0 and cb.ktab[-1] == 1.0 and np.all(np.diff(cb.ktab) > 0)
    assert np.array_equal(cb.kthr.astype(F64), (cb.ktab[:-1] + cb.ktab[1:]) / 2)
    # key levels are the value levels renormalised to [0, 1]
    lam = (cb.levels - cb.levels[0]) / (cb.levels[-1] - cb.levels[0])
    assert np.max(np.abs(cb.ktab - lam)) <= 2.0 ** -11


# ---------------------------------------------------------------- storage roundings

def test_directed_fp16_rounding():
    r = np.random.default_rng(3)
    x = (r.standard_normal(20000) * 5).astype(F32)
    dn, up = o.f16_round_down(x), o.f16_round_up(x)
    assert np.all(dn.astype(F32) <= x) and np.all(up.astype(F32) >= x)
    # tightest: the next fp16 past each bound crosses x
    nxt = np.nextafter(dn, F16(np.inf)).astype(F32)
    assert np.all((dn.astype(F32) == x) | (nxt > x))
    prv = np.nextafter(up, F16(-np.inf)).astype(F32)
    assert np.all((up.astype(F32) == x) | (prv < x))


# ---------------------------------------------------------------- key groups

def _brute_nearest(x, levels):
    """argmin_j |x - level_j|, ties to the lower index, by enumeration."""
    d = np.abs(np.asarray(x, F64)[..., None] - np.asarray(levels, F64))
    return np.argmin(d, axis=-1).astype(np.uint8)


@pytest.mark.parametrize("bits", [2, 4])
def test_key_group_codes_bounds_and_brute_force(bits):
    cb = o.make_codebook(bits)
    r = np.random.default_rng(4 + bits)
    s = o.hadamard_signs(3, 128)
    k = (r.standard_normal((32, 128)) * r.uniform(0.5, 4, 128) + 0.7).astype(F16)
    kp = o.rotate_keys_f32(k, s)
    mn, rg, codes, bnd = o.quantize_key_group(kp, cb)
    mn64, rg64 = mn.astype(F64), rg.astype(F64)
    # the stored interval contains every member, and both ends are the tightest fp16
    assert np.all(mn64 <= kp.min(0)) and np.all(mn64 + rg64 >= kp.max(0))
    assert np.all(np.nextafter(mn, F16(np.inf)).astype(F64) > kp.min(0))
    assert np.all(mn64 + np.nextafter(rg, F16(-np.inf)).astype(F64) < kp.max(0))
    u = (kp.astype(F64) - mn64) / rg64
    ref = _brute_nearest(u, cb.ktab)
    ok = ~bnd
    assert np.array_equal(codes[ok], ref[ok])
    rec = mn64 + cb.ktab[codes] * rg64
    assert np.all(rec >= mn64 - 1e-12) and np.all(rec <= mn64 + rg64 + 1e-12)
    gap = np.max(np.diff(cb.ktab))
    assert np.all(np.abs(rec - kp) <= rg64 * gap / 2 + 1e-6)
    # every code of a wide group is used somewhere; the top and bottom levels are hit
    assert codes.min() == 0 and codes.max() == (1 << bits) - 1


def test_key_group_degenerate_range_gives_code_zero():
    cb = o.make_codebook(2)
    kp = np.full((32, 128), 1.25, F32)
    mn, rg, codes, _ = o.quantize_key_group(kp, cb)
    assert np.all(rg == 0) and np.all(codes == 0)


def test_f16_round_up_of_exact_values():
    x = np.array([0.0, 1.0, 1.0 + 2.0 ** -12, 3.0 - 2.0 ** -30, 65504.0], F64)
    up = o.f16_round_up_f64(x).astype(F64)
    assert up.tolist() == [0.0, 1.0, 1.0 + 2.0 ** -10, 3.0, 65504.0]


# ---------------------------------------------------------------- values

@pytest.mark.parametrize("bits", [2, 4])
def test_value_codes_brute_force_and_error_identity(bits):
    cb = o.make_codebook(bits)
    r = np.random.default_rng(10 + bits)
    v = (r.standard_normal((50, 128)) * 2 + 0.5).astype(F16)
    R = np.linalg.qr(r.standard_normal((128, 128)))[0].astype(F32)
    nrm, codes, bnd, nb = o.quantize_values(v, R, cb)
    v64 = v.astype(F64)
    n = np.linalg.norm(v64, axis=1)
    assert np.array_equal(nrm, n.astype(F16))
    w = math.sqrt(128) * (v64 / n[:, None]) @ R.astype(F64).T
    ref = _brute_nearest(w, cb.levels)
    assert np.array_equal(codes[~bnd], ref[~bnd])
    # per-coordinate bound: half the widest gap inside the table, clipping outside
    gap = np.max(np.diff(cb.levels))
    err = np.abs(w - cb.levels[codes])
    bound = np.maximum(gap / 2, np.maximum(0, np.abs(w) - cb.levels[-1]))
    assert np.all(err <= bound + 1e-9)
    # orthogonality: |v - v_hat| = n |u - u_hat| with u_hat = R^T l / sqrt d
    uh = (cb.levels[codes] / math.sqrt(128)) @ R.astype(F64)
    vh = n[:, None] * uh
    lhs = np.linalg.norm(v64 - vh, axis=1)
    rhs = n * np.linalg.norm(v64 / n[:, None] - uh, axis=1)
    assert np.allclose(lhs, rhs, rtol=1e-12)
    assert np.allclose(np.linalg.norm(uh, axis=1), np.linalg.norm(cb.levels[codes], axis=1) / math.sqrt(128))


def test_zero_value_vector():
    cb = o.make_codebook(2)
    R = np.eye(128, dtype=F32)
    nrm, codes, _, _ = o.quantize_values(np.zeros((1, 128), F16), R, cb)
    assert nrm[0] == 0 and np.all(codes == 1)       # nearest level to 0, tie -> lower middle level


@pytest.mark.parametrize("bits", [2, 4])
def test_pack_roundtrip_and_bit_positions(bits):
    r = np.random.default_rng(20)
    c = r.integers(0, 1 << bits, (3, 128)).astype(np.uint8)
    p = o.pack_codes(c, bits)
    assert p.shape == (3, 128 * bits // 8)
    assert np.array_equal(o.unpack_codes(p, bits), c)
    one = np.zeros((1, 128), np.uint8)
    one[0, 5] = (1 << bits) - 1
    pk = o.pack_codes(one, bits)
    if bits == 2:
        assert pk[0, 1] == 0b00001100 and pk.sum() == 12
    else:
        assert pk[0, 2] == 0xF0 and pk.sum() == 0xF0


# ---------------------------------------------------------------- attention

def _rotations(w):
    V, mod = w.calibration_slice()
    return o.calibrate_rotations(V, mod, w.shape.num_modalities)[0].astype(F32)


def _unit(bits=2, G=32, T=203, seed=0, Gq=4):
    cb = o.make_codebook(bits)
    r = np.random.default_rng(seed)
    R = np.stack([np.linalg.qr(r.standard_normal((128, 128)))[0] for _ in range(3)]).astype(F32)
    u = o.OracleUnit(128, G, cb, o.hadamard_signs(99, 128), R, Gq, 1024)
    T1 = T // 2
    for a, b in ((0, T1), (T1, T)):
        K = (r.standard_normal((b - a, 128)) * 2 + np.linspace(0, 1, b - a)[:, None]).astype(F16)
        V = (r.standard_normal((b - a, 128)) * 1.5 + 0.3).astype(F16)
        mod = r.integers(0, 3, b - a).astype(np.uint8)
        u.append(K, V, mod)
    return u, r


@pytest.mark.parametrize("bits,G,T", [(2, 32, 203), (2, 64, 130), (4, 32, 96), (4, 64, 31)])
def test_fused_scores_equal_bruteforce(bits, G, T):
    u, r = _unit(bits, G, T, seed=bits * 100 + G + T)
    q = (r.standard_normal((4, 128)) * 1.5).astype(F16)
    a = u.decode(q)
    b = u.decode_bruteforce(q)
    assert np.max(np.abs(a - b)) < 1e-10


def test_single_token_output_is_its_dequantized_value():
    u, r = _unit(T=1)
    q = r.standard_normal((4, 128)).astype(F16)
    _, Vh = u.dequantized()
    assert np.allclose(u.decode(q), np.broadcast_to(Vh[0], (4, 128)), atol=1e-12)


def test_zero_query_gives_mean_value():
    u, r = _unit(T=150)
    _, Vh = u.dequantized()
    out = u.decode(np.zeros((4, 128), F16))
    assert np.allclose(out, np.broadcast_to(Vh.mean(0), (4, 128)), atol=1e-12)


def test_empty_unit_outputs_zero():
    cb = o.make_codebook(2)
    R = np.stack([np.eye(128, dtype=F32)] * 3)
    u = o.OracleUnit(128, 32, cb, o.hadamard_signs(1, 128), R, 2, 64)
    assert np.all(u.decode(np.ones((2, 128), F16)) == 0)


def test_grid_keys_reproduce_exact_attention():
    """Keys built so their rotated coordinates sit on the group's grid: the codec
    is then lossless for keys (up to the fp16 rounding of the constructed keys),
    so the fused output must match exact attention over those keys."""
    G, T, d = 32, 96, 128
    cb = o.make_codebook(2)
    r = np.random.default_rng(5)
    s = o.hadamard_signs(42, d)
    H = o.sylvester_hadamard(d).astype(F64)
    codes = r.integers(0, 4, (T, d))
    codes[0::G] = 0
    codes[1::G] = 3                                      # every channel reaches both ends
    mn = np.repeat(r.uniform(-3, -1, (T // G, d)), G, 0)
    mx = mn + np.repeat(r.uniform(1, 4, (T // G, d)), G, 0)
    kp = mn + cb.ktab[codes] * (mx - mn)
    K = ((kp @ H.T) * s / math.sqrt(d)).astype(F16)      # k = D H^T k' / sqrt d
    V = (r.standard_normal((T, d)) * 2).astype(F16)
    mod = np.zeros(T, np.uint8)
    R = np.stack([np.eye(d, dtype=F32)] * 3)
    u = o.OracleUnit(d, G, cb, s, R, 2, T)
    u.append(K, V, mod)
    assert np.mean(u.kcodes[:T] == codes) > 0.97
    q = r.standard_normal((2, d)).astype(F16)
    _, Vh = u.dequantized()
    sc = q.astype(F64) @ K.astype(F64).T / math.sqrt(d)
    p = np.exp(sc - sc.max(1, keepdims=True))
    exact = (p / p.sum(1, keepdims=True)) @ Vh
    assert np.max(np.abs(u.decode(q) - exact)) < 5e-3


def test_streaming_chunking_invariance():
    w = synth.tiny(seed=7)
    R = _rotations(w)
    K, V = w.session_kv(0)
    mod = w.sessions[0].modality()

    def build(bounds):
        c = o.OracleCache(1, 1, 8, 2, 128, 32, 2, 2048, w.hadamard_seed, R)
        for a, b in bounds:
            c.append(0, K[a:b], V[a:b], mod[a:b])
        return c

    T = len(mod)
    one = build([(0, T)])
    r = np.random.default_rng(0)
    cuts = np.sort(r.choice(np.arange(1, T), 20, replace=False))
    rand = build(list(zip([0, *cuts], [*cuts, T])))
    by97 = build([(a, min(a + 97, T)) for a in range(0, T, 97)])
    for h in range(2):
        e0 = one.units[(0, 0, h)].export()
        for other in (rand, by97):
            e1 = other.units[(0, 0, h)].export()
            for key in e0:
                assert np.array_equal(e0[key], e1[key]), key


# ---------------------------------------------------------------- synthetic inputs

def test_calibrated_rotations_on_the_slice_orthogonal_and_diagonalising():
    """The multi-unit calibration on the synthetic calibration slice: every basis is
    orthonormal and diagonalises np.cov of its modality's tokens (the unweighted,
    n-1 normalised covariance has the same eigenvectors)."""
    w = synth.tiny(seed=3)
    Vc, mod = w.calibration_slice()
    assert Vc.shape == (synth.CALIB_TOKENS, 1, 2, 128) and Vc.dtype == F16
    R, lam = o.calibrate_rotations(Vc, mod, 3)
    assert R.shape == (1, 2, 3, 128, 128) and lam.shape == (1, 2, 3, 128)
    for h in range(2):
        for m in range(3):
            Rm = R[0, h, m]
            assert np.max(np.abs(Rm @ Rm.T - np.eye(128))) < 1e-10
            C = np.cov(Vc[mod == m, 0, h].astype(F64), rowvar=False)
            D = Rm @ C @ Rm.T
            off = D - np.diag(np.diag(D))
            assert np.max(np.abs(off)) < 1e-10 * np.trace(C)
            assert np.all(np.diff(np.diag(D)) <= 1e-10 * np.trace(C))
            n = int((mod == m).sum())
            assert np.allclose(lam[0, h, m] * n / (n - 1), np.diag(D), atol=1e-10 * np.trace(C))
    # ids beyond the modality count are ignored
    R2, _ = o.calibrate_rotations(Vc, np.where(mod == 2, 7, mod).astype(np.uint8), 3)
    assert np.array_equal(R2[0, :, :2], R[0, :, :2]) and np.array_equal(R2[0, 0, 2], np.eye(128))


def test_workload_streams():
    w = synth.qwen3b(tokens=32768)
    m = w.sessions[0].modality()
    assert len(m) == 32768 and set(np.unique(m)) == {0, 1, 2}
    c = w.sessions[0].chunks
    assert len(c[0]) == 665 and len(c[29]) == 697
    t = synth.tiny()
    mt = t.sessions[0].modality()
    assert len(mt) == 2048 and mt[:64].tolist() == [0] * 64 and mt[64:89].tolist() == [1] * 25
    assert mt[2037:].tolist() == [0] * 11


# ---------------------------------------------------------------- TurboQuant key codec

def test_hadamard_rotation_matrix_matches_butterfly():
    """(1/sqrt d) H D as a matrix (Sylvester construction) equals the butterfly
    rotation and is orthogonal."""
    s = o.hadamard_signs(7, 128)
    Rh = o.hadamard_rotation(s)
    x = np.random.default_rng(1).standard_normal((5, 128))
    assert np.allclose(x @ Rh.T, o.rotate_f64(x, s), atol=1e-12)
    assert np.allclose(Rh @ Rh.T, np.eye(128), atol=1e-12)


def _turbo_unit(bits=2, T=203, seed=0, Gq=4):
    cb = o.make_codebook(bits)
    r = np.random.default_rng(seed)
    R = np.stack([np.linalg.qr(r.standard_normal((128, 128)))[0] for _ in range(3)]).astype(F32)
    u = o.OracleUnit(128, 32, cb, o.hadamard_signs(99, 128), R, Gq, 1024, key_codec="turbo")
    T1 = T // 2
    for a, b in ((0, T1), (T1, T)):
        K = (r.standard_normal((b - a, 128)) * 2 + np.linspace(0, 1, b - a)[:, None]).astype(F16)
        V = (r.standard_normal((b - a, 128)) * 1.5 + 0.3).astype(F16)
        u.append(K, V, r.integers(0, 3, b - a).astype(np.uint8))
    return u, r


@pytest.mark.parametrize("bits,T", [(2, 203), (4, 31), (2, 1)])
def test_turbo_fused_scores_equal_bruteforce(bits, T):
    u, r = _turbo_unit(bits, T, seed=bits * 10 + T)
    assert u.T_full == T                                  # every key is quantized on arrival
    q = (r.standard_normal((4, 128)) * 1.5).astype(F16)
    assert np.max(np.abs(u.decode(q) - u.decode_bruteforce(q))) < 1e-10


@pytest.mark.parametrize("bits,mse", [(2, 0.1175), (4, 0.009497)])
def test_turbo_key_distortion_is_the_gaussian_quantizer_mse(bits, mse):
    """Isotropic Gaussian keys: after the randomized Hadamard rotation and the
    sqrt(d)/|k| scale the coordinates are ~N(0,1), so the relative squared error of
    the reconstructed key is the Lloyd-Max MSE of the unit Gaussian (Max 1960:
    0.1175 for 4 levels, 0.009497 for 16)."""
    r = np.random.default_rng(3)
    K = r.standard_normal((3000, 128)).astype(F16)
    u = o.OracleUnit(128, 32, o.make_codebook(bits), o.hadamard_signs(5, 128),
                     np.stack([np.eye(128, dtype=F32)] * 3), 1, 3000, key_codec="turbo")
    u.append(K, K, np.zeros(3000, np.uint8))
    Kh, _ = u.dequantized()
    Kf = K.astype(F64)
    rel = np.sum((Kh - Kf) ** 2, axis=1) / np.sum(Kf ** 2, axis=1)
    assert abs(rel.mean() / mse - 1.0) < 0.06, rel.mean()


def _key_errors(key_codec, K, V, q, bits=2):
    cb = o.make_codebook(bits)
    u = o.OracleUnit(128, 32, cb, o.hadamard_signs(11, 128), np.stack([np.eye(128, dtype=F32)] * 3),
                     q.shape[0], len(K), key_codec=key_codec)
    u.append(K, V, np.zeros(len(K), np.uint8))
    Kh, _ = u.dequantized()
    Kf = K.astype(F64)
    key_err = np.sum((Kh - Kf) ** 2) / np.sum(Kf ** 2)
    s = q.astype(F64) @ Kf.T / math.sqrt(128)
    p = np.exp(s - s.max(1, keepdims=True))
    _, Vh = u.dequantized()
    exact = (p / p.sum(1, keepdims=True)) @ Vh           # same dequantized values, exact keys
    att_err = np.sqrt(np.mean((u.decode(q) - exact) ** 2) / np.mean(exact ** 2))
    return key_err, att_err


def test_local_key_ranges_beat_turbo_scale_on_drifted_keys():
    """The comparison the pages make (section 2, Table 3: local key ranges lower the
    quantization error of TurboQuant's fixed scale at the same bit width, because
    keys drift over the stream) on the full 32,768-token synthetic drifted stream:
    the 2-bit key reconstruction error and the attention output error it causes are
    both lower with per-group ranges (measured: 0.057 vs 0.113 and 0.071 vs 0.105)."""
    w = synth.qwen3b(tokens=32768, layers=1)
    K, V = w.layer_kv(0, 0)
    K, V = K[:, 0], V[:, 0]
    q = w.queries(0)[0, 0, :8]
    ko, ao = _key_errors("omni", K, V, q)
    kt, at = _key_errors("turbo", K, V, q)
    assert ko < 0.7 * kt, (ko, kt)
    assert ao < at, (ao, at)


# ---------------------------------------------------------------- rotation calibration

def _exact_cloud(U, lam):
    """Points +-sqrt(d lam_i) u_i (2d of them): mean 0, covariance exactly U diag(lam) U^T."""
    d = len(lam)
    pts = []
    for i in range(d):
        pts.append(np.sqrt(d * lam[i]) * U[:, i])
        pts.append(-np.sqrt(d * lam[i]) * U[:, i])
    return np.array(pts)


def test_calibration_recovers_a_constructed_eigenbasis():
    d = 128
    r = np.random.default_rng(8)
    U = np.linalg.qr(r.standard_normal((d, d)))[0]
    lam = np.sort(r.uniform(0.1, 5.0, d))[::-1] + np.arange(d)[::-1] * 1e-3    # distinct, descending
    X = _exact_cloud(U, lam)
    R, ev = o.calibrate_rotation(X)
    assert np.allclose(ev, lam, rtol=1e-9, atol=1e-12)
    dots = np.abs(np.sum(R * U.T, axis=1))                   # |<r_i, u_i>|
    assert np.all(dots > 1 - 1e-8)
    assert np.all(R[np.arange(d), np.argmax(np.abs(R), axis=1)] > 0)   # sign convention


def test_calibration_weights_equal_duplication_and_shift_invariance():
    r = np.random.default_rng(9)
    X = r.standard_normal((40, 128)) * r.uniform(0.5, 3, 128)
    a = r.integers(1, 4, 40).astype(float)
    Rw, ew = o.calibrate_rotation(X, a)
    Rd, ed = o.calibrate_rotation(np.repeat(X, a.astype(int), axis=0))
    assert np.allclose(ew, ed, rtol=1e-10, atol=1e-12)
    Rs, es = o.calibrate_rotation(X + 7.0, a)                 # the weighted mean is removed
    assert np.allclose(es, ew, rtol=1e-9, atol=1e-9)
    top = ew[:-1] - ew[1:] > 1e-3 * ew[0]                     # well-separated directions are unique
    ok = np.abs(np.sum(Rw * Rd, axis=1))[:-1][top]
    assert np.all(ok > 1 - 1e-8)


def test_calibration_eigen_equation_and_degenerate_cases():
    r = np.random.default_rng(10)
    X = r.standard_normal((300, 128)) * np.linspace(0.2, 3, 128)
    R, ev = o.calibrate_rotation(X)
    C = np.cov(X, rowvar=False, bias=True)
    assert np.allclose(R @ R.T, np.eye(128), atol=1e-10)
    assert np.allclose(R @ C @ R.T, np.diag(ev), atol=1e-9 * ev[0])
    assert np.all(np.diff(ev) <= 1e-12)
    R1, e1 = o.calibrate_rotation(X[:1])
    assert np.array_equal(R1, np.eye(128)) and not e1.any()
    R0, _ = o.calibrate_rotation(X, np.zeros(300))
    assert np.array_equal(R0, np.eye(128))


# ---------------------------------------------------------------- eviction and compaction

def _stream(r, n):
    K = (r.standard_normal((n, 128)) * 2 + np.linspace(0, 1, n)[:, None]).astype(F16)
    V = (r.standard_normal((n, 128)) * 1.5 + 0.3).astype(F16)
    return K, V, r.integers(0, 3, n).astype(np.uint8)


def _fresh(key_codec, bits=2, G=32, seed=0):
    cb = o.make_codebook(bits)
    r = np.random.default_rng(seed)
    R = np.stack([np.linalg.qr(r.standard_normal((128, 128)))[0] for _ in range(3)]).astype(F32)
    return o.OracleUnit(128, G, cb, o.hadamard_signs(99, 128), R, 4, 2048, key_codec=key_codec)


@pytest.mark.parametrize("key_codec,bits,G", [("omni", 2, 32), ("omni", 4, 64), ("turbo", 2, 32)])
def test_eviction_fused_decode_equals_attention_over_live_tokens(key_codec, bits, G):
    """Masked fused decode = brute-force softmax over the explicitly dequantized
    live tokens; deleted tokens' data does not matter; deleting all gives zeros."""
    r = np.random.default_rng(31)
    u = _fresh(key_codec, bits, G)
    K, V, mod = _stream(r, 203)
    u.append(K[:150], V[:150], mod[:150])
    u.append(K[150:], V[150:], mod[150:])
    for a, b in ((0, 3), (40, 97), (130, 131), (195, 203)):     # sinks, whole groups, a tail token
        u.evict(a, b)
    q = (r.standard_normal((4, 128)) * 1.5).astype(F16)
    out = u.decode(q)
    assert np.max(np.abs(out - u.decode_bruteforce(q))) < 1e-10
    Kh, Vh = u.dequantized()
    live = ~u.dead[:u.T]
    s = q.astype(F64) @ Kh[live].T / math.sqrt(128)
    p = np.exp(s - s.max(1, keepdims=True))
    assert np.max(np.abs(out - (p / p.sum(1, keepdims=True)) @ Vh[live])) < 1e-10
    # a deleted token's codes can be anything
    u.vcodes[50] ^= 1
    u.vnorm[50] = F16(100.0)
    u.kcodes[60] ^= 1
    assert np.array_equal(u.decode(q), out)
    u.evict(0, u.T)
    assert np.all(u.decode(q) == 0) and np.all(u.decode_bruteforce(q) == 0)
    with pytest.raises(ValueError):
        u.evict(10, u.T + 1)


def _brute_plan(dead, T, gran, min_pages):
    """Every granule-aligned suffix start, packed explicitly; the largest start that
    saves enough pages."""
    best = None
    for sg in range(-(-T // gran)):
        slots = list(range(sg * gran))
        for j in range(sg, -(-T // gran)):
            toks = list(range(j * gran, min((j + 1) * gran, T)))
            if not all(dead[t] for t in toks):
                slots += toks
        if -(-T // 64) - (-(-len(slots) // 64)) >= min_pages:
            best = (sg, len(slots))
    return best


def test_suffix_plan_is_the_shortest_suffix_saving_enough_pages():
    r = np.random.default_rng(5)
    for trial in range(300):
        gran = int(r.choice([16, 32, 64]))
        T = int(r.integers(1, 700))
        dead = np.zeros(T, bool)
        for _ in range(int(r.integers(0, 8))):                  # runs of deletions
            a = int(r.integers(0, T))
            dead[a:a + int(r.integers(1, 200))] = True
        if trial % 7 == 0:
            dead[:] = True
        mp = int(r.integers(1, 5))
        plan = o.plan_suffix_compaction(dead, T, gran, mp)
        ref = _brute_plan(dead, T, gran, mp)
        if ref is None:
            assert plan is None
            continue
        sg, T2, moves = plan
        assert (sg, T2) == ref
        assert all(d < s for s, d in moves) and moves == sorted(moves)
        assert [d for _, d in moves] == sorted(set(d for _, d in moves))
    with pytest.raises(ValueError):
        o.plan_suffix_compaction(np.zeros(10, bool), 10, 32, 0)


@pytest.mark.parametrize("key_codec,bits,G", [("omni", 2, 32), ("omni", 4, 64), ("turbo", 2, 32)])
def test_compaction_equals_never_having_appended_the_removed_granules(key_codec, bits, G):
    """Evict, compact: the state equals a cache that received only the surviving
    granules (same partial deletions), and stays equal after further appends
    (the trailing group continues in its new place). Decode is unchanged."""
    r = np.random.default_rng(77 + bits + G)
    gran = o.compaction_granule(key_codec, G)
    n = 64 * 7 + 37                                              # ragged: the last granule is partial
    K, V, mod = _stream(r, n + 90)
    A = _fresh(key_codec, bits, G)
    for a, b in ((0, 100), (100, 300), (300, n)):
        A.append(K[a:b], V[a:b], mod[a:b])
    ng = -(-n // gran)
    dead = np.zeros(n, bool)
    for j in (1, 3, 4, ng - 3):                                  # whole granules, one of them early
        dead[j * gran:(j + 1) * gran] = True
    dead[5:9] = True                                             # partial deletions
    dead[6 * gran + 3:6 * gran + 7] = True
    for t in np.nonzero(dead)[0]:
        A.evict(int(t), int(t) + 1)
    q = (r.standard_normal((4, 128)) * 1.5).astype(F16)
    before = A.decode(q)
    plan = o.plan_suffix_compaction(A.dead, A.T, gran, 1)
    assert plan is not None
    sg, T2, moves = plan
    A.move_granules(moves, gran, T2)
    assert np.allclose(A.decode(q), before, rtol=1e-12, atol=1e-12)
    # the same tokens appended without the removed granules
    keep = np.ones(n, bool)
    for j in range(sg, ng):
        if dead[j * gran:min((j + 1) * gran, n)].all():
            keep[j * gran:(j + 1) * gran] = False
    idx = np.nonzero(keep)[0]
    assert len(idx) == T2
    B = _fresh(key_codec, bits, G)
    B.append(K[idx], V[idx], mod[idx])
    for t in np.nonzero(dead[idx])[0]:
        B.evict(int(t), int(t) + 1)
    ea, eb = A.export(), B.export()
    for key in eb:
        assert np.array_equal(ea[key], eb[key]), key
    A.append(K[n:], V[n:], mod[n:])
    B.append(K[n:], V[n:], mod[n:])
    ea, eb = A.export(), B.export()
    for key in eb:
        assert np.array_equal(ea[key], eb[key]), key
    assert np.allclose(A.decode(q), B.decode(q), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- pseudo-token far memory

def _far(r, n_proto, per, scale=1.0):
    c = r.standard_normal((n_proto, 128)) * 2.0                              # prototype centres
    kf = (np.repeat(c, per, axis=0) + 0.3 * r.standard_normal((n_proto * per, 128))) * scale
    vf = np.repeat(r.standard_normal((n_proto, 128)), per, axis=0) + 0.2 * r.standard_normal((n_proto * per, 128))
    return kf.astype(F16), vf.astype(F16)


@pytest.mark.parametrize("key_codec", ["omni", "turbo"])
def test_log_mass_bias_equals_duplicated_pseudo_tokens(key_codec):
    """b_k = log n_k is exactly the effect of n_k copies of each of the
    prototype's pseudo tokens (the pages' motivation for the bias): integer masses
    against brute-force attention over [dequantized near window; repeated far
    tokens] with no bias; inactive prototypes (n = 0) contribute nothing."""
    r = np.random.default_rng(41)
    u = _fresh(key_codec)
    K, V, mod = _stream(r, 150)
    u.append(K, V, mod)
    u.evict(20, 40)
    P, S = 6, 4
    kf, vf = _far(r, P, S)
    mass = np.array([1, 3, 0, 7, 2, 12], np.float32)
    q = (r.standard_normal((4, 128)) * 1.2).astype(F16)
    out = u.decode_with_pseudo(q, kf, vf, mass, S)
    Kh, Vh = u.dequantized()
    live = ~u.dead[:u.T]
    reps = np.repeat(mass.astype(int), S)
    Kall = np.concatenate([Kh[live], np.repeat(kf.astype(F64), reps, axis=0)])
    Vall = np.concatenate([Vh[live], np.repeat(vf.astype(F64), reps, axis=0)])
    s = q.astype(F64) @ Kall.T / math.sqrt(128)
    p = np.exp(s - s.max(1, keepdims=True))
    assert np.max(np.abs(out - (p / p.sum(1, keepdims=True)) @ Vall)) < 1e-10


def test_pseudo_decode_reduces_to_plain_decode_and_to_far_only():
    r = np.random.default_rng(42)
    u = _fresh("omni")
    K, V, mod = _stream(r, 203)
    u.append(K, V, mod)
    q = (r.standard_normal((4, 128)) * 1.5).astype(F16)
    kf, vf = _far(r, 5, 8)
    assert np.max(np.abs(u.decode_with_pseudo(q, kf[:0], vf[:0], np.zeros(0), 8) - u.decode(q))) < 1e-12
    assert np.max(np.abs(u.decode_with_pseudo(q, kf, vf, np.zeros(5), 8) - u.decode(q))) < 1e-12
    e = _fresh("omni")                                                       # empty near window
    mass = np.array([2.5, 1.0, 4.0, 0.5, 9.0])
    s = q.astype(F64) @ kf.astype(F64).T / math.sqrt(128) + np.log(np.repeat(mass, 8))[None]
    p = np.exp(s - s.max(1, keepdims=True))
    ref = (p / p.sum(1, keepdims=True)) @ vf.astype(F64)
    assert np.max(np.abs(e.decode_with_pseudo(q, kf, vf, mass, 8) - ref)) < 1e-12
    assert np.all(e.decode_with_pseudo(q, kf, vf, np.zeros(5), 8) == 0)
