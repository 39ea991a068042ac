"""okvq_calibrate_rotations (the value-rotation calibration kernel) against the
oracle's calibrate_rotations on the same seeded calibration streams.

What is unique is compared directly: the eigenvalues (descending), and for an
eigenvalue separated from the others, its eigenvector with the sign rule (the
largest-magnitude entry positive). Where eigenvalues cluster (a rank-deficient
modality has a null space of near-zero eigenvalues; any basis of it is
correct), the cluster's projector is compared instead, and the GPU basis is
checked to be orthonormal and to diagonalise the oracle's covariance.
Degenerate modalities (no token, one token, zero total weight) give the
identity, exactly."""
import numpy as np
import pytest

from oracle import okvq_oracle as o
from bit_kv_cache_rht_gb300 import synth
import parity_util as pu

F64 = np.float64
EPS_C = 2e-5          # covariance + Jacobi error budget, relative to the largest eigenvalue


def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pu.ensure_built()
    return torch


def _run(torch, V, mod, M, weight=None):
    from bit_kv_cache_rht_gb300 import okvq
    Vd = torch.from_numpy(np.ascontiguousarray(V)).cuda()
    Md = torch.from_numpy(np.ascontiguousarray(mod)).cuda()
    Wd = None if weight is None else torch.from_numpy(np.ascontiguousarray(weight, np.float32)).cuda()
    rot, eig, sweeps = okvq.calibrate_rotations(Vd, Md, M, weight=Wd, return_sweeps=True)
    torch.cuda.synchronize()
    sw = sweeps.cpu().numpy()
    assert np.all(sw >= 0), "Jacobi did not converge: %s" % sw
    return rot.cpu().numpy().astype(F64), eig.cpu().numpy().astype(F64)


def _clusters(lam, delta):
    """Index ranges [a, b) of eigenvalues (descending) whose neighbours differ by < delta."""
    out, a = [], 0
    for i in range(1, len(lam) + 1):
        if i == len(lam) or lam[i - 1] - lam[i] >= delta:
            out.append((a, i))
            a = i
    return out


def _check_unit(Rg, lg, Ro, lo, what):
    d = len(lo)
    scale = max(float(lo[0]), 1e-30)
    tol = EPS_C * scale
    assert np.all(np.diff(lg) <= 0), what + ": eigenvalues not descending"
    np.testing.assert_allclose(lg, lo, rtol=0, atol=tol, err_msg=what + ": eigenvalues")
    assert np.max(np.abs(Rg @ Rg.T - np.eye(d))) < 2e-5, what + ": not orthonormal"
    C = Ro.T @ np.diag(lo) @ Ro                      # the oracle's covariance
    Dg = Rg @ C @ Rg.T
    assert np.max(np.abs(Dg - np.diag(np.diag(Dg)))) < 2 * tol, what + ": does not diagonalise"
    for a, b in _clusters(lo, 1e-3 * scale):
        rest = np.concatenate([lo[:a], lo[b:]])
        gap = np.min(np.abs(rest[:, None] - lo[None, a:b])) if len(rest) else scale
        bound = 10 * tol / gap
        if bound >= 0.5:
            continue                                 # nothing is determined at this separation
        Pg = Rg[a:b].T @ Rg[a:b]
        Po = Ro[a:b].T @ Ro[a:b]
        assert np.max(np.abs(Pg - Po)) < bound, "%s: eigenspace [%d, %d)" % (what, a, b)
        if b == a + 1:
            mag = np.sort(np.abs(Ro[a]))[::-1]
            if mag[0] - mag[1] > 2 * bound:          # the sign rule decides unambiguously
                assert np.max(np.abs(Rg[a] - Ro[a])) < bound, "%s: eigenvector %d" % (what, a)
    for i in range(d):                               # the sign rule, on the GPU's own vectors
        j = int(np.argmax(np.abs(Rg[i])))
        assert Rg[i, j] > 0, "%s: row %d sign" % (what, i)


def _check_all(Rg, lg, Ro, lo, what):
    L, H, M = Ro.shape[:3]
    for l in range(L):
        for h in range(H):
            for m in range(M):
                if not np.any(lo[l, h, m]):
                    assert np.array_equal(Rg[l, h, m], np.eye(Ro.shape[-1])), "%s (%d,%d,%d): identity" % (
                        what, l, h, m)
                    assert not np.any(lg[l, h, m])
                    continue
                _check_unit(Rg[l, h, m], lg[l, h, m], Ro[l, h, m], lo[l, h, m], "%s (%d,%d,%d)" % (what, l, h, m))


@pytest.mark.gpu
def test_calibration_tiny_slice_unweighted():
    torch = _gpu()
    w = synth.tiny(seed=5)
    V, mod = w.calibration_slice()
    Ro, lo = o.calibrate_rotations(V, mod, 3)
    Rg, lg = _run(torch, V, mod, 3)
    _check_all(Rg, lg, Ro, lo, "tiny")


@pytest.mark.gpu
def test_calibration_full_model_slice():
    """Every (layer, kv head, modality) of the 36-layer model's calibration slice:
    the launch the benchmark makes (216 CTAs)."""
    torch = _gpu()
    w = synth.qwen3b()
    V, mod = w.calibration_slice()
    Ro, lo = o.calibrate_rotations(V, mod, 3)
    Rg, lg = _run(torch, V, mod, 3)
    _check_all(Rg, lg, Ro, lo, "qwen3b")


@pytest.mark.gpu
def test_calibration_attention_weighted():
    """Contribution weights a_t >= 0 per (token, layer, kv head): attention-like
    (a softmax of random scores, summing to 1 per unit) with a quarter of the
    tokens given weight 0."""
    torch = _gpu()
    w = synth.tiny(seed=6)
    r = np.random.default_rng(11)
    V, mod = w.calibration_slice()
    V = np.concatenate([V, V[:, :1]], axis=1)              # 2 layers
    n, L, H = V.shape[:3]
    s = r.standard_normal((n, L, H)) * 2.0
    a = np.exp(s - s.max(0, keepdims=True))
    a /= a.sum(0, keepdims=True)
    a[r.random((n, L, H)) < 0.25] = 0.0
    a = a.astype(np.float32)
    Ro, lo = o.calibrate_rotations(V, mod, 3, a)
    Rg, lg = _run(torch, V, mod, 3, a)
    _check_all(Rg, lg, Ro, lo, "weighted")
    # the weights matter: the weighted spectrum is not the plain one
    _, lp = o.calibrate_rotations(V, mod, 3)
    assert np.max(np.abs(lp - lg)) > 0.1 * np.max(lp)


@pytest.mark.gpu
def test_calibration_long_stream_and_ragged_modalities():
    """4,099 tokens in irregular order; modality 2 never occurs and ids 5 and 9
    (beyond the modality count) are ignored."""
    torch = _gpu()
    r = np.random.default_rng(12)
    n, L, H = 4099, 1, 3
    scale = np.exp(r.uniform(np.log(0.3), np.log(5.0), (L, H, 128)))
    mod = r.choice(np.array([0, 1, 5, 9], np.uint8), n, p=[0.55, 0.35, 0.05, 0.05]).astype(np.uint8)
    V = (r.standard_normal((n, L, H, 128)) * scale[None] + 3.0).astype(np.float16)
    Ro, lo = o.calibrate_rotations(V, mod, 3)
    Rg, lg = _run(torch, V, mod, 3)
    assert not np.any(lo[:, :, 2])
    _check_all(Rg, lg, Ro, lo, "long")


@pytest.mark.gpu
def test_calibration_constructed_spectrum():
    """Tokens built so that the covariance has a known orthonormal eigenbasis U and
    well-separated eigenvalues (+-sqrt(lambda) along each axis, mirrored): both
    sides recover U, signed by the rule."""
    torch = _gpu()
    r = np.random.default_rng(13)
    U, _ = np.linalg.qr(r.standard_normal((128, 128)))
    lam = np.linspace(9.0, 0.5, 128)
    X = np.concatenate([np.sqrt(lam)[:, None] * U.T, -np.sqrt(lam)[:, None] * U.T]) * np.sqrt(128)
    V = X.astype(np.float16)[:, None, None, :]
    mod = np.zeros(256, np.uint8)
    Ro, lo = o.calibrate_rotations(V, mod, 1)
    Rg, lg = _run(torch, V, mod, 1)
    _check_all(Rg, lg, Ro, lo, "constructed")
    Us = U.T * np.sign(U.T[np.arange(128), np.argmax(np.abs(U.T), axis=1)])[:, None]
    assert np.max(np.abs(Rg[0, 0, 0] - Us)) < 0.1         # fp16 rounding of the tokens moves U slightly


@pytest.mark.gpu
def test_calibration_degenerate_modalities_give_identity():
    torch = _gpu()
    r = np.random.default_rng(14)
    n = 200
    V = r.standard_normal((n, 1, 2, 128)).astype(np.float16)
    mod = np.zeros(n, np.uint8)
    mod[7] = 1                                             # modality 1: one token
    mod[100:150] = 2                                       # modality 2: weight 0 below
    a = np.ones((n, 1, 2), np.float32)
    a[100:150] = 0.0
    Rg, lg = _run(torch, V, mod, 3, a)
    for h in range(2):
        for m in (1, 2):
            assert np.array_equal(Rg[0, h, m], np.eye(128)) and not np.any(lg[0, h, m])
    Ro, lo = o.calibrate_rotations(V, mod, 3, a)
    _check_all(Rg, lg, Ro, lo, "degenerate")
    # no calibration token at all: every modality gets the identity
    from bit_kv_cache_rht_gb300 import okvq
    rot = torch.full((1, 2, 3, 128, 128), float("nan"), device="cuda")
    st = okvq.okvq_calibrate_rotations(1, 2, 3, 0, 0, 0, 0, rot.data_ptr(), 0, 0)
    torch.cuda.synchronize()
    assert st == okvq.OKVQ_OK
    assert torch.equal(rot.cpu(), torch.eye(128).expand(1, 2, 3, 128, 128))


def test_calibration_rejects_bad_arguments_before_cuda():
    pu.ensure_built()
    from bit_kv_cache_rht_gb300 import okvq
    E = okvq.OKVQ_EINVAL
    assert okvq.okvq_calibrate_rotations(0, 2, 3, 1, 1, 0, 10, 1, 0, 0) == E       # no layer
    assert okvq.okvq_calibrate_rotations(1, 2, 4, 1, 1, 0, 10, 1, 0, 0) == E       # more modalities than slots
    assert okvq.okvq_calibrate_rotations(1, 2, 3, 1, 1, 0, -1, 1, 0, 0) == E       # negative token count
    assert okvq.okvq_calibrate_rotations(1, 2, 3, 1, 1, 0, 10, 0, 0, 0) == E       # no output
    assert okvq.okvq_calibrate_rotations(1, 2, 3, 0, 1, 0, 10, 1, 0, 0) == E       # tokens but no values
