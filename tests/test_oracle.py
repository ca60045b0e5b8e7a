"""Pins for the CPU oracle (no GPU).

The oracle is checked against facts fixed by the KATA paper and by mathematics,
never against itself:

  * printed values: the packed width 2080 at d = 64 (Sec. 4.1) and the rotary
    factor r_KATA = cos^2(0.1024) = 0.9896 (Sec. 5.3), both in tests/golden/;
  * the lift identity <psi(u), psi(v)> = <u u^T, v v^T>_F = (u^T v)^2 and
    ||psi(u)|| = ||u||^2 (Sec. 3.1, Thm. 4);
  * closed forms: equal keys give the running mean of the values; orthonormal
    keys give exact recall (the zero-interference case);
  * Prop. 1: o_1 = v_1, outputs lie in the convex hull of the values, and the
    convex-gate recursion o_t = alpha_t o_{t|t-1} + beta_t v_t;
  * invariances implied by the squared kernel and the ratio (rotation, scale,
    sign flips of keys);
  * brute force in exact rational arithmetic through the Frobenius route on
    tiny integer inputs;
  * the oracle's two self-check forms (Eq. 2 recurrence, Algorithm 1 /
    Eq. 17-20 at several chunk sizes) and the decode step.

Each pin set is also run against numpy mutants with one planted mistake each,
to show that a plausible error (exclusive mask, missing square, transposed
q/k, missing normaliser, ...) fails at least one pin.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _rand_qkv(rng, B=2, H=2, T=37, d=8, dv=5, sphere=True):
    q = rng.standard_normal((B, H, T, d))
    k = rng.standard_normal((B, H, T, d))
    if sphere:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    return q, k, v


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------- lift


def test_feature_width_printed():
    (d, direct, packed), = _golden_rows("feature_widths.txt")
    d, direct, packed = int(d), int(direct), int(packed)
    assert oracle.feature_dim(d) == packed
    assert d * d == direct
    assert oracle.lift(np.ones(d)).shape == (packed,)


@pytest.mark.parametrize("d", [1, 2, 3, 7, 16, 31, 32, 64])
def test_lift_identity_random(d):
    rng = np.random.default_rng(d)
    u = rng.standard_normal((64, d))
    w = rng.standard_normal((64, d))
    pu, pw = oracle.lift(u), oracle.lift(w)
    got = np.sum(pu * pw, axis=-1)
    want = np.einsum("ri,ri->r", u, w) ** 2
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # Frobenius route: <u u^T, w w^T>_F
    frob = np.einsum("rij,rij->r", np.einsum("ri,rj->rij", u, u), np.einsum("ri,rj->rij", w, w))
    np.testing.assert_allclose(got, frob, rtol=1e-12, atol=1e-12)
    # ||psi(u)||_2 = ||u||^2  (= 1 on the sphere, Sec. 3.1)
    np.testing.assert_allclose(np.linalg.norm(pu, axis=-1), np.sum(u * u, axis=-1), rtol=1e-12)


@pytest.mark.parametrize("d", [2, 5, 32, 64])
def test_lift_identity_adversarial(d):
    rng = np.random.default_rng(100 + d)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    e = np.eye(d)
    cases = [
        (e[0], e[0], 1.0),            # axis aligned
        (e[0], e[d - 1], 0.0),        # orthogonal axes
        (u, -u, 1.0),                 # antipodal: squared kernel is sign blind
        (u, u, 1.0),                  # identical unit vectors
        (3.0 * u, -2.0 * u, 36.0),    # scaled
    ]
    v = rng.standard_normal(d)
    v -= v.dot(u) * u                 # exactly orthogonal to u (up to rounding)
    cases.append((u, v, u.dot(v) ** 2))
    for a, b, want in cases:
        got = float(np.dot(oracle.lift(a), oracle.lift(b)))
        assert abs(got - want) <= 1e-12 * max(1.0, abs(want)), (a, b, got, want)


def test_lift_unpacks_to_outer_product():
    """The stated packing: upper triangle row-major, sqrt(2) off the diagonal."""
    rng = np.random.default_rng(7)
    for d in (1, 4, 16, 33):
        x = rng.standard_normal(d)
        phi = oracle.lift(x)
        M = np.zeros((d, d))
        f = 0
        for i in range(d):
            for j in range(i, d):
                val = phi[f] if i == j else phi[f] / math.sqrt(2.0)
                M[i, j] = M[j, i] = val
                f += 1
        assert f == phi.shape[0]
        np.testing.assert_allclose(M, np.outer(x, x), rtol=1e-14, atol=1e-14)
    # position of a single off-diagonal pair (i, j) = (1, 3) at d = 4: f = 1*4 - 0 + 2 = 6
    x = np.zeros(4)
    x[1] = x[3] = 1.0
    phi = oracle.lift(x)
    assert np.flatnonzero(np.abs(phi) > 0).tolist() == [4, 6, 9]
    assert phi[6] == pytest.approx(math.sqrt(2.0))


def test_printed_rope_factor_lift():
    (angle, printed, decimals), = _golden_rows("rope_factor.txt")
    a, printed, decimals = float(angle), float(printed), int(decimals)
    for d in (2, 16, 64):
        q = np.zeros(d)
        k = np.zeros(d)
        q[0] = 1.0
        k[0], k[1] = math.cos(a), math.sin(a)
        r = float(np.dot(oracle.lift(q), oracle.lift(k)))
        assert round(r, decimals) == printed


# ------------------------------------------------------------------- pin checks
# Each check takes a forward implementation fwd(q, k, v) -> o and raises
# AssertionError when the pin fails.


def check_rope_forward(fwd, tol=1e-12):
    (angle, printed, decimals), = _golden_rows("rope_factor.txt")
    a, printed, decimals = float(angle), float(printed), int(decimals)
    d = 4
    q = np.zeros((1, 1, 2, d))
    k = np.zeros((1, 1, 2, d))
    v = np.zeros((1, 1, 2, 1))
    q[0, 0, :, 0] = 1.0
    k[0, 0, 0, 0] = 1.0                              # aligned key: weight 1
    k[0, 0, 1, 0], k[0, 0, 1, 1] = math.cos(a), math.sin(a)
    v[0, 0, 1, 0] = 1.0
    o = fwd(q, k, v)[0, 0, 1, 0]                     # = r / (1 + r)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = o / (1.0 - o)
    assert round(r, decimals) == printed, r


def check_equal_keys_mean(fwd, tol=1e-12):
    rng = np.random.default_rng(11)
    B, H, T, d, dv = 1, 2, 29, 6, 3
    kk = rng.standard_normal(d)
    kk /= np.linalg.norm(kk)
    q = rng.standard_normal((B, H, T, d)) + 3.0 * kk   # |q.k| bounded away from 0
    k = np.broadcast_to(kk, (B, H, T, d)).copy()
    v = rng.standard_normal((B, H, T, dv))
    o = fwd(q, k, v)
    want = np.cumsum(v, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    assert _rel(o, want) < tol


def check_orthonormal_recall(fwd, tol=1e-12):
    B, H, d, dv = 1, 1, 8, 4
    T = d
    rng = np.random.default_rng(12)
    k = np.eye(d)[None, None]                        # k_s = e_s
    v = rng.standard_normal((B, H, T, dv))
    for j in range(d):
        q = np.zeros((B, H, T, d))
        q[..., j] = 1.0                              # q_t = e_j for all t
        o = fwd(q, k, v)
        for t in range(T):
            want = v[0, 0, j] if t >= j else np.zeros(dv)
            assert np.max(np.abs(o[0, 0, t] - want)) < tol, (j, t)


def check_first_token(fwd, tol=1e-12):
    rng = np.random.default_rng(13)
    q, k, v = _rand_qkv(rng, B=2, H=3, T=5, d=7, dv=4)
    o = fwd(q, k, v)
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0])) < tol


def check_convex_hull(fwd, tol=1e-12):
    rng = np.random.default_rng(14)
    q, k, v = _rand_qkv(rng, B=2, H=2, T=40, d=5, dv=6, sphere=False)
    o = fwd(q, k, v)
    lo = np.minimum.accumulate(v, axis=2)
    hi = np.maximum.accumulate(v, axis=2)
    assert np.all(o >= lo - tol) and np.all(o <= hi + tol)


def check_prop1_recursion(fwd, tol=1e-12):
    """o_t = (D_{t-1}/D_t) obar_{t|t-1} + (c_t/D_t) v_t, where obar uses the
    current query against the previous state (Prop. 1)."""
    rng = np.random.default_rng(15)
    q, k, v = _rand_qkv(rng, B=1, H=1, T=12, d=5, dv=3)
    o = fwd(q, k, v)[0, 0]
    for t in range(1, 12):
        qt = q[0, 0, t]
        prev = np.einsum("sd,d->s", k[0, 0, :t], qt) ** 2     # c_s for s < t
        D_prev = prev.sum()
        c_t = np.dot(qt, k[0, 0, t]) ** 2
        D_t = D_prev + c_t
        alpha, beta = D_prev / D_t, c_t / D_t
        assert alpha >= 0 and beta >= 0 and abs(alpha + beta - 1) < 1e-15
        qq = q[:, :, : t].copy()
        qq[0, 0, t - 1] = qt                       # current query, previous state
        obar = fwd(qq, k[:, :, :t], v[:, :, :t])[0, 0, t - 1]
        want = alpha * obar + beta * v[0, 0, t]
        assert np.max(np.abs(o[t] - want)) < tol, t


def check_invariances(fwd, tol=1e-12):
    rng = np.random.default_rng(16)
    q, k, v = _rand_qkv(rng, B=1, H=2, T=33, d=6, dv=4, sphere=False)
    base = fwd(q, k, v)
    U, _ = np.linalg.qr(rng.standard_normal((6, 6)))
    tol = max(tol, 1e-11)
    assert _rel(fwd(q @ U.T, k @ U.T, v), base) < tol             # common rotation
    a = rng.uniform(0.5, 3.0, size=(1, 2, 33, 1)) * rng.choice([-1, 1], size=(1, 2, 33, 1))
    assert _rel(fwd(q * a, k, v), base) < tol                     # per-query scale/sign
    assert _rel(fwd(q, 2.5 * k, v), base) < tol                   # common key scale
    s = rng.choice([-1.0, 1.0], size=(1, 2, 33, 1))
    assert _rel(fwd(q, k * s, v), base) < tol                     # key sign flips


def _exact_forward(q, k, v):
    """Exact rationals through the Frobenius route <q q^T, k k^T>_F."""
    T, d = q.shape
    dv = v.shape[1]
    out = []
    for t in range(T):
        num = [Fraction(0)] * dv
        den = Fraction(0)
        for s in range(t + 1):
            w = Fraction(0)
            for i in range(d):
                for j in range(d):
                    w += Fraction(int(q[t, i]) * int(q[t, j])) * Fraction(int(k[s, i]) * int(k[s, j]))
            den += w
            for jj in range(dv):
                num[jj] += w * Fraction(int(v[s, jj]))
        out.append([float(x / den) if den != 0 else 0.0 for x in num])
    return np.array(out)


def check_bruteforce_exact(fwd, tol=1e-12):
    rng = np.random.default_rng(17)
    for T, d, dv in [(1, 1, 1), (3, 2, 2), (6, 3, 2), (8, 4, 3)]:
        for _ in range(3):
            q = rng.integers(-3, 4, size=(T, d)).astype(np.float64)
            k = rng.integers(-3, 4, size=(T, d)).astype(np.float64)
            v = rng.integers(-5, 6, size=(T, dv)).astype(np.float64)
            got = fwd(q[None, None], k[None, None], v[None, None])[0, 0]
            want = _exact_forward(q, k, v)
            assert np.max(np.abs(got - want)) <= tol * max(1.0, np.max(np.abs(want)))


ALL_CHECKS = [check_rope_forward, check_equal_keys_mean, check_orthonormal_recall,
              check_first_token, check_convex_hull, check_prop1_recursion,
              check_invariances, check_bruteforce_exact]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_forward_pins(check):
    check(oracle.forward)


# The feature-space forms sum psi(q)_f psi(k)_f with mixed signs, so they lose
# up to log10(|q|^2 |k|^2 / (q.k)^2) digits to cancellation; 1e-9 covers the
# conditioning of these inputs.
FEATURE_FORM_TOL = 1e-9


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_recurrent_pins(check):
    check(oracle.recurrent, tol=FEATURE_FORM_TOL)


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_chunked_pins(check):
    check(lambda q, k, v: oracle.chunked(q, k, v, 3), tol=FEATURE_FORM_TOL)


# ------------------------------------------------------------- planted mistakes


def _mutant(kind):
    def fwd(q, k, v):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        T = q.shape[2]
        s = np.einsum("bhtd,bhsd->bhts", q, k)
        if kind == "transposed_qk":
            s = np.swapaxes(s, -1, -2)
        w = np.abs(s) if kind == "no_square" else s * s
        mask = np.tril(np.ones((T, T)), -1 if kind == "exclusive_mask" else 0)
        if kind == "anticausal":
            mask = mask.T
        w = w * mask
        num = np.einsum("bhts,bhsj->bhtj", w, v)
        den = w.sum(-1, keepdims=True)
        if kind == "no_normaliser":
            return num
        if kind == "den_plus_one":
            den = den + 1.0
        with np.errstate(invalid="ignore", divide="ignore"):
            o = np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)
        if kind == "off_by_one_row":
            o = np.concatenate([o[:, :, :1], o[:, :, :-1]], axis=2)
        return o
    return fwd


def test_reference_numpy_form_passes_pins():
    """The unmutated numpy form passes every pin (so mutants fail for their mistake)."""
    for check in ALL_CHECKS:
        check(_mutant("none"))


@pytest.mark.parametrize("kind", ["transposed_qk", "no_square", "exclusive_mask", "anticausal",
                                  "no_normaliser", "den_plus_one", "off_by_one_row"])
def test_planted_mistake_fails_a_pin(kind):
    fwd = _mutant(kind)
    failed = []
    for check in ALL_CHECKS:
        try:
            check(fwd)
        except (AssertionError, ZeroDivisionError, FloatingPointError):
            failed.append(check.__name__)
    assert failed, f"mutant {kind} passed every pin"


def test_planted_lift_mistakes_fail():
    x = np.array([0.3, -1.2, 0.7, 2.0])
    y = np.array([1.1, 0.4, -0.9, 0.2])
    want = np.dot(x, y) ** 2

    def no_sqrt2(z):
        return np.array([z[i] * z[j] for i in range(4) for j in range(i, 4)])

    def column_major_upper(z):
        r2 = math.sqrt(2.0)
        return np.array([z[i] * z[j] * (1 if i == j else r2) for j in range(4) for i in range(j + 1)])

    assert abs(np.dot(no_sqrt2(x), no_sqrt2(y)) - want) > 1e-3
    # another packing order keeps the identity but not the stated layout
    other = column_major_upper(x)
    assert abs(np.dot(other, column_major_upper(y)) - want) < 1e-12
    assert not np.allclose(other, oracle.lift(x))


# ------------------------------------------------------- self-check agreement


@pytest.mark.parametrize("T,C", [(1, 4), (7, 3), (32, 8), (37, 8), (50, 50), (50, 64)])
def test_chunked_and_recurrent_equal_direct(T, C):
    rng = np.random.default_rng(T * 100 + C)
    q, k, v = _rand_qkv(rng, B=2, H=2, T=T, d=6, dv=5)
    ref = oracle.forward(q, k, v)
    assert _rel(oracle.chunked(q, k, v, C), ref) < FEATURE_FORM_TOL
    assert _rel(oracle.recurrent(q, k, v), ref) < FEATURE_FORM_TOL


def test_forward_rows_equal_full():
    rng = np.random.default_rng(21)
    q, k, v = _rand_qkv(rng, B=2, H=3, T=45, d=5, dv=4)
    full = oracle.forward(q, k, v).reshape(-1, 4)
    rows = np.array([0, 1, 44, 45, 100, 200, 269])
    np.testing.assert_array_equal(oracle.forward_rows(q, k, v, rows), full[rows])


def test_zero_denominator_gives_zero():
    d = 4
    q = np.zeros((1, 1, 3, d))
    k = np.zeros((1, 1, 3, d))
    v = np.ones((1, 1, 3, 2))
    q[0, 0, :, 0] = 1.0
    k[0, 0, :2, 1] = 1.0          # first two keys orthogonal to the query
    k[0, 0, 2, 0] = 1.0
    o = oracle.forward(q, k, v)
    assert np.all(o[0, 0, :2] == 0.0)
    assert np.allclose(o[0, 0, 2], 1.0)


def test_decode_steps_equal_forward():
    rng = np.random.default_rng(22)
    B, H, T, d, dv = 2, 2, 9, 6, 3
    q, k, v = _rand_qkv(rng, B=B, H=H, T=T, d=d, dv=dv, sphere=False)
    ref = oracle.forward(q, k, v)
    n = oracle.feature_dim(d)
    S = np.zeros((B, H, n, dv))
    z = np.zeros((B, H, n))
    for t in range(T):
        S, z, o = oracle.decode_step(S, z, q[:, :, t], k[:, :, t], v[:, :, t])
        assert _rel(o, ref[:, :, t]) < FEATURE_FORM_TOL
    S2, z2 = oracle.prefix_state(k, v)
    assert _rel(S2, S) < 1e-12 and _rel(z2, z) < 1e-12
    # the state itself: S = sum psi(k) v^T, z = sum psi(k) (Eq. 2)
    pk = oracle.lift(k)
    assert _rel(z, pk.sum(axis=2)) < 1e-12
    assert _rel(S, np.einsum("bhtf,bhtj->bhfj", pk, v)) < 1e-12
