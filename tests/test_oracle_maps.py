"""Pins for the oracle's reduced PSD families (no GPU).

[KATA] Sec. 4.1 ("two reduced PSD families") cuts u in R^d into g blocks u_a
of width m = d/g and defines

  * KATA-M_g:     psi(u) = (u_1 u_1^T, ..., u_g u_g^T),
                  <psi(q), psi(k)> = sum_a (q_a . k_a)^2, state g m(m+1)/2 x d_v;
  * KATA-Sigma_g: psi(u) = sum_a u_a u_a^T,
                  <psi(q), psi(k)>_F = sum_{a,b} (q_a . k_b)^2, state m(m+1)/2 x d_v,

and states that both recover the full rank-one map at g = 1.  The Sigma
configuration adds eps I (eps = 1e-4) and a scale s (1/4 for Sigma_4), so
psi(u) = eps I + s sum_a u_a u_a^T and, expanding the Frobenius product,
<psi(q), psi(k)> = eps^2 m + eps s (|q|^2 + |k|^2) + s^2 sum_{a,b} (q_a . k_b)^2.

The oracle computes the weights as entrywise products of the map's matrices
and the lift by packing those matrices; these tests pin both to the printed
inner-product identities and state sizes, to the g = 1 reduction, to the block
structure (through the already pinned full lift and forward), to the
equal-keys closed form and the convex-hull invariant, and to the packed
recurrence.  Planted mistakes in a numpy copy of the weight fail them.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

CASES = [("M", 16, 2), ("M", 32, 4), ("M", 64, 2), ("Sigma", 16, 2), ("Sigma", 32, 4),
         ("Sigma", 64, 2)]


def _blocks(x, g):
    m = x.shape[-1] // g
    return [x[..., a * m:(a + 1) * m] for a in range(g)]


def _closed_form(q, k, map_name, g, eps, s):
    """The printed inner-product identities (plus the eps/scale expansion)."""
    qb, kb = _blocks(q, g), _blocks(k, g)
    if map_name == "M":
        return sum(float(qa @ ka) ** 2 for qa, ka in zip(qb, kb))
    m = q.shape[-1] // g
    cross = sum(float(qa @ kb_) ** 2 for qa in qb for kb_ in kb)
    return eps * eps * m + eps * s * (float(q @ q) + float(k @ k)) + s * s * cross


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _rand_qkv(rng, B=1, H=2, T=29, d=16, dv=5):
    q = rng.standard_normal((B, H, T, d)) / np.sqrt(d)
    k = rng.standard_normal((B, H, T, d)) / np.sqrt(d)
    v = rng.standard_normal((B, H, T, dv))
    return q, k, v


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("g", [1, 2, 4])
def test_map_widths_are_the_printed_state_sizes(d, g):
    m = d // g
    assert oracle.map_dim("Sigma", d, g) == m * (m + 1) // 2
    assert oracle.map_dim("M", d, g) == g * m * (m + 1) // 2 == d * (d // g + 1) // 2
    assert oracle.map_dim("full", d, 1) == d * (d + 1) // 2
    # the packed lift has exactly that many coordinates
    x = np.ones((3, d))
    assert oracle.lift_map(x, "M", g).shape == (3, oracle.map_dim("M", d, g))
    assert oracle.lift_map(x, "Sigma", g).shape == (3, oracle.map_dim("Sigma", d, g))


@pytest.mark.parametrize("map_name,d,g", CASES)
@pytest.mark.parametrize("eps,s", [(0.0, 1.0), (1e-4, 1.0), (1e-4, 0.25), (0.3, 2.0)])
def test_lift_inner_product_is_the_closed_form(map_name, d, g, eps, s):
    rng = np.random.default_rng(d * 10 + g)
    for _ in range(20):
        q, k = rng.standard_normal(d), rng.standard_normal(d)
        e, sc = (eps, s) if map_name == "Sigma" else (0.0, 1.0)
        pq = oracle.lift_map(q, map_name, g, e, sc)
        pk = oracle.lift_map(k, map_name, g, e, sc)
        want = _closed_form(q, k, map_name, g, e, sc)
        assert abs(float(pq @ pk) - want) <= 1e-12 * max(1.0, abs(want))


@pytest.mark.parametrize("d", [16, 32, 64])
def test_g1_recovers_the_full_map(d):
    x = np.random.default_rng(d).standard_normal((4, d))
    full = oracle.lift(x)   # equal up to the rounding order of sqrt(2) x_i x_j
    assert _rel(oracle.lift_map(x, "M", 1), full) <= 1e-15
    assert _rel(oracle.lift_map(x, "Sigma", 1, 0.0, 1.0), full) <= 1e-15
    assert _rel(oracle.lift_map(x, "full", 1), full) <= 1e-15


@pytest.mark.parametrize("d,g", [(16, 2), (32, 4), (64, 2), (64, 4)])
def test_M_lift_is_the_block_lifts_in_order(d, g):
    x = np.random.default_rng(d + g).standard_normal((3, d))
    want = np.concatenate([oracle.lift(b) for b in _blocks(x, g)], axis=-1)
    assert _rel(oracle.lift_map(x, "M", g), want) <= 1e-15


@pytest.mark.parametrize("d,g", [(16, 2), (32, 4), (64, 2)])
def test_Sigma_lift_of_a_single_block(d, g):
    """Only block a nonzero: psi = eps I + s u_a u_a^T, i.e. eps vech(I) + s lift(u_a)."""
    m = d // g
    rng = np.random.default_rng(d * g)
    eye = oracle.lift(np.zeros(m))
    diag = [i * m - i * (i - 1) // 2 for i in range(m)]   # packed positions of (i, i)
    eye[diag] = 1.0
    for a in range(g):
        x = np.zeros(d)
        x[a * m:(a + 1) * m] = rng.standard_normal(m)
        got = oracle.lift_map(x, "Sigma", g, 1e-4, 0.25)
        want = 1e-4 * eye + 0.25 * oracle.lift(x[a * m:(a + 1) * m])
        assert _rel(got, want) <= 1e-14


def test_full_map_forward_is_the_pinned_forward():
    q, k, v = _rand_qkv(np.random.default_rng(1), d=16)
    assert _rel(oracle.forward_map(q, k, v, "full"), oracle.forward(q, k, v)) <= 1e-12


@pytest.mark.parametrize("map_name,d,g", CASES[:2] + CASES[3:5])
def test_block_supported_inputs_reduce_to_the_full_map(map_name, d, g):
    """q and k supported on one block a: M_g and Sigma_g (eps = 0) weights are the
    full map's on that block (times s^2, which cancels in the ratio)."""
    m = d // g
    rng = np.random.default_rng(7 * d + g)
    for a in (0, g - 1):
        q, k, v = _rand_qkv(rng, T=23, d=d)
        mask = np.zeros(d)
        mask[a * m:(a + 1) * m] = 1.0
        q, k = q * mask, k * mask
        want = oracle.forward(q[..., a * m:(a + 1) * m], k[..., a * m:(a + 1) * m], v)
        got = oracle.forward_map(q, k, v, map_name, g, 0.0, 0.25 if map_name == "Sigma" else 1.0)
        assert _rel(got, want) <= 1e-12


@pytest.mark.parametrize("map_name,d,g", CASES)
def test_equal_keys_give_the_running_mean(map_name, d, g):
    rng = np.random.default_rng(d + 3 * g)
    q, _, v = _rand_qkv(rng, T=17, d=d)
    k = np.broadcast_to(rng.standard_normal(d), q.shape).copy()
    eps, s = (1e-4, 0.25) if map_name == "Sigma" else (0.0, 1.0)
    got = oracle.forward_map(q, k, v, map_name, g, eps, s)
    want = np.cumsum(v, axis=2) / np.arange(1, v.shape[2] + 1)[None, None, :, None]
    assert _rel(got, want) <= 1e-12


@pytest.mark.parametrize("map_name,d,g", CASES)
def test_outputs_in_the_convex_hull(map_name, d, g):
    q, k, v = _rand_qkv(np.random.default_rng(5 + d + g), T=41, d=d)
    eps, s = (1e-4, 0.25) if map_name == "Sigma" else (0.0, 1.0)
    o = oracle.forward_map(q, k, v, map_name, g, eps, s)
    lo = np.minimum.accumulate(v, axis=2)
    hi = np.maximum.accumulate(v, axis=2)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)


@pytest.mark.parametrize("map_name,d,g", CASES)
def test_direct_form_equals_the_packed_recurrence(map_name, d, g):
    q, k, v = _rand_qkv(np.random.default_rng(11 + d + g), T=19, d=d)
    eps, s = (1e-4, 0.25) if map_name == "Sigma" else (0.0, 1.0)
    a = oracle.forward_map(q, k, v, map_name, g, eps, s)
    b = oracle.recurrent_map(q, k, v, map_name, g, eps, s)
    assert _rel(a, b) <= 1e-11
    rows = np.array([0, 5, 18, 19 + 7, 2 * 19 - 1])
    r = oracle.forward_rows_map(q, k, v, rows, map_name, g, eps, s)
    assert _rel(r, a.reshape(-1, a.shape[-1])[rows]) <= 1e-14


# ---- planted mistakes: a numpy weight with one error must fail the closed-form pin
def _weight_numpy(q, k, map_name, g, eps, s, mistake=None):
    qb, kb = _blocks(q, g), _blocks(k, g)
    m = q.shape[-1] // g
    if map_name == "M":
        if mistake == "cross_blocks":      # Sigma's sum over all block pairs
            return sum(float(a @ b) ** 2 for a in qb for b in kb)
        if mistake == "no_square":
            return sum(float(a @ b) for a, b in zip(qb, kb))
        return sum(float(a @ b) ** 2 for a, b in zip(qb, kb))
    A = eps * np.eye(m) + s * sum(np.outer(a, a) for a in qb)
    Bm = eps * np.eye(m) + s * sum(np.outer(b, b) for b in kb)
    if mistake == "no_eps":
        A, Bm = A - eps * np.eye(m), Bm - eps * np.eye(m)
    if mistake == "diag_blocks_only":   # M's pairing instead of all pairs
        return s * s * sum(float(a @ b) ** 2 for a, b in zip(qb, kb)) + eps * eps * m
    if mistake == "scale_once":
        Bm = eps * np.eye(m) + sum(np.outer(b, b) for b in kb)
    return float(np.sum(A * Bm))


def test_numpy_weight_passes_the_pin():
    rng = np.random.default_rng(3)
    for map_name, d, g in CASES:
        q, k = rng.standard_normal(d), rng.standard_normal(d)
        e, s = (1e-2, 0.25) if map_name == "Sigma" else (0.0, 1.0)
        assert abs(_weight_numpy(q, k, map_name, g, e, s) - _closed_form(q, k, map_name, g, e, s)) \
            <= 1e-10 * abs(_closed_form(q, k, map_name, g, e, s))


@pytest.mark.parametrize("map_name,mistake", [("M", "cross_blocks"), ("M", "no_square"),
                                              ("Sigma", "no_eps"), ("Sigma", "diag_blocks_only"),
                                              ("Sigma", "scale_once")])
def test_planted_weight_mistakes_fail(map_name, mistake):
    rng = np.random.default_rng(9)
    d, g = 32, 4
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    e, s = (0.3, 0.25) if map_name == "Sigma" else (0.0, 1.0)
    bad = _weight_numpy(q, k, map_name, g, e, s, mistake)
    want = _closed_form(q, k, map_name, g, e, s)
    assert abs(bad - want) > 1e-6 * abs(want)


# ---- orthant map (the pages' linear-state family): psi(u)_i = max(u_i, 0) + eps, n = d
def _orthant_identity(q, k, eps):
    """Expanded inner product: sum q+ k+ + eps (sum q+ + sum k+) + d eps^2."""
    qp, kp = np.maximum(q, 0.0), np.maximum(k, 0.0)
    return float(qp @ kp) + eps * (float(qp.sum()) + float(kp.sum())) + q.shape[-1] * eps * eps


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.25])
def test_orthant_width_and_inner_product(d, eps):
    assert oracle.map_dim("orthant", d, 1) == d
    rng = np.random.default_rng(d + int(eps * 100))
    for _ in range(20):
        q, k = rng.standard_normal(d), rng.standard_normal(d)
        pq, pk = oracle.lift_map(q, "orthant", 1, eps), oracle.lift_map(k, "orthant", 1, eps)
        assert pq.shape == (d,) and np.all(pq >= eps)
        want = _orthant_identity(q, k, eps)
        assert abs(float(pq @ pk) - want) <= 1e-12 * max(1.0, abs(want))


def test_orthant_one_hot_lookup():
    """eps = 0, one-hot keys and queries: the weight is 1 exactly when the indices
    match, so o_t is the mean of the values stored under the query's index so far
    (a zero row when there are none)."""
    rng = np.random.default_rng(2)
    d, T, dv = 8, 40, 3
    ki, qi = rng.integers(0, d, T), rng.integers(0, d, T)
    k = np.eye(d)[ki][None, None]
    q = np.eye(d)[qi][None, None]
    v = rng.standard_normal((1, 1, T, dv))
    got = oracle.forward_map(q, k, v, "orthant", 1, 0.0)
    want = np.zeros((T, dv))
    for t in range(T):
        hits = [s for s in range(t + 1) if ki[s] == qi[t]]
        if hits:
            want[t] = v[0, 0, hits].mean(axis=0)
    assert _rel(got[0, 0], want) <= 1e-13


@pytest.mark.parametrize("eps", [1e-6, 0.1])
def test_orthant_equal_keys_convex_hull_and_recurrence(eps):
    rng = np.random.default_rng(17)
    q, k, v = _rand_qkv(rng, T=33, d=16)
    keq = np.broadcast_to(np.abs(rng.standard_normal(16)), q.shape).copy()
    got = oracle.forward_map(q, keq, v, "orthant", 1, eps)
    want = np.cumsum(v, axis=2) / np.arange(1, v.shape[2] + 1)[None, None, :, None]
    assert _rel(got, want) <= 1e-12
    o = oracle.forward_map(q, k, v, "orthant", 1, eps)
    lo, hi = np.minimum.accumulate(v, axis=2), np.maximum.accumulate(v, axis=2)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)
    assert _rel(o, oracle.recurrent_map(q, k, v, "orthant", 1, eps)) <= 1e-11


@pytest.mark.parametrize("mistake", ["no_relu", "eps_on_query_only"])
def test_orthant_planted_mistakes_fail(mistake):
    rng = np.random.default_rng(23)
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    eps = 0.2
    if mistake == "no_relu":
        bad = float((q + eps) @ (k + eps))
    else:
        bad = float((np.maximum(q, 0) + eps) @ np.maximum(k, 0))
    assert abs(bad - _orthant_identity(q, k, eps)) > 1e-6


# ---- the map's state after a prefix and one decode step (Eq. 2's recurrence
# with the map's psi): pinned to the direct definition and the printed identities
STATE_CASES = [("M", 16, 2, 0.0, 1.0), ("M", 32, 4, 0.0, 1.0), ("Sigma", 16, 2, 1e-4, 1.0),
               ("Sigma", 64, 4, 1e-4, 0.25), ("Sigma", 32, 2, 0.3, 2.0), ("orthant", 16, 1, 1e-6, 1.0)]


@pytest.mark.parametrize("map_name,d,g,eps,s", STATE_CASES)
def test_prefix_then_decode_is_the_direct_row(map_name, d, g, eps, s):
    """State of tokens 0..T-1, then one step with token T: its output is row T
    of the direct O(T^2) definition."""
    q, k, v = _rand_qkv(np.random.default_rng(d + g), B=2, H=1, T=23, d=d, dv=6)
    T = q.shape[2] - 1
    S, z = oracle.prefix_state_map(k[:, :, :T], v[:, :, :T], map_name, g, eps, s)
    S2, z2, o = oracle.decode_step_map(S, z, q[:, :, T], k[:, :, T], v[:, :, T], map_name, g,
                                       eps, s)
    ref = oracle.forward_map(q, k, v, map_name, g, eps, s)[:, :, T]
    assert _rel(o, ref) < 1e-12
    # the step's state is the prefix state of all T + 1 tokens
    S_all, z_all = oracle.prefix_state_map(k, v, map_name, g, eps, s)
    assert _rel(S2, S_all) < 1e-12 and _rel(z2, z_all) < 1e-12


@pytest.mark.parametrize("map_name,d,g,eps,s", STATE_CASES[:5])
def test_state_contracts_to_the_printed_weights(map_name, d, g, eps, s):
    """psi(q)^T S = sum_s w(q, k_s) v_s and psi(q)^T z = sum_s w(q, k_s), with w
    the printed inner-product identity (computed here in numpy)."""
    q, k, v = _rand_qkv(np.random.default_rng(3 * d + g), B=1, H=1, T=17, d=d, dv=4)
    S, z = oracle.prefix_state_map(k, v, map_name, g, eps, s)
    pq = oracle.lift_map(q[0, 0, 5], map_name, g, eps, s)
    w = np.array([_closed_form(q[0, 0, 5], k[0, 0, t], map_name, g, eps, s) for t in range(17)])
    assert _rel(pq @ S[0, 0], w @ v[0, 0]) < 1e-12
    assert abs(float(pq @ z[0, 0]) - float(w.sum())) < 1e-12 * float(w.sum())


def test_full_map_state_is_the_pinned_prefix_state():
    q, k, v = _rand_qkv(np.random.default_rng(5), B=1, H=2, T=19, d=16, dv=5)
    S, z = oracle.prefix_state_map(k, v, "M", 1)
    S0, z0 = oracle.prefix_state(k, v)
    assert _rel(S, S0) < 1e-12 and _rel(z, z0) < 1e-12


def test_decode_read_before_update_fails_the_pin():
    """A step that reads the state before adding its own key misses the token's
    own weight: it differs from the direct row."""
    q, k, v = _rand_qkv(np.random.default_rng(9), B=1, H=1, T=12, d=16, dv=3)
    T = 11
    S, z = oracle.prefix_state_map(k[:, :, :T], v[:, :, :T], "Sigma", 2, 1e-4, 1.0)
    pq = oracle.lift_map(q[0, 0, T], "Sigma", 2, 1e-4, 1.0)
    wrong = (pq @ S[0, 0]) / (pq @ z[0, 0])
    ref = oracle.forward_map(q, k, v, "Sigma", 2, 1e-4, 1.0)[0, 0, T]
    assert _rel(wrong, ref) > 1e-6


# ---- a reduced map's state from full-map states of its blocks (the composition
# the tensor routes use), checked on the oracle alone
def _vech_index(i, j, m):
    return i * m - i * (i - 1) // 2 + (j - i)


@pytest.mark.parametrize("map_name,d,g,eps,s,pad", [
    ("M", 32, 2, 0.0, 1.0, 0), ("M", 64, 4, 0.0, 1.0, 16), ("M", 32, 2, 0.0, 1.0, 16),
    ("Sigma", 64, 2, 1e-4, 1.0, 0), ("Sigma", 32, 2, 0.5, 0.25, 0), ("Sigma", 32, 1, 3.0, 1.0, 0),
])
def test_map_state_is_composed_from_block_states(map_name, d, g, eps, s, pad):
    """M_g: block a's features are those of the full-map state of u_a (here also
    of u_a zero-padded to m + pad coordinates, restricted to the first m);
    Sigma_g: s sum_a S(u_a) + eps sum_t v_t on the diagonal features, and
    z = s sum_a z(u_a) + eps T there (psi = eps I + s sum_a u_a u_a^T, term by term)."""
    q, k, v = _rand_qkv(np.random.default_rng(d + 7 * g + pad), B=1, H=2, T=21, d=d, dv=5)
    m = d // g
    S, z = oracle.prefix_state_map(k, v, map_name, g, eps, s)
    blocks = []
    for a in range(g):
        ka = k[..., a * m:(a + 1) * m]
        if pad:
            ka = np.concatenate([ka, np.zeros(ka.shape[:-1] + (pad,))], axis=-1)
        blocks.append(oracle.prefix_state(ka, v))   # the full map of width m + pad
    nm, mp = m * (m + 1) // 2, m + pad
    sel = [_vech_index(i, j, mp) for i in range(m) for j in range(i, m)]   # first m coordinates
    if map_name == "M":
        S_c = np.concatenate([Sa[:, :, sel] for Sa, _ in blocks], axis=2)
        z_c = np.concatenate([za[:, :, sel] for _, za in blocks], axis=2)
    else:
        diag = np.zeros(nm)
        diag[[_vech_index(i, i, m) for i in range(m)]] = 1.0
        T = k.shape[2]
        S_c = s * sum(Sa[:, :, sel] for Sa, _ in blocks) + eps * diag[None, None, :, None] * \
            v.sum(axis=2)[:, :, None, :]
        z_c = s * sum(za[:, :, sel] for _, za in blocks) + eps * T * diag[None, None, :]
    assert _rel(S_c, S) < 1e-12 and _rel(z_c, z) < 1e-12


def test_map_state_composition_without_eps_fails_the_pin():
    """Leaving out the eps diagonal (or the scale) breaks the Sigma composition."""
    q, k, v = _rand_qkv(np.random.default_rng(77), B=1, H=1, T=15, d=32, dv=4)
    S, _ = oracle.prefix_state_map(k, v, "Sigma", 2, 0.5, 0.25)
    S_a = sum(oracle.prefix_state(k[..., a * 16:(a + 1) * 16], v)[0] for a in range(2))
    assert _rel(0.25 * S_a, S) > 1e-3
    assert _rel(S_a, S) > 1e-3
