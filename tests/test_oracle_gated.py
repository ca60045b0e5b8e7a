"""Pins for the oracle's GatedKATA forward and decode step (no GPU).

The pages' gated variant (the appendix on recurrent variants, "multiplicative
scalar state gate"; Sec. 5.2) puts a scalar gate gamma_t in [0, 1] inside the
recurrence, S_t = gamma_t S_{t-1} + psi(k_t) v_t^T, which unrolls so that write
s carries the weight prod_{r=s+1}^{t} gamma_r.  Readings: Z_t is gated the same
way, so the normalised readout stays the convex output gate of Prop. 1; the
no-denominator readout psi(q_t)^T S_t of the MQAR appendix is the
normalize=False form.

The pins tie the oracle to things other than itself: the already pinned plain
forward (gamma = 1), a reset (gamma_r = 0 drops every earlier write but keeps
write r), scipy's linear filter for the exponentially weighted mean that equal
keys and a constant gate give, a cumulative-product identity for time-varying
gates, invariants, and the decode step against the forward.  A numpy copy of
the weight with one planted mistake fails them.
"""
from __future__ import annotations

import numpy as np
import pytest
from scipy.signal import lfilter

import oracle


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _qkv(rng, B=1, H=2, T=23, d=8, dv=5):
    q = rng.standard_normal((B, H, T, d)) / np.sqrt(d)
    k = rng.standard_normal((B, H, T, d)) / np.sqrt(d)
    v = rng.standard_normal((B, H, T, dv))
    return q, k, v


def _gates(rng, shape, zeros=True):
    g = rng.uniform(0.0, 1.0, shape)
    if zeros:
        g.reshape(-1)[::7] = 1.0
        g.reshape(-1)[3::11] = 0.0
    return g


def test_unit_gate_is_plain_kata():
    q, k, v = _qkv(np.random.default_rng(1))
    one = np.ones(q.shape[:3])
    assert _rel(oracle.forward_gated(q, k, v, one), oracle.forward(q, k, v)) <= 1e-13
    # no denominator: the plain numerator psi(q_t) . sum_{s<=t} psi(k_s) v_s^T,
    # formed from the pinned lift and running sums
    pq, pk = oracle.lift(q), oracle.lift(k)
    S = np.cumsum(pk[..., :, None] * v[..., None, :], axis=2)
    want = np.einsum("bhtf,bhtfj->bhtj", pq, S)
    assert _rel(oracle.forward_gated(q, k, v, one, normalize=False), want) <= 1e-12


@pytest.mark.parametrize("r0", [1, 9, 22])
@pytest.mark.parametrize("normalize", [True, False])
def test_zero_gate_resets_the_state(r0, normalize):
    """gamma_r0 = 0: rows t >= r0 see only tokens r0 .. t (write r0 itself kept)."""
    rng = np.random.default_rng(r0)
    q, k, v = _qkv(rng)
    g = rng.uniform(0.3, 1.0, q.shape[:3])
    g[..., r0] = 0.0
    full = oracle.forward_gated(q, k, v, g, normalize)
    tail = oracle.forward_gated(q[..., r0:, :], k[..., r0:, :], v[..., r0:, :], g[..., r0:],
                                normalize)
    assert _rel(full[..., r0:, :], tail) <= 1e-13
    # earlier rows do not see the later gate (causality)
    head = oracle.forward_gated(q[..., :r0, :], k[..., :r0, :], v[..., :r0, :], g[..., :r0],
                                normalize)
    assert _rel(full[..., :r0, :], head) <= 1e-13
    if normalize:   # and with gamma_r0 = 0, row r0 is v_r0 exactly (o_1 = v_1 of Prop. 1)
        assert _rel(full[..., r0, :], v[..., r0, :]) <= 1e-13


@pytest.mark.parametrize("gamma", [0.0, 0.5, 0.9, 1.0])
def test_equal_keys_constant_gate_is_the_ewma(gamma):
    """All keys equal and gamma constant: o_t = sum gamma^{t-s} v_s / sum gamma^{t-s},
    the exponentially weighted mean; numerator and weights by scipy's IIR filter."""
    rng = np.random.default_rng(int(gamma * 10) + 3)
    q, _, v = _qkv(rng, T=31)
    k = np.broadcast_to(rng.standard_normal(8), q.shape).copy()
    g = np.full(q.shape[:3], gamma)
    num = lfilter([1.0], [1.0, -gamma], v, axis=2)
    den = lfilter([1.0], [1.0, -gamma], np.ones(v.shape[:3]), axis=2)
    assert _rel(oracle.forward_gated(q, k, v, g), num / den[..., None]) <= 1e-12
    # unit weights (q_t = k_s = e_1): the no-denominator readout is the filter output
    e1 = np.zeros(q.shape)
    e1[..., 0] = 1.0
    assert _rel(oracle.forward_gated(e1, e1, v, g, normalize=False), num) <= 1e-12


def test_time_varying_gate_unit_weights():
    """q_t = k_s = e_1: o_t = sum_s (prod_{r=s+1}^t gamma_r) v_s = P_t sum_{s<=t} v_s / P_s
    with P_t = prod_{r<=t} gamma_r (gates bounded away from 0)."""
    rng = np.random.default_rng(8)
    _, _, v = _qkv(rng, T=40)
    e1 = np.zeros(v.shape[:3] + (8,))
    e1[..., 0] = 1.0
    g = rng.uniform(0.6, 1.0, v.shape[:3])
    P = np.cumprod(g, axis=2)[..., None]
    want = P * np.cumsum(v / P, axis=2)
    assert _rel(oracle.forward_gated(e1, e1, v, g, normalize=False), want) <= 1e-12
    # normalised: the same with v replaced by 1 in the denominator
    den = P * np.cumsum(1.0 / P, axis=2)
    assert _rel(oracle.forward_gated(e1, e1, v, g), want / den) <= 1e-12


def test_outputs_in_the_convex_hull():
    rng = np.random.default_rng(4)
    q, k, v = _qkv(rng, T=60)
    o = oracle.forward_gated(q, k, v, _gates(rng, q.shape[:3]))
    lo, hi = np.minimum.accumulate(v, axis=2), np.maximum.accumulate(v, axis=2)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)


def test_scale_invariance_of_the_normalised_readout():
    rng = np.random.default_rng(6)
    q, k, v = _qkv(rng)
    g = _gates(rng, q.shape[:3])
    a = oracle.forward_gated(q, k, v, g)
    b = oracle.forward_gated(3.0 * q, -0.5 * k, v, g)
    assert _rel(b, a) <= 1e-12


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d", [4, 8, 16])
def test_direct_form_equals_the_gated_recurrence(normalize, d):
    rng = np.random.default_rng(20 + d)
    q, k, v = _qkv(rng, T=37, d=d)
    g = _gates(rng, q.shape[:3])
    a = oracle.forward_gated(q, k, v, g, normalize)
    assert _rel(a, oracle.recurrent_gated(q, k, v, g, normalize)) <= 1e-11
    rows = np.array([0, 3, 36, 37, 40, 73])
    r = oracle.forward_rows_gated(q, k, v, g, rows, normalize)
    assert _rel(r, a.reshape(-1, a.shape[-1])[rows]) <= 1e-14


@pytest.mark.parametrize("normalize", [True, False])
def test_decode_step_continues_the_forward(normalize):
    rng = np.random.default_rng(12)
    q, k, v = _qkv(rng, B=2, H=2, T=19, d=8)
    g = _gates(rng, q.shape[:3])
    S, z = oracle.prefix_state_gated(k[..., :-1, :], v[..., :-1, :], g[..., :-1])
    S1, z1, o = oracle.decode_step_gated(S, z, q[..., -1, :], k[..., -1, :], v[..., -1, :],
                                         g[..., -1], normalize)
    full = oracle.forward_gated(q, k, v, g, normalize)
    assert _rel(o, full[..., -1, :]) <= 1e-12
    S2, z2 = oracle.prefix_state_gated(k, v, g)
    assert _rel(S1, S2) <= 1e-13 and _rel(z1, z2) <= 1e-13
    # the gated state with unit gates is the plain prefix state
    S3, z3 = oracle.prefix_state_gated(k, v, np.ones(g.shape))
    S4, z4 = oracle.prefix_state(k, v)
    assert _rel(S3, S4) <= 1e-14 and _rel(z3, z4) <= 1e-14


# ---- planted mistakes: a numpy copy of the gated weight with one error fails a pin
def _gated_numpy(q, k, v, g, normalize=True, mistake=None):
    B, H, T, _ = q.shape
    out = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                num, den = np.zeros(v.shape[-1]), 0.0
                for s in range(t + 1):
                    lo = s if mistake == "own_gate" else s + 1
                    hi = t if mistake == "last_gate_dropped" else t + 1
                    a = float(np.prod(g[b, h, lo:hi]))
                    if mistake == "last_gate_dropped" and s == t:
                        a = 1.0
                    w = float(q[b, h, t] @ k[b, h, s]) ** 2
                    num += a * w * v[b, h, s]
                    den += (1.0 if mistake == "ungated_denominator" else a) * w
                out[b, h, t] = (num / den if den > 0 else 0.0 * num) if normalize else num
    return out


def test_numpy_gated_weight_matches_the_oracle():
    rng = np.random.default_rng(30)
    q, k, v = _qkv(rng, T=12)
    g = _gates(rng, q.shape[:3])
    for normalize in (True, False):
        assert _rel(_gated_numpy(q, k, v, g, normalize), oracle.forward_gated(q, k, v, g, normalize)) \
            <= 1e-12


@pytest.mark.parametrize("mistake", ["own_gate", "last_gate_dropped", "ungated_denominator"])
def test_planted_gate_mistakes_fail_a_pin(mistake):
    """Each mistake breaks the reset pin or the EWMA pin (both computed here for the
    numpy copy exactly as the pins above compute them for the oracle)."""
    rng = np.random.default_rng(40)
    q, k, v = _qkv(rng, T=14)
    # reset pin
    g = rng.uniform(0.3, 1.0, q.shape[:3])
    r0 = 6
    g[..., r0] = 0.0
    full = _gated_numpy(q, k, v, g, True, mistake)
    tail_gated = oracle.forward_gated(q[..., r0:, :], k[..., r0:, :], v[..., r0:, :], g[..., r0:])
    reset_ok = _rel(full[..., r0:, :], tail_gated) <= 1e-10
    # EWMA pin (equal keys, constant gate)
    k2 = np.broadcast_to(rng.standard_normal(8), q.shape).copy()
    gc = np.full(q.shape[:3], 0.7)
    num = lfilter([1.0], [1.0, -0.7], v, axis=2)
    den = lfilter([1.0], [1.0, -0.7], np.ones(v.shape[:3]), axis=2)
    ewma_ok = _rel(_gated_numpy(q, k2, v, gc, True, mistake), num / den[..., None]) <= 1e-10
    assert not (reset_ok and ewma_ok), mistake
