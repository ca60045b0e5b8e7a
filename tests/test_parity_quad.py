"""GPU parity of the quadratic (flash-style) forward kata_fwd_quadratic against
the oracle's direct definition (the same function as the chunked form, [KATA]
Sec. 2 Eq. 2 with the rank-one PSD lift): element by element at sizes the
oracle finishes in seconds (several tiles and ragged tails), and sampled rows
at full workload sizes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import TOL, require_gpu, slice_rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kg():
    return require_gpu()


def _check(kg, q, k, v):
    out = kg.kata_fwd_quadratic(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward(to_f64(q), to_f64(k), to_f64(v))
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[q.dtype], f"{err:.3e}"
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("name", ["lm_layer_bf16", "mid_bf16", "recall_bf16", "long_ctx_bf16"])
@pytest.mark.parametrize("T", [1, 127, 128, 129, 300, 700])
def test_quadratic_parity(kg, name, T):
    w = workloads.WORKLOADS[name].scaled(B=1, H=3, T=T)
    _check(kg, *workloads.make_qkv(w))


def test_quadratic_many_heads(kg):
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=4, H=9, T=260)
    _check(kg, *workloads.make_qkv(w))


def test_quadratic_zero_denominator_rows(kg):
    # queries along e_0, the first 70 keys along e_1: rows t < 70 have D_t = 0
    B, H, T, d, dv = 1, 1, 150, 32, 64
    q = torch.zeros(B, H, T, d)
    k = torch.zeros(B, H, T, d)
    q[..., 0] = 1.0
    k[..., :70, 1] = 1.0
    k[..., 70:, 0] = 1.0
    v = torch.randn(B, H, T, dv, generator=torch.Generator().manual_seed(5))
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    out = kg.kata_fwd_quadratic(q.cuda(), k.cuda(), v.cuda()).float().cpu()
    assert torch.all(out[..., :70, :] == 0)
    ref = oracle.forward(to_f64(q), to_f64(k), to_f64(v))
    assert slice_rel_err(out.numpy().astype(np.float64), ref) <= TOL[torch.bfloat16]


def test_quadratic_deterministic(kg):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=2, H=2, T=1000)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_quadratic(q, k, v)
    b = kg.kata_fwd_quadratic(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("d,dv", [(16, 16), (16, 64), (16, 128), (32, 32), (32, 128), (64, 16),
                                  (64, 128)])
@pytest.mark.parametrize("T", [129, 300])
def test_quadratic_adapted_shapes(kg, d, dv, T):
    """Other bf16 head sizes: q, k padded to d = 32 and v in 64-column parts, each
    part one pass of the quadratic kernel."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=3, T=T, d=d, dv=dv)
    _check(kg, *workloads.make_qkv(w))


def test_quadratic_unsupported_shapes(kg):
    w = workloads.WORKLOADS["small_fp32"]
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    with pytest.raises(kg.KataError) as e:
        kg.kata_fwd_quadratic(q, k, v)
    assert e.value.status == kg.KATA_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["lm_layer_bf16", "mid_bf16", "recall_bf16"])
def test_quadratic_full_size_sampled_rows(kg, name):
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w, device="cuda")
    out = kg.kata_fwd_quadratic(q, k, v)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    assert torch.isfinite(out).all()
    BH = w.B * w.H
    rng = np.random.default_rng(w.index + 100)
    worst = 0.0
    for h in sorted(set([0, BH - 1] + rng.integers(0, BH, size=2).tolist())):
        ts = np.array(sorted(set([0, 1, 127, 128, 129, w.T // 2, w.T - 2, w.T - 1] +
                                 rng.integers(0, w.T, size=16).tolist())), dtype=np.int64)
        ref = oracle.forward_rows(to_f64(q.reshape(BH, 1, w.T, w.d)[h:h + 1]),
                                  to_f64(k.reshape(BH, 1, w.T, w.d)[h:h + 1]),
                                  to_f64(v.reshape(BH, 1, w.T, w.dv)[h:h + 1]), ts)
        got = to_f64(out.reshape(BH, w.T, w.dv)[h][ts])
        worst = max(worst, slice_rel_err(got, ref))
    assert worst <= TOL[w.dtype], f"{name}: {worst:.3e}"


@pytest.mark.parametrize("gated", [False, True])
def test_long_context_sampled_rows(kg, gated):
    """The long-context shape (B=1, H=16, T=131072, d=32: 1024 query tiles per head,
    the longest walking 1024 key tiles) in the quadratic form, plain and gated,
    sampled rows against the oracle (first, last, tile edges, random)."""
    w = workloads.WORKLOADS["long_ctx_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    g = workloads.make_gate(w, device="cuda") if gated else None
    out = kg.kata_fwd_quadratic_gated(q, k, v, g) if gated else kg.kata_fwd_quadratic(q, k, v)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(91)
    worst = 0.0
    for h in (0, 7, w.H - 1):
        ts = np.array(sorted(set([0, 127, 128, w.T // 2, w.T - 1] +
                                 rng.integers(0, w.T, size=6).tolist())), dtype=np.int64)
        sl = (slice(0, 1), slice(h, h + 1))
        qf, kf, vf = to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl])
        if gated:
            ref = oracle.forward_rows_gated(qf, kf, vf, to_f64(g[sl]), ts)
        else:
            ref = oracle.forward_rows(qf, kf, vf, ts)
        worst = max(worst, slice_rel_err(to_f64(out[0, h])[ts], ref))
    assert worst <= TOL[torch.bfloat16], f"{worst:.3e}"
