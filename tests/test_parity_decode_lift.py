"""GPU parity of the decode step and the standalone feature lift against the
CPU oracle, and prefill/decode consistency."""
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


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [1, 5, 16, 32, 64])
def test_lift_matches_oracle(kg, dtype, d):
    g = torch.Generator().manual_seed(d)
    x = torch.randn(37, 3, d, generator=g).to(dtype)
    phi = kg.kata_lift(x.cuda())
    torch.cuda.synchronize()
    ref = oracle.lift(to_f64(x))
    got = to_f64(phi)
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=2e-6, atol=1e-6)


def _state_from_prefix(w, length):
    kp, vp = workloads.make_decode_prefix(w, length)
    S, z = oracle.prefix_state(to_f64(kp), to_f64(vp))
    return S, z


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d,dv", [(16, 16), (32, 64), (64, 64), (64, 128)])
def test_decode_step_matches_oracle(kg, dtype, d, dv):
    w = workloads.DECODE.scaled(B=3, H=5, d=d, dv=dv, dtype=dtype)
    S, z = _state_from_prefix(w, 16)
    q, k, v = workloads.make_decode_inputs(w)
    S_d = torch.from_numpy(S).float().cuda()
    z_d = torch.from_numpy(z).float().cuda()
    # the oracle continues from the same fp32 state the GPU receives
    S0, z0 = to_f64(S_d), to_f64(z_d)
    out = kg.kata_decode_step(S_d, z_d, q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    S_ref, z_ref, o_ref = oracle.decode_step(S0, z0, to_f64(q), to_f64(k), to_f64(v))
    err = slice_rel_err(to_f64(out)[..., None, :], o_ref[..., None, :])
    assert err <= TOL[dtype], err
    # the updated state: fp32 adds of fp32 products
    np.testing.assert_allclose(to_f64(S_d), S_ref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(to_f64(z_d), z_ref, rtol=1e-5, atol=1e-5)


def test_decode_full_workload(kg):
    """B=256, H=16, d=64, dv=64 decode from a state built by the oracle's
    recurrence over a seeded 16-token prefix; all heads checked."""
    w = workloads.DECODE
    S_np, z_np = _state_from_prefix(w, 16)
    S = torch.from_numpy(S_np).float().cuda()
    z = torch.from_numpy(z_np).float().cuda()
    q, k, v = workloads.make_decode_inputs(w, device="cuda")
    S0, z0 = to_f64(S), to_f64(z)
    out = kg.kata_decode_step(S, z, q, k, v)
    torch.cuda.synchronize()
    _, _, o_ref = oracle.decode_step(S0, z0, to_f64(q), to_f64(k), to_f64(v))
    got = to_f64(out)
    scale = np.max(np.abs(o_ref), axis=-1)
    err = np.max(np.abs(got - o_ref), axis=-1) / scale
    assert float(err.max()) <= TOL[w.dtype], float(err.max())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_steps_continue_prefill(kg, dtype):
    """T decode steps from the zero state reproduce the chunked forward."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=2, H=2, T=70, d=32, dv=64, dtype=dtype, C=32)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    fwd = kg.kata_fwd_chunked(q, k, v, w.C)
    n = kg.kata_feature_dim(w.d)
    S = torch.zeros(w.B, w.H, n, w.dv, device="cuda")
    z = torch.zeros(w.B, w.H, n, device="cuda")
    outs = []
    for t in range(w.T):
        outs.append(kg.kata_decode_step(S, z, q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                        v[:, :, t].contiguous()))
    dec = torch.stack(outs, dim=2)
    torch.cuda.synchronize()
    ref = oracle.forward(to_f64(q), to_f64(k), to_f64(v))
    assert slice_rel_err(to_f64(dec), ref) <= TOL[dtype]
    assert slice_rel_err(to_f64(fwd), ref) <= TOL[dtype]
    # final state equals the oracle's prefix state
    S_ref, z_ref = oracle.prefix_state(to_f64(k), to_f64(v))
    np.testing.assert_allclose(to_f64(S), S_ref, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(to_f64(z), z_ref, rtol=1e-4, atol=1e-4)
