"""GPU parity of kata_fwd_chunked_state: the state after the last token, in the
decode layout, against the oracle's feature-state recurrence ([KATA] Eq. 2,
App. D.1), and prefill -> decode consistency against the direct definition.

Metric for a state: per (b, h), max |S - S_ref| / max |S_ref| (same for z).  The
fp32 path accumulates fp32 products of the inputs (bar 1e-5).  The tensor-core
path accumulates products of bf16-rounded lifted keys with v in fp32, so each
term carries a relative rounding of at most 2^-9 (bar 1e-2)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import TOL, require_gpu, slice_rel_err, to_f64

pytestmark = pytest.mark.gpu

STATE_TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}


@pytest.fixture(scope="module")
def kg():
    return require_gpu()


def _state_err(got, ref):
    """got, ref: [B, H, ...]; max over (b, h) of max|got - ref| / max|ref|."""
    g = got.reshape(got.shape[0] * got.shape[1], -1)
    r = ref.reshape(g.shape)
    return max(float(np.max(np.abs(a - b)) / np.max(np.abs(b))) for a, b in zip(g, r))


def _check_state(kg, w, expect_path=None):
    q, k, v = workloads.make_qkv(w)
    if expect_path is not None:
        assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == expect_path
    out, S, z = kg.kata_fwd_chunked_state(q.cuda(), k.cuda(), v.cuda(), w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    S_ref, z_ref = oracle.prefix_state(to_f64(k), to_f64(v))
    tol = STATE_TOL[w.dtype]
    es, ez = _state_err(to_f64(S), S_ref), _state_err(to_f64(z), z_ref)
    assert es <= tol and ez <= tol, f"state {es:.2e}, z {ez:.2e} (bar {tol:.0e})"
    # the output of the same call is the forward's
    ref = oracle.forward(to_f64(q), to_f64(k), to_f64(v))
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


# With the state exported every segment is summed (the last one too) and the
# scan's inclusive totals are the state.
@pytest.mark.parametrize("B,H,T", [
    (1, 2, 1100),    # 9 one-chunk segments per head, ragged last chunk
    (16, 8, 700),    # one segment per head
    (4, 8, 4096),    # 4 segments of 8 chunks
    (1, 4, 5000),    # 20 segments of 2 chunks
    (1, 1, 129),     # last chunk holds one token
    (3, 1, 5),       # a single partial chunk
])
def test_state_tensor_path(kg, B, H, T):
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=B, H=H, T=T)
    _check_state(kg, w, kg.KATA_PATH_TC)


@pytest.mark.parametrize("name,overrides", [
    ("small_fp32", dict(B=2, H=3, T=300)),
    ("small_fp32", dict(B=1, H=2, T=97, d=32, dv=64, C=32)),
])
def test_state_cuda_core_path(kg, name, overrides):
    w = workloads.WORKLOADS[name].scaled(**overrides)
    _check_state(kg, w, kg.KATA_PATH_SIMT)


@pytest.mark.parametrize("d,dv,B,H,T", [
    (32, 128, 1, 2, 200),    # two v parts, one column block of the state each
    (16, 16, 1, 2, 1100),    # q, k padded to d = 32: 136 of the 528 features kept
    (16, 128, 3, 1, 129),
    (32, 32, 2, 2, 5),
    (64, 128, 2, 19, 300),   # the d = 64 kernels, two v parts
])
def test_state_adapted_shapes(kg, d, dv, B, H, T):
    """bf16 shapes the tensor kernels take through padded q, k and 64-column
    parts of v: each part's state is a column block of the state, and the
    padded features that mix in a zero column are dropped."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=B, H=H, T=T, d=d, dv=dv, C=64)
    _check_state(kg, w, kg.KATA_PATH_TC)


@pytest.mark.parametrize("B,H,T", [
    (1, 2, 333),     # 2 heads: SMs left idle, chunks in order
    (2, 19, 300),    # 38 heads, ragged tail
    (2, 19, 129),    # last chunk holds one token (the state records follow an odd-sized workspace part)
    (4, 10, 5),      # a single partial chunk
])
def test_state_d64_tensor_path(kg, B, H, T):
    """d = 64 with the state split over four CTAs per head: each CTA writes the
    running state of its feature blocks after the last chunk, group 0 also the
    Gram matrix, and a reorder kernel maps them to the decode layout."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T)
    _check_state(kg, w, kg.KATA_PATH_TC)


@pytest.mark.parametrize("name,overrides", [
    ("long_ctx_bf16", dict(B=2, H=2, T=1000)),
    ("small_fp32", dict(B=1, H=2, T=150)),
    ("long_ctx_bf16", dict(B=1, H=3, T=700, d=16, dv=128)),   # padded q, k; two v parts
])
def test_prefill_then_decode(kg, name, overrides):
    """Forward over T-1 tokens with state export, then one decode step with
    token T-1: its output is the definition's output at row T-1."""
    w = workloads.WORKLOADS[name].scaled(**overrides)
    q, k, v = workloads.make_qkv(w)
    Tp = w.T - 1
    _, S, z = kg.kata_fwd_chunked_state(q[:, :, :Tp].contiguous().cuda(),
                                        k[:, :, :Tp].contiguous().cuda(),
                                        v[:, :, :Tp].contiguous().cuda(), w.C)
    o = kg.kata_decode_step(S, z, q[:, :, Tp].contiguous().cuda(), k[:, :, Tp].contiguous().cuda(),
                            v[:, :, Tp].contiguous().cuda())
    torch.cuda.synchronize()
    rows = np.arange(w.B * w.H, dtype=np.int64) * w.T + Tp
    ref = oracle.forward_rows(to_f64(q), to_f64(k), to_f64(v), rows)
    got = to_f64(o).reshape(w.B, w.H, 1, w.dv)
    assert slice_rel_err(got, ref.reshape(got.shape)) <= TOL[w.dtype]


def test_state_full_size_sampled_heads(kg):
    """The long-context workload in the bench's call configuration: the exported
    state of two heads against the oracle recurrence over all 131072 tokens."""
    w = workloads.WORKLOADS["long_ctx_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    out, S, z = kg.kata_fwd_chunked_state(q, k, v, w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    BH = w.B * w.H
    for h in (0, BH - 1):
        kh = k.reshape(BH, 1, 1, w.T, w.d)[h]
        vh = v.reshape(BH, 1, 1, w.T, w.dv)[h]
        S_ref, z_ref = oracle.prefix_state(to_f64(kh), to_f64(vh))
        Sg = to_f64(S.reshape(BH, 1, -1, w.dv)[h:h + 1])
        zg = to_f64(z.reshape(BH, 1, -1)[h:h + 1])
        assert _state_err(Sg, S_ref) <= STATE_TOL[w.dtype]
        assert _state_err(zg, z_ref) <= STATE_TOL[w.dtype]


def test_state_d64_full_size_sampled_heads(kg):
    """The LM-layer workload (d = 64) in the bench's call configuration: the
    exported state of two heads against the oracle recurrence."""
    w = workloads.WORKLOADS["lm_layer_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    out, S, z = kg.kata_fwd_chunked_state(q, k, v, w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    BH = w.B * w.H
    for h in (0, BH - 1):
        kh = k.reshape(BH, 1, 1, w.T, w.d)[h]
        vh = v.reshape(BH, 1, 1, w.T, w.dv)[h]
        S_ref, z_ref = oracle.prefix_state(to_f64(kh), to_f64(vh))
        Sg = to_f64(S.reshape(BH, 1, -1, w.dv)[h:h + 1])
        zg = to_f64(z.reshape(BH, 1, -1)[h:h + 1])
        assert _state_err(Sg, S_ref) <= STATE_TOL[w.dtype]
        assert _state_err(zg, z_ref) <= STATE_TOL[w.dtype]


# ---- reduced maps: the map's state after a prefill, and a decode step from it
_MAP_NAMES = {1: "M", 2: "Sigma", 3: "orthant"}


def _map_params(map_, g):
    if map_ == 2:
        return 1e-4, (0.25 if g == 4 else 1.0)
    if map_ == 3:
        return 1e-6, 1.0
    return 0.0, 1.0


@pytest.mark.parametrize("map_,g,d,dtype", [
    (2, 4, 64, torch.bfloat16),   # Sigma_4: the explicit-feature path exports its scanned records
    (2, 2, 32, torch.bfloat16),
    (3, 1, 64, torch.bfloat16),   # orthant
    (1, 4, 16, torch.bfloat16),
    (1, 2, 64, torch.bfloat16),   # M_2 at d = 64: its sub-heads' states are its blocks
    (2, 2, 64, torch.bfloat16),   # Sigma_2 at d = 64: composed from the key halves' states
    (2, 1, 32, torch.bfloat16),   # Sigma_1 at d = 32: the full map's state plus the eps terms
    (2, 2, 16, torch.float32),    # fp32: CUDA cores
])
@pytest.mark.parametrize("dv", [64, 128])
def test_map_prefill_then_decode(kg, map_, g, d, dtype, dv):
    """kata_fwd_chunked_map_state over T-1 tokens: its state against the oracle's
    map recurrence, its output against the direct definition; then
    kata_decode_step_map with token T-1: the direct definition's row T-1."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=2, H=2, T=301, d=d, dv=dv, dtype=dtype)
    name = _MAP_NAMES[map_]
    eps, scale = _map_params(map_, g)
    q, k, v = workloads.make_qkv(w)
    Tp = w.T - 1
    sl = (slice(None), slice(None), slice(0, Tp))
    out, S, z = kg.kata_fwd_chunked_map_state(q[sl].contiguous().cuda(), k[sl].contiguous().cuda(),
                                              v[sl].contiguous().cuda(), w.C, map_, g, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    S_ref, z_ref = oracle.prefix_state_map(to_f64(k[sl]), to_f64(v[sl]), name, g, eps, scale)
    tol = STATE_TOL[dtype]
    es, ez = _state_err(to_f64(S), S_ref), _state_err(to_f64(z), z_ref)
    assert es <= tol and ez <= tol, f"state {es:.2e}, z {ez:.2e} (bar {tol:.0e})"
    ref = oracle.forward_map(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), name, g, eps, scale)
    assert slice_rel_err(to_f64(out), ref) <= TOL[dtype]
    o = kg.kata_decode_step_map(S, z, q[:, :, Tp].contiguous().cuda(), k[:, :, Tp].contiguous().cuda(),
                                v[:, :, Tp].contiguous().cuda(), map_, g, eps, scale)
    torch.cuda.synchronize()
    rows = np.arange(w.B * w.H, dtype=np.int64) * w.T + Tp
    refo = oracle.forward_rows_map(to_f64(q), to_f64(k), to_f64(v), rows, name, g, eps, scale)
    got = to_f64(o).reshape(w.B, w.H, 1, w.dv)
    assert slice_rel_err(got, refo.reshape(got.shape)) <= TOL[dtype]


@pytest.mark.parametrize("map_,g,d,dv", [(2, 4, 64, 64), (1, 2, 32, 16), (3, 1, 16, 128),
                                         (2, 2, 64, 32)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_map_decode_step_parity(kg, map_, g, d, dv, dtype):
    """One decode step from an oracle state (a 16-token prefix) against the
    oracle's map step: the output and the updated state and z."""
    name = _MAP_NAMES[map_]
    eps, scale = _map_params(map_, g)
    rng = torch.Generator().manual_seed(d + dv + map_)
    B, H = 3, 5
    kp = torch.randn(B, H, 16, d, generator=rng) / d ** 0.5
    vp = torch.randn(B, H, 16, dv, generator=rng)
    S0, z0 = oracle.prefix_state_map(to_f64(kp), to_f64(vp), name, g, eps, scale)
    q = (torch.randn(B, H, d, generator=rng) / d ** 0.5).to(dtype)
    k = (torch.randn(B, H, d, generator=rng) / d ** 0.5).to(dtype)
    v = torch.randn(B, H, dv, generator=rng).to(dtype)
    S = torch.from_numpy(S0).float().cuda()
    z = torch.from_numpy(z0).float().cuda()
    Sf, zf = to_f64(S), to_f64(z)
    o = kg.kata_decode_step_map(S, z, q.cuda(), k.cuda(), v.cuda(), map_, g, eps, scale)
    torch.cuda.synchronize()
    S1, z1, oref = oracle.decode_step_map(Sf, zf, to_f64(q), to_f64(k), to_f64(v), name, g, eps,
                                          scale)
    assert slice_rel_err(to_f64(o)[:, :, None, :], oref[:, :, None, :]) <= TOL[dtype]
    assert _state_err(to_f64(S), S1) <= 1e-5 and _state_err(to_f64(z), z1) <= 1e-5


# (map, g, d, eps, scale): the tensor routes built from full-map sub-heads, whose
# map state is composed from the sub-heads' states; eps of the size of the
# s^2 (q.k)^2 terms puts weight on the eps diagonal of the Sigma states
_COMPOSED = [(1, 2, 64, 0.0, 1.0), (1, 4, 64, 0.0, 1.0), (2, 2, 64, 1e-4, 1.0),
             (2, 2, 64, 0.5, 0.25), (2, 1, 64, 1e-4, 1.0), (2, 1, 64, 3.0, 1.0),
             (1, 2, 32, 0.0, 1.0), (2, 1, 32, 1e-4, 1.0), (2, 1, 32, 0.5, 0.25)]


@pytest.mark.parametrize("map_,g,d,eps,scale", _COMPOSED)
@pytest.mark.parametrize("B,H,T,dv", [(2, 2, 300, 64), (1, 2, 1100, 64), (1, 3, 129, 128)])
def test_map_state_composed_routes(kg, map_, g, d, eps, scale, B, H, T, dv):
    """M_2, M_4, Sigma_2, Sigma_1 at d = 64 and M_2, Sigma_1 at d = 32 on the tensor
    cores with the state exported: S and z against the oracle's map recurrence
    (several segments at T = 1100; 64-column parts of v at dv = 128), the output
    against the direct definition."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T, d=d, dv=dv)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, map_, g) == \
        kg.KATA_PATH_TC
    name = _MAP_NAMES[map_]
    q, k, v = workloads.make_qkv(w)
    out, S, z = kg.kata_fwd_chunked_map_state(q.cuda(), k.cuda(), v.cuda(), w.C, map_, g, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    S_ref, z_ref = oracle.prefix_state_map(to_f64(k), to_f64(v), name, g, eps, scale)
    es, ez = _state_err(to_f64(S), S_ref), _state_err(to_f64(z), z_ref)
    tol = STATE_TOL[w.dtype]
    assert es <= tol and ez <= tol, f"state {es:.2e}, z {ez:.2e} (bar {tol:.0e})"
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), name, g, eps, scale)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


def test_map_state_composed_eps_diagonal(kg):
    """Zero keys: psi(0) = eps I for Sigma_g, so the state is eps sum_t v_t on the
    diagonal features and zero elsewhere, and z is eps T there: the eps terms
    alone, checked exactly up to fp32 rounding."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=2, T=300)
    q, k, v = workloads.make_qkv(w)
    k.zero_()
    for g in (1, 2):
        out, S, z = kg.kata_fwd_chunked_map_state(q.cuda(), k.cuda(), v.cuda(), w.C, 2, g, 0.5, 0.25)
        torch.cuda.synchronize()
        S_ref, z_ref = oracle.prefix_state_map(to_f64(k), to_f64(v), "Sigma", g, 0.5, 0.25)
        assert _state_err(to_f64(S), S_ref) <= 1e-5 and _state_err(to_f64(z), z_ref) <= 1e-6, g
