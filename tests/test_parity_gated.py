"""GPU parity of GatedKATA (the pages' multiplicative scalar state gate:
S_t = gamma_t S_{t-1} + psi(k_t) v_t^T, Z_t alike) against the CPU oracle:
kata_fwd_chunked_gated element by element at sizes the oracle finishes in
seconds (several chunks and a ragged tail, resets and unit gates at chunk
edges, both readouts), the exported final state, the gated decode step, and
sampled rows at the mid-size workload."""
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


def _gates(w, edges=True):
    g = workloads.make_gate(w)
    if edges:   # exact resets and unit gates, on and next to chunk boundaries
        T, C = w.T, w.C
        for t in (0, C - 1, C, 2 * C + 1, T - 1):
            if t < T:
                g[..., t] = 0.0
        for t in (1, C + 1, 2 * C):
            if t < T:
                g[..., t] = 1.0
        g[..., 3::17] = 0.5
    return g.contiguous()


def _check(kg, w, g, normalize):
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C, normalize)
    torch.cuda.synchronize()
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[w.dtype], f"{w.name} normalize={normalize}: {err:.3e}"


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d,dv,C,dtype", [
    (16, 16, 32, torch.float32), (32, 64, 64, torch.bfloat16), (64, 64, 64, torch.bfloat16),
    (32, 128, 128, torch.float32), (16, 32, 32, torch.bfloat16), (64, 16, 128, torch.float32)])
def test_gated_forward_parity(kg, normalize, d, dv, C, dtype):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=2, H=2, T=3 * C + 7, d=d, dv=dv, C=C,
                                               dtype=dtype)
    _check(kg, w, _gates(w), normalize)


@pytest.mark.parametrize("T", [1, 31, 32, 33, 95])
def test_gated_forward_ragged(kg, T):
    w = workloads.WORKLOADS["small_fp32"].scaled(B=1, H=3, T=T)
    for normalize in (True, False):
        _check(kg, w, _gates(w, edges=T > 40), normalize)


def test_gated_unit_and_zero_gates(kg):
    """gamma = 1 everywhere is plain KATA; gamma = 0 everywhere keeps only the
    token's own write (o_t = v_t where (q_t . k_t) != 0)."""
    w = workloads.WORKLOADS["small_fp32"].scaled(B=1, H=2, T=100)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    one = torch.ones((w.B, w.H, w.T), device="cuda")
    a = kg.kata_fwd_chunked_gated(q, k, v, one, w.C)
    torch.cuda.synchronize()
    ref = oracle.forward(to_f64(q), to_f64(k), to_f64(v))
    assert slice_rel_err(to_f64(a), ref) <= TOL[torch.float32]
    zero = torch.zeros_like(one)
    b = kg.kata_fwd_chunked_gated(q, k, v, zero, w.C)
    torch.cuda.synchronize()
    assert slice_rel_err(to_f64(b), to_f64(v)) <= TOL[torch.float32]


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d,dv,C,dtype", [(16, 16, 32, torch.float32),
                                          (32, 64, 64, torch.bfloat16),
                                          (64, 32, 64, torch.float32)])
def test_gated_state_export_and_decode(kg, normalize, d, dv, C, dtype):
    """The state after the last token equals the oracle's gated recurrence, and a
    gated decode step from it continues the forward."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=2, H=2, T=2 * C + 5, d=d, dv=dv, C=C,
                                               dtype=dtype)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    T = w.T - 1   # the forward covers tokens 0 .. T-1; the decode step takes token T
    g[..., T] = 0.9   # a reset here would make the step's output independent of the state
    sl = (slice(None), slice(None), slice(0, T))
    out, S, z = kg.kata_fwd_chunked_gated(q[sl].contiguous().cuda(), k[sl].contiguous().cuda(),
                                          v[sl].contiguous().cuda(), g[sl].contiguous().cuda(),
                                          C, normalize, with_state=True)
    torch.cuda.synchronize()
    S_ref, z_ref = oracle.prefix_state_gated(to_f64(k[sl]), to_f64(v[sl]), to_f64(g[sl]))
    # the tensor path sums products of bf16 lifted keys (scaled by the gates) with v
    tc = kg.kata_fwd_path_gated(w.B, w.H, T, d, dv, C, dtype) == kg.KATA_PATH_TC
    stol = 1e-2 if tc else TOL[torch.float32]
    assert slice_rel_err(to_f64(S), S_ref) <= stol
    assert slice_rel_err(to_f64(z)[..., None], z_ref[..., None]) <= stol
    o = kg.kata_decode_step_gated(S, z, q[..., T, :].contiguous().cuda(),
                                  k[..., T, :].contiguous().cuda(),
                                  v[..., T, :].contiguous().cuda(),
                                  g[..., T].contiguous().cuda(), normalize)
    torch.cuda.synchronize()
    full = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    err = slice_rel_err(to_f64(o)[:, :, None, :], full[:, :, T:T + 1, :])
    assert err <= TOL[dtype], f"{err:.3e}"


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gated_decode_parity(kg, normalize, dtype):
    w = workloads.DECODE.scaled(B=4, H=4, dtype=dtype)
    kp, vp = workloads.make_decode_prefix(w, length=12)
    gp = torch.sigmoid(torch.randn(w.B, w.H, 12, generator=torch.Generator().manual_seed(5)) + 2)
    S0, z0 = oracle.prefix_state_gated(to_f64(kp), to_f64(vp), to_f64(gp))
    q, k, v = workloads.make_decode_inputs(w)
    g = workloads.make_decode_gate(w)
    S = torch.from_numpy(S0).float().cuda()
    z = torch.from_numpy(z0).float().cuda()
    o = kg.kata_decode_step_gated(S, z, q.cuda(), k.cuda(), v.cuda(), g.cuda(), normalize)
    torch.cuda.synchronize()
    S1, z1, o_ref = oracle.decode_step_gated(S0, z0, to_f64(q), to_f64(k), to_f64(v), to_f64(g),
                                             normalize)
    assert slice_rel_err(to_f64(o)[:, :, None, :], o_ref[:, :, None, :]) <= TOL[dtype]
    assert slice_rel_err(to_f64(S), S1) <= 1e-5
    assert slice_rel_err(to_f64(z)[..., None], z1[..., None]) <= 1e-5


def test_plain_decode_unchanged_by_a_unit_gate(kg):
    w = workloads.DECODE.scaled(B=2, H=3)
    q, k, v = (t.cuda() for t in workloads.make_decode_inputs(w))
    S, z = (t.cuda() for t in workloads.make_decode_state_fill(w))
    S2, z2 = S.clone(), z.clone()
    a = kg.kata_decode_step(S, z, q, k, v)
    b = kg.kata_decode_step_gated(S2, z2, q, k, v, torch.ones((w.B, w.H), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(S, S2) and torch.equal(z, z2)


@pytest.mark.parametrize("normalize", [True, False])
def test_gated_full_size_sampled_rows(kg, normalize):
    """The mid-size workload (B=4, H=8, T=4096, d=32, dv=64, C=64, bf16) with its
    seeded gates, sampled rows against the oracle."""
    w = workloads.WORKLOADS["mid_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    g = workloads.make_gate(w, device="cuda")
    out = kg.kata_fwd_chunked_gated(q, k, v, g, w.C, normalize)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    BH = w.B * w.H
    rng = np.random.default_rng(77)
    worst = 0.0
    qf, kf, vf, gf = to_f64(q), to_f64(k), to_f64(v), to_f64(g)
    for h in sorted(set([0, BH - 1] + rng.integers(0, BH, size=2).tolist())):
        b, hh = divmod(h, w.H)
        ts = np.array(sorted(set([0, 1, w.C - 1, w.C, w.T // 2, w.T - 1] +
                                 rng.integers(0, w.T, size=10).tolist())), dtype=np.int64)
        ref = oracle.forward_rows_gated(qf[b:b + 1, hh:hh + 1], kf[b:b + 1, hh:hh + 1],
                                        vf[b:b + 1, hh:hh + 1], gf[b:b + 1, hh:hh + 1], ts,
                                        normalize)
        got = to_f64(out[b, hh])[ts]
        worst = max(worst, slice_rel_err(got, ref))
    assert worst <= TOL[w.dtype], f"{worst:.3e}"


# ---- GatedKATA in the quadratic form on the tensor cores (bf16, d in {32, 64}, dv = 64)
@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d,T", [(32, 129), (32, 300), (64, 257), (64, 1000)])
def test_gated_quadratic_parity(kg, normalize, d, T):
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=2, H=2, T=T, d=d, C=128)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out = kg.kata_fwd_quadratic_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), normalize)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[torch.bfloat16], f"d={d} T={T} normalize={normalize}: {err:.3e}"


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d,dv", [(16, 64), (16, 128), (32, 16), (64, 32), (64, 128)])
def test_gated_quadratic_adapted_shapes(kg, normalize, d, dv):
    """Other bf16 head sizes in the gated quadratic form: q, k padded to d = 32,
    v in 64-column parts, each part one pass of the kernel."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=2, H=2, T=300, d=d, dv=dv, C=128)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out = kg.kata_fwd_quadratic_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), normalize)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[torch.bfloat16], f"d={d} dv={dv} normalize={normalize}: {err:.3e}"


@pytest.mark.parametrize("T", [1, 127, 128, 129])
def test_gated_quadratic_ragged(kg, T):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=3, T=T, C=128)
    q, k, v = workloads.make_qkv(w)
    g = workloads.make_gate(w)
    g[..., T // 2] = 0.0
    out = kg.kata_fwd_quadratic_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda())
    torch.cuda.synchronize()
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g))
    assert slice_rel_err(to_f64(out), ref) <= TOL[torch.bfloat16]


def test_gated_quadratic_unit_gate_is_the_plain_kernel(kg):
    """gamma = 1: scaled keys equal the keys, every factor is 1, so the gated
    kernel produces the plain quadratic kernel's output bit for bit."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=2, H=3, T=700)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    one = torch.ones((w.B, w.H, w.T), device="cuda")
    a = kg.kata_fwd_quadratic_gated(q, k, v, one)
    b = kg.kata_fwd_quadratic(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("normalize", [True, False])
def test_gated_quadratic_full_size_sampled_rows(kg, normalize):
    """The LM-layer workload (B=8, H=16, T=2048, d=64, dv=64, bf16) with its seeded
    gates, sampled rows against the oracle."""
    w = workloads.WORKLOADS["lm_layer_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    g = workloads.make_gate(w, device="cuda")
    out = kg.kata_fwd_quadratic_gated(q, k, v, g, normalize)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    assert torch.isfinite(out).all()
    BH = w.B * w.H
    rng = np.random.default_rng(78)
    worst = 0.0
    qf, kf, vf, gf = to_f64(q), to_f64(k), to_f64(v), to_f64(g)
    for h in sorted(set([0, BH - 1] + rng.integers(0, BH, size=2).tolist())):
        b, hh = divmod(h, w.H)
        ts = np.array(sorted(set([0, 1, 127, 128, w.T // 2, w.T - 1] +
                                 rng.integers(0, w.T, size=10).tolist())), dtype=np.int64)
        ref = oracle.forward_rows_gated(qf[b:b + 1, hh:hh + 1], kf[b:b + 1, hh:hh + 1],
                                        vf[b:b + 1, hh:hh + 1], gf[b:b + 1, hh:hh + 1], ts,
                                        normalize)
        worst = max(worst, slice_rel_err(to_f64(out[b, hh])[ts], ref))
    assert worst <= TOL[w.dtype], f"{worst:.3e}"


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d,dtype,form", [
    (32, torch.bfloat16, "quadratic"),   # tensor-core quadratic form
    (64, torch.bfloat16, "quadratic"),
    (32, torch.float32, "chunked"),      # fp32: the chunked CUDA-core form
])
def test_gated_auto_form(kg, normalize, d, dtype, form):
    """kata_fwd_gated takes the form kata_fwd_gated_form names, and either form
    matches the oracle's gated forward."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=2, T=300, d=d, C=64, dtype=dtype)
    want = {"quadratic": kg.KATA_FORM_QUADRATIC, "chunked": kg.KATA_FORM_CHUNKED}[form]
    assert kg.kata_fwd_gated_form(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == want
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out = kg.kata_fwd_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C, normalize)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[w.dtype], f"{form} normalize={normalize}: {err:.3e}"


# ---- GatedKATA chunked on the tensor cores (bf16, d = 32, dv = 64): the d = 32
# segments with gated keys, a gated segment scan and decayed running state
def _seam_rows(kg, w):
    nseg, seg_tokens = kg.kata_fwd_segments(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype)
    rows = []
    for g in range(1, nseg):
        s0 = g * seg_tokens
        rows += [s0 - 2, s0 - 1, s0, s0 + 1, s0 + 127, s0 + 128]
    return [t for t in rows if 0 <= t < w.T]


_TC_SHAPES = [
    (1, 2, 1100),    # nine one-chunk segments per head: state kernel, gated scan
    (4, 15, 1000),   # 60 heads: 2 segments of 4 chunks, sums from 2 pieces of 2 chunks
    (1, 4, 5000),    # 20 segments of 2 chunks, one-chunk pieces
    (8, 8, 1000),    # 2 segments of 4 chunks, ragged tail
    (1, 1, 129),     # last chunk holds one token
    (3, 1, 5),       # a single partial chunk
]


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("B,H,T", _TC_SHAPES)
def test_gated_tensor_path(kg, normalize, B, H, T):
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path_gated(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)   # resets and unit gates at 128-token chunk edges, runs of 0.5
    out = kg.kata_fwd_chunked_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C, normalize)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[w.dtype], f"normalize={normalize}: {err:.3e}"


@pytest.mark.parametrize("B,H,T", [(1, 2, 1100), (4, 15, 1000), (1, 1, 129)])
def test_gated_tensor_path_unit_gates_are_the_plain_path(kg, B, H, T):
    """gamma = 1: every scale is exactly 1 and every decay exactly 1, so the
    gated tensor path reproduces the plain one bit for bit."""
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=B, H=H, T=T)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    one = torch.ones((w.B, w.H, w.T), device="cuda")
    a = kg.kata_fwd_chunked_gated(q, k, v, one, w.C)
    b = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_gated_tensor_path_zero_gates(kg):
    """gamma = 0 everywhere keeps only each token's own write: o_t = v_t."""
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=1, H=2, T=1100)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    zero = torch.zeros((w.B, w.H, w.T), device="cuda")
    for normalize in (True, False):
        out = kg.kata_fwd_chunked_gated(q, k, v, zero, w.C, normalize)
        torch.cuda.synchronize()
        ref = oracle.forward_gated(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()),
                                   to_f64(zero.cpu()), normalize)
        assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]
    out = kg.kata_fwd_chunked_gated(q, k, v, zero, w.C, True)
    torch.cuda.synchronize()
    assert slice_rel_err(to_f64(out), to_f64(v)) <= TOL[w.dtype]


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("B,H,T", [(1, 2, 1100), (4, 15, 1000), (1, 4, 5000), (16, 10, 700)])
def test_gated_tensor_path_state(kg, normalize, B, H, T):
    """The state after the last token: the last segment's running state and Gram,
    which start from the gated prefix of the segments before (160 heads at
    T = 700: one segment each)."""
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=B, H=H, T=T)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out, S, z = kg.kata_fwd_chunked_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C, normalize,
                                          with_state=True)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    S_ref, z_ref = oracle.prefix_state_gated(to_f64(k), to_f64(v), to_f64(g))
    assert slice_rel_err(to_f64(S), S_ref) <= 1e-2
    assert slice_rel_err(to_f64(z)[..., None], z_ref[..., None]) <= 1e-2
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


@pytest.mark.parametrize("normalize", [True, False])
def test_gated_tensor_path_long_context_sampled_rows(kg, normalize):
    """The long-context workload (B=1, H=16, T=131072) with its seeded gates plus
    resets and unit gates at chunk edges, sampled rows (the rows on both sides of
    every segment seam among them) against the oracle."""
    w = workloads.WORKLOADS["long_ctx_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    g = workloads.make_gate(w, device="cuda")
    g[..., 128 * 300] = 0.0          # a reset at a chunk start
    g[..., 128 * 301 - 1] = 0.0      # and at a chunk end
    g[..., 5000:5300] = 1.0          # a run of unit gates
    g[..., 70000:70100] = 0.5        # a run of halving gates
    out = kg.kata_fwd_chunked_gated(q, k, v, g, w.C, normalize)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    assert torch.isfinite(out).all()
    BH = w.B * w.H
    rng = np.random.default_rng(131)
    seams = _seam_rows(kg, w)
    fixed = [0, 1, 127, 128, 128 * 300 - 1, 128 * 300, 128 * 300 + 1, 128 * 301 - 1,
             128 * 301, 5299, 70050, 70100, w.T - 1]
    worst = 0.0
    for h in sorted(set([0, BH - 1] + rng.integers(0, BH, size=2).tolist())):
        ts = np.array(sorted(set(fixed + seams + rng.integers(0, w.T, size=16).tolist())),
                      dtype=np.int64)
        qh, kh, vh = (to_f64(t.reshape(BH, 1, w.T, -1)[h:h + 1]) for t in (q, k, v))
        gh = to_f64(g.reshape(BH, 1, w.T)[h:h + 1])
        ref = oracle.forward_rows_gated(qh, kh, vh, gh, ts, normalize)
        got = to_f64(out.reshape(BH, w.T, w.dv)[h])[ts]
        worst = max(worst, slice_rel_err(got, ref))
    print(f"long-context gated: {len(seams)} seam rows, worst slice metric {worst:.3e}")
    assert worst <= TOL[w.dtype], f"{worst:.3e}"


@pytest.mark.parametrize("d,T,form", [
    (32, 10240, "quadratic"), (32, 10241, "chunked"), (32, 32768, "chunked"),
    (64, 32768, "quadratic"), (64, 65536, "quadratic"), (64, 65537, "chunked"),
])
def test_gated_form_bounds(kg, d, T, form):
    """kata_fwd_gated's form at and past its measured bounds (bf16, dv = 64)."""
    want = {"quadratic": kg.KATA_FORM_QUADRATIC, "chunked": kg.KATA_FORM_CHUNKED}[form]
    assert kg.kata_fwd_gated_form(1, 1, T, d, 64, 64, torch.bfloat16) == want


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d", [32, 64])
def test_gated_auto_form_32k_sampled_rows(kg, normalize, d):
    """kata_fwd_gated at T = 32768 (d = 32: the chunked tensor form; d = 64: the
    quadratic form) with the seeded gates plus resets, unit gates and runs of
    0.5 gates, sampled rows against the oracle."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=2, T=32768, d=d, C=64)
    q, k, v = workloads.make_qkv(w, device="cuda")
    g = workloads.make_gate(w, device="cuda")
    for t in (0, 127, 128, 4095, 4096, 20000):
        g[..., t] = 0.0
    g[..., 1000:1400] = 1.0
    g[..., 9000:9300] = 0.5
    g[..., 30000:30040] = 0.5
    out = kg.kata_fwd_gated(q, k, v, g, w.C, normalize)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    assert torch.isfinite(out).all()
    BH = w.B * w.H
    rng = np.random.default_rng(32768 + d)
    fixed = [0, 1, 127, 128, 129, 1399, 4095, 4096, 4097, 9299, 19999, 20000, 20001, 30039,
             w.T - 1]
    worst = 0.0
    for h in range(BH):
        ts = np.array(sorted(set(fixed + rng.integers(0, w.T, size=12).tolist())), dtype=np.int64)
        qh, kh, vh = (to_f64(t.reshape(BH, 1, w.T, -1)[h:h + 1]) for t in (q, k, v))
        gh = to_f64(g.reshape(BH, 1, w.T)[h:h + 1])
        ref = oracle.forward_rows_gated(qh, kh, vh, gh, ts, normalize)
        worst = max(worst, slice_rel_err(to_f64(out.reshape(BH, w.T, w.dv)[h])[ts], ref))
    assert worst <= TOL[w.dtype], f"d={d}: {worst:.3e}"


# ---- GatedKATA at d = 64 on the tensor cores (bf16, dv = 64): the output from the
# gated quadratic form, the state from the chunked d = 64 path on sqrt(A_s) k_s
@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("B,H,T", [
    (1, 38, 300),    # 38 heads: the fewest with the d = 64 chunked path for the state
    (2, 19, 129),    # last tile holds one token
    (4, 10, 5),      # a single partial tile
])
def test_gated_d64_tensor_path_state(kg, normalize, B, H, T):
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path_gated(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out, S, z = kg.kata_fwd_chunked_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C, normalize,
                                          with_state=True)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]
    S_ref, z_ref = oracle.prefix_state_gated(to_f64(k), to_f64(v), to_f64(g))
    assert slice_rel_err(to_f64(S), S_ref) <= 1e-2
    assert slice_rel_err(to_f64(z)[..., None], z_ref[..., None]) <= 1e-2


def test_gated_d64_prefill_then_decode(kg):
    """Gated prefill of T-1 tokens at the decode shape's head size (d = 64) with the
    state exported on the tensor path, then one gated decode step: the step's
    output is the definition's output at row T-1."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=2, H=19, T=257)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    Tp = w.T - 1
    g[..., Tp] = 0.9   # a reset here would make the step's output independent of the state
    sl = (slice(None), slice(None), slice(0, Tp))
    _, S, z = kg.kata_fwd_chunked_gated(q[sl].contiguous().cuda(), k[sl].contiguous().cuda(),
                                        v[sl].contiguous().cuda(), g[sl].contiguous().cuda(),
                                        w.C, True, with_state=True)
    o = kg.kata_decode_step_gated(S, z, q[..., Tp, :].contiguous().cuda(),
                                  k[..., Tp, :].contiguous().cuda(),
                                  v[..., Tp, :].contiguous().cuda(), g[..., Tp].contiguous().cuda())
    torch.cuda.synchronize()
    full = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g))
    assert slice_rel_err(to_f64(o)[:, :, None, :], full[:, :, Tp:Tp + 1, :]) <= TOL[w.dtype]


def test_gated_d64_few_heads_state(kg):
    """Fewer than 38 heads with the state exported: the state comes from the d = 64
    chunked kernels with SMs left idle."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=3, T=200)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out, S, z = kg.kata_fwd_chunked_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C, True,
                                          with_state=True)
    torch.cuda.synchronize()
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g))
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]
    S_ref, _ = oracle.prefix_state_gated(to_f64(k), to_f64(v), to_f64(g))
    assert kg.kata_fwd_path_gated(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    assert slice_rel_err(to_f64(S), S_ref) <= 1e-2


# ---- other bf16 head sizes (d = 16, dv != 64) on the gated tensor routes: q, k
# padded to d = 32, v in 64-column parts, each part one gated forward
_ADAPTED_GATED = [
    (16, 64, 1, 2, 1100),    # the d = 32 gated segments, q and k padded
    (16, 128, 2, 2, 300),
    (32, 16, 1, 3, 700),
    (32, 128, 1, 2, 1100),
    (64, 32, 1, 2, 300),     # d = 64: output from the gated quadratic form
    (64, 128, 2, 2, 129),
]


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d,dv,B,H,T", _ADAPTED_GATED)
def test_gated_adapted_shapes(kg, normalize, d, dv, B, H, T):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=B, H=H, T=T, d=d, dv=dv, C=128)
    assert kg.kata_fwd_path_gated(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    _check(kg, w, _gates(w), normalize)
    assert kg.kata_sync_status() == kg.KATA_OK


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("d,dv,B,H,T", [
    (16, 128, 1, 2, 1100),   # padded features gathered, two column blocks
    (32, 32, 2, 2, 300),
    (64, 128, 2, 19, 300),   # d = 64: the state from the chunked d = 64 kernels
])
def test_gated_adapted_shapes_state(kg, normalize, d, dv, B, H, T):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=B, H=H, T=T, d=d, dv=dv, C=128)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out, S, z = kg.kata_fwd_chunked_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C, normalize,
                                          with_state=True)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), normalize)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]
    S_ref, z_ref = oracle.prefix_state_gated(to_f64(k), to_f64(v), to_f64(g))
    assert slice_rel_err(to_f64(S), S_ref) <= 1e-2
    assert slice_rel_err(to_f64(z)[..., None], z_ref[..., None]) <= 1e-2


def test_gated_adapted_prefill_then_decode(kg):
    """Gated prefill at d = 16, dv = 128 on the tensor route, then a gated decode
    step from the exported state: the definition's output at the last row."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=3, T=500, d=16, dv=128, C=128)
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    Tp = w.T - 1
    g[..., Tp] = 0.9   # a reset here would make the step's output independent of the state
    sl = (slice(None), slice(None), slice(0, Tp))
    _, S, z = kg.kata_fwd_chunked_gated(q[sl].contiguous().cuda(), k[sl].contiguous().cuda(),
                                        v[sl].contiguous().cuda(), g[sl].contiguous().cuda(),
                                        w.C, True, with_state=True)
    o = kg.kata_decode_step_gated(S, z, q[..., Tp, :].contiguous().cuda(),
                                  k[..., Tp, :].contiguous().cuda(),
                                  v[..., Tp, :].contiguous().cuda(), g[..., Tp].contiguous().cuda())
    torch.cuda.synchronize()
    full = oracle.forward_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g))
    assert slice_rel_err(to_f64(o)[:, :, None, :], full[:, :, Tp:Tp + 1, :]) <= TOL[w.dtype]


@pytest.mark.parametrize("d,dv,T,form", [(16, 128, 300, "quadratic"), (32, 16, 20000, "chunked")])
def test_gated_auto_form_adapted_shapes(kg, d, dv, T, form):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=2, T=T, d=d, dv=dv, C=128)
    want = {"quadratic": kg.KATA_FORM_QUADRATIC, "chunked": kg.KATA_FORM_CHUNKED}[form]
    assert kg.kata_fwd_gated_form(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == want
    q, k, v = workloads.make_qkv(w)
    g = _gates(w)
    out = kg.kata_fwd_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda(), w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    rows = np.array(sorted(set([0, 1, 127, 128, T // 2, T - 1, T + 3, 2 * T - 1])),
                    dtype=np.int64)
    ref = oracle.forward_rows_gated(to_f64(q), to_f64(k), to_f64(v), to_f64(g), rows)
    got = to_f64(out).reshape(-1, w.dv)[rows]
    assert slice_rel_err(got, ref) <= TOL[w.dtype]
