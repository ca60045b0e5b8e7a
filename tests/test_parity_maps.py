"""GPU parity of the reduced PSD families (KATA-M_g, KATA-Sigma_g; [KATA] Sec. 4.1)
against the CPU oracle: kata_fwd_chunked_map element by element at sizes the
oracle finishes in seconds (several chunks and a ragged tail), kata_lift_map,
and sampled rows at the LM-layer size (B=8, H=16, T=2048, d=64)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import TOL, require_gpu, slice_rel_err, to_f64

pytestmark = pytest.mark.gpu

NAMES = {1: "M", 2: "Sigma"}


@pytest.fixture(scope="module")
def kg():
    return require_gpu()


def _params(kg, map_, g):
    # the Sigma configuration: eps = 1e-4, scale 1 (Sigma_2) or 1/4 (Sigma_4)
    if map_ == kg.KATA_MAP_SUM:
        return 1e-4, (0.25 if g == 4 else 1.0)
    return 0.0, 1.0


@pytest.mark.parametrize("map_", [1, 2])
@pytest.mark.parametrize("g", [2, 4])
@pytest.mark.parametrize("d,dv,C", [(16, 16, 32), (32, 64, 64), (64, 64, 64)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_map_forward_parity(kg, map_, g, d, dv, C, dtype):
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=2, T=3 * C + 7, d=d, dv=dv, C=C,
                                                    dtype=dtype)
    q, k, v = workloads.make_qkv(w)
    eps, scale = _params(kg, map_, g)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), C, map_, g, eps, scale)
    torch.cuda.synchronize()
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), NAMES[map_], g, eps, scale)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[dtype], f"{NAMES[map_]}_{g} d={d}: {err:.3e}"


@pytest.mark.parametrize("map_,g", [(1, 2), (1, 4), (2, 2), (2, 4)])
def test_map_forward_ragged(kg, map_, g):
    eps, scale = _params(kg, map_, g)
    for T in (1, 31, 32, 33):
        w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=1, T=T, C=32, dtype=torch.float32)
        q, k, v = workloads.make_qkv(w)
        out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), 32, map_, g, eps, scale)
        torch.cuda.synchronize()
        ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), NAMES[map_], g, eps, scale)
        assert slice_rel_err(to_f64(out), ref) <= TOL[torch.float32]


def test_full_map_is_the_plain_forward(kg):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=2, T=300)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_chunked_map(q, k, v, w.C, kg.KATA_MAP_FULL, 1)
    b = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("map_,g,d", [(1, 2, 64), (1, 4, 32), (2, 2, 64), (2, 4, 16)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_map_lift_parity(kg, map_, g, d, dtype):
    x = torch.randn(37, d, generator=torch.Generator().manual_seed(d + g)).to(dtype)
    eps, scale = _params(kg, map_, g)
    phi = kg.kata_lift_map(x.cuda(), map_, g, eps, scale)
    torch.cuda.synchronize()
    ref = oracle.lift_map(to_f64(x), NAMES[map_], g, eps, scale)
    err = float(np.max(np.abs(to_f64(phi) - ref)) / np.max(np.abs(ref)))
    assert err <= 1e-6


@pytest.mark.parametrize("map_,g", [(1, 2), (2, 2), (1, 4), (2, 4), (2, 1)])
def test_map_full_size_sampled_rows(kg, map_, g):
    """The LM-layer workload with M_2 / Sigma_2 / M_4 / Sigma_4 / Sigma_1, sampled
    rows against the oracle."""
    w = workloads.WORKLOADS["lm_layer_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    eps, scale = _params(kg, map_, g)
    out = kg.kata_fwd_chunked_map(q, k, v, w.C, map_, g, eps, scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    BH = w.B * w.H
    rng = np.random.default_rng(w.index + 10 * map_)
    worst = 0.0
    for h in sorted(set([0, BH - 1] + rng.integers(0, BH, size=1).tolist())):
        ts = np.array(sorted(set([0, 1, w.C - 1, w.C, w.T // 2, w.T - 1] +
                                 rng.integers(0, w.T, size=10).tolist())), dtype=np.int64)
        ref = oracle.forward_rows_map(to_f64(q.reshape(BH, 1, w.T, w.d)[h:h + 1]),
                                      to_f64(k.reshape(BH, 1, w.T, w.d)[h:h + 1]),
                                      to_f64(v.reshape(BH, 1, w.T, w.dv)[h:h + 1]), ts,
                                      NAMES[map_], g, eps, scale)
        got = to_f64(out.reshape(BH, w.T, w.dv)[h][ts])
        worst = max(worst, slice_rel_err(got, ref))
    assert worst <= TOL[w.dtype], f"{NAMES[map_]}_{g}: {worst:.3e}"


@pytest.mark.parametrize("B,H,T", [
    (1, 2, 1100),    # 4 sub-heads: many one-chunk segments (state kernel + scan per sub-head)
    (8, 8, 700),     # 128 sub-heads, one segment each, ragged tail
    (2, 3, 129),     # last chunk holds one token
    (3, 1, 5),       # a single partial chunk
])
def test_m2_tensor_path(kg, B, H, T):
    """KATA-M_2 at d = 64 (bf16, dv = 64): two d = 32 sub-heads on the tensor path,
    numerators and denominators summed."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, 1, 2) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 1, 2)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "M", 2)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


@pytest.mark.parametrize("B,H,T", [
    (1, 2, 1100),    # 8 sub-heads: 9 one-chunk segments (state kernel on the key halves + scan)
    (8, 8, 700),     # 256 sub-heads, one segment each, ragged tail
    (2, 3, 129),     # last chunk holds one token
    (3, 1, 5),       # a single partial chunk
])
@pytest.mark.parametrize("eps,scale", [
    (1e-4, 1.0),     # the Sigma_2 configuration
    (0.5, 0.25),     # eps terms of the size of the (q_a . k_b)^2 terms
    (3.0, 1.0),      # eps terms dominant
])
def test_sigma2_tensor_path(kg, B, H, T, eps, scale):
    """KATA-Sigma_2 at d = 64 (bf16, dv = 64): four crosswise d = 32 sub-heads on
    the tensor path plus the eps terms as a linear attention."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, 2, 2) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 2, 2, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "Sigma", 2, eps, scale)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


def test_sigma2_tensor_path_eps_only_rows(kg):
    """Zero queries: <psi(0), psi(k)> = eps^2 m + eps s |k|^2, so those rows come
    from the eps terms alone; zero keys in one half leave only the other half's
    cross terms."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=2, T=300)
    q, k, v = workloads.make_qkv(w)
    q[:, :, ::3] = 0
    k[:, :, 100:200, 32:] = 0
    for eps, scale in ((1e-4, 1.0), (0.5, 0.25)):
        out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 2, 2, eps, scale)
        torch.cuda.synchronize()
        ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "Sigma", 2, eps, scale)
        assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype], (eps, scale)


def test_sigma2_eps_zero_is_four_cross_terms(kg):
    """eps = 0: the weight is scale^2 sum_{a,b} (q_a . k_b)^2, and the scale cancels."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=3, T=400)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_chunked_map(q, k, v, w.C, 2, 2, 0.0, 1.0)
    b = kg.kata_fwd_chunked_map(q, k, v, w.C, 2, 2, 0.0, 0.5)
    torch.cuda.synchronize()
    ref = oracle.forward_map(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()), "Sigma", 2, 0.0, 1.0)
    assert slice_rel_err(to_f64(a), ref) <= TOL[w.dtype]
    assert slice_rel_err(to_f64(b), to_f64(a)) <= 1e-2


@pytest.mark.parametrize("B,H,T", [
    (1, 2, 1100),    # 8 sub-heads: 9 one-chunk segments
    (8, 8, 700),     # 256 sub-heads, one segment each, ragged tail
    (2, 3, 129),     # last chunk holds one token
    (3, 1, 5),       # a single partial chunk
])
def test_m4_tensor_path(kg, B, H, T):
    """KATA-M_4 at d = 64 (bf16, dv = 64): each 16-wide block zero-padded to 32
    and run as a d = 32 sub-head; the zero coordinates contribute nothing."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, 1, 4) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 1, 4)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "M", 4)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


def test_m4_tensor_path_zero_block(kg):
    """A query block that is zero in every row leaves only the other blocks'
    weights; a key block that is zero everywhere does the same."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=2, T=300)
    q, k, v = workloads.make_qkv(w)
    q[..., 16:32] = 0
    k[..., 48:64] = 0
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 1, 4)
    torch.cuda.synchronize()
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "M", 4)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


def test_map_paths(kg):
    """bf16, dv = 64: M_2, Sigma_2, M_4 at d = 64 as d = 32 sub-heads; Sigma_1 as
    the full map plus its eps terms; Sigma_4 at d = 64, every map at d = 16 and
    all but M_2 / M_1 / Sigma_1 at d = 32 (more than 192 features) on the
    explicit-feature path; fp32 on CUDA cores."""
    w = workloads.WORKLOADS["lm_layer_bf16"]

    def path(d=w.d, dv=w.dv, dtype=w.dtype, map_=1, g=2):
        return kg.kata_fwd_path_map(w.B, w.H, w.T, d, dv, w.C, dtype, map_, g)

    for map_, g in ((1, 2), (2, 2), (1, 4), (2, 4)):
        assert path(map_=map_, g=g) == kg.KATA_PATH_TC
        assert path(d=16, map_=map_, g=g) == kg.KATA_PATH_TC
        assert path(dtype=torch.float32, map_=map_, g=g) == kg.KATA_PATH_SIMT
    for map_, g in ((2, 2), (1, 4), (2, 4)):
        assert path(d=32, map_=map_, g=g) == kg.KATA_PATH_TC
    assert path(d=32, map_=1, g=2) == kg.KATA_PATH_TC       # padded d = 64 sub-heads
    assert path(d=32, map_=2, g=1) == kg.KATA_PATH_TC       # the d = 32 full map + eps terms
    assert path(map_=2, g=1) == kg.KATA_PATH_TC             # the d = 64 full map + eps terms
    assert path(dv=128, map_=2, g=1) == kg.KATA_PATH_TC     # 64-column parts of v
    assert path(dtype=torch.float32, map_=2, g=1) == kg.KATA_PATH_SIMT
    assert path(d=32, dv=128, map_=2, g=2) == kg.KATA_PATH_TC     # 64-column parts of v
    assert path(d=32, dv=128, dtype=torch.float32, map_=2, g=2) == kg.KATA_PATH_SIMT
    for d in (16, 32, 64):
        assert path(d=d, map_=kg.KATA_MAP_ORTHANT, g=1) == kg.KATA_PATH_TC


# ---- explicit-feature tensor path (kata_feat.cu): the map's features written
# out, chunk states and outputs on tcgen05 around the chunk scan
_FEAT_MAPS = [
    (2, 4, 64),   # Sigma_4 at the LM-layer head size: 136 features, 3 boxes, 2 blocks
    (2, 2, 32),   # 136
    (2, 4, 32),   # 36: one box, one block
    (1, 4, 32),   # 144
    (1, 2, 16),
    (2, 2, 16),
    (1, 4, 16),
    (2, 4, 16),   # 10 features
    (1, 1, 16),   # M_1 = the rank-one lift: the full map's path
    (2, 1, 16),   # Sigma_1: eps I + s x x^T, 136 features; weights s^2 (q.k)^2 + eps
                  # terms near zero for near-orthogonal pairs (the hi/lo X)
    (3, 1, 64),   # orthant: n = d
    (3, 1, 32),
    (3, 1, 16),
]


def _feat_params(kg, map_, g):
    return (1e-6, 1.0) if map_ == kg.KATA_MAP_ORTHANT else _params(kg, map_, g)


def _feat_name(map_):
    return "orthant" if map_ == 3 else NAMES[map_]


@pytest.mark.parametrize("map_,g,d", _FEAT_MAPS)
@pytest.mark.parametrize("B,H,T", [(1, 3, 300), (2, 2, 129), (1, 1, 5)])
def test_feature_path_parity(kg, map_, g, d, B, H, T):
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T, d=d)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, map_, g) == \
        kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    eps, scale = _feat_params(kg, map_, g)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, map_, g, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), _feat_name(map_), g, eps, scale)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[w.dtype], f"{_feat_name(map_)}_{g} d={d}: {err:.3e}"


def test_feature_path_deterministic(kg):
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=2, H=3, T=700)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_chunked_map(q, k, v, w.C, 2, 4, 1e-4, 0.25)
    b = kg.kata_fwd_chunked_map(q, k, v, w.C, 2, 4, 1e-4, 0.25)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("map_,g,d", [(2, 4, 64), (3, 1, 64)])
def test_feature_path_long_sequence_sampled_rows(kg, map_, g, d):
    """256 chunks per head (the two-level chunk scan), sampled rows."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=4, T=32768, d=d)
    q, k, v = workloads.make_qkv(w, device="cuda")
    eps, scale = _feat_params(kg, map_, g)
    out = kg.kata_fwd_chunked_map(q, k, v, w.C, map_, g, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    BH = w.B * w.H
    rng = np.random.default_rng(7)
    worst = 0.0
    for h in range(BH):
        ts = np.array(sorted(set([0, 1, 127, 128, 129, w.T // 2, w.T - 1] +
                                 rng.integers(0, w.T, size=12).tolist())), dtype=np.int64)
        ref = oracle.forward_rows_map(to_f64(q.reshape(BH, 1, w.T, w.d)[h:h + 1]),
                                      to_f64(k.reshape(BH, 1, w.T, w.d)[h:h + 1]),
                                      to_f64(v.reshape(BH, 1, w.T, w.dv)[h:h + 1]), ts,
                                      _feat_name(map_), g, eps, scale)
        got = to_f64(out.reshape(BH, w.T, w.dv)[h][ts])
        worst = max(worst, slice_rel_err(got, ref))
    assert worst <= TOL[w.dtype], f"{worst:.3e}"


# ---- orthant map (psi_i = max(u_i, 0) + eps, n = d) and the two-level chunk scan
@pytest.mark.parametrize("d,dv,C,dtype", [(16, 16, 32, torch.float32), (32, 64, 64, torch.bfloat16),
                                          (64, 64, 128, torch.bfloat16), (64, 32, 64, torch.float32)])
def test_orthant_forward_parity(kg, d, dv, C, dtype):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=3, T=3 * C + 5, d=d, dv=dv, C=C, dtype=dtype)
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), C, kg.KATA_MAP_ORTHANT, 1, 1e-6)
    torch.cuda.synchronize()
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "orthant", 1, 1e-6)
    assert slice_rel_err(to_f64(out), ref) <= TOL[dtype]
    x = q.reshape(-1, d)[:50].cuda()
    phi = kg.kata_lift_map(x, kg.KATA_MAP_ORTHANT, 1, 1e-6)
    torch.cuda.synchronize()
    refl = oracle.lift_map(to_f64(x.cpu()), "orthant", 1, 1e-6)
    assert float(np.max(np.abs(to_f64(phi) - refl))) <= 1e-6 * float(np.max(np.abs(refl)))


@pytest.mark.parametrize("mapname,d,dv", [("orthant", 64, 64), ("full", 16, 16)])
def test_two_level_scan(kg, monkeypatch, mapname, d, dv):
    """Few heads, small states, many chunks: the two-level chunk scan (forced) and
    the one-pass scan (forced) both match the oracle and each other; the state
    exported through the two-level scan matches the oracle's recurrence."""
    w = workloads.WORKLOADS["small_fp32"].scaled(B=1, H=2, T=64 * 32 + 9, d=d, dv=dv, C=32)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    code = kg.KATA_MAP_ORTHANT if mapname == "orthant" else kg.KATA_MAP_FULL
    eps = 1e-6 if mapname == "orthant" else 0.0
    outs = {}
    for mode in ("sequential", "blocked"):
        monkeypatch.setenv("KATA_CHUNK_SCAN", mode)
        outs[mode] = kg.kata_fwd_chunked_map(q, k, v, w.C, code, 1, eps)
        torch.cuda.synchronize()
    monkeypatch.delenv("KATA_CHUNK_SCAN")
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), mapname, 1, eps)
    for mode, o in outs.items():
        assert slice_rel_err(to_f64(o), ref) <= TOL[torch.float32], mode
    assert slice_rel_err(to_f64(outs["blocked"]), to_f64(outs["sequential"])) <= 1e-5
    if mapname == "full":
        monkeypatch.setenv("KATA_CHUNK_SCAN", "blocked")
        _, S, z = kg.kata_fwd_chunked_state(q, k, v, w.C)
        torch.cuda.synchronize()
        S_ref, z_ref = oracle.prefix_state(to_f64(k), to_f64(v))
        assert slice_rel_err(to_f64(S), S_ref) <= 1e-5
        assert slice_rel_err(to_f64(z)[..., None], z_ref[..., None]) <= 1e-5


@pytest.mark.parametrize("map_,g,d,dv", [
    (1, 2, 64, 128),   # M_2 sub-heads, two parts
    (2, 2, 64, 32),    # Sigma_2 crosswise sub-heads, one zero-padded part
    (1, 4, 64, 16),    # M_4 padded sub-heads
    (2, 4, 64, 128),   # Sigma_4, explicit features
    (2, 2, 32, 16),
    (3, 1, 64, 32),    # orthant
    (2, 1, 64, 128),   # Sigma_1: the d = 64 full map plus eps terms, two parts
])
def test_map_value_parts(kg, map_, g, d, dv):
    """bf16 with dv != 64: the map's dv = 64 route on 64-column parts of v."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=3, T=300, d=d, dv=dv)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, map_, g) == \
        kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    eps, scale = _feat_params(kg, map_, g)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, map_, g, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), _feat_name(map_), g, eps, scale)
    err = slice_rel_err(to_f64(out), ref)
    assert err <= TOL[w.dtype], f"{_feat_name(map_)}_{g} d={d} dv={dv}: {err:.3e}"


@pytest.mark.parametrize("B,H,T,dv", [(1, 3, 300, 64), (2, 2, 129, 64), (1, 2, 1100, 64),
                                      (1, 2, 300, 128)])
def test_m2_d32_padded_sub_heads(kg, B, H, T, dv):
    """KATA-M_2 at d = 32 (272 features) as M_2 at d = 64 on [u_1 0 | u_2 0]: two
    d = 32 sub-heads whose padded halves add nothing."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T, d=32, dv=dv)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, 1, 2) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 1, 2)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "M", 2)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


@pytest.mark.parametrize("B,H,T,dv", [(1, 3, 300, 64), (2, 2, 129, 64), (1, 2, 300, 128)])
@pytest.mark.parametrize("eps,scale", [(1e-4, 1.0), (0.05, 0.5)])
def test_sigma1_d32_tensor_path(kg, B, H, T, dv, eps, scale):
    """KATA-Sigma_1 at d = 32 (eps I + s u u^T, 528 features): s^2 times the full
    map's (q . k)^2 on the d = 32 tensor path, plus eps s (|q|^2 + |k|^2) + eps^2 m
    as a linear attention (m = 32)."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T, d=32, dv=dv)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, 2, 1) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 2, 1, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "Sigma", 1, eps, scale)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


@pytest.mark.parametrize("B,H,T", [
    (1, 2, 1100),    # 8 CTAs: each head's chunks in order, ragged tail
    (4, 10, 700),    # 160 CTAs, ragged tail
    (2, 3, 129),     # last chunk holds one token
    (3, 1, 5),       # a single partial chunk
])
@pytest.mark.parametrize("eps,scale", [
    (1e-4, 1.0),     # the Sigma configuration
    (0.5, 0.25),     # eps terms of the size of the s^2 (q . k)^2 term
    (3.0, 1.0),      # eps terms dominant
])
def test_sigma1_d64_tensor_path(kg, B, H, T, eps, scale):
    """KATA-Sigma_1 at d = 64 (eps I + s u u^T, 2080 features): s^2 times the full
    map on the d = 64 tensor path (four feature groups' fp32 numerators and one
    denominator), plus the eps terms as a linear attention (m = 64)."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, 2, 1) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 2, 1, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "Sigma", 1, eps, scale)
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]


def test_sigma1_d64_eps_only_rows(kg):
    """Zero queries: <psi(0), psi(k)> = eps^2 m + eps s |k|^2, so those rows come
    from the eps terms alone; with eps = 0 the map is s^2 (q . k)^2 and the scale
    cancels, leaving the plain forward."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=2, T=300)
    q, k, v = workloads.make_qkv(w)
    q[:, :, ::3] = 0
    for eps, scale in ((1e-4, 1.0), (0.5, 0.25)):
        out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, 2, 1, eps, scale)
        torch.cuda.synchronize()
        ref = oracle.forward_map(to_f64(q), to_f64(k), to_f64(v), "Sigma", 1, eps, scale)
        assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype], (eps, scale)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_chunked_map(q, k, v, w.C, 2, 1, 0.0, 0.5)
    b = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert slice_rel_err(to_f64(a), to_f64(b)) <= 1e-2


@pytest.mark.parametrize("map_,g,B,H,path", [
    (1, 2, 1, 32767, "tc"),      # M_2: 65534 sub-heads along grid.y
    (2, 2, 1, 16383, "tc"),      # Sigma_2: 65532 crosswise sub-heads
    (2, 2, 1, 16384, "simt"),    # one head more would pass grid.y: the CUDA cores
    (1, 4, 1, 16384, "simt"),
    (2, 1, 3, 21845, "tc"),      # Sigma_1 on the d = 64 path: 65535 heads
])
def test_map_head_count_limits(kg, map_, g, B, H, path):
    """The sub-head routes launch nsub sub-heads per head along grid.y (at most
    65535); past that the map takes the CUDA cores.  T = 3, sampled heads
    against the oracle."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=3)
    want = kg.KATA_PATH_TC if path == "tc" else kg.KATA_PATH_SIMT
    assert kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, map_, g) == want
    q, k, v = workloads.make_qkv(w)
    eps, scale = (0.5, 0.25) if map_ == 2 else (0.0, 1.0)
    out = kg.kata_fwd_chunked_map(q.cuda(), k.cuda(), v.cuda(), w.C, map_, g, eps, scale)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    for b, h in [(0, 0), (B - 1, H - 1), (0, H // 2)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.forward_map(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), NAMES[map_], g, eps,
                                 scale)
        assert slice_rel_err(to_f64(out[sl]), ref) <= TOL[w.dtype], (b, h)
