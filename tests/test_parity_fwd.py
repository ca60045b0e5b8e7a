"""GPU forward parity: libkata's kata_fwd_chunked against the CPU oracle.

Element by element at sizes the oracle finishes in seconds (several chunks and a
ragged tail), and on sampled rows at the workloads' full sizes in the same call
configuration the benchmark times.  Inputs come from workloads.py; the oracle
reads exactly the stored (bf16-rounded) values."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import TOL, elem_rel_err, require_gpu, slice_rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kg():
    return require_gpu()


def _run(kg, q, k, v, C):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out = kg.kata_fwd_chunked(qd, kd, vd, C)
    torch.cuda.synchronize()
    return out


def _check_full(kg, q, k, v, C, tol=None):
    out = _run(kg, q, k, v, C)
    ref = oracle.forward(to_f64(q), to_f64(k), to_f64(v))
    err = slice_rel_err(to_f64(out), ref)
    tol = TOL[q.dtype] if tol is None else tol
    assert err <= tol, (f"max relative error {err:.3e} > {tol:.1e} "
                        f"(element-wise {elem_rel_err(to_f64(out), ref):.3e})")
    assert torch.isfinite(out).all()
    return err


def test_small_fp32_workload_full(kg):
    w = workloads.WORKLOADS["small_fp32"]
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, w.C)


@pytest.mark.parametrize("name,overrides", [
    ("mid_bf16", dict(B=2, H=2, T=517)),
    ("recall_bf16", dict(B=2, H=2, T=700)),
    ("lm_layer_bf16", dict(B=1, H=3, T=333)),
    ("long_ctx_bf16", dict(B=1, H=2, T=1100)),
    ("small_fp32", dict(B=2, H=3, T=300)),
])
def test_workload_recipes_scaled(kg, name, overrides):
    w = workloads.WORKLOADS[name].scaled(**overrides)
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, w.C)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("C", [32, 64, 128])
def test_ragged_lengths(kg, dtype, C):
    for T in (1, C - 1, C, C + 1, 3 * C + 5):
        w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=2, T=T, dtype=dtype, C=C)
        q, k, v = workloads.make_qkv(w)
        _check_full(kg, q, k, v, C)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("dv", [16, 32, 64, 128])
def test_head_dims(kg, dtype, d, dv):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=2, T=200, d=d, dv=dv, dtype=dtype, C=64)
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, 64)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zero_denominator_rows_are_zero(kg, dtype):
    # queries along e_0, the first 70 keys along e_1: rows t < 70 have D_t = 0
    B, H, T, d, dv = 1, 1, 150, 32, 64
    q = torch.zeros(B, H, T, d)
    k = torch.zeros(B, H, T, d)
    q[..., 0] = 1.0
    k[..., :70, 1] = 1.0
    k[..., 70:, 0] = 1.0
    v = torch.randn(B, H, T, dv, generator=torch.Generator().manual_seed(5))
    q, k, v = (t.to(dtype) for t in (q, k, v))
    out = _run(kg, q, k, v, 64).float().cpu()
    assert torch.all(out[..., :70, :] == 0)
    ref = oracle.forward(to_f64(q), to_f64(k), to_f64(v))
    assert slice_rel_err(out.numpy().astype(np.float64), ref) <= TOL[dtype]


def test_deterministic(kg):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=2, H=2, T=1000)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_chunked(q, k, v, w.C)
    b = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def _seam_rows(kg, w):
    """Rows where the tensor path changes hands: the first and last rows of
    every segment (the first rows after a seam start from the scanned prefix
    state) and of the first and last 128-token chunks it walks."""
    nseg, seg_tokens = kg.kata_fwd_segments(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype)
    rows = []
    for g in range(1, nseg):
        s0 = g * seg_tokens
        rows += [s0 - 2, s0 - 1, s0, s0 + 1, s0 + 127, s0 + 128]
    for c in (128, 256, w.T - w.T % 128):
        rows += [c - 1, c, c + 1]
    return [t for t in rows if 0 <= t < w.T]


def _sample_rows(w, heads, rng, per_head=24, extra=()):
    T, C = w.T, w.C
    fixed = [0, 1, C - 1, C, C + 1, 2 * C - 1, T // 2, T - 2, T - 1] + list(extra)
    rows = []
    for h in heads:
        ts = sorted(set([t for t in fixed if 0 <= t < T] +
                        rng.integers(0, T, size=per_head).tolist()))
        rows.append(ts)
    return rows


@pytest.mark.parametrize("name", ["small_fp32", "mid_bf16", "recall_bf16", "lm_layer_bf16",
                                  "long_ctx_bf16"])
def test_full_size_sampled_rows(kg, name):
    """Full workload size, the exact call the benchmark times, checked on
    sampled rows computed one by one by the oracle."""
    _sampled_check(kg, workloads.WORKLOADS[name], name)


def _sampled_check(kg, w, name):
    q, k, v = workloads.make_qkv(w, device="cuda")
    out = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(w.index)
    BH = w.B * w.H
    heads = sorted(set([0, BH - 1] + rng.integers(0, BH, size=2).tolist()))
    # copy only the sampled heads to the host for the oracle
    qf = q.reshape(BH, 1, w.T, w.d)[heads]
    kf = k.reshape(BH, 1, w.T, w.d)[heads]
    vf = v.reshape(BH, 1, w.T, w.dv)[heads]
    of = out.reshape(BH, w.T, w.dv)[heads]
    seams = _seam_rows(kg, w)
    rows = _sample_rows(w, heads, rng, extra=seams)
    worst = worst_elem = 0.0
    for hi, ts in enumerate(rows):
        flat = np.array(ts, dtype=np.int64)
        ref = oracle.forward_rows(to_f64(qf[hi:hi + 1]), to_f64(kf[hi:hi + 1]),
                                  to_f64(vf[hi:hi + 1]), flat)
        got = to_f64(of[hi][flat])
        worst = max(worst, slice_rel_err(got, ref))
        worst_elem = max(worst_elem, elem_rel_err(got, ref))
    print(f"{name}: {len(seams)} seam rows, slice metric {worst:.3e}, element-wise {worst_elem:.3e}")
    assert worst <= TOL[w.dtype], f"{name}: {worst:.3e} (element-wise {worst_elem:.3e})"


def test_long_context_dense_sampled_rows(kg):
    """The long-context configuration (B=1, H=16, T=131072, d=32, dv=64, C=128) on
    a dense row sample: for the first and the last head, the first and last 256
    rows, the last row of every 8th chunk and both sides of every segment seam;
    64 random rows of four more heads.  About 1500 rows, each computed by the
    oracle's direct O(T) sum."""
    w = workloads.WORKLOADS["long_ctx_bf16"]
    q, k, v = workloads.make_qkv(w, device="cuda")
    out = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    BH, T = w.B * w.H, w.T
    seams = _seam_rows(kg, w)
    dense = sorted(set(list(range(256)) + list(range(T - 256, T)) +
                   list(range(127, T, 8 * 128)) + seams))
    rng = np.random.default_rng(11)
    plan = {0: dense, BH - 1: dense}
    for h in (3, 6, 9, 12):
        plan[h] = sorted(set(rng.integers(0, T, size=64).tolist()))
    worst = worst_elem = 0.0
    nrows = 0
    for h, ts in plan.items():
        flat = np.array(ts, dtype=np.int64)
        ref = oracle.forward_rows(to_f64(q.reshape(BH, 1, T, w.d)[h:h + 1]),
                                  to_f64(k.reshape(BH, 1, T, w.d)[h:h + 1]),
                                  to_f64(v.reshape(BH, 1, T, w.dv)[h:h + 1]), flat)
        got = to_f64(out.reshape(BH, T, w.dv)[h][flat])
        worst = max(worst, slice_rel_err(got, ref))
        worst_elem = max(worst_elem, elem_rel_err(got, ref))
        nrows += len(ts)
    print(f"long context: {nrows} rows, slice metric {worst:.3e}, element-wise {worst_elem:.3e}")
    assert nrows > 1400
    assert worst <= TOL[w.dtype], f"{worst:.3e} (element-wise {worst_elem:.3e})"


# Segmentations (one-CTA output kernel: G = min(152 // BH, chunks) segments per
# head, segment sums from m = 152 // ((G - 1) BH) pieces per segment)
_SEGMENTATIONS = [
    (1, 2, 1100),    # nine one-chunk segments per head
    (16, 8, 700),    # 128 heads: a single segment of 6 chunks per head
    (8, 8, 1000),    # 64 heads: 2 segments of 4 chunks, ragged tail
    (4, 15, 1000),   # 60 heads: 2 segments of 4 chunks, sums from 2 pieces of 2 chunks
    (4, 8, 4096),    # 32 heads: 4 segments of 8 chunks
    (1, 4, 5000),    # 4 heads: 20 segments of 2 chunks, 2 one-chunk pieces each
    (1, 1, 129),     # 1 head: 2 chunks, second has one token
    (3, 1, 5),       # a single partial chunk
]


def _segments(BH, T, span, sms=152):
    """(segments per head, tokens per segment) when `span` CTAs take a segment."""
    chunks = -(-T // 128)
    lc = -(-chunks // max(1, min(chunks, sms // (span * BH))))
    return -(-chunks // lc), 128 * lc


@pytest.mark.parametrize("B,H,T", _SEGMENTATIONS)
def test_tensor_path_segmentation(kg, B, H, T):
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert kg.kata_fwd_segments(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == _segments(B * H, T, 1)
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, w.C)
    assert kg.kata_sync_status() == kg.KATA_OK


@pytest.mark.parametrize("B,H,T", _SEGMENTATIONS)
def test_tensor_path_pair_output(kg, B, H, T, monkeypatch):
    """The CTA-pair output kernel (feature blocks split over two SMs, partial
    numerators exchanged through distributed shared memory), selected by
    KATA_TC_OUTPUT=pair; it halves the segment count per head."""
    monkeypatch.setenv("KATA_TC_OUTPUT", "pair")
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=B, H=H, T=T)
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, w.C)
    assert kg.kata_sync_status() == kg.KATA_OK
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert kg.kata_fwd_segments(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == _segments(B * H, T, 2)


@pytest.mark.parametrize("B,H,T", [
    (1, 38, 300),    # 38 heads: the fewest that fill 152 SMs with four CTAs each; ragged tail
    (2, 19, 129),    # last chunk holds one token
    (4, 10, 5),      # a single partial chunk
    (8, 16, 640),    # the layer's 128 heads, five whole chunks
])
def test_d64_tensor_path(kg, B, H, T):
    """d = 64: the state (17 feature blocks) split over four CTAs per head,
    partial numerators summed in a separate pass."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T)
    assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, w.C)
    assert kg.kata_sync_status() == kg.KATA_OK


# bf16 shapes outside the tensor kernels' own (d = 16, or dv != 64): q and k
# padded with zero columns to d = 32, v cut into 64-column parts, each part one
# forward on the kernels (exact: the padding adds zero features, and output
# columns depend on their own v column only).
_ADAPTED = [
    (16, 16, 1, 2, 1100),    # nine one-chunk segments per head
    (16, 64, 2, 3, 129),     # last chunk holds one token
    (16, 128, 1, 2, 700),    # two v parts
    (16, 32, 3, 1, 5),       # a single partial chunk
    (32, 16, 1, 2, 1100),
    (32, 32, 2, 2, 517),
    (32, 128, 1, 3, 1100),
    (64, 16, 1, 38, 300),    # the d = 64 kernels
    (64, 32, 1, 2, 300),     # two heads: SMs left idle
    (64, 32, 2, 19, 129),
    (64, 128, 1, 38, 300),
]


@pytest.mark.parametrize("d,dv,B,H,T", _ADAPTED)
def test_adapted_shapes_take_the_tensor_path(kg, d, dv, B, H, T):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=B, H=H, T=T, d=d, dv=dv, C=64)
    assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, w.C)
    assert kg.kata_sync_status() == kg.KATA_OK
    if d < 64 and torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert kg.kata_fwd_segments(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == _segments(B * H, T, 1)


@pytest.mark.parametrize("d,dv", [(16, 128), (32, 16)])
def test_adapted_shapes_long_context_sampled_rows(kg, d, dv):
    """The long-context shape (B=1, H=16, T=131072) at the other head sizes,
    on sampled rows (segment seams included)."""
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(d=d, dv=dv)
    assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    _sampled_check(kg, w, f"long_ctx d={d} dv={dv}")


def test_adapted_shapes_deterministic(kg):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=3, T=1100, d=16, dv=128)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_chunked(q, k, v, w.C)
    b = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,T,dv", [(1, 37, 200, 64), (1, 1, 1100, 64), (1, 3, 300, 128),
                                      (2, 1, 129, 32)])
def test_d64_few_heads_tensor_path(kg, B, H, T, dv):
    """Fewer than 38 heads at d = 64: the four CTAs per head leave SMs idle but
    still outpace the CUDA cores; every head's chunks run in order."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=B, H=H, T=T, dv=dv)
    assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    q, k, v = workloads.make_qkv(w)
    _check_full(kg, q, k, v, w.C)
    assert kg.kata_sync_status() == kg.KATA_OK


@pytest.mark.parametrize("B,H,T,form", [(1, 1, 65536, "quadratic"), (1, 16, 16384, "quadratic"),
                                        (1, 16, 32768, "chunked"), (8, 16, 16384, "chunked")])
def test_d64_form_follows_the_head_count(kg, B, H, T, form):
    """At d = 64 the quadratic form is taken while B H T < 420000 x the waves of
    four CTAs per head (the chunked kernels walk a head's chunks in order)."""
    want = kg.KATA_FORM_QUADRATIC if form == "quadratic" else kg.KATA_FORM_CHUNKED
    assert kg.kata_fwd_form(B, H, T, 64, 64, 64, torch.bfloat16) == want


def test_d64_tensor_path_deterministic(kg):
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=2, H=19, T=700)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    a = kg.kata_fwd_chunked(q, k, v, w.C)
    b = kg.kata_fwd_chunked(q, k, v, w.C)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["long_ctx_bf16", "lm_layer_bf16", "small_fp32"])
def test_host_entry_point(kg, name):
    """kata_fwd_chunked_host (host buffers; large transfers pipelined over groups of
    heads): sampled rows against the oracle and the whole output against the
    device entry point within the tolerance (a head group may be segmented
    differently from the whole call, which changes only the rounding)."""
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    out = kg.kata_fwd_chunked_host(qh, kh, vh, w.C)
    dev = kg.kata_fwd_chunked(q.cuda(), k.cuda(), v.cuda(), w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    assert torch.isfinite(out).all()
    assert slice_rel_err(to_f64(out), to_f64(dev)) <= TOL[w.dtype]
    BH = w.B * w.H
    rng = np.random.default_rng(5)
    worst = 0.0
    for h in sorted(set([0, BH - 1])):
        b, hh = divmod(h, w.H)
        ts = np.array(sorted(set([0, w.T // 2, w.T - 1] + rng.integers(0, w.T, size=5).tolist())),
                      dtype=np.int64)
        sl = (slice(b, b + 1), slice(hh, hh + 1))
        ref = oracle.forward_rows(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), ts)
        worst = max(worst, slice_rel_err(to_f64(out[b, hh])[ts], ref))
    assert worst <= TOL[w.dtype], f"{worst:.3e}"


@pytest.mark.parametrize("form", ["simt_fp32", "tc_bf16", "quadratic", "gated", "tc64_bf16",
                                  "sigma4_features", "d16_dv128"])
def test_maximum_head_count(kg, form):
    """B * H = 65535 (the grid limit every path checks) at T = 3: one partial chunk
    per head.  Sampled heads against the oracle."""
    if form == "simt_fp32":
        w = workloads.WORKLOADS["small_fp32"].scaled(B=3, H=21845, T=3)
    elif form in ("tc64_bf16", "sigma4_features"):
        w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=3, H=21845, T=3)
    elif form == "d16_dv128":
        w = workloads.WORKLOADS["mid_bf16"].scaled(B=3, H=21845, T=3, d=16, dv=128)
    else:
        w = workloads.WORKLOADS["mid_bf16"].scaled(B=3, H=21845, T=3)
    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    g = None
    if form == "quadratic":
        out = kg.kata_fwd_quadratic(qd, kd, vd)
    elif form == "gated":
        g = workloads.make_gate(w)
        out = kg.kata_fwd_chunked_gated(qd, kd, vd, g.cuda(), w.C)
    elif form == "sigma4_features":
        out = kg.kata_fwd_chunked_map(qd, kd, vd, w.C, 2, 4, 1e-4, 0.25)
    else:
        out = kg.kata_fwd_chunked(qd, kd, vd, w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    heads = [(0, 0), (1, 12345), (2, w.H - 1)]
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        if g is not None:
            ref = oracle.forward_gated(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), to_f64(g[sl]))
        elif form == "sigma4_features":
            ref = oracle.forward_map(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), "Sigma", 4, 1e-4,
                                     0.25)
        else:
            ref = oracle.forward(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]))
        assert slice_rel_err(to_f64(out[sl]), ref) <= TOL[w.dtype], (form, b, h)


@pytest.mark.parametrize("name,T,form,dims", [("lm_layer_bf16", 700, "quadratic", None),
                                              ("mid_bf16", 4096, "quadratic", None),
                                              ("recall_bf16", 8192, "chunked", None),
                                              ("small_fp32", 256, "chunked", None),
                                              ("mid_bf16", 2000, "quadratic", (16, 128)),
                                              ("lm_layer_bf16", 700, "quadratic", (64, 32)),
                                              ("mid_bf16", 7000, "chunked", (16, 32))])
def test_fwd_picks_the_faster_form(kg, name, T, form, dims):
    """kata_fwd: the quadratic form up to the crossover on the tensor cores, the
    chunked form beyond it and for fp32; sampled rows against the oracle."""
    w = workloads.WORKLOADS[name].scaled(B=1, H=2, T=T)
    if dims is not None:
        w = w.scaled(d=dims[0], dv=dims[1])
    want = kg.KATA_FORM_QUADRATIC if form == "quadratic" else kg.KATA_FORM_CHUNKED
    assert kg.kata_fwd_form(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == want
    q, k, v = workloads.make_qkv(w)
    out = kg.kata_fwd(q.cuda(), k.cuda(), v.cuda(), w.C)
    torch.cuda.synchronize()
    assert kg.kata_sync_status() == kg.KATA_OK
    rows = np.array(sorted(set([0, 1, T // 3, T // 2, T - 1, T + 5, 2 * T - 1])), dtype=np.int64)
    ref = oracle.forward_rows(to_f64(q), to_f64(k), to_f64(v), rows)
    got = to_f64(out).reshape(-1, w.dv)[rows]
    assert slice_rel_err(got, ref) <= TOL[w.dtype]
