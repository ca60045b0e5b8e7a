"""Out-of-range writes, caught without a sanitizer: every path writes its output
into the middle of a buffer whose guard regions hold a byte pattern, and the
inputs are compared byte for byte before and after the call.  A kernel that
stored past either end of its output, or into an input, changes them."""
from __future__ import annotations

import pytest
import torch

import workloads
from parity_util import require_gpu

pytestmark = pytest.mark.gpu

GUARD = 4096   # bytes on each side (a multiple of 16, so the output stays aligned)
PATTERN = 0x5A


@pytest.fixture(scope="module")
def kg():
    return require_gpu()


def _guarded(shape, dtype):
    """(full byte buffer, output view in its middle)."""
    es = torch.tensor([], dtype=dtype).element_size()
    n = 1
    for x in shape:
        n *= x
    buf = torch.full((2 * GUARD + n * es,), PATTERN, dtype=torch.uint8, device="cuda")
    out = buf[GUARD:GUARD + n * es].view(dtype).view(*shape)
    return buf, out


def _check(buf, inputs, before):
    torch.cuda.synchronize()
    assert bool((buf[:GUARD] == PATTERN).all()), "write below the output"
    assert bool((buf[-GUARD:] == PATTERN).all()), "write past the output"
    for t, b in zip(inputs, before):
        assert torch.equal(t, b), "an input changed"


def _fwd_case(kg, w, call):
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    ins = [q, k, v]
    before = [t.clone() for t in ins]
    buf, out = _guarded((w.B, w.H, w.T, w.dv), w.dtype)
    call(q, k, v, out)
    _check(buf, ins, before)
    assert torch.isfinite(out.float()).all()
    assert kg.kata_sync_status() == kg.KATA_OK


@pytest.mark.parametrize("name,overrides", [
    ("long_ctx_bf16", dict(B=1, H=2, T=1100)),   # d = 32 tensor path, nine segments
    ("long_ctx_bf16", dict(B=2, H=3, T=129)),    # one-token last chunk
    ("lm_layer_bf16", dict(B=2, H=19, T=300)),   # d = 64 tensor path
    ("small_fp32", dict(B=2, H=3, T=97)),        # CUDA cores
    ("mid_bf16", dict(B=1, H=2, T=77, dv=128)),  # tensor path, two v parts
    ("mid_bf16", dict(B=1, H=3, T=130, d=16, dv=16)),   # q, k padded to d = 32
    ("lm_layer_bf16", dict(B=1, H=38, T=129, dv=32)),   # d = 64 kernels, one v part
    ("lm_layer_bf16", dict(B=1, H=37, T=100, dv=128)),  # d = 64 kernels, 37 heads, two v parts
    ("small_fp32", dict(B=2, H=3, T=97, d=64, dv=128)),  # CUDA cores, fp32
])
def test_chunked_forward_stays_in_bounds(kg, name, overrides):
    w = workloads.WORKLOADS[name].scaled(**overrides)
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_chunked(q, k, v, w.C, out=out))


@pytest.mark.parametrize("map_,g,d", [(1, 2, 64), (2, 2, 64), (1, 4, 64), (2, 4, 64), (1, 4, 32),
                                      (1, 2, 32), (2, 1, 32), (3, 1, 16)])
def test_map_sub_heads_stay_in_bounds(kg, map_, g, d):
    """Sub-head routes at d = 64 and the explicit-feature path (Sigma_4, M_4 at
    d = 32, the orthant map)."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=3, T=333, d=d)
    eps, scale = ((1e-4, 1.0) if map_ == kg.KATA_MAP_SUM else (1e-6, 1.0) if map_ == 3
                  else (0.0, 1.0))
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_chunked_map(q, k, v, w.C, map_, g, eps,
                                                                  scale, out=out))


@pytest.mark.parametrize("d,T", [(32, 1100), (32, 129), (64, 300)])
def test_gated_and_quadratic_stay_in_bounds(kg, d, T):
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=3, T=T, d=d, C=64)
    gate = workloads.make_gate(w, device="cuda")
    g_before = gate.clone()
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_chunked_gated(q, k, v, gate, w.C, out=out))
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_quadratic(q, k, v, out=out))
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_quadratic_gated(q, k, v, gate, out=out))
    assert torch.equal(gate, g_before)


@pytest.mark.parametrize("d,dv,T", [(16, 128, 300), (32, 16, 1100), (64, 32, 129)])
def test_adapted_gated_and_quadratic_stay_in_bounds(kg, d, dv, T):
    """Other bf16 head sizes (padded q, k; 64-column parts of v) in the gated
    chunked and both quadratic forms."""
    w = workloads.WORKLOADS["mid_bf16"].scaled(B=1, H=3, T=T, d=d, dv=dv, C=64)
    gate = workloads.make_gate(w, device="cuda")
    g_before = gate.clone()
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_chunked_gated(q, k, v, gate, w.C, out=out))
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_quadratic(q, k, v, out=out))
    _fwd_case(kg, w, lambda q, k, v, out: kg.kata_fwd_quadratic_gated(q, k, v, gate, out=out))
    assert torch.equal(gate, g_before)


def test_decode_stays_in_bounds(kg):
    w = workloads.DECODE.scaled(B=4, H=3)
    q, k, v = (t.cuda() for t in workloads.make_decode_inputs(w))
    S, z = (t.cuda() for t in workloads.make_decode_state_fill(w))
    ins = [q, k, v]
    before = [t.clone() for t in ins]
    buf, out = _guarded((w.B, w.H, w.dv), w.dtype)
    kg.kata_decode_step(S, z, q, k, v, out=out)
    _check(buf, ins, before)
    assert torch.isfinite(out.float()).all()
