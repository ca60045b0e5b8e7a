"""The allocation-free forward entry point, kata_fwd_chunked_noalloc.

It exists for callers that cannot allocate device memory where they run the
forward (framework-owned memory pools, hosts that must not allocate after
start-up, replays of pre-recorded GPU work); its scratch is a fixed 32 MiB
device array inside the library.  These tests call it through the C ABI and
check it against kata_fwd_chunked on two calls in a row, so a second call
that reuses the array's leftover contents is covered.  This file is collected
last so that a failing run stopped at the first failure has run every other
test first; it also passes when run alone in a fresh process.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import workloads
from parity_util import TOL, require_gpu, slice_rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kg():
    return require_gpu()


def _noalloc_raw(kg, q, k, v, out, C):
    """Direct C-ABI call (no binding logic besides pointers)."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    dt = kg.KATA_BF16 if q.dtype == torch.bfloat16 else kg.KATA_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return kg.lib().kata_fwd_chunked_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             out.data_ptr(), B, H, T, d, dv, C, dt, stream)


@pytest.mark.parametrize("name,overrides", [
    ("long_ctx_bf16", dict(B=1, H=4, T=2000)),     # tensor-core path, 16 segments
    ("mid_bf16", dict(B=2, H=8, T=1500)),          # tensor-core path, C = 64
    ("lm_layer_bf16", dict(B=1, H=38, T=300)),     # d = 64 tensor path (state over 4 CTAs)
    ("lm_layer_bf16", dict(B=1, H=64, T=256)),     # d = 64 tensor path, ~17 MB of scratch
    ("small_fp32", dict()),                        # CUDA-core fp32 path
    ("mid_bf16", dict(B=1, H=4, T=1000, d=16, dv=128)),   # padded q, k; two v parts
])
def test_noalloc_matches_allocating_forward_twice(kg, name, overrides):
    w = workloads.WORKLOADS[name].scaled(**overrides)
    assert kg.kata_fwd_workspace_size(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) <= \
        kg.KATA_NOALLOC_SCRATCH_BYTES
    if w.dtype == torch.bfloat16:   # the same kernel family as the allocating call
        assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    q1, k1, v1 = (t.cuda() for t in workloads.make_qkv(w))
    # a second, different batch: its call must not depend on what the first left behind
    q2, k2, v2 = (t.cuda() for t in workloads.make_qkv(w.scaled(index=w.index + 10)))
    for q, k, v in ((q1, k1, v1), (q2, k2, v2)):
        ref = kg.kata_fwd_chunked(q, k, v, w.C)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_raw(kg, q, k, v, out, w.C) == kg.KATA_OK
        torch.cuda.synchronize()
        assert kg.kata_sync_status() == kg.KATA_OK
        assert torch.isfinite(out).all()
        err = slice_rel_err(to_f64(out), to_f64(ref))
        assert err <= TOL[w.dtype], err


def test_noalloc_rejects_oversized_scratch(kg):
    # fp32 chunk states of 64 heads x 64 chunks x 136 x 17 floats exceed 32 MiB
    w = workloads.WORKLOADS["small_fp32"].scaled(B=8, H=8, T=2048)
    assert kg.kata_fwd_workspace_size(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) > \
        kg.KATA_NOALLOC_SCRATCH_BYTES
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    out = torch.zeros(w.B, w.H, w.T, w.dv, device="cuda")
    assert _noalloc_raw(kg, q, k, v, out, w.C) == kg.KATA_ERR_SCRATCH_LIMIT
    assert "scratch" in kg.kata_status_str(kg.KATA_ERR_SCRATCH_LIMIT)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_noalloc_rejects_oversized_d64_tensor_path(kg):
    # the d = 64 tensor path keeps ~1 KB of fp32 partials per token and head:
    # 64 heads x 1024 tokens need ~67 MB, more than the 32 MiB array
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=64, T=1024)
    assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    assert kg.kata_fwd_workspace_size(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) > \
        kg.KATA_NOALLOC_SCRATCH_BYTES
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    out = torch.zeros(w.B, w.H, w.T, w.dv, device="cuda", dtype=torch.bfloat16)
    assert _noalloc_raw(kg, q, k, v, out, w.C) == kg.KATA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(out == 0)
