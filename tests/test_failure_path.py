"""The bounded-wait failure path of the tensor-core kernels, run once on the GPU.

kata_test_arm_stall makes the next segment-state launch issue no tile loads.
Every wait on those tiles then runs out its bounded limit (a %globaltimer
deadline of about 2 s), the kernel leaves through its abort path (no copy or
MMA in flight, TMEM released) and records the error word that kata_sync_status
reads.  Nothing faults, traps or hangs: the kernel returns normally."""
from __future__ import annotations

import time

import torch

import oracle
import workloads
from parity_util import TOL, require_gpu, slice_rel_err, to_f64

import pytest

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_next_call_is_correct():
    kg = require_gpu()
    # 2 heads, 9 one-chunk segments each: the segment-state kernel runs 16 CTAs
    w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=1, H=2, T=1100)
    assert kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype) == kg.KATA_PATH_TC
    assert kg.kata_fwd_segments(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype)[0] >= 2
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    assert kg.kata_sync_status() == kg.KATA_OK

    kg.kata_test_arm_stall()
    t0 = time.monotonic()
    kg.kata_fwd_chunked(q, k, v, w.C)
    assert kg.kata_sync_status() == kg.KATA_ERR_TIMEOUT
    waited = time.monotonic() - t0
    assert 1.0 < waited < 30.0, waited
    # the error word was cleared by reading it
    assert kg.kata_sync_status() == kg.KATA_OK

    # the context is intact and the next call is correct
    out = kg.kata_fwd_chunked(q, k, v, w.C)
    assert kg.kata_sync_status() == kg.KATA_OK
    ref = oracle.forward(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()))
    assert slice_rel_err(to_f64(out), ref) <= TOL[w.dtype]
    assert torch.isfinite(out).all()
