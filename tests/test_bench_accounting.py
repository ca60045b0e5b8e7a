"""The work accounting bench.py divides by its kernel times (CPU only): the causal
intra-chunk pair count against brute-force enumeration, the map widths against
the oracle's pinned packed widths, the whole-call flops against a count built
from those, and the source digests that key the DRAM-traffic records."""
from __future__ import annotations

import importlib.util
import os

import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _pairs_brute(T, C):
    return sum(1 for t in range(T) for s in range(t + 1) if s // C == t // C)


@pytest.mark.parametrize("T,C", [(1, 32), (31, 32), (32, 32), (33, 32), (300, 64), (1100, 128),
                                 (129, 128), (257, 256)])
def test_intra_pairs_is_the_causal_pair_count(bench, T, C):
    assert bench._intra_pairs(T, C) == _pairs_brute(T, C)
    # the quadratic form counts every causal pair of the head
    assert bench._intra_pairs(T, T) == T * (T + 1) // 2


@pytest.mark.parametrize("name,g,d", [("full", 1, 16), ("full", 1, 64), ("M", 2, 32), ("M", 4, 64),
                                      ("Sigma", 1, 64), ("Sigma", 2, 64), ("Sigma", 4, 32),
                                      ("orthant", 1, 64)])
def test_feature_widths_are_the_oracle_map_widths(bench, name, g, d):
    fm = bench.FeatureMap(name, g)
    ref = oracle.map_dim("M" if name == "full" else name, d, g) if name != "orthant" else d
    assert fm.n(d) == ref


def test_call_flops_at_the_long_context_size(bench):
    """State and inter output 2 n (dv + 1) each per token and head, plus 2 (d + dv + 1)
    per causal in-chunk pair: 149,793 flop per token and head at d = 32, dv = 64,
    C = 128 (T a multiple of C)."""
    w = workloads.WORKLOADS["long_ctx_bf16"]
    n = oracle.map_dim("M", w.d, 1)
    per_token = 4 * n * (w.dv + 1) + 2 * (w.d + w.dv + 1) * (w.C + 1) / 2
    assert per_token == 149793
    assert bench.call_flops(w) == pytest.approx(per_token * w.B * w.H * w.T, rel=1e-12)


def test_call_flops_counts_ragged_chunks_and_the_sigma_weight(bench):
    """A ragged last chunk contributes its own causal pairs; Sigma_g's weight takes
    g d multiply-adds per pair (all g x g block products)."""
    w = workloads.WORKLOADS["lm_layer_bf16"].scaled(B=1, H=2, T=300)
    for name, g in (("full", 1), ("Sigma", 2), ("M", 2)):
        fm = bench.FeatureMap(name, g)
        n = fm.n(w.d)
        wd = g * w.d if name == "Sigma" else w.d
        ref = (4 * n * (w.dv + 1) * w.T + 2 * (wd + w.dv + 1) * _pairs_brute(w.T, w.C)) * w.B * w.H
        assert bench.call_flops(w, fm) == pytest.approx(ref, rel=1e-12)


def test_source_digest_follows_the_stage_sources(bench):
    """A stage's digest covers its own .cu file and the headers it includes: the
    d = 32 output stage and its state stage share kata_tc.cu, the d = 64 stages
    another file."""
    a = bench._source_digest("tc_segment_output")
    assert a == bench._source_digest("tc_segment_state")
    assert a != bench._source_digest("tc64_output")
    assert len(a) == 16 and int(a, 16) >= 0
