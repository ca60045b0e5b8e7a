"""C ABI checks that need no GPU: the library builds, loads and exports every
function include/kata.h declares, and host-side argument validation rejects
bad calls before any device work (these calls return before the library
touches the CUDA runtime)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kata.h")


@pytest.fixture(scope="module")
def L():
    from kernelized_causal_linear_gb300 import build
    build.build()
    import kernelized_causal_linear_gb300 as kg
    return kg.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kata_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("kata_fwd_chunked", "kata_decode_step", "kata_feature_dim", "kata_status_str",
                 "kata_lift"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    import kernelized_causal_linear_gb300 as kg
    for name in _declared_functions():
        assert hasattr(L, name), name
    assert set(_declared_functions()) <= set(kg.EXPORTED) | set()


def test_feature_dim_and_status_text(L):
    import kernelized_causal_linear_gb300 as kg
    assert kg.kata_feature_dim(16) == 136
    assert kg.kata_feature_dim(32) == 528
    assert kg.kata_feature_dim(64) == 2080
    assert kg.kata_feature_dim(0) == -1
    for code in (0, -1, -2, -3, -4, -5):
        assert kg.kata_status_str(code) != "unknown status"
    assert kg.kata_status_str(7) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


def _fwd(L, q=FAKE, k=FAKE, v=FAKE, out=FAKE + 0x1000000, B=1, H=1, T=8, d=16, dv=16, C=32,
         dtype=1):
    return L.kata_fwd_chunked(q, k, v, out, B, H, T, d, dv, C, dtype, None)


def test_fwd_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    assert _fwd(L, q=0) == kg.KATA_ERR_ARG
    assert _fwd(L, out=0) == kg.KATA_ERR_ARG
    assert _fwd(L, v=FAKE + 8) == kg.KATA_ERR_ARG              # misaligned
    assert _fwd(L, B=0) == kg.KATA_ERR_ARG
    assert _fwd(L, T=0) == kg.KATA_ERR_ARG
    assert _fwd(L, H=-3) == kg.KATA_ERR_ARG
    assert _fwd(L, dtype=2) == kg.KATA_ERR_ARG
    assert _fwd(L, d=24) == kg.KATA_ERR_UNSUPPORTED
    assert _fwd(L, dv=48) == kg.KATA_ERR_UNSUPPORTED
    assert _fwd(L, C=16) == kg.KATA_ERR_UNSUPPORTED
    assert _fwd(L, B=300, H=300) == kg.KATA_ERR_UNSUPPORTED     # grid limit on B*H
    # out overlapping an input
    assert _fwd(L, out=FAKE + 16) == kg.KATA_ERR_ARG


def test_workspace_and_path_queries_reject_bad_shapes(L):
    import kernelized_causal_linear_gb300 as kg
    n = ctypes.c_size_t(0)
    assert L.kata_fwd_workspace_size(1, 1, 8, 16, 16, 32, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd_workspace_size(1, 1, 8, 20, 16, 32, 1, ctypes.byref(n)) == \
        kg.KATA_ERR_UNSUPPORTED
    assert L.kata_fwd_path(1, 1, 8, 20, 16, 32, 1) == kg.KATA_PATH_NONE
    assert L.kata_fwd_path(0, 1, 8, 16, 16, 32, 1) == kg.KATA_PATH_NONE


def test_host_variant_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    assert L.kata_fwd_chunked_host(0, FAKE, FAKE, FAKE, 1, 1, 8, 16, 16, 32, 1, None) == \
        kg.KATA_ERR_ARG
    assert L.kata_fwd_chunked_host(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 16, 17, 32, 1, None) == \
        kg.KATA_ERR_UNSUPPORTED


def test_decode_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    S, z, q, k, v, o = (FAKE * (i + 1) * 256 for i in range(6))
    assert L.kata_decode_step(0, z, q, k, v, o, 1, 1, 16, 16, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_decode_step(S, z, q, k, v + 4, o, 1, 1, 16, 16, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_decode_step(S, z, q, k, v, o, 0, 1, 16, 16, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_decode_step(S, z, q, k, v, o, 1, 1, 8, 16, 1, None) == kg.KATA_ERR_UNSUPPORTED
    assert L.kata_decode_step(S, z, q, k, v, o, 1, 1, 16, 20, 1, None) == kg.KATA_ERR_UNSUPPORTED
    # z overlapping the state
    assert L.kata_decode_step(S, S + 64, q, k, v, o, 1, 1, 16, 16, 1, None) == kg.KATA_ERR_ARG


def test_lift_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    assert L.kata_lift(0, FAKE, 4, 16, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_lift(FAKE, FAKE * 2, 0, 16, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_lift(FAKE, FAKE * 2, 4, 65, 1, None) == kg.KATA_ERR_UNSUPPORTED
    assert L.kata_lift(FAKE + 2, FAKE * 2, 4, 16, 1, None) == kg.KATA_ERR_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import kernelized_causal_linear_gb300 as kg
    monkeypatch.setattr(kg, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(kg, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        kg.lib()


def test_state_variant_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    q, k, v, o, S, z = (FAKE * (i + 1) * 4096 for i in range(6))

    def st(**kw):
        a = dict(q=q, k=k, v=v, out=o, S=S, z=z, B=1, H=1, T=8, d=16, dv=16, C=32, dtype=1)
        a.update(kw)
        return L.kata_fwd_chunked_state(a["q"], a["k"], a["v"], a["out"], a["S"], a["z"],
                                        a["B"], a["H"], a["T"], a["d"], a["dv"], a["C"],
                                        a["dtype"], None)

    assert st(S=0) == kg.KATA_ERR_ARG
    assert st(z=0) == kg.KATA_ERR_ARG
    assert st(q=0) == kg.KATA_ERR_ARG
    assert st(S=S + 8) == kg.KATA_ERR_ARG                      # misaligned state
    assert st(z=z + 4) == kg.KATA_ERR_ARG                      # misaligned z
    assert st(z=S + 64) == kg.KATA_ERR_ARG                     # z inside the state
    assert st(S=q) == kg.KATA_ERR_ARG                          # state over an input
    assert st(z=o + 16) == kg.KATA_ERR_ARG                     # z over the output
    assert st(d=20) == kg.KATA_ERR_UNSUPPORTED
    assert st(T=0) == kg.KATA_ERR_ARG


def test_map_feature_dims(L):
    import kernelized_causal_linear_gb300 as kg
    assert L.kata_map_feature_dim(kg.KATA_MAP_FULL, 64, 1) == 2080
    assert L.kata_map_feature_dim(kg.KATA_MAP_BLOCK, 64, 2) == 1056     # g m(m+1)/2
    assert L.kata_map_feature_dim(kg.KATA_MAP_BLOCK, 64, 4) == 544
    assert L.kata_map_feature_dim(kg.KATA_MAP_SUM, 64, 2) == 528        # m(m+1)/2
    assert L.kata_map_feature_dim(kg.KATA_MAP_SUM, 32, 4) == 36
    assert L.kata_map_feature_dim(kg.KATA_MAP_FULL, 64, 2) == -1        # full map is g = 1
    assert L.kata_map_feature_dim(kg.KATA_MAP_BLOCK, 16, 3) == -1       # g must divide d, in {1,2,4}
    assert L.kata_map_feature_dim(7, 16, 2) == -1


def test_map_forward_rejects_bad_maps(L):
    import kernelized_causal_linear_gb300 as kg
    q, k, v, o = (FAKE * (i + 1) * 4096 for i in range(4))

    def fm(map_, g, eps=0.0, scale=1.0, **kw):
        a = dict(B=1, H=1, T=8, d=16, dv=16, C=32, dtype=1)
        a.update(kw)
        return L.kata_fwd_chunked_map(q, k, v, o, a["B"], a["H"], a["T"], a["d"], a["dv"],
                                      a["C"], a["dtype"], map_, g, eps, scale, None)

    assert fm(3, 2) == kg.KATA_ERR_ARG                                   # unknown map
    assert fm(kg.KATA_MAP_FULL, 2) == kg.KATA_ERR_ARG                    # full map needs g = 1
    assert fm(kg.KATA_MAP_BLOCK, 3) == kg.KATA_ERR_ARG                   # g in {1, 2, 4}
    assert fm(kg.KATA_MAP_BLOCK, 2, eps=1e-4) == kg.KATA_ERR_ARG         # eps only for Sigma
    assert fm(kg.KATA_MAP_SUM, 2, eps=-1.0) == kg.KATA_ERR_ARG
    assert fm(kg.KATA_MAP_SUM, 2, scale=0.0) == kg.KATA_ERR_ARG
    assert fm(kg.KATA_MAP_SUM, 2, eps=float("nan")) == kg.KATA_ERR_ARG
    assert fm(kg.KATA_MAP_SUM, 4, d=16, T=0) == kg.KATA_ERR_ARG          # shape rules as the forward
    assert L.kata_lift_map(q, o, 4, 16, 1, kg.KATA_MAP_BLOCK, 3, 0.0, 1.0, None) == kg.KATA_ERR_ARG


def test_gated_forward_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    q, k, v, g, o, S, z = (FAKE * (i + 1) * 4096 for i in range(7))

    def fw(**kw):
        a = dict(q=q, k=k, v=v, g=g, out=o, S=0, z=0, B=1, H=1, T=8, d=16, dv=16, C=32,
                 dtype=1, norm=1)
        a.update(kw)
        return L.kata_fwd_chunked_gated(a["q"], a["k"], a["v"], a["g"], a["out"], a["S"] or None,
                                        a["z"] or None, a["B"], a["H"], a["T"], a["d"], a["dv"],
                                        a["C"], a["dtype"], a["norm"], None)

    assert fw(g=0) == kg.KATA_ERR_ARG                          # no gate
    assert fw(q=0) == kg.KATA_ERR_ARG
    assert fw(g=g + 4) == kg.KATA_ERR_ARG                      # misaligned gate
    assert fw(norm=2) == kg.KATA_ERR_ARG
    assert fw(S=S) == kg.KATA_ERR_ARG                          # state without z
    assert fw(z=z) == kg.KATA_ERR_ARG                          # z without state
    assert fw(S=S, z=S + 64) == kg.KATA_ERR_ARG                # z inside the state
    assert fw(S=g, z=z) == kg.KATA_ERR_ARG                     # state over the gate
    assert fw(out=g) == kg.KATA_ERR_ARG                        # output over the gate
    assert fw(d=20) == kg.KATA_ERR_UNSUPPORTED
    assert fw(C=16) == kg.KATA_ERR_UNSUPPORTED
    assert fw(T=0) == kg.KATA_ERR_ARG


def test_gated_decode_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    S, z, q, k, v, g, o = (FAKE * (i + 1) * 256 for i in range(7))

    def dc(**kw):
        a = dict(S=S, z=z, q=q, k=k, v=v, g=g, out=o, B=1, H=1, d=16, dv=16, dtype=1, norm=1)
        a.update(kw)
        return L.kata_decode_step_gated(a["S"], a["z"], a["q"], a["k"], a["v"], a["g"], a["out"],
                                        a["B"], a["H"], a["d"], a["dv"], a["dtype"], a["norm"],
                                        None)

    assert dc(g=0) == kg.KATA_ERR_ARG
    assert dc(g=g + 8) == kg.KATA_ERR_ARG
    assert dc(norm=-1) == kg.KATA_ERR_ARG
    assert dc(g=S + 16) == kg.KATA_ERR_ARG                     # gate inside the state
    assert dc(d=8) == kg.KATA_ERR_UNSUPPORTED
    assert dc(B=0) == kg.KATA_ERR_ARG


def test_gated_quadratic_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    q, k, v, g, o = (FAKE * (i + 1) * 4096 for i in range(5))

    def fq(**kw):
        a = dict(q=q, k=k, v=v, g=g, out=o, B=1, H=1, T=8, d=32, dv=64, dtype=1, norm=1)
        a.update(kw)
        return L.kata_fwd_quadratic_gated(a["q"], a["k"], a["v"], a["g"], a["out"], a["B"],
                                          a["H"], a["T"], a["d"], a["dv"], a["dtype"], a["norm"],
                                          None)

    assert fq(g=0) == kg.KATA_ERR_ARG
    assert fq(g=g + 4) == kg.KATA_ERR_ARG
    assert fq(norm=3) == kg.KATA_ERR_ARG
    assert fq(out=g) == kg.KATA_ERR_ARG                        # output over the gate
    assert fq(T=0) == kg.KATA_ERR_ARG
    assert fq(d=24) == kg.KATA_ERR_UNSUPPORTED


def test_orthant_map_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    assert kg.kata_map_feature_dim(kg.KATA_MAP_ORTHANT, 64, 1) == 64
    assert kg.kata_map_feature_dim(kg.KATA_MAP_ORTHANT, 64, 2) == -1     # one feature per coordinate
    q, k, v, o = (FAKE * (i + 1) * 4096 for i in range(4))
    bad_scale = L.kata_fwd_chunked_map(q, k, v, o, 1, 1, 8, 16, 16, 32, 0, 3, 1,
                                       ctypes.c_float(1e-6), ctypes.c_float(2.0), None)
    bad_eps = L.kata_fwd_chunked_map(q, k, v, o, 1, 1, 8, 16, 16, 32, 0, 3, 1,
                                     ctypes.c_float(-1.0), ctypes.c_float(1.0), None)
    assert bad_scale == kg.KATA_ERR_ARG and bad_eps == kg.KATA_ERR_ARG


def test_fwd_auto_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    q, k, v, o = (FAKE * (i + 1) * 4096 for i in range(4))
    assert L.kata_fwd(0, k, v, o, 1, 1, 8, 32, 64, 64, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd(q, k, v, 0, 1, 1, 8, 32, 64, 64, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd(q, k, v, o, 1, 1, 0, 32, 64, 64, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd(q, k, v, o, 1, 1, 8, 24, 64, 64, 1, None) == kg.KATA_ERR_UNSUPPORTED
    assert L.kata_fwd_form(1, 1, 8, 24, 64, 64, 1) == kg.KATA_FORM_NONE


def test_fwd_gated_auto_rejects_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    q, k, v, o, g = (FAKE * (i + 1) * 4096 for i in range(5))
    assert L.kata_fwd_gated(0, k, v, g, o, 1, 1, 8, 32, 64, 64, 1, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd_gated(q, k, v, 0, o, 1, 1, 8, 32, 64, 64, 1, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd_gated(q, k, v, g, 0, 1, 1, 8, 32, 64, 64, 1, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd_gated(q, k, v, g, o, 1, 1, 0, 32, 64, 64, 1, 1, None) == kg.KATA_ERR_ARG
    assert L.kata_fwd_gated(q, k, v, g, o, 1, 1, 8, 24, 64, 64, 1, 1, None) == kg.KATA_ERR_UNSUPPORTED
    assert L.kata_fwd_gated_form(1, 1, 8, 24, 64, 64, 1) == kg.KATA_FORM_NONE


def test_map_state_and_decode_reject_bad_arguments(L):
    import kernelized_causal_linear_gb300 as kg
    q, k, v, o, S, z = (FAKE * (i + 1) * 4096 for i in range(6))

    def fs(**kw):
        a = dict(q=q, S=S, z=z, B=1, H=1, T=8, d=16, dv=16, C=32, dtype=1,
                 map_=kg.KATA_MAP_SUM, g=2, eps=1e-4, scale=1.0)
        a.update(kw)
        return L.kata_fwd_chunked_map_state(a["q"], k, v, o, a["S"] or None, a["z"] or None,
                                            a["B"], a["H"], a["T"], a["d"], a["dv"], a["C"],
                                            a["dtype"], a["map_"], a["g"], a["eps"], a["scale"],
                                            None)

    assert fs(map_=kg.KATA_MAP_ORTHANT, g=2) == kg.KATA_ERR_ARG   # the orthant map needs g = 1
    assert fs(map_=kg.KATA_MAP_BLOCK, eps=1e-4) == kg.KATA_ERR_ARG
    assert fs(S=0) == kg.KATA_ERR_ARG                              # no state
    assert fs(z=0) == kg.KATA_ERR_ARG
    assert fs(S=S + 4) == kg.KATA_ERR_ARG                          # misaligned state
    assert fs(T=0) == kg.KATA_ERR_ARG                              # shape rules as the forward
    assert fs(d=24, g=4) == kg.KATA_ERR_UNSUPPORTED
    assert fs(z=S + 64) == kg.KATA_ERR_ARG                         # z inside the state

    def dm(**kw):
        a = dict(S=S, q=q, B=1, H=1, d=16, dv=16, dtype=1, map_=kg.KATA_MAP_BLOCK, g=2, eps=0.0,
                 scale=1.0)
        a.update(kw)
        return L.kata_decode_step_map(a["S"] or None, z, a["q"] or None, k, v, o, a["B"], a["H"],
                                      a["d"], a["dv"], a["dtype"], a["map_"], a["g"], a["eps"],
                                      a["scale"], None)

    assert dm(S=0) == kg.KATA_ERR_ARG
    assert dm(q=0) == kg.KATA_ERR_ARG
    assert dm(g=3) == kg.KATA_ERR_ARG
    assert dm(map_=kg.KATA_MAP_SUM, eps=-1.0) == kg.KATA_ERR_ARG
    assert dm(d=20) == kg.KATA_ERR_UNSUPPORTED
    assert dm(dv=48) == kg.KATA_ERR_UNSUPPORTED
    assert dm(B=0) == kg.KATA_ERR_ARG
