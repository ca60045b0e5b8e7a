"""CPU oracle for KATA rank-one PSD causal linear attention.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the CUDA library and its Python
binding never do, and share no code with it.

The arithmetic lives in ``kata_oracle.c`` (plain C, double precision, OpenMP
over independent rows/heads).  This module compiles it with gcc on first use and
marshals numpy arrays.  Every function takes float64 arrays in the layouts

    q, k : [B, H, T, d]      v, out : [B, H, T, dv]
    S    : [B, H, n, dv]     z      : [B, H, n]        n = d(d+1)/2

and follows the paper "Kernelized Linear Attention: Breaking the Capacity Wall
with Symmetric Cones" (KATA): Eq. 2 (normalised linear attention and its additive
recurrence), Sec. 3.1 (rank-one PSD lift), Sec. 4.1 (packed width, Eq. 17-20) and
App. D.2 Algorithm 1 (chunkwise forward).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kata_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkata_oracle.so")

_lib = None
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i = ctypes.c_int
            lib.kata_oracle_feature_dim.argtypes = [i]
            lib.kata_oracle_feature_dim.restype = i
            lib.kata_oracle_set_threads.argtypes = [i]
            lib.kata_oracle_get_threads.restype = i
            lib.kata_oracle_lift.argtypes = [_D, ctypes.c_int64, i, _D]
            lib.kata_oracle_forward.argtypes = [_D, _D, _D, _D, i, i, i, i]
            lib.kata_oracle_forward_rows.argtypes = [_D, _D, _D, _I64, ctypes.c_int64,
                                                     _D, i, i, i, i]
            lib.kata_oracle_recurrent.argtypes = [_D, _D, _D, _D, i, i, i, i]
            lib.kata_oracle_chunked.argtypes = [_D, _D, _D, _D, i, i, i, i, i]
            lib.kata_oracle_prefix_state.argtypes = [_D, _D, _D, _D, i, i, i, i]
            lib.kata_oracle_decode_step.argtypes = [_D, _D, _D, _D, _D, _D, i, i, i]
            dd = ctypes.c_double
            lib.kata_oracle_map_dim.argtypes = [i, i, i]
            lib.kata_oracle_map_dim.restype = i
            lib.kata_oracle_lift_map.argtypes = [_D, ctypes.c_int64, i, i, i, dd, dd, _D]
            lib.kata_oracle_forward_map.argtypes = [_D, _D, _D, _D, i, i, i, i, i, i, dd, dd]
            lib.kata_oracle_forward_rows_map.argtypes = [_D, _D, _D, _I64, ctypes.c_int64, _D,
                                                         i, i, i, i, i, i, dd, dd]
            lib.kata_oracle_recurrent_map.argtypes = [_D, _D, _D, _D, i, i, i, i, i, i, dd, dd]
            lib.kata_oracle_prefix_state_map.argtypes = [_D, _D, _D, _D, i, i, i, i, i, i, dd, dd]
            lib.kata_oracle_decode_step_map.argtypes = [_D, _D, _D, _D, _D, _D, i, i, i, i, i, dd,
                                                        dd]
            lib.kata_oracle_forward_gated.argtypes = [_D, _D, _D, _D, _D, i, i, i, i, i]
            lib.kata_oracle_forward_rows_gated.argtypes = [_D, _D, _D, _D, _I64, ctypes.c_int64,
                                                           _D, i, i, i, i, i]
            lib.kata_oracle_recurrent_gated.argtypes = [_D, _D, _D, _D, _D, i, i, i, i, i]
            lib.kata_oracle_prefix_state_gated.argtypes = [_D, _D, _D, _D, _D, i, i, i, i]
            lib.kata_oracle_decode_step_gated.argtypes = [_D, _D, _D, _D, _D, _D, _D, i, i, i, i]
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def set_threads(n: int) -> None:
    """Number of OpenMP threads the oracle uses (0 = all cores)."""
    _load().kata_oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().kata_oracle_get_threads())


def feature_dim(d: int) -> int:
    """Packed width n = d(d+1)/2 of the rank-one PSD lift (Sec. 4.1)."""
    return int(_load().kata_oracle_feature_dim(int(d)))


def lift(x) -> np.ndarray:
    """Rank-one PSD lift psi(x) = vech(x x^T), sqrt(2) on off-diagonals (Sec. 3.1)."""
    x = _f64(x)
    d = x.shape[-1]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    n = feature_dim(d)
    out = np.empty(x.shape[:-1] + (n,), dtype=np.float64)
    _load().kata_oracle_lift(_p(x), rows, d, _p(out))
    return out


def _dims(q, v):
    B, H, T, d = q.shape
    dv = v.shape[-1]
    return B, H, T, d, dv


def forward(q, k, v) -> np.ndarray:
    """Direct O(T^2) definition: o_t = sum_{s<=t} (q_t.k_s)^2 v_s / sum_{s<=t} (q_t.k_s)^2."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    out = np.empty((B, H, T, dv), dtype=np.float64)
    _load().kata_oracle_forward(_p(q), _p(k), _p(v), _p(out), B * H, T, d, dv)
    return out


def forward_rows(q, k, v, rows) -> np.ndarray:
    """The direct definition at sampled rows; rows are flat (b*H + h)*T + t indices."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.shape[0], dv), dtype=np.float64)
    _load().kata_oracle_forward_rows(_p(q), _p(k), _p(v), rows.ctypes.data_as(_I64),
                                     rows.shape[0], _p(out), B * H, T, d, dv)
    return out


def recurrent(q, k, v) -> np.ndarray:
    """Self-check form: explicit feature-state recurrence of Eq. 2."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    out = np.empty((B, H, T, dv), dtype=np.float64)
    _load().kata_oracle_recurrent(_p(q), _p(k), _p(v), _p(out), B * H, T, d, dv)
    return out


def chunked(q, k, v, C: int) -> np.ndarray:
    """Self-check form: App. D.2 Algorithm 1 with Eq. 17-20 at chunk size C."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    out = np.empty((B, H, T, dv), dtype=np.float64)
    _load().kata_oracle_chunked(_p(q), _p(k), _p(v), _p(out), B * H, T, d, dv, int(C))
    return out


def prefix_state(k, v):
    """(S_T, Z_T) after all T tokens, by the additive recurrence (Eq. 2, App. D.1)."""
    k, v = _f64(k), _f64(v)
    B, H, T, d = k.shape
    dv = v.shape[-1]
    n = feature_dim(d)
    S = np.empty((B, H, n, dv), dtype=np.float64)
    z = np.empty((B, H, n), dtype=np.float64)
    _load().kata_oracle_prefix_state(_p(k), _p(v), _p(S), _p(z), B * H, T, d, dv)
    return S, z


def decode_step(S, z, q, k, v):
    """One recurrent step (App. D.1): returns (S', z', o) without modifying inputs.

    q, k: [B, H, d]; v: [B, H, dv]; S: [B, H, n, dv]; z: [B, H, n]."""
    S = _f64(S).copy()
    z = _f64(z).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, d = q.shape
    dv = v.shape[-1]
    out = np.empty((B, H, dv), dtype=np.float64)
    _load().kata_oracle_decode_step(_p(S), _p(z), _p(q), _p(k), _p(v), _p(out), B * H,
                                    d, dv)
    return S, z, out


# ---------------------------------------------------------------------------
# Reduced PSD families (Sec. 4.1, "two reduced PSD families"): u in R^d cut into
# g blocks u_a of width m = d/g.  map "M": psi(u) = (u_1 u_1^T, ..., u_g u_g^T);
# map "Sigma": psi(u) = eps I + s * sum_a u_a u_a^T (eps and s as the Sigma
# configuration sets them: 1e-4, and 1/4 for Sigma_4); map "full": u u^T; map
# "orthant": psi(u)_i = max(u_i, 0) + eps, one feature per coordinate (the pages'
# linear-state family, eps = 1e-6 in their configuration).
MAPS = {"full": 0, "M": 1, "Sigma": 2, "orthant": 3}


def map_dim(map_name: str, d: int, g: int) -> int:
    """Packed width of the map: d(d+1)/2, g m(m+1)/2 (M_g) or m(m+1)/2 (Sigma_g)."""
    return int(_load().kata_oracle_map_dim(MAPS[map_name], int(d), int(g)))


def lift_map(x, map_name: str, g: int = 1, eps: float = 0.0, scale: float = 1.0) -> np.ndarray:
    """Packed psi(x) under a map: each matrix vech'd with sqrt(2) off the diagonal."""
    x = _f64(x)
    d = x.shape[-1]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    n = map_dim(map_name, d, g)
    out = np.empty(x.shape[:-1] + (n,), dtype=np.float64)
    _load().kata_oracle_lift_map(_p(x), rows, d, MAPS[map_name], int(g), float(eps),
                                 float(scale), _p(out))
    return out


def forward_map(q, k, v, map_name: str, g: int = 1, eps: float = 0.0,
                scale: float = 1.0) -> np.ndarray:
    """Direct O(T^2) definition (Eq. 2) with w_ts = <psi(q_t), psi(k_s)>_F of the map."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    out = np.empty((B, H, T, dv), dtype=np.float64)
    _load().kata_oracle_forward_map(_p(q), _p(k), _p(v), _p(out), B * H, T, d, dv,
                                    MAPS[map_name], int(g), float(eps), float(scale))
    return out


def forward_rows_map(q, k, v, rows, map_name: str, g: int = 1, eps: float = 0.0,
                     scale: float = 1.0) -> np.ndarray:
    """forward_map at sampled rows (flat (b*H + h)*T + t indices)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.shape[0], dv), dtype=np.float64)
    _load().kata_oracle_forward_rows_map(_p(q), _p(k), _p(v), rows.ctypes.data_as(_I64),
                                         rows.shape[0], _p(out), B * H, T, d, dv,
                                         MAPS[map_name], int(g), float(eps), float(scale))
    return out


def recurrent_map(q, k, v, map_name: str, g: int = 1, eps: float = 0.0,
                  scale: float = 1.0) -> np.ndarray:
    """Self-check form: the packed-feature recurrence of Eq. 2 under a map."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    out = np.empty((B, H, T, dv), dtype=np.float64)
    _load().kata_oracle_recurrent_map(_p(q), _p(k), _p(v), _p(out), B * H, T, d, dv,
                                      MAPS[map_name], int(g), float(eps), float(scale))
    return out


def prefix_state_map(k, v, map_name: str, g: int = 1, eps: float = 0.0, scale: float = 1.0):
    """(S_T, Z_T) after all T tokens under a map (Eq. 2's recurrence with the
    map's psi), features in lift_map's packed order."""
    k, v = _f64(k), _f64(v)
    B, H, T, d = k.shape
    dv = v.shape[-1]
    n = map_dim(map_name, d, g)
    S = np.empty((B, H, n, dv), dtype=np.float64)
    z = np.empty((B, H, n), dtype=np.float64)
    _load().kata_oracle_prefix_state_map(_p(k), _p(v), _p(S), _p(z), B * H, T, d, dv,
                                         MAPS[map_name], int(g), float(eps), float(scale))
    return S, z


def decode_step_map(S, z, q, k, v, map_name: str, g: int = 1, eps: float = 0.0,
                    scale: float = 1.0):
    """One decode step under a map: returns (S', z', o) without modifying inputs."""
    S = _f64(S).copy()
    z = _f64(z).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, d = q.shape
    dv = v.shape[-1]
    out = np.empty((B, H, dv), dtype=np.float64)
    _load().kata_oracle_decode_step_map(_p(S), _p(z), _p(q), _p(k), _p(v), _p(out), B * H, d,
                                        dv, MAPS[map_name], int(g), float(eps), float(scale))
    return S, z, out


# ---------------------------------------------------------------------------
# GatedKATA (the appendix on recurrent variants, "multiplicative scalar state
# gate"; Sec. 5.2): S_t = gamma_t S_{t-1} + psi(k_t) v_t^T with gamma_t in [0, 1],
# Z_t gated the same way; readout psi(q)^T S_t / psi(q)^T Z_t (normalize=True) or
# psi(q)^T S_t (normalize=False, the MQAR appendix's no-denominator form).
# gamma: [B, H, T] for the forward, [B, H] for one decode step.


def _gate(gamma, shape) -> np.ndarray:
    g = _f64(gamma)
    if g.shape != tuple(shape):
        raise ValueError(f"gamma must have shape {tuple(shape)}, got {g.shape}")
    return g


def forward_gated(q, k, v, gamma, normalize: bool = True) -> np.ndarray:
    """Direct O(T^2) definition: weights prod_{r=s+1}^{t} gamma_r (q_t.k_s)^2."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    g = _gate(gamma, (B, H, T))
    out = np.empty((B, H, T, dv), dtype=np.float64)
    _load().kata_oracle_forward_gated(_p(q), _p(k), _p(v), _p(g), _p(out), B * H, T, d, dv,
                                      int(bool(normalize)))
    return out


def forward_rows_gated(q, k, v, gamma, rows, normalize: bool = True) -> np.ndarray:
    """The gated direct definition at flat rows (b*H + h)*T + t."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    g = _gate(gamma, (B, H, T))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.shape[0], dv), dtype=np.float64)
    _load().kata_oracle_forward_rows_gated(_p(q), _p(k), _p(v), _p(g), rows.ctypes.data_as(_I64),
                                           rows.shape[0], _p(out), B * H, T, d, dv,
                                           int(bool(normalize)))
    return out


def recurrent_gated(q, k, v, gamma, normalize: bool = True) -> np.ndarray:
    """Self-check form: the gated feature-state recurrence."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d, dv = _dims(q, v)
    g = _gate(gamma, (B, H, T))
    out = np.empty((B, H, T, dv), dtype=np.float64)
    _load().kata_oracle_recurrent_gated(_p(q), _p(k), _p(v), _p(g), _p(out), B * H, T, d, dv,
                                        int(bool(normalize)))
    return out


def prefix_state_gated(k, v, gamma):
    """(S_T, Z_T) after all T tokens under the gated recurrence."""
    k, v = _f64(k), _f64(v)
    B, H, T, d = k.shape
    dv = v.shape[-1]
    g = _gate(gamma, (B, H, T))
    n = feature_dim(d)
    S = np.empty((B, H, n, dv), dtype=np.float64)
    z = np.empty((B, H, n), dtype=np.float64)
    _load().kata_oracle_prefix_state_gated(_p(k), _p(v), _p(g), _p(S), _p(z), B * H, T, d, dv)
    return S, z


def decode_step_gated(S, z, q, k, v, gamma, normalize: bool = True):
    """One gated step: returns (S', z', o) without modifying the inputs."""
    S = _f64(S).copy()
    z = _f64(z).copy()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, d = q.shape
    dv = v.shape[-1]
    g = _gate(gamma, (B, H))
    out = np.empty((B, H, dv), dtype=np.float64)
    _load().kata_oracle_decode_step_gated(_p(S), _p(z), _p(q), _p(k), _p(v), _p(g), _p(out),
                                          B * H, d, dv, int(bool(normalize)))
    return S, z, out
