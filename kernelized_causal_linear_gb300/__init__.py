"""Python binding of libkata: KATA rank-one PSD causal linear attention on GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of libkata.so, reached through its C ABI (include/kata.h) with ctypes.
PyTorch tensors supply device memory and the current CUDA stream; nothing here
computes.  If libkata.so has not been built, every call raises -- there is no
CPU fallback.

Names follow the C ABI: kata_fwd_chunked, kata_decode_step, kata_lift,
kata_fwd_chunked_host, kata_fwd_workspace_size, kata_fwd_path, kata_fwd_segments,
kata_feature_dim, kata_status_str.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkata.so")

KATA_OK = 0
KATA_ERR_ARG = -1
KATA_ERR_UNSUPPORTED = -2
KATA_ERR_CUDA = -3
KATA_ERR_ALLOC = -4
KATA_ERR_TIMEOUT = -5
KATA_ERR_SCRATCH_LIMIT = -6
KATA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

KATA_F32 = 0
KATA_BF16 = 1

KATA_MAP_FULL = 0
KATA_MAP_BLOCK = 1
KATA_MAP_SUM = 2
KATA_MAP_ORTHANT = 3
KATA_FORM_NONE = 0
KATA_FORM_CHUNKED = 1
KATA_FORM_QUADRATIC = 2

KATA_PATH_NONE = 0
KATA_PATH_SIMT = 1
KATA_PATH_TC = 2

EXPORTED = ("kata_feature_dim", "kata_status_str", "kata_fwd_chunked",
            "kata_fwd_workspace_size", "kata_fwd_path", "kata_fwd_chunked_host",
            "kata_decode_step", "kata_lift", "kata_trace_begin", "kata_trace_end",
            "kata_sync_status", "kata_fwd_chunked_noalloc", "kata_fwd_chunked_state",
            "kata_fwd_chunked_map", "kata_lift_map", "kata_map_feature_dim",
            "kata_fwd_path_map", "kata_fwd_quadratic", "kata_fwd_chunked_gated",
            "kata_decode_step_gated", "kata_fwd_quadratic_gated", "kata_fwd", "kata_fwd_form",
            "kata_fwd_gated", "kata_fwd_gated_form", "kata_fwd_segments",
            "kata_test_arm_stall", "kata_fwd_path_gated", "kata_fwd_chunked_map_state",
            "kata_decode_step_map")

_lib = None


class TraceStage(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


class KataError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_str(status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libkata.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkata.so is not built ({LIB_PATH}); run "
                               "kernelized_causal_linear_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        i, p, vp = ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        L.kata_feature_dim.argtypes = [i]
        L.kata_feature_dim.restype = i
        L.kata_status_str.argtypes = [i]
        L.kata_status_str.restype = ctypes.c_char_p
        L.kata_fwd_chunked.argtypes = [p, p, p, p, i, i, i, i, i, i, i, vp]
        L.kata_fwd_chunked.restype = i
        L.kata_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        L.kata_fwd_workspace_size.restype = i
        L.kata_fwd_path.argtypes = [i, i, i, i, i, i, i]
        L.kata_fwd_path.restype = i
        L.kata_fwd_segments.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
        L.kata_fwd_segments.restype = i
        L.kata_fwd_chunked_host.argtypes = [p, p, p, p, i, i, i, i, i, i, i, vp]
        L.kata_fwd_chunked_host.restype = i
        L.kata_decode_step.argtypes = [p, p, p, p, p, p, i, i, i, i, i, vp]
        L.kata_decode_step.restype = i
        L.kata_lift.argtypes = [p, p, ctypes.c_int64, i, i, vp]
        L.kata_lift.restype = i
        L.kata_fwd_chunked_noalloc.argtypes = [p, p, p, p, i, i, i, i, i, i, i, vp]
        L.kata_fwd_chunked_noalloc.restype = i
        L.kata_fwd_chunked_state.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, vp]
        f = ctypes.c_float
        L.kata_fwd_chunked_map.argtypes = [p, p, p, p, i, i, i, i, i, i, i, i, i, f, f, vp]
        L.kata_fwd_chunked_map_state.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, i, i, f, f,
                                                 vp]
        L.kata_decode_step_map.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, f, f, vp]
        L.kata_lift_map.argtypes = [p, p, ctypes.c_int64, i, i, i, i, f, f, vp]
        L.kata_map_feature_dim.argtypes = [i, i, i]
        L.kata_map_feature_dim.restype = i
        L.kata_fwd_path_map.argtypes = [i, i, i, i, i, i, i, i, i]
        L.kata_fwd_path_map.restype = i
        L.kata_fwd_quadratic.argtypes = [p, p, p, p, i, i, i, i, i, i, vp]
        L.kata_fwd_quadratic.restype = i
        L.kata_fwd_chunked_gated.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, vp]
        L.kata_fwd_chunked_gated.restype = i
        L.kata_decode_step_gated.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, vp]
        L.kata_decode_step_gated.restype = i
        L.kata_fwd_quadratic_gated.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, vp]
        L.kata_fwd_quadratic_gated.restype = i
        L.kata_fwd.argtypes = [p, p, p, p, i, i, i, i, i, i, i, vp]
        L.kata_fwd.restype = i
        L.kata_fwd_form.argtypes = [i, i, i, i, i, i, i]
        L.kata_fwd_form.restype = i
        L.kata_fwd_gated.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, i, vp]
        L.kata_fwd_gated.restype = i
        L.kata_fwd_gated_form.argtypes = [i, i, i, i, i, i, i]
        L.kata_fwd_gated_form.restype = i
        L.kata_fwd_path_gated.argtypes = [i, i, i, i, i, i, i]
        L.kata_fwd_path_gated.restype = i
        L.kata_fwd_chunked_state.restype = i
        L.kata_sync_status.argtypes = [vp]
        L.kata_sync_status.restype = i
        L.kata_test_arm_stall.argtypes = []
        L.kata_test_arm_stall.restype = i
        L.kata_trace_begin.argtypes = []
        L.kata_trace_begin.restype = i
        L.kata_trace_end.argtypes = [ctypes.POINTER(TraceStage), i, ctypes.POINTER(i)]
        L.kata_trace_end.restype = i
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return kata_status_str(status)


def kata_status_str(status: int) -> str:
    return lib().kata_status_str(int(status)).decode()


def kata_feature_dim(d: int) -> int:
    return int(lib().kata_feature_dim(int(d)))


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return KATA_F32
    if t == torch.bfloat16:
        return KATA_BF16
    raise TypeError(f"unsupported dtype {t}")


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str) -> None:
    if rc != KATA_OK:
        raise KataError(rc, where)


def _contig(*ts):
    for t in ts:
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def kata_fwd_chunked(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, C: int,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal KATA forward (chunked O(T) form). q,k: [B,H,T,d]; v: [B,H,T,dv] on CUDA."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    _contig(q, k, v, out)
    rc = lib().kata_fwd_chunked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                B, H, T, d, dv, int(C), _dtype_code(q.dtype),
                                _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_chunked")
    return out


def kata_fwd_chunked_state(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, C: int,
                           out: torch.Tensor | None = None, state: torch.Tensor | None = None,
                           z: torch.Tensor | None = None, stream=None):
    """Forward plus the state after the last token in the decode layout:
    returns (out, state [B,H,n,dv] fp32, z [B,H,n] fp32), ready for
    kata_decode_step to continue the sequence."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    n = d * (d + 1) // 2
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    if state is None:
        state = torch.empty((B, H, n, dv), dtype=torch.float32, device=v.device)
    if z is None:
        z = torch.empty((B, H, n), dtype=torch.float32, device=v.device)
    _contig(q, k, v, out, state, z)
    rc = lib().kata_fwd_chunked_state(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      state.data_ptr(), z.data_ptr(), B, H, T, d, dv, int(C),
                                      _dtype_code(q.dtype), _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_chunked_state")
    return out, state, z


def kata_fwd_chunked_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, C: int,
                             out: torch.Tensor, stream=None) -> torch.Tensor:
    """The forward without any device allocation, for callers that cannot
    allocate where they run it: scratch comes from a fixed 32 MiB device array
    inside the library, shared by all calls (order calls that could overlap).
    `out` must be provided, so this function allocates nothing either."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    _contig(q, k, v, out)
    rc = lib().kata_fwd_chunked_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        out.data_ptr(), B, H, T, d, dv, int(C),
                                        _dtype_code(q.dtype), _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_chunked_noalloc")
    return out


def kata_fwd_chunked_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, C: int,
                          out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Same forward on HOST tensors (pinned for async copies); synchronous."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, pin_memory=True)
    _contig(q, k, v, out)
    rc = lib().kata_fwd_chunked_host(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     out.data_ptr(), B, H, T, d, dv, int(C),
                                     _dtype_code(q.dtype), _stream_handle(stream, None))
    _check(rc, "kata_fwd_chunked_host")
    return out


def kata_fwd_workspace_size(B, H, T, d, dv, C, dtype: torch.dtype) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().kata_fwd_workspace_size(B, H, T, d, dv, C, _dtype_code(dtype),
                                         ctypes.byref(n)), "kata_fwd_workspace_size")
    return int(n.value)


def kata_fwd_path(B, H, T, d, dv, C, dtype: torch.dtype) -> int:
    return int(lib().kata_fwd_path(B, H, T, d, dv, C, _dtype_code(dtype)))


def kata_fwd_segments(B, H, T, d, dv, C, dtype: torch.dtype) -> tuple[int, int]:
    """(segments per head, tokens per segment but the last) of kata_fwd_chunked."""
    tok = ctypes.c_int(0)
    n = int(lib().kata_fwd_segments(B, H, T, d, dv, C, _dtype_code(dtype), ctypes.byref(tok)))
    if n < 0:
        _check(n, "kata_fwd_segments")
    return n, int(tok.value)


def kata_decode_step(state: torch.Tensor, z: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
                     v: torch.Tensor, out: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """One recurrent decode step, state [B,H,n,dv] f32 and z [B,H,n] f32 updated in place."""
    B, H, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, dv), dtype=v.dtype, device=v.device)
    _contig(state, z, q, k, v, out)
    if state.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("state and z must be float32")
    rc = lib().kata_decode_step(state.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(),
                                v.data_ptr(), out.data_ptr(), B, H, d, dv,
                                _dtype_code(q.dtype), _stream_handle(stream, q.device))
    _check(rc, "kata_decode_step")
    return out


def kata_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, C: int,
             out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The forward in whichever exact form is faster for the shape (quadratic for
    short sequences on the tensor cores, else chunked); kata_fwd_form tells which."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    _contig(q, k, v, out)
    rc = lib().kata_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, T, d, dv,
                        int(C), _dtype_code(q.dtype), _stream_handle(stream, q.device))
    _check(rc, "kata_fwd")
    return out


def kata_fwd_form(B, H, T, d, dv, C, dtype: torch.dtype) -> int:
    return int(lib().kata_fwd_form(B, H, T, d, dv, C, _dtype_code(dtype)))


def kata_fwd_quadratic(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Quadratic (flash-style) KATA forward. q,k: [B,H,T,d]; v: [B,H,T,dv] on CUDA."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    _contig(q, k, v, out)
    rc = lib().kata_fwd_quadratic(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  B, H, T, d, dv, _dtype_code(q.dtype),
                                  _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_quadratic")
    return out


def kata_fwd_chunked_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                           gamma: torch.Tensor, C: int, normalize: bool = True,
                           out: torch.Tensor | None = None, with_state: bool = False,
                           stream=None):
    """GatedKATA forward: S_t = gamma_t S_{t-1} + psi(k_t) v_t^T (Z_t alike),
    read out as psi(q)^T S / psi(q)^T Z (normalize) or psi(q)^T S.
    gamma: [B,H,T] float32 in [0, 1] on the same device.  Returns out, or
    (out, state [B,H,n,dv], z [B,H,n]) with with_state."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if gamma.dtype != torch.float32 or tuple(gamma.shape) != (B, H, T):
        raise TypeError("gamma must be float32 of shape [B, H, T]")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    state = z = None
    if with_state:
        n = d * (d + 1) // 2
        state = torch.empty((B, H, n, dv), dtype=torch.float32, device=v.device)
        z = torch.empty((B, H, n), dtype=torch.float32, device=v.device)
        _contig(state, z)
    _contig(q, k, v, gamma, out)
    rc = lib().kata_fwd_chunked_gated(q.data_ptr(), k.data_ptr(), v.data_ptr(), gamma.data_ptr(),
                                      out.data_ptr(), state.data_ptr() if with_state else None,
                                      z.data_ptr() if with_state else None, B, H, T, d, dv,
                                      int(C), _dtype_code(q.dtype), int(bool(normalize)),
                                      _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_chunked_gated")
    return (out, state, z) if with_state else out


def kata_fwd_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, gamma: torch.Tensor,
                   C: int, normalize: bool = True, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """GatedKATA in whichever exact form is faster for the shape (the quadratic form
    on the tensor cores up to T = 32768 where supported, else chunked);
    kata_fwd_gated_form tells which.  gamma: [B,H,T] float32."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if gamma.dtype != torch.float32 or tuple(gamma.shape) != (B, H, T):
        raise TypeError("gamma must be float32 of shape [B, H, T]")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    _contig(q, k, v, gamma, out)
    rc = lib().kata_fwd_gated(q.data_ptr(), k.data_ptr(), v.data_ptr(), gamma.data_ptr(),
                              out.data_ptr(), B, H, T, d, dv, int(C), _dtype_code(q.dtype),
                              int(bool(normalize)), _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_gated")
    return out


def kata_fwd_gated_form(B, H, T, d, dv, C, dtype: torch.dtype) -> int:
    return int(lib().kata_fwd_gated_form(B, H, T, d, dv, C, _dtype_code(dtype)))


def kata_fwd_path_gated(B, H, T, d, dv, C, dtype: torch.dtype) -> int:
    """Path kata_fwd_chunked_gated takes for a shape (a KATA_PATH_* value)."""
    return int(lib().kata_fwd_path_gated(B, H, T, d, dv, C, _dtype_code(dtype)))


def kata_fwd_quadratic_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                             gamma: torch.Tensor, normalize: bool = True,
                             out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """GatedKATA in the quadratic form on the tensor cores (bf16, d in {32, 64},
    dv = 64): weights prod_{r=s+1}^{t} gamma_r (q_t.k_s)^2; gamma [B,H,T] float32."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if gamma.dtype != torch.float32 or tuple(gamma.shape) != (B, H, T):
        raise TypeError("gamma must be float32 of shape [B, H, T]")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    _contig(q, k, v, gamma, out)
    rc = lib().kata_fwd_quadratic_gated(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        gamma.data_ptr(), out.data_ptr(), B, H, T, d, dv,
                                        _dtype_code(q.dtype), int(bool(normalize)),
                                        _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_quadratic_gated")
    return out


def kata_decode_step_gated(state: torch.Tensor, z: torch.Tensor, q: torch.Tensor,
                           k: torch.Tensor, v: torch.Tensor, gamma: torch.Tensor,
                           normalize: bool = True, out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """One GatedKATA step (S = gamma S + psi(k) v^T, z = gamma z + psi(k)) in place;
    gamma: [B,H] float32."""
    B, H, d = q.shape
    dv = v.shape[-1]
    if gamma.dtype != torch.float32 or tuple(gamma.shape) != (B, H):
        raise TypeError("gamma must be float32 of shape [B, H]")
    if state.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("state and z must be float32")
    if out is None:
        out = torch.empty((B, H, dv), dtype=v.dtype, device=v.device)
    _contig(state, z, q, k, v, gamma, out)
    rc = lib().kata_decode_step_gated(state.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(),
                                      v.data_ptr(), gamma.data_ptr(), out.data_ptr(), B, H, d, dv,
                                      _dtype_code(q.dtype), int(bool(normalize)),
                                      _stream_handle(stream, q.device))
    _check(rc, "kata_decode_step_gated")
    return out


def kata_fwd_path_map(B, H, T, d, dv, C, dtype, map: int, g: int) -> int:
    """Path kata_fwd_chunked_map takes for a shape and map (a KATA_PATH_* value)."""
    return int(lib().kata_fwd_path_map(B, H, T, d, dv, C, _dtype_code(dtype), int(map), int(g)))


def kata_map_feature_dim(map: int, d: int, g: int) -> int:
    """Packed width of a feature map (-1 if invalid)."""
    return int(lib().kata_map_feature_dim(int(map), int(d), int(g)))


def kata_fwd_chunked_map(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, C: int, map: int,
                         g: int, eps: float = 0.0, scale: float = 1.0,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal KATA forward with a reduced PSD map (KATA_MAP_BLOCK: M_g, KATA_MAP_SUM: Sigma_g)."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    _contig(q, k, v, out)
    rc = lib().kata_fwd_chunked_map(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    B, H, T, d, dv, int(C), _dtype_code(q.dtype), int(map),
                                    int(g), float(eps), float(scale),
                                    _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_chunked_map")
    return out


def kata_fwd_chunked_map_state(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, C: int,
                               map: int, g: int, eps: float = 0.0, scale: float = 1.0,
                               out: torch.Tensor | None = None, state: torch.Tensor | None = None,
                               z: torch.Tensor | None = None, stream=None):
    """kata_fwd_chunked_map plus the map's state after the last token: returns
    (out, state [B,H,n,dv] fp32, z [B,H,n] fp32) for kata_decode_step_map."""
    B, H, T, d = q.shape
    dv = v.shape[-1]
    n = kata_map_feature_dim(map, d, g)
    if n < 0:
        raise KataError(KATA_ERR_ARG, "kata_fwd_chunked_map_state")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=v.dtype, device=v.device)
    if state is None:
        state = torch.empty((B, H, n, dv), dtype=torch.float32, device=v.device)
    if z is None:
        z = torch.empty((B, H, n), dtype=torch.float32, device=v.device)
    _contig(q, k, v, out, state, z)
    rc = lib().kata_fwd_chunked_map_state(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          out.data_ptr(), state.data_ptr(), z.data_ptr(), B, H, T,
                                          d, dv, int(C), _dtype_code(q.dtype), int(map), int(g),
                                          float(eps), float(scale),
                                          _stream_handle(stream, q.device))
    _check(rc, "kata_fwd_chunked_map_state")
    return out, state, z


def kata_decode_step_map(state: torch.Tensor, z: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
                         v: torch.Tensor, map: int, g: int, eps: float = 0.0, scale: float = 1.0,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One decode step under a map; state [B,H,n,dv] and z [B,H,n] (fp32) in place."""
    B, H, d = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, dv), dtype=v.dtype, device=v.device)
    _contig(state, z, q, k, v, out)
    if state.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("state and z must be float32")
    rc = lib().kata_decode_step_map(state.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(),
                                    v.data_ptr(), out.data_ptr(), B, H, d, dv,
                                    _dtype_code(q.dtype), int(map), int(g), float(eps),
                                    float(scale), _stream_handle(stream, q.device))
    _check(rc, "kata_decode_step_map")
    return out


def kata_lift_map(x: torch.Tensor, map: int, g: int, eps: float = 0.0, scale: float = 1.0,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Packed psi(x) of a map for each row of x [..., d] -> fp32 [..., n]."""
    d = x.shape[-1]
    rows = x.numel() // d
    n = kata_map_feature_dim(map, d, g)
    if n < 0:
        raise KataError(KATA_ERR_ARG, "kata_lift_map")
    if out is None:
        out = torch.empty(x.shape[:-1] + (n,), dtype=torch.float32, device=x.device)
    _contig(x, out)
    rc = lib().kata_lift_map(x.data_ptr(), out.data_ptr(), rows, d, _dtype_code(x.dtype),
                             int(map), int(g), float(eps), float(scale),
                             _stream_handle(stream, x.device))
    _check(rc, "kata_lift_map")
    return out


def kata_lift(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """psi(x) for each row of x [..., d] -> fp32 [..., n]."""
    d = x.shape[-1]
    rows = x.numel() // d
    n = d * (d + 1) // 2
    if out is None:
        out = torch.empty(x.shape[:-1] + (n,), dtype=torch.float32, device=x.device)
    _contig(x, out)
    rc = lib().kata_lift(x.data_ptr(), out.data_ptr(), rows, d, _dtype_code(x.dtype),
                         _stream_handle(stream, x.device))
    _check(rc, "kata_lift")
    return out


def kata_trace_begin() -> None:
    """Start per-stage device timing of every libkata launch."""
    _check(lib().kata_trace_begin(), "kata_trace_begin")


def kata_trace_end() -> dict:
    """Stop tracing; {stage: (launches, total_ms)} since kata_trace_begin."""
    buf = (TraceStage * 64)()
    n = ctypes.c_int(0)
    _check(lib().kata_trace_end(buf, 64, ctypes.byref(n)), "kata_trace_end")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n.value, 64))}


def kata_sync_status(stream=None) -> int:
    """Wait for the stream; KATA_ERR_TIMEOUT if a device-side bounded wait expired."""
    return int(lib().kata_sync_status(_stream_handle(stream, None)))


def kata_test_arm_stall() -> None:
    """Test hook: the next segment-state launch of the d = 32 tensor path issues
    no tile loads, so its bounded waits expire and kata_sync_status reports
    KATA_ERR_TIMEOUT for that call."""
    _check(lib().kata_test_arm_stall(), "kata_test_arm_stall")
