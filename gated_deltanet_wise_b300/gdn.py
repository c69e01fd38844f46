"""Thin Python binding over the C ABI of libgdn_b300.so (include/gdn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  If the
library is missing or fails to load, every call raises — there is no fallback.

The raw C entry points are exposed under their C names (``gdn_frame_fwd`` ...)
taking torch tensors; ``frame_fwd`` / ``frame_step`` / ``frame_fwd_f32`` are
conveniences that allocate outputs and workspace with torch and check status.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn_b300.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_CUDA = 3
GDN_ERR_TIMEOUT = 4
GDN_ERR_WORKSPACE = 5

EXPORTED = [
    "gdn_version", "gdn_status_string", "gdn_frame_fwd_workspace_size", "gdn_frame_fwd",
    "gdn_frame_step_workspace_size", "gdn_frame_step", "gdn_frame_fwd_f32", "gdn_device_status",
    "gdn_frame_fwd_profiled", "gdn_frame_fwd_host_buffer_size", "gdn_frame_fwd_host",
    "gdn_frame_step_noalloc_limit_bytes", "gdn_frame_step_noalloc",
    "gdn_frame_composite_workspace_size", "gdn_frame_composite", "gdn_state_compose",
    "gdn_frame_fwd_product_workspace_size", "gdn_frame_fwd_product",
    "gdn_frame_fwd_ex_workspace_size", "gdn_frame_fwd_ex",
    "gdn_frame_bwd_workspace_size", "gdn_frame_bwd", "gdn_test_frame_fwd_expired_wait",
    "gdn_block_in_proj", "gdn_block_out_proj", "gdn_block_fwd_workspace_size", "gdn_block_fwd",
    "gdn_frame_fwd_resume",
]

GDN_FWD_PRODUCT = 1
GDN_FWD_REVERSE = 2
GDN_FWD_FUSED = 4

_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libgdn_b300.so (built in-tree by gated_deltanet_wise_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libgdn_b300.so not built ({LIB_PATH}); run python -m gated_deltanet_wise_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.gdn_version.restype = I
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_status_string.argtypes = [I]
        L.gdn_frame_fwd_workspace_size.restype = Z
        L.gdn_frame_fwd_workspace_size.argtypes = [I] * 5
        L.gdn_frame_step_workspace_size.restype = Z
        L.gdn_frame_step_workspace_size.argtypes = [I] * 4
        L.gdn_frame_fwd.restype = I
        L.gdn_frame_fwd.argtypes = [P] * 8 + [I] * 5 + [F, P, Z, P]
        L.gdn_frame_step.restype = I
        L.gdn_frame_step.argtypes = [P] * 8 + [I] * 4 + [F, P, Z, P]
        L.gdn_frame_fwd_f32.restype = I
        L.gdn_frame_fwd_f32.argtypes = [P] * 8 + [I] * 5 + [F, P]
        L.gdn_device_status.restype = I
        L.gdn_device_status.argtypes = [P]
        L.gdn_frame_fwd_profiled.restype = I
        L.gdn_frame_fwd_profiled.argtypes = [P] * 8 + [I] * 5 + [F, P, Z, P, P]
        L.gdn_frame_fwd_host_buffer_size.restype = Z
        L.gdn_frame_fwd_host_buffer_size.argtypes = [I] * 5
        L.gdn_frame_fwd_host.restype = I
        L.gdn_frame_fwd_host.argtypes = [P] * 8 + [I] * 5 + [F, P, Z, P]
        L.gdn_frame_step_noalloc_limit_bytes.restype = Z
        L.gdn_frame_step_noalloc_limit_bytes.argtypes = []
        L.gdn_frame_step_noalloc.restype = I
        L.gdn_frame_step_noalloc.argtypes = [P] * 8 + [I] * 4 + [F, P]
        L.gdn_frame_composite_workspace_size.restype = Z
        L.gdn_frame_composite_workspace_size.argtypes = [I] * 5
        L.gdn_frame_composite.restype = I
        L.gdn_frame_composite.argtypes = [P] * 6 + [I] * 5 + [F, P, Z, P]
        L.gdn_state_compose.restype = I
        L.gdn_state_compose.argtypes = [P] * 4 + [I] * 2 + [P]
        L.gdn_frame_fwd_product_workspace_size.restype = Z
        L.gdn_frame_fwd_product_workspace_size.argtypes = [I] * 5
        L.gdn_frame_fwd_product.restype = I
        L.gdn_frame_fwd_product.argtypes = [P] * 8 + [I] * 5 + [F, P, Z, P]
        L.gdn_frame_fwd_ex_workspace_size.restype = Z
        L.gdn_frame_fwd_ex_workspace_size.argtypes = [I] * 5 + [ctypes.c_uint]
        L.gdn_frame_fwd_ex.restype = I
        L.gdn_frame_fwd_ex.argtypes = [P] * 8 + [I] * 5 + [F, ctypes.c_uint, P, Z, P]
        L.gdn_frame_bwd_workspace_size.restype = Z
        L.gdn_frame_bwd_workspace_size.argtypes = [I] * 5
        L.gdn_frame_bwd.restype = I
        L.gdn_frame_bwd.argtypes = [P] * 14 + [I] * 5 + [F, P, Z, P]
        L.gdn_frame_fwd_resume.restype = I
        L.gdn_frame_fwd_resume.argtypes = [P] * 5 + [I] * 5 + [P, Z, P]
        L.gdn_block_in_proj.restype = I
        L.gdn_block_in_proj.argtypes = [P] * 7 + [I] * 5 + [P]
        L.gdn_block_out_proj.restype = I
        L.gdn_block_out_proj.argtypes = [P] * 3 + [I] * 5 + [P]
        L.gdn_block_fwd_workspace_size.restype = Z
        L.gdn_block_fwd_workspace_size.argtypes = [I] * 5
        L.gdn_block_fwd.restype = I
        L.gdn_block_fwd.argtypes = [P] * 6 + [I] * 5 + [F, P, Z, P]
        L.gdn_test_frame_fwd_expired_wait.restype = I
        L.gdn_test_frame_fwd_expired_wait.argtypes = [P] * 8 + [I] * 5 + [F, P, Z, P]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_status(st: int, what: str):
    if st != GDN_OK:
        raise GdnError(st, what)


# ---------------------------------------------------------------- raw C entry points
def gdn_frame_fwd_workspace_size(B: int, H: int, F: int, N: int, D: int) -> int:
    return int(lib().gdn_frame_fwd_workspace_size(B, H, F, N, D))


def gdn_frame_fwd_resume(q, gamma, S_in, S_out, o, B, H, F, N, D, workspace, workspace_bytes, stream=None) -> int:
    return int(lib().gdn_frame_fwd_resume(_p(q), _p(gamma), _p(S_in), _p(S_out), _p(o), B, H, F, N, D,
                                          _p(workspace), int(workspace_bytes), _stream(stream)))


def gdn_block_in_proj(x, W_in, q, k, v, beta, gamma, B, H, F, N, D, stream=None) -> int:
    return int(lib().gdn_block_in_proj(_p(x), _p(W_in), _p(q), _p(k), _p(v), _p(beta), _p(gamma), B, H, F, N, D,
                                       _stream(stream)))


def gdn_block_out_proj(o, W_out, y, B, H, F, N, D, stream=None) -> int:
    return int(lib().gdn_block_out_proj(_p(o), _p(W_out), _p(y), B, H, F, N, D, _stream(stream)))


def gdn_block_fwd_workspace_size(B: int, H: int, F: int, N: int, D: int) -> int:
    return int(lib().gdn_block_fwd_workspace_size(B, H, F, N, D))


def gdn_block_fwd(x, W_in, W_out, S_in, S_out, y, B, H, F, N, D, key_scale, workspace, workspace_bytes,
                  stream=None) -> int:
    return int(lib().gdn_block_fwd(_p(x), _p(W_in), _p(W_out), _p(S_in), _p(S_out), _p(y), B, H, F, N, D,
                                   float(key_scale), _p(workspace), int(workspace_bytes), _stream(stream)))


def gdn_test_frame_fwd_expired_wait(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, workspace,
                                    workspace_bytes, stream=None) -> int:
    return int(lib().gdn_test_frame_fwd_expired_wait(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out),
                                                     _p(o), B, H, F, N, D, float(key_scale), _p(workspace),
                                                     int(workspace_bytes), _stream(stream)))


def gdn_frame_step_workspace_size(B: int, H: int, N: int, D: int) -> int:
    return int(lib().gdn_frame_step_workspace_size(B, H, N, D))


def gdn_frame_fwd(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, workspace, workspace_bytes,
                  stream=None) -> int:
    return int(lib().gdn_frame_fwd(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                   B, H, F, N, D, float(key_scale), _p(workspace), int(workspace_bytes),
                                   _stream(stream)))


def gdn_frame_fwd_product_workspace_size(B: int, H: int, F: int, N: int, D: int) -> int:
    return int(lib().gdn_frame_fwd_product_workspace_size(B, H, F, N, D))


def gdn_frame_fwd_product(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, workspace,
                          workspace_bytes, stream=None) -> int:
    return int(lib().gdn_frame_fwd_product(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                           B, H, F, N, D, float(key_scale), _p(workspace), int(workspace_bytes),
                                           _stream(stream)))


def gdn_frame_fwd_ex_workspace_size(B: int, H: int, F: int, N: int, D: int, flags: int) -> int:
    return int(lib().gdn_frame_fwd_ex_workspace_size(B, H, F, N, D, flags))


def gdn_frame_fwd_ex(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, flags, workspace,
                     workspace_bytes, stream=None) -> int:
    return int(lib().gdn_frame_fwd_ex(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                      B, H, F, N, D, float(key_scale), int(flags), _p(workspace),
                                      int(workspace_bytes), _stream(stream)))


def gdn_frame_bwd_workspace_size(B: int, H: int, F: int, N: int, D: int) -> int:
    return int(lib().gdn_frame_bwd_workspace_size(B, H, F, N, D))


def gdn_frame_bwd(q, k, v, beta, gamma, S_in, dO, dS_out, dq, dk, dv, dbeta, dgamma, dS_in, B, H, F, N, D,
                  key_scale, workspace, workspace_bytes, stream=None) -> int:
    return int(lib().gdn_frame_bwd(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(dO), _p(dS_out),
                                   _p(dq), _p(dk), _p(dv), _p(dbeta), _p(dgamma), _p(dS_in), B, H, F, N, D,
                                   float(key_scale), _p(workspace), int(workspace_bytes), _stream(stream)))


def gdn_frame_step(q, k, v, beta, gamma, S_in, S_out, o, B, H, N, D, key_scale, workspace, workspace_bytes,
                   stream=None) -> int:
    return int(lib().gdn_frame_step(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                    B, H, N, D, float(key_scale), _p(workspace), int(workspace_bytes),
                                    _stream(stream)))


def gdn_frame_fwd_f32(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, stream=None) -> int:
    return int(lib().gdn_frame_fwd_f32(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                       B, H, F, N, D, float(key_scale), _stream(stream)))


def gdn_device_status(stream=None) -> int:
    return int(lib().gdn_device_status(_stream(stream)))


def gdn_frame_fwd_profiled(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, workspace,
                           workspace_bytes, events, stream=None) -> int:
    """``events``: 4 torch.cuda.Event(enable_timing=True) recorded around the internal launches."""
    arr = None
    if events:
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
                e.record(torch.cuda.current_stream() if stream is None else stream)
        arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    return int(lib().gdn_frame_fwd_profiled(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                            B, H, F, N, D, float(key_scale), _p(workspace), int(workspace_bytes),
                                            _stream(stream), arr))


def gdn_frame_fwd_host_buffer_size(B: int, H: int, F: int, N: int, D: int) -> int:
    return int(lib().gdn_frame_fwd_host_buffer_size(B, H, F, N, D))


def gdn_frame_fwd_host(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, device_buffer,
                       device_buffer_bytes, stream=None) -> int:
    """Host tensors in (pinned CPU memory for asynchronous copies), host tensors out."""
    return int(lib().gdn_frame_fwd_host(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                        B, H, F, N, D, float(key_scale), _p(device_buffer),
                                        int(device_buffer_bytes), _stream(stream)))


def gdn_frame_step_noalloc_limit_bytes() -> int:
    return int(lib().gdn_frame_step_noalloc_limit_bytes())


def gdn_frame_step_noalloc(q, k, v, beta, gamma, S_in, S_out, o, B, H, N, D, key_scale, stream=None) -> int:
    """Streaming step whose scratch is the library's fixed device array (no workspace argument)."""
    return int(lib().gdn_frame_step_noalloc(_p(q), _p(k), _p(v), _p(beta), _p(gamma), _p(S_in), _p(S_out), _p(o),
                                            B, H, N, D, float(key_scale), _stream(stream)))


def gdn_frame_composite_workspace_size(B: int, H: int, F: int, N: int, D: int) -> int:
    return int(lib().gdn_frame_composite_workspace_size(B, H, F, N, D))


def gdn_frame_composite(k, v, beta, gamma, C_out, H_out, B, H, F, N, D, key_scale, workspace, workspace_bytes,
                        stream=None) -> int:
    return int(lib().gdn_frame_composite(_p(k), _p(v), _p(beta), _p(gamma), _p(C_out), _p(H_out), B, H, F, N, D,
                                         float(key_scale), _p(workspace), int(workspace_bytes), _stream(stream)))


def gdn_state_compose(S, C, Hc, S_out, BH, D, stream=None) -> int:
    return int(lib().gdn_state_compose(_p(S), _p(C), _p(Hc), _p(S_out), BH, D, _stream(stream)))


# ---------------------------------------------------------------- conveniences
def _shape(q: torch.Tensor, gamma: torch.Tensor) -> Tuple[int, int, int, int, int]:
    B, FN, H, D = q.shape
    F = gamma.shape[1]
    if F == 0:
        return B, H, 0, 0, D
    if FN % F:
        raise ValueError("q.shape[1] must be F * N")
    return B, H, F, FN // F, D


def _check(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Workspace:
    """Grow-only device workspace owned by the caller (the library never allocates)."""

    def __init__(self):
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int, device) -> Optional[torch.Tensor]:
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != torch.device(device):
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        return self.buf


_default_ws = Workspace()


def frame_fwd(q, k, v, beta, gamma, S_in=None, *, key_scale: float = 0.0, o=None, S_out=None,
              workspace: Optional[Workspace] = None, stream=None):
    """bf16 frame-wise GDN forward.  Returns (o [B, F*N, H, D] bf16, S_out [B, H, D, D] fp32)."""
    B, H, F, N, D = _shape(q, gamma)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, torch.bfloat16, n)
    _check(beta, torch.float32, "beta")
    _check(gamma, torch.float32, "gamma")
    if S_in is not None:
        _check(S_in, torch.float32, "S_in")
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=q.device) if S_out is None else S_out
    nbytes = gdn_frame_fwd_workspace_size(B, H, F, N, D)
    if nbytes == 2 ** 64 - 1:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_frame_fwd_workspace_size")
    ws = (workspace or _default_ws).get(nbytes, q.device)
    st = gdn_frame_fwd(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, ws, nbytes, stream)
    _check_status(st, "gdn_frame_fwd")
    return o, S_out


def frame_fwd_product(q, k, v, beta, gamma, S_in=None, *, key_scale: float = 0.0, o=None, S_out=None,
                      workspace: Optional[Workspace] = None, stream=None):
    """Token-ordered reading (gdn_frame_fwd_product); same arguments and results as frame_fwd."""
    B, H, F, N, D = _shape(q, gamma)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, torch.bfloat16, n)
    _check(beta, torch.float32, "beta")
    _check(gamma, torch.float32, "gamma")
    if S_in is not None:
        _check(S_in, torch.float32, "S_in")
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=q.device) if S_out is None else S_out
    nbytes = gdn_frame_fwd_product_workspace_size(B, H, F, N, D)
    if nbytes == 2 ** 64 - 1:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_frame_fwd_product_workspace_size")
    ws = (workspace or _default_ws).get(nbytes, q.device)
    st = gdn_frame_fwd_product(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, ws, nbytes, stream)
    _check_status(st, "gdn_frame_fwd_product")
    return o, S_out


def frame_fwd_ex(q, k, v, beta, gamma, S_in=None, *, product: bool = False, reverse: bool = False,
                 fused: bool = False, key_scale: float = 0.0, o=None, S_out=None,
                 workspace: Optional[Workspace] = None, stream=None):
    """gdn_frame_fwd_ex: the sum or product reading, forward or reverse frame order, the sum
    reading optionally as the fused chained-scan launch."""
    B, H, F, N, D = _shape(q, gamma)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, torch.bfloat16, n)
    _check(beta, torch.float32, "beta")
    _check(gamma, torch.float32, "gamma")
    if S_in is not None:
        _check(S_in, torch.float32, "S_in")
    flags = (GDN_FWD_PRODUCT if product else 0) | (GDN_FWD_REVERSE if reverse else 0) | \
        (GDN_FWD_FUSED if fused else 0)
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=q.device) if S_out is None else S_out
    nbytes = gdn_frame_fwd_ex_workspace_size(B, H, F, N, D, flags)
    if nbytes == 2 ** 64 - 1:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_frame_fwd_ex_workspace_size")
    ws = (workspace or _default_ws).get(nbytes, q.device)
    st = gdn_frame_fwd_ex(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, flags, ws, nbytes, stream)
    _check_status(st, "gdn_frame_fwd_ex")
    return o, S_out


def frame_bwd(q, k, v, beta, gamma, S_in, dO, dS_out=None, *, key_scale: float = 0.0,
              workspace: Optional[Workspace] = None, stream=None):
    """gdn_frame_bwd: returns (dq, dk, dv, dbeta, dgamma, dS_in), fp32."""
    B, H, F, N, D = _shape(q, gamma)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dO, "dO")):
        _check(t, torch.bfloat16, n)
    _check(beta, torch.float32, "beta")
    _check(gamma, torch.float32, "gamma")
    for t, n in ((S_in, "S_in"), (dS_out, "dS_out")):
        if t is not None:
            _check(t, torch.float32, n)
    dev = q.device
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    dbeta = torch.empty(beta.shape, dtype=torch.float32, device=dev)
    dgamma = torch.empty(gamma.shape, dtype=torch.float32, device=dev)
    dS_in = torch.empty(B, H, D, D, dtype=torch.float32, device=dev)
    nbytes = gdn_frame_bwd_workspace_size(B, H, F, N, D)
    if nbytes == 2 ** 64 - 1:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_frame_bwd_workspace_size")
    ws = (workspace or _default_ws).get(nbytes, dev)
    st = gdn_frame_bwd(q, k, v, beta, gamma, S_in, dO, dS_out, dq, dk, dv, dbeta, dgamma, dS_in, B, H, F, N, D,
                       key_scale, ws, nbytes, stream)
    _check_status(st, "gdn_frame_bwd")
    return dq, dk, dv, dbeta, dgamma, dS_in


def frame_step(q, k, v, beta, gamma, S_in=None, *, key_scale: float = 0.0, o=None, S_out=None,
               workspace: Optional[Workspace] = None, stream=None):
    """One latent frame: q/k/v [B, N, H, D] bf16, beta [B, N, H], gamma [B, H]."""
    B, N, H, D = q.shape
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=q.device) if S_out is None else S_out
    nbytes = gdn_frame_step_workspace_size(B, H, N, D)
    if nbytes == 2 ** 64 - 1:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_frame_step_workspace_size")
    ws = (workspace or _default_ws).get(nbytes, q.device)
    st = gdn_frame_step(q, k, v, beta, gamma, S_in, S_out, o, B, H, N, D, key_scale, ws, nbytes, stream)
    _check_status(st, "gdn_frame_step")
    return o, S_out


def frame_fwd_f32(q, k, v, beta, gamma, S_in=None, *, key_scale: float = 0.0, stream=None):
    """fp32 validation path.  Returns (o fp32, S_out fp32)."""
    B, H, F, N, D = _shape(q, gamma)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, torch.float32, n)
    o = torch.empty_like(q)
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=q.device)
    st = gdn_frame_fwd_f32(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, stream)
    _check_status(st, "gdn_frame_fwd_f32")
    return o, S_out


def frame_composite(k, v, beta, gamma, *, key_scale: float = 0.0, workspace: Optional[Workspace] = None,
                    stream=None, outputs: bool = True):
    """Per-chain composites (C, H) of the frames given, each [B, H, D, D] fp32.  With
    outputs=False only the frame-statistics pass runs (C_out = H_out = NULL) and (None, None)
    comes back: the workspace still holds what gdn_frame_fwd_resume needs."""
    B, H, F, N, D = _shape(k, gamma)
    for t, n in ((k, "k"), (v, "v")):
        _check(t, torch.bfloat16, n)
    C = torch.empty(B, H, D, D, dtype=torch.float32, device=k.device) if outputs else None
    Hc = torch.empty_like(C) if outputs else None
    nbytes = gdn_frame_composite_workspace_size(B, H, F, N, D)
    if nbytes == 2 ** 64 - 1:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_frame_composite_workspace_size")
    ws = (workspace or _default_ws).get(nbytes, k.device)
    st = gdn_frame_composite(k, v, beta, gamma, C, Hc, B, H, F, N, D, key_scale, ws, nbytes, stream)
    _check_status(st, "gdn_frame_composite")
    return C, Hc


def frame_fwd_resume(q, gamma, S_in=None, *, workspace: Workspace, o=None, S_out=None, stream=None):
    """Finish the forward of the frames whose composites the last frame_composite call on
    `workspace` computed (gdn_frame_fwd_resume).  Returns (o, S_out)."""
    B, H, F, N, D = _shape(q, gamma)
    _check(q, torch.bfloat16, "q")
    _check(gamma, torch.float32, "gamma")
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=q.device) if S_out is None else S_out
    nbytes = gdn_frame_composite_workspace_size(B, H, F, N, D)
    ws = workspace.get(nbytes, q.device)
    st = gdn_frame_fwd_resume(q, gamma, S_in, S_out, o, B, H, F, N, D, ws, nbytes, stream)
    _check_status(st, "gdn_frame_fwd_resume")
    return o, S_out


def state_compose(S, C, Hc, *, out=None, stream=None):
    """S C + Hc per chain (S None: zero); tensors [..., D, D] fp32."""
    D = C.shape[-1]
    BH = C.numel() // (D * D)
    out = torch.empty_like(C) if out is None else out
    st = gdn_state_compose(S, C, Hc, out, BH, D, stream)
    _check_status(st, "gdn_state_compose")
    return out


def block_fwd(x, W_in, W_out, S_in=None, *, F: int, key_scale: float = 0.0, y=None, S_out=None,
              workspace: Optional[Workspace] = None, stream=None):
    """GDN block with its projections (gdn_block_fwd).  x: bf16 [B, F*N, H*D];
    W_in: bf16 [3*H*D + 2*H, H*D]; W_out: bf16 [H*D, H*D].  Returns (y, S_out)."""
    _check(x, torch.bfloat16, "x")
    _check(W_in, torch.bfloat16, "W_in")
    _check(W_out, torch.bfloat16, "W_out")
    B, FN, HD = x.shape
    D = 112
    H = HD // D
    N = FN // F
    if H * D != HD or F * N != FN or W_in.shape != (3 * HD + 2 * H, HD) or W_out.shape != (HD, HD):
        raise ValueError("block shapes: x [B, F*N, H*112], W_in [3HD+2H, HD], W_out [HD, HD]")
    if S_in is not None:
        _check(S_in, torch.float32, "S_in")
    y = torch.empty_like(x) if y is None else y
    S_out = torch.empty(B, H, D, D, dtype=torch.float32, device=x.device) if S_out is None else S_out
    nbytes = gdn_block_fwd_workspace_size(B, H, F, N, D)
    if nbytes == 2 ** 64 - 1:
        raise GdnError(GDN_ERR_UNSUPPORTED, "gdn_block_fwd_workspace_size")
    ws = (workspace or _default_ws).get(nbytes, x.device)
    st = gdn_block_fwd(x, W_in, W_out, S_in, S_out, y, B, H, F, N, D, key_scale, ws, nbytes, stream)
    _check_status(st, "gdn_block_fwd")
    return y, S_out
