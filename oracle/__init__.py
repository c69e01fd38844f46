"""fp64 CPU oracle for the frame-wise Gated DeltaNet forward pass.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline may use this package; the product library never does.  The arithmetic
lives in ``gdn_oracle.c`` (plain C, fp64); this module only marshals numpy
arrays into it.  Every function states the passage it follows, on the summary
page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid Linear
Diffusion Transformer":

* section 方法步骤详情 (method details), module 2: the recurrence
  S_t = S_{t-1}(gamma_t I - K^ beta K^T) + V beta K^T and the output O_t = S_t Q^_t;
* section 前置知识 "Gated DeltaNet": S_t = S_{t-1} M_t + U_t;
* section 技术新颖性 (novelty): ||M_t||_2 <= gamma_t <= 1 and the exact
  composite prefix scan (C_p, H_p) used for context parallelism.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        Dbl = ctypes.c_double
        lib.oracle_gdn_frame_fwd.argtypes = [P] * 6 + [I] * 5 + [Dbl, P, P]
        lib.oracle_gdn_frame_fwd_tokacc.argtypes = [P] * 6 + [I] * 5 + [Dbl, P, P]
        lib.oracle_gdn_frame_transitions.argtypes = [P] * 4 + [I] * 5 + [Dbl, P, P]
        lib.oracle_gdn_frame_fwd_product.argtypes = [P] * 6 + [I] * 5 + [Dbl, P, P]
        lib.oracle_gdn_frame_transitions_product.argtypes = [P] * 4 + [I] * 5 + [Dbl, P, P]
        lib.oracle_gdn_frame_bwd.argtypes = [P] * 8 + [I] * 5 + [Dbl] + [P] * 6
        lib.oracle_gdn_composite.argtypes = [P, P, I, I, P, P]
        lib.oracle_gdn_compose.argtypes = [P, P, P, P, I, P, P]
        lib.oracle_num_threads.restype = I
        _lib = lib
    return _lib


def _f32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> exact fp32 copy on the host
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shapes(q):
    B, FN, H, D = q.shape
    return B, FN, H, D


def _flip_frames(x, F):
    """Reverse the frame order of a [B, F*N, ...] token array (or [B, F, H] per-frame array)."""
    B, FN = x.shape[:2]
    return np.ascontiguousarray(x.reshape(B, F, FN // F, *x.shape[2:])[:, ::-1].reshape(x.shape))


def frame_fwd(q, k, v, beta, gamma, S_in=None, N=None, key_scale=0.0, formulation="recurrence",
              mode="sum", reverse=False):
    """Frame-wise GDN forward in fp64.

    Shapes: q, k, v [B, F*N, H, D]; beta [B, F*N, H]; gamma [B, F, H];
    S_in [B, H, D, D] or None.  Returns (o [B, F*N, H, D] fp64, S_out [B, H, D, D] fp64).
    ``mode="sum"`` is the transition as printed in module 2 of the
    method-details section, M_f = gamma_f I - sum_n beta_n k^_n k^_n^T; there
    ``formulation`` picks the printed recurrence ("recurrence") or the
    token-accumulation rewrite ("tokacc").  ``mode="product"`` is the
    token-ordered reading M_f = gamma_f I - (I - prod_n (I - beta_n k^_n k^_n^T))
    with the frame's tokens applied in order from zero for U_f, computed by the
    plain definition, one token at a time.

    ``reverse=True`` is the reverse-direction scan of the bidirectional stage-1
    model (summary page, section 局限与改进): the frames are visited from the
    last to the first, starting from S_in, each frame's output read from the
    state after its own update, and S_out is the state after frame 0.  It is
    computed literally as the forward scan of the frame-reversed sequence,
    with the outputs put back in frame order.
    """
    if reverse:
        q, k, v, beta, gamma = (_f32(x) for x in (q, k, v, beta, gamma))
        F = gamma.shape[1]
        o, S_out = frame_fwd(*(_flip_frames(x, F) for x in (q, k, v, beta, gamma)), S_in, N=N, key_scale=key_scale,
                             formulation=formulation, mode=mode)
        return _flip_frames(o, F), S_out
    q, k, v, beta, gamma, S_in = (_f32(x) for x in (q, k, v, beta, gamma, S_in))
    B, FN, H, D = _shapes(q)
    F = gamma.shape[1]
    N = FN // F if N is None else N
    assert F * N == FN and k.shape == q.shape and v.shape == q.shape
    assert beta.shape == (B, FN, H) and gamma.shape == (B, F, H)
    if S_in is not None:
        assert S_in.shape == (B, H, D, D)
    o = np.zeros((B, FN, H, D), np.float64)
    S_out = np.zeros((B, H, D, D), np.float64)
    if mode == "product":
        _load().oracle_gdn_frame_fwd_product(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gamma), _ptr(S_in),
                                             B, H, F, N, D, float(key_scale), _ptr(o), _ptr(S_out))
        return o, S_out
    assert mode == "sum", mode
    fn = {"recurrence": _load().oracle_gdn_frame_fwd,
          "tokacc": _load().oracle_gdn_frame_fwd_tokacc}[formulation]
    fn(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gamma), _ptr(S_in),
       B, H, F, N, D, float(key_scale), _ptr(o), _ptr(S_out))
    return o, S_out


def frame_transitions(k, v, beta, gamma, key_scale=0.0, mode="sum"):
    """Per-frame (M_f, U_f), each [B, H, F, D, D] fp64 (module 2: M_t = gamma_t I - K^ beta K^T).

    ``mode`` as in ``frame_fwd``.
    """
    k, v, beta, gamma = (_f32(x) for x in (k, v, beta, gamma))
    B, FN, H, D = _shapes(k)
    F = gamma.shape[1]
    N = FN // F
    M = np.zeros((B, H, F, D, D), np.float64)
    U = np.zeros((B, H, F, D, D), np.float64)
    if mode == "product":
        _load().oracle_gdn_frame_transitions_product(_ptr(k), _ptr(v), _ptr(beta), _ptr(gamma),
                                                     B, H, F, N, D, float(key_scale), _ptr(M), _ptr(U))
        return M, U
    assert mode == "sum", mode
    _load().oracle_gdn_frame_transitions(_ptr(k), _ptr(v), _ptr(beta), _ptr(gamma),
                                         B, H, F, N, D, float(key_scale), _ptr(M), _ptr(U))
    return M, U


def frame_bwd(q, k, v, beta, gamma, S_in, dO, dS_out=None, key_scale=0.0):
    """Backward pass of the sum reading in fp64 (gradients by the chain rule through
    the printed recurrence; see oracle_gdn_frame_bwd in gdn_oracle.c).

    dO [B, F*N, H, D] is dL/do, dS_out [B, H, D, D] is dL/dS_out (None: zero).
    Returns (dq, dk, dv [B, F*N, H, D], dbeta [B, F*N, H], dgamma [B, F, H], dS_in [B, H, D, D]), fp64.
    """
    q, k, v, beta, gamma, S_in, dO, dS_out = (_f32(x) for x in (q, k, v, beta, gamma, S_in, dO, dS_out))
    B, FN, H, D = _shapes(q)
    F = gamma.shape[1]
    N = FN // F if F else 0
    dq = np.zeros((B, FN, H, D), np.float64)
    dk = np.zeros_like(dq)
    dv = np.zeros_like(dq)
    dbeta = np.zeros((B, FN, H), np.float64)
    dgamma = np.zeros((B, F, H), np.float64)
    dS_in = np.zeros((B, H, D, D), np.float64)
    _load().oracle_gdn_frame_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(gamma), _ptr(S_in), _ptr(dO),
                                 _ptr(dS_out), B, H, F, N, D, float(key_scale), _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(dbeta), _ptr(dgamma), _ptr(dS_in))
    return dq, dk, dv, dbeta, dgamma, dS_in


def _round_bf16(a):
    """Round-to-nearest-even to bf16, returned as float32 (the layer's input type)."""
    a32 = np.ascontiguousarray(a, dtype=np.float32)
    u = a32.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def block_in_proj(x, W_in, F, D=112):
    """The GDN block's input projection in fp64 (summary page, section 方法步骤详情 module 1:
    d_model = H * D; the projection shapes are a reading, the pages print none):
    [q | k | v | a | g] = x W_in^T, beta = sigmoid(a), gamma_f = exp(-softplus(mean over the
    frame's tokens of g)).  q, k, v are rounded to bf16, the layer's input type.
    x [B, F*N, H*D]; returns (q, k, v [B, F*N, H, D] fp32 holding bf16 values, beta [B, F*N, H],
    gamma [B, F, H] fp64)."""
    x = np.asarray(_f32(x), dtype=np.float64)
    W = np.asarray(_f32(W_in), dtype=np.float64)
    B, FN, HD = x.shape
    H = HD // D
    N = FN // F
    P = x @ W.T                      # library matmul as one step: [B, F*N, 3HD + 2H]
    q, k, v = (_round_bf16(P[..., i * HD:(i + 1) * HD]).reshape(B, FN, H, D) for i in range(3))
    a = P[..., 3 * HD:3 * HD + H]
    g = P[..., 3 * HD + H:3 * HD + 2 * H]
    beta = 1.0 / (1.0 + np.exp(-a))
    gmean = g.reshape(B, F, N, H).mean(axis=2)
    gamma = np.exp(-np.logaddexp(0.0, gmean))   # exp(-softplus)
    return q, k, v, beta, gamma


def block_fwd(x, W_in, W_out, S_in=None, F=None, key_scale=0.0, D=112):
    """The whole GDN block in fp64: input projection, the frame-wise forward (frame_fwd, sum
    reading), output projection y = o W_out^T (o kept in fp64).  Returns (y [B, F*N, H*D],
    S_out [B, H, D, D])."""
    q, k, v, beta, gamma = block_in_proj(x, W_in, F, D)
    o, S_out = frame_fwd(q, k, v, beta, gamma, S_in, key_scale=key_scale)
    B, FN, H, _ = o.shape
    y = o.reshape(B, FN, H * D) @ np.asarray(_f32(W_out), dtype=np.float64).T
    return y, S_out


def composite(M, U):
    """(C, H) of a run of frames: C = prod M_f, H = state reached from zero (novelty section, C_p / H_p)."""
    M = np.ascontiguousarray(M, dtype=np.float64)
    U = np.ascontiguousarray(U, dtype=np.float64)
    nF, D, _ = M.shape
    C = np.zeros((D, D)); Hc = np.zeros((D, D))
    _load().oracle_gdn_composite(_ptr(M), _ptr(U), nF, D, _ptr(C), _ptr(Hc))
    return C, Hc


def compose(C1, H1, C2, H2):
    """(C1, H1) followed by (C2, H2) -> (C1 C2, H1 C2 + H2)."""
    arrs = [np.ascontiguousarray(x, dtype=np.float64) for x in (C1, H1, C2, H2)]
    D = arrs[0].shape[0]
    C = np.zeros((D, D)); Hc = np.zeros((D, D))
    _load().oracle_gdn_compose(*(_ptr(a) for a in arrs), D, _ptr(C), _ptr(Hc))
    return C, Hc


def num_threads() -> int:
    return int(_load().oracle_num_threads())
