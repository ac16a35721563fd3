"""Python front end of the fp64 CPU oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module; the library never does.
It shares no code with the CUDA path.

The oracle is the plain token-by-token KDA recurrence
``S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T``,
``o_t = scale * S_t^T q_t`` (decay first, then the delta-rule write), with the
state pool semantics of the sglang PR 30169 digest ("pool state I/O fused into
the h kernel", section 实现拆解 items 1-3): slot index -1 maps to the last slot.
Inputs are widened exactly to fp64 before the call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/libkda_oracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        d = ctypes.POINTER(ctypes.c_double)
        i = ctypes.POINTER(ctypes.c_int)
        lib.kda_oracle_recurrence.restype = ctypes.c_int
        lib.kda_oracle_recurrence.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            d, d, d, d, d, i, d, i, ctypes.c_longlong, d, d, ctypes.c_int]
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> exact fp64 on the host
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def recurrence(q, k, v, g, beta, cu_seqlens, *, scale=None, state=None, state_indices=None,
               num_threads: int = 0):
    """Run the oracle.

    q, k: [T, Hk, K]; v: [T, Hv, V]; g: [T, Hv, K]; beta: [T, Hv];
    cu_seqlens: [N+1] int.  ``state`` is a dense h0 [N, Hv, K, V] (no indices),
    a pool [num_slots, Hv, K, V] (with ``state_indices`` [N]) or None (zeros).
    ``scale`` defaults to K**-0.5.

    Returns ``(o, final)``: o [T, Hv, V] fp64; ``final`` is the dense final state
    [N, Hv, K, V] (no indices) or the updated pool copy (with indices).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if g.ndim == 2:  # scalar (GDN) gate [T, Hv]: the same decay on every key channel
        g = np.ascontiguousarray(np.repeat(g[:, :, None], q.shape[2], axis=2))
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int32))
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu.shape[0] - 1
    if scale is None:
        scale = K ** -0.5
    st = _f64(state)
    idx = None
    num_slots = 0
    if state_indices is not None:
        idx = np.ascontiguousarray(np.asarray(
            state_indices.cpu().numpy() if hasattr(state_indices, "cpu") else state_indices,
            dtype=np.int32))
        num_slots = st.shape[0]
        out_state = np.empty_like(st)
    else:
        out_state = np.empty((N, Hv, K, V), dtype=np.float64)
    o = np.zeros((T, Hv, V), dtype=np.float64)
    # g and beta may be longer than T (padding); only the first T rows are read.
    g = np.ascontiguousarray(g[:T])
    beta = np.ascontiguousarray(beta[:T])
    rc = _load().kda_oracle_recurrence(
        N, Hk, Hv, K, V, float(scale),
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        _ptr(g, ctypes.c_double), _ptr(beta, ctypes.c_double), _ptr(cu, ctypes.c_int),
        _ptr(st, ctypes.c_double), _ptr(idx, ctypes.c_int), int(num_slots),
        _ptr(o, ctypes.c_double), _ptr(out_state, ctypes.c_double), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return o, out_state


def decode(q, k, v, g, beta, *, pool, state_indices, scale=None, num_threads: int = 0):
    """One token per row: the prefill recurrence with every length equal to 1."""
    n = q.shape[0]
    cu = np.arange(n + 1, dtype=np.int32)
    return recurrence(q, k, v, g, beta, cu, scale=scale, state=pool,
                      state_indices=state_indices, num_threads=num_threads)


def gate_activation(a, A_log, dt_bias=None, lower_bound=None):
    """Log-decay from the gate pre-activation, in fp64:
    ``g[t,h,c] = max(-exp(A_log[h]) * softplus(a[t,h,c] + dt_bias[h,c]), lower_bound)``.

    The ``-exp(A_log) * softplus(a + dt_bias)`` form is the gate the pages' tests build
    (sglang PR 30169 digest, 关键源码片段: the GDN pool test, one scalar per head there);
    the KDA prefill entry takes ``A_log``, ``dt_bias`` and ``lower_bound``
    (PR 27488 digest, 关键源码片段: ``CuteDSLKDAKernel.extend``).  Here ``a`` and
    ``dt_bias`` carry a key-channel axis, as KDA's per-channel gate does.  The pages
    name ``lower_bound`` without a formula; it is read as a floor on g.

    softplus(x) = log(1 + e^x), evaluated as max(x, 0) + log1p(e^-|x|) so that no
    intermediate overflows.  a [T, Hv, K]; A_log [Hv]; dt_bias [Hv, K] or None.  A scalar
    (GDN) gate, as on the pages: a [T, Hv] and dt_bias [Hv], giving g [T, Hv].
    """
    a = _f64(a)
    A = np.exp(_f64(A_log))
    x = a + (_f64(dt_bias)[None] if dt_bias is not None else 0.0)
    sp = np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))
    g = -(A[None, :, None] if a.ndim == 3 else A[None, :]) * sp
    if lower_bound is not None:
        g = np.maximum(g, float(lower_bound))
    return g


def l2norm(x, eps=1e-12):
    """Rows of x (last axis) divided by max(||row||_2, eps), in fp64: the q/k normalisation
    the pages' callers apply before the prefill (sglang PR 27488 digest, 关键源码片段
    ``CuteDSLKDAKernel.extend``), which the kernels can do in place (KDA_FLAG_QK_L2NORM)."""
    x = _f64(x)
    return x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), eps)
