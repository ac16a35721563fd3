"""Thin Python binding of ``libkda_gb300.so`` (argument marshalling only).

Every step of the prefill and decode runs in the library's CUDA kernels; this
module only checks tensors, builds the ``kda_desc_t`` descriptor, allocates the
workspace and outputs with ``torch.empty`` and passes raw device pointers and
the current CUDA stream.  There is no CPU fallback: if the library cannot be
loaded the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

KDA_BF16, KDA_F32 = 0, 1
KDA_FLAG_CUDA_CORE_PATH = 0x1
KDA_FLAG_SCALAR_GATE = 0x2
KDA_FLAG_QK_L2NORM = 0x4
KDA_FLAG_STATE_VK = 0x8
KDA_DEVICE_BAD_SLOT, KDA_DEVICE_BAD_SEQLENS, KDA_DEVICE_PIPE_TIMEOUT = 0x1, 0x2, 0x4
KDA_DEVICE_DEBUG_BOUNDS = 0x8
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
           3: "workspace too small", 4: "CUDA error", 5: "invalid device data"}


class KdaError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {_STATUS.get(code, code)} (status {code})")


class KdaDesc(ctypes.Structure):
    """Mirror of ``kda_desc_t`` in include/kda.h."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("num_k_heads", ctypes.c_int32),
        ("num_v_heads", ctypes.c_int32),
        ("head_k_dim", ctypes.c_int32),
        ("head_v_dim", ctypes.c_int32),
        ("qkv_dtype", ctypes.c_int),
        ("state_dtype", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("chunk_size", ctypes.c_int32),
        ("num_slots", ctypes.c_int64),
        ("slot_stride_elems", ctypes.c_int64),
        ("flags", ctypes.c_uint32),
    ]


EXPORTS = ("kda_chunk_prefill_workspace_size", "kda_chunk_prefill_min_workspace_size",
           "kda_decode_workspace_size", "kda_chunk_prefill",
           "kda_decode", "kda_read_device_status", "kda_chunk_prefill_path", "kda_status_string",
           "kda_chunk_prefill_noalloc", "kda_chunk_prefill_act", "kda_decode_draft",
           "kda_set_pipeline_wait_limit")

_lib = None


def debug_build() -> bool:
    """KDA_DEBUG=1 selects the bounds-checked library (libkda_gb300_debug.so)."""
    return os.environ.get("KDA_DEBUG", "") == "1"


def library_path() -> str:
    return _build.LIB_DEBUG if debug_build() else _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed) the CUDA library and declare its prototypes."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path) and not build_if_missing:
        raise RuntimeError(f"{path} is missing; run __graft_entry__.build()")
    if build_if_missing:
        _build.build(debug=debug_build())  # no-op unless a source is newer than the library
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    D = ctypes.POINTER(KdaDesc)
    lib.kda_chunk_prefill_workspace_size.argtypes = [D]
    lib.kda_chunk_prefill_workspace_size.restype = ctypes.c_size_t
    lib.kda_chunk_prefill_min_workspace_size.argtypes = [D]
    lib.kda_chunk_prefill_min_workspace_size.restype = ctypes.c_size_t
    lib.kda_decode_workspace_size.argtypes = [D]
    lib.kda_decode_workspace_size.restype = ctypes.c_size_t
    lib.kda_chunk_prefill.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.kda_chunk_prefill.restype = ctypes.c_int
    lib.kda_decode.argtypes = [D, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.kda_decode.restype = ctypes.c_int
    lib.kda_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.kda_read_device_status.restype = ctypes.c_int
    lib.kda_chunk_prefill_path.argtypes = [D]
    lib.kda_chunk_prefill_path.restype = ctypes.c_int
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_chunk_prefill_noalloc.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P]
    lib.kda_chunk_prefill_noalloc.restype = ctypes.c_int
    lib.kda_chunk_prefill_act.argtypes = [D, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, P, P, P,
                                          ctypes.c_size_t, P]
    lib.kda_chunk_prefill_act.restype = ctypes.c_int
    lib.kda_decode_draft.argtypes = [D, P, P, P, P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int32,
                                     ctypes.c_int, P, P, ctypes.c_size_t, P]
    lib.kda_decode_draft.restype = ctypes.c_int
    lib.kda_set_pipeline_wait_limit.argtypes = [ctypes.c_uint64]
    lib.kda_set_pipeline_wait_limit.restype = ctypes.c_int
    _lib = lib
    return lib


def _dt(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return KDA_BF16
    if t == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t}; use bfloat16 or float32")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _shape(t, name, dims, min_rows=None):
    """t has len(dims) dimensions matching dims (None matches any size); with min_rows its
    first dimension is at least that.  The C ABI takes plain pointers, so this is where a
    tensor too small for the descriptor is caught, before any launch."""
    if t.dim() != len(dims) or any(d is not None and t.shape[i] != d for i, d in enumerate(dims)):
        want = "[" + ", ".join("*" if d is None else str(d) for d in dims) + "]"
        raise ValueError(f"{name} must have shape {want}, got {list(t.shape)}")
    if min_rows is not None and t.shape[0] < min_rows:
        raise ValueError(f"{name} needs at least {min_rows} rows, got {t.shape[0]}")


def _gate_shape(gate, name, T, Hv, K):
    """[>=T, Hv, K] per key channel, or [>=T, Hv] for a scalar gate."""
    if gate.dim() == 2:
        _shape(gate, name, (None, Hv), min_rows=T)
    else:
        _shape(gate, name, (None, Hv, K), min_rows=T)


def _pool_shape(pool, name, Hv, K, V, slot_stride):
    if slot_stride == 0:
        _shape(pool, name, (None, Hv, K, V))
    elif pool.dim() < 1 or pool.numel() < (pool.shape[0] - 1) * slot_stride + Hv * K * V:
        raise ValueError(f"{name} is too small for {pool.shape[0]} slots of pitch {slot_stride}")


def _state_dims(K, V, state_layout):
    """Trailing dims of one head's state: (K, V), or (V, K) for the transposed layout."""
    if state_layout not in ("kv", "vk"):
        raise ValueError(f"state_layout must be 'kv' or 'vk', got {state_layout!r}")
    return (K, V) if state_layout == "kv" else (V, K)


def check_prefill_shapes(q, k, v, gate, beta, cu_seqlens, *, state=None, state_indices=None,
                         final_state=None, out=None, A_log=None, dt_bias=None, slot_stride=0,
                         state_layout="kv"):
    """Shape checks of a prefill call (host only; see :func:`chunk_prefill`)."""
    _shape(q, "q", (None, None, None))
    T, Hk, K = q.shape
    _shape(k, "k", (T, Hk, K))
    _shape(v, "v", (T, None, None))
    Hv, V = v.shape[1], v.shape[2]
    SA, SB = _state_dims(K, V, state_layout)
    if Hk == 0 or Hv % Hk != 0:
        raise ValueError(f"the v-head count {Hv} must be a multiple of the k-head count {Hk}")
    _gate_shape(gate, "g" if A_log is None else "a", T, Hv, K)
    _shape(beta, "beta", (None, Hv), min_rows=T)
    _shape(cu_seqlens, "cu_seqlens", (None,), min_rows=1)
    N = cu_seqlens.shape[0] - 1
    if A_log is not None:
        _shape(A_log, "A_log", (Hv,))
        if dt_bias is not None:
            _shape(dt_bias, "dt_bias", (Hv,) if gate.dim() == 2 else (Hv, K))
    if state_indices is not None:
        _shape(state_indices, "state_indices", (N,))
        if state is not None:
            _pool_shape(state, "state", Hv, SA, SB, slot_stride)
    else:
        if state is not None:
            _shape(state, "state", (N, Hv, SA, SB))
        if final_state is not None:
            _shape(final_state, "final_state", (N, Hv, SA, SB))
        # the kernels write the final state in the element type of the initial one: a
        # final_state of another dtype would be written past its end (or only half filled)
        if state is not None and final_state is not None and state.dtype != final_state.dtype:
            raise TypeError(f"final_state must be {state.dtype} like state, got {final_state.dtype}")
    if out is not None:
        _shape(out, "out", (T, Hv, V))
        if out.dtype != q.dtype:
            raise TypeError(f"out must be {q.dtype}, got {out.dtype}")


def check_decode_shapes(q, k, v, g, beta, pool, *, state_indices=None, out=None, slot_stride=0,
                        cu_seqlens=None, state_layout="kv"):
    """Shape checks of a decode call (one row per token, or draft steps per request when
    ``cu_seqlens`` is given; host only)."""
    _shape(q, "q", (None, None, None))
    T, Hk, K = q.shape
    _shape(k, "k", (T, Hk, K))
    _shape(v, "v", (T, None, None))
    Hv, V = v.shape[1], v.shape[2]
    if Hk == 0 or Hv % Hk != 0:
        raise ValueError(f"the v-head count {Hv} must be a multiple of the k-head count {Hk}")
    _gate_shape(g, "g", T, Hv, K)
    _shape(beta, "beta", (None, Hv), min_rows=T)
    _pool_shape(pool, "pool", Hv, *_state_dims(K, V, state_layout), slot_stride)
    N = T
    if cu_seqlens is not None:
        _shape(cu_seqlens, "cu_seqlens", (None,), min_rows=1)
        N = cu_seqlens.shape[0] - 1
    if state_indices is not None:
        _shape(state_indices, "state_indices", (N,))
    if out is not None:
        _shape(out, "out", (T, Hv, V))
        if out.dtype != q.dtype:
            raise TypeError(f"out must be {q.dtype}, got {out.dtype}")


def make_desc(*, num_seqs, total_tokens, Hk, Hv, K, V, qkv_dtype, state_dtype=torch.float32,
              scale=None, num_slots=0, slot_stride=0, flags=0) -> KdaDesc:
    d = KdaDesc()
    d.num_seqs = num_seqs
    d.total_tokens = total_tokens
    d.num_k_heads, d.num_v_heads, d.head_k_dim, d.head_v_dim = Hk, Hv, K, V
    d.qkv_dtype = _dt(qkv_dtype)
    d.state_dtype = _dt(state_dtype)
    d.scale = 0.0 if scale is None else float(scale)
    d.chunk_size = 64
    d.num_slots = num_slots
    d.slot_stride_elems = slot_stride
    d.flags = flags
    return d


def prefill_workspace_size(desc: KdaDesc) -> int:
    return int(load().kda_chunk_prefill_workspace_size(ctypes.byref(desc)))


def prefill_min_workspace_size(desc: KdaDesc) -> int:
    """Least workspace the prefill accepts: no sequence is cut in two with less than
    :func:`prefill_workspace_size`."""
    return int(load().kda_chunk_prefill_min_workspace_size(ctypes.byref(desc)))


def prefill_path(desc: KdaDesc) -> int:
    """1 = fused tensor-core path, 0 = CUDA-core path, -1 = invalid descriptor."""
    return int(load().kda_chunk_prefill_path(ctypes.byref(desc)))


def set_pipeline_wait_limit(nanoseconds: int = 0) -> None:
    """Bound of the tensor-core prefill's internal waits for later launches (0: the default
    2 s).  A timeout sets KDA_DEVICE_PIPE_TIMEOUT in the device status; the call returns."""
    rc = load().kda_set_pipeline_wait_limit(int(nanoseconds))
    if rc != 0:
        raise KdaError(rc, "kda_set_pipeline_wait_limit")


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the device status bits of the last call."""
    bits = ctypes.c_uint32(0)
    rc = load().kda_read_device_status(_ptr(workspace), ctypes.byref(bits), _stream(stream))
    if rc not in (0, 5):
        raise KdaError(rc, "kda_read_device_status")
    return int(bits.value)


def chunk_prefill(q, k, v, g, beta, cu_seqlens, *, state=None, state_indices=None,
                  final_state=None, output_final_state=True, scale=None, slot_stride=0,
                  out=None, workspace=None, stream=None, cuda_core_path=False, qk_l2norm=False,
                  state_layout="kv"):
    """Chunked KDA prefill.  Returns ``(o, final)``.

    q, k [T, Hk, K]; v [T, Hv, V] (bf16 or fp32, same dtype); g [>=T, Hv, K] fp32, or
    [>=T, Hv] for a scalar (per token and head, GDN) gate; beta [>=T, Hv] fp32;
    cu_seqlens [N+1] int32.
    Pool mode (``state_indices`` [N] int32 given): ``state`` is the pool
    [num_slots, Hv, K, V], updated in place and returned as ``final``.
    Dense mode: ``state`` is h0 [N, Hv, K, V] or None; ``final`` is a new
    [N, Hv, K, V] tensor (or ``final_state`` if given, may be ``state``) or None
    when ``output_final_state`` is False.  ``qk_l2norm`` normalises q and k per
    (token, head) inside the kernel (KDA_FLAG_QK_L2NORM).  ``state_layout="vk"`` stores every
    head's state transposed, [V, K] (the pages' pool layout; KDA_FLAG_STATE_VK).
    """
    _need(g, "g", torch.float32)
    return _prefill(q, k, v, g, None, beta, cu_seqlens, state, state_indices, final_state,
                    output_final_state, scale, slot_stride, out, workspace, stream,
                    cuda_core_path, chunk_prefill, qk_l2norm, state_layout)


def chunk_prefill_act(q, k, v, a, A_log, dt_bias, beta, cu_seqlens, *, lower_bound=None,
                      state=None, state_indices=None, final_state=None, output_final_state=True,
                      scale=None, slot_stride=0, out=None, workspace=None, stream=None,
                      cuda_core_path=False, qk_l2norm=False, state_layout="kv"):
    """Chunked KDA prefill with the gate computed in the kernel (kda_chunk_prefill_act):
    ``g = max(-exp(A_log[h]) * softplus(a + dt_bias[h]), lower_bound)``.

    a [>=T, Hv, K] in the dtype of q/k/v; A_log [Hv] fp32; dt_bias [Hv, K] fp32 or None;
    lower_bound a float <= 0 or None.  A scalar (GDN) gate: a [>=T, Hv], dt_bias [Hv].
    Everything else as :func:`chunk_prefill`.
    """
    _need(a, "a", q.dtype)
    _need(A_log, "A_log", torch.float32)
    if dt_bias is not None:
        _need(dt_bias, "dt_bias", torch.float32)
    lb = float("-inf") if lower_bound is None else float(lower_bound)
    return _prefill(q, k, v, None, (a, A_log, dt_bias, lb), beta, cu_seqlens, state,
                    state_indices, final_state, output_final_state, scale, slot_stride, out,
                    workspace, stream, cuda_core_path, chunk_prefill_act, qk_l2norm, state_layout)


def _prefill(q, k, v, g, act, beta, cu_seqlens, state, state_indices, final_state,
             output_final_state, scale, slot_stride, out, workspace, stream, cuda_core_path,
             owner, qk_l2norm=False, state_layout="kv"):
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name)
    _need(beta, "beta", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k and v must share one dtype")
    for name, t in (("state", state), ("final_state", final_state), ("out", out)):
        if t is not None:
            _need(t, name)
    check_prefill_shapes(q, k, v, g if act is None else act[0], beta, cu_seqlens, state=state,
                         state_indices=state_indices, final_state=final_state, out=out,
                         A_log=None if act is None else act[1],
                         dt_bias=None if act is None else act[2], slot_stride=slot_stride,
                         state_layout=state_layout)
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    pool = state_indices is not None
    sdt = state.dtype if state is not None else (final_state.dtype if final_state is not None
                                                 else torch.float32)
    num_slots = 0
    if pool:
        _need(state_indices, "state_indices", torch.int32)
        if state is None:
            raise ValueError("pool mode needs the pool in `state`")
        num_slots = state.shape[0]
        final_state = state
    else:
        if state is not None:
            _need(state, "state")
        if final_state is None and output_final_state:
            final_state = torch.empty((N, Hv, *_state_dims(K, V, state_layout)), dtype=sdt,
                                      device=q.device)
    if state is not None and not pool:
        _need(state, "state")
    gate = g if act is None else act[0]
    scalar = gate.dim() == 2
    d = make_desc(num_seqs=N, total_tokens=T, Hk=Hk, Hv=Hv, K=K, V=V, qkv_dtype=q.dtype,
                  state_dtype=sdt, scale=scale, num_slots=num_slots, slot_stride=slot_stride,
                  flags=(KDA_FLAG_CUDA_CORE_PATH if cuda_core_path else 0)
                  | (KDA_FLAG_SCALAR_GATE if scalar else 0)
                  | (KDA_FLAG_QK_L2NORM if qk_l2norm else 0)
                  | (KDA_FLAG_STATE_VK if state_layout == "vk" else 0))
    if out is None:
        out = torch.empty((T, Hv, V), dtype=q.dtype, device=q.device)
    ws_size = lib.kda_chunk_prefill_workspace_size(ctypes.byref(d))
    if ws_size == 0:
        raise KdaError(1, "kda_chunk_prefill_workspace_size")
    if workspace is None or workspace.numel() < lib.kda_chunk_prefill_min_workspace_size(
            ctypes.byref(d)):
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=q.device)
    if act is None:
        rc = lib.kda_chunk_prefill(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   _ptr(cu_seqlens), _ptr(state), _ptr(state_indices),
                                   _ptr(final_state), _ptr(out), _ptr(workspace),
                                   workspace.numel(), _stream(stream))
        name = "kda_chunk_prefill"
    else:
        a, A_log, dt_bias, lb = act
        rc = lib.kda_chunk_prefill_act(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                       _ptr(A_log), _ptr(dt_bias), lb, _ptr(beta),
                                       _ptr(cu_seqlens), _ptr(state), _ptr(state_indices),
                                       _ptr(final_state), _ptr(out), _ptr(workspace),
                                       workspace.numel(), _stream(stream))
        name = "kda_chunk_prefill_act"
    if rc != 0:
        raise KdaError(rc, name)
    owner.last_workspace = workspace
    chunk_prefill.last_workspace = workspace
    return out, final_state


def decode(q, k, v, g, beta, pool, state_indices=None, *, scale=None, slot_stride=0, out=None,
           workspace=None, stream=None, qk_l2norm=False, state_layout="kv"):
    """One-token-per-row decode, updating ``pool`` [num_slots, Hv, K, V] (or [.., V, K] with
    ``state_layout="vk"``) in place.  Returns o.

    g [>=N, Hv, K] fp32, or [>=N, Hv] for a scalar (per row and head, GDN) gate."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("pool", pool)):
        _need(t, name)
    _need(g, "g", torch.float32)
    _need(beta, "beta", torch.float32)
    if state_indices is not None:
        _need(state_indices, "state_indices", torch.int32)
    if out is not None:
        _need(out, "out")
    check_decode_shapes(q, k, v, g, beta, pool, state_indices=state_indices, out=out,
                        slot_stride=slot_stride, state_layout=state_layout)
    N, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    d = make_desc(num_seqs=N, total_tokens=N, Hk=Hk, Hv=Hv, K=K, V=V, qkv_dtype=q.dtype,
                  state_dtype=pool.dtype, scale=scale, num_slots=pool.shape[0],
                  slot_stride=slot_stride,
                  flags=(KDA_FLAG_SCALAR_GATE if g.dim() == 2 else 0)
                  | (KDA_FLAG_QK_L2NORM if qk_l2norm else 0)
                  | (KDA_FLAG_STATE_VK if state_layout == "vk" else 0))
    if out is None:
        out = torch.empty((N, Hv, V), dtype=q.dtype, device=q.device)
    ws_size = lib.kda_decode_workspace_size(ctypes.byref(d))
    if ws_size == 0:
        raise KdaError(1, "kda_decode_workspace_size")
    if workspace is None or workspace.numel() < ws_size:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=q.device)
    rc = lib.kda_decode(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                        _ptr(pool), _ptr(state_indices), _ptr(out), _ptr(workspace),
                        workspace.numel(), _stream(stream))
    if rc != 0:
        raise KdaError(rc, "kda_decode")
    decode.last_workspace = workspace
    return out


def decode_draft(q, k, v, g, beta, cu_seqlens, pool, state_indices=None, *, cache=None,
                 max_steps=None, update_pool=False, scale=None, slot_stride=0, out=None,
                 workspace=None, stream=None, qk_l2norm=False, state_layout="kv"):
    """Speculative draft steps (kda_decode_draft).  Request n runs its tokens
    cu_seqlens[n]..cu_seqlens[n+1]-1 from pool[slot n]; the state after step j goes to
    ``cache[n].view(-1)[j*Hv*K*V:(j+1)*Hv*K*V]`` when ``cache`` is given: a tensor whose
    first dimension is the request and whose row pitch (``cache.stride(0)`` elements) is
    passed to the kernel as is.  The pool row gets the last state only if ``update_pool``.
    Returns o [T, Hv, V]."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("pool", pool)):
        _need(t, name)
    _need(g, "g", torch.float32)
    _need(beta, "beta", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    if state_indices is not None:
        _need(state_indices, "state_indices", torch.int32)
    if out is not None:
        _need(out, "out")
    check_decode_shapes(q, k, v, g, beta, pool, state_indices=state_indices, out=out,
                        slot_stride=slot_stride, cu_seqlens=cu_seqlens, state_layout=state_layout)
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    if max_steps is None:
        max_steps = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 1
    pitch = 0
    if cache is not None:
        if not isinstance(cache, torch.Tensor) or not cache.is_cuda or cache.dtype != pool.dtype:
            raise TypeError("cache must be a CUDA tensor of the pool's dtype")
        pitch = cache.stride(0)
        step = Hv * K * V
        avail = cache.untyped_storage().nbytes() // cache.element_size() - cache.storage_offset()
        if cache.dim() < 1 or cache.shape[0] < N or pitch < max_steps * step or \
                (N > 0 and (N - 1) * pitch + max_steps * step > avail):
            raise ValueError(f"cache must hold {N} requests of {max_steps} states "
                             f"({step} elements each) at its row pitch {pitch}")
    d = make_desc(num_seqs=N, total_tokens=T, Hk=Hk, Hv=Hv, K=K, V=V, qkv_dtype=q.dtype,
                  state_dtype=pool.dtype, scale=scale, num_slots=pool.shape[0],
                  slot_stride=slot_stride,
                  flags=(KDA_FLAG_SCALAR_GATE if g.dim() == 2 else 0)
                  | (KDA_FLAG_QK_L2NORM if qk_l2norm else 0)
                  | (KDA_FLAG_STATE_VK if state_layout == "vk" else 0))
    if out is None:
        out = torch.empty((T, Hv, V), dtype=q.dtype, device=q.device)
    ws_size = lib.kda_decode_workspace_size(ctypes.byref(d))
    if ws_size == 0:
        raise KdaError(1, "kda_decode_workspace_size")
    if workspace is None or workspace.numel() < ws_size:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=q.device)
    rc = lib.kda_decode_draft(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              _ptr(cu_seqlens), _ptr(pool), _ptr(state_indices), _ptr(cache),
                              pitch, int(max_steps), 1 if update_pool else 0, _ptr(out),
                              _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != 0:
        raise KdaError(rc, "kda_decode_draft")
    decode_draft.last_workspace = workspace
    return out
