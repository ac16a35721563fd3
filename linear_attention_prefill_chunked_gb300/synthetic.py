"""Seeded synthetic inputs for the KDA prefill / decode workloads.

This module only draws random inputs; it holds none of the method's
arithmetic, and both the CUDA path's tests/benchmarks and the CPU oracle take
their inputs from it.  Every draw uses a ``torch.Generator`` seeded per
workload, in a fixed order: lengths, q, k, v, gate input, beta input, states,
slot indices.

Shapes and distributions follow the workloads the KDA prefill pages test
(sglang PR 27488 digest, 关键文件 test_kda_prefill_cutedsl.py: varlen
correctness and a realistic-gate test; sglang PR 30169 digest, 关键源码片段
test_gdn_chunk_cutedsl_pool_mode_matches_dense: 5 sequences of random length
below 130, 4 k-heads / 8 v-heads, 128x128 heads, a random-permutation slot
pool).  q and k are drawn N(0,1), L2-normalised per head in fp32
(x / max(||x||, 1e-12)) and then cast, exactly like the callers on those pages
normalise outside the kernel (PR 27488 digest, CuteDSLKDAKernel.extend).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

BF16 = torch.bfloat16
F32 = torch.float32


@dataclass
class Workload:
    name: str
    q: torch.Tensor            # [T, Hk, K]
    k: torch.Tensor            # [T, Hk, K]
    v: torch.Tensor            # [T, Hv, V]
    g: torch.Tensor            # [T, Hv, K] fp32 log-decay
    beta: torch.Tensor         # [T, Hv] fp32
    cu_seqlens: torch.Tensor   # [N+1] int32
    state: Optional[torch.Tensor]          # pool [slots,Hv,K,V] or dense [N,Hv,K,V] or None
    state_indices: Optional[torch.Tensor]  # [N] int32 or None
    scale: float
    lens: list = field(default_factory=list)

    @property
    def T(self):
        return int(self.cu_seqlens[-1])

    @property
    def N(self):
        return self.cu_seqlens.numel() - 1

    @property
    def dims(self):
        return dict(Hk=self.q.shape[1], Hv=self.v.shape[1], K=self.q.shape[2], V=self.v.shape[2])


def _normal(shape, gen, std=1.0):
    return torch.randn(*shape, generator=gen, dtype=F32) * std


def _unit(x):
    n = torch.linalg.vector_norm(x, dim=-1, keepdim=True)
    return x / torch.clamp(n, min=1e-12)


def _cu(lens):
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    if lens:
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return cu


def make(lens, *, Hk, Hv, K, V, dtype=BF16, seed=0, gate="softplus", gate_scale_log_max=None,
         state="pool", num_slots=None, state_dtype=F32, last_index_pad=False, state_std=0.1,
         g_pad_rows=0, name="custom", gen=None) -> Workload:
    """General generator used by every named workload.

    gate: "softplus"    g = -softplus(x), x ~ N(0,1)
          "large"       g = -exp(a_h) * softplus(x), a_h ~ U(0, gate_scale_log_max) per v-head
          "zero"        g = 0
    state: "pool"  -> pool of ``num_slots`` rows, indices = randperm(num_slots-1)[:N]
           "dense" -> dense [N,Hv,K,V]
           None    -> no initial state
    last_index_pad: set the last sequence's index to -1 (the sentinel slot).
    g_pad_rows: extra rows appended to g and beta (padding past T, never read).
    gen: continue drawing from this generator (after the lengths were drawn
         from it) instead of a fresh one seeded with ``seed``.
    """
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in lens]
    T = sum(lens)
    q = _unit(_normal((T, Hk, K), gen)).to(dtype)
    k = _unit(_normal((T, Hk, K), gen)).to(dtype)
    v = _normal((T, Hv, V), gen).to(dtype)
    if gate == "large":
        a = torch.rand(Hv, generator=gen, dtype=F32) * gate_scale_log_max
        x = _normal((T + g_pad_rows, Hv, K), gen)
        g = -torch.exp(a).view(1, Hv, 1) * torch.nn.functional.softplus(x)
    elif gate == "zero":
        g = torch.zeros(T + g_pad_rows, Hv, K, dtype=F32)
    else:
        g = -torch.nn.functional.softplus(_normal((T + g_pad_rows, Hv, K), gen))
    beta = torch.sigmoid(_normal((T + g_pad_rows, Hv), gen))
    st = None
    idx = None
    N = len(lens)
    if state == "pool":
        st = _normal((num_slots, Hv, K, V), gen, state_std).to(state_dtype)
        idx = torch.randperm(num_slots - 1, generator=gen)[:N].to(torch.int32)
        if last_index_pad and N > 0:
            idx[-1] = -1
    elif state == "dense":
        st = _normal((N, Hv, K, V), gen, state_std).to(state_dtype)
    return Workload(name, q, k, v, g.contiguous(), beta.contiguous(), _cu(lens), st, idx,
                    K ** -0.5, lens)


# ----------------------------------------------------------------------------
# Named workloads (the five configurations the path is specified on).
# ----------------------------------------------------------------------------

def tiny_varlen(seed=0) -> Workload:
    """3 sequences [1, 37, 130]; Hk=Hv=2, K=V=64; fp32 q/k/v; dense fp32 h0 N(0, 0.1)."""
    return make([1, 37, 130], Hk=2, Hv=2, K=64, V=64, dtype=F32, seed=seed, state="dense",
                name="tiny_varlen_fp32_3seq_K64")


def pool_varlen(state_dtype=F32, seed=11) -> Workload:
    """5 sequences, lengths uniform in [1, 130); Hk=4, Hv=8, K=V=128; bf16 q/k/v;
    16-slot pool N(0, 0.1); random slots, last sequence index -1 (sentinel 15)."""
    gen = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, 130, (5,), generator=gen).tolist()
    return make(lens, Hk=4, Hv=8, K=128, V=128, dtype=BF16, gen=gen, state="pool",
                num_slots=16, state_dtype=state_dtype, last_index_pad=True,
                name=f"pool_varlen_5seq_Hv8_{'bf16' if state_dtype == BF16 else 'fp32'}_pool")


def large_decay(seed=0, num_seqs=8, seqlen=4096) -> Workload:
    """8 x 4096 tokens; Hk=Hv=32, K=V=128; bf16; g = -exp(a_h) softplus(x), a_h ~ U(0, ln 1000)."""
    return make([seqlen] * num_seqs, Hk=32, Hv=32, K=128, V=128, dtype=BF16, seed=seed,
                gate="large", gate_scale_log_max=math.log(1000.0), state="pool", num_slots=64,
                name=f"large_decay_{num_seqs}x{seqlen}_Hv32")


def throughput_lengths(seed=0, num_seqs=16, total=32768, lo=64, hi=8192, gen=None):
    """Lengths log-uniform in [lo, hi], rescaled to ``total`` (floor, >= 1, residual to the longest)."""
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    u = torch.rand(num_seqs, generator=gen, dtype=torch.float64)
    lf = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    lf = lf * total / lf.sum()
    L = torch.clamp(torch.floor(lf), min=1).long()
    L[torch.argmax(L)] += total - int(L.sum())
    return L.tolist()


def throughput(seed=0) -> Workload:
    """32768 tokens as 16 log-uniform sequences; Hk=Hv=32, K=V=128; bf16; 256-slot fp32 pool."""
    gen = torch.Generator().manual_seed(seed)
    lens = throughput_lengths(gen=gen)
    return make(lens, Hk=32, Hv=32, K=128, V=128, dtype=BF16, gen=gen, state="pool",
                num_slots=256, name="throughput_T32768_16seq_Hv32_K128")


def decode_batch(seed=0, num_rows=4096, num_pad=64, num_slots=8192, Hv=32, K=128, V=128,
                 device="cpu", pool_device=None, pad_shuffled=False) -> Workload:
    """4096 rows of one token; the last ``num_pad`` rows are padding (-1 -> sentinel).

    The pool ([num_slots, Hv, K, V] fp32, N(0, 0.1)) is large (16 GiB at the
    default sizes); it is drawn on ``pool_device`` with a generator of that
    device seeded from ``seed`` so it never has to pass through host memory.
    """
    gen = torch.Generator().manual_seed(seed)
    lens = [1] * num_rows
    T = num_rows
    q = _unit(_normal((T, Hv, K), gen)).to(BF16)
    k = _unit(_normal((T, Hv, K), gen)).to(BF16)
    v = _normal((T, Hv, V), gen).to(BF16)
    g = -torch.nn.functional.softplus(_normal((T, Hv, K), gen))
    beta = torch.sigmoid(_normal((T, Hv), gen))
    pdev = torch.device(pool_device or device)
    pgen = torch.Generator(device=pdev).manual_seed(seed + 7)
    pool = torch.empty((num_slots, Hv, K, V), dtype=F32, device=pdev)
    step = max(1, num_slots // 16)
    for s in range(0, num_slots, step):
        e = min(num_slots, s + step)
        pool[s:e].normal_(0.0, 0.1, generator=pgen)
    real = torch.randperm(num_slots - 1, generator=gen)[: num_rows - num_pad].to(torch.int32)
    idx = torch.cat([real, torch.full((num_pad,), -1, dtype=torch.int32)])
    if pad_shuffled:
        idx = idx[torch.randperm(num_rows, generator=gen)]
    return Workload(f"decode_{num_rows}rows_{num_slots}slots", q, k, v, g, beta, _cu(lens),
                    pool, idx, K ** -0.5, lens)


WORKLOADS = {
    "tiny_varlen": tiny_varlen,
    "pool_varlen": pool_varlen,
    "large_decay": large_decay,
    "throughput": throughput,
    "decode_batch": decode_batch,
}


def gate_act_inputs(T, Hv, K, *, dtype=BF16, seed=0, rows=None, A_max=16.0):
    """Inputs of the in-kernel gate activation, drawn like the pages' gate tests
    (sglang PR 30169 digest, 关键源码片段, the GDN pool test: A ~ U(0, 16) per head,
    dt log-uniform in [1e-3, 1e-1] and floored at 1e-4, dt_bias the value whose
    softplus is dt), with a key-channel axis for the KDA gate.

    Returns ``(a, A_log, dt_bias)``: a [rows or T, Hv, K] ~ N(0, 1) in ``dtype``;
    A_log [Hv] fp32; dt_bias [Hv, K] fp32.  Drawn from its own generator (seed)
    so that the workloads of :func:`make` keep their values.
    """
    gen = torch.Generator().manual_seed(seed + 7919)
    n = T if rows is None else rows
    a = _normal((n, Hv, K), gen).to(dtype)
    A = torch.rand(Hv, generator=gen, dtype=F32) * A_max
    A_log = torch.log(torch.clamp(A, min=1e-6))
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt = torch.exp(torch.rand(Hv, K, generator=gen, dtype=F32) * (hi - lo) + lo).clamp(min=1e-4)
    dt_bias = torch.log(torch.expm1(dt))  # softplus(dt_bias) = dt
    return a.contiguous(), A_log.contiguous(), dt_bias.contiguous()


def scalar_gate_inputs(T, Hv, *, dtype=BF16, seed=0, act=False, A_max=16.0):
    """Scalar (gated-delta-net) gate inputs, one value per (token, v-head).

    act=False: g [T, Hv] fp32 = -softplus(x), x ~ N(0, 1).
    act=True: ``(a, A_log, dt_bias)`` drawn like the pages' GDN pool test (sglang PR 30169
    digest, 关键源码片段): a [T, Hv] ~ N(0, 1) in ``dtype``, A ~ U(0, 16) -> A_log [Hv],
    dt log-uniform in [1e-3, 1e-1] (floored at 1e-4) -> dt_bias [Hv] with softplus(dt_bias) = dt.
    """
    gen = torch.Generator().manual_seed(seed + 104729)
    if not act:
        return (-torch.nn.functional.softplus(_normal((T, Hv), gen))).contiguous()
    a = _normal((T, Hv), gen).to(dtype)
    A_log = torch.log(torch.clamp(torch.rand(Hv, generator=gen, dtype=F32) * A_max, min=1e-6))
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt = torch.exp(torch.rand(Hv, generator=gen, dtype=F32) * (hi - lo) + lo).clamp(min=1e-4)
    return a.contiguous(), A_log.contiguous(), torch.log(torch.expm1(dt)).contiguous()
