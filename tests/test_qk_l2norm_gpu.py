"""GPU parity of the in-kernel q/k L2 normalisation (KDA_FLAG_QK_L2NORM):
x / max(||x||, 1e-12) per (token, head), the step the pages' callers run before the prefill
(sglang PR 27488 digest, 关键源码片段 CuteDSLKDAKernel.extend).  Inputs here are NOT
normalised; the oracle normalises them in fp64.  Bars: relative L2 1e-2 (bf16), 1e-4 (fp32).
"""
import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from oracle import kda_oracle
from tests._util import assert_close, to_dev

pytestmark = pytest.mark.gpu

# The kernels normalise in fp32 (the tensor-core kernel then re-rounds to bf16), the reference
# in fp64: q and k themselves then differ by up to one bf16 step in some elements, on top of
# the bf16 rounding every other test shares.  The whole-tensor bar (relative L2 1e-2) is
# unchanged; the per-element bound gets that one extra rounding step of room.
MAX_RMS_NORM = 0.15


def _raw_qk(w, seed, scale=3.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(w.q.shape, generator=g) * scale).to(w.q.dtype)
    k = (torch.randn(w.k.shape, generator=g) * scale).to(w.k.dtype)
    return q, k


def _unit(x, rounded):
    """Normalised rows; ``rounded``: cast back to the input dtype first, as the tensor-core
    kernel (like a caller's normalise-then-cast) does."""
    y = kda_oracle.l2norm(x)
    return torch.from_numpy(y).to(x.dtype).double().numpy() if rounded else y


def _oracle(w, q, k, pool_mode=True, g=None, rounded=True):
    return kda_oracle.recurrence(_unit(q, rounded), _unit(k, rounded), w.v,
                                 w.g if g is None else g, w.beta, w.cu_seqlens, scale=w.scale,
                                 state=w.state,
                                 state_indices=w.state_indices if pool_mode else None)


def _slots(d, pool):
    i = d["state_indices"]
    return torch.where(i >= 0, i, torch.full_like(i, pool.shape[0] - 1)).long()


@pytest.mark.parametrize("cuda_core", [False, True])
def test_l2norm_pool_bf16(cuda_core):
    w = synthetic.pool_varlen(seed=31)
    q, k = _raw_qk(w, 1)
    d = to_dev(w)
    o, pool = kda.chunk_prefill(q.cuda(), k.cuda(), d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"],
                                cuda_core_path=cuda_core, qk_l2norm=True)
    torch.cuda.synchronize()
    o_ref, pool_ref = _oracle(w, q, k, rounded=not cuda_core)
    s = _slots(d, pool)
    assert_close(o, o_ref, torch.bfloat16, "o", max_rms=MAX_RMS_NORM)
    assert_close(pool[s], pool_ref[s.cpu().numpy()], torch.bfloat16, "pool rows",
                 max_rms=MAX_RMS_NORM)


def test_l2norm_fp32_dense():
    w = synthetic.tiny_varlen(seed=4)
    q, k = _raw_qk(w, 2)
    d = to_dev(w)
    o, ht = kda.chunk_prefill(q.cuda(), k.cuda(), d["v"], d["g"], d["beta"], d["cu_seqlens"],
                              state=d["state"], scale=w.scale, qk_l2norm=True)
    o_ref, ht_ref = _oracle(w, q, k, pool_mode=False, rounded=False)
    assert_close(o, o_ref, torch.float32, "o")
    assert_close(ht, ht_ref, torch.float32, "ht")


def test_l2norm_large_decay_pairwise_path():
    w = synthetic.make([150, 66], Hk=2, Hv=4, K=128, V=128, seed=32, gate="large",
                       gate_scale_log_max=6.9, state="pool", num_slots=4)
    q, k = _raw_qk(w, 3, scale=0.2)
    d = to_dev(w)
    o, pool = kda.chunk_prefill(q.cuda(), k.cuda(), d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"],
                                qk_l2norm=True)
    torch.cuda.synchronize()
    o_ref, pool_ref = _oracle(w, q, k)
    assert_close(o, o_ref, torch.bfloat16, "o", max_rms=MAX_RMS_NORM)


def test_l2norm_with_gate_activation():
    w = synthetic.pool_varlen(seed=33)
    q, k = _raw_qk(w, 4)
    a, A_log, dt_bias = synthetic.gate_act_inputs(w.T, 8, 128, seed=9)
    d = to_dev(w)
    o, _ = kda.chunk_prefill_act(q.cuda(), k.cuda(), d["v"], a.cuda(), A_log.cuda(),
                                 dt_bias.cuda(), d["beta"], d["cu_seqlens"], state=d["state"],
                                 state_indices=d["state_indices"], qk_l2norm=True)
    torch.cuda.synchronize()
    o_ref, _ = _oracle(w, q, k, g=kda_oracle.gate_activation(a, A_log, dt_bias))
    assert_close(o, o_ref, torch.bfloat16, "o", max_rms=MAX_RMS_NORM)


def test_l2norm_decode():
    N, Hk, Hv, K, V = 80, 4, 8, 128, 128
    w = synthetic.make([1] * N, Hk=Hk, Hv=Hv, K=K, V=V, seed=34, state="pool", num_slots=96)
    q, k = _raw_qk(w, 5)
    d = to_dev(w)
    pool = d["state"]
    o = kda.decode(q.cuda(), k.cuda(), d["v"], d["g"], d["beta"], pool, d["state_indices"],
                   qk_l2norm=True)
    torch.cuda.synchronize()
    o_ref, pool_ref = kda_oracle.decode(_unit(q, False), _unit(k, False), w.v, w.g,
                                        w.beta, pool=w.state, state_indices=w.state_indices)
    s = d["state_indices"].long()
    assert_close(o, o_ref, torch.bfloat16, "o", max_rms=MAX_RMS_NORM)
    assert_close(pool[s], pool_ref[s.cpu().numpy()], torch.bfloat16, "pool rows",
                 max_rms=MAX_RMS_NORM)
