"""GPU parity of the prefill with the in-kernel gate activation
(kda_chunk_prefill_act: ``g = max(-exp(A_log) softplus(a + dt_bias), lower_bound)``)
against the fp64 oracle, through the C ABI.  Same bars as the plain prefill: relative L2
1e-2 with bf16 inputs, 1e-4 with fp32 inputs, finite outputs, pool == dense bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from oracle import kda_oracle
from tests._util import assert_close, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _oracle(w, a, A_log, dt_bias, lb=None, pool_mode=True):
    g = kda_oracle.gate_activation(a[:w.T], A_log, dt_bias, lb)
    return kda_oracle.recurrence(w.q, w.k, w.v, g, w.beta, w.cu_seqlens, scale=w.scale,
                                 state=w.state,
                                 state_indices=w.state_indices if pool_mode else None)


def _run(d, a, A_log, dt_bias, lb=None, **kw):
    return kda.chunk_prefill_act(d["q"], d["k"], d["v"], a.cuda(), A_log.cuda(),
                                 None if dt_bias is None else dt_bias.cuda(), d["beta"],
                                 d["cu_seqlens"], lower_bound=lb, **kw)


@pytest.mark.parametrize("cuda_core", [False, True])
def test_act_pool_bf16_matches_oracle(cuda_core):
    w = synthetic.pool_varlen()
    a, A_log, dt_bias = synthetic.gate_act_inputs(w.T, 8, 128, seed=3)
    d = to_dev(w)
    o, pool = _run(d, a, A_log, dt_bias, state=d["state"], state_indices=d["state_indices"],
                   cuda_core_path=cuda_core)
    torch.cuda.synchronize()
    assert kda.read_device_status(kda.chunk_prefill_act.last_workspace) == 0
    o_ref, pool_ref = _oracle(w, a, A_log, dt_bias)
    slots = torch.where(d["state_indices"] >= 0, d["state_indices"],
                        torch.full_like(d["state_indices"], pool.shape[0] - 1)).long().cpu()
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(pool[slots.cuda()], pool_ref[slots.numpy()], torch.bfloat16, "pool rows")


def test_act_matches_explicit_gate_path():
    # the same gate given as fp32 g to kda_chunk_prefill: both paths agree closely
    w = synthetic.pool_varlen(seed=12)
    a, A_log, dt_bias = synthetic.gate_act_inputs(w.T, 8, 128, seed=4)
    d = to_dev(w)
    g = torch.from_numpy(kda_oracle.gate_activation(a, A_log, dt_bias)).float().cuda()
    o1, p1 = kda.chunk_prefill(d["q"], d["k"], d["v"], g, d["beta"], d["cu_seqlens"],
                               state=d["state"].clone(), state_indices=d["state_indices"])
    o2, p2 = _run(d, a, A_log, dt_bias, state=d["state"].clone(),
                  state_indices=d["state_indices"])
    torch.cuda.synchronize()
    assert rel_l2(o2.double().cpu(), o1.double().cpu()) < 2e-3
    assert rel_l2(p2.double().cpu(), p1.double().cpu()) < 2e-3


def test_act_fp32_cuda_core_dense_no_bias():
    w = synthetic.tiny_varlen()
    a, A_log, _ = synthetic.gate_act_inputs(w.T, 2, 64, dtype=torch.float32, seed=5)
    d = to_dev(w)
    o, ht = _run(d, a, A_log, None, state=d["state"], scale=w.scale)
    o_ref, ht_ref = _oracle(w, a, A_log, None, pool_mode=False)
    assert_close(o, o_ref, torch.float32, "o")
    assert_close(ht, ht_ref, torch.float32, "ht")


@pytest.mark.parametrize("lb", [-0.05, -1.0])
def test_act_lower_bound(lb):
    w = synthetic.pool_varlen(seed=13)
    a, A_log, dt_bias = synthetic.gate_act_inputs(w.T, 8, 128, seed=6)
    a = (a.float() + 4.0).to(torch.bfloat16)  # large gates, so the bound binds
    d = to_dev(w)
    o, pool = _run(d, a, A_log, dt_bias, lb=lb, state=d["state"],
                   state_indices=d["state_indices"])
    torch.cuda.synchronize()
    o_ref, _ = _oracle(w, a, A_log, dt_bias, lb)
    assert_close(o, o_ref, torch.bfloat16, "o")
    g = kda_oracle.gate_activation(a, A_log, dt_bias)
    assert np.mean(g < lb) > 0.1  # the bound is active on a good share of the gates


def test_act_large_decay_unsafe_channels():
    # A up to ~e^9: sub-chunk gate products underflow, so the exact pairwise path runs
    w = synthetic.make([200, 64, 17], Hk=2, Hv=4, K=128, V=128, seed=21, state="pool",
                       num_slots=8)
    a, _, dt_bias = synthetic.gate_act_inputs(w.T, 4, 128, seed=7)
    A_log = torch.tensor([0.0, 3.0, 6.0, 9.0])
    d = to_dev(w)
    o, pool = _run(d, a, A_log, dt_bias, state=d["state"], state_indices=d["state_indices"])
    torch.cuda.synchronize()
    o_ref, pool_ref = _oracle(w, a, A_log, dt_bias)
    assert_close(o, o_ref, torch.bfloat16, "o")
    slots = d["state_indices"].long().cpu()
    assert_close(pool[slots.cuda()], pool_ref[slots.numpy()], torch.bfloat16, "pool rows")


def test_act_pool_equals_dense_bitwise():
    w = synthetic.pool_varlen(seed=14)
    a, A_log, dt_bias = synthetic.gate_act_inputs(w.T, 8, 128, seed=8)
    d = to_dev(w)
    pool = d["state"]
    slots = torch.where(d["state_indices"] >= 0, d["state_indices"],
                        torch.full_like(d["state_indices"], pool.shape[0] - 1)).long()
    o_dense, ht_dense = _run(d, a, A_log, dt_bias, state=pool[slots].clone())
    o_pool, _ = _run(d, a, A_log, dt_bias, state=pool, state_indices=d["state_indices"])
    torch.cuda.synchronize()
    assert torch.equal(o_pool, o_dense)
    assert torch.equal(pool[slots], ht_dense)


def test_act_rejects_positive_lower_bound():
    w = synthetic.pool_varlen()
    a, A_log, dt_bias = synthetic.gate_act_inputs(w.T, 8, 128, seed=3)
    d = to_dev(w)
    with pytest.raises(kda.KdaError):
        _run(d, a, A_log, dt_bias, lb=0.5, state=d["state"], state_indices=d["state_indices"])
