"""GPU parity of the scalar-gate (gated delta net, GDN) form: one log-decay per (token,
v-head) shared by every key channel (KDA_FLAG_SCALAR_GATE), through the same prefill
kernels and pool I/O and through decode, against the fp64 oracle.  The pages ship this
twin with its pool-vs-dense test (sglang PR 30169 digest, 关键源码片段).  Bars as for the
per-channel gate: relative L2 1e-2 (bf16) / 1e-4 (fp32), pool == dense bit for bit.
"""
import numpy as np
import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from oracle import kda_oracle
from tests._util import assert_close, to_dev

pytestmark = pytest.mark.gpu


def _slots(d, pool):
    i = d["state_indices"]
    return torch.where(i >= 0, i, torch.full_like(i, pool.shape[0] - 1)).long()


def _oracle(w, g, pool_mode=True):
    return kda_oracle.recurrence(w.q, w.k, w.v, g, w.beta, w.cu_seqlens, scale=w.scale,
                                 state=w.state,
                                 state_indices=w.state_indices if pool_mode else None)


@pytest.mark.parametrize("cuda_core", [False, True])
def test_scalar_gate_pool_matches_oracle(cuda_core):
    w = synthetic.pool_varlen(seed=21)
    g2 = synthetic.scalar_gate_inputs(w.T, 8, seed=1)
    d = to_dev(w)
    o, pool = kda.chunk_prefill(d["q"], d["k"], d["v"], g2.cuda(), d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"],
                                cuda_core_path=cuda_core)
    torch.cuda.synchronize()
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    o_ref, pool_ref = _oracle(w, g2)
    s = _slots(d, pool)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(pool[s], pool_ref[s.cpu().numpy()], torch.bfloat16, "pool rows")


@pytest.mark.parametrize("cuda_core", [False, True])
def test_scalar_gate_activation_like_the_pages_gdn_test(cuda_core):
    w = synthetic.pool_varlen(seed=22)
    a, A_log, dt_bias = synthetic.scalar_gate_inputs(w.T, 8, seed=2, act=True)
    d = to_dev(w)
    o, pool = kda.chunk_prefill_act(d["q"], d["k"], d["v"], a.cuda(), A_log.cuda(),
                                    dt_bias.cuda(), d["beta"], d["cu_seqlens"],
                                    state=d["state"], state_indices=d["state_indices"],
                                    cuda_core_path=cuda_core)
    torch.cuda.synchronize()
    o_ref, pool_ref = _oracle(w, kda_oracle.gate_activation(a, A_log, dt_bias))
    s = _slots(d, pool)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(pool[s], pool_ref[s.cpu().numpy()], torch.bfloat16, "pool rows")


def test_scalar_gate_pool_equals_dense_bitwise():
    w = synthetic.pool_varlen(seed=23)
    g2 = synthetic.scalar_gate_inputs(w.T, 8, seed=3).cuda()
    d = to_dev(w)
    pool = d["state"]
    s = _slots(d, pool)
    o_dense, ht = kda.chunk_prefill(d["q"], d["k"], d["v"], g2, d["beta"], d["cu_seqlens"],
                                    state=pool[s].clone())
    o_pool, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], g2, d["beta"], d["cu_seqlens"],
                                  state=pool, state_indices=d["state_indices"])
    torch.cuda.synchronize()
    assert torch.equal(o_pool, o_dense)
    assert torch.equal(pool[s], ht)


def test_scalar_gate_heads_not_multiple_of_8_use_cuda_cores():
    w = synthetic.make([40, 131, 7], Hk=2, Hv=4, K=128, V=128, seed=24, state="pool",
                       num_slots=6)
    g2 = synthetic.scalar_gate_inputs(w.T, 4, seed=4)
    d = to_dev(w)
    desc = kda.make_desc(num_seqs=3, total_tokens=w.T, Hk=2, Hv=4, K=128, V=128,
                         qkv_dtype=torch.bfloat16, num_slots=6, flags=0x2)
    assert kda.prefill_path(desc) == 0
    o, pool = kda.chunk_prefill(d["q"], d["k"], d["v"], g2.cuda(), d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"])
    torch.cuda.synchronize()
    o_ref, pool_ref = _oracle(w, g2)
    assert_close(o, o_ref, torch.bfloat16, "o")


def test_scalar_gate_fp32_dense():
    w = synthetic.tiny_varlen(seed=3)
    g2 = synthetic.scalar_gate_inputs(w.T, 2, seed=5)
    d = to_dev(w)
    o, ht = kda.chunk_prefill(d["q"], d["k"], d["v"], g2.cuda(), d["beta"], d["cu_seqlens"],
                              state=d["state"], scale=w.scale)
    o_ref, ht_ref = _oracle(w, g2, pool_mode=False)
    assert_close(o, o_ref, torch.float32, "o")
    assert_close(ht, ht_ref, torch.float32, "ht")


def test_scalar_gate_decode():
    N, Hk, Hv, K, V = 96, 4, 8, 128, 128
    w = synthetic.make([1] * N, Hk=Hk, Hv=Hv, K=K, V=V, seed=25, state="pool", num_slots=128)
    g2 = synthetic.scalar_gate_inputs(N, Hv, seed=6)
    d = to_dev(w)
    pool = d["state"]
    o = kda.decode(d["q"], d["k"], d["v"], g2.cuda(), d["beta"], pool, d["state_indices"])
    torch.cuda.synchronize()
    o_ref, pool_ref = kda_oracle.decode(w.q, w.k, w.v, g2, w.beta, pool=w.state,
                                        state_indices=w.state_indices)
    s = d["state_indices"].long()
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(pool[s], pool_ref[s.cpu().numpy()], torch.bfloat16, "pool rows")
