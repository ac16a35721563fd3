"""The tensor-core prefill's failure path, made to run on purpose without faulting the GPU.

Every wait between the kernel's warp groups is bounded; kda_set_pipeline_wait_limit sets the
bound.  At 1 ns every wait that is not already complete gives up at once: the kernel must set
KDA_DEVICE_PIPE_TIMEOUT, stop taking work, let its own loads and matrix operations finish and
return (no trap, no hang), and the next call on the same device must be correct with a clean
status word.
"""
import time

import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import api, synthetic
from oracle import kda_oracle
from tests._util import assert_items_close, assert_rows_close, to_dev

pytestmark = pytest.mark.gpu


def _call(d):
    pool = d["state"].clone()
    o, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             state=pool, state_indices=d["state_indices"])
    return o, pool


def test_wait_timeout_sets_status_returns_and_next_call_is_clean():
    w = synthetic.make([2000, 300, 70, 5], Hk=2, Hv=4, K=128, V=128, seed=51, state="pool",
                       num_slots=5)
    d = to_dev(w)
    torch.cuda.synchronize()
    api.set_pipeline_wait_limit(1)
    try:
        t0 = time.perf_counter()
        _call(d)
        bits = kda.read_device_status(kda.chunk_prefill.last_workspace)  # synchronises
        dt = time.perf_counter() - t0
    finally:
        api.set_pipeline_wait_limit(0)
    assert bits & api.KDA_DEVICE_PIPE_TIMEOUT
    # no wait ran to its full 2 s bound: the drains found everything they waited for
    assert dt < 1.5, dt
    o, pool = _call(d)
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    o_ref, pool_ref = kda_oracle.recurrence(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens,
                                            scale=w.scale, state=w.state,
                                            state_indices=w.state_indices)
    assert_items_close(o, o_ref, w.cu_seqlens.tolist(), torch.bfloat16, "o")
    slots = w.state_indices.long()
    assert_rows_close(pool[slots.cuda()], pool_ref[slots.numpy()], torch.bfloat16, "pool rows")
