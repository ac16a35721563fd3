"""GPU parity of the speculative draft-step decode with a per-step state cache
(kda_decode_draft) against the fp64 oracle: each request's draft tokens run in order from
its pool row; the state after step j must equal the oracle's state after the first j+1
tokens, read through the explicit per-request pitch (sglang PR 37317 digest, 实现拆解
item 2).  Bars: relative L2 1e-2 (bf16 inputs), no NaN/Inf.
"""
import numpy as np
import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from oracle import kda_oracle
from tests._util import assert_close, to_dev

pytestmark = pytest.mark.gpu

LENS = [1, 2, 3, 4, 1, 3]
HK, HV, K, V = 4, 8, 128, 128


def _workload(seed=41):
    return synthetic.make(LENS, Hk=HK, Hv=HV, K=K, V=V, seed=seed, state="pool", num_slots=16)


def _oracle_steps(w, n):
    """Oracle o rows and per-step states of request n."""
    cu = w.cu_seqlens.tolist()
    a, b = cu[n], cu[n + 1]
    slot = int(w.state_indices[n])
    S0 = w.state[slot:slot + 1]
    o, _ = kda_oracle.recurrence(w.q[a:b], w.k[a:b], w.v[a:b], w.g[a:b], w.beta[a:b],
                                 [0, b - a], scale=w.scale, state=S0)
    steps = []
    for j in range(b - a):
        _, fin = kda_oracle.recurrence(w.q[a:a + j + 1], w.k[a:a + j + 1], w.v[a:a + j + 1],
                                       w.g[a:a + j + 1], w.beta[a:a + j + 1], [0, j + 1],
                                       scale=w.scale, state=S0)
        steps.append(fin[0])
    return o, steps


@pytest.mark.parametrize("update_pool", [False, True])
def test_draft_steps_match_oracle_prefixes(update_pool):
    w = _workload()
    d = to_dev(w)
    pool = d["state"]
    before = pool.clone()
    max_steps, pitch_steps = 4, 5  # a pitch wider than max_steps: read it, do not infer it
    cache = torch.full((len(LENS), pitch_steps, HV, K, V), float("nan"), device="cuda")
    o = kda.decode_draft(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], pool,
                         d["state_indices"], cache=cache, max_steps=max_steps,
                         update_pool=update_pool)
    torch.cuda.synchronize()
    assert kda.read_device_status(kda.decode_draft.last_workspace) == 0
    cu = w.cu_seqlens.tolist()
    for n in range(len(LENS)):
        o_ref, steps = _oracle_steps(w, n)
        assert_close(o[cu[n]:cu[n + 1]], o_ref, torch.bfloat16, f"o of request {n}")
        for j, st in enumerate(steps):
            assert_close(cache[n, j], st, torch.bfloat16, f"state after step {j} of request {n}")
        assert torch.isnan(cache[n, len(steps):]).all()  # steps past the request: untouched
        slot = int(w.state_indices[n])
        if update_pool:
            assert_close(pool[slot], steps[-1], torch.bfloat16, f"pool row of request {n}")
        else:
            assert torch.equal(pool[slot], before[slot])


def test_single_steps_equal_plain_decode_bitwise():
    w = synthetic.make([1] * 40, Hk=HK, Hv=HV, K=K, V=V, seed=42, state="pool", num_slots=48)
    d = to_dev(w)
    p1, p2 = d["state"].clone(), d["state"].clone()
    o1 = kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], p1, d["state_indices"])
    o2 = kda.decode_draft(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], p2,
                          d["state_indices"], update_pool=True, max_steps=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(p1, p2)


def test_request_longer_than_max_steps_is_flagged_and_skipped():
    w = _workload(seed=43)
    d = to_dev(w)
    cache = torch.zeros((len(LENS), 3, HV, K, V), device="cuda")
    o = torch.full((w.T, HV, V), 7.0, dtype=torch.bfloat16, device="cuda")
    kda.decode_draft(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["state"],
                     d["state_indices"], cache=cache, max_steps=3, out=o)
    torch.cuda.synchronize()
    assert kda.read_device_status(kda.decode_draft.last_workspace) & 0x2  # BAD_SEQLENS
    cu = w.cu_seqlens.tolist()
    assert torch.all(o[cu[3]:cu[4]] == 7.0)  # the 4-token request was skipped
    o_ref, _ = _oracle_steps(w, 2)
    assert_close(o[cu[2]:cu[3]], o_ref, torch.bfloat16, "o of a request within the limit")
