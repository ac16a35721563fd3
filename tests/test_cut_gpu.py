"""Long sequences cut in two (tensor-core prefill), through the C ABI, against the oracle.

A sequence much longer than the batch's share per SM is cut at a chunk boundary: its head
runs as usual; its tail runs from a zero state and, with the values set to zero, from the
identity matrix; a combine step finishes the tail exactly (the state is affine in its start
value: S_end = M S_p + S_loc, o_t = o_loc_t + S_p^T y_t).  The fp64 model of that algebra is
checked against the oracle in tests/test_chunked_model.py; here the kernels are.
"""
import ctypes

import numpy as np
import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from oracle import kda_oracle
from tests._util import assert_close, assert_items_close, assert_rows_close, to_dev

pytestmark = pytest.mark.gpu


def _cuts(ws):
    """Number of sequences the planning step cut (the fourth word of the workspace header)."""
    return int(ws[12:16].cpu().view(torch.int32)[0])


def _run(w, pool_mode=True, workspace=None, **kw):
    d = to_dev(w)
    st = d["state"]
    o, fin = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                               state=st, state_indices=d["state_indices"] if pool_mode else None,
                               workspace=workspace, **kw)
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    return o, (st if pool_mode else fin), kda.chunk_prefill.last_workspace


def _check_pool(w, o, pool, dtype=torch.bfloat16):
    o_ref, pool_ref = kda_oracle.recurrence(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens,
                                            scale=w.scale, state=w.state,
                                            state_indices=w.state_indices)
    assert_items_close(o, o_ref, w.cu_seqlens.tolist(), dtype, "o")
    slots = torch.where(w.state_indices >= 0, w.state_indices,
                        torch.full_like(w.state_indices, w.state.shape[0] - 1)).long()
    assert_rows_close(pool[slots.cuda()], pool_ref[slots.numpy()], dtype, "written pool rows")
    untouched = torch.ones(w.state.shape[0], dtype=torch.bool)
    untouched[slots] = False
    assert torch.equal(pool[untouched.cuda()].cpu(), w.state[untouched])


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_one_long_sequence_is_cut_and_matches_oracle(state_dtype):
    w = synthetic.make([3000, 100, 37, 0], Hk=2, Hv=4, K=128, V=128, seed=41, state="pool",
                       num_slots=8, state_dtype=state_dtype, last_index_pad=True)
    o, pool, ws = _run(w)
    assert _cuts(ws) == 1
    _check_pool(w, o, pool)


def test_several_cuts_pool_equals_dense_bitwise():
    """Four long sequences cut (the most the workspace allows), a fifth long one and the short
    ones run whole; pool and dense calls cut alike and agree bit for bit."""
    w = synthetic.make([2000, 1500, 1300, 1100, 900, 20, 64], Hk=1, Hv=2, K=128, V=128, seed=42,
                       state="pool", num_slots=9)
    o_pool, pool, ws = _run(w)
    assert _cuts(ws) == 4
    _check_pool(w, o_pool, pool)
    d = to_dev(w)
    slots = w.state_indices.long().cuda()
    h0 = d["state"][slots].clone()
    o_dense, ht = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                    state=h0)
    assert _cuts(kda.chunk_prefill.last_workspace) == 4
    assert torch.equal(o_dense, o_pool)
    assert torch.equal(ht, pool[slots])


def test_cut_and_whole_runs_agree_and_min_workspace_equals_noalloc():
    """With the least workspace nothing is cut: the same within the tolerance, and bit for bit
    what the allocation-free entry point (whose scratch has no room for cuts) computes."""
    w = synthetic.make([2500, 300, 64], Hk=2, Hv=4, K=128, V=128, seed=43, state="pool",
                       num_slots=6)
    o_cut, pool_cut, ws = _run(w)
    assert _cuts(ws) == 1
    desc = kda.make_desc(num_seqs=w.N, total_tokens=w.T, Hk=2, Hv=4, K=128, V=128,
                         qkv_dtype=torch.bfloat16, num_slots=6)
    small = torch.empty(kda.prefill_min_workspace_size(desc), dtype=torch.uint8, device="cuda")
    assert small.numel() < kda.prefill_workspace_size(desc)
    o_whole, pool_whole, ws2 = _run(w, workspace=small)
    assert _cuts(ws2) == 0
    assert_close(o_cut, o_whole.double().cpu().numpy(), torch.bfloat16, "o cut vs whole")
    _check_pool(w, o_whole, pool_whole)
    # the allocation-free entry point on the same inputs
    d = to_dev(w)
    pool_na = d["state"]
    o_na = torch.empty_like(o_whole)
    lib = kda.load()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.kda_chunk_prefill_noalloc(ctypes.byref(desc), P(d["q"]), P(d["k"]), P(d["v"]),
                                       P(d["g"]), P(d["beta"]), P(d["cu_seqlens"]), P(pool_na),
                                       P(d["state_indices"]), None, P(o_na),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(o_na, o_whole) and torch.equal(pool_na, pool_whole)


def test_cut_dense_without_final_state_and_zero_initial_state():
    w = synthetic.make([2600, 70], Hk=2, Hv=2, K=128, V=128, seed=44, state=None)
    d = to_dev(w)
    o, fin = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                               output_final_state=False)
    assert fin is None
    assert _cuts(kda.chunk_prefill.last_workspace) == 1
    o_ref, _ = kda_oracle.recurrence(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, scale=w.scale)
    assert_items_close(o, o_ref, w.cu_seqlens.tolist(), torch.bfloat16, "o")


def test_cut_tail_too_long_for_the_scratch_runs_whole_then_cut_fits():
    """A tail longer than the 8192 y rows of the workspace is not cut; a shorter one is."""
    w = synthetic.make([20000], Hk=1, Hv=2, K=128, V=128, seed=45, state="pool", num_slots=2)
    o, pool, ws = _run(w)
    assert _cuts(ws) == 0
    _check_pool(w, o, pool)
    w = synthetic.make([16000], Hk=1, Hv=2, K=128, V=128, seed=46, state="pool", num_slots=2)
    o, pool, ws = _run(w)
    assert _cuts(ws) == 1
    _check_pool(w, o, pool)


def test_cut_at_large_decay():
    """Per-chunk log-decay sums near -6e4 (the unsafe-channel path) across the cut."""
    w = synthetic.make([4096, 200], Hk=2, Hv=4, K=128, V=128, seed=47, gate="large",
                       gate_scale_log_max=float(np.log(1000.0)), state="pool", num_slots=4)
    o, pool, ws = _run(w)
    assert _cuts(ws) == 1
    assert torch.isfinite(o).all() and torch.isfinite(pool).all()
    _check_pool(w, o, pool)


@pytest.mark.parametrize("variant", ["act", "scalar", "l2norm"])
def test_cut_with_kernel_variants(variant):
    """The gate activation, the scalar gate and the in-kernel q/k normalisation across a cut."""
    w = synthetic.make([2200, 90], Hk=8, Hv=8, K=128, V=128, seed=48, state="pool", num_slots=4)
    d = to_dev(w)
    T = w.T
    if variant == "act":
        a, A_log, dtb = synthetic.gate_act_inputs(T, 8, 128, seed=5)
        o, _ = kda.chunk_prefill_act(d["q"], d["k"], d["v"], a.cuda(), A_log.cuda(), dtb.cuda(),
                                     d["beta"], d["cu_seqlens"], state=d["state"],
                                     state_indices=d["state_indices"])
        g = torch.from_numpy(kda_oracle.gate_activation(a, A_log, dtb))
        q, k = w.q, w.k
    elif variant == "scalar":
        g = synthetic.scalar_gate_inputs(T, 8, seed=6)
        o, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], g.cuda(), d["beta"], d["cu_seqlens"],
                                 state=d["state"], state_indices=d["state_indices"])
        q, k = w.q, w.k
    else:
        gen = torch.Generator().manual_seed(7)
        q = (torch.randn(T, 8, 128, generator=gen) * 3).to(torch.bfloat16)
        k = (torch.randn(T, 8, 128, generator=gen) * 0.5).to(torch.bfloat16)
        o, _ = kda.chunk_prefill(q.cuda(), k.cuda(), d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 state=d["state"], state_indices=d["state_indices"], qk_l2norm=True)
        g = w.g
        q, k = torch.from_numpy(kda_oracle.l2norm(q)), torch.from_numpy(kda_oracle.l2norm(k))
    assert _cuts(kda.chunk_prefill.last_workspace if variant != "act"
                 else kda.chunk_prefill_act.last_workspace) == 1
    o_ref, pool_ref = kda_oracle.recurrence(q, k, w.v, g, w.beta, w.cu_seqlens, scale=w.scale,
                                            state=w.state, state_indices=w.state_indices)
    rms = 0.15 if variant == "l2norm" else None
    assert_items_close(o, o_ref, w.cu_seqlens.tolist(), torch.bfloat16, "o", max_rms=rms)
    slots = w.state_indices.long()
    assert_rows_close(d["state"][slots.cuda()], pool_ref[slots.numpy()], torch.bfloat16, "pool")
