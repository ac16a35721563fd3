"""GPU parity of the chunked prefill against the fp64 oracle, through the C ABI.

Tolerances (relative L2 over the tensor): 1e-2 with bf16 inputs, 1e-4 with fp32
inputs; every output finite; pool mode bit-identical to dense gather/scatter
(sglang PR 30169 digest, 关键源码片段 test_gdn_chunk_cutedsl_pool_mode_matches_dense).
"""
import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from oracle import kda_oracle
from tests._util import assert_close, assert_items_close, assert_rows_close, to_dev

pytestmark = pytest.mark.gpu


def _full_oracle(w, state=None, pool_mode=True):
    st = w.state if state is None else state
    return kda_oracle.recurrence(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, scale=w.scale,
                                 state=st, state_indices=w.state_indices if pool_mode else None)


def test_tiny_varlen_fp32_dense():
    w = synthetic.tiny_varlen()
    d = to_dev(w)
    o, ht = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                              state=d["state"], scale=w.scale)
    o_ref, ht_ref = _full_oracle(w, pool_mode=False)
    assert_close(o, o_ref, torch.float32, "o")
    assert_close(ht, ht_ref, torch.float32, "ht")


@pytest.mark.parametrize("layout", ["kv", "vk"])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_pool_mode_matches_dense_bitwise_and_oracle(state_dtype, layout):
    """Pool mode against dense gather/scatter, bit for bit, in both state layouts: [K][V] per
    head, and the pages' transposed [V][K] pool (PR 30169 digest, 关键源码片段), which must give
    the [K][V] run's results transposed, bit for bit."""
    w = synthetic.pool_varlen(state_dtype=state_dtype)
    d = to_dev(w)
    if layout == "vk":
        kv_pool = d["state"].clone()
        o_kv, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                    state=kv_pool, state_indices=d["state_indices"])
        d["state"] = d["state"].transpose(-1, -2).contiguous()
    pool = d["state"]
    slots = torch.where(d["state_indices"] >= 0, d["state_indices"],
                        torch.full_like(d["state_indices"], pool.shape[0] - 1)).long()
    h0_dense = pool[slots].clone()
    pool_before = pool.clone()
    o_dense, ht_dense = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                          d["cu_seqlens"], state=h0_dense.clone(),
                                          state_layout=layout)
    o_pool, ht_pool = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                        d["cu_seqlens"], state=pool,
                                        state_indices=d["state_indices"], state_layout=layout)
    torch.cuda.synchronize()
    assert ht_pool is pool
    assert torch.equal(o_pool, o_dense)
    assert torch.equal(pool[slots], ht_dense)
    untouched = torch.ones(pool.shape[0], dtype=torch.bool, device=pool.device)
    untouched[slots] = False
    assert torch.equal(pool[untouched], pool_before[untouched])
    if layout == "vk":  # the transposed layout's results are the [K][V] run's, transposed
        assert torch.equal(o_pool, o_kv)
        assert torch.equal(pool.transpose(-1, -2), kv_pool)
        pool = pool.transpose(-1, -2)
    # against the oracle (the -1 sequence lands in the sentinel slot 15)
    o_ref, pool_ref = _full_oracle(w)
    assert_close(o_pool, o_ref, torch.bfloat16, "o")
    assert_close(pool[slots], pool_ref[slots.cpu().numpy()], torch.bfloat16, "pool rows")
    assert int(slots[-1]) == pool.shape[0] - 1


def _full_size_case(w):
    """One prefill of a full-size workload in pool mode, compared in full with one
    whole-workload oracle call: every (sequence, v-head) item of o and every written pool
    row, each on its own; pool rows no sequence names stay bit-identical."""
    d = to_dev(w)
    pool_before = w.state.clone()
    o, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             state=d["state"], state_indices=d["state_indices"])
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    assert torch.isfinite(o).all()
    assert torch.isfinite(d["state"]).all()
    o_ref, pool_ref = _full_oracle(w, state=pool_before)
    e_o = assert_items_close(o, o_ref, w.cu_seqlens.tolist(), torch.bfloat16, "o")
    slots = torch.where(w.state_indices >= 0, w.state_indices,
                        torch.full_like(w.state_indices, w.state.shape[0] - 1)).long()
    e_s = assert_rows_close(d["state"][slots.cuda()], pool_ref[slots.numpy()], torch.bfloat16,
                            "written pool rows")
    untouched = torch.ones(w.state.shape[0], dtype=torch.bool)
    untouched[slots] = False
    assert torch.equal(d["state"][untouched.cuda()].cpu(), pool_before[untouched])
    return e_o, e_s


def test_large_decay_full():
    """Config 3: 8 x 4096 tokens, Hv = 32, per-chunk log-decay sums near -6e4 (the gate
    magnitude at which the pages' fp32 exponent overflowed: PR 27488 digest, 功能与动机)."""
    _full_size_case(synthetic.large_decay())


def test_throughput_workload_full():
    """Config 4, the benchmark's workload (32768 tokens in 16 sequences, Hv = 32), in the
    launch configuration the benchmark times."""
    _full_size_case(synthetic.throughput())


@pytest.mark.parametrize("K,V,dtype", [(64, 128, torch.float32), (128, 64, torch.bfloat16),
                                       (64, 64, torch.bfloat16), (128, 128, torch.float32)])
def test_head_dims_and_dtypes(K, V, dtype):
    w = synthetic.make([3, 64, 129, 1, 200], Hk=2, Hv=4, K=K, V=V, dtype=dtype, seed=K + V,
                       state="pool", num_slots=8)
    d = to_dev(w)
    o, pool = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"])
    o_ref, pool_ref = _full_oracle(w)
    assert_close(o, o_ref, dtype, "o")
    assert_close(pool, pool_ref, dtype, "pool")


@pytest.mark.parametrize("p", [1, 37, 63, 64, 65, 130])
def test_split_invariance_through_pool(p):
    w = synthetic.make([200], Hk=4, Hv=8, K=128, V=128, dtype=torch.bfloat16, seed=p,
                       state="pool", num_slots=4)
    d = to_dev(w)
    pool_a = d["state"].clone()
    o_full, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                  state=pool_a, state_indices=d["state_indices"])
    pool_b = d["state"].clone()
    cu1 = torch.tensor([0, p], dtype=torch.int32, device="cuda")
    cu2 = torch.tensor([0, 200 - p], dtype=torch.int32, device="cuda")
    o1, _ = kda.chunk_prefill(d["q"][:p].contiguous(), d["k"][:p].contiguous(),
                              d["v"][:p].contiguous(), d["g"][:p].contiguous(),
                              d["beta"][:p].contiguous(), cu1, state=pool_b,
                              state_indices=d["state_indices"])
    o2, _ = kda.chunk_prefill(d["q"][p:].contiguous(), d["k"][p:].contiguous(),
                              d["v"][p:].contiguous(), d["g"][p:].contiguous(),
                              d["beta"][p:].contiguous(), cu2, state=pool_b,
                              state_indices=d["state_indices"])
    o_ref, pool_ref = _full_oracle(w)
    assert_close(torch.cat([o1, o2]), o_ref, torch.bfloat16, "split o")
    assert_close(pool_b, pool_ref, torch.bfloat16, "split pool")
    assert_close(o_full, o_ref, torch.bfloat16, "whole o")


def test_run_to_run_bit_identical():
    w = synthetic.pool_varlen()
    d = to_dev(w)
    outs = []
    for _ in range(2):
        pool = d["state"].clone()
        o, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 state=pool, state_indices=d["state_indices"])
        outs.append((o, pool))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_zero_length_sequences_and_empty_batch():
    w = synthetic.make([0, 70, 0, 5], Hk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16, seed=3,
                       state="dense")
    d = to_dev(w)
    o, ht = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                              state=d["state"])
    o_ref, ht_ref = _full_oracle(w, pool_mode=False)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert torch.equal(ht[0], d["state"][0]) and torch.equal(ht[2], d["state"][2])
    assert_close(ht, ht_ref, torch.bfloat16, "ht")
    # N = 0, T = 0
    e = torch.empty((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    o0, h0 = kda.chunk_prefill(e, e, torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda"),
                               torch.empty((0, 2, 128), device="cuda"),
                               torch.empty((0, 2), device="cuda"),
                               torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert o0.shape == (0, 2, 128) and h0.shape == (0, 2, 128, 128)


def test_many_short_items_claimed_late():
    """Four times more (sequence, head) items than SMs, most of them 0 to 3 chunks long and
    empty sequences among them: every CTA claims many items, each near the end of the one
    before it (at its first chunk when the item has at most three), and items run back to
    back with and without the next chunk known one chunk ahead."""
    pattern = [0, 1, 5, 63, 64, 65, 130, 200, 17, 0, 129, 3]
    lens = (pattern * 50)[:600]
    w = synthetic.make(lens, Hk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16, seed=77,
                       state="pool", num_slots=640)
    d = to_dev(w)
    pool_before = w.state.clone()
    o, pool = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"])
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    o_ref, pool_ref = _full_oracle(w, state=pool_before)
    # relative L2 at the stated bar; the element-wise guard at 0.15 of the RMS over these 8.7 M
    # outputs (the largest of bf16 rounding errors grows with the element count; an item run
    # with a wrong state or chunk would be off by the values themselves, ~1 RMS)
    assert_close(o, o_ref, torch.bfloat16, "o", max_rms=0.15)
    assert_close(pool, pool_ref, torch.bfloat16, "pool")


def test_sixteen_thousand_sequences_longest_first():
    """16384 sequences, most of 0 to 5 tokens with longer ones spread among them: the
    longest-first order of the work list is built on the device (a counting sort over chunk
    counts, no host sync) for a batch of this size too, and every item is claimed and run
    once.  Every (sequence, head) item and every written pool row against the oracle."""
    gen = torch.Generator().manual_seed(123)
    lens = torch.randint(0, 6, (16384,), generator=gen)
    longer = torch.randperm(16384, generator=gen)[:40]
    lens[longer] = torch.randint(60, 400, (40,), generator=gen)
    w = synthetic.make(lens.tolist(), Hk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16, seed=124,
                       state="pool", num_slots=16385, state_dtype=torch.bfloat16)
    d = to_dev(w)
    pool_before = w.state.clone()
    o, pool = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"])
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    o_ref, pool_ref = _full_oracle(w, state=pool_before)
    assert_items_close(o, o_ref, w.cu_seqlens.tolist(), torch.bfloat16, "o", max_rms=0.15)
    slots = w.state_indices.long()
    assert_rows_close(pool[slots.cuda()], pool_ref[slots.numpy()], torch.bfloat16, "pool rows")


def test_zero_initial_state_and_padded_gate_rows():
    w = synthetic.make([90, 33], Hk=2, Hv=2, K=128, V=128, dtype=torch.bfloat16, seed=5,
                       state=None, g_pad_rows=17)
    d = to_dev(w)
    d["g"][-17:] = float("nan")      # padding rows past T must never be read
    d["beta"][-17:] = float("nan")
    o, ht = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    T = w.T
    o_ref, ht_ref = kda_oracle.recurrence(w.q, w.k, w.v, w.g[:T], w.beta[:T], w.cu_seqlens,
                                          scale=w.scale)
    assert_close(o, o_ref, torch.bfloat16, "o")
    assert_close(ht, ht_ref, torch.bfloat16, "ht")


def test_bad_slot_and_bad_seqlens_set_device_status():
    w = synthetic.make([20, 30, 40], Hk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16, seed=9,
                       state="pool", num_slots=6)
    d = to_dev(w)
    idx = d["state_indices"].clone()
    idx[1] = 6  # out of range
    pool = d["state"].clone()
    o = torch.zeros((w.T, 2, 128), dtype=torch.bfloat16, device="cuda")
    kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], state=pool,
                      state_indices=idx, out=o)
    bits = kda.read_device_status(kda.chunk_prefill.last_workspace)
    assert bits & kda.api.KDA_DEVICE_BAD_SLOT
    o_ref, pool_ref = _full_oracle(w)
    cu = w.cu_seqlens.tolist()
    assert torch.count_nonzero(o[cu[1]:cu[2]]) == 0          # skipped sequence untouched
    for n in (0, 2):
        s = int(w.state_indices[n])
        assert_close(o[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]], torch.bfloat16, f"o seq {n}")
        assert_close(pool[s], pool_ref[s], torch.bfloat16, f"slot {s}")
    # a clean call clears the word
    kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                      state=d["state"].clone(), state_indices=d["state_indices"])
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    # non-monotone cu_seqlens
    cu_bad = d["cu_seqlens"].clone()
    cu_bad[2] = 10
    kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_bad,
                      state=d["state"].clone(), state_indices=d["state_indices"])
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) & kda.api.KDA_DEVICE_BAD_SEQLENS


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_tensor_core_path_matches_cuda_core_path_and_oracle(state_dtype):
    """The fused tcgen05 kernel and the fp32 CUDA-core kernel on identical inputs."""
    w = synthetic.make([1, 63, 64, 65, 200, 130, 17], Hk=2, Hv=4, K=128, V=128,
                       dtype=torch.bfloat16, seed=21, state="pool", num_slots=12,
                       state_dtype=state_dtype, last_index_pad=True)
    d = to_dev(w)
    desc = kda.make_desc(num_seqs=w.N, total_tokens=w.T, Hk=2, Hv=4, K=128, V=128,
                         qkv_dtype=torch.bfloat16, num_slots=12)
    assert kda.prefill_path(desc) == 1
    pool_tc, pool_cc = d["state"].clone(), d["state"].clone()
    o_tc, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=pool_tc, state_indices=d["state_indices"])
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    o_cc, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=pool_cc, state_indices=d["state_indices"],
                                cuda_core_path=True)
    o_ref, pool_ref = _full_oracle(w)
    assert_close(o_tc, o_ref, torch.bfloat16, "tensor-core o")
    assert_close(pool_tc, pool_ref, torch.bfloat16, "tensor-core pool")
    assert_close(o_cc, o_ref, torch.bfloat16, "cuda-core o")
    assert_close(o_tc, o_cc.double().cpu().numpy(), torch.bfloat16, "tc vs cuda-core o")


@pytest.mark.parametrize("K,V,dtype", [(64, 128, torch.float32), (128, 128, torch.bfloat16)])
def test_transposed_state_layout_cuda_core_path_and_cut(K, V, dtype):
    """The [V][K] state layout on the CUDA-core kernel (fp32 inputs, 64-wide keys) and on the
    tensor-core kernel with a cut sequence (the combine writes the transposed final state):
    the [K][V] run's results, transposed."""
    w = synthetic.make([1500, 63, 130], Hk=2, Hv=4, K=K, V=V, dtype=dtype, seed=K + 7,
                       state="pool", num_slots=6)
    d = to_dev(w)
    pool_kv = d["state"].clone()
    o_kv, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=pool_kv, state_indices=d["state_indices"])
    pool_vk = d["state"].transpose(-1, -2).contiguous()
    o_vk, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=pool_vk, state_indices=d["state_indices"], state_layout="vk")
    ws = kda.chunk_prefill.last_workspace
    if dtype == torch.bfloat16:
        assert int(ws[12:16].cpu().view(torch.int32)[0]) == 1  # the 1500-token sequence is cut
    assert torch.equal(o_vk, o_kv)
    assert torch.equal(pool_vk.transpose(-1, -2), pool_kv)
    o_ref, pool_ref = _full_oracle(w)
    assert_close(o_vk, o_ref, dtype, "o")
    assert_close(pool_vk.transpose(-1, -2), pool_ref, dtype, "pool")


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_chunk_forms_alternate_within_an_item(state_dtype):
    """Chunks whose every key channel keeps its whole-chunk decay product above 2^-100 run as
    one 64-token sub-chunk; the others as four 16-token sub-chunks with the exact pairwise
    fallback.  Gates 40x stronger on every other 64-token block (aligned to the sequence
    starts) make consecutive chunks of one item alternate between the two forms, and a
    partial last chunk end each sequence."""
    lens = [64 * 9 + 17, 64 * 4, 64 * 7 + 1]
    w = synthetic.make(lens, Hk=2, Hv=4, K=128, V=128, seed=61, state="pool", num_slots=5,
                       state_dtype=state_dtype)
    cu = w.cu_seqlens.tolist()
    f = torch.ones(w.T)
    for n in range(len(lens)):
        for c0 in range(cu[n] + 64, cu[n + 1], 128):
            f[c0:c0 + 64] = 40.0
    w.g = (w.g * f[:, None, None]).contiguous()
    d = to_dev(w)
    pool_before = w.state.clone()
    o, pool = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                state=d["state"], state_indices=d["state_indices"])
    assert kda.read_device_status(kda.chunk_prefill.last_workspace) == 0
    o_ref, pool_ref = _full_oracle(w, state=pool_before)
    assert_items_close(o, o_ref, cu, torch.bfloat16, "o")
    slots = w.state_indices.long()
    assert_rows_close(pool[slots.cuda()], pool_ref[slots.numpy()], torch.bfloat16, "pool rows")
