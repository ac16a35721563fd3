"""GPU parity of the one-token decode against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from oracle import kda_oracle
from tests._util import assert_close, assert_rows_close

pytestmark = pytest.mark.gpu


def _oracle_rows(w, rows, pool_rows_before):
    """Oracle o and final state for the given rows (each with its own slot)."""
    o_all, s_all = [], []
    for j, n in enumerate(rows):
        o, fin = kda_oracle.recurrence(
            w.q[n:n + 1], w.k[n:n + 1], w.v[n:n + 1], w.g[n:n + 1], w.beta[n:n + 1], [0, 1],
            scale=w.scale, state=pool_rows_before[j:j + 1])
        o_all.append(o[0])
        s_all.append(fin[0])
    return np.stack(o_all), np.stack(s_all)


def test_decode_large_batch_all_rows():
    """Config 5: 4096 rows x 32 heads (N*Hv = 131072 > 65535), 8192-slot fp32 pool (16 GiB),
    64 padding rows on the sentinel.  Every real row's o and updated pool row against the
    oracle (in batches, each row from its own slot's prior state), each row on its own;
    pool rows no row names stay bit-identical."""
    w = synthetic.decode_batch(pool_device="cuda")
    pool = w.state
    q, k, v, g, beta = (t.cuda() for t in (w.q, w.k, w.v, w.g, w.beta))
    idx = w.state_indices.cuda()
    real = np.flatnonzero(w.state_indices.numpy() >= 0)
    assert real.size == 4032
    slots = w.state_indices[real].long().cuda()
    before = pool[slots].clone()  # 8 GB on the device
    rng = np.random.default_rng(0)
    used = set(w.state_indices[real].tolist()) | {pool.shape[0] - 1}
    free = np.array([s for s in range(pool.shape[0]) if s not in used])
    untouched = torch.from_numpy(rng.choice(free, size=256, replace=False)).cuda()
    untouched_before = pool[untouched].clone()
    o = kda.decode(q, k, v, g, beta, pool, idx, scale=w.scale)
    assert kda.read_device_status(kda.decode.last_workspace) == 0
    assert torch.isfinite(o[torch.from_numpy(real).cuda()]).all()
    B = 336
    for b0 in range(0, real.size, B):
        rows = real[b0:b0 + B]
        st0 = before[b0:b0 + B].cpu()
        o_ref, s_ref = kda_oracle.recurrence(
            w.q[rows], w.k[rows], w.v[rows], w.g[rows], w.beta[rows],
            np.arange(rows.size + 1), scale=w.scale, state=st0)
        assert_rows_close(o[torch.from_numpy(rows).cuda()], o_ref, torch.bfloat16,
                          f"o rows {b0}..")
        assert_rows_close(pool[slots[b0:b0 + B]], s_ref, torch.float32, f"pool rows {b0}..")
    assert torch.equal(pool[untouched], untouched_before)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_decode_equals_prefill_with_unit_lengths(state_dtype):
    w = synthetic.make([1] * 300, Hk=4, Hv=8, K=128, V=128, dtype=torch.bfloat16, seed=2,
                       state="pool", num_slots=512, state_dtype=state_dtype)
    q, k, v, g, beta = (t.cuda() for t in (w.q, w.k, w.v, w.g, w.beta))
    idx = w.state_indices.cuda()
    pool_d = w.state.cuda()
    pool_p = pool_d.clone()
    o_d = kda.decode(q, k, v, g, beta, pool_d, idx)
    o_p, _ = kda.chunk_prefill(q, k, v, g, beta, w.cu_seqlens.cuda(), state=pool_p,
                               state_indices=idx)
    o_ref, pool_ref = kda_oracle.recurrence(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens,
                                            state=w.state, state_indices=w.state_indices)
    assert_close(o_d, o_ref, torch.bfloat16, "decode o")
    assert_close(o_p, o_ref, torch.bfloat16, "prefill o")
    tol_dtype = torch.bfloat16
    assert_close(pool_d, pool_ref, tol_dtype, "decode pool")
    assert_close(pool_p, pool_ref, tol_dtype, "prefill pool")


def test_decode_fp32_inputs_and_shuffled_padding():
    w = synthetic.make([1] * 200, Hk=2, Hv=4, K=64, V=128, dtype=torch.float32, seed=4,
                       state="pool", num_slots=300)
    idx = w.state_indices.clone()
    perm = torch.randperm(200, generator=torch.Generator().manual_seed(1))
    idx[perm[:7]] = -1  # padding rows spread through the batch
    q, k, v, g, beta = (t.cuda() for t in (w.q, w.k, w.v, w.g, w.beta))
    pool = w.state.cuda()
    o = kda.decode(q, k, v, g, beta, pool, idx.cuda())
    real = np.array(sorted(set(range(200)) - set(perm[:7].tolist())))
    before = w.state[idx[real].long()]
    o_ref, s_ref = _oracle_rows(w, real, before)
    assert_close(o[real], o_ref, torch.float32, "o")
    assert_close(pool[idx[real].long().cuda()], s_ref, torch.float32, "pool rows")


def test_decode_bad_slot_sets_status():
    w = synthetic.make([1] * 10, Hk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16, seed=6,
                       state="pool", num_slots=16)
    idx = w.state_indices.clone()
    idx[3] = 16
    q, k, v, g, beta = (t.cuda() for t in (w.q, w.k, w.v, w.g, w.beta))
    pool = w.state.cuda()
    kda.decode(q, k, v, g, beta, pool, idx.cuda())
    assert kda.read_device_status(kda.decode.last_workspace) & kda.api.KDA_DEVICE_BAD_SLOT


@pytest.mark.parametrize("K,state_dtype", [(128, torch.float32), (64, torch.bfloat16)])
def test_decode_transposed_state_layout(K, state_dtype):
    """Decode on a [V][K] (transposed) pool: the key-channel reductions are shuffles within a
    row's threads there, so the results match the [K][V] decode within the tolerance and the
    oracle; rows no index names stay bit-identical."""
    w = synthetic.make([1] * 300, Hk=4, Hv=8, K=K, V=128, dtype=torch.bfloat16, seed=9,
                       state="pool", num_slots=400, state_dtype=state_dtype, last_index_pad=True)
    q, k, v, g, beta = (t.cuda() for t in (w.q, w.k, w.v, w.g, w.beta))
    idx = w.state_indices.cuda()
    pool_vk = w.state.transpose(-1, -2).contiguous().cuda()
    before = pool_vk.clone()
    o = kda.decode(q, k, v, g, beta, pool_vk, idx, state_layout="vk")
    assert kda.read_device_status(kda.decode.last_workspace) == 0
    o_ref, pool_ref = kda_oracle.recurrence(w.q[:-1], w.k[:-1], w.v[:-1], w.g[:-1], w.beta[:-1],
                                            np.arange(300), scale=w.scale, state=w.state,
                                            state_indices=w.state_indices[:-1])
    assert_close(o[:-1], o_ref, torch.bfloat16, "o")
    slots = w.state_indices[:-1].long()
    tol = torch.float32 if state_dtype == torch.float32 else torch.bfloat16
    assert_close(pool_vk[slots.cuda()].transpose(-1, -2), pool_ref[slots.numpy()], tol, "pool rows")
    untouched = torch.ones(400, dtype=torch.bool)
    untouched[slots] = False
    untouched[-1] = False  # the sentinel (padding row)
    assert torch.equal(pool_vk[untouched.cuda()], before[untouched.cuda()])
