"""The seeded input recipes, checked against the workload specification they stand for
(shapes, length mix, value ranges, slot indices): inputs are part of every parity and
timing claim, so a drifted recipe would silently change both."""
import math

import torch

from linear_attention_prefill_chunked_gb300 import synthetic


def _unit_rows(x, tol):
    n = x.float().norm(dim=-1)
    return bool(((n - 1).abs() <= tol).all())


def test_throughput_workload_recipe():
    lens = synthetic.throughput_lengths()
    assert len(lens) == 16 and sum(lens) == 32768 and min(lens) >= 1
    # log-uniform in [64, 8192] before the rescale to 32768 tokens; the longest takes the residual
    assert max(lens) <= 2 * 8192 and sorted(lens)[-2] < 8192
    w = synthetic.throughput()
    assert w.q.shape == (32768, 32, 128) and w.v.shape == (32768, 32, 128)
    assert w.q.dtype == torch.bfloat16 and w.state.shape == (256, 32, 128, 128)
    assert w.state.dtype == torch.float32
    assert w.cu_seqlens.tolist()[-1] == 32768 and w.lens == lens
    idx = w.state_indices.tolist()
    assert len(set(idx)) == 16 and all(0 <= i < 255 for i in idx)  # distinct, never the sentinel
    assert bool((w.g <= 0).all()) and bool(((w.beta > 0) & (w.beta < 1)).all())
    assert _unit_rows(w.q[:4096], 2e-2) and _unit_rows(w.k[:4096], 2e-2)  # unit rows, then bf16
    assert abs(float(w.state[:8].std()) - 0.1) < 5e-3


def test_small_configurations():
    t = synthetic.tiny_varlen()
    assert t.lens == [1, 37, 130] and t.q.shape == (168, 2, 64) and t.q.dtype == torch.float32
    assert t.state.shape == (3, 2, 64, 64) and t.state_indices is None
    p = synthetic.pool_varlen()
    assert len(p.lens) == 5 and all(1 <= n < 130 for n in p.lens)
    assert p.q.shape[1:] == (4, 128) and p.v.shape[1:] == (8, 128)
    assert p.state.shape == (16, 8, 128, 128) and p.state_indices.tolist()[-1] == -1
    assert len(set(p.state_indices.tolist()[:-1])) == 4
    assert p.scale == 128 ** -0.5


def test_large_decay_reaches_the_stress_range():
    w = synthetic.large_decay(num_seqs=2, seqlen=256)
    assert bool(torch.isfinite(w.g).all()) and bool((w.g <= 0).all())
    # g = -exp(a_h) softplus(x) with a_h up to ln 1000: per-chunk sums reach the 1e4 range
    chunk_sums = w.g[:64].sum(dim=0)  # [Hv, K] over one 64-token chunk
    assert float(chunk_sums.min()) < -1e4
    a_max = float((-w.g[:64]).max())
    assert a_max <= 1000 * (math.log1p(math.exp(8.0))) + 1


def test_decode_batch_recipe_small():
    w = synthetic.decode_batch(num_rows=64, num_pad=4, num_slots=96)
    assert w.lens == [1] * 64 and w.q.shape == (64, 32, 128)
    idx = w.state_indices.tolist()
    assert idx[-4:] == [-1] * 4 and len(set(idx[:-4])) == 60 and all(0 <= i < 95 for i in idx[:-4])
    assert w.state.shape == (96, 32, 128, 128)
