"""Pins for the fp64 CPU oracle: checks against facts fixed by the mathematics,
not against the oracle's own formula.

Each test is chosen so that a plausible slip in the oracle fails it:
  * hand-worked example        -- any arithmetic slip
  * explicit-matrix brute force -- transposed S, wrong index, wrong sign
  * beta = 0 closed form       -- dropped/duplicated decay, exp base, cumsum
  * beta = 1 delta write       -- decay after the write, sign of u, o from S_{t-1}
  * orthonormal keys           -- row/column confusion in the write
  * scalar-gate identity       -- order of decay and write
  * GQA repeat, packing, split, pool/dense, sentinel, padding rows
"""
import os

import numpy as np
import pytest

from oracle import kda_oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, lens, Hk, Hv, K, V, unit=True, gate="softplus", beta=None):
    T = sum(lens)
    q = rng.standard_normal((T, Hk, K))
    k = rng.standard_normal((T, Hk, K))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, V))
    if gate == "softplus":
        g = -np.log1p(np.exp(rng.standard_normal((T, Hv, K))))
    elif gate == "zero":
        g = np.zeros((T, Hv, K))
    else:
        g = gate(T, Hv, K)
    b = (1.0 / (1.0 + np.exp(-rng.standard_normal((T, Hv))))) if beta is None else np.full((T, Hv), beta)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, g, b, cu


def _brute(q, k, v, g, b, cu, S0, scale):
    """Explicit matrices: M_t = (I - b k k^T) Diag(exp g), S_t = M_t S_{t-1} + b k v^T."""
    T, Hk, K = q.shape
    Hv, V = v.shape[1:]
    N = len(cu) - 1
    o = np.zeros((T, Hv, V))
    fin = np.zeros((N, Hv, K, V))
    for n in range(N):
        for h in range(Hv):
            kh = h // (Hv // Hk)
            S = S0[n, h].copy()
            for t in range(cu[n], cu[n + 1]):
                kt = k[t, kh][:, None]
                M = (np.eye(K) - b[t, h] * kt @ kt.T) @ np.diag(np.exp(g[t, h]))
                S = M @ S + b[t, h] * kt @ v[t, h][None, :]
                o[t, h] = scale * S.T @ q[t, kh]
            fin[n, h] = S
    return o, fin


def test_hand_worked_example():
    vals = {}
    with open(os.path.join(GOLD, "hand_worked_k2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            vals[key] = np.array([float(x) for x in rest.split()])
    q = vals["q"].reshape(2, 1, 2)
    k = vals["k"].reshape(2, 1, 2)
    v = vals["v"].reshape(2, 1, 2)
    g = vals["g"].reshape(2, 1, 2)
    b = vals["beta"].reshape(2, 1)
    S0 = vals["S0"].reshape(1, 1, 2, 2)
    o, fin = kda_oracle.recurrence(q, k, v, g, b, [0, 2], scale=1.0, state=S0)
    np.testing.assert_allclose(o.reshape(-1), vals["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin.reshape(-1), vals["S_final"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_matrix_form(seed):
    rng = np.random.default_rng(seed)
    K, V = (3, 4) if seed % 2 else (4, 3)
    Hk, Hv = (1, 2) if seed % 3 == 0 else (2, 2)
    lens = [int(x) for x in rng.integers(0, 7, size=3)]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, Hk, Hv, K, V, unit=bool(seed % 2))
    S0 = rng.standard_normal((3, Hv, K, V)) * 0.3
    scale = 0.7
    o, fin = kda_oracle.recurrence(q, k, v, g, b, cu, scale=scale, state=S0)
    ob, fb = _brute(q, k, v, g, b, cu, S0, scale)
    np.testing.assert_allclose(o, ob, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin, fb, rtol=1e-13, atol=1e-13)


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(1)
    lens = [5, 0, 9]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, 2, 4, 6, 5, beta=0.0)
    S0 = rng.standard_normal((3, 4, 6, 5))
    scale = 6 ** -0.5
    o, fin = kda_oracle.recurrence(q, k, v, g, b, cu, state=S0)
    for n in range(3):
        for h in range(4):
            kh = h // 2
            G = np.cumsum(g[cu[n]:cu[n + 1], h], axis=0)  # inclusive
            for j, t in enumerate(range(cu[n], cu[n + 1])):
                want = scale * S0[n, h].T @ (np.exp(G[j]) * q[t, kh])
                np.testing.assert_allclose(o[t, h], want, rtol=1e-12, atol=1e-14)
            tot = G[-1] if lens[n] else np.zeros(6)
            np.testing.assert_allclose(fin[n, h], np.exp(tot)[:, None] * S0[n, h], rtol=1e-12,
                                       atol=1e-14)


def test_beta_one_writes_value_exactly():
    # With ||k_t|| = 1 and beta_t = 1 the write makes S_t^T k_t = v_t whatever the gate;
    # with q_t = k_t and scale 1 the output must equal v_t.
    rng = np.random.default_rng(2)
    lens = [11, 4]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, 1, 2, 8, 5, beta=1.0,
                                     gate=lambda T, H, K: -3.0 * rng.random((T, H, K)))
    S0 = rng.standard_normal((2, 2, 8, 5))
    o, _ = kda_oracle.recurrence(k, k, v, g, b, cu, scale=1.0, state=S0)
    np.testing.assert_allclose(o, v, rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_replace_rows():
    rng = np.random.default_rng(3)
    K, V, T = 5, 4, 7
    rows = [2, 0, 2, 4, 1, 0, 3]
    k = np.zeros((T, 1, K))
    for t, r in enumerate(rows):
        k[t, 0, r] = 1.0
    q = rng.standard_normal((T, 1, K))
    v = rng.standard_normal((T, 1, V))
    g = np.zeros((T, 1, K))
    b = np.ones((T, 1))
    S0 = rng.standard_normal((1, 1, K, V))
    o, fin = kda_oracle.recurrence(q, k, v, g, b, [0, T], scale=1.0, state=S0)
    S = S0[0, 0].copy()
    for t, r in enumerate(rows):
        S[r] = v[t, 0]
        np.testing.assert_allclose(o[t, 0], S.T @ q[t, 0], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], S, rtol=0, atol=1e-15)


def test_scalar_gate_equals_rescaled_ungated_delta_rule():
    # With g_t constant over channels (decay a_t), S_t / A_t (A_t = prod a) follows the
    # ungated delta rule driven by v_t / A_t; this holds only for decay-then-write.
    rng = np.random.default_rng(4)
    T, K, V = 13, 6, 5
    q, k, v, _, b, cu = _rand_inputs(rng, [T], 1, 1, K, V)
    a = -0.4 * rng.random(T)
    g = np.repeat(a[:, None, None], K, axis=2)
    S0 = rng.standard_normal((1, 1, K, V))
    o, fin = kda_oracle.recurrence(q, k, v, g, b, cu, scale=1.0, state=S0)
    A = np.exp(np.cumsum(a))
    o2, fin2 = kda_oracle.recurrence(q, k, v / A[:, None, None], np.zeros_like(g), b, cu,
                                     scale=1.0, state=S0)
    np.testing.assert_allclose(o, o2 * A[:, None, None], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fin, fin2 * A[-1], rtol=1e-11, atol=1e-12)


def test_linearity_in_v_and_state():
    rng = np.random.default_rng(5)
    q, k, v, g, b, cu = _rand_inputs(rng, [9, 3], 2, 2, 4, 4)
    S0 = rng.standard_normal((2, 2, 4, 4))
    o1, f1 = kda_oracle.recurrence(q, k, v, g, b, cu, state=S0)
    o2, f2 = kda_oracle.recurrence(q, k, 2 * v, g, b, cu, state=2 * S0)
    assert np.array_equal(o2, 2 * o1) and np.array_equal(f2, 2 * f1)


@pytest.mark.parametrize("p", [1, 37, 63, 64, 65, 130])
def test_split_invariance_through_pool(p):
    rng = np.random.default_rng(6)
    L = 140
    q, k, v, g, b, cu = _rand_inputs(rng, [L], 1, 2, 8, 8)
    pool = rng.standard_normal((4, 2, 8, 8))
    idx = np.array([2], dtype=np.int32)
    o, pool_full = kda_oracle.recurrence(q, k, v, g, b, cu, state=pool, state_indices=idx)
    oa, pa = kda_oracle.recurrence(q[:p], k[:p], v[:p], g[:p], b[:p], [0, p], state=pool,
                                   state_indices=idx)
    ob, pb = kda_oracle.recurrence(q[p:], k[p:], v[p:], g[p:], b[p:], [0, L - p], state=pa,
                                   state_indices=idx)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(pb, pool_full, rtol=1e-13, atol=1e-14)


def test_packing_independence_and_zero_length():
    rng = np.random.default_rng(7)
    lens = [6, 0, 10]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, 1, 1, 4, 3)
    S0 = rng.standard_normal((3, 1, 4, 3))
    o, fin = kda_oracle.recurrence(q, k, v, g, b, cu, state=S0)
    o3, f3 = kda_oracle.recurrence(q[6:], k[6:], v[6:], g[6:], b[6:], [0, 10], state=S0[2:])
    assert np.array_equal(o[6:], o3) and np.array_equal(fin[2], f3[0])
    assert np.array_equal(fin[1], S0[1])  # empty sequence keeps its state


def test_gqa_head_mapping_contiguous_groups():
    rng = np.random.default_rng(8)
    q, k, v, g, b, cu = _rand_inputs(rng, [12], 2, 4, 4, 4)
    S0 = rng.standard_normal((1, 4, 4, 4))
    o, fin = kda_oracle.recurrence(q, k, v, g, b, cu, state=S0)
    qr, kr = np.repeat(q, 2, axis=1), np.repeat(k, 2, axis=1)  # v-head h <- k-head h // 2
    o2, fin2 = kda_oracle.recurrence(qr, kr, v, g, b, cu, state=S0)
    assert np.array_equal(o, o2) and np.array_equal(fin, fin2)


def test_pool_mode_equals_dense_gather_scatter_and_sentinel():
    rng = np.random.default_rng(9)
    lens = [5, 9, 3]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, 1, 2, 4, 4)
    pool = rng.standard_normal((6, 2, 4, 4))
    idx = np.array([3, 0, -1], dtype=np.int32)
    slots = np.array([3, 0, 5])
    o_p, pool_out = kda_oracle.recurrence(q, k, v, g, b, cu, state=pool, state_indices=idx)
    o_d, fin_d = kda_oracle.recurrence(q, k, v, g, b, cu, state=pool[slots])
    assert np.array_equal(o_p, o_d)
    assert np.array_equal(pool_out[slots], fin_d)
    untouched = np.setdiff1d(np.arange(6), slots)
    assert np.array_equal(pool_out[untouched], pool[untouched])


def test_padding_rows_of_g_and_beta_are_ignored():
    rng = np.random.default_rng(10)
    q, k, v, g, b, cu = _rand_inputs(rng, [7], 1, 1, 3, 3)
    g_pad = np.concatenate([g, np.full((5, 1, 3), np.nan)])
    b_pad = np.concatenate([b, np.full((5, 1), np.nan)])
    o1, f1 = kda_oracle.recurrence(q, k, v, g, b, cu)
    o2, f2 = kda_oracle.recurrence(q, k, v, g_pad, b_pad, cu)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_rejects_out_of_range_slot():
    rng = np.random.default_rng(11)
    q, k, v, g, b, cu = _rand_inputs(rng, [3], 1, 1, 2, 2)
    pool = np.zeros((4, 1, 2, 2))
    with pytest.raises(ValueError):
        kda_oracle.recurrence(q, k, v, g, b, cu, state=pool, state_indices=np.array([4], np.int32))
    with pytest.raises(ValueError):
        kda_oracle.recurrence(q, k, v, g, b, cu, state=pool, state_indices=np.array([-2], np.int32))
