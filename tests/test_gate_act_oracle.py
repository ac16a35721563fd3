"""Pins of the oracle's gate activation ``g = max(-exp(A_log) softplus(a + dt_bias), lb)``
against closed forms of softplus and of the recurrence (no GPU needed).

The gate form is the one the pages' tests build (sglang PR 30169 digest, 关键源码片段, the
GDN pool test; PR 27488 digest, 关键源码片段 ``CuteDSLKDAKernel.extend`` takes A_log,
dt_bias and lower_bound).  Each check below would fail for a plausible slip: a wrong
softplus (log(1 + x), or log(1 + e^x) evaluated naively), a dropped or mis-signed exp(A_log),
dt_bias not added inside softplus, or the bound applied as a ceiling.
"""
import math

import numpy as np

from oracle import kda_oracle

rng = np.random.default_rng(5)


def test_softplus_at_zero_is_ln2():
    g = kda_oracle.gate_activation(np.zeros((3, 2, 4)), np.zeros(2))
    assert np.allclose(g, -math.log(2.0), rtol=0, atol=1e-15)


def test_odd_part_of_softplus_is_identity():
    # softplus(x) - softplus(-x) = x for every x
    a = rng.normal(size=(5, 3, 8)) * 4
    d = kda_oracle.gate_activation(a, np.zeros(3)) - kda_oracle.gate_activation(-a, np.zeros(3))
    assert np.allclose(d, -a, rtol=0, atol=1e-13)


def test_A_log_scales_the_gate_by_exp():
    a = rng.normal(size=(4, 2, 6))
    g1 = kda_oracle.gate_activation(a, np.zeros(2))
    g3 = kda_oracle.gate_activation(a, np.full(2, math.log(3.0)))
    assert np.allclose(g3, 3.0 * g1, rtol=1e-14, atol=0)
    assert np.all(g1 < 0)


def test_dt_bias_shifts_the_argument_per_channel():
    a = rng.normal(size=(4, 2, 6))
    db = rng.normal(size=(2, 6))
    assert np.allclose(kda_oracle.gate_activation(a, np.zeros(2), db),
                       kda_oracle.gate_activation(a + db[None], np.zeros(2)), rtol=1e-14, atol=0)


def test_softplus_tails():
    # large x: softplus(x) = x + log1p(e^-x); very negative x: softplus(x) = e^x (1 - e^x/2 ...)
    g_hi = kda_oracle.gate_activation(np.full((1, 1, 1), 40.0), np.zeros(1))
    assert abs(g_hi[0, 0, 0] + 40.0) <= 1e-14 * 40
    g_lo = kda_oracle.gate_activation(np.full((1, 1, 1), -40.0), np.zeros(1))
    assert abs(g_lo[0, 0, 0] / -math.exp(-40.0) - 1.0) < 1e-12


def test_lower_bound_is_a_floor():
    a = rng.normal(size=(6, 2, 8)) * 3
    g = kda_oracle.gate_activation(a, np.full(2, math.log(5.0)))
    gb = kda_oracle.gate_activation(a, np.full(2, math.log(5.0)), lower_bound=-1.0)
    assert np.all(gb >= -1.0)
    assert np.array_equal(gb[g > -1.0], g[g > -1.0])
    assert np.all(gb[g <= -1.0] == -1.0)
    assert np.any(g < -1.0) and np.any(g > -1.0)


def test_gate_feeds_the_recurrence_as_a_decay():
    # beta = 0: S_T = Diag(exp(sum_t g_t)) S_0; with a = 0, A_log = 0 each step halves S
    T, K, V = 5, 4, 3
    a = np.zeros((T, 1, K))
    g = kda_oracle.gate_activation(a, np.zeros(1))
    S0 = rng.normal(size=(1, 1, K, V))
    q = rng.normal(size=(T, 1, K))
    k = rng.normal(size=(T, 1, K))
    v = rng.normal(size=(T, 1, V))
    _, fin = kda_oracle.recurrence(q, k, v, g, np.zeros((T, 1)), [0, T], state=S0)
    assert np.allclose(fin, S0 * 2.0 ** -T, rtol=1e-13, atol=0)


def test_scalar_gate_is_the_channel_broadcast():
    # a [T, Hv] gate (GDN form) must act like the same value on every key channel
    T, Hk, Hv, K, V = 9, 1, 2, 4, 3
    q = rng.normal(size=(T, Hk, K))
    k = rng.normal(size=(T, Hk, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, Hv, V))
    beta = rng.uniform(size=(T, Hv))
    g2 = -rng.uniform(0.0, 2.0, size=(T, Hv))
    g3 = np.repeat(g2[:, :, None], K, axis=2)
    o2, s2 = kda_oracle.recurrence(q, k, v, g2, beta, [0, 4, T])
    o3, s3 = kda_oracle.recurrence(q, k, v, g3, beta, [0, 4, T])
    assert np.array_equal(o2, o3) and np.array_equal(s2, s3)
    a = rng.normal(size=(T, Hv))
    ga = kda_oracle.gate_activation(a, np.zeros(Hv), np.zeros(Hv))
    assert ga.shape == (T, Hv)
    assert np.allclose(ga - kda_oracle.gate_activation(-a, np.zeros(Hv), np.zeros(Hv)), -a,
                       rtol=0, atol=1e-13)


def test_l2norm_rows():
    x = rng.normal(size=(7, 3, 16)) * 5
    x[2, 1] = 0.0
    y = kda_oracle.l2norm(x)
    n = np.linalg.norm(y, axis=-1)
    assert np.allclose(np.delete(n.reshape(-1), 2 * 3 + 1), 1.0, rtol=0, atol=1e-14)
    assert np.all(y[2, 1] == 0.0)                             # zero rows stay zero
    assert np.allclose(kda_oracle.l2norm(3.5 * x), y, rtol=1e-14, atol=0)  # scale-free
    assert np.all(np.sign(y) == np.sign(x))
