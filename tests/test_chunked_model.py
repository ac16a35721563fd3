"""The chunked algebra the kernels implement, checked in fp64 against the oracle
(this pins the chunked form -- gate factorisation, sub-chunk references,
unsafe-channel fallback, blocked inverse, U/W, state and output updates --
before any GPU code runs)."""
import numpy as np
import pytest

from oracle import kda_oracle
from tests.chunked_model import chunked_forward, split_state_passing, tri_inv_unit_lower_blocked


def _inputs(rng, lens, Hk, Hv, K, V, gate_scale=None):
    T = sum(lens)
    q = rng.standard_normal((T, Hk, K))
    k = rng.standard_normal((T, Hk, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, V))
    x = rng.standard_normal((T, Hv, K))
    sp = np.log1p(np.exp(x))
    if gate_scale is None:
        g = -sp
    else:
        g = -np.exp(rng.random(Hv) * gate_scale)[None, :, None] * sp
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, Hv))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, g, b, cu


def test_blocked_inverse_matches_dense_inverse():
    rng = np.random.default_rng(0)
    for C in (16, 37, 64):
        A = np.tril(rng.standard_normal((C, C)) * 0.2, -1)
        X = tri_inv_unit_lower_blocked(A, 16)
        np.testing.assert_allclose(X, np.linalg.inv(np.eye(C) + A), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("lens,gate_scale", [
    ([1, 37, 130], None),
    ([64, 65, 16, 3], None),
    ([150, 20], np.log(1000.0)),  # large decay: exercises the unsafe-channel path
])
def test_chunked_model_equals_token_recurrence(lens, gate_scale):
    rng = np.random.default_rng(sum(lens))
    Hk, Hv, K, V = 1, 2, 16, 8
    q, k, v, g, b, cu = _inputs(rng, lens, Hk, Hv, K, V, gate_scale)
    S0 = rng.standard_normal((len(lens), Hv, K, V)) * 0.1
    scale = K ** -0.5
    o_ref, f_ref = kda_oracle.recurrence(q, k, v, g, b, cu, scale=scale, state=S0)
    o, f = chunked_forward(q, k, v, g, b, cu, S0, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(f, f_ref, rtol=1e-10, atol=1e-12)
    assert np.all(np.isfinite(o))


@pytest.mark.parametrize("split_chunks,gate_scale", [(1, None), (2, None), (1, np.log(1000.0))])
def test_split_state_passing_equals_token_recurrence(split_chunks, gate_scale):
    """A long sequence cut in two segments that run independently (the second one twice: from
    zero with the values, from the identity without them) and combined by two products gives
    the recurrence's outputs and final state: the algebra a split of the longest chains across
    CTAs would use."""
    rng = np.random.default_rng(7 + split_chunks)
    lens = [200, 40, 129]
    Hk, Hv, K, V = 1, 2, 16, 8
    q, k, v, g, b, cu = _inputs(rng, lens, Hk, Hv, K, V, gate_scale)
    S0 = rng.standard_normal((len(lens), Hv, K, V)) * 0.1
    scale = K ** -0.5
    o_ref, f_ref = kda_oracle.recurrence(q, k, v, g, b, cu, scale=scale, state=S0)
    o, f = split_state_passing(q, k, v, g, b, cu, S0, scale, split_chunks)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(f, f_ref, rtol=1e-10, atol=1e-12)
