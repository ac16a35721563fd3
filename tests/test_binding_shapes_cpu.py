"""Host-side shape checks of the Python binding: the C ABI takes plain pointers, so a tensor
too small for the descriptor must be refused before any launch (it would be read or
written out of bounds otherwise).  Runs on CPU tensors: the checks look at shapes only."""
import pytest
import torch

from linear_attention_prefill_chunked_gb300 import api

T, N, HK, HV, K, V, SLOTS = 70, 3, 2, 4, 128, 128, 8
BF = torch.bfloat16


def _prefill_args(**over):
    a = dict(q=torch.zeros(T, HK, K, dtype=BF), k=torch.zeros(T, HK, K, dtype=BF),
             v=torch.zeros(T, HV, V, dtype=BF), gate=torch.zeros(T + 5, HV, K),
             beta=torch.zeros(T, HV), cu_seqlens=torch.tensor([0, 10, 40, T], dtype=torch.int32))
    kw = dict(state=torch.zeros(SLOTS, HV, K, V), state_indices=torch.zeros(N, dtype=torch.int32),
              out=torch.zeros(T, HV, V, dtype=BF))
    for key, val in over.items():
        (a if key in a else kw)[key] = val
    return a, kw


def _check_prefill(**over):
    a, kw = _prefill_args(**over)
    api.check_prefill_shapes(a["q"], a["k"], a["v"], a["gate"], a["beta"], a["cu_seqlens"], **kw)


def test_valid_prefill_shapes_pass():
    _check_prefill()
    _check_prefill(gate=torch.zeros(T, HV))  # scalar gate
    _check_prefill(state_indices=None, state=torch.zeros(N, HV, K, V),
                   final_state=torch.zeros(N, HV, K, V))  # dense mode
    a, kw = _prefill_args(gate=torch.zeros(T, HV, K, dtype=BF))
    api.check_prefill_shapes(a["q"], a["k"], a["v"], a["gate"], a["beta"], a["cu_seqlens"],
                             A_log=torch.zeros(HV), dt_bias=torch.zeros(HV, K), **kw)


@pytest.mark.parametrize("over", [
    dict(k=torch.zeros(T, HK, 64, dtype=BF)),                 # k and q differ
    dict(v=torch.zeros(T - 1, HV, V, dtype=BF)),              # v shorter than q
    dict(v=torch.zeros(T, 3, V, dtype=BF)),                   # Hv not a multiple of Hk
    dict(gate=torch.zeros(T - 1, HV, K)),                     # gate shorter than T
    dict(gate=torch.zeros(T, HV, 64)),                        # gate of the wrong width
    dict(beta=torch.zeros(T, HV - 1)),                        # beta of the wrong width
    dict(state_indices=torch.zeros(N + 1, dtype=torch.int32)),  # one index per sequence
    dict(state=torch.zeros(SLOTS, HV, K, 64)),                # pool rows of the wrong shape
    dict(out=torch.zeros(T - 1, HV, V, dtype=BF)),            # out too short
])
def test_prefill_shape_errors_are_refused(over):
    with pytest.raises(ValueError):
        _check_prefill(**over)


def test_prefill_out_dtype_and_dense_state_checked():
    with pytest.raises(TypeError):
        _check_prefill(out=torch.zeros(T, HV, V))  # fp32 out for bf16 inputs
    with pytest.raises(ValueError):
        _check_prefill(state_indices=None, state=torch.zeros(N + 1, HV, K, V))
    with pytest.raises(ValueError):
        a, kw = _prefill_args()
        api.check_prefill_shapes(a["q"], a["k"], a["v"], a["gate"], a["beta"], a["cu_seqlens"],
                                 A_log=torch.zeros(HV), dt_bias=torch.zeros(HV), **kw)


def test_decode_shape_checks():
    rows = 6
    q = torch.zeros(rows, HK, K, dtype=BF)
    ok = dict(q=q, k=q.clone(), v=torch.zeros(rows, HV, V, dtype=BF), g=torch.zeros(rows, HV, K),
              beta=torch.zeros(rows, HV), pool=torch.zeros(SLOTS, HV, K, V))
    api.check_decode_shapes(*ok.values(), state_indices=torch.zeros(rows, dtype=torch.int32))
    with pytest.raises(ValueError):
        api.check_decode_shapes(*ok.values(), state_indices=torch.zeros(rows - 1, dtype=torch.int32))
    with pytest.raises(ValueError):
        api.check_decode_shapes(*ok.values(), out=torch.zeros(rows, HV, V - 1, dtype=BF))
    bad = dict(ok, g=torch.zeros(rows - 1, HV, K))
    with pytest.raises(ValueError):
        api.check_decode_shapes(*bad.values())
    # draft steps: one index per request, not per token
    cu = torch.tensor([0, 2, 6], dtype=torch.int32)
    api.check_decode_shapes(*ok.values(), state_indices=torch.zeros(2, dtype=torch.int32),
                            cu_seqlens=cu)
    with pytest.raises(ValueError):
        api.check_decode_shapes(*ok.values(), state_indices=torch.zeros(rows, dtype=torch.int32),
                                cu_seqlens=cu)
    # a pitched pool (rows of `pitch` elements) must reach the end of its last slot's state
    pitch = HV * K * V + 64
    api.check_decode_shapes(*dict(ok, pool=torch.zeros(SLOTS, pitch)).values(), slot_stride=pitch)
    with pytest.raises(ValueError):
        api.check_decode_shapes(*dict(ok, pool=torch.zeros(SLOTS, 64)).values(), slot_stride=pitch)


def test_dense_final_state_dtype_must_match_state():
    """Dense mode writes the final state in the initial state's element type, so a mismatched
    final_state would be overrun (fp32 state, bf16 final) or half filled (the reverse)."""
    for sdt, fdt in ((torch.float32, BF), (BF, torch.float32)):
        with pytest.raises(TypeError):
            _check_prefill(state_indices=None, state=torch.zeros(N, HV, K, V, dtype=sdt),
                           final_state=torch.zeros(N, HV, K, V, dtype=fdt))
    _check_prefill(state_indices=None, state=torch.zeros(N, HV, K, V, dtype=BF),
                   final_state=torch.zeros(N, HV, K, V, dtype=BF))
