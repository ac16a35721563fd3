"""Shared helpers of the GPU tests: device transfer, oracle on sampled heads,
error metrics."""
import numpy as np
import torch

from oracle import kda_oracle

# Tolerances of the path: relative L2 error over a whole tensor (fp64), per input dtype.
REL_L2 = {torch.bfloat16: 1e-2, torch.float32: 1e-4}
# Element-wise bound, in units of the reference's RMS: bf16 outputs carry a 2^-9
# relative rounding each, so a few percent of the RMS bounds any single element.
MAX_ERR_RMS = {torch.bfloat16: 0.1, torch.float32: 1e-3}


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def assert_close(x, ref, dtype, what="", max_rms=None):
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    e = rel_l2(x, ref)
    assert e <= REL_L2[dtype], f"{what}: relative L2 error {e:.3e} > {REL_L2[dtype]:.0e}"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    if rms > 0:
        m = float(np.max(np.abs(x - ref))) / rms
        bound = MAX_ERR_RMS[dtype] if max_rms is None else max_rms
        assert m <= bound, f"{what}: max element error {m:.3e} RMS > {bound}"
    return e


def to_dev(w, device="cuda"):
    """Copy a synthetic Workload's tensors to the device (returns a dict)."""
    d = dict(q=w.q, k=w.k, v=w.v, g=w.g, beta=w.beta, cu_seqlens=w.cu_seqlens,
             state=w.state, state_indices=w.state_indices)
    return {k: (v.to(device).contiguous() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def oracle_sampled(w, pairs, state_before=None, pool_mode=True):
    """Oracle outputs for selected (sequence, v-head) pairs.

    Returns {(n, h): (o [len, V], S_final [K, V])}.  ``state_before`` is the
    initial state array (pool or dense h0) as it was before the GPU call.
    """
    cu = w.cu_seqlens.tolist()
    Hk, Hv = w.q.shape[1], w.v.shape[1]
    st = w.state if state_before is None else state_before
    out = {}
    for n, h in pairs:
        a, b = cu[n], cu[n + 1]
        kh = h // (Hv // Hk)
        if st is None:
            S0 = None
        elif pool_mode and w.state_indices is not None:
            s = int(w.state_indices[n])
            s = st.shape[0] - 1 if s < 0 else s
            S0 = st[s, h:h + 1].unsqueeze(0)
        else:
            S0 = st[n, h:h + 1].unsqueeze(0)
        o, fin = kda_oracle.recurrence(
            w.q[a:b, kh:kh + 1], w.k[a:b, kh:kh + 1], w.v[a:b, h:h + 1], w.g[a:b, h:h + 1],
            w.beta[a:b, h:h + 1], [0, b - a], scale=w.scale, state=S0)
        out[(n, h)] = (o[:, 0], fin[0, 0])
    return out
