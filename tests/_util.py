"""Shared helpers of the GPU tests: device transfer, oracle on sampled heads,
error metrics."""
import numpy as np
import torch

from oracle import kda_oracle

# Tolerances of the path: relative L2 error over a whole tensor (fp64), per input dtype.
REL_L2 = {torch.bfloat16: 1e-2, torch.float32: 1e-4}
# Element-wise guard against localised faults (not part of the stated bar): an element may be
# off by MAX_ERR_RMS of the reference's RMS plus ELEM_REL of its own magnitude.  bf16 outputs
# and operands carry a 2^-9 relative rounding each and the chunked form chains a few of them,
# so the error of a large element grows with the element (the full-size workloads have
# outputs beyond 20x their RMS); a value from a wrong tile, item or state is off by about
# the values themselves.
MAX_ERR_RMS = {torch.bfloat16: 0.1, torch.float32: 1e-3}
ELEM_REL = {torch.bfloat16: 2.0 ** -6, torch.float32: 0.0}
# Per-item guard (each (sequence, v-head) item on its own): three times the stated bar.  Items
# of one to a few tokens hold only 128 to a few hundred outputs, whose relative L2 scatters
# around the tensor's (up to 1.3e-2 over 27,000 such items); a wrong item is off by ~1.
ITEM_REL_L2 = {k: 3.0 * v for k, v in REL_L2.items()}


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
        bound = MAX_ERR_RMS[dtype] if max_rms is None else max_rms
        excess = np.abs(x - ref) - (bound * rms + ELEM_REL[dtype] * np.abs(ref))
        i = int(np.argmax(excess))
        assert excess.flat[i] <= 0, (
            f"{what}: element {np.unravel_index(i, x.shape)} error {abs(x.flat[i] - ref.flat[i]) / rms:.3e} "
            f"RMS > {bound} RMS + {ELEM_REL[dtype]:.3g} x |ref| ({abs(ref.flat[i]) / rms:.2f} RMS)")
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


def assert_items_close(o, o_ref, cu, dtype, what="o", max_rms=None):
    """The whole tensor at the stated bar, then every (sequence, v-head) item of o [T, Hv, V]
    on its own at ITEM_REL_L2: a fault confined to some items (a wrong chunk, state or claim)
    cannot hide behind the others.  Returns the worst item error."""
    x = o.detach().cpu().double().numpy() if hasattr(o, "detach") else np.asarray(o, np.float64)
    ref = np.asarray(o_ref, np.float64)
    assert_close(x, ref, dtype, what, max_rms=max_rms)
    worst, where = 0.0, None
    cu = [int(c) for c in cu]
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if b <= a:
            continue
        d = np.linalg.norm(x[a:b] - ref[a:b], axis=(0, 2))
        r = np.linalg.norm(ref[a:b], axis=(0, 2))
        e = d / np.where(r > 0, r, 1.0)
        h = int(np.argmax(e))
        if e[h] > worst:
            worst, where = float(e[h]), (n, h)
    assert worst <= ITEM_REL_L2[dtype], \
        f"{what}: item {where} relative L2 {worst:.3e} > {ITEM_REL_L2[dtype]:.0e}"
    return worst


def assert_rows_close(x, ref, dtype, what="state"):
    """The whole tensor at the stated bar, then each leading-axis row of x (e.g. a state
    [Hv, K, V] per slot) on its own, per (row, v-head), at ITEM_REL_L2."""
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert_close(x, ref, dtype, what)
    ax = tuple(range(2, x.ndim))
    d = np.linalg.norm(x - ref, axis=ax)
    r = np.linalg.norm(ref, axis=ax)
    e = d / np.where(r > 0, r, 1.0)
    i = np.unravel_index(int(np.argmax(e)), e.shape)
    assert e[i] <= ITEM_REL_L2[dtype], f"{what}: row {i} relative L2 {e[i]:.3e} > {ITEM_REL_L2[dtype]:.0e}"
    return float(e[i])
