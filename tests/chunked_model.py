"""fp64 numpy model of the chunked KDA algorithm exactly as the CUDA kernels
organise it (test-side blueprint; never imported by the library or the oracle).

Per chunk of C tokens (aligned to the sequence start, last one partial):

  e_r      = exp(g_r)                                    [C, K], 1 on padded rows
  rho_r    = prod_{j = start(sub(r))}^{r} e_j            inclusive, within the sub-chunk
  kap_r    = prod_{j = r+1}^{end(sub(r))} e_j            exclusive, within the sub-chunk
  pi_s     = product of e over sub-chunk s
  E_s, F_s = products of pi over the sub-chunks before / after s
  KG = k rho E,  QG = scale q rho E,  KR = k kap F,  gamma = prod e     (all factors <= 1)

  A[r,i] = beta_r sum_c k_r k_i prod_{j=i+1}^{r} e_j   (i < r)
  B[r,i] = scale  sum_c q_r k_i prod_{j=i+1}^{r} e_j   (i <= r)

  off-diagonal sub-chunk blocks (row block a > column block b) factor as
      (k_r rho_r) . (k_i kap_i prod_{b<s<a} pi_s)            every factor <= 1
  diagonal blocks use (k_r rho_r) . (k_i / rho_i) on channels whose sub-chunk
  product pi_a >= 2**-100 (so 1/rho <= 2**100), and the explicit pairwise product
  on the remaining ("unsafe") channels.

  Tm = (I + A)^-1 diag(beta)   (16x16 diagonal blocks by forward substitution,
                                merged pairwise: X21 = -X22 A21 X11)
  U~ = Tm V,  W = Tm KG,  U = U~ - W S,  O = QG S + B U,  S <- diag(gamma) S + KR^T U
"""
import numpy as np

SAFE_MIN = 2.0 ** -100


def tri_inv_unit_lower_blocked(A, bs=16):
    """(I + A)^-1 for strictly lower A, 16x16 diagonal blocks then pairwise merges."""
    C = A.shape[0]
    X = np.zeros_like(A)
    for b0 in range(0, C, bs):  # diagonal blocks: forward substitution
        blk = A[b0:b0 + bs, b0:b0 + bs]
        n = blk.shape[0]
        Xi = np.eye(n)
        for r in range(n):
            for i in range(r):
                Xi[r] -= blk[r, i] * Xi[i]
        X[b0:b0 + bs, b0:b0 + bs] = Xi
    w = bs
    while w < C:  # merge [[X11, 0], [A21, X22]] blocks of width w into 2w
        for b0 in range(0, C, 2 * w):
            m = b0 + w
            if m >= C:
                continue
            e = min(b0 + 2 * w, C)
            X[m:e, b0:m] = -X[m:e, m:e] @ A[m:e, b0:m] @ X[b0:m, b0:m]
        w *= 2
    return X


def chunk_quantities(q, k, v, g, beta, c, C=64, s=16, scale=1.0):
    """S-independent quantities of one chunk (inputs already padded to C rows)."""
    K = k.shape[1]
    valid = np.arange(C) < c
    e = np.where(valid[:, None], np.exp(g), 1.0)
    k = np.where(valid[:, None], k, 0.0)
    q = np.where(valid[:, None], q, 0.0)
    b = np.where(valid, beta, 0.0)
    ns = C // s
    sub = np.arange(C) // s
    rho = np.empty((C, K))
    kap = np.empty((C, K))
    for a in range(ns):
        p = np.ones(K)
        for r in range(a * s, a * s + s):
            p = p * e[r]
            rho[r] = p
        p = np.ones(K)
        for r in range(a * s + s - 1, a * s - 1, -1):
            kap[r] = p
            p = p * e[r]
    pi = np.stack([rho[a * s + s - 1] for a in range(ns)])
    E = np.ones((ns, K))
    F = np.ones((ns, K))
    for a in range(1, ns):
        E[a] = E[a - 1] * pi[a - 1]
    for a in range(ns - 2, -1, -1):
        F[a] = F[a + 1] * pi[a + 1]
    gamma = E[ns - 1] * pi[ns - 1]
    KG = k * rho * E[sub]
    QG = scale * q * rho * E[sub]
    KR = k * kap * F[sub]
    Krho, Qrho = k * rho, q * rho

    A = np.zeros((C, C))
    B = np.zeros((C, C))
    for a in range(ns):
        rows = slice(a * s, a * s + s)
        for bb in range(a):  # off-diagonal blocks, reference = start of row block a
            cols = slice(bb * s, bb * s + s)
            mid = np.ones(K)
            for t in range(bb + 1, a):
                mid = mid * pi[t]
            Ccol = k[cols] * kap[cols] * mid
            A[rows, cols] = Krho[rows] @ Ccol.T
            B[rows, cols] = Qrho[rows] @ Ccol.T
        safe = pi[a] >= SAFE_MIN
        DG = np.where(safe, k[rows] / np.where(safe, rho[rows], 1.0), 0.0)
        Ad = Krho[rows] @ DG.T
        Bd = Qrho[rows] @ DG.T
        for ch in np.nonzero(~safe)[0]:  # pairwise products on unsafe channels
            for i in range(s):
                f = 1.0
                for r in range(i, s):
                    if r > i:
                        f *= e[a * s + r, ch]
                    Ad[r, i] += k[a * s + r, ch] * k[a * s + i, ch] * f
                    Bd[r, i] += q[a * s + r, ch] * k[a * s + i, ch] * f
        A[rows, rows] = Ad
        B[rows, rows] = Bd
    A = np.tril(A, -1) * b[:, None]
    B = np.tril(B) * scale
    Tm = tri_inv_unit_lower_blocked(A, s) * b[None, :]
    vv = np.where(valid[:, None], v, 0.0)
    return dict(Ut=Tm @ vv, W=Tm @ KG, QG=QG, KR=KR, B=B, gamma=gamma, A=A, Tm=Tm)


def chunked_forward(q, k, v, g, beta, cu, S0, scale, C=64, s=16):
    """Chunked prefill over packed sequences; S0 is dense [N, Hv, K, V]."""
    T, Hk, K = q.shape
    Hv, V = v.shape[1:]
    N = len(cu) - 1
    o = np.zeros((T, Hv, V))
    fin = np.zeros((N, Hv, K, V))
    for n in range(N):
        for h in range(Hv):
            kh = h // (Hv // Hk)
            S = S0[n, h].astype(np.float64).copy()
            for t0 in range(cu[n], cu[n + 1], C):
                c = min(C, cu[n + 1] - t0)
                pad = lambda x: np.concatenate([x, np.zeros((C - c,) + x.shape[1:])]) if c < C else x
                Qc = chunk_quantities(pad(q[t0:t0 + c, kh]), pad(k[t0:t0 + c, kh]),
                                      pad(v[t0:t0 + c, h]), pad(g[t0:t0 + c, h]),
                                      pad(beta[t0:t0 + c, h]), c, C, s, scale)
                U = Qc["Ut"] - Qc["W"] @ S
                O = Qc["QG"] @ S + Qc["B"] @ U
                o[t0:t0 + c, h] = O[:c]
                S = Qc["gamma"][:, None] * S + Qc["KR"].T @ U
            fin[n, h] = S
    return o, fin


def split_state_passing(q, k, v, g, beta, cu, S0, scale, split_chunks, C=64, s=16):
    """The same prefill with every sequence longer than split_chunks chunks cut at that
    chunk boundary into two segments that need not run one after the other.

    The update is affine in the state, S_t = M_t S_p + S_t^loc with M_t the product of the
    per-token maps (I - beta k k^T) Diag(e^g) since the cut, so the second segment runs twice
    from the cut on, independently of the first: once from a zero state with the real values
    (o^loc, S^loc), once from the identity with zero values (its outputs are
    y_t = scale M_t^T q_t, its final state M_end).  The combine, once the first segment has
    produced S_p, is two products:  o_t = o_t^loc + y_t^T S_p  and  S_end = M_end S_p + S^loc.
    """
    T, Hk, K = q.shape
    Hv, V = v.shape[1:]
    N = len(cu) - 1
    o = np.zeros((T, Hv, V))
    fin = np.zeros((N, Hv, K, V))
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        cut = a + split_chunks * C
        if cut >= b:  # too short to split
            on, fn = chunked_forward(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], [0, b - a],
                                     S0[n:n + 1], scale, C, s)
            o[a:b], fin[n] = on, fn[0]
            continue
        seg1 = lambda x: x[a:cut]
        seg2 = lambda x: x[cut:b]
        o1, Sp = chunked_forward(seg1(q), seg1(k), seg1(v), seg1(g), seg1(beta), [0, cut - a],
                                 S0[n:n + 1], scale, C, s)
        o2l, S2l = chunked_forward(seg2(q), seg2(k), seg2(v), seg2(g), seg2(beta), [0, b - cut],
                                   np.zeros((1, Hv, K, V)), scale, C, s)
        eye = np.broadcast_to(np.eye(K), (1, Hv, K, K)).copy()
        y, Mend = chunked_forward(seg2(q), seg2(k), np.zeros((b - cut, Hv, K)), seg2(g),
                                  seg2(beta), [0, b - cut], eye, scale, C, s)
        o[a:cut] = o1
        for h in range(Hv):
            o[cut:b, h] = o2l[:, h] + y[:, h] @ Sp[0, h]
            fin[n, h] = Mend[0, h] @ Sp[0, h] + S2l[0, h]
    return o, fin
