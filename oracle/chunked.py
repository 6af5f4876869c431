"""Independent chunk-form (WY/UT) KDA formulation in numpy fp64.
TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Shares no code with ``kda_oracle.c``; the two must agree to ~1e-12.  It
follows the chunk decomposition that the vLLM kimi_k3 AMD ``kda_chunk`` page
describes (``fused_kda_prologue``: gate cumsum, two intra-chunk passes, the
w/u recompute; ``fused_kda_chunk``: the inter-chunk walk fused with the
output) and the chunk-group scan of ``_chunk_groups`` (transfer operator
M_g = prod_c (diag(d_c) - w_c^T kg_c)).

Notation per chunk of C rows r = 0..C-1 (K = V = 128), S is K x V:
  Lam_r   = sum_{j<=r} gate_j                       (per key channel)
  A_kk    = [beta_r sum_c k^_rc k^_ic e^{Lam_rc - Lam_ic}]_{i<r}
  A_qk    = [sum_c q~_rc k^_ic e^{Lam_rc - Lam_ic}]_{i<=r}
  T       = (I + A_kk)^{-1} diag(beta)
  w       = T (e^{Lam} * k^),   u = T v
  U       = u - w S
  o       = (e^{Lam} * q~) S + A_qk U
  S'      = diag(e^{Lam_C}) S + (e^{Lam_C - Lam} * k^)^T U
where Lam_C is the last row.  In the V-first storage the update reads
S'^T = S^T (diag(d) - w^T kg) + u^T kg, the page's transfer operator.
"""
from __future__ import annotations

import numpy as np

D = 128


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def activations(q, k, g, beta, A_log_h, dt_bias_h, scale, lower_bound, l2norm=True):
    """Per-token activations for one head: q~, k^, gate (log decay), beta."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    g = np.asarray(g, np.float64)
    if A_log_h is None:
        gate = g
    else:
        gate = lower_bound * _sig(np.exp(float(A_log_h)) * (g + np.asarray(dt_bias_h, np.float64)))
    if l2norm:
        kh = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
        qh = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
    else:
        kh, qh = k, q
    return scale * qh, kh, gate, _sig(np.asarray(beta, np.float64))


def commit_from_records(S0, kg_raw, corr, A_log_h, dt_bias_h, lower_bound):
    """The state after an accepted prefix, rebuilt from speculative verify's
    records (the vLLM kimi_k3 verify page writes corr = U_t and kg = raw k_t,
    raw g_t so that it can be rebuilt).  Unrolling S_t = diag(e^{gate_t})
    S_{t-1} + k^_t U_t^T over the accepted tokens t = 1..a gives

        S_a = diag(e^{L_a}) S_0 + sum_{t <= a} diag(e^{L_a - L_t}) k^_t U_t^T

    with L_t the per-channel cumsum of the gates.  S0 is V-first [V, K];
    kg_raw [a, 2K] (raw k, raw g); corr [a, V].  Returns the V-first S_a."""
    kg_raw = np.asarray(kg_raw, np.float64)
    corr = np.asarray(corr, np.float64)
    a = corr.shape[0]
    S = np.asarray(S0, np.float64).T.copy()  # K x V
    if a == 0:
        return S.T
    k, g = kg_raw[:, :D], kg_raw[:, D:]
    _, kh, gate, _ = activations(k, k, g, np.zeros(a), A_log_h, dt_bias_h, 1.0, lower_bound)
    L = np.cumsum(gate, axis=0)                        # [a, K]
    S *= np.exp(L[-1])[:, None]
    for t in range(a):
        S += np.outer(np.exp(L[-1] - L[t]) * kh[t], corr[t])
    return S.T


def chunk_operands(qh, kh, gate, b):
    """Intra-chunk quantities for one chunk (rows beyond the chunk absent)."""
    C = kh.shape[0]
    lam = np.cumsum(gate, axis=0)                     # [C, K]
    diff = lam[:, None, :] - lam[None, :, :]          # [r, i, K]
    low = np.tril(np.ones((C, C), bool), -1)
    lowd = np.tril(np.ones((C, C), bool), 0)
    ex = np.exp(np.where(lowd[:, :, None], diff, -np.inf))
    Akk = b[:, None] * np.einsum("rc,ic,ric->ri", kh, kh, ex) * low
    Aqk = np.einsum("rc,ic,ric->ri", qh, kh, ex) * lowd
    Tm = np.linalg.solve(np.eye(C) + Akk, np.diag(b))
    kd = np.exp(lam) * kh
    w = Tm @ kd
    qg = np.exp(lam) * qh
    d = np.exp(lam[-1])
    kg = np.exp(lam[-1][None, :] - lam) * kh
    return dict(Akk=Akk, Aqk=Aqk, T=Tm, w=w, qg=qg, kg=kg, d=d)


def chunk_step(ops, v, S):
    """One chunk of the walk: returns (o, U, S_next).  S is K x V."""
    u = ops["T"] @ v
    U = u - ops["w"] @ S
    o = ops["qg"] @ S + ops["Aqk"] @ U
    S_next = ops["d"][:, None] * S + ops["kg"].T @ U
    return o, U, S_next


def sequence_chunked(q, k, v, g, beta, A_log_h, dt_bias_h, scale, lower_bound,
                     S0=None, chunk=64, l2norm=True):
    """One (sequence, head): inputs [L, 128] (beta [L]).  S0 is the V-first
    state [V, K] or None.  Returns (o [L, V], corr [L, V], final V-first)."""
    qh, kh, gate, b = activations(q, k, g, beta, A_log_h, dt_bias_h, scale, lower_bound, l2norm)
    L = qh.shape[0]
    S = np.zeros((D, D)) if S0 is None else np.asarray(S0, np.float64).T.copy()
    o = np.zeros((L, D))
    corr = np.zeros((L, D))
    v = np.asarray(v, np.float64)
    for s in range(0, L, chunk):
        e = min(L, s + chunk)
        ops = chunk_operands(qh[s:e], kh[s:e], gate[s:e], b[s:e])
        o[s:e], corr[s:e], S = chunk_step(ops, v[s:e], S)
    return o, corr, S.T.copy()


def sequence_group_scan(q, k, v, g, beta, A_log_h, dt_bias_h, scale, lower_bound,
                        S0=None, chunk=64, groups=4, l2norm=True):
    """The chunk-group parallel scan for one (sequence, head).

    Pass one walks every group from a zero state to get B_g and composes its
    exact transfer operator M_g (S_end = M_g S_start + B_g); the serial scan
    then gives each group's incoming state; pass two re-walks each group from
    that state for the outputs.  Same results as :func:`sequence_chunked`.
    """
    qh, kh, gate, b = activations(q, k, g, beta, A_log_h, dt_bias_h, scale, lower_bound, l2norm)
    L = qh.shape[0]
    v = np.asarray(v, np.float64)
    starts = list(range(0, L, chunk))
    n_chunks = len(starts)
    per = -(-n_chunks // groups)
    bounds = [(gi * per, min(n_chunks, (gi + 1) * per)) for gi in range(groups)]
    bounds = [bb for bb in bounds if bb[0] < bb[1]]
    ops_all = []
    for s in starts:
        e = min(L, s + chunk)
        ops_all.append((chunk_operands(qh[s:e], kh[s:e], gate[s:e], b[s:e]), v[s:e]))
    # pass one: (M_g, B_g) per group, independent of every other group
    Ms, Bs = [], []
    for c0, c1 in bounds:
        M = np.eye(D)
        Bg = np.zeros((D, D))
        for c in range(c0, c1):
            ops, vc = ops_all[c]
            Ac = np.diag(ops["d"]) - ops["kg"].T @ ops["w"]
            bc = ops["kg"].T @ (ops["T"] @ vc)
            M = Ac @ M
            Bg = Ac @ Bg + bc
        Ms.append(M)
        Bs.append(Bg)
    # serial composition over groups
    S = np.zeros((D, D)) if S0 is None else np.asarray(S0, np.float64).T.copy()
    S_in = []
    for M, Bg in zip(Ms, Bs):
        S_in.append(S)
        S = M @ S + Bg
    final = S
    # pass two: outputs from each group's incoming state
    o = np.zeros((L, D))
    for (c0, c1), Sg in zip(bounds, S_in):
        St = Sg
        for c in range(c0, c1):
            ops, vc = ops_all[c]
            s = starts[c]
            e = min(L, s + chunk)
            o[s:e], _, St = chunk_step(ops, vc, St)
    return o, final.T.copy()


def run(x, *, chunk=64, groups=None, l2norm=True):
    """Chunked oracle over a whole KdaInputs batch (all sequences, heads).
    Returns out [T, Hv, 128] and final states [N, Hv, 128, 128] (V-first)."""
    import torch

    f = lambda t: t.detach().to("cpu", torch.float32).numpy().astype(np.float64)
    q, k, v, g, beta = f(x.q), f(x.k), f(x.v), f(x.g), f(x.beta)
    A_log = None if x.A_log is None else f(x.A_log)
    dt = None if x.dt_bias is None else f(x.dt_bias)
    cu = x.cu_seqlens.cpu().numpy()
    n = len(cu) - 1
    r = x.hv // x.hqk
    out = np.zeros((x.t_total, x.hv, D))
    final = np.zeros((n, x.hv, D, D))
    for i in range(n):
        s, e = int(cu[i]), int(cu[i + 1])
        for h in range(x.hv):
            hq = h // r
            S0 = None
            if x.initial_state is not None:
                S0 = f(x.initial_state[i, h])
            elif x.state_pool is not None:
                idx = int(x.state_indices[i])
                hi = True if x.has_initial_state is None else bool(x.has_initial_state[i])
                if idx >= 0 and hi:
                    S0 = f(x.state_pool[idx, h])
            args = (q[s:e, hq], k[s:e, hq], v[s:e, h], g[s:e, h], beta[s:e, h],
                    None if A_log is None else A_log[h], None if dt is None else dt[h],
                    x.scale, x.lower_bound)
            if groups:
                o, St = sequence_group_scan(*args, S0=S0, chunk=chunk, groups=groups,
                                            l2norm=l2norm)
            else:
                o, _, St = sequence_chunked(*args, S0=S0, chunk=chunk, l2norm=l2norm)
            out[s:e, h] = o
            final[i, h] = St
    return out, final
