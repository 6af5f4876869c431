"""CPU oracle for the KDA forward path.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library (``linear_attention_
serving_fwd_gb300``) never imports it and has no CPU fallback.

Contents
--------
* ``kda_oracle.c`` - the fp64 token-by-token recurrence (the definition),
  built with gcc + OpenMP into ``_build/libkda_oracle.so`` and called through
  ctypes by :func:`recurrence`.
* ``chunked.py`` - an independent numpy fp64 chunk-form (WY/UT) formulation
  and the chunk-group scan; it shares no code with the C file and checks it.
* :func:`prefill` / :func:`window` - host-side arrangement (slot gathers and
  scatters, null slots) around :func:`recurrence` for the prefill, decode and
  verify entry points.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkda_oracle.so")
_SRC = os.path.join(_HERE, "kda_oracle.c")
_lock = threading.Lock()
_lib = None

D = 128


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc -O2 -fopenmp).  Plain fp64 code: no fast-math,
    so the compiler keeps IEEE semantics and the operation order written."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


def open_library(path: str):
    """ctypes handle with the oracle's signatures for a built copy at ``path``."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.kda_oracle_recurrence.argtypes = [
        P, P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_double, ctypes.c_int, P, P, P, P, ctypes.c_int]
    lib.kda_oracle_recurrence.restype = ctypes.c_int
    lib.kda_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = open_library(_SO)
    return _lib


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def _f32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> numpy (bf16 values are exact in fp32)
        import torch
        x = x.detach().to("cpu", torch.float32).numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def recurrence(q, k, v, g, beta, cu_seqlens, *, A_log=None, dt_bias=None,
               scale=D ** -0.5, lower_bound=-5.0, use_qk_l2norm=True, h0=None,
               want_out=True, want_state=True, want_corr=False, n_threads=0):
    """Run the fp64 token recurrence over every sequence and head.

    q, k: [T, Hqk, 128]; v, g: [T, Hv, 128]; beta: [T, Hv] (logits);
    cu_seqlens: [N+1]; h0: [N, Hv, 128, 128] (V-first) or None.
    Returns dict(out=[T,Hv,128], state=[N,Hv,128,128], corr=[T,Hv,128]) fp64.
    """
    lib = _load()
    q, k, v, g, beta = (_f32(t) for t in (q, k, v, g, beta))
    A_log, dt_bias = _f32(A_log), _f32(dt_bias)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens), dtype=np.int64)
    T, hqk = q.shape[0], q.shape[1]
    hv = v.shape[1]
    n = cu.shape[0] - 1
    assert q.shape == (T, hqk, D) and k.shape == q.shape
    assert v.shape == (T, hv, D) and g.shape == v.shape and beta.shape == (T, hv)
    if h0 is not None:
        if hasattr(h0, "detach"):
            h0 = h0.detach().cpu().double().numpy()
        h0 = np.ascontiguousarray(h0, dtype=np.float64)
        assert h0.shape == (n, hv, D, D)
    out = np.zeros((T, hv, D)) if want_out else None
    hT = np.zeros((n, hv, D, D)) if want_state else None
    corr = np.zeros((T, hv, D)) if want_corr else None
    rc = lib.kda_oracle_recurrence(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
        _ptr(cu), n, hqk, hv, float(scale), float(lower_bound), int(bool(use_qk_l2norm)),
        _ptr(h0), _ptr(out), _ptr(hT), _ptr(corr), int(n_threads))
    if rc != 0:
        raise ValueError("kda_oracle_recurrence rejected its arguments")
    return dict(out=out, state=hT, corr=corr)


def round_bf16(a):
    """fp64 values rounded to bf16 as a kernel holding them in fp32 would:
    to fp32, then to bf16, each to nearest even (torch's casts)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def _is_bf16(t):
    if t is None:
        return False
    import torch
    return getattr(t, "dtype", None) == torch.bfloat16


def prefill(x, *, want_corr=False, n_threads=0):
    """Oracle for ``kda_chunk_fwd`` on a :class:`KdaInputs` batch.

    Initial states come from ``initial_state`` or from the paged cache rows
    ``state_pool[state_indices[n]]`` (zero where ``has_initial_state[n]`` is
    false).  Returns out, the final states [N, Hv, 128, 128], and, for the
    paged form, the whole updated pool (final states written to their rows).
    With bf16 states (the pool or initial state stored as bf16) the states
    are read widened and the final ones rounded to bf16 once, at the end:
    the chunk path keeps its state in fp32 across the whole sequence.
    """
    n = x.n_seqs
    h0 = None
    pool = None
    if x.state_pool is not None:
        pool = x.state_pool.detach().cpu().double().numpy().copy()
        idx = x.state_indices.cpu().numpy().astype(np.int64)
        hi = (x.has_initial_state.cpu().numpy().astype(bool)
              if x.has_initial_state is not None else np.ones(n, bool))
        h0 = np.zeros((n, x.hv, D, D))
        for i in range(n):
            if idx[i] >= 0 and hi[i]:
                h0[i] = pool[idx[i]]
    elif x.initial_state is not None:
        h0 = x.initial_state.detach().cpu().double().numpy()
    res = recurrence(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, A_log=x.A_log,
                     dt_bias=x.dt_bias, scale=x.scale, lower_bound=x.lower_bound,
                     h0=h0, want_corr=want_corr, n_threads=n_threads)
    if _is_bf16(x.state_pool) or _is_bf16(x.initial_state):
        res["state"] = round_bf16(res["state"])
    if pool is not None:
        idx = x.state_indices.cpu().numpy().astype(np.int64)
        for i in range(n):
            if idx[i] >= 0:
                pool[idx[i]] = res["state"][i]
        res["pool"] = pool
    return res


def _token_steps(x, h0, starts, lens, *, bf16, n_threads=0):
    """Run each live request's tokens one at a time from h0 [R, Hv, 128, 128]
    (request r's tokens starts[r] .. starts[r] + lens[r] - 1), rounding the
    carried state to bf16 after every token when ``bf16``: the MATE decode
    page's bf16 state, stored after each decoded token.  Returns the per
    token outputs and corrections [T, Hv, 128] and the states after every
    token, states[t][r] (None past a request's length)."""
    T, hv = x.t_total, x.hv
    out = np.zeros((T, hv, D))
    corr = np.zeros((T, hv, D))
    S = [h0[r] for r in range(len(starts))]
    states = []
    for t in range(max(lens, default=0)):
        live = [r for r in range(len(starts)) if lens[r] > t]
        tok = np.asarray([starts[r] + t for r in live])
        res = recurrence(x.q[tok], x.k[tok], x.v[tok], x.g[tok], x.beta[tok],
                         np.arange(len(live) + 1), A_log=x.A_log, dt_bias=x.dt_bias,
                         scale=x.scale, lower_bound=x.lower_bound, h0=np.stack([S[r] for r in live]),
                         want_corr=True, n_threads=n_threads)
        out[tok] = res["out"]
        corr[tok] = res["corr"]
        st = round_bf16(res["state"]) if bf16 else res["state"]
        row = [None] * len(starts)
        for i, r in enumerate(live):
            S[r] = st[i]
            row[r] = st[i]
        states.append(row)
    return out, corr, states


def window(x, *, n_threads=0):
    """Oracle for ``kda_decode`` / ``kda_verify`` on a decode batch.

    Request b runs its tokens cu_seqlens[b]..cu_seqlens[b+1]-1 from pool row
    ``state_indices[b]``.  A negative slot is a padding entry: zero output,
    no correction records, and its (nonexistent) row untouched.  Returns
    out [T, Hv, 128], corr [T, Hv, 128] (U_t), and the pool after the decode
    (the verify pool is the input pool, unchanged).  A bf16 pool is read
    widened and the carried state rounded to bf16 after every token.
    """
    if _is_bf16(x.state_pool):
        return _window_bf16(x, n_threads=n_threads)
    n = x.n_seqs
    pool = x.state_pool.detach().cpu().double().numpy().copy()
    idx = x.state_indices.cpu().numpy().astype(np.int64)
    h0 = np.zeros((n, x.hv, D, D))
    for b in range(n):
        if idx[b] >= 0:
            h0[b] = pool[idx[b]]
    res = recurrence(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, A_log=x.A_log,
                     dt_bias=x.dt_bias, scale=x.scale, lower_bound=x.lower_bound,
                     h0=h0, want_corr=True, n_threads=n_threads)
    cu = x.cu_seqlens.cpu().numpy()
    for b in range(n):
        if idx[b] >= 0:
            pool[idx[b]] = res["state"][b]
        else:
            res["out"][cu[b]:cu[b + 1]] = 0.0
            res["corr"][cu[b]:cu[b + 1]] = 0.0
    res["pool"] = pool
    return res


def _window_bf16(x, *, n_threads=0):
    pool = x.state_pool.detach().cpu().double().numpy().copy()
    idx = x.state_indices.cpu().numpy().astype(np.int64)
    cu = x.cu_seqlens.cpu().numpy().astype(np.int64)
    live = [b for b in range(x.n_seqs) if idx[b] >= 0 and cu[b + 1] > cu[b]]
    h0 = np.stack([pool[idx[b]] for b in live]) if live else np.zeros((0, x.hv, D, D))
    out, corr, states = _token_steps(x, h0, [int(cu[b]) for b in live],
                                     [int(cu[b + 1] - cu[b]) for b in live], bf16=True,
                                     n_threads=n_threads)
    for b in range(x.n_seqs):
        if idx[b] < 0:
            out[cu[b]:cu[b + 1]] = 0.0
            corr[cu[b]:cu[b + 1]] = 0.0
    for i, b in enumerate(live):
        pool[idx[b]] = states[int(cu[b + 1] - cu[b]) - 1][i]
    return dict(out=out, corr=corr, pool=pool, state=None)


def window_steps(x, table, num_accepted=None, *, n_threads=0):
    """Oracle for ``kda_decode_steps``: decode with a [request, step] slot table.

    Follows the MATE ``gated_delta_rule_decode`` arguments ``state_indices``
    ([B, T]) and ``num_accepted_tokens`` as read here: request b starts from
    pool row ``table[b, c]`` with c = num_accepted[b] - 1 (0 without counts),
    and the state after its token t is stored to row ``table[b, t]``
    (negative: no store), rows written in token order.  A negative start row
    makes b padding (zero output, nothing stored).  A start column outside
    the table, or a row >= the pool size at the start column or at any of
    b's token columns, flags the call and b is treated as padding.

    Every state is the recurrence itself: the state after token t is the
    final state of the recurrence run on b's first t + 1 tokens (with a bf16
    pool: run token by token, the carried state rounded to bf16 after each).
    Returns out [T, Hv, 128], the pool after the call, and ``bad``.
    """
    n = x.n_seqs
    pool0 = x.state_pool.detach().cpu().double().numpy()
    pool = pool0.copy()
    n_slots = pool.shape[0]
    tab = np.asarray(table.cpu().numpy() if hasattr(table, "cpu") else table, dtype=np.int64)
    na = None
    if num_accepted is not None:
        na = np.asarray(num_accepted.cpu().numpy() if hasattr(num_accepted, "cpu") else num_accepted,
                        dtype=np.int64)
    cu = np.asarray(x.cu_seqlens.cpu().numpy(), dtype=np.int64)
    q, k, v, g, beta = (_f32(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    out = np.zeros((int(cu[-1]), x.hv, D))
    bad = False
    live = []  # (request, start row, length)
    for b in range(n):
        L = int(cu[b + 1] - cu[b])
        col = int(na[b]) - 1 if na is not None else 0
        if col < 0 or col >= tab.shape[1]:
            bad = True
            continue
        if L <= 0:
            continue
        r0 = int(tab[b, col])
        if r0 >= n_slots or np.any(tab[b, :L] >= n_slots):
            bad = True
            continue
        if r0 >= 0:
            live.append((b, r0, L))
    if _is_bf16(x.state_pool):
        if live:
            o, _, states = _token_steps(x, np.stack([pool0[r0] for _, r0, _ in live]),
                                        [int(cu[b]) for b, _, _ in live], [L for _, _, L in live],
                                        bf16=True, n_threads=n_threads)
            for i, (b, r0, L) in enumerate(live):
                out[int(cu[b]):int(cu[b]) + L] = o[int(cu[b]):int(cu[b]) + L]
                for t in range(L):
                    row = int(tab[b, t])
                    if row >= 0:
                        pool[row] = states[t][i]
        return dict(out=out, pool=pool, bad=bad)
    # one sequence per (request, prefix length): tokens cu[b] .. cu[b] + t
    sel, starts, h0 = [], [0], []
    for b, r0, L in live:
        for t in range(L):
            sel.extend(range(int(cu[b]), int(cu[b]) + t + 1))
            starts.append(len(sel))
            h0.append(pool0[r0])
    if live:
        sel = np.asarray(sel)
        res = recurrence(q[sel], k[sel], v[sel], g[sel], beta[sel], np.asarray(starts),
                         A_log=x.A_log, dt_bias=x.dt_bias, scale=x.scale,
                         lower_bound=x.lower_bound, h0=np.stack(h0), n_threads=n_threads)
        piece = 0
        for b, r0, L in live:
            for t in range(L):
                if t == L - 1:  # the full window: its outputs are the decode's
                    a, e = starts[piece], starts[piece + 1]
                    out[int(cu[b]):int(cu[b]) + L] = res["out"][a:e]
                row = int(tab[b, t])
                if row >= 0:
                    pool[row] = res["state"][piece]
                piece += 1
    return dict(out=out, pool=pool, bad=bad)
