"""Pins for the CPU oracle: every check here ties the oracle to something
other than itself - closed forms the recurrence must reduce to, brute-force
matrix products, an independently written chunk form, the group-scan
composition, invariances, and hand-derived gate values under tests/golden/.
CPU only (no GPU)."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from linear_attention_serving_fwd_gb300 import workloads as W

D = 128
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(T, hqk=1, hv=1, seed=0, lb=-5.0, g_shift=0.0, bf16=True):
    gen = torch.Generator().manual_seed(seed)
    t = lambda *s: torch.randn(*s, generator=gen)
    q, k = t(T, hqk, D), t(T, hqk, D)
    v, g = t(T, hv, D), t(T, hv, D) + g_shift
    b = t(T, hv)
    if bf16:
        q, k, v, g, b = (x.bfloat16().float() for x in (q, k, v, g, b))
    A_log = torch.log(torch.rand(hv, generator=gen) * 15 + 1)
    dt = t(hv, D) * 0.1
    return q, k, v, g, b, A_log, dt


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# --- closed forms -----------------------------------------------------------

def test_gate_golden_values():
    """Per-token log decay equals the hand-derived values in the fixture.
    With beta = 0 one token maps S0 to diag(exp(gate)) S0, so the log ratio
    of final to initial state exposes the gate of every key channel."""
    fx = json.load(open(os.path.join(GOLDEN, "gate_closed_form.json")))
    for case in fx["cases"]:
        q = torch.randn(1, 1, D)
        k = torch.randn(1, 1, D)
        v = torch.randn(1, 1, D)
        g = torch.full((1, 1, D), case["g"])
        b = torch.full((1, 1), -1e4)  # sigmoid -> exactly 0 in fp64
        A_log = torch.tensor([case["A_log"]])
        dt = torch.full((1, D), case["dt_bias"])
        h0 = np.random.default_rng(1).uniform(0.5, 1.5, (1, 1, D, D))
        res = oracle.recurrence(q, k, v, g, b, [0, 1], A_log=A_log, dt_bias=dt,
                                lower_bound=case["lower_bound"], h0=h0)
        with np.errstate(invalid="ignore", divide="ignore"):  # a planted mistake may give a negative ratio
            gate = np.log(res["state"][0, 0] / h0[0, 0])
        np.testing.assert_allclose(gate, case["expected_gate"], atol=fx["tolerance"], rtol=0)


def test_beta_zero_gate_zero_leaves_state_and_reads_it():
    """beta = 0 and gate = 0 (lower_bound 0): the state is unchanged bit for
    bit and o_t = scale * S0^T q^_t (q^ the normalised query)."""
    T = 37
    q, k, v, g, b, A_log, dt = _rand_inputs(T)
    b[:] = -np.inf
    h0 = np.random.default_rng(2).normal(0, 0.5, (1, 1, D, D))
    scale = 0.3
    res = oracle.recurrence(q, k, v, g, b, [0, T], A_log=A_log, dt_bias=dt,
                            lower_bound=0.0, scale=scale, h0=h0)
    assert np.array_equal(res["state"], h0)
    qn = q[:, 0].double().numpy()
    qn = qn / np.sqrt((qn * qn).sum(-1, keepdims=True) + 1e-6)
    expect = scale * qn @ h0[0, 0].T  # S0^T q with S0^T stored [V][K]
    np.testing.assert_allclose(res["out"][:, 0], expect, rtol=1e-12, atol=1e-14)


def test_single_token_from_zero_state():
    """One token from a zero state: S = beta k^ v^T and o = scale beta (k^.q^) v."""
    q, k, v, g, b, A_log, dt = _rand_inputs(1, seed=3)
    scale = D ** -0.5
    res = oracle.recurrence(q, k, v, g, b, [0, 1], A_log=A_log, dt_bias=dt, scale=scale)
    kk = k[0, 0].double().numpy()
    qq = q[0, 0].double().numpy()
    vv = v[0, 0].double().numpy()
    kh = kk / np.sqrt(kk @ kk + 1e-6)
    qh = qq / np.sqrt(qq @ qq + 1e-6)
    beta = 1 / (1 + np.exp(-float(b[0, 0])))
    np.testing.assert_allclose(res["out"][0, 0], scale * beta * (kh @ qh) * vv, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(res["state"][0, 0], beta * np.outer(vv, kh), rtol=1e-12, atol=1e-15)


def test_delta_rule_overwrite():
    """gate = 0, beta = 1: a token whose query equals its key reads back
    exactly its value, times |k^|^2, whatever the state held, because
    (I - k^ k^T) k^ = k^ (1 - |k^|^2) and the old content is erased."""
    q, k, v, g, b, A_log, dt = _rand_inputs(1, seed=4)
    q = k.clone()
    b[:] = np.inf
    h0 = np.random.default_rng(5).normal(0, 3.0, (1, 1, D, D))
    res = oracle.recurrence(q, k, v, g, b, [0, 1], A_log=A_log, dt_bias=dt,
                            lower_bound=0.0, scale=1.0, h0=h0)
    kk = k[0, 0].double().numpy()
    n2 = (kk @ kk) / (kk @ kk + 1e-6)
    # o = S0^T k^ (1 - n2) + v n2; with |k|^2 ~ 128, (1 - n2) ~ 8e-9
    kh = kk / np.sqrt(kk @ kk + 1e-6)
    expect = h0[0, 0] @ kh * (1 - n2) + v[0, 0].double().numpy() * n2
    np.testing.assert_allclose(res["out"][0, 0], expect, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(res["out"][0, 0], v[0, 0].double().numpy(), rtol=1e-6, atol=1e-6)


# --- brute force -------------------------------------------------------------

def _bruteforce(q, k, v, g, b, A_log, dt, scale, lb, h0):
    """Full 128x128 matrix form S_t = (I - b k k^T) diag(e^gate) S_{t-1} + b k v^T,
    o_t = S_t^T q, with S as K x V: an explicit product per token."""
    T = q.shape[0]
    S = h0.T.copy()
    outs = []
    a = np.exp(float(A_log[0]))
    for t in range(T):
        kk = k[t, 0].double().numpy()
        qq = q[t, 0].double().numpy()
        kh = kk / np.sqrt(kk @ kk + 1e-6)
        qh = scale * qq / np.sqrt(qq @ qq + 1e-6)
        gate = lb / (1 + np.exp(-a * (g[t, 0].double().numpy() + dt[0].double().numpy())))
        beta = 1 / (1 + np.exp(-float(b[t, 0])))
        P = np.eye(D) - beta * np.outer(kh, kh)
        S = P @ np.diag(np.exp(gate)) @ S + beta * np.outer(kh, v[t, 0].double().numpy())
        outs.append(S.T @ qh)
    return np.array(outs), S.T


@pytest.mark.parametrize("T,lb", [(1, -5.0), (5, -5.0), (8, -0.05)])
def test_bruteforce_tiny(T, lb):
    q, k, v, g, b, A_log, dt = _rand_inputs(T, seed=10 + T)
    h0 = np.random.default_rng(T).normal(0, 0.3, (1, 1, D, D))
    res = oracle.recurrence(q, k, v, g, b, [0, T], A_log=A_log, dt_bias=dt,
                            lower_bound=lb, h0=h0)
    o_bf, S_bf = _bruteforce(q, k, v, g, b, A_log, dt, D ** -0.5, lb, h0[0, 0])
    np.testing.assert_allclose(res["out"][:, 0], o_bf, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["state"][0, 0], S_bf, rtol=1e-11, atol=1e-13)


# --- independent chunk form and group scan -----------------------------------

@pytest.mark.parametrize("T,lb,g_shift", [(63, -5.0, 0.0), (64, -5.0, 0.0), (65, -0.05, 0.0),
                                          (200, -1.0, 0.0), (257, -5.0, -6.0)])
def test_chunk_form_matches_recurrence(T, lb, g_shift):
    x = W.dense_prefill(1, T, 1, 1, seed=T, lower_bound=lb, g_shift=g_shift)
    res = oracle.prefill(x, want_corr=True)
    out_c, fin_c = chunked.run(x)
    assert _rel(out_c, res["out"]) < 1e-11
    assert _rel(fin_c, res["state"]) < 1e-11


def test_chunk_form_varlen_gva():
    x = W.varlen_paged([70, 1, 129, 64], 2, 4, slots=6, seed=3, lower_bound=-0.3,
                       has_initial=[1, 0, 1, 1])
    res = oracle.prefill(x)
    out_c, fin_c = chunked.run(x)
    assert _rel(out_c, res["out"]) < 1e-11
    assert _rel(fin_c, res["state"]) < 1e-11


@pytest.mark.parametrize("groups", [2, 4, 5])
def test_group_scan_matches_recurrence(groups):
    """The chunk-group scan composes exact transfer operators, so it equals
    the serial recurrence to rounding for any group count."""
    x = W.dense_prefill(1, 64 * 9 + 17, 1, 1, seed=groups, lower_bound=-0.05)
    res = oracle.prefill(x)
    out_g, fin_g = chunked.run(x, groups=groups)
    assert _rel(out_g, res["out"]) < 1e-10
    assert _rel(fin_g, res["state"]) < 1e-10


# --- invariances ---------------------------------------------------------------

def test_split_invariance():
    """run(T) == run(T1) then run(T2) from the carried state."""
    x = W.dense_prefill(1, 150, 2, 2, seed=7, lower_bound=-0.1)
    full = oracle.prefill(x)
    T1 = 61
    a = oracle.recurrence(x.q[:T1], x.k[:T1], x.v[:T1], x.g[:T1], x.beta[:T1], [0, T1],
                          A_log=x.A_log, dt_bias=x.dt_bias, lower_bound=x.lower_bound,
                          h0=x.initial_state)
    b = oracle.recurrence(x.q[T1:], x.k[T1:], x.v[T1:], x.g[T1:], x.beta[T1:], [0, 150 - T1],
                          A_log=x.A_log, dt_bias=x.dt_bias, lower_bound=x.lower_bound,
                          h0=a["state"])
    np.testing.assert_allclose(np.concatenate([a["out"], b["out"]]), full["out"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b["state"], full["state"], rtol=1e-12, atol=1e-15)


def test_varlen_equals_dense_per_sequence():
    x = W.dense_prefill(3, 40, 1, 2, seed=8, lower_bound=-0.2)
    full = oracle.prefill(x)
    for i in range(3):
        s = slice(40 * i, 40 * (i + 1))
        one = oracle.recurrence(x.q[s], x.k[s], x.v[s], x.g[s], x.beta[s], [0, 40],
                                A_log=x.A_log, dt_bias=x.dt_bias, lower_bound=x.lower_bound,
                                h0=x.initial_state[i:i + 1])
        np.testing.assert_array_equal(one["out"], full["out"][s])
        np.testing.assert_array_equal(one["state"][0], full["state"][i])


def test_gva_equals_repeated_heads():
    """Value head h reads query/key head h // (Hv/Hqk): GVA equals running
    with q and k repeat-interleaved to Hv heads."""
    x = W.dense_prefill(1, 50, 2, 6, seed=9, lower_bound=-0.2)
    gva = oracle.prefill(x)
    rep = oracle.recurrence(x.q.repeat_interleave(3, dim=1), x.k.repeat_interleave(3, dim=1),
                            x.v, x.g, x.beta, x.cu_seqlens, A_log=x.A_log, dt_bias=x.dt_bias,
                            lower_bound=x.lower_bound, h0=x.initial_state)
    np.testing.assert_array_equal(gva["out"], rep["out"])
    np.testing.assert_array_equal(gva["state"], rep["state"])


def test_window_equals_repeated_single_tokens():
    """A Q-token decode equals Q single-token decodes on the carried state,
    and padding requests (slot -1) give zeros and touch no pool row."""
    x = W.decode_batch(6, 4, 2, 4, slots=10, seed=11, qlens=[4, 1, 0, 3, 4, 2],
                       null_requests=(4,), lower_bound=-0.5)
    res = oracle.window(x)
    pool = x.state_pool.double().numpy().copy()
    cu = x.cu_seqlens.tolist()
    idx = x.state_indices.tolist()
    for b in range(6):
        if idx[b] < 0:
            assert np.all(res["out"][cu[b]:cu[b + 1]] == 0)
            continue
        S = pool[idx[b]][None]
        for t in range(cu[b], cu[b + 1]):
            one = oracle.recurrence(x.q[t:t + 1], x.k[t:t + 1], x.v[t:t + 1], x.g[t:t + 1],
                                    x.beta[t:t + 1], [0, 1], A_log=x.A_log, dt_bias=x.dt_bias,
                                    lower_bound=x.lower_bound, h0=S, want_corr=True)
            np.testing.assert_allclose(res["out"][t], one["out"][0], rtol=1e-13, atol=1e-16)
            np.testing.assert_allclose(res["corr"][t], one["corr"][0], rtol=1e-13, atol=1e-16)
            S = one["state"]
        np.testing.assert_allclose(res["pool"][idx[b]], S[0], rtol=1e-13, atol=1e-16)
    untouched = [s for s in range(10) if s not in idx]
    assert np.array_equal(res["pool"][untouched], pool[untouched])


def test_slot_table_decode_states_and_reads():
    """The slot-table decode stores, at each column t, the state after t + 1
    single-token decodes from the start row (the accepted column), and with
    every column of a request on one slot it is the in-place window decode."""
    x = W.decode_batch(5, 4, 2, 4, slots=24, seed=12, qlens=[4, 3, 1, 4, 2], lower_bound=-0.7)
    pool = x.state_pool.double().numpy().copy()
    table = np.array([[0, 1, 2, 3], [4, -1, 6, 7], [8, 9, 10, 11], [-1, 12, 13, 14],
                      [15, 16, -1, -1]], dtype=np.int64)
    acc = np.array([2, 1, 4, 1, 3])
    res = oracle.window_steps(x, torch.from_numpy(table), torch.from_numpy(acc))
    assert not res["bad"]
    cu = x.cu_seqlens.tolist()
    written = set()
    for b in range(5):
        r0 = table[b, acc[b] - 1]
        if r0 < 0:
            assert np.all(res["out"][cu[b]:cu[b + 1]] == 0)
            continue
        S = pool[r0][None]
        for j, t in enumerate(range(cu[b], cu[b + 1])):
            one = oracle.recurrence(x.q[t:t + 1], x.k[t:t + 1], x.v[t:t + 1], x.g[t:t + 1],
                                    x.beta[t:t + 1], [0, 1], A_log=x.A_log, dt_bias=x.dt_bias,
                                    lower_bound=x.lower_bound, h0=S)
            np.testing.assert_allclose(res["out"][t], one["out"][0], rtol=1e-12, atol=1e-15)
            S = one["state"]
            if table[b, j] >= 0:
                np.testing.assert_allclose(res["pool"][table[b, j]], S[0], rtol=1e-12, atol=1e-15)
                written.add(int(table[b, j]))
    untouched = [r for r in range(24) if r not in written]
    assert np.array_equal(res["pool"][untouched], pool[untouched])
    # one slot per request in every column: the in-place decode
    same = np.repeat(x.state_indices.numpy()[:, None], 4, axis=1)
    a = oracle.window_steps(x, torch.from_numpy(same))
    w = oracle.window(x)
    np.testing.assert_allclose(a["out"], w["out"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(a["pool"], w["pool"], rtol=1e-12, atol=1e-15)
    # a start column outside the table, or a row past the pool, is flagged
    assert oracle.window_steps(x, torch.from_numpy(table), torch.from_numpy(acc * 0))["bad"]
    t2 = table.copy()
    t2[2, 3] = 24
    assert oracle.window_steps(x, torch.from_numpy(t2), torch.from_numpy(acc))["bad"]


def test_bf16_state_decode_is_repeated_single_token_decode():
    """The MATE decode page's bf16 state: a Q-token decode on a bf16 pool
    equals Q single-token decodes, each widening the stored bf16 row and
    storing its result back as bf16.  Every stored value is bf16."""
    x = W.decode_batch(5, 4, 1, 2, slots=9, seed=17, qlens=[4, 2, 3, 0, 4], null_requests=(1,),
                       lower_bound=-0.7, state_dtype=torch.bfloat16)
    res = oracle.window(x)
    pool = x.state_pool.clone()
    cu = x.cu_seqlens.tolist()
    idx = x.state_indices.tolist()
    for b in range(5):
        if idx[b] < 0:
            assert np.all(res["out"][cu[b]:cu[b + 1]] == 0)
            continue
        for t in range(cu[b], cu[b + 1]):
            one = oracle.recurrence(x.q[t:t + 1], x.k[t:t + 1], x.v[t:t + 1], x.g[t:t + 1],
                                    x.beta[t:t + 1], [0, 1], A_log=x.A_log, dt_bias=x.dt_bias,
                                    lower_bound=x.lower_bound,
                                    h0=pool[idx[b]].double().numpy()[None])
            np.testing.assert_allclose(res["out"][t], one["out"][0], rtol=1e-13, atol=1e-16)
            pool[idx[b]] = torch.from_numpy(one["state"][0]).float().bfloat16()
    np.testing.assert_array_equal(res["pool"], pool.double().numpy())
    assert np.array_equal(res["pool"], pool.double().numpy())


def test_bf16_state_closed_forms():
    """beta = 0, gate = 0: a bf16 state is unchanged bit for bit; one token
    from a zero bf16 state stores bf16(beta k^ v^T)."""
    x = W.decode_batch(2, 3, 1, 1, slots=3, seed=19, state_dtype=torch.bfloat16)
    x.beta[:] = -float("inf")
    x.A_log, x.dt_bias, x.lower_bound = None, None, 0.0
    x.g[:] = 0
    res = oracle.window(x)
    assert np.array_equal(res["pool"], x.state_pool.double().numpy())
    y = W.decode_batch(1, 1, 1, 1, slots=2, seed=20, state_dtype=torch.bfloat16)
    y.state_pool[:] = 0
    res = oracle.window(y)
    kk, vv = y.k[0, 0].double().numpy(), y.v[0, 0].double().numpy()
    kh = kk / np.sqrt(kk @ kk + 1e-6)
    beta = 1 / (1 + np.exp(-float(y.beta[0, 0])))
    want = torch.from_numpy(beta * np.outer(vv, kh)).float().bfloat16().double().numpy()
    np.testing.assert_array_equal(res["pool"][int(y.state_indices[0]), 0], want)


def test_corr_matches_windowed_solve():
    """The correction records U_t equal the windowed forward substitution of
    the verify page (probes p_t = e^{L_t} k^_t against the start state and
    coupling scalars c_ti = sum_c e^{L_t - L_i} k^_t k^_i), an algebraic
    unrolling of the recurrence over the window."""
    x = W.decode_batch(1, 6, 1, 1, slots=2, seed=12, lower_bound=-0.7)
    res = oracle.window(x)
    S0 = x.state_pool[int(x.state_indices[0]), 0].double().numpy().T  # K x V
    qh, kh, gate, b = chunked.activations(x.q[:, 0].float().numpy(), x.k[:, 0].float().numpy(),
                                          x.g[:, 0].float().numpy(), x.beta[:, 0].float().numpy(),
                                          x.A_log[0].item(), x.dt_bias[0].numpy(), x.scale,
                                          x.lower_bound)
    L = np.cumsum(gate, 0)
    v = x.v[:, 0].double().numpy()
    U = []
    for t in range(6):
        acc = v[t] - S0.T @ (np.exp(L[t]) * kh[t])
        for i in range(t):
            c_ti = np.sum(np.exp(L[t] - L[i]) * kh[t] * kh[i])
            acc = acc - c_ti * U[i]
        U.append(b[t] * acc)
        o = S0.T @ (np.exp(L[t]) * qh[t])
        for i in range(t + 1):
            o = o + np.sum(np.exp(L[t] - L[i]) * qh[t] * kh[i]) * U[i]
        np.testing.assert_allclose(res["out"][t, 0], o, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(res["corr"][:, 0], np.array(U), rtol=1e-11, atol=1e-14)


def test_no_gate_params_uses_g_directly():
    """Without A_log/dt_bias the gate input is the log decay itself."""
    q, k, v, g, b, A_log, dt = _rand_inputs(3, seed=13)
    g = -torch.rand(3, 1, D)
    b[:] = -np.inf
    h0 = np.ones((1, 1, D, D))
    res = oracle.recurrence(q, k, v, g, b, [0, 3], h0=h0)
    np.testing.assert_allclose(res["state"][0, 0], np.exp(g.double().sum(0)[0].numpy())[None, :]
                               * np.ones((D, 1)), rtol=1e-13)


@pytest.mark.parametrize("gated", [True, False])
def test_commit_from_records_equals_prefix_recurrence(gated):
    """Rebuilding the state after an accepted prefix from verify's records
    (corr = U_t, raw k_t, raw g_t) equals the recurrence run on the first a
    tokens alone, for every a = 0..qlen (GVA: v-head h reads the raw k of
    its q/k head)."""
    x = W.decode_batch(3, 5, 1, 2, slots=6, seed=13, qlens=[5, 3, 4], lower_bound=-0.8,
                       g_shift=0.0 if gated else -3.0)
    if not gated:
        x.A_log, x.dt_bias = None, None
    res = oracle.window(x)
    pool = x.state_pool.double().numpy()
    cu = x.cu_seqlens.tolist()
    idx = x.state_indices.tolist()
    f = lambda t: t.float().numpy().astype(np.float64)
    for b in range(3):
        qs, qe = cu[b], cu[b + 1]
        for a in range(qe - qs + 1):
            want = oracle.recurrence(x.q[qs:qs + a], x.k[qs:qs + a], x.v[qs:qs + a], x.g[qs:qs + a],
                                     x.beta[qs:qs + a], [0, a], A_log=x.A_log, dt_bias=x.dt_bias,
                                     lower_bound=x.lower_bound, h0=pool[idx[b]][None])["state"][0]
            for h in range(x.hv):
                kg_raw = np.concatenate([f(x.k[qs:qs + a, h // (x.hv // x.hqk)]), f(x.g[qs:qs + a, h])], axis=1)
                got = chunked.commit_from_records(
                    pool[idx[b], h], kg_raw, res["corr"][qs:qs + a, h],
                    None if x.A_log is None else float(x.A_log[h]),
                    None if x.dt_bias is None else f(x.dt_bias[h]), x.lower_bound)
                np.testing.assert_allclose(got, want[h], rtol=1e-11, atol=1e-14,
                                           err_msg=f"request {b} head {h} accepted {a}")
