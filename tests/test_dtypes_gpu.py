"""GPU parity of the dtype variants through the C ABI: fp16 activations
(q, k, v, g, beta and the output o in fp16, MATE's supported q/k/v types)
and bf16 recurrent states (read widened; prefill rounds the final state
once, decode and verify round the carried state after every token, the
MATE decode page's bf16 state), against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state, check_state_bf16, np64

pytestmark = pytest.mark.gpu

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32


def _check_states(got, ref, what):
    if got.dtype == BF16:
        return check_state_bf16(got, ref, what)
    return check_state(got, ref, what)


def _prefill(x, groups=1, dense=False, ckpt=None):
    import linear_attention_serving_fwd_gb300 as kda
    xd = x.to("cuda")
    kw = dict(A_log=xd.A_log, dt_bias=xd.dt_bias, scale=x.scale, lower_bound=x.lower_bound, groups=groups)
    pool = None
    if xd.state_pool is not None:
        pool = xd.state_pool.clone()
        out, fin = kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, cu_seqlens=xd.cu_seqlens,
                                     state_cache=pool, state_indices=xd.state_indices,
                                     has_initial_state=xd.has_initial_state, **(ckpt or {}), **kw)
    else:
        out, fin = kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, n_seqs=x.n_seqs,
                                     initial_state=xd.initial_state, output_final_state=True, **kw)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    assert out.dtype == x.q.dtype
    return out, fin, pool


@pytest.mark.parametrize("act,state,groups", [(F16, F32, 1), (F16, BF16, 3), (BF16, BF16, 1)])
def test_prefill_dense_dtypes(act, state, groups):
    x = W.dense_prefill(2, 64 * 9 + 17, 2, 4, seed=41, lower_bound=-0.3, act_dtype=act, state_dtype=state)
    ref = oracle.prefill(x)
    out, fin, _ = _prefill(x, groups=groups)
    assert fin.dtype == state
    check_out(out, ref["out"], f"{act} out")
    _check_states(fin, ref["state"], f"{state} final state")


@pytest.mark.parametrize("act,state,groups", [(F16, F32, 1), (BF16, BF16, 4), (F16, BF16, 1)])
def test_prefill_paged_dtypes(act, state, groups):
    """Varlen paged (GVA), a sequence without initial state, one without a
    row, and a mid-prefill snapshot in the state dtype."""
    x = W.varlen_paged([70, 1, 129, 64, 5, 700], 2, 4, slots=11, seed=42, lower_bound=-0.2,
                       has_initial=[1, 0, 1, 1, 1, 1], act_dtype=act, state_dtype=state)
    x.state_indices[4] = -1
    ref = oracle.prefill(x)
    ck = torch.zeros((6, 4, 128, 128), dtype=state, device="cuda") + 7
    offs = torch.tensor([64, 0, 128, 64, 0, 640], dtype=torch.int32, device="cuda")
    out, _, pool = _prefill(x, groups=groups, ckpt=dict(checkpoint_state=ck, checkpoint_offsets=offs))
    check_out(out, ref["out"], f"{act} varlen out")
    live = [s for s in x.state_indices.tolist() if s >= 0]
    _check_states(pool[live], ref["pool"][live], f"{state} cache rows")
    untouched = [s for s in range(pool.shape[0]) if s not in live]
    assert torch.equal(pool[untouched].cpu(), x.state_pool[untouched])
    # the snapshots: the state after offs[n] tokens (rounded once if bf16)
    cu = x.cu_seqlens.tolist()
    pool0 = x.state_pool.double().numpy()
    for n, o in enumerate(offs.tolist()):
        if o == 0:
            assert torch.all(ck[n] == 7)
            continue
        idx = x.state_indices.tolist()[n]
        h0 = pool0[idx][None] if idx >= 0 and x.has_initial_state[n] else None
        s = oracle.recurrence(x.q[cu[n]:cu[n] + o], x.k[cu[n]:cu[n] + o], x.v[cu[n]:cu[n] + o],
                              x.g[cu[n]:cu[n] + o], x.beta[cu[n]:cu[n] + o], [0, o], A_log=x.A_log,
                              dt_bias=x.dt_bias, lower_bound=x.lower_bound, h0=h0)["state"]
        if state == BF16:
            s = oracle.round_bf16(s)
        _check_states(ck[n:n + 1], s, f"snapshot {n}")


def _decode(x, verify=False, table=None, acc=None):
    import linear_attention_serving_fwd_gb300 as kda
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    kw = dict(A_log=xd.A_log, dt_bias=xd.dt_bias, scale=x.scale, lower_bound=x.lower_bound)
    corr = kg = None
    if verify:
        out, corr, kg = kda.kda_verify(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens,
                                       xd.state_indices, x.window, **kw)
    elif table is not None:
        out = kda.kda_decode_steps(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens, table.cuda(),
                                   x.window, num_accepted_tokens=None if acc is None else acc.cuda(), **kw)
    else:
        out = kda.kda_decode(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens, xd.state_indices,
                             x.window, **kw)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    assert out.dtype == x.q.dtype
    return out, pool, corr, kg


@pytest.mark.parametrize("act,state,window", [(F16, F32, 1), (F16, F32, 4), (BF16, BF16, 1), (BF16, BF16, 4),
                                              (F16, BF16, 1), (F16, BF16, 8)])
def test_decode_dtypes(act, state, window):
    qlens = [window, 1, 0, max(1, window - 1), window, 2 if window > 1 else 1]
    x = W.decode_batch(6, window, 2, 4, slots=17, seed=43 + window, qlens=qlens, null_requests=(4,),
                       lower_bound=-0.6, act_dtype=act, state_dtype=state)
    ref = oracle.window(x)
    out, pool, _, _ = _decode(x)
    check_out(out, ref["out"], f"{act} decode out")
    live = [s for s in x.state_indices.tolist() if s >= 0]
    _check_states(pool[live], ref["pool"][live], f"{state} decode rows")
    untouched = [s for s in range(pool.shape[0]) if s not in live]
    assert torch.equal(pool[untouched].cpu(), x.state_pool[untouched])


@pytest.mark.parametrize("window", [1, 4])
def test_decode_bf16_state_serving_batch(window):
    """256 requests x window, H=32, 512-slot bf16 pool."""
    x = W.decode_batch(256, window, 32, 32, slots=512, seed=44, state_dtype=BF16)
    ref = oracle.window(x)
    out, pool, _, _ = _decode(x)
    check_out(out, ref["out"], "bf16-state decode out")
    live = x.state_indices.tolist()
    _check_states(pool[live], ref["pool"][live], "bf16-state decode rows")


@pytest.mark.parametrize("act,state", [(F16, BF16), (BF16, BF16), (F16, F32)])
def test_verify_and_commit_dtypes(act, state):
    """Verify reads the pool only; its corr records follow the per-token
    rounded states; commit rebuilds the accepted prefix in the pool's dtype
    from fp16 or bf16 kg records."""
    import linear_attention_serving_fwd_gb300 as kda
    qlens = [4, 3, 4, 1, 4]
    x = W.decode_batch(5, 4, 1, 2, slots=9, seed=45, qlens=qlens, null_requests=(3,), lower_bound=-0.6,
                       act_dtype=act, state_dtype=state)
    ref = oracle.window(x)
    out, pool, corr, kg = _decode(x, verify=True)
    check_out(out, ref["out"], "verify out")
    assert torch.equal(pool.cpu(), x.state_pool), "verify changed the pool"
    assert kg.dtype == act
    cu = x.cu_seqlens.tolist()
    idx = x.state_indices.tolist()
    c = np64(corr)
    for b in range(5):
        if idx[b] < 0:
            continue
        for t in range(qlens[b]):
            r_u = ref["corr"][cu[b] + t]
            assert np.linalg.norm(c[b, :, t] - r_u) / np.linalg.norm(r_u) < 2e-3, (b, t)
            assert torch.equal(kg[b, :, t, 128:].cpu(), x.g[cu[b] + t])
    accepted = [2, 3, 4, 0, 1]
    acc = torch.tensor(accepted, dtype=torch.int32, device="cuda")
    xd = x.to("cuda")
    kda.kda_commit(pool, xd.state_indices, acc, corr, kg, 4, A_log=xd.A_log, dt_bias=xd.dt_bias,
                   lower_bound=x.lower_bound)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    pool0 = x.state_pool.double().numpy()
    for b in range(5):
        if idx[b] < 0:
            continue
        a = accepted[b]
        # the state after the accepted prefix, token by token (per-token
        # rounding with a bf16 pool, as decode would have left it)
        S = pool0[idx[b]][None]
        for t in range(cu[b], cu[b] + a):
            S = oracle.recurrence(x.q[t:t + 1], x.k[t:t + 1], x.v[t:t + 1], x.g[t:t + 1], x.beta[t:t + 1],
                                  [0, 1], A_log=x.A_log, dt_bias=x.dt_bias, lower_bound=x.lower_bound,
                                  h0=S)["state"]
            if state == BF16:
                S = oracle.round_bf16(S)
        _check_states(pool[idx[b]:idx[b] + 1], S, f"commit request {b} accepted {a}")


def test_decode_steps_bf16_state():
    x = W.decode_batch(5, 4, 1, 2, slots=24, seed=46, qlens=[4, 3, 1, 4, 2], lower_bound=-0.6,
                       act_dtype=F16, state_dtype=BF16)
    table, acc = W.decode_slot_table(5, 4, 24, seed=46)
    ref = oracle.window_steps(x, table, acc)
    out, pool, _, _ = _decode(x, table=table, acc=acc)
    check_out(out, ref["out"], "slot-table out")
    changed = sorted({int(r) for r in np.flatnonzero(
        np.any(ref["pool"] != x.state_pool.double().numpy(), axis=(1, 2, 3)))})
    _check_states(pool[changed], ref["pool"][changed], "slot-table bf16 rows")
    untouched = [r for r in range(24) if r not in changed]
    assert torch.equal(pool[untouched].cpu(), x.state_pool[untouched])


def test_dense_prefill_full_fp16_bf16_state():
    """The B=2, T=4096, H=16 prefill with fp16 activations and bf16 initial
    and final states."""
    x = W.dense_prefill(2, 4096, 16, 16, seed=47, act_dtype=F16, state_dtype=BF16)
    ref = oracle.prefill(x)
    out, fin, _ = _prefill(x, dense=True)
    check_out(out, ref["out"], "fp16 dense out")
    check_state_bf16(fin, ref["state"], "bf16 dense final state")
