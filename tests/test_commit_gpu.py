"""GPU parity of kda_commit (speculative-decode commit) through the C ABI:
kda_verify on a decode batch, then kda_commit with per-request accepted
counts, against the fp64 recurrence run on each request's accepted prefix
alone.  Rows not committed (padding, a = 0, other slots) stay bit-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_state

pytestmark = pytest.mark.gpu


def _prefix_states(x, accepted):
    """Per request b: the fp64 state after its first accepted[b] tokens."""
    pool = x.state_pool.double().numpy()
    cu = x.cu_seqlens.tolist()
    idx = x.state_indices.tolist()
    out = {}
    for b in range(len(idx)):
        if idx[b] < 0:
            continue
        qs, a = cu[b], accepted[b]
        out[b] = oracle.recurrence(x.q[qs:qs + a], x.k[qs:qs + a], x.v[qs:qs + a], x.g[qs:qs + a],
                                   x.beta[qs:qs + a], [0, a], A_log=x.A_log, dt_bias=x.dt_bias,
                                   lower_bound=x.lower_bound, h0=pool[idx[b]][None])["state"][0]
    return out


@pytest.mark.parametrize("window,qlens,accepted,nulls,hqk,hv", [
    (4, [4, 1, 0, 3, 4, 2, 4, 4], [3, 1, 0, 0, 4, 2, 1, 4], (6,), 2, 4),
    (8, [8, 5, 1, 8], [8, 2, 1, 5], (), 1, 2),
    (1, [1, 1, 1], [1, 0, 1], (1,), 2, 2),
])
def test_commit_matches_prefix_recurrence(window, qlens, accepted, nulls, hqk, hv):
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(len(qlens), window, hqk, hv, slots=29, seed=31 + window, qlens=qlens,
                       null_requests=nulls, lower_bound=-0.6)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    kw = dict(A_log=xd.A_log, dt_bias=xd.dt_bias, scale=x.scale, lower_bound=x.lower_bound)
    _, corr, kg = kda.kda_verify(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens, xd.state_indices,
                                 window, **kw)
    acc = torch.tensor(accepted, dtype=torch.int32, device="cuda")
    kda.kda_commit(pool, xd.state_indices, acc, corr, kg, window, A_log=xd.A_log, dt_bias=xd.dt_bias,
                   lower_bound=x.lower_bound)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    want = _prefix_states(x, accepted)
    got = pool.cpu()
    idx = x.state_indices.tolist()
    for b, S in want.items():
        if accepted[b] == 0:
            assert torch.equal(got[idx[b]], x.state_pool[idx[b]]), f"request {b}: a = 0 changed its row"
        else:
            check_state(got[idx[b]:idx[b] + 1], S[None], f"request {b} accepted {accepted[b]}")
    touched = [idx[b] for b in want if accepted[b] > 0]
    untouched = [s for s in range(x.state_pool.shape[0]) if s not in touched]
    assert torch.equal(got[untouched], x.state_pool[untouched]), "rows outside the commit changed"


def test_commit_decode_workload_sampled():
    """The 256-request x H=32 window-4 workload: every request accepts a
    random prefix; sampled requests against the prefix recurrence."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.workload("decode", window=4, seed=5)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    kw = dict(A_log=xd.A_log, dt_bias=xd.dt_bias, scale=x.scale, lower_bound=x.lower_bound)
    _, corr, kg = kda.kda_verify(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens, xd.state_indices,
                                 4, **kw)
    gen = torch.Generator().manual_seed(7)
    accepted = torch.randint(0, 5, (x.n_seqs,), generator=gen, dtype=torch.int32)
    kda.kda_commit(pool, xd.state_indices, accepted.cuda(), corr, kg, 4, A_log=xd.A_log,
                   dt_bias=xd.dt_bias, lower_bound=x.lower_bound)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    acc = accepted.tolist()
    sample = [0, 1, 77, 128, 200, 255]
    idx = x.state_indices.tolist()
    cu = x.cu_seqlens.tolist()
    pool0 = x.state_pool.double().numpy()
    got = pool.cpu()
    for b in sample:
        qs, a = cu[b], acc[b]
        S = oracle.recurrence(x.q[qs:qs + a], x.k[qs:qs + a], x.v[qs:qs + a], x.g[qs:qs + a],
                              x.beta[qs:qs + a], [0, a], A_log=x.A_log, dt_bias=x.dt_bias,
                              lower_bound=x.lower_bound, h0=pool0[idx[b]][None])["state"]
        check_state(got[idx[b]:idx[b] + 1], S, f"request {b} accepted {a}")


def test_commit_flags_bad_accepted_count():
    """An accepted count above the window is reported (KDA_ERR_DEVICE_INDEX)
    and that request's row is left as it was."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(2, 2, 1, 1, slots=4, seed=3)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    _, corr, kg = kda.kda_verify(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens, xd.state_indices, 2,
                                 A_log=xd.A_log, dt_bias=xd.dt_bias, lower_bound=x.lower_bound)
    acc = torch.tensor([3, 1], dtype=torch.int32, device="cuda")
    kda.kda_commit(pool, xd.state_indices, acc, corr, kg, 2, A_log=xd.A_log, dt_bias=xd.dt_bias,
                   lower_bound=x.lower_bound)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 5  # KDA_ERR_DEVICE_INDEX
    s0 = int(x.state_indices[0])
    assert torch.equal(pool[s0].cpu(), x.state_pool[s0])
