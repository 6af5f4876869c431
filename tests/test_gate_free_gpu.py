"""GPU parity of the mode without gate parameters, through the C ABI.

With A_log = dt_bias = NULL the raw g is the per-channel log decay itself and
lower_bound is unused (mate.kda, ``chunk_kda`` docstring, gate parameters:
the lower bound applies only when the gate parameters are enabled).  The
kernels take their ``has_gate = false`` branches: prefill (dense and varlen,
serial walk and chunk-group scan), decode, verify and commit, each against
the fp64 oracle on the same draws.  The log decays are drawn U[lo, 0] with
lo >= -10, inside the exponent range the chunk kernels factor.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state

pytestmark = pytest.mark.gpu

STRONG = (-5.0, 0.0)   # a serving-like range of per-token decays
WEAK = (-0.1, 0.0)     # the state survives whole chunks: the walk matters


def _prefill(x, groups, dense):
    import linear_attention_serving_fwd_gb300 as kda
    xd = x.to("cuda")
    assert xd.A_log is None and xd.dt_bias is None
    kw = dict(scale=x.scale, lower_bound=x.lower_bound, groups=groups)
    if xd.state_pool is not None:
        pool = xd.state_pool.clone()
        out, _ = kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, cu_seqlens=xd.cu_seqlens,
                                   state_cache=pool, state_indices=xd.state_indices,
                                   has_initial_state=xd.has_initial_state, **kw)
        fin = None
    else:
        pool = None
        out, fin = kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta,
                                     **(dict(n_seqs=x.n_seqs) if dense else dict(cu_seqlens=xd.cu_seqlens)),
                                     initial_state=xd.initial_state, output_final_state=True, **kw)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    return out, fin, pool


@pytest.mark.parametrize("decay", [STRONG, WEAK], ids=["strong", "weak"])
@pytest.mark.parametrize("groups", [1, 4])
def test_dense_prefill_gate_free(decay, groups):
    x = W.dense_prefill(2, 64 * 17 + 23, 2, 4, seed=41 + groups, log_decay=decay, state_std=0.3)
    ref = oracle.prefill(x)
    out, fin, _ = _prefill(x, groups, dense=True)
    check_out(out, ref["out"], f"dense G={groups} out")
    check_state(fin, ref["state"], f"dense G={groups} final state")


@pytest.mark.parametrize("groups", [1, -1], ids=["two-launch", "pipelined"])
def test_dense_prefill_at_the_log_decay_limit(groups):
    """Log decays U[-10.5, -10], at the limit of the range the chunk kernels
    factor: 8 consecutive rows span e^{+-84}, so the operands' scale factors
    (running products of the rows' decays from one anchor each) reach their
    largest anchors, and every decay product beyond a few rows underflows."""
    x = W.dense_prefill(2, 64 * 9 + 5, 2, 4, seed=47 + groups, log_decay=(-10.5, -10.0), state_std=0.3)
    assert float(x.g.min()) >= -10.5
    ref = oracle.prefill(x)
    out, fin, _ = _prefill(x, groups, dense=True)
    check_out(out, ref["out"], f"dense G={groups} out at the log decay limit")
    check_state(fin, ref["state"], f"dense G={groups} final state at the log decay limit")


@pytest.mark.parametrize("decay", [STRONG, WEAK], ids=["strong", "weak"])
@pytest.mark.parametrize("groups", [1, 4])
def test_varlen_paged_prefill_gate_free(decay, groups):
    x = W.varlen_paged([700, 64, 1300, 33, 1], 2, 4, slots=11, seed=43 + groups, log_decay=decay,
                       has_initial=[1, 1, 0, 1, 1], state_std=0.3)
    ref = oracle.prefill(x)
    out, _, pool = _prefill(x, groups, dense=False)
    check_out(out, ref["out"], f"varlen G={groups} out")
    live = [s for s in x.state_indices.tolist() if s >= 0]
    check_state(pool[live], ref["pool"][live], f"varlen G={groups} cache rows")
    untouched = [s for s in range(pool.shape[0]) if s not in live]
    assert torch.equal(pool[untouched].cpu(), x.state_pool[untouched]), "untouched rows changed"


@pytest.mark.parametrize("window,qlens,nulls", [(1, [1] * 9, (4,)), (4, [4, 1, 0, 3, 4, 2, 4], (5,))])
def test_decode_and_verify_gate_free(window, qlens, nulls):
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(len(qlens), window, 2, 4, slots=21, seed=47 + window, qlens=qlens,
                       null_requests=nulls, log_decay=WEAK, state_std=0.3)
    ref = oracle.window(x)
    xd = x.to("cuda")
    args = (xd.q, xd.k, xd.v, xd.g, xd.beta)
    pool = xd.state_pool.clone()
    od = kda.kda_decode(*args, pool, xd.cu_seqlens, xd.state_indices, window, scale=x.scale)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    ov, corr, _ = kda.kda_verify(*args, xd.state_pool, xd.cu_seqlens, xd.state_indices, window,
                                 scale=x.scale, work_counter=counter)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    check_out(od, ref["out"], "decode out")
    check_out(ov, ref["out"], "verify out")
    live = [s for s in x.state_indices.tolist() if s >= 0]
    check_state(pool[live], ref["pool"][live], "decode state")
    assert torch.equal(xd.state_pool.cpu(), x.state_pool), "verify modified the pool"
    assert int(counter.item()) == 0


def test_commit_gate_free():
    """verify then commit of per-request accepted prefixes, no gate
    parameters, against the fp64 recurrence over each accepted prefix."""
    import linear_attention_serving_fwd_gb300 as kda
    qlens, accepted = [4, 1, 3, 4, 2, 4], [3, 1, 0, 4, 2, 1]
    x = W.decode_batch(len(qlens), 4, 2, 4, slots=17, seed=53, qlens=qlens, log_decay=STRONG,
                       state_std=0.3)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    _, corr, kg = kda.kda_verify(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens,
                                 xd.state_indices, 4, scale=x.scale)
    acc = torch.tensor(accepted, dtype=torch.int32, device="cuda")
    kda.kda_commit(pool, xd.state_indices, acc, corr, kg, 4)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    cu, idx = x.cu_seqlens.tolist(), x.state_indices.tolist()
    pool0 = x.state_pool.double().numpy()
    got = pool.cpu()
    for b, a in enumerate(accepted):
        if a == 0:
            assert torch.equal(got[idx[b]], x.state_pool[idx[b]])
            continue
        qs = cu[b]
        S = oracle.recurrence(x.q[qs:qs + a], x.k[qs:qs + a], x.v[qs:qs + a], x.g[qs:qs + a],
                              x.beta[qs:qs + a], [0, a], h0=pool0[idx[b]][None])["state"]
        check_state(got[idx[b]:idx[b] + 1], S, f"request {b} accepted {a}")


def test_log_decay_out_of_range_is_reported():
    """A raw log decay below -10.5 leaves the exponent range the chunk
    kernels factor: the prefill reports KDA_ERR_DEVICE_RANGE (and a clean
    call afterwards reports nothing)."""
    import linear_attention_serving_fwd_gb300 as kda
    from linear_attention_serving_fwd_gb300 import _native
    x = W.dense_prefill(1, 130, 1, 2, seed=59, log_decay=STRONG).to("cuda")
    g = x.g.clone()
    g[70, 1, 5] = -11.0
    kda.kda_chunk_fwd(x.q, x.k, x.v, g, x.beta, n_seqs=1, output_final_state=True)
    assert kda.kda_device_status(clear=True) == _native.KDA_ERR_DEVICE_RANGE
    kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, n_seqs=1, output_final_state=True)
    assert kda.kda_device_status(clear=True) == 0
