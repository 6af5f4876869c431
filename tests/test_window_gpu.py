"""GPU parity of kda_decode / kda_verify against the fp64 oracle, through the
C ABI (the package's ctypes binding)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state, np64

pytestmark = pytest.mark.gpu


def _run_decode(x, verify=False):
    import linear_attention_serving_fwd_gb300 as kda
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    args = (xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens, xd.state_indices, x.window)
    kw = dict(A_log=xd.A_log, dt_bias=xd.dt_bias, scale=x.scale, lower_bound=x.lower_bound)
    if verify:
        counter = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, corr, kg = kda.kda_verify(*args, work_counter=counter, **kw)
        torch.cuda.synchronize()
        return dict(out=out, pool=pool, corr=corr, kg=kg, counter=counter, x=xd)
    out = kda.kda_decode(*args, **kw)
    torch.cuda.synchronize()
    return dict(out=out, pool=pool, x=xd)


def _status_clean():
    import linear_attention_serving_fwd_gb300 as kda
    assert kda.kda_device_status(clear=True) == 0


def _check_decode(x, res, ref):
    check_out(res["out"], ref["out"], "decode out")
    idx = x.state_indices.tolist()
    live = [s for s in idx if s >= 0]
    check_state(res["pool"][live], ref["pool"][live], "decode state")
    untouched = [s for s in range(x.state_pool.shape[0]) if s not in live]
    assert torch.equal(res["pool"][untouched].cpu(), x.state_pool[untouched]), "untouched slots changed"


@pytest.mark.parametrize("window,qlens,nulls", [
    (1, None, ()),
    (4, [4, 1, 0, 3, 4, 2, 4, 4, 1, 4, 3], (2, 5)),
    (8, [8, 5, 1], (1,)),
])
def test_decode_small(window, qlens, nulls):
    n = len(qlens) if qlens else 7
    x = W.decode_batch(n, window, 2, 4, slots=23, seed=window, qlens=qlens, null_requests=nulls)
    ref = oracle.window(x)
    res = _run_decode(x)
    _check_decode(x, res, ref)
    cu = x.cu_seqlens.tolist()
    for b in nulls:
        assert torch.count_nonzero(res["out"][cu[b]:cu[b + 1]]) == 0
    _status_clean()


@pytest.mark.parametrize("window", [1, 4])
def test_decode_full_batch(window):
    """256 requests x window, H=32, 512-slot pool: the serving batch."""
    x = W.workload("decode", window=window)
    ref = oracle.window(x)
    res = _run_decode(x)
    _check_decode(x, res, ref)
    _status_clean()


@pytest.mark.parametrize("window", [1, 4])
def test_verify_matches_oracle_and_leaves_state(window):
    x = W.workload("decode", window=window)
    ref = oracle.window(x)
    res = _run_decode(x, verify=True)
    check_out(res["out"], ref["out"], "verify out")
    assert torch.equal(res["pool"].cpu(), x.state_pool), "verify modified the state pool"
    assert int(res["counter"].item()) == 0, "work counter not left at zero"
    # corr [n_req, Hv, window, 128] = U_t of each request's tokens
    cu = x.cu_seqlens.tolist()
    corr = np64(res["corr"])
    kg = res["kg"].cpu()
    for b in range(x.n_seqs):
        for t in range(cu[b + 1] - cu[b]):
            ref_u = ref["corr"][cu[b] + t]
            got = corr[b, :, t]
            err = np.linalg.norm(got - ref_u) / np.linalg.norm(ref_u)
            assert err < 1e-3, (b, t, err)
            r = x.hv // x.hqk
            raw_k = x.k[cu[b] + t].repeat_interleave(r, dim=0)
            assert torch.equal(kg[b, :, t, :128], raw_k)
            assert torch.equal(kg[b, :, t, 128:], x.g[cu[b] + t])
    _status_clean()


def test_verify_equals_decode_outputs_and_padding():
    """Verify and decode give the same outputs (verify runs the windowed solve
    for 2..4 tokens, decode the token loop: both within the output tolerance
    of the oracle, zeros on the padding), and verify leaves the pool as it
    was."""
    x = W.decode_batch(9, 4, 1, 2, slots=12, seed=5, qlens=[4, 3, 4, 0, 1, 4, 2, 4, 4],
                       null_requests=(4, 7), lower_bound=-0.3)
    ref = oracle.window(x)
    dec = _run_decode(x)
    ver = _run_decode(x, verify=True)
    check_out(ver["out"], ref["out"], "verify out")
    check_out(dec["out"], ref["out"], "decode out")
    cu = x.cu_seqlens.tolist()
    for b in (4, 7):  # padding: zeros from both
        assert torch.count_nonzero(ver["out"][cu[b]:cu[b + 1]]) == 0
        assert torch.count_nonzero(dec["out"][cu[b]:cu[b + 1]]) == 0
    assert torch.equal(ver["pool"].cpu(), x.state_pool)
    _status_clean()


def test_bad_slot_sets_device_index_error():
    """A slot beyond the pool is reported through the device error word and
    treated as padding; the other requests are unaffected."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(4, 1, 1, 1, slots=6, seed=6)
    x.state_indices[2] = 6  # one past the end
    ref_x = W.decode_batch(4, 1, 1, 1, slots=6, seed=6)
    ref_x.state_indices[2] = -1
    ref = oracle.window(ref_x)
    res = _run_decode(x)
    check_out(res["out"], ref["out"], "out with bad slot")
    assert kda.kda_device_status(clear=True) == 5
    _status_clean()


def test_repeated_single_token_decodes_equal_window():
    """Q single-token decodes on the carried pool equal one Q-token decode."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(5, 4, 2, 2, slots=8, seed=7, lower_bound=-0.5)
    full = _run_decode(x)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    outs = []
    for t in range(4):
        sel = torch.arange(5, device="cuda") * 4 + t
        qs = torch.arange(6, dtype=torch.int32, device="cuda")
        o = kda.kda_decode(xd.q[sel], xd.k[sel], xd.v[sel], xd.g[sel], xd.beta[sel], pool, qs,
                           xd.state_indices, 1, A_log=xd.A_log, dt_bias=xd.dt_bias,
                           lower_bound=x.lower_bound)
        outs.append(o)
    torch.cuda.synchronize()
    step = torch.stack(outs, 1).reshape(20, 2, 128)
    np.testing.assert_allclose(np64(step), np64(full["out"]), rtol=2e-2, atol=1e-3)
    live = x.state_indices.tolist()
    d = (pool[live] - full["pool"][live]).norm() / full["pool"][live].norm()
    assert float(d) < 1e-5
