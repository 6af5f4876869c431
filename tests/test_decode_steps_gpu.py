"""GPU parity of kda_decode_steps (decode with a [request, step] slot table
and accepted-token counts, the MATE gated_delta_rule_decode [B, T]
state_indices / num_accepted_tokens form) against the fp64 oracle, through
the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state

pytestmark = pytest.mark.gpu


def _run(x, table, acc):
    import linear_attention_serving_fwd_gb300 as kda
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    out = kda.kda_decode_steps(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens,
                               table.to("cuda"), x.window,
                               num_accepted_tokens=None if acc is None else acc.to("cuda"),
                               A_log=xd.A_log, dt_bias=xd.dt_bias, scale=x.scale,
                               lower_bound=x.lower_bound)
    torch.cuda.synchronize()
    return out, pool


def _compare(x, table, acc, out, pool, ref, what):
    check_out(out, ref["out"], f"{what} out")
    changed = sorted({int(r) for r in np.flatnonzero(
        np.any(ref["pool"] != x.state_pool.double().numpy(), axis=(1, 2, 3)))})
    if changed:
        check_state(pool[changed], ref["pool"][changed], f"{what} stored states")
    untouched = [r for r in range(x.state_pool.shape[0]) if r not in changed]
    assert torch.equal(pool[untouched].cpu(), x.state_pool[untouched]), f"{what}: untouched rows changed"


def test_slot_table_small():
    """Ragged windows (an empty request among them), accepted counts 1..4,
    disabled store columns, a padding request (negative start row)."""
    qlens = [4, 3, 1, 4, 2, 0, 4, 3]
    x = W.decode_batch(len(qlens), 4, 2, 4, slots=40, seed=21, qlens=qlens, lower_bound=-0.6)
    table, acc = W.decode_slot_table(len(qlens), 4, 40, seed=21)
    table[1, 0] = -1
    table[4, 1] = -1
    acc[6] = 2
    table[6, 1] = -1   # request 6 starts from a negative row: padding
    ref = oracle.window_steps(x, table, acc)
    assert not ref["bad"]
    out, pool = _run(x, table, acc)
    _compare(x, table, acc, out, pool, ref, "slot table")
    cu = x.cu_seqlens.tolist()
    assert torch.count_nonzero(out[cu[6]:cu[7]]) == 0
    import linear_attention_serving_fwd_gb300 as kda
    assert kda.kda_device_status(clear=True) == 0


def test_slot_table_without_counts_and_repeated_rows():
    """No counts: start from column 0.  A row repeated across columns ends
    with the later token's state; all columns on one slot give kda_decode's
    result (within tolerance: the slot table runs token by token, the
    in-place decode of a 2..4-token window runs the windowed solve)."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(6, 4, 2, 2, slots=30, seed=22, qlens=[4, 4, 2, 3, 1, 4], lower_bound=-0.6)
    table, _ = W.decode_slot_table(6, 4, 30, seed=22)
    table[0, 2] = table[0, 0]
    table[3, 1] = table[3, 2]
    ref = oracle.window_steps(x, table, None)
    out, pool = _run(x, table, None)
    _compare(x, table, None, out, pool, ref, "no counts")
    same = x.state_indices[:, None].repeat(1, 4).contiguous()
    out_s, pool_s = _run(x, same, None)
    xd = x.to("cuda")
    pool_d = xd.state_pool.clone()
    out_d = kda.kda_decode(xd.q, xd.k, xd.v, xd.g, xd.beta, pool_d, xd.cu_seqlens, xd.state_indices,
                           x.window, A_log=xd.A_log, dt_bias=xd.dt_bias, lower_bound=x.lower_bound)
    torch.cuda.synchronize()
    ref_d = oracle.window(x)
    check_out(out_s, ref_d["out"], "slot table, one slot per request")
    check_out(out_d, ref_d["out"], "kda_decode")
    live = x.state_indices.tolist()
    check_state(pool_s[live], ref_d["pool"][live], "slot table rows")
    check_state(pool_d[live], ref_d["pool"][live], "kda_decode rows")
    assert torch.equal(pool_s[[r for r in range(30) if r not in live]],
                       pool_d[[r for r in range(30) if r not in live]])
    assert kda.kda_device_status(clear=True) == 0


def test_slot_table_bad_rows_are_reported():
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(3, 4, 1, 1, slots=16, seed=23, qlens=[4, 4, 4])
    table, acc = W.decode_slot_table(3, 4, 16, seed=23)
    table[1, 2] = 16           # past the pool
    acc[2] = 5                 # start column past the table
    out, pool = _run(x, table, acc)
    assert kda.kda_device_status(clear=True) == 5
    cu = x.cu_seqlens.tolist()
    assert torch.count_nonzero(out[cu[1]:cu[3]]) == 0
    ref = oracle.window_steps(x, table, acc)
    assert ref["bad"]
    _compare(x, table, acc, out, pool, ref, "bad rows")


def test_slot_table_serving_batch_sampled():
    """256 requests x 4 tokens, H=32, a 1280-row pool with four rows per
    request (the timed workload): every output and stored state of 12
    sampled requests against the oracle, and rows no request owns unchanged."""
    x = W.decode_batch(256, 4, 32, 32, slots=1280, seed=24, device="cuda", name="decode_steps_q4")
    table, acc = W.decode_slot_table(256, 4, 1280, seed=24, device="cuda")
    out, pool = _run(x, table, acc)
    gen = torch.Generator().manual_seed(5)
    reqs = sorted(torch.randperm(256, generator=gen)[:12].tolist())
    cu = x.cu_seqlens.tolist()
    tok = torch.cat([torch.arange(cu[b], cu[b + 1]) for b in reqs]).to("cuda")
    rows = table[reqs].cpu()
    uniq = sorted({int(r) for r in rows.flatten().tolist()})
    remap = {r: i for i, r in enumerate(uniq)}
    c = lambda t: t.cpu()
    sub = W.KdaInputs(name="sample", q=c(x.q[tok]), k=c(x.k[tok]), v=c(x.v[tok]), g=c(x.g[tok]),
                      beta=c(x.beta[tok]), A_log=c(x.A_log), dt_bias=c(x.dt_bias),
                      cu_seqlens=torch.tensor([0] + [4 * (i + 1) for i in range(len(reqs))],
                                              dtype=torch.int32),
                      B=0, T=0, lower_bound=x.lower_bound, state_pool=c(x.state_pool[uniq]),
                      state_indices=None, window=4)
    sub_table = rows.clone().apply_(lambda r: remap[r])
    ref = oracle.window_steps(sub, sub_table, acc[reqs].cpu())
    got_out = torch.cat([out[cu[b]:cu[b + 1]] for b in reqs])
    check_out(got_out, ref["out"], "sampled out")
    check_state(pool[uniq], ref["pool"], "sampled stored states")
    owned = set(table.flatten().tolist())
    free = torch.tensor([r for r in range(1280) if r not in owned], device="cuda")
    assert torch.equal(pool[free], x.state_pool[free])
    import linear_attention_serving_fwd_gb300 as kda
    assert kda.kda_device_status(clear=True) == 0
