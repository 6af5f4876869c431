"""GPU parity of the 128-column walk through the C ABI: the pipelined prefill
launch (groups = -1) and the same walk as a launch of its own.

The pipelined launch is one cooperative kernel: one CTA per (sequence, head)
chain walks all 128 value columns while the other SMs run the prologue in
level-major order, and a walk CTA takes each chunk's record once the prologue
has flagged it ready.  With more chains than the 32-column walk fits on the
SMs in one wave, the 128-column walk runs as a launch of its own after the
prologue.  Every case checks, through the library's kernel trace, which
kernels ran, and compares outputs and states with the fp64 oracle at the
spec's tolerances.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import conv as oconv
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state, check_state_bf16

pytestmark = pytest.mark.gpu


def _traced(fn):
    """Run fn with the kernel trace on; return (fn's result, kernel names)."""
    from linear_attention_serving_fwd_gb300 import _native
    _native.trace_enable(True)
    try:
        r = fn()
        torch.cuda.synchronize()
        names = set(_native.trace_read())
    finally:
        _native.trace_enable(False)
    return r, names


def _dense(x, groups=-1, **extra):
    import linear_attention_serving_fwd_gb300 as kda
    xd = x.to("cuda")

    def call():
        return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 scale=x.scale, lower_bound=x.lower_bound, n_seqs=x.n_seqs,
                                 initial_state=xd.initial_state, output_final_state=True, groups=groups,
                                 **extra)
    (out, fin), names = _traced(call)
    assert kda.kda_device_status(clear=True) == 0
    return out, fin, names


def _assert_pipelined(names):
    assert "kda_pipelined" in names, f"pipelined kernel did not run: {sorted(names)}"
    assert "kda_walk" not in names and "kda_prologue" not in names, sorted(names)


@pytest.mark.parametrize("B,T,hqk,hv,init", [(1, 256, 1, 1, False), (2, 64 * 17 + 23, 2, 4, True),
                                             (3, 64, 1, 2, True), (1, 1, 1, 1, True), (2, 130, 2, 2, False),
                                             (1, 700, 4, 4, True)],
                         ids=["tiny", "ragged-gva", "one-chunk", "one-token", "two-chunks", "gva1"])
def test_pipelined_matches_oracle(B, T, hqk, hv, init):
    x = W.dense_prefill(B, T, hqk, hv, seed=71 + T, init_state=init, state_std=0.3)
    ref = oracle.prefill(x)
    out, fin, names = _dense(x)
    _assert_pipelined(names)
    check_out(out, ref["out"], "pipelined out")
    check_state(fin, ref["state"], "pipelined final state")


@pytest.mark.parametrize("lb,shift", [(-0.05, 0.0), (-5.0, -6.0)], ids=["lb-0.05", "g-6"])
def test_pipelined_weak_decay(lb, shift):
    """The state survives every chunk: the walk chain and h0 reach every output."""
    x = W.dense_prefill(2, 64 * 30 + 5, 2, 4, seed=73, lower_bound=lb, g_shift=shift, state_std=0.3)
    ref = oracle.prefill(x)
    out, fin, names = _dense(x)
    _assert_pipelined(names)
    check_out(out, ref["out"], "pipelined weak out")
    check_state(fin, ref["state"], "pipelined weak final state")


@pytest.mark.parametrize("g_shift", [4.0, 0.0], ids=["gates-near-limit", "gates-spread"])
@pytest.mark.parametrize("groups", [-1, 1], ids=["pipelined", "two-launch"])
def test_gated_prefill_at_the_lower_bound_limit(groups, g_shift):
    """lower_bound = -10.5, the API's limit.  With g shifted up the sigmoid
    sits near 1 and most gates near -10.5: the operands' scale factors reach
    their largest anchors (e^{+-84} over 8 rows).  With g ~ N(0, 1) the
    channels decay at very different rates, and 16 rows of gates often sum
    below -87: a later sub-chunk's Y factor must not pass through
    e^{m_R2 - m_Rq}, which would flush to zero there (o_intra was once 5 %
    off at the sub-chunks' first rows)."""
    x = W.dense_prefill(2, 64 * 9 + 5, 2, 4, seed=79, lower_bound=-10.5, g_shift=g_shift, state_std=0.3)
    ref = oracle.prefill(x)
    out, fin, names = _dense(x, groups=groups)
    if groups == -1:
        _assert_pipelined(names)
    check_out(out, ref["out"], f"G={groups} out at lower_bound -10.5")
    check_state(fin, ref["state"], f"G={groups} final state at lower_bound -10.5")


def test_pipelined_gate_free():
    x = W.dense_prefill(2, 64 * 9 + 40, 2, 4, seed=75, log_decay=(-0.1, 0.0), state_std=0.3)
    ref = oracle.prefill(x)
    out, fin, names = _dense(x)
    _assert_pipelined(names)
    check_out(out, ref["out"], "pipelined gate-free out")
    check_state(fin, ref["state"], "pipelined gate-free final state")


@pytest.mark.parametrize("act,state", [(torch.float16, torch.float32), (torch.bfloat16, torch.bfloat16),
                                       (torch.float16, torch.bfloat16)])
def test_pipelined_dtypes(act, state):
    x = W.dense_prefill(2, 64 * 9 + 17, 2, 4, seed=77, lower_bound=-0.3, act_dtype=act, state_dtype=state)
    ref = oracle.prefill(x)
    out, fin, names = _dense(x)
    _assert_pipelined(names)
    assert out.dtype == act
    check_out(out, ref["out"], "pipelined out")
    if state == torch.bfloat16:
        check_state_bf16(fin, ref["state"], "pipelined bf16 final state")
    else:
        check_state(fin, ref["state"], "pipelined final state")


def test_pipelined_paged_cache_dense():
    """Dense sequences on a paged cache: rows read and written back in place,
    one sequence without an initial state, one with a negative row."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(3, 300, 2, 4, seed=79, lower_bound=-0.3, state_std=0.3)
    slots = 7
    g = torch.Generator().manual_seed(79)
    pool0 = torch.randn((slots, 4, 128, 128), generator=g) * 0.3
    idx = torch.tensor([5, -1, 2], dtype=torch.int32)
    has = torch.tensor([1, 1, 0], dtype=torch.uint8)
    h0 = torch.zeros((3, 4, 128, 128))
    h0[0] = pool0[5]
    ref = oracle.prefill(dataclasses.replace(x, initial_state=h0))
    xd = x.to("cuda")
    pool = pool0.to("cuda")

    def call():
        return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 scale=x.scale, lower_bound=x.lower_bound, n_seqs=3, state_cache=pool,
                                 state_indices=idx.to("cuda"), has_initial_state=has.to("cuda"), groups=-1)
    (out, _), names = _traced(call)
    assert kda.kda_device_status(clear=True) == 0
    _assert_pipelined(names)
    check_out(out, ref["out"], "pipelined paged out")
    check_state(pool[5:6], ref["state"][0:1], "row 5 (sequence 0)")
    check_state(pool[2:3], ref["state"][2:3], "row 2 (sequence 2, zero start)")
    untouched = [s for s in range(slots) if s not in (5, 2)]
    assert torch.equal(pool[untouched].cpu(), pool0[untouched]), "untouched rows changed"


@pytest.mark.parametrize("scratch", [True, False])
def test_pipelined_conv(scratch):
    """With the fused conv: a scratch pass before the kernel, or each
    prologue item convolving its own tiles (the kernel's conv instantiation)."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(2, 64 * 5 + 9, 2, 4, seed=81, lower_bound=-0.3, state_std=0.3)
    w, st = W.conv_inputs(x.hqk, x.hv, 4, 4, taps="bf16", seed=81)
    cidx = torch.tensor([3, 0], dtype=torch.int32)
    chas = torch.tensor([1, 1], dtype=torch.uint8)
    (q2, k2, v2), st_ref = oconv.prefill(x.q, x.k, x.v, x.cu_seqlens, w, "bf16", st, cidx, chas)
    ref = oracle.prefill(dataclasses.replace(x, q=q2.bfloat16(), k=k2.bfloat16(), v=v2.bfloat16()))
    xd = x.to("cuda")
    cst = st.to("cuda")

    def call():
        return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 scale=x.scale, lower_bound=x.lower_bound, n_seqs=2,
                                 initial_state=xd.initial_state, output_final_state=True, groups=-1,
                                 conv_weight=w.to("cuda"), conv_state=cst, conv_state_indices=cidx.to("cuda"),
                                 conv_has_initial_state=chas.to("cuda"), conv_scratch=scratch)
    (out, fin), names = _traced(call)
    assert kda.kda_device_status(clear=True) == 0
    _assert_pipelined(names)
    check_out(out, ref["out"], "pipelined conv out")
    check_state(fin, ref["state"], "pipelined conv final state")
    np.testing.assert_array_equal(cst.float().cpu().numpy(), st_ref, err_msg="conv state")


def test_pipelined_most_chains():
    """48 chains (3 sequences x 16 heads), the most the launch takes, and the
    49th rejected."""
    x = W.dense_prefill(3, 64 * 6 + 3, 4, 16, seed=83, lower_bound=-0.3, state_std=0.3)
    ref = oracle.prefill(x)
    out, fin, names = _dense(x)
    _assert_pipelined(names)
    check_out(out, ref["out"], "48 chains out")
    check_state(fin, ref["state"], "48 chains final state")
    y = W.dense_prefill(7, 64, 1, 7, seed=84)
    with pytest.raises(ValueError, match="pipelined"):
        _dense(y)


def test_pipelined_rejects_varlen():
    import linear_attention_serving_fwd_gb300 as kda
    x = W.varlen_paged([70, 130], 1, 2, slots=4, seed=85).to("cuda")
    with pytest.raises(ValueError, match="pipelined"):
        kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias,
                          cu_seqlens=x.cu_seqlens, state_cache=x.state_pool.clone(),
                          state_indices=x.state_indices, groups=-1)
    assert kda.kda_device_status(clear=True) == 0


def test_pipelined_is_the_auto_choice_at_the_dense_and_long_workloads():
    """groups = 0 picks the pipelined launch for the dense (B=2, T=4096,
    H=16) and long (B=1, T=131072, H=32) prefills, and two launches for a
    one-chain prefill of four chunks."""
    for name in ("dense", "long"):
        x = W.workload(name)
        _, _, names = _dense(x, groups=0)
        _assert_pipelined(names)
    _, _, names = _dense(W.workload("tiny"), groups=0)
    assert "kda_walk" in names and "kda_pipelined" not in names, sorted(names)


def test_pipelined_repeats_bit_identical():
    """32 repeats of the dense workload through the pipelined launch, half
    after an L2 flush, give bit-identical outputs and final states: the
    record hand-over through the ready flags leaves no order dependence."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.workload("dense").to("cuda")
    T, hv, n = x.t_total, x.hv, x.n_seqs
    ws = torch.empty(kda.chunk_workspace_bytes(n, T, hv, -1), dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((T, hv, 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((n, hv, 128, 128), dtype=torch.float32, device="cuda")

    def run():
        kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias, scale=x.scale,
                          lower_bound=x.lower_bound, n_seqs=n, initial_state=x.initial_state,
                          final_state=fin, out=out, workspace=ws, groups=-1)
    run()
    torch.cuda.synchronize()
    ref_o, ref_f = out.clone(), fin.clone()
    for i in range(32):
        if i % 2:
            flush.random_()
        out.zero_()
        fin.zero_()
        run()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o), f"repeat {i}: outputs differ"
        assert torch.equal(fin, ref_f), f"repeat {i}: final states differ"
    assert kda.kda_device_status(clear=True) == 0


# ---- the 128-column walk as a launch of its own (more chains than the
# 32-column walk fits on the SMs in one wave: 4 x chains > SMs)

def test_walk128_varlen_many_chains():
    """8 ragged sequences x 8 heads = 64 chains on a paged cache: the
    prologue and then the 128-column walk, against the oracle."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.varlen_paged([70, 1, 129, 64, 5, 300, 700, 33], 2, 8, slots=12, seed=87, lower_bound=-0.4,
                       has_initial=[1, 1, 0, 1, 1, 1, 0, 1], state_std=0.3)
    ref = oracle.prefill(x)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()

    def call():
        return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 scale=x.scale, lower_bound=x.lower_bound, cu_seqlens=xd.cu_seqlens,
                                 state_cache=pool, state_indices=xd.state_indices,
                                 has_initial_state=xd.has_initial_state)
    (out, _), names = _traced(call)
    assert kda.kda_device_status(clear=True) == 0
    assert "kda_walk128" in names and "kda_walk" not in names, sorted(names)
    check_out(out, ref["out"], "walk128 out")
    live = [s for s in x.state_indices.tolist() if s >= 0]
    check_state(pool[live], ref["pool"][live], "walk128 cache rows")
    untouched = [s for s in range(pool.shape[0]) if s not in live]
    assert torch.equal(pool[untouched].cpu(), x.state_pool[untouched]), "untouched rows changed"


def _prefix_state(x, n, o, h0):
    bos = int(x.cu_seqlens[n])
    return oracle.recurrence(x.q[bos:bos + o], x.k[bos:bos + o], x.v[bos:bos + o], x.g[bos:bos + o],
                             x.beta[bos:bos + o], [0, o], A_log=x.A_log, dt_bias=x.dt_bias,
                             lower_bound=x.lower_bound, h0=h0[None])["state"][0]


@pytest.mark.parametrize("form", ["walk128", "pipelined"])
def test_128_column_walk_checkpoints(form):
    """Mid-prefill snapshots from the 128-column walk: on its own launch
    (5 sequences x 8 heads = 40 chains) and in the pipelined launch (dense,
    3 x 4 = 12 chains).  Valid offsets snapshot; 0, a misaligned offset and
    one past the sequence's end leave their rows untouched."""
    import linear_attention_serving_fwd_gb300 as kda
    if form == "walk128":
        lens = [200, 130, 517, 256, 640]
        offs = [128, 0, 512, 100, 704]
        x = W.varlen_paged(lens, 2, 8, slots=12, seed=89, lower_bound=-0.7, state_std=0.3)
        h0 = [x.state_pool[int(x.state_indices[n])].double().numpy()
              if int(x.state_indices[n]) >= 0 and bool(x.has_initial_state[n]) else np.zeros((x.hv, 128, 128))
              for n in range(len(lens))]
    else:
        lens = [320, 320, 320]
        offs = [64, 320, 100]
        x = W.dense_prefill(3, 320, 2, 4, seed=91, lower_bound=-0.7, state_std=0.3)
        h0 = [x.initial_state[n].double().numpy() for n in range(3)]
    ref = oracle.prefill(x)
    xd = x.to("cuda")
    sentinel = torch.full((len(lens), x.hv, 128, 128), 7.0, dtype=torch.float32, device="cuda")
    ck = sentinel.clone()
    offs_d = torch.tensor(offs, dtype=torch.int32, device="cuda")

    def call():
        if form == "walk128":
            pool = xd.state_pool.clone()
            return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                     lower_bound=x.lower_bound, cu_seqlens=xd.cu_seqlens, state_cache=pool,
                                     state_indices=xd.state_indices, has_initial_state=xd.has_initial_state,
                                     checkpoint_state=ck, checkpoint_offsets=offs_d)
        return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 lower_bound=x.lower_bound, n_seqs=3, initial_state=xd.initial_state,
                                 output_final_state=True, groups=-1, checkpoint_state=ck,
                                 checkpoint_offsets=offs_d)
    (out, _), names = _traced(call)
    assert kda.kda_device_status(clear=True) == 0
    assert ("kda_walk128" if form == "walk128" else "kda_pipelined") in names, sorted(names)
    check_out(out, ref["out"], f"{form} out with checkpoints")
    for n, o in enumerate(offs):
        if o > 0 and o % 64 == 0 and o <= lens[n]:
            check_state(ck[n:n + 1], _prefix_state(x, n, o, h0[n])[None], f"{form} snapshot {n} at {o}")
        else:
            assert torch.equal(ck[n], sentinel[n]), f"{form} sequence {n}: skipped snapshot wrote its row"


def test_pipelined_workspace_offset_16_bytes():
    """A workspace that is only 16-byte aligned (the API's requirement): the
    records then straddle 128-byte lines, so the walk must not drop them
    from L2; results as from an aligned workspace, against the oracle."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(2, 64 * 12 + 7, 2, 4, seed=93, lower_bound=-0.3, state_std=0.3)
    ref = oracle.prefill(x)
    xd = x.to("cuda")
    need = kda.chunk_workspace_bytes(2, x.t_total, x.hv, -1)
    raw = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    ws = raw[16:16 + need]
    assert ws.data_ptr() % 128 == 16

    def call():
        return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 scale=x.scale, lower_bound=x.lower_bound, n_seqs=2,
                                 initial_state=xd.initial_state, output_final_state=True, groups=-1,
                                 workspace=ws)
    (out, fin), names = _traced(call)
    assert kda.kda_device_status(clear=True) == 0
    _assert_pipelined(names)
    check_out(out, ref["out"], "offset workspace out")
    check_state(fin, ref["state"], "offset workspace final state")


@pytest.mark.parametrize("act,state,decay", [(torch.float16, torch.float32, None),
                                             (torch.bfloat16, torch.bfloat16, None),
                                             (torch.bfloat16, torch.float32, (-0.1, 0.0))],
                         ids=["fp16-act", "bf16-state", "gate-free"])
def test_walk128_dtypes_and_gate_free(act, state, decay):
    """The 128-column walk on its own launch (6 sequences x 8 heads = 48
    chains) with fp16 activations, a bf16 cache, or raw log decays."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.varlen_paged([70, 129, 64, 5, 300, 33], 2, 8, slots=9, seed=95, lower_bound=-0.3, state_std=0.3,
                       act_dtype=act, state_dtype=state, log_decay=decay)
    ref = oracle.prefill(x)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()

    def call():
        return kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 scale=x.scale, lower_bound=x.lower_bound, cu_seqlens=xd.cu_seqlens,
                                 state_cache=pool, state_indices=xd.state_indices,
                                 has_initial_state=xd.has_initial_state)
    (out, _), names = _traced(call)
    assert kda.kda_device_status(clear=True) == 0
    assert "kda_walk128" in names, sorted(names)
    assert out.dtype == act
    check_out(out, ref["out"], "walk128 out")
    live = [s for s in x.state_indices.tolist() if s >= 0]
    if state == torch.bfloat16:
        check_state_bf16(pool[live], ref["pool"][live], "walk128 bf16 cache rows")
    else:
        check_state(pool[live], ref["pool"][live], "walk128 cache rows")
