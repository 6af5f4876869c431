"""GPU parity of the fused width-4 conv + SiLU (raw q/k/v projection bands)
in prefill (kda_chunk_fwd_ex with a conv) and verify (kda_verify_ex), against
the conv oracle followed by the fp64 recurrence, through the C ABI."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import conv as oconv
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state, np64

pytestmark = pytest.mark.gpu


def _layout(st, dim_first):
    """Device copy of a token-major [rows, positions, C] conv state in the
    requested layout."""
    st = st.to("cuda")
    return st.transpose(1, 2).contiguous() if dim_first else st.clone()


def _token_major(st, dim_first):
    return (st.transpose(1, 2) if dim_first else st).float().cpu().numpy()


def _bf16_close(got, want, what):
    """bf16 tensors equal or one bf16 step apart (a SiLU rounding boundary
    between the kernel's fp32 and the oracle's fp64 evaluation)."""
    g = got.float().cpu().numpy()
    w = np.asarray(want, np.float32)
    step = np.maximum(np.abs(w), 1e-30) * 2.0 ** -7
    bad = np.abs(g - w) > step * 1.0001
    assert not bad.any(), f"{what}: {int(bad.sum())} values beyond one bf16 step"
    frac = float(np.mean(g != w))
    assert frac < 0.01, f"{what}: {frac:.3%} of values differ"


def _conv_inputs(x, dense_bands=False):
    """The raw bands as the library sees them: separate tensors, or strided
    views of one fused [T, C] projection."""
    if not dense_bands:
        return x.q, x.k, x.v
    T, hqk, hv = x.t_total, x.hqk, x.hv
    qkv = torch.cat([x.q.reshape(T, -1), x.k.reshape(T, -1), x.v.reshape(T, -1)], dim=1)
    a, b = hqk * 128, 2 * hqk * 128
    return (qkv[:, :a].view(T, hqk, 128), qkv[:, a:b].view(T, hqk, 128), qkv[:, b:].view(T, hv, 128))


def _prefill_case(x, taps, dim_first, cidx, chas, groups=1, fused=False, positions=4, scratch=True):
    import linear_attention_serving_fwd_gb300 as kda
    w, st = W.conv_inputs(x.hqk, x.hv, x.state_pool.shape[0], positions, taps=taps, seed=x.t_total)
    (q2, k2, v2), st_ref = oconv.prefill(x.q, x.k, x.v, x.cu_seqlens, w, taps, st, cidx, chas)
    xc = dataclasses.replace(x, q=q2.bfloat16(), k=k2.bfloat16(), v=v2.bfloat16())
    ref = oracle.prefill(xc)
    xd = x.to("cuda")
    q, k, v = _conv_inputs(xd, fused)
    pool = xd.state_pool.clone()
    cst = _layout(st, dim_first)
    out, _ = kda.kda_chunk_fwd(q, k, v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                               scale=x.scale, lower_bound=x.lower_bound, cu_seqlens=xd.cu_seqlens,
                               state_cache=pool, state_indices=xd.state_indices,
                               has_initial_state=xd.has_initial_state, groups=groups,
                               conv_weight=w.to("cuda"), conv_state=cst,
                               conv_state_indices=cidx.to("cuda"),
                               conv_has_initial_state=None if chas is None else chas.to("cuda"),
                               conv_dim_first=dim_first, conv_scratch=scratch)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    check_out(out, ref["out"], "conv prefill out")
    live = [s for s in x.state_indices.tolist() if s >= 0]
    check_state(pool[live], ref["pool"][live], "conv prefill cache rows")
    np.testing.assert_array_equal(_token_major(cst, dim_first), st_ref, err_msg="conv state")


@pytest.mark.parametrize("scratch", [True, False])
@pytest.mark.parametrize("taps,dim_first", [("bf16", False), ("f32", True), ("bf16", True)])
def test_prefill_conv_small(taps, dim_first, scratch):
    """Ragged sequences (lengths 1 and 2 below the conv history, chunk
    multiples, a 300-token chain), conv rows without history, a sequence
    with no conv row; the conv in its own pass (scratch) or in each
    prologue item."""
    x = W.varlen_paged([70, 1, 2, 129, 64, 5, 300], 2, 4, slots=9, seed=31, lower_bound=-0.4,
                       has_initial=[1, 0, 1, 1, 1, 0, 1])
    cidx = x.state_indices.clone()
    cidx[4] = -1
    chas = torch.tensor([1, 1, 0, 1, 1, 1, 0], dtype=torch.uint8)
    _prefill_case(x, taps, dim_first, cidx, chas, scratch=scratch)


@pytest.mark.parametrize("scratch", [True, False])
def test_prefill_conv_group_scan_and_fused_bands(scratch):
    """The chunk-group scan on convolved inputs, with q/k/v as strided views
    of one fused projection and a longer conv state row."""
    x = W.varlen_paged([700, 64, 1300], 1, 2, slots=5, seed=33, lower_bound=-0.1,
                       has_initial=[1, 1, 0])
    cidx = torch.tensor([3, 0, 4], dtype=torch.int32)
    _prefill_case(x, "f32", False, cidx, None, groups=4, fused=True, positions=6, scratch=scratch)


def test_prefill_conv_paths_agree_bitwise():
    """The conv in its own pass and the conv in each prologue item evaluate
    the same roundings in the same order: bit-identical outputs, states and
    conv rows on the varlen workload's shapes (GVA 4)."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.varlen_paged([300, 1000, 7, 700], 2, 8, slots=6, seed=37, lower_bound=-0.3).to("cuda")
    w, st = W.conv_inputs(x.hqk, x.hv, 6, 4, taps="bf16", seed=37, device="cuda")
    res = []
    for scratch in (True, False):
        pool, cst = x.state_pool.clone(), st.clone()
        out, _ = kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias,
                                   cu_seqlens=x.cu_seqlens, state_cache=pool, state_indices=x.state_indices,
                                   conv_weight=w, conv_state=cst, conv_state_indices=x.state_indices,
                                   conv_scratch=scratch)
        res.append((out, pool, cst))
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    for a, b, what in zip(res[0], res[1], ("out", "state cache", "conv state")):
        assert torch.equal(a, b), what


def test_prefill_conv_varlen_full():
    """8 sequences summing to 32768 tokens, Hqk=8, Hv=32, bf16 taps, fused
    projection bands, conv rows = cache rows."""
    x = W.workload("varlen")
    _prefill_case(x, "bf16", False, x.state_indices.clone(), x.has_initial_state, fused=True)


def _verify_case(x, taps, dim_first, acc, positions):
    import linear_attention_serving_fwd_gb300 as kda
    w, st = W.conv_inputs(x.hqk, x.hv, x.state_pool.shape[0], positions, taps=taps, seed=x.n_seqs)
    (q2, k2, v2), st_ref = oconv.verify(x.q, x.k, x.v, x.cu_seqlens, w, taps, st, x.state_indices, acc)
    xc = dataclasses.replace(x, q=q2.bfloat16(), k=k2.bfloat16(), v=v2.bfloat16())
    ref = oracle.window(xc)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    cst = _layout(st, dim_first)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, corr, kg = kda.kda_verify(xd.q, xd.k, xd.v, xd.g, xd.beta, pool, xd.cu_seqlens,
                                   xd.state_indices, x.window, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                   scale=x.scale, lower_bound=x.lower_bound, work_counter=counter,
                                   conv_weight=w.to("cuda"), conv_state=cst,
                                   num_accepted_tokens=acc.to("cuda"), conv_dim_first=dim_first)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    check_out(out, ref["out"], "conv verify out")
    assert torch.equal(pool, xd.state_pool), "verify modified the state pool"
    assert int(counter.item()) == 0
    np.testing.assert_array_equal(_token_major(cst, dim_first), st_ref, err_msg="rolled conv state")
    cu = x.cu_seqlens.tolist()
    corr = np64(corr)
    kg = kg.cpu()
    r = x.hv // x.hqk
    for b in range(x.n_seqs):
        if x.state_indices[b] < 0:
            continue
        for t in range(cu[b + 1] - cu[b]):
            ref_u = ref["corr"][cu[b] + t]
            err = np.linalg.norm(corr[b, :, t] - ref_u) / np.linalg.norm(ref_u)
            assert err < 1e-3, (b, t, err)
            _bf16_close(kg[b, :, t, :128], k2[cu[b] + t].repeat_interleave(r, dim=0).numpy(),
                        f"kg record (convolved k) of request {b} token {t}")
            assert torch.equal(kg[b, :, t, 128:], x.g[cu[b] + t])


@pytest.mark.parametrize("taps,dim_first", [("bf16", True), ("f32", False)])
def test_verify_conv_small(taps, dim_first):
    """Ragged windows, an empty and a padding request, accepted counts 1..4
    reading histories at every position of a window + 2 row."""
    x = W.decode_batch(7, 4, 2, 4, slots=12, seed=32, qlens=[4, 1, 0, 3, 4, 2, 4],
                       null_requests=(5,), lower_bound=-0.6)
    acc = torch.tensor([1, 4, 2, 3, 1, 2, 4], dtype=torch.int32)
    _verify_case(x, taps, dim_first, acc, positions=6)


def test_verify_conv_window8():
    """Windows of up to 8 tokens: 16 (token, channel-half) conv units on the
    CTA's 8 warps, two per warp; accepted counts up to 8 on a 10-position
    conv row."""
    x = W.decode_batch(4, 8, 2, 4, slots=8, seed=35, qlens=[8, 5, 1, 7], lower_bound=-0.6)
    acc = torch.tensor([1, 8, 3, 6], dtype=torch.int32)
    _verify_case(x, "bf16", False, acc, positions=10)


def test_verify_conv_serving_batch():
    """256 requests x 4 tokens, Hqk=Hv=32, 512-slot pool, accepted counts
    U{1..4}, bf16 taps, token-major conv state of window + 2 positions."""
    x = W.workload("decode", window=4)
    acc = torch.randint(1, 5, (x.n_seqs,), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    _verify_case(x, "bf16", False, acc, positions=6)


def test_verify_conv_bad_accepted_is_padding():
    import linear_attention_serving_fwd_gb300 as kda
    x = W.decode_batch(3, 4, 1, 1, slots=5, seed=34, qlens=[4, 4, 4])
    w, st = W.conv_inputs(1, 1, 5, 6, seed=34)
    xd = x.to("cuda")
    cst = st.to("cuda")
    before = cst.clone()
    out, _, _ = kda.kda_verify(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.state_pool.clone(), xd.cu_seqlens,
                               xd.state_indices, 4, A_log=xd.A_log, dt_bias=xd.dt_bias,
                               conv_weight=w.to("cuda"), conv_state=cst,
                               num_accepted_tokens=torch.tensor([1, 0, 5], dtype=torch.int32,
                                                                device="cuda"))
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 5
    cu = x.cu_seqlens.tolist()
    assert torch.count_nonzero(out[cu[1]:cu[3]]) == 0
    slots = x.state_indices.tolist()
    assert torch.equal(cst[slots[1]], before[slots[1]]) and torch.equal(cst[slots[2]], before[slots[2]])
    assert not torch.equal(cst[slots[0]], before[slots[0]])
