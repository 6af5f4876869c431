"""GPU parity of kda_chunk_fwd_host (prefill on host-memory tensors, cut
into chunk-aligned segments with the fp32 state carried between them, the
copies overlapped with the kernels) against the fp64 oracle and against the
device-resident kda_chunk_fwd, through the C ABI."""
from __future__ import annotations

import dataclasses

import pytest
import torch

import oracle
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state

pytestmark = pytest.mark.gpu


def _host(x, *, segment, pinned=True, dense=False, fused=False, groups=0):
    import linear_attention_serving_fwd_gb300 as kda

    def h(t):
        return t.pin_memory() if pinned else t.clone()

    q, k, v = x.q, x.k, x.v
    if fused:  # q, k, v as strided views of one fused projection row
        T = x.t_total
        qkv = h(torch.cat([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], dim=1))
        a, b = x.hqk * 128, 2 * x.hqk * 128
        q, k, v = (qkv[:, :a].view(T, x.hqk, 128), qkv[:, a:b].view(T, x.hqk, 128),
                   qkv[:, b:].view(T, x.hv, 128))
    else:
        q, k, v = h(q), h(k), h(v)
    out, fin = kda.kda_chunk_fwd_host(
        q, k, v, h(x.g), h(x.beta), A_log=x.A_log, dt_bias=x.dt_bias, scale=x.scale,
        lower_bound=x.lower_bound, cu_seqlens=None if dense else x.cu_seqlens, n_seqs=x.n_seqs,
        initial_state=None if x.initial_state is None else h(x.initial_state.contiguous()),
        output_final_state=True, segment_tokens=segment, groups=groups)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    assert not out.is_cuda and not fin.is_cuda
    return out, fin


def _varlen_with_initial(lens, hqk, hv, seed, **kw):
    x = W.varlen_paged(lens, hqk, hv, slots=len(lens) + 2, seed=seed, **kw)
    h0 = x.state_pool[x.state_indices.long()].clone()
    return dataclasses.replace(x, initial_state=h0, state_pool=None, state_indices=None,
                               has_initial_state=None, output_final_state=True)


def test_dense_segments():
    """B=2 x 700 tokens in 128-token segments (five full, one of 60): weak
    decay, so each segment's output depends on the carried state."""
    x = W.dense_prefill(2, 700, 2, 4, seed=5, lower_bound=-0.05, state_std=0.3)
    ref = oracle.prefill(x)
    out, fin = _host(x, segment=128, dense=True)
    check_out(out, ref["out"], "host dense out")
    check_state(fin, ref["state"], "host dense final state")


def test_varlen_shrinking_calls_fused_rows():
    """Ragged sequences (one empty, one of a single token) in 64-token
    segments: later calls hold fewer sequences and pieces of unequal length;
    q, k, v are strided views of one fused host row."""
    x = _varlen_with_initial([70, 1, 0, 129, 300, 64], 2, 4, seed=41, lower_bound=-0.3, state_std=0.2)
    ref = oracle.prefill(x)
    out, fin = _host(x, segment=64, fused=True)
    check_out(out, ref["out"], "host varlen out")
    check_state(fin, ref["state"], "host varlen final state")
    assert torch.equal(fin[2], x.initial_state[2]), "an empty sequence's final state is its initial state"


def test_pageable_host_memory():
    """Pageable (not page-locked) host tensors: the copies do not overlap but
    the results are the same."""
    x = W.dense_prefill(1, 320, 1, 2, seed=6, lower_bound=-0.2, state_std=0.2)
    ref = oracle.prefill(x)
    out, fin = _host(x, segment=256, pinned=False, dense=True)
    check_out(out, ref["out"], "pageable out")
    check_state(fin, ref["state"], "pageable final state")


def test_full_dense_workload_matches_device_path():
    """The timed prefill workload (B=2, T=4096, H=16) through the host path
    against the device-resident prefill of the same inputs."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.workload("dense")
    xd = x.to("cuda")
    out_d, fin_d = kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                     scale=x.scale, lower_bound=x.lower_bound, n_seqs=x.n_seqs,
                                     initial_state=xd.initial_state, output_final_state=True)
    out_h, fin_h = _host(x, segment=0, dense=True)
    od, oh = out_d.float().cpu(), out_h.float()
    assert torch.allclose(oh, od, rtol=2e-2, atol=2e-3), float((oh - od).abs().max())
    rel = float((fin_h - fin_d.cpu()).norm() / fin_d.norm().cpu())
    assert rel < 1e-4, rel


def test_fp16_activations_default_segments():
    """fp16 q/k/v/g/beta and output through the default (shrinking)
    segments: one sequence of 300 tokens runs as segments of 64 and 236
    tokens (a 256-token segment cut short by the sequence's end)."""
    x = W.dense_prefill(1, 300, 2, 2, seed=8, lower_bound=-0.3, state_std=0.2, act_dtype=torch.float16)
    ref = oracle.prefill(x)
    out, fin = _host(x, segment=0, dense=True)
    assert out.dtype == torch.float16
    check_out(out, ref["out"], "host fp16 out")
    check_state(fin, ref["state"], "host fp16 final state")


def test_empty_batch_returns_initial_states():
    """Every sequence empty: no segment call runs; the final states are the
    initial ones and the output is empty."""
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(2, 64, 1, 2, seed=9)
    e = lambda t: t[:0].pin_memory()
    h0 = x.initial_state.contiguous().pin_memory()
    out, fin = kda.kda_chunk_fwd_host(e(x.q), e(x.k), e(x.v), e(x.g), e(x.beta), A_log=x.A_log,
                                      dt_bias=x.dt_bias, cu_seqlens=torch.zeros(3, dtype=torch.int32),
                                      initial_state=h0, output_final_state=True)
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 128)
    assert torch.equal(fin, h0)


def test_group_scan_inside_segment_calls():
    """Each 256-token segment call runs the chunk-group scan (G = 4) on its
    pieces, the state carried between calls through the cache table."""
    x = _varlen_with_initial([700, 1300, 64], 1, 2, seed=42, lower_bound=-0.1, state_std=0.2)
    ref = oracle.prefill(x)
    out, fin = _host(x, segment=256, groups=4)
    check_out(out, ref["out"], "host group-scan out")
    check_state(fin, ref["state"], "host group-scan final state")
