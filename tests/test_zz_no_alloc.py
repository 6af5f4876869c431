"""kda_chunk_fwd_noalloc: the prefill for callers that cannot allocate device
memory (runtimes that reserve all memory up front or forbid cudaMalloc after
graph capture, plugins whose host owns the allocator, code that must not
synchronise).  Its scratch is a fixed 64 MiB array inside the library.

This file is collected last on purpose.  Each call is checked against the
regular entry point (same inputs, caller-provided workspace) bit for bit:
both run the same kernels on the same inputs and the prefill is
deterministic.  Calls come two in a row with different inputs, so stale
scratch contents from the first call cannot leak into the second: varlen
with the serial walk, varlen with four chunk groups (the group planes in
the scratch), and dense sequences (closed-form chunk tables, so the
scratch's chunk table is skipped and left stale).  It passes alone in a
fresh process and after the other tests."""
from __future__ import annotations

import pytest
import torch

from linear_attention_serving_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(kind, seed):
    if kind == "dense":
        return W.dense_prefill(2, 64 * 5 + 17, 2, 4, seed=seed, lower_bound=-0.5).to("cuda")
    return W.varlen_paged([300, 64, 777, 1], 2, 4, slots=7, seed=seed, lower_bound=-0.5,
                          has_initial=[1, 0, 1, 1]).to("cuda")


def _call(kda, fn, x, groups, **extra):
    kw = dict(A_log=x.A_log, dt_bias=x.dt_bias, lower_bound=x.lower_bound, groups=groups)
    out = torch.empty((x.t_total, x.hv, 128), dtype=torch.bfloat16, device="cuda")
    if x.state_pool is not None:
        pool = x.state_pool.clone()
        fn(x.q, x.k, x.v, x.g, x.beta, out=out, cu_seqlens=x.cu_seqlens, state_cache=pool,
           state_indices=x.state_indices, has_initial_state=x.has_initial_state, **kw, **extra)
        return out, pool
    fin = torch.empty((x.n_seqs, x.hv, 128, 128), dtype=torch.float32, device="cuda")
    fn(x.q, x.k, x.v, x.g, x.beta, out=out, n_seqs=x.n_seqs, initial_state=x.initial_state,
       final_state=fin, **kw, **extra)
    return out, fin


@pytest.mark.parametrize("kind,groups", [("varlen", 1), ("varlen", 4), ("dense", 1)])
def test_noalloc_matches_regular_entry_point_twice(kind, groups):
    import linear_attention_serving_fwd_gb300 as kda
    for seed in (11, 12):  # two calls in a row, different inputs
        x = _inputs(kind, seed)
        out_r, st_r = _call(kda, kda.kda_chunk_fwd, x, groups)
        out_n, st_n = _call(kda, kda.kda_chunk_fwd_noalloc, x, groups)
        torch.cuda.synchronize()
        assert kda.kda_device_status(clear=True) == 0
        assert torch.equal(out_n, out_r), f"{kind} G={groups} seed {seed}: outputs differ"
        assert torch.equal(st_n, st_r), f"{kind} G={groups} seed {seed}: states differ"
        if x.state_pool is not None:
            live = [s for s in x.state_indices.tolist() if s >= 0]
            untouched = [s for s in range(st_n.shape[0]) if s not in live]
            assert torch.equal(st_n[untouched], x.state_pool[untouched])


def test_noalloc_rejects_calls_beyond_its_scratch():
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(1, 64 * 600, 1, 4, seed=1, init_state=False, device="cuda")
    assert kda.chunk_workspace_bytes(1, x.t_total, x.hv, 0) > 64 << 20
    out = torch.empty((x.t_total, x.hv, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="64 MiB"):
        kda.kda_chunk_fwd_noalloc(x.q, x.k, x.v, x.g, x.beta, out=out, A_log=x.A_log,
                                  dt_bias=x.dt_bias, n_seqs=1)
