"""kda_chunk_fwd_noalloc: the prefill for callers that cannot allocate device
memory (runtimes that reserve all memory up front or forbid cudaMalloc after
graph capture, plugins whose host owns the allocator, code that must not
synchronise).  Its scratch is a fixed 64 MiB array inside the library.

This file is collected last on purpose.  Each call is checked against the
regular entry point (same inputs, caller-provided workspace) within the
parity tolerances, on two calls in a row with different inputs, so stale
scratch contents from the first call cannot leak into the second.  It passes
alone in a fresh process and after the other tests."""
from __future__ import annotations

import pytest
import torch

from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import OUT_ATOL, OUT_RTOL, OUT_REL_FRO, STATE_REL_FRO, np64, rel_fro

pytestmark = pytest.mark.gpu


def _inputs(seed):
    x = W.varlen_paged([300, 64, 777, 1], 2, 4, slots=7, seed=seed, lower_bound=-0.5,
                       has_initial=[1, 0, 1, 1]).to("cuda")
    return x


def _regular(kda, x):
    pool = x.state_pool.clone()
    out, _ = kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias,
                               lower_bound=x.lower_bound, cu_seqlens=x.cu_seqlens,
                               state_cache=pool, state_indices=x.state_indices,
                               has_initial_state=x.has_initial_state)
    return out, pool


def _noalloc(kda, x):
    pool = x.state_pool.clone()
    out = torch.empty((x.t_total, x.hv, 128), dtype=torch.bfloat16, device="cuda")
    kda.kda_chunk_fwd_noalloc(x.q, x.k, x.v, x.g, x.beta, out=out, A_log=x.A_log,
                              dt_bias=x.dt_bias, lower_bound=x.lower_bound,
                              cu_seqlens=x.cu_seqlens, state_cache=pool,
                              state_indices=x.state_indices,
                              has_initial_state=x.has_initial_state)
    return out, pool


def test_noalloc_matches_regular_entry_point_twice():
    import linear_attention_serving_fwd_gb300 as kda
    for seed in (11, 12):  # two calls in a row, different inputs
        x = _inputs(seed)
        out_r, pool_r = _regular(kda, x)
        out_n, pool_n = _noalloc(kda, x)
        torch.cuda.synchronize()
        assert kda.kda_device_status(clear=True) == 0
        a, b = np64(out_n), np64(out_r)
        assert abs(a - b).max() <= OUT_ATOL + OUT_RTOL * abs(b).max()
        assert rel_fro(a, b) <= OUT_REL_FRO
        assert rel_fro(np64(pool_n), np64(pool_r)) <= STATE_REL_FRO
        live = [s for s in x.state_indices.tolist() if s >= 0]
        untouched = [s for s in range(pool_n.shape[0]) if s not in live]
        assert torch.equal(pool_n[untouched], x.state_pool[untouched])


def test_noalloc_rejects_calls_beyond_its_scratch():
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(1, 64 * 600, 1, 4, seed=1, init_state=False, device="cuda")
    assert kda.chunk_workspace_bytes(1, x.t_total, x.hv, 0) > 64 << 20
    out = torch.empty((x.t_total, x.hv, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="64 MiB"):
        kda.kda_chunk_fwd_noalloc(x.q, x.k, x.v, x.g, x.beta, out=out, A_log=x.A_log,
                                  dt_bias=x.dt_bias, n_seqs=1)
