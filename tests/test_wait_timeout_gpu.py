"""The bounded device waits give up cleanly (no fault, no trap, no hang).

kda_selftest_wait_timeout runs the chunk kernels' bounded mbarrier wait on a
barrier that nothing arrives at, with a 1 ms limit, in a CTA that holds
tensor memory.  The wait must expire, the device error word must report
KDA_ERR_DEVICE_TIMEOUT, the kernel must return (the synchronise inside
kda_device_status finishes), and the next regular call must be clean."""
from __future__ import annotations

import time

import pytest
import torch

import oracle
from linear_attention_serving_fwd_gb300 import _native
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    import linear_attention_serving_fwd_gb300 as kda
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    t0 = time.perf_counter()
    kda.kda_selftest_wait_timeout(1000)
    assert kda.kda_device_status(clear=True) == _native.KDA_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0, "the expired wait took far longer than its limit"
    assert kda.kda_device_status(clear=True) == 0, "the error word was not cleared"
    # the context is usable: a regular prefill right after is clean and correct
    x = W.dense_prefill(1, 200, 1, 2, seed=5, lower_bound=-1.0)
    ref = oracle.prefill(x)
    xd = x.to("cuda")
    out, fin = kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                                 lower_bound=x.lower_bound, n_seqs=1, initial_state=xd.initial_state,
                                 output_final_state=True)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    check_out(out, ref["out"])
    check_state(fin, ref["state"])

