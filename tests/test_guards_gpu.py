"""Guard regions around every buffer the kernels write: outputs, final
states, verify records and the prefill workspace (including the chunk-group
scan's operators) are views into larger buffers whose margins hold a
sentinel, and every margin must come back untouched."""
from __future__ import annotations

import pytest
import torch

from linear_attention_serving_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

G = 1024  # guard elements on each side (16-byte multiples for every dtype here)
SENT = {torch.bfloat16: -12345.0, torch.float32: -7.5e30, torch.uint8: 0xA5}


def _guarded(shape, dtype):
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 2 * G,), SENT[dtype], dtype=dtype, device="cuda")
    return buf, buf[G:G + n].view(shape)


def _check(buf, what):
    ref = torch.full((G,), SENT[buf.dtype], dtype=buf.dtype, device="cuda")
    assert torch.equal(buf[:G], ref), f"{what}: front guard overwritten"
    assert torch.equal(buf[-G:], ref), f"{what}: back guard overwritten"


@pytest.mark.parametrize("groups", [1, 4])
def test_prefill_guards(groups):
    import linear_attention_serving_fwd_gb300 as kda
    x = W.varlen_paged([700, 64, 1300, 5], 1, 2, slots=6, seed=51, lower_bound=-0.2).to("cuda")
    n, T, hv = x.n_seqs, x.t_total, x.hv
    ob, out = _guarded((T, hv, 128), torch.bfloat16)
    h0 = x.state_pool[x.state_indices.long()].contiguous()
    fb, fin = _guarded((n, hv, 128, 128), torch.float32)
    ws_bytes = kda.chunk_workspace_bytes(n, T, hv, groups)
    wb = torch.full((ws_bytes + 4096,), SENT[torch.uint8], dtype=torch.uint8, device="cuda")
    kda.kda_chunk_fwd(x.q, x.k, x.v, x.g, x.beta, A_log=x.A_log, dt_bias=x.dt_bias, cu_seqlens=x.cu_seqlens,
                      initial_state=h0, final_state=fin, out=out, groups=groups, workspace=wb[:ws_bytes])
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    _check(ob, "out")
    _check(fb, "final_state")
    assert torch.equal(wb[ws_bytes:], torch.full((4096,), SENT[torch.uint8], dtype=torch.uint8,
                                                 device="cuda")), "workspace overrun"
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()


@pytest.mark.parametrize("window", [1, 4])
def test_decode_and_verify_guards(window):
    import linear_attention_serving_fwd_gb300 as kda
    qlens = [window, 1, 0, window] if window > 1 else None
    x = W.decode_batch(4, window, 2, 4, slots=9, seed=52, qlens=qlens, null_requests=(1,)).to("cuda")
    T, hv, n = x.t_total, x.hv, x.n_seqs
    pool = x.state_pool.clone()
    ob, out = _guarded((T, hv, 128), torch.bfloat16)
    kda.kda_decode(x.q, x.k, x.v, x.g, x.beta, pool, x.cu_seqlens, x.state_indices, window,
                   A_log=x.A_log, dt_bias=x.dt_bias, out=out)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    _check(ob, "decode out")
    ob, out = _guarded((T, hv, 128), torch.bfloat16)
    cb, corr = _guarded((n, hv, window, 128), torch.float32)
    kb, kg = _guarded((n, hv, window, 256), torch.bfloat16)
    kda.kda_verify(x.q, x.k, x.v, x.g, x.beta, pool, x.cu_seqlens, x.state_indices, window,
                   A_log=x.A_log, dt_bias=x.dt_bias, out=out, corr=corr, kg=kg)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    for buf, what in ((ob, "verify out"), (cb, "corr"), (kb, "kg")):
        _check(buf, what)
