"""The prefill's per-(chunk, head) records against the oracle's chunk form.

kda_chunk_fwd's prologue writes, for every (chunk, head), the tensor-core
operands of the walk into the caller's workspace (fp16, K-major core-matrix
layout):  WQ = [w ; qg - A_qk w] (128 x 128), KGT = kg^T (128 x 64),
TT = [T ; A_qk T] (128 x 64) and d (fp32 128).  This test decodes them and
compares each with the same quantity built by oracle/chunked.py, which pins
the prologue's intermediates, not only the end result.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import chunked
from linear_attention_serving_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

D, C = 128, 64
MAIN = 128 * 128 * 2 + 128 * 64 * 2 * 2 + 128 * 4
VB_LBO = 528
VB = VB_LBO * 8
REC = MAIN + 4 * VB


def _kmajor_decode(raw: np.ndarray, R: int, K: int) -> np.ndarray:
    """Inverse of byte(row, k) = (k/8)(R*16) + (row/8)128 + (row%8)16 + (k%8)2."""
    h = raw.view(np.float16).astype(np.float64)
    rows = np.arange(R)[:, None]
    ks = np.arange(K)[None, :]
    idx = ((ks // 8) * (R * 16) + (rows // 8) * 128 + (rows % 8) * 16 + (ks % 8) * 2) // 2
    return h[idx]


def _kmajor_decode_lbo(raw: np.ndarray, R: int, K: int, lbo: int) -> np.ndarray:
    h = raw.view(np.float16).astype(np.float64)
    rows = np.arange(R)[:, None]
    ks = np.arange(K)[None, :]
    idx = ((ks // 8) * lbo + (rows // 8) * 128 + (rows % 8) * 16 + (ks % 8) * 2) // 2
    return h[idx]


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("T,lb", [(130, -0.3), (64, -5.0)])
def test_prologue_records_match_chunk_form(T, lb):
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(1, T, 1, 2, seed=21, lower_bound=lb, init_state=False)
    xd = x.to("cuda")
    ws_bytes = kda.chunk_workspace_bytes(1, T, 2, 1)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                      lower_bound=lb, n_seqs=1, output_final_state=True, groups=1, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    raw = ws.cpu().numpy()
    max_chunks = T // C + 1
    int_words = (4 + 2 + 2 * max_chunks + 63) // 64 * 64
    n_chunks = int(raw[:4].view(np.int32)[0])
    assert n_chunks == -(-T // C)
    base = int_words * 4
    f = lambda t: t.float().numpy().astype(np.float64)
    for h in range(2):
        qh, kh, gate, b = chunked.activations(f(x.q[:, 0]), f(x.k[:, 0]), f(x.g[:, h]),
                                              f(x.beta[:, h]), float(x.A_log[h]), f(x.dt_bias[h]),
                                              x.scale, lb)
        for c in range(n_chunks):
            s, e = c * C, min(T, (c + 1) * C)
            ops = chunked.chunk_operands(qh[s:e], kh[s:e], gate[s:e], b[s:e])
            L = e - s
            pad = lambda a, shape: np.pad(a, [(0, shape[i] - a.shape[i]) for i in range(a.ndim)])
            Tm = pad(ops["T"], (C, C))
            w = pad(ops["w"], (C, D))
            Aqk = pad(ops["Aqk"], (C, C))
            qg = pad(ops["qg"], (C, D))
            kg = pad(ops["kg"], (C, D))
            want_wq = np.vstack([w, qg - Aqk @ w])
            want_kgt = kg.T
            want_tt = np.vstack([Tm, Aqk @ Tm])
            off = base + (c * 2 + h) * REC
            rec = raw[off:off + REC]
            got_wq = _kmajor_decode(rec[0:32768], 128, 128)
            got_kgt = _kmajor_decode(rec[32768:49152], 128, 64)
            got_tt = _kmajor_decode(rec[49152:65536], 128, 64)
            got_d = rec[65536:66048].view(np.float32).astype(np.float64)
            tag = f"T={T} head {h} chunk {c} (len {L})"
            assert _rel(got_tt[:64], want_tt[:64]) < 2e-3, f"T block {tag}: {_rel(got_tt[:64], want_tt[:64])}"
            assert _rel(got_tt[64:], want_tt[64:]) < 1e-2, f"A_qk T {tag}: {_rel(got_tt[64:], want_tt[64:])}"
            assert _rel(got_kgt, want_kgt) < 2e-3, f"kg {tag}"
            assert _rel(got_d, ops["d"]) < 1e-4, f"d {tag}"
            assert _rel(got_wq[:64], want_wq[:64]) < 5e-3, f"w {tag}: {_rel(got_wq[:64], want_wq[:64])}"
            assert _rel(got_wq[64:], want_wq[64:]) < 1e-2, f"qg' {tag}: {_rel(got_wq[64:], want_wq[64:])}"
            # v^T blocks, fp16 [32 value columns][64 rows]: bf16 v converted to
            # fp16, exact except below fp16's normal range (absolute 3e-8)
            vv = pad(f(x.v[s:e, h]), (C, D))
            for jb in range(4):
                got_v = _kmajor_decode_lbo(rec[MAIN + jb * VB:MAIN + (jb + 1) * VB], 32, 64, VB_LBO)
                np.testing.assert_allclose(got_v, vv[:, 32 * jb:32 * (jb + 1)].T, rtol=0, atol=3e-8,
                                           err_msg=f"v block {jb} {tag}")
