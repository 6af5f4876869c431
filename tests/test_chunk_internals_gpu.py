"""The prefill's per-(chunk, head) records against the oracle's chunk form.

kda_chunk_fwd's prologue writes, for every (chunk, head), the walk's
tensor-core operands into the caller's workspace (fp16, K-major core-matrix
layout): P = -kg^T w (128 x 128), R = kg^T T (128 x 64), d (fp32 128),
qg' = qg - A_qk w (64 x 128), o_intra = A_qk T v (bf16, four blocks of
[64 rows][32 value columns], row r's 16-byte chunks rotated by r // 2) and
v^T (128 value columns x 64 rows).  This test decodes them and compares each with the same
quantity built by oracle/chunked.py, which pins the prologue's
intermediates, not only the end result.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import chunked
from linear_attention_serving_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

D, C = 128, 64
OFF_P, OFF_R, OFF_D, OFF_QG, OFF_OI, OFF_V = 0, 32768, 49152, 49664, 66048, 82432
REC = OFF_V + 128 * 64 * 2


def _kmajor_decode(raw: np.ndarray, R: int, K: int) -> np.ndarray:
    """Inverse of byte(row, k) = (k/8)(R*16) + (row/8)128 + (row%8)16 + (k%8)2."""
    h = raw.view(np.float16).astype(np.float64)
    rows = np.arange(R)[:, None]
    ks = np.arange(K)[None, :]
    idx = ((ks // 8) * (R * 16) + (rows // 8) * 128 + (rows % 8) * 16 + (ks % 8) * 2) // 2
    return h[idx]


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _err(a, b):
    """Relative Frobenius error with an absolute floor of 1e-6 per element:
    fp16 records flush entries below its subnormal range (6e-8) to zero, and
    under strong decay a whole operand can sit there."""
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-6 * np.sqrt(b.size)))


@pytest.mark.parametrize("T,lb", [(130, -0.3), (64, -5.0), (130, -10.5)])
def test_prologue_records_match_chunk_form(T, lb):
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(1, T, 1, 2, seed=21, lower_bound=lb, init_state=False)
    xd = x.to("cuda")
    ws_bytes = kda.chunk_workspace_bytes(1, T, 2, 1)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    # cu_seqlens: the device-built chunk table (dense calls use closed-form tables)
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                      lower_bound=lb, cu_seqlens=cu, output_final_state=True, groups=1, workspace=ws)
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
            want_P = -kg.T @ w
            want_R = kg.T @ Tm
            want_qg = qg - Aqk @ w
            vv = pad(f(x.v[s:e, h]), (C, D))
            want_oi = Aqk @ Tm @ vv
            off = base + (c * 2 + h) * REC
            rec = raw[off:off + REC]
            got_P = _kmajor_decode(rec[OFF_P:OFF_R], 128, 128)
            got_R = _kmajor_decode(rec[OFF_R:OFF_D], 128, 64)
            got_d = rec[OFF_D:OFF_QG].view(np.float32).astype(np.float64)
            got_qg = _kmajor_decode(rec[OFF_QG:OFF_OI], 64, 128)
            oi_raw = rec[OFF_OI:OFF_V].view(np.uint16).astype(np.uint32) << 16
            oi_blocks = oi_raw.view(np.float32).astype(np.float64).reshape(4, 64, 4, 8)  # block, row, slot, 8 cols
            # row r's 16-byte chunk j (value columns 8 j ..) sits at slot (j + r // 2) % 4
            rows = np.arange(64)[:, None]
            slots = (np.arange(4)[None, :] + rows // 2) % 4
            got_oi = np.concatenate([oi_blocks[jb][rows, slots].reshape(64, 32) for jb in range(4)], axis=1)
            tag = f"T={T} head {h} chunk {c} (len {L})"
            assert _rel(got_d, ops["d"]) < 1e-4, f"d {tag}"
            assert _err(got_R, want_R) < 5e-3, f"R {tag}: {_err(got_R, want_R)}"
            assert _err(got_P, want_P) < 1e-2, f"P {tag}: {_err(got_P, want_P)}"
            assert _err(got_qg, want_qg) < 1e-2, f"qg' {tag}: {_err(got_qg, want_qg)}"
            assert _err(got_oi, want_oi) < 1e-2, f"o_intra {tag}: {_err(got_oi, want_oi)}"
            # v^T, fp16 [128 value columns][64 rows]: bf16 v converted to fp16,
            # exact except below fp16's normal range (absolute 3e-8)
            got_v = _kmajor_decode(rec[OFF_V:REC], 128, 64)
            np.testing.assert_allclose(got_v, vv.T, rtol=0, atol=3e-8, err_msg=f"v^T {tag}")
