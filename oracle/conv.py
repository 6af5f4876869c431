"""Width-4 depthwise causal convolution + SiLU with a rolled conv state.
TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows the conv path of ``KdaTcVerify`` on the vLLM kimi_k3 CuTeDSL verify
page (step 2, "Activations", with ``conv``) and the conv arguments of
``fused_kda_prologue`` on the vLLM kimi_k3 AMD ``kda_chunk`` page
(``conv_weight``, ``conv_state``, ``conv_state_indices``,
``conv_has_initial_state``: q/k/v are then the raw bands of the QKV
projection and the conv state is updated in place).

Channels: the projection's bands are numbered q (Hqk*128 channels), then k
(Hqk*128), then v (Hv*128); channel = band offset + head * 128 + c.

Per channel, with the three history inputs h_0, h_1, h_2 (oldest first)
followed by the raw inputs x_0, x_1, ...:
    win   = [h_0, h_1, h_2, x_0, x_1, ...]
    acc_t = sum_{j=0..3} w_j * win_{t+j}        (w_3 multiplies x_t)
    y_t   = bf16( acc_t / (1 + exp(-acc_t)) )   (SiLU, rounded to bf16)
in the page's precision: with bf16 taps every product is rounded to bf16
and the four are added in fp32 in tap order; with fp32 taps the sum is an
fp32 fused multiply-add chain in tap order.  SiLU itself is evaluated here
in fp64 from the fp32 sum, so a result may sit one bf16 step from a kernel
that evaluates it in fp32 (a rounding boundary between the two).

Conv state rows are [positions, C] (token major).  Prefill reads its history
from positions 0..2 and leaves the last three raw inputs of the sequence
there.  Verify reads positions a-1 .. a+1 (a = accepted tokens of the
previous step) and writes the rolled state: positions 0, 1 = the last two
history inputs, position 2 + t = raw input t of the window.
"""
from __future__ import annotations

import numpy as np
import torch

D = 128
WIDTH = 4
HIST = WIDTH - 1


def to_bf16(a) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), returned as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _np(t) -> np.ndarray:
    if hasattr(t, "detach"):
        return t.detach().to("cpu", torch.float32).numpy()
    return np.asarray(t, dtype=np.float32)


def preact(x, w, hist, taps: str) -> np.ndarray:
    """The fp32 sums acc_t [L, C] of raw inputs x [L, C] with taps w [C, 4]
    after history hist [3, C]; ``taps`` is "bf16" or "f32" (the taps'
    storage type, which fixes the summation precision)."""
    x = _np(x)
    w = _np(w)
    hist = _np(hist)
    L, C = x.shape
    assert w.shape == (C, WIDTH) and hist.shape == (HIST, C)
    win = np.concatenate([hist, x], axis=0).astype(np.float64)
    acc = np.zeros((L, C), dtype=np.float32)
    for j in range(WIDTH):
        prod = win[j:j + L] * w[None, :, j].astype(np.float64)  # exact in fp64
        if taps == "bf16":
            acc = (acc + to_bf16(prod)).astype(np.float32)
        elif taps == "f32":
            acc = (acc.astype(np.float64) + prod).astype(np.float32)  # one rounding: an fma
        else:
            raise ValueError(taps)
    return acc


def silu_bf16(acc) -> np.ndarray:
    a = np.asarray(acc, dtype=np.float64)
    return to_bf16(a / (1.0 + np.exp(-a)))


def conv_silu(x, w, hist, taps: str) -> np.ndarray:
    """y [L, C] (bf16 values as float32) for raw inputs x after history hist."""
    return silu_bf16(preact(x, w, hist, taps))


def channels(q, k, v) -> np.ndarray:
    """[T, C] raw projection rows from the q [T,Hqk,128], k, v [T,Hv,128] bands."""
    T = q.shape[0]
    return np.concatenate([_np(q).reshape(T, -1), _np(k).reshape(T, -1), _np(v).reshape(T, -1)],
                          axis=1)


def bands(y, hqk, hv):
    T = y.shape[0]
    a, b = hqk * D, 2 * hqk * D
    return (torch.from_numpy(np.ascontiguousarray(y[:, :a].reshape(T, hqk, D))),
            torch.from_numpy(np.ascontiguousarray(y[:, a:b].reshape(T, hqk, D))),
            torch.from_numpy(np.ascontiguousarray(y[:, b:].reshape(T, hv, D))))


def prefill(q, k, v, cu_seqlens, weight, taps, state, indices, has_initial_state=None):
    """Conv + SiLU over every sequence of a varlen batch.

    state: [rows, positions >= 3, C] (token major); sequence n reads its
    history from row indices[n] (zero history when has_initial_state[n] is
    false or indices[n] < 0) and that row ends holding the sequence's last
    three raw inputs at positions 0..2 (a shorter sequence keeps the tail of
    its history in front of them).  Returns (q', k', v') as torch float32
    bands and the updated state (numpy float32).
    """
    hqk, hv = q.shape[1], v.shape[1]
    x = channels(q, k, v)
    st = _np(state).copy()
    cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    idx = [int(i) for i in (indices.tolist() if hasattr(indices, "tolist") else indices)]
    hi = None if has_initial_state is None else [bool(b) for b in np.asarray(_np(has_initial_state))]
    y = np.zeros_like(x)
    for n in range(len(cu) - 1):
        a, e = cu[n], cu[n + 1]
        r = idx[n]
        hist = np.zeros((HIST, x.shape[1]), np.float32)
        if r >= 0 and (hi is None or hi[n]):
            hist = st[r, :HIST].copy()
        y[a:e] = conv_silu(x[a:e], weight, hist, taps)
        if r >= 0:
            st[r, :HIST] = np.concatenate([hist, x[a:e]], axis=0)[-HIST:]
    return bands(y, hqk, hv), st


def verify(q, k, v, cu_seqlens, weight, taps, state, slots, accepted):
    """Conv + SiLU of each request's window after the history at positions
    accepted[b]-1 .. accepted[b]+1 of row slots[b], and the rolled state
    (positions 0, 1 = the history's last two inputs, 2 + t = raw input t).
    Requests with a negative slot are skipped (zero outputs, row untouched).
    Returns (q', k', v') as torch float32 bands and the updated state."""
    hqk, hv = q.shape[1], v.shape[1]
    x = channels(q, k, v)
    st = _np(state).copy()
    cu = [int(c) for c in cu_seqlens.tolist()]
    sl = [int(s) for s in slots.tolist()]
    acc = [int(a) for a in accepted.tolist()]
    y = np.zeros_like(x)
    for b in range(len(cu) - 1):
        a, e = cu[b], cu[b + 1]
        if sl[b] < 0 or e == a:
            continue
        first = acc[b] - 1
        hist = st[sl[b], first:first + HIST].copy()
        y[a:e] = conv_silu(x[a:e], weight, hist, taps)
        st[sl[b], 0:2] = hist[1:]
        st[sl[b], 2:2 + (e - a)] = x[a:e]
    return bands(y, hqk, hv), st
