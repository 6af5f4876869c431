"""Pins for the conv + SiLU oracle (oracle/conv.py): closed forms, tap
order, a library convolution, the bf16-product rounding the verify page
prescribes, and the rolled state across split prefills and verify steps.
CPU only."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import conv

C = 6


def _bf(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).float().numpy()


def _rand(L, seed=0):
    g = np.random.default_rng(seed)
    return _bf(g.standard_normal((L, C))), _bf(g.standard_normal((3, C)))


def test_silu_limits():
    """SiLU(0) = 0, SiLU(x) = x for large x (the logistic is 1 in fp32),
    SiLU(-x) tiny and negative, and SiLU(x) - SiLU(-x) = x."""
    y = conv.silu_bf16(np.array([0.0, 64.0, -64.0, 1.5, -1.5], np.float32))
    assert y[0] == 0.0 and y[1] == 64.0
    assert -1e-20 < y[2] < 0.0
    assert abs((y[3] - y[4]) - 1.5) <= 1.5 * 2 ** -7


@pytest.mark.parametrize("taps", ["bf16", "f32"])
def test_current_tap_is_pointwise(taps):
    """Taps (0, 0, 0, 1): y_t = SiLU(x_t), whatever the history."""
    x, h = _rand(9, 1)
    w = np.tile(np.array([0.0, 0.0, 0.0, 1.0], np.float32), (C, 1))
    np.testing.assert_array_equal(conv.conv_silu(x, w, h, taps), conv.silu_bf16(x))


def test_oldest_tap_reads_history_then_inputs():
    """Taps (1, 0, 0, 0): y_t = SiLU(win_t), the input three steps back."""
    x, h = _rand(7, 2)
    w = np.tile(np.array([1.0, 0.0, 0.0, 0.0], np.float32), (C, 1))
    want = conv.silu_bf16(np.concatenate([h, x])[:7])
    np.testing.assert_array_equal(conv.conv_silu(x, w, h, "f32"), want)


def test_matches_library_convolution():
    """fp32 taps: per channel, the sum is numpy's full convolution of the
    history-extended input with the reversed taps (a correlation)."""
    x, h = _rand(20, 3)
    w = np.random.default_rng(4).uniform(-0.5, 0.5, (C, 4)).astype(np.float32)
    got = conv.preact(x, w, h, "f32")
    win = np.concatenate([h, x]).astype(np.float64)
    for c in range(C):
        ref = np.convolve(win[:, c], w[c, ::-1].astype(np.float64), mode="valid")
        np.testing.assert_allclose(got[:, c], ref, rtol=3e-7, atol=1e-7)


def test_bf16_taps_round_each_product():
    """x = w = 1 + 2^-7: the exact product 1 + 2^-6 + 2^-14 rounds to
    1 + 2^-6 in bf16, so four taps sum to 4.0625 exactly; fp32 taps keep
    the 2^-14 terms."""
    v = 1.0 + 2.0 ** -7
    x = np.full((1, C), v, np.float32)
    h = np.full((3, C), v, np.float32)
    w = np.full((C, 4), v, np.float32)
    assert np.all(conv.preact(x, w, h, "bf16") == np.float32(4.0625))
    assert np.all(conv.preact(x, w, h, "f32") == np.float32(4.0625 + 4 * 2.0 ** -14))


def test_prefill_split_carries_the_rolled_state():
    """A sequence run in two prefills (the state carried between them)
    equals one prefill; a sequence shorter than the history keeps the tail
    of its history in front of its inputs."""
    hqk, hv = 1, 2
    g = torch.Generator().manual_seed(5)
    T = 11
    q, k = (torch.randn(T, hqk, 128, generator=g).bfloat16().float() for _ in range(2))
    v = torch.randn(T, hv, 128, generator=g).bfloat16().float()
    Cn = (2 * hqk + hv) * 128
    w = torch.rand(Cn, 4, generator=g) - 0.5
    st = torch.randn(2, 5, Cn, generator=g).bfloat16().float().numpy()
    (q1, k1, v1), s1 = conv.prefill(q, k, v, [0, T], w, "f32", st, [1])
    (qa, ka, va), sa = conv.prefill(q[:6], k[:6], v[:6], [0, 6], w, "f32", st, [1])
    (qb, kb, vb), sb = conv.prefill(q[6:], k[6:], v[6:], [0, T - 6], w, "f32", sa, [1])
    for one, two in ((q1, torch.cat([qa, qb])), (k1, torch.cat([ka, kb])), (v1, torch.cat([va, vb]))):
        assert torch.equal(one, two)
    np.testing.assert_array_equal(s1, sb)
    np.testing.assert_array_equal(s1[0], st[0])
    x = conv.channels(q, k, v)
    np.testing.assert_array_equal(s1[1, :3], x[T - 3:])
    np.testing.assert_array_equal(s1[1, 3:], st[1, 3:])
    (_, _, _), s2 = conv.prefill(q[:2], k[:2], v[:2], [0, 2], w, "f32", st, [0])
    np.testing.assert_array_equal(s2[0, :3], np.concatenate([st[0, 2:3], x[:2]]))
    # no initial state: zero history
    (q0, _, _), _ = conv.prefill(q[:1], k[:1], v[:1], [0, 1], w, "f32", st, [0], [False])
    wq = w[:128].numpy()
    want = conv.silu_bf16(q[0, 0].numpy() * wq[:, 3])
    np.testing.assert_array_equal(q0[0, 0].numpy(), want)


def test_verify_history_follows_accepted_tokens():
    """Two verify steps: the second one's history is the inputs at the
    end of the tokens accepted in the first, so its outputs equal the conv
    over the stream of accepted inputs followed by the new window."""
    hqk = hv = 1
    g = torch.Generator().manual_seed(6)
    Cn = 3 * 128
    w = (torch.rand(Cn, 4, generator=g) - 0.5).bfloat16().float()
    st = torch.randn(1, 6, Cn, generator=g).bfloat16().float().numpy()
    mk = lambda n: [torch.randn(n, h, 128, generator=g).bfloat16().float() for h in (hqk, hqk, hv)]
    x1, x2 = mk(4), mk(4)
    one = torch.tensor([1], dtype=torch.int32)
    (_, _, _), s1 = conv.verify(*x1, torch.tensor([0, 4]), w, "bf16", st, torch.tensor([0]), one)
    for a in (1, 2, 3, 4):
        (q2, k2, v2), _ = conv.verify(*x2, torch.tensor([0, 4]), w, "bf16", s1, torch.tensor([0]),
                                      torch.tensor([a]))
        stream = np.concatenate([st[0, :3], conv.channels(*x1)[:a], conv.channels(*x2)])
        want = conv.conv_silu(stream[3:], w, stream[:3], "bf16")[a:]
        got = conv.channels(q2, k2, v2)
        np.testing.assert_array_equal(got, want)
