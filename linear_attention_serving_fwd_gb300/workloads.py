"""Seeded synthetic inputs for the KDA forward path.

This module only draws random numbers and arranges them into the layouts the
kernels and the CPU oracle both consume.  It holds none of the method's
arithmetic (no gate, no norm, no recurrence), so both sides can share it.

Draw order for every workload is fixed: q, k, v, g, beta, A_log, dt_bias,
state, lengths, slots.  Draws are fp32 from one seeded generator and are cast
to bf16 afterwards (activations may be cast to fp16 and states to bf16
instead, ``act_dtype`` / ``state_dtype``, from the same draws).  "N(0, s)"
means standard deviation s.

Workloads (the shapes and distributions of the chunk_kda / decode pages'
intended serving traffic):

* ``tiny``     B=1, T=256, Hqk=Hv=1, no initial state, final state returned.
* ``dense``    B=2, T=4096, Hqk=Hv=16, initial state N(0, 0.02).
* ``varlen``   8 sequences, lengths U[64, 8192] rescaled to sum 32768,
               Hqk=8, Hv=32, paged fp32 cache [64 slots], 8 slots permuted.
* ``long``     B=1, T=131072, Hqk=Hv=32, zero initial state.
* ``decode``   256 requests x window Q in {1, 4}, H=32, pool of 512 slots,
               256 slots drawn without replacement.

q, k, v, g and the beta logits are N(0, 1); A_log = log(U[1, 16]) per head,
dt_bias ~ N(0, 0.1) per head and channel, lower_bound = -5, scale = 128^-0.5.

Without gate parameters (``log_decay=(lo, hi)``) g is drawn U[lo, hi] in its
place in the draw order and used as the per-channel log decay itself; A_log
and dt_bias are still drawn (the order stays fixed) and then dropped.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

D = 128  # head dimension (K = V = 128)
CHUNK = 64


@dataclasses.dataclass
class KdaInputs:
    """One batch of inputs in the flattened token-major layout.

    q, k: [T_tot, Hqk, 128] bf16.  v, g: [T_tot, Hv, 128] bf16.
    beta: [T_tot, Hv] bf16 (logits).  A_log: [Hv] fp32.  dt_bias: [Hv, 128] fp32.
    cu_seqlens: [N+1] int32 (token offsets of each sequence / request).
    initial_state: [N, Hv, 128, 128] fp32 (V-first, K contiguous) or None.
    state_pool: [slots, Hv, 128, 128] fp32 or None, with state_indices [N] int32.
    """

    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    A_log: Optional[torch.Tensor]
    dt_bias: Optional[torch.Tensor]
    cu_seqlens: torch.Tensor
    B: int  # dense batch (0 for varlen / paged)
    T: int  # dense sequence length (0 for varlen / paged)
    scale: float = D ** -0.5
    lower_bound: float = -5.0
    initial_state: Optional[torch.Tensor] = None
    state_pool: Optional[torch.Tensor] = None
    state_indices: Optional[torch.Tensor] = None
    has_initial_state: Optional[torch.Tensor] = None
    window: int = 0  # decode window Q (0 for prefill)
    output_final_state: bool = True

    @property
    def n_seqs(self) -> int:
        return int(self.cu_seqlens.numel() - 1)

    @property
    def t_total(self) -> int:
        return int(self.q.shape[0])

    @property
    def hqk(self) -> int:
        return int(self.q.shape[1])

    @property
    def hv(self) -> int:
        return int(self.v.shape[1])

    def seq_lens(self) -> list:
        cu = self.cu_seqlens.cpu().tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    def to(self, device) -> "KdaInputs":
        out = dataclasses.replace(self)
        for f in dataclasses.fields(self):
            val = getattr(self, f.name)
            if isinstance(val, torch.Tensor):
                setattr(out, f.name, val.to(device))
        return out


def _gen(seed: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return gen


def _normal(gen, shape, std, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def _uniform(gen, shape, lo, hi, device):
    return torch.rand(shape, generator=gen, device=device, dtype=torch.float32) * (hi - lo) + lo


def _draw_activations(gen, t_total, hqk, hv, device, g_std=1.0, g_shift=0.0, dtype=torch.bfloat16,
                      log_decay=None):
    bf = dtype  # activation storage: bf16 (default) or fp16, from the same fp32 draws
    q = _normal(gen, (t_total, hqk, D), 1.0, device).to(bf)
    k = _normal(gen, (t_total, hqk, D), 1.0, device).to(bf)
    v = _normal(gen, (t_total, hv, D), 1.0, device).to(bf)
    if log_decay is None:
        g = (_normal(gen, (t_total, hv, D), g_std, device) + g_shift).to(bf)
    else:
        g = _uniform(gen, (t_total, hv, D), log_decay[0], log_decay[1], device).to(bf)
    beta = _normal(gen, (t_total, hv), 1.0, device).to(bf)
    A_log = torch.log(_uniform(gen, (hv,), 1.0, 16.0, device))
    dt_bias = _normal(gen, (hv, D), 0.1, device)
    if log_decay is not None:  # no gate parameters: g is the log decay
        A_log = dt_bias = None
    return q, k, v, g, beta, A_log, dt_bias


def dense_prefill(B: int, T: int, hqk: int, hv: int, *, seed: int = 0, device="cpu",
                  init_state: bool = True, state_std: float = 0.02,
                  lower_bound: float = -5.0, g_shift: float = 0.0,
                  scale: float = D ** -0.5, name: str = "dense",
                  act_dtype=torch.bfloat16, state_dtype=torch.float32,
                  log_decay=None) -> KdaInputs:
    """Dense [B, T] prefill flattened to T_tot = B*T tokens."""
    gen = _gen(seed, device)
    q, k, v, g, beta, A_log, dt_bias = _draw_activations(gen, B * T, hqk, hv, device,
                                                         g_shift=g_shift, dtype=act_dtype,
                                                         log_decay=log_decay)
    h0 = _normal(gen, (B, hv, D, D), state_std, device).to(state_dtype) if init_state else None
    cu = torch.arange(0, B + 1, dtype=torch.int32, device=device) * T
    return KdaInputs(name=name, q=q, k=k, v=v, g=g, beta=beta, A_log=A_log,
                     dt_bias=dt_bias, cu_seqlens=cu, B=B, T=T, scale=scale,
                     lower_bound=lower_bound, initial_state=h0)


def rescaled_lengths(gen, n: int, total: int, lo: float, hi: float, device) -> list:
    """n lengths drawn U[lo, hi], rescaled to sum to ``total``; the last one
    takes the remainder."""
    x = _uniform(gen, (n,), lo, hi, device).cpu().double().tolist()
    s = sum(x)
    lens = [int(round(xi * total / s)) for xi in x[:-1]]
    lens.append(total - sum(lens))
    return lens


def varlen_paged(lens_or_n, hqk: int, hv: int, *, total: Optional[int] = None,
                 slots: int = 64, seed: int = 0, device="cpu",
                 lower_bound: float = -5.0, g_shift: float = 0.0,
                 state_std: float = 0.02, has_initial=None,
                 name: str = "varlen", act_dtype=torch.bfloat16,
                 state_dtype=torch.float32, log_decay=None) -> KdaInputs:
    """Varlen prefill on a paged state cache (fp32 unless ``state_dtype``).

    ``lens_or_n`` is either an explicit list of lengths or a sequence count,
    in which case lengths are drawn U[64, 8192] and rescaled to ``total``.
    Lengths are drawn after the activations, as the fixed draw order demands,
    so T_tot must be known first: with a count, ``total`` fixes it.
    """
    gen = _gen(seed, device)
    if isinstance(lens_or_n, int):
        assert total is not None
        n = lens_or_n
        t_total = total
    else:
        n = len(lens_or_n)
        t_total = int(sum(lens_or_n))
    q, k, v, g, beta, A_log, dt_bias = _draw_activations(gen, t_total, hqk, hv, device,
                                                         g_shift=g_shift, dtype=act_dtype,
                                                         log_decay=log_decay)
    pool = _normal(gen, (slots, hv, D, D), state_std, device).to(state_dtype)
    if isinstance(lens_or_n, int):
        lens = rescaled_lengths(gen, n, total, 64.0, 8192.0, device)
    else:
        lens = list(lens_or_n)
    idx = torch.randperm(slots, generator=gen, device=device)[:n].to(torch.int32)
    cu = torch.tensor([0] + list(_cumsum(lens)), dtype=torch.int32, device=device)
    if has_initial is None:
        hi = torch.ones(n, dtype=torch.uint8, device=device)
    else:
        hi = torch.tensor([1 if x else 0 for x in has_initial], dtype=torch.uint8, device=device)
    return KdaInputs(name=name, q=q, k=k, v=v, g=g, beta=beta, A_log=A_log,
                     dt_bias=dt_bias, cu_seqlens=cu, B=0, T=0,
                     lower_bound=lower_bound, state_pool=pool, state_indices=idx,
                     has_initial_state=hi, output_final_state=False)


def decode_batch(n_req: int, window: int, hqk: int, hv: int, *, slots: int = 512,
                 seed: int = 0, device="cpu", qlens=None, null_requests=(),
                 lower_bound: float = -5.0, g_shift: float = 0.0,
                 state_std: float = 0.02, name: str = "decode",
                 act_dtype=torch.bfloat16, state_dtype=torch.float32,
                 log_decay=None) -> KdaInputs:
    """Batched decode / verify: each request has ``window`` new tokens (or
    ``qlens[b]`` <= window), one state slot each, drawn without replacement.
    Requests listed in ``null_requests`` get slot -1 (a padding entry)."""
    gen = _gen(seed, device)
    if qlens is None:
        qlens = [window] * n_req
    assert all(0 <= x <= window for x in qlens)
    t_total = int(sum(qlens))
    q, k, v, g, beta, A_log, dt_bias = _draw_activations(gen, t_total, hqk, hv, device,
                                                         g_shift=g_shift, dtype=act_dtype,
                                                         log_decay=log_decay)
    pool = _normal(gen, (slots, hv, D, D), state_std, device).to(state_dtype)
    idx = torch.randperm(slots, generator=gen, device=device)[:n_req].to(torch.int32)
    for b in null_requests:
        idx[b] = -1
    cu = torch.tensor([0] + list(_cumsum(qlens)), dtype=torch.int32, device=device)
    return KdaInputs(name=name, q=q, k=k, v=v, g=g, beta=beta, A_log=A_log,
                     dt_bias=dt_bias, cu_seqlens=cu, B=0, T=0,
                     lower_bound=lower_bound, state_pool=pool, state_indices=idx,
                     window=window, output_final_state=False)


def decode_slot_table(n_req: int, steps: int, slots: int, *, seed: int = 0, device="cpu"):
    """A [n_req, steps] int32 slot table of distinct pool rows (a row per
    request and decode step, as speculative decode keeps them) drawn from
    randperm(slots), and per-request accepted-token counts U{1..steps}."""
    assert n_req * steps <= slots
    gen = _gen(seed + 7919, device)
    rows = torch.randperm(slots, generator=gen, device=device)[:n_req * steps]
    table = rows.to(torch.int32).view(n_req, steps).contiguous()
    acc = torch.randint(1, steps + 1, (n_req,), generator=gen, device=device, dtype=torch.int32)
    return table, acc


def conv_inputs(hqk: int, hv: int, rows: int, positions: int, *, taps: str = "bf16",
                seed: int = 0, device="cpu"):
    """Width-4 depthwise conv parameters and state for the raw q/k/v
    projection bands (C = (2 Hqk + Hv) * 128 channels): weight [C, 4] drawn
    U(-1/2, 1/2) (the default init of a conv1d with fan-in 4), bf16 or fp32,
    and a bf16 conv state [rows, positions, C] (token major) of N(0, 1)
    values, the scale of the projection outputs it holds."""
    gen = _gen(seed + 104729, device)
    C = (2 * hqk + hv) * D
    w = _uniform(gen, (C, 4), -0.5, 0.5, device)
    w = w.to(torch.bfloat16) if taps == "bf16" else w
    st = _normal(gen, (rows, positions, C), 1.0, device).to(torch.bfloat16)
    return w, st


def _cumsum(xs):
    s = 0
    for x in xs:
        s += x
        yield s


# The five serving workloads, by name.  Each returns a KdaInputs.
def workload(name: str, *, seed: int = 0, device="cpu", window: int = 1) -> KdaInputs:
    if name == "tiny":
        x = dense_prefill(1, 256, 1, 1, seed=seed, device=device, init_state=False, name=name)
        return x
    if name == "dense":
        return dense_prefill(2, 4096, 16, 16, seed=seed, device=device, name=name)
    if name == "varlen":
        return varlen_paged(8, 8, 32, total=32768, slots=64, seed=seed, device=device,
                            name=name)
    if name == "long":
        return dense_prefill(1, 131072, 32, 32, seed=seed, device=device, init_state=False,
                             name=name)
    if name == "decode":
        return decode_batch(256, window, 32, 32, slots=512, seed=seed, device=device,
                            name=f"decode_q{window}")
    raise KeyError(name)


WORKLOADS = ("tiny", "dense", "varlen", "long", "decode")


def flop_per_token_head(chunk: int = CHUNK) -> int:
    """Algorithmic prefill flop per (token, v-head): three 64x128x128
    contractions of the inter-chunk walk (6*K*V) plus five C x C x 128
    intra-chunk products (10*C*K), full tiles."""
    return 6 * D * D + 10 * chunk * D


def prefill_bytes_per_token_head(hqk: int, hv: int) -> float:
    """Algorithmic HBM bytes per (token, v-head) of one prefill pass: q and k
    shared by Hv/Hqk v-heads, v and g read, beta read, o written (all bf16)."""
    r = hv // hqk
    return 2 * 256 / r + 512 + 2 + 256


def state_bytes() -> int:
    return D * D * 4


def _self_check():  # pragma: no cover - manual aid
    x = workload("tiny")
    assert x.q.shape == (256, 1, 128)
    assert math.isclose(x.scale, 128 ** -0.5)
