"""GPU parity of mid-prefill state snapshots (kda_chunk_fwd_ex's
checkpoint_state / checkpoint_offsets / checkpoint_state_indices, the vLLM
kda_chunk page's fused_kda_chunk arguments) through the C ABI: each
snapshot equals the fp64 recurrence run on the sequence's first
checkpoint_offsets[n] tokens; rows whose snapshot is disabled or skipped
stay bit-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_fwd_gb300 import workloads as W
from tests.helpers import check_out, check_state

pytestmark = pytest.mark.gpu


def _prefix_state(x, n, o, h0):
    cu = x.cu_seqlens.tolist() if x.cu_seqlens is not None else None
    bos = cu[n] if cu is not None else n * (x.t_total // x.n_seqs)
    return oracle.recurrence(x.q[bos:bos + o], x.k[bos:bos + o], x.v[bos:bos + o], x.g[bos:bos + o],
                             x.beta[bos:bos + o], [0, o], A_log=x.A_log, dt_bias=x.dt_bias,
                             lower_bound=x.lower_bound, h0=h0[None])["state"][0]


def _initial(x, n):
    idx = int(x.state_indices[n])
    if idx < 0 or not bool(x.has_initial_state[n]):
        return np.zeros((x.hv, 128, 128))
    return x.state_pool[idx].double().numpy()


@pytest.mark.parametrize("groups", [1, 4])
def test_checkpoint_staging_buffer(groups):
    """Staging rows by sequence: valid offsets snapshot; 0, a misaligned
    offset and one past the sequence's end leave their rows untouched."""
    import linear_attention_serving_fwd_gb300 as kda
    lens = [200, 64, 130, 517, 256, 640]
    offs = [128, 64, 0, 512, 100, 704]  # 0 disabled, 100 misaligned, 704 > 640
    x = W.varlen_paged(lens, 2, 4, slots=16, seed=41, lower_bound=-0.7)
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    sentinel = torch.full((len(lens), x.hv, 128, 128), 7.0, dtype=torch.float32, device="cuda")
    ck = sentinel.clone()
    out, _ = kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                               lower_bound=x.lower_bound, cu_seqlens=xd.cu_seqlens, state_cache=pool,
                               state_indices=xd.state_indices, has_initial_state=xd.has_initial_state,
                               groups=groups, checkpoint_state=ck,
                               checkpoint_offsets=torch.tensor(offs, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    ref = oracle.prefill(x)
    check_out(out, ref["out"], "out with checkpoints")
    for n, o in enumerate(offs):
        if o > 0 and o % 64 == 0 and o <= lens[n]:
            check_state(ck[n:n + 1], _prefix_state(x, n, o, _initial(x, n))[None], f"snapshot {n} at {o}")
        else:
            assert torch.equal(ck[n], sentinel[n]), f"sequence {n}: skipped snapshot wrote its row"


def test_checkpoint_into_state_cache():
    """Snapshots written into spare rows of the paged cache the prefill also
    updates in place; a negative row disables, and an offset equal to the
    length gives the final state."""
    import linear_attention_serving_fwd_gb300 as kda
    lens = [192, 256, 128]
    x = W.varlen_paged(lens, 1, 2, slots=12, seed=43, lower_bound=-0.9)
    live = set(x.state_indices.tolist())
    spare = [s for s in range(12) if s not in live]
    ck_rows = [spare[0], -1, spare[1]]
    offs = [64, 128, 128]
    xd = x.to("cuda")
    pool = xd.state_pool.clone()
    kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                      lower_bound=x.lower_bound, cu_seqlens=xd.cu_seqlens, state_cache=pool,
                      state_indices=xd.state_indices, has_initial_state=xd.has_initial_state, groups=1,
                      checkpoint_state=pool, checkpoint_offsets=torch.tensor(offs, dtype=torch.int32,
                                                                           device="cuda"),
                      checkpoint_state_indices=torch.tensor(ck_rows, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 0
    ref = oracle.prefill(x)
    got = pool.cpu()
    check_state(got[[spare[0]]], _prefix_state(x, 0, 64, _initial(x, 0))[None], "snapshot of sequence 0")
    final2 = ref["pool"][int(x.state_indices[2])]
    check_state(got[[spare[1]]], final2[None], "snapshot at the end of sequence 2")
    others = [s for s in range(12) if s not in live and s not in (spare[0], spare[1])]
    assert torch.equal(got[others], x.state_pool[others]), "rows outside the call changed"
    for n in range(3):
        s = int(x.state_indices[n])
        check_state(got[[s]], ref["pool"][s][None], f"final state of sequence {n}")


def test_checkpoint_bad_row_is_reported():
    import linear_attention_serving_fwd_gb300 as kda
    x = W.dense_prefill(2, 128, 1, 1, seed=45)
    xd = x.to("cuda")
    ck = torch.zeros((2, 1, 128, 128), dtype=torch.float32, device="cuda")
    kda.kda_chunk_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, A_log=xd.A_log, dt_bias=xd.dt_bias,
                      lower_bound=x.lower_bound, n_seqs=2, initial_state=xd.initial_state, groups=1,
                      checkpoint_state=ck,
                      checkpoint_offsets=torch.tensor([64, 64], dtype=torch.int32, device="cuda"),
                      checkpoint_state_indices=torch.tensor([0, 5], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert kda.kda_device_status(clear=True) == 5  # KDA_ERR_DEVICE_INDEX
    S = _prefix_state(x, 0, 64, x.initial_state[0].double().numpy())
    check_state(ck[0:1], S[None], "snapshot of sequence 0")
    assert torch.count_nonzero(ck[1]) == 0
