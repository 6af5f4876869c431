"""The C ABI without a GPU: the library builds, loads, exports every function
include/kda.h declares, and its host-side validation rejects each broken
argument rule (the MATE chunk_kda / gated_delta_rule_decode checks and the
fused_kda_chunk state-cache rules) with the documented status code, before
touching the device.  Pointers here are fake, aligned addresses that are
never dereferenced: validation fails first."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from linear_attention_serving_fwd_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INVALID, DTYPE, CUDA = 1, 2, 3
FAKE = 0x10000  # aligned, never dereferenced


def _header_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    lib = _native.lib()
    declared = _header_functions()
    assert set(declared) == set(_native.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.kda_version().decode().startswith("kda-gb300")


def _acts(**over):
    a = _native.KdaActivations()
    for name in ("q", "k", "v", "g", "beta"):
        setattr(a, name, FAKE)
    a.q_stride_tok = a.k_stride_tok = 2 * 128
    a.q_stride_head = a.k_stride_head = 128
    a.v_stride_tok = a.g_stride_tok = 4 * 128
    a.v_stride_head = a.g_stride_head = 128
    a.beta_stride_tok, a.beta_stride_head = 4, 1
    a.A_log, a.dt_bias = FAKE, FAKE
    a.dtype, a.t_total, a.hqk, a.hv = 0, 64, 2, 4
    a.use_qk_l2norm, a.scale, a.lower_bound = 1, 128 ** -0.5, -5.0
    for k, v in over.items():
        setattr(a, k, v)
    return a


def _chunk(a, **kw):
    lib = _native.lib()
    args = dict(out=FAKE, cu=None, n=1, h0=None, hT=None, cache=None, stride=0, slots=0,
                idx=None, hi=None, groups=1, ws=FAKE, ws_bytes=1 << 40, stream=None)
    args.update(kw)
    return lib.kda_chunk_fwd(ctypes.byref(a), args["out"], args["cu"], args["n"], args["h0"],
                             args["hT"], args["cache"], args["stride"], args["slots"],
                             args["idx"], args["hi"], args["groups"], args["ws"],
                             args["ws_bytes"], args["stream"])


def _msg():
    return _native.lib().kda_last_error().decode()


@pytest.mark.parametrize("over,code,text", [
    (dict(dtype=7), DTYPE, "bfloat16 or float16"),
    (dict(state_bf16=2), INVALID, "state_bf16"),
    (dict(hv=3), INVALID, "GVA requires"),
    (dict(hqk=0), INVALID, "positive"),
    (dict(A_log=None), INVALID, "provided together"),
    (dict(use_qk_l2norm=0), INVALID, "L2 norm"),
    (dict(lower_bound=-12.0), INVALID, "lower_bound"),
    (dict(q=FAKE + 2), INVALID, "16-byte aligned"),
    (dict(v_stride_tok=4 * 128 + 1), INVALID, "multiples of 8"),
    (dict(k=None), INVALID, "must not be NULL"),
    (dict(t_total=-1), INVALID, "t_total"),
])
def test_chunk_validation(over, code, text):
    assert _chunk(_acts(**over)) == code
    assert text in _msg()


def test_chunk_rules_on_states_and_workspace():
    a = _acts()
    assert _chunk(a, cache=FAKE, h0=FAKE, idx=FAKE, stride=4 * 16384, slots=3) == INVALID
    assert "replaces initial_state" in _msg()
    assert _chunk(a, cache=FAKE, stride=4 * 16384, slots=3) == INVALID
    assert "needs state_indices" in _msg()
    assert _chunk(a, cache=FAKE, idx=FAKE, stride=4 * 16384 + 2, slots=3) == INVALID
    assert "slot_stride" in _msg()
    # bf16 states: 16-byte rows need strides in multiples of 8 elements
    assert _chunk(_acts(state_bf16=1), cache=FAKE, idx=FAKE, stride=4 * 16384 + 4, slots=3) == INVALID
    assert "multiple of 8" in _msg()
    assert _chunk(a, cache=FAKE, idx=FAKE, stride=4 * 16384, slots=0) == INVALID
    assert "at least one slot" in _msg()
    assert _chunk(a, ws_bytes=16) == INVALID
    assert "workspace needs" in _msg()
    assert _chunk(a, n=0) == INVALID
    assert _chunk(_acts(t_total=65), n=2) == INVALID
    assert "divisible" in _msg()


def _chunk_ex(a, **kw):
    lib = _native.lib()
    args = dict(out=FAKE, cu=None, n=1, h0=None, hT=None, cache=None, stride=0, slots=0,
                idx=None, hi=None, ck=None, ck_stride=0, ck_rows=0, ck_off=None, ck_idx=None,
                conv=None, groups=1, ws=FAKE, ws_bytes=1 << 40, stream=None)
    args.update(kw)
    return lib.kda_chunk_fwd_ex(ctypes.byref(a), args["out"], args["cu"], args["n"], args["h0"],
                                args["hT"], args["cache"], args["stride"], args["slots"],
                                args["idx"], args["hi"], args["ck"], args["ck_stride"],
                                args["ck_rows"], args["ck_off"], args["ck_idx"],
                                None if args["conv"] is None else ctypes.byref(args["conv"]),
                                args["groups"],
                                args["ws"], args["ws_bytes"], args["stream"])


def test_checkpoint_argument_rules():
    a = _acts()
    row = 4 * 16384
    assert _chunk_ex(a, ck=FAKE, ck_stride=row, ck_rows=1) == INVALID
    assert "needs checkpoint_offsets" in _msg()
    assert _chunk_ex(a, ck_off=FAKE) == INVALID
    assert "without checkpoint_state" in _msg()
    assert _chunk_ex(a, ck_idx=FAKE) == INVALID
    assert "without checkpoint_state" in _msg()
    assert _chunk_ex(_acts(t_total=128), n=2, ck=FAKE, ck_stride=row, ck_rows=1, ck_off=FAKE) == INVALID
    assert "row per sequence" in _msg()
    assert _chunk_ex(a, ck=FAKE, ck_stride=row + 2, ck_rows=1, ck_off=FAKE) == INVALID
    assert "checkpoint_row_stride" in _msg()
    assert _chunk_ex(a, ck=FAKE, ck_stride=row, ck_rows=0, ck_off=FAKE, ck_idx=FAKE) == INVALID
    assert "checkpoint_state must contain" in _msg()
    assert _chunk_ex(a, ck=FAKE + 4, ck_stride=row, ck_rows=1, ck_off=FAKE) == INVALID
    assert "checkpoint_state must be 16-byte aligned" in _msg()


def _conv_desc(**over):
    cv = _native.KdaConv()
    cv.weight, cv.weight_f32, cv.state = FAKE, 0, FAKE
    cv.row_stride, cv.pos_stride, cv.chan_stride = 10 * 1024, 1024, 1
    cv.rows, cv.positions = 4, 10
    cv.state_indices, cv.has_initial_state, cv.num_accepted = FAKE, None, FAKE
    for k, v in over.items():
        setattr(cv, k, v)
    return cv


def test_conv_argument_rules():
    a = _acts()
    assert _chunk_ex(a, conv=_conv_desc(weight=None)) == INVALID and "conv weight" in _msg()
    assert _chunk_ex(a, conv=_conv_desc(weight=FAKE + 8)) == INVALID and "16-byte" in _msg()
    assert _chunk_ex(a, conv=_conv_desc(weight_f32=2)) == INVALID and "weight_f32" in _msg()
    assert _chunk_ex(a, conv=_conv_desc(positions=2)) == INVALID and "at least 3 positions" in _msg()
    assert _chunk_ex(a, conv=_conv_desc(state_indices=None)) == INVALID and "state_indices" in _msg()
    assert _chunk_ex(a, conv=_conv_desc(pos_stride=0)) == INVALID and "positive" in _msg()
    assert _chunk_ex(_acts(dtype=1), conv=_conv_desc()) == DTYPE and "bfloat16 activations" in _msg()
    lib = _native.lib()

    def verify(cv, win=4, slots=4):
        return lib.kda_verify_ex(ctypes.byref(a), FAKE, FAKE, 4 * 16384, slots, FAKE, FAKE, 2, win,
                                 FAKE, FAKE, FAKE, ctypes.byref(cv), None)
    assert verify(_conv_desc(positions=5)) == INVALID and "at least 6 positions" in _msg()
    assert verify(_conv_desc(num_accepted=None)) == INVALID and "num_accepted" in _msg()
    assert verify(_conv_desc(), slots=5) == INVALID and "row per state slot" in _msg()
    assert verify(_conv_desc(scratch=FAKE, scratch_bytes=1 << 30)) == INVALID and "no conv scratch" in _msg()
    # the optional prefill scratch: (2 Hqk + Hv) x 128 bf16 values a token
    need = lib.kda_conv_scratch_bytes(64, 2, 4)
    assert need == 64 * (2 * 2 + 4) * 128 * 2
    assert _chunk_ex(a, conv=_conv_desc(scratch=FAKE, scratch_bytes=need - 2)) == INVALID
    assert "conv scratch needs" in _msg()
    assert _chunk_ex(a, conv=_conv_desc(scratch=FAKE + 8, scratch_bytes=need)) == INVALID
    assert "conv scratch must be 16-byte aligned" in _msg()
    assert lib.kda_conv_scratch_bytes(64, 0, 4) == 0


def test_workspace_query():
    lib = _native.lib()
    assert lib.kda_chunk_workspace_bytes(0, 64, 4, 1) == 0
    one = lib.kda_chunk_workspace_bytes(2, 8192, 16, 1)
    four = lib.kda_chunk_workspace_bytes(2, 8192, 16, 4)
    assert one > 0 and four > one
    # three 64 KB planes per (sequence, head, group) for the group scan
    assert four - one == 3 * 2 * 16 * 4 * 128 * 128 * 4


def _window(a, verify=False, **kw):
    lib = _native.lib()
    args = dict(out=FAKE, pool=FAKE, stride=4 * 16384, slots=8, qs=FAKE, sl=FAKE, n=2, win=1,
                corr=FAKE, kg=FAKE, ctr=FAKE, stream=None)
    args.update(kw)
    if verify:
        return lib.kda_verify(ctypes.byref(a), args["out"], args["pool"], args["stride"],
                              args["slots"], args["qs"], args["sl"], args["n"], args["win"],
                              args["corr"], args["kg"], args["ctr"], args["stream"])
    return lib.kda_decode(ctypes.byref(a), args["out"], args["pool"], args["stride"],
                          args["slots"], args["qs"], args["sl"], args["n"], args["win"],
                          args["stream"])


@pytest.mark.parametrize("verify", [False, True])
def test_window_validation(verify):
    a = _acts()
    assert _window(a, verify, win=0) == INVALID and "window" in _msg()
    assert _window(a, verify, win=9) == INVALID and "window" in _msg()
    assert _window(a, verify, pool=None) == INVALID and "state_pool" in _msg()
    assert _window(a, verify, slots=0) == INVALID and "at least one slot" in _msg()
    assert _window(a, verify, qs=None) == INVALID
    assert _window(a, verify, n=-1) == INVALID
    assert _window(a, verify, n=0) == 0  # nothing to do
    assert _window(_acts(hv=3), verify) == INVALID
    if verify:
        assert _window(a, True, ctr=None) == INVALID and "work_counter" in _msg()


def test_slot_table_decode_validation():
    lib = _native.lib()
    a = _acts()

    def steps(**kw):
        args = dict(out=FAKE, pool=FAKE, stride=4 * 16384, slots=8, qs=FAKE, tab=FAKE, ts=4,
                    acc=None, n=2, win=4)
        args.update(kw)
        return lib.kda_decode_steps(ctypes.byref(a), args["out"], args["pool"], args["stride"],
                                    args["slots"], args["qs"], args["tab"], args["ts"], args["acc"],
                                    args["n"], args["win"], None)
    assert steps(ts=3) == INVALID and "at least window" in _msg()
    assert steps(tab=None) == INVALID and "state_indices" in _msg()
    assert steps(qs=None) == INVALID
    assert steps(win=9, ts=9) == INVALID and "window" in _msg()
    assert steps(pool=None) == INVALID and "state_pool" in _msg()
    assert steps(n=0) == 0  # nothing to do


def test_valid_call_without_gpu_reports_cuda_error():
    """Arguments that pass validation reach the CUDA runtime, which on a host
    without a GPU fails cleanly with KDA_ERR_CUDA."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    assert _window(_acts(), False) == CUDA


def _commit(**kw):
    lib = _native.lib()
    args = dict(pool=FAKE, stride=4 * 16384, slots=8, sl=FAKE, acc=FAKE, n=2, hv=4, win=4, corr=FAKE,
                kg=FAKE, A_log=FAKE, dt=FAKE, lb=-5.0, stream=None)
    args.update(kw)
    return lib.kda_commit(args["pool"], args["stride"] * args["hv"], args["slots"], args["sl"], args["acc"], args["n"], args["hv"], args["win"],
                          args["corr"], args["kg"], args["A_log"], args["dt"], ctypes.c_float(args["lb"]),
                          args["stream"])


def test_commit_validation():
    assert _commit(win=0) == INVALID and "window" in _msg()
    assert _commit(win=9) == INVALID and "window" in _msg()
    assert _commit(n=-1) == INVALID
    assert _commit(n=0) == 0  # nothing to do
    assert _commit(hv=0) == INVALID and "hv" in _msg()
    assert _commit(sl=None) == INVALID and "must not be NULL" in _msg()
    assert _commit(acc=None) == INVALID and "must not be NULL" in _msg()
    assert _commit(corr=None) == INVALID and "corr and kg" in _msg()
    assert _commit(kg=FAKE + 8) == INVALID and "16-byte aligned" in _msg()
    assert _commit(A_log=None) == INVALID and "provided together" in _msg()
    assert _commit(lb=-11.0) == INVALID and "lower_bound" in _msg()
    assert _commit(pool=None) == INVALID and "state_pool" in _msg()
    assert _commit(slots=0) == INVALID and "at least one slot" in _msg()
    lib = _native.lib()

    def commit_ex(sb, kf, stride=4 * 16384):
        return lib.kda_commit_ex(FAKE, stride, 8, FAKE, FAKE, 2, 4, 4, FAKE, FAKE, FAKE, FAKE, -5.0, sb, kf,
                                 None)
    assert commit_ex(2, 0) == INVALID and "state_bf16 and kg_fp16" in _msg()
    assert commit_ex(0, 3) == INVALID and "state_bf16 and kg_fp16" in _msg()
    assert commit_ex(1, 0, stride=4 * 16384 + 4) == INVALID and "multiple of 8" in _msg()


def _host_call(a, cu=None, n=1, segment=0, ws_bytes=1 << 40):
    lib = _native.lib()
    return lib.kda_chunk_fwd_host(ctypes.byref(a), FAKE, cu, n, None, None, segment, 0, FAKE, ws_bytes, None)


def test_host_prefill_validation():
    """The host-memory prefill's own rules, checked before any CUDA call."""
    lib = _native.lib()
    a = _acts(t_total=128)
    assert _host_call(a, segment=100) == INVALID and "segment_tokens" in _msg()
    assert _host_call(_acts(t_total=128, state_bf16=1)) == INVALID and "fp32 states" in _msg()
    assert _host_call(_acts(t_total=128, q_stride_head=256, q_stride_tok=512)) == INVALID
    assert "contiguous heads" in _msg()
    assert _host_call(_acts(t_total=128, v_stride_tok=128)) == INVALID and "token strides" in _msg()
    bad = (ctypes.c_int32 * 3)(0, 100, 90)
    assert _host_call(_acts(t_total=90), cu=bad, n=2) == INVALID and "non-decreasing" in _msg()
    short = (ctypes.c_int32 * 3)(0, 10, 80)
    assert _host_call(_acts(t_total=90), cu=short, n=2) == INVALID and "0 to t_total" in _msg()
    assert _host_call(_acts(t_total=129), n=2) == INVALID and "divisible" in _msg()
    assert _host_call(a, ws_bytes=64) == INVALID and "workspace needs" in _msg()
    # the size query: mirrors of every band and the output, the carried
    # states, per-call tables and one call's prefill scratch
    cu = (ctypes.c_int32 * 3)(0, 100, 128)
    need = lib.kda_chunk_fwd_host_workspace_bytes(ctypes.byref(a), cu, 2, 64, 0)
    T, hqk, hv = 128, 2, 4
    mirrors = T * (2 * hqk + 3 * hv) * 128 * 2 + T * hv * 2
    assert need > mirrors + 2 * hv * 128 * 128 * 4
    assert lib.kda_chunk_fwd_host_workspace_bytes(ctypes.byref(a), cu, 2, 100, 0) == 0
    assert "segment_tokens" in _msg()


def test_wait_selftest_rejects_out_of_range_limits():
    """The bounded-wait self-test validates its limit before any launch."""
    lib = _native.lib()
    for bad in (0, 2_000_000):
        assert lib.kda_selftest_wait_timeout(bad, None) == INVALID
        assert "limit_us" in lib.kda_last_error().decode()
