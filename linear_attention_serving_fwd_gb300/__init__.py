"""GB300 (sm_103a) Kimi Delta Attention forward path.

Python binding of the C ABI in ``include/kda.h``: these functions only
marshal torch tensors into pointers, strides and the current CUDA stream;
every step of the computation runs in the library's CUDA kernels.

* :func:`kda_chunk_fwd` - chunked prefill (dense, varlen, paged state cache,
  optional chunk-group scan).
* :func:`kda_decode` - in-place window decode on a paged fp32 state cache.
* :func:`kda_decode_steps` - window decode with a [request, step] slot table
  and accepted-token counts (speculative multi-token decode).
* :func:`kda_verify` - speculative verify (state read only, correction
  records).
* :func:`kda_device_status` - read (and clear) the device error word.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _native
from ._native import KdaError

D = 128
__all__ = ["kda_chunk_fwd", "kda_chunk_fwd_noalloc", "kda_chunk_fwd_host", "kda_decode", "kda_decode_steps",
           "kda_verify", "kda_commit", "kda_device_status", "chunk_workspace_bytes",
           "chunk_fwd_host_workspace_bytes", "conv_scratch_bytes", "KdaError", "library_path"]


def library_path() -> str:
    return _native.lib_path()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _as_tokens(x: torch.Tensor, name: str, heads_dim: bool = True) -> torch.Tensor:
    """[T, H, 128] (or [T, H] for beta) view; [B, T, ...] dense input is
    flattened when its batch and time strides allow a single token stride."""
    want = 3 if heads_dim else 2
    if x.dim() == want + 1:
        x = x.reshape(-1, *x.shape[2:])
    if x.dim() != want:
        raise ValueError(f"{name} must be [T, H, 128] / [B, T, H, 128] (got {tuple(x.shape)}).")
    if heads_dim and (x.shape[-1] != D or x.stride(-1) != 1):
        raise ValueError(f"{name} needs a contiguous last dimension of 128.")
    return x


_STATE_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


def _state_bf16(*states) -> int:
    """0 for fp32 recurrent states, 1 for bf16; every given state tensor of
    a call must have the same dtype."""
    kinds = {t.dtype for t in states if t is not None}
    if not kinds:
        return 0
    if len(kinds) > 1:
        raise TypeError("all recurrent states of a call must share one dtype.")
    dt = kinds.pop()
    if dt not in _STATE_DTYPES:
        raise TypeError(f"recurrent states must be float32 or bfloat16 (got {dt}).")
    return _STATE_DTYPES[dt]


def _activations(q, k, v, g, beta, A_log, dt_bias, scale, lower_bound, host=False):
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if host and t.is_cuda:
            raise ValueError(f"{name} must be a host (CPU) tensor.")
        if not host and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor.")
    if q.dtype == torch.float16:
        dtype = _native.KDA_DTYPE_FP16
    elif q.dtype == torch.bfloat16:
        dtype = _native.KDA_DTYPE_BF16
    else:
        raise TypeError("chunk_kda supports torch.float16 and torch.bfloat16 inputs.")
    for name, t in (("k", k), ("v", v), ("g", g), ("beta", beta)):
        if t.dtype != q.dtype:
            raise TypeError("k, v, g and beta must have the same dtype as q.")
    if k.shape != q.shape:
        raise ValueError("k must have the same shape as q.")
    if g.shape != v.shape:
        raise ValueError("g must have the same shape as v.")
    if q.shape[0] != v.shape[0]:
        raise ValueError("q, v and g must have matching token counts.")
    if tuple(beta.shape) != tuple(v.shape[:2]):
        raise ValueError("beta must have shape [T, Hv].")
    if (A_log is None) != (dt_bias is None):
        raise ValueError("A_log and dt_bias must be provided together.")
    if A_log is not None:
        if A_log.dtype != torch.float32 or dt_bias.dtype != torch.float32:
            raise TypeError("A_log and dt_bias must be float32.")
        A_log = A_log.contiguous()
        dt_bias = dt_bias.contiguous()
    a = _native.KdaActivations()
    a.q, a.q_stride_tok, a.q_stride_head = q.data_ptr(), q.stride(0), q.stride(1)
    a.k, a.k_stride_tok, a.k_stride_head = k.data_ptr(), k.stride(0), k.stride(1)
    a.v, a.v_stride_tok, a.v_stride_head = v.data_ptr(), v.stride(0), v.stride(1)
    a.g, a.g_stride_tok, a.g_stride_head = g.data_ptr(), g.stride(0), g.stride(1)
    a.beta, a.beta_stride_tok, a.beta_stride_head = beta.data_ptr(), beta.stride(0), beta.stride(1)
    a.A_log = None if A_log is None else A_log.data_ptr()
    a.dt_bias = None if dt_bias is None else dt_bias.data_ptr()
    a.dtype = dtype
    a.t_total, a.hqk, a.hv = q.shape[0], q.shape[1], v.shape[1]
    a.use_qk_l2norm = 1
    a.scale = D ** -0.5 if scale is None else float(scale)
    a.lower_bound = float(lower_bound)
    a.state_bf16 = 0  # set by the caller from its state tensors
    return a, (A_log, dt_bias)  # keep contiguous copies alive


def _conv(conv_weight, conv_state, conv_dim_first, hqk, hv, *, state_indices=None,
          has_initial_state=None, num_accepted=None):
    """The kda_conv descriptor (or None) and the tensors it points into."""
    if conv_weight is None and conv_state is None:
        return None, []
    if conv_weight is None or conv_state is None:
        raise ValueError("conv_weight and conv_state must be given together.")
    C = (2 * hqk + hv) * D
    w = conv_weight.reshape(C, 4).contiguous()
    if w.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("conv_weight must be bfloat16 or float32.")
    if conv_state.dtype != torch.bfloat16 or conv_state.dim() != 3:
        raise ValueError("conv_state must be a bfloat16 [rows, positions, C] (or [rows, C, positions] "
                         "with conv_dim_first) tensor.")
    ch_dim, pos_dim = (1, 2) if conv_dim_first else (2, 1)
    if conv_state.shape[ch_dim] != C:
        raise ValueError(f"conv_state needs {C} channels (2 Hqk + Hv bands of 128).")
    cv = _native.KdaConv()
    cv.weight, cv.weight_f32 = w.data_ptr(), int(w.dtype == torch.float32)
    cv.state = conv_state.data_ptr()
    cv.row_stride, cv.pos_stride = conv_state.stride(0), conv_state.stride(pos_dim)
    cv.chan_stride = conv_state.stride(ch_dim)
    cv.rows, cv.positions = conv_state.shape[0], conv_state.shape[pos_dim]
    keep = [w]
    if state_indices is not None:
        state_indices = state_indices.to(torch.int32).contiguous()
        keep.append(state_indices)
        cv.state_indices = state_indices.data_ptr()
    if has_initial_state is not None:
        has_initial_state = has_initial_state.to(torch.uint8).contiguous()
        keep.append(has_initial_state)
        cv.has_initial_state = has_initial_state.data_ptr()
    if num_accepted is not None:
        num_accepted = num_accepted.to(torch.int32).contiguous()
        keep.append(num_accepted)
        cv.num_accepted = num_accepted.data_ptr()
    return cv, keep


def conv_scratch_bytes(t_total: int, hqk: int, hv: int) -> int:
    """Bytes of the optional conv scratch of a prefill with a conv."""
    return int(_native.lib().kda_conv_scratch_bytes(t_total, hqk, hv))


def chunk_workspace_bytes(n_seqs: int, t_total: int, hv: int, groups: int = 0) -> int:
    return int(_native.lib().kda_chunk_workspace_bytes(n_seqs, t_total, hv, groups))


def kda_chunk_fwd(q, k, v, g, beta, *, A_log=None, dt_bias=None, scale=None, lower_bound=-5.0,
                  cu_seqlens=None, n_seqs=None, initial_state=None, output_final_state=False,
                  final_state=None, out=None, state_cache=None, state_indices=None,
                  has_initial_state=None, groups: int = 0, workspace=None, stream=None,
                  checkpoint_state=None, checkpoint_offsets=None, checkpoint_state_indices=None,
                  conv_weight=None, conv_state=None, conv_state_indices=None,
                  conv_has_initial_state=None, conv_dim_first=False, conv_scratch=True):
    """Chunked KDA prefill.  Returns (out, final_state or None).

    q, k: [T, Hqk, 128] or [B, T, Hqk, 128]; v, g: [T, Hv, 128]; beta:
    [T, Hv] logits; bf16 or fp16 (o has the same dtype).  Dense [B, T] input
    without ``cu_seqlens`` runs B sequences of T tokens.  Recurrent states
    (initial_state, final_state, state_cache, checkpoint_state) are all fp32
    or all bf16; a bf16 final state is rounded once at the end.
    ``state_cache`` [slots, Hv, 128, 128] with
    ``state_indices`` [N] int32 (and optional ``has_initial_state`` [N])
    replaces initial_state / final_state and is updated in place.
    ``checkpoint_state`` [rows, Hv, 128, 128] with ``checkpoint_offsets``
    [N] (and optional ``checkpoint_state_indices`` [N]) receives each
    sequence's state after its first checkpoint_offsets[n] tokens (a positive
    multiple of 64 no larger than its length; other offsets are skipped).
    ``conv_weight`` [C, 4] (bf16 or fp32) with ``conv_state`` bf16
    [rows, positions >= 3, C] (``conv_dim_first``: [rows, C, positions]) and
    ``conv_state_indices`` [N] makes q, k, v the raw projection bands
    (C = (2 Hqk + Hv) * 128): they pass a width-4 depthwise conv and SiLU
    first, and each sequence's conv row is left holding its last three raw
    inputs.  ``conv_scratch`` (True: allocated here; or a uint8 CUDA tensor of
    ``conv_scratch_bytes(T, Hqk, Hv)``) lets the conv run once per (token,
    channel) in its own pass; False makes each prologue item convolve its
    own rows.  Both give the same results.
    ``groups``: 0 lets the library choose; 1 walks each chain in a launch of
    its own after the prologue; G > 1 runs the chunk-group scan; -1 runs the
    pipelined launch (dense sequences, at most 48 (sequence, head) chains), in
    which one CTA per chain walks while the prologue still runs on the other
    SMs.
    """
    dense_b = q.shape[0] if q.dim() == 4 else None
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    v, g = _as_tokens(v, "v"), _as_tokens(g, "g")
    beta = _as_tokens(beta, "beta", heads_dim=False)
    a, keep = _activations(q, k, v, g, beta, A_log, dt_bias, scale, lower_bound)
    T, hv = q.shape[0], v.shape[1]
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must have dtype torch.int32.")
        cu_seqlens = cu_seqlens.contiguous()
        n = cu_seqlens.numel() - 1
    else:
        n = n_seqs if n_seqs is not None else (dense_b if dense_b is not None else 1)
    if out is None:
        out = torch.empty((T, hv, D), dtype=q.dtype, device=q.device)
    elif out.shape != (T, hv, D) or not out.is_contiguous():
        out = out.view(T, hv, D)
    slot_stride, n_slots = 0, 0
    if state_cache is not None:
        if state_indices is None:
            raise ValueError("state_cache needs state_indices.")
        state_indices = state_indices.to(torch.int32).contiguous()
        if has_initial_state is not None:
            has_initial_state = has_initial_state.to(torch.uint8).contiguous()
        slot_stride, n_slots = state_cache.stride(0), state_cache.shape[0]
        if tuple(state_cache.shape[1:]) != (hv, D, D) or state_cache[0].stride() != (D * D, D, 1):
            raise ValueError("state_cache must be [slots, Hv, 128, 128] with contiguous rows.")
    a.state_bf16 = _state_bf16(initial_state, final_state, state_cache, checkpoint_state)
    if output_final_state and final_state is None:
        final_state = torch.empty((n, hv, D, D), dtype=torch.bfloat16 if a.state_bf16 else torch.float32,
                                  device=q.device)
    if initial_state is not None:
        initial_state = initial_state.contiguous()
    ws_bytes = chunk_workspace_bytes(n, T, hv, groups)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ck_stride, ck_rows = 0, 0
    cv, cv_keep = _conv(conv_weight, conv_state, conv_dim_first, a.hqk, hv,
                        state_indices=conv_state_indices, has_initial_state=conv_has_initial_state)
    if cv is not None and conv_state_indices is None:
        raise ValueError("conv_state needs conv_state_indices.")
    if cv is not None and conv_scratch is not False and conv_scratch is not None:
        if conv_scratch is True:
            conv_scratch = torch.empty(conv_scratch_bytes(T, a.hqk, hv), dtype=torch.uint8, device=q.device)
        cv.scratch, cv.scratch_bytes = conv_scratch.data_ptr(), conv_scratch.numel() * conv_scratch.element_size()
        cv_keep.append(conv_scratch)
    if checkpoint_state is not None or cv is not None:
        if checkpoint_state is not None:
            if checkpoint_offsets is None:
                raise ValueError("checkpoint_state needs checkpoint_offsets.")
            if (tuple(checkpoint_state.shape[1:]) != (hv, D, D)
                    or checkpoint_state[0].stride() != (D * D, D, 1)):
                raise ValueError("checkpoint_state must be [rows, Hv, 128, 128] with contiguous rows.")
            ck_stride, ck_rows = checkpoint_state.stride(0), checkpoint_state.shape[0]
            checkpoint_offsets = checkpoint_offsets.to(torch.int32).contiguous()
            if checkpoint_state_indices is not None:
                checkpoint_state_indices = checkpoint_state_indices.to(torch.int32).contiguous()
        rc = _native.lib().kda_chunk_fwd_ex(
            ctypes.byref(a), _ptr(out), _ptr(cu_seqlens), n, _ptr(initial_state), _ptr(final_state),
            _ptr(state_cache), slot_stride, n_slots, _ptr(state_indices), _ptr(has_initial_state),
            _ptr(checkpoint_state), ck_stride, ck_rows, _ptr(checkpoint_offsets),
            _ptr(checkpoint_state_indices), None if cv is None else ctypes.byref(cv), int(groups),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
        del cv_keep
    else:
        rc = _native.lib().kda_chunk_fwd(
            ctypes.byref(a), _ptr(out), _ptr(cu_seqlens), n, _ptr(initial_state), _ptr(final_state),
            _ptr(state_cache), slot_stride, n_slots, _ptr(state_indices), _ptr(has_initial_state),
            int(groups), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream_handle(stream))
    _native.check(rc)
    del keep
    return out, final_state


def kda_chunk_fwd_host(q, k, v, g, beta, *, A_log=None, dt_bias=None, scale=None, lower_bound=-5.0,
                       cu_seqlens=None, n_seqs=None, initial_state=None, output_final_state=False,
                       final_state=None, out=None, segment_tokens: int = 0, groups: int = 0,
                       workspace=None, device=None, stream=None):
    """Chunked prefill on host (CPU) tensors; returns (out, final_state or None),
    both host tensors.

    The same shapes and rules as ``kda_chunk_fwd`` with every tensor in host
    memory (``cu_seqlens`` an int32 CPU tensor; A_log, dt_bias, states fp32
    CPU tensors).  The library copies segments of ``segment_tokens`` tokens
    of every sequence to the GPU, runs them as chunked prefill with the
    state carried between segments, and copies the outputs back, the copies
    overlapping the kernels when the host tensors are page-locked
    (``pin_memory()``; ``out`` and ``final_state`` are allocated page-locked
    when not given).  ``workspace`` is a uint8 CUDA tensor of at least
    ``chunk_fwd_host_workspace_bytes(..)`` bytes, allocated on ``device``
    when not given.  The call returns once the work is queued on ``stream``:
    synchronise it before reading ``out``.
    """
    dense_b = q.shape[0] if q.dim() == 4 else None
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    v, g = _as_tokens(v, "v"), _as_tokens(g, "g")
    beta = _as_tokens(beta, "beta", heads_dim=False)
    if any(t is not None and t.is_cuda for t in (A_log, dt_bias)):
        raise ValueError("A_log and dt_bias must be CPU tensors.")
    a, keep = _activations(q, k, v, g, beta, A_log, dt_bias, scale, lower_bound, host=True)
    T, hv = q.shape[0], v.shape[1]
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.is_cuda:
            raise TypeError("cu_seqlens must be an int32 CPU tensor.")
        cu_seqlens = cu_seqlens.contiguous()
        n = cu_seqlens.numel() - 1
    else:
        n = n_seqs if n_seqs is not None else (dense_b if dense_b is not None else 1)
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is not None and (t.is_cuda or t.dtype != torch.float32 or tuple(t.shape) != (n, hv, D, D)
                              or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous fp32 CPU tensor [N, Hv, 128, 128].")
    if out is None:
        out = torch.empty((T, hv, D), dtype=q.dtype).pin_memory()
    elif out.is_cuda or tuple(out.shape) != (T, hv, D) or not out.is_contiguous() or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous CPU tensor [T, Hv, 128] of the input dtype.")
    if output_final_state and final_state is None:
        final_state = torch.empty((n, hv, D, D), dtype=torch.float32).pin_memory()
    lib = _native.lib()
    need = int(lib.kda_chunk_fwd_host_workspace_bytes(ctypes.byref(a), _ptr(cu_seqlens), n,
                                                      int(segment_tokens), int(groups)))
    if need == 0:
        raise _native.KdaError(_native.KDA_ERR_INVALID_ARGUMENT, lib.kda_last_error().decode())
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8,
                                device=device if device is not None else torch.cuda.current_device())
    elif not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor.")
    with torch.cuda.device(workspace.device):
        rc = lib.kda_chunk_fwd_host(ctypes.byref(a), _ptr(out), _ptr(cu_seqlens), n, _ptr(initial_state),
                                    _ptr(final_state), int(segment_tokens), int(groups), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _native.check(rc)
    del keep
    return out, final_state


def chunk_fwd_host_workspace_bytes(q, k, v, g, beta, *, A_log=None, dt_bias=None, cu_seqlens=None,
                                   n_seqs=None, segment_tokens: int = 0, groups: int = 0) -> int:
    """Workspace bytes ``kda_chunk_fwd_host`` needs for these host tensors."""
    dense_b = q.shape[0] if q.dim() == 4 else None
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    v, g = _as_tokens(v, "v"), _as_tokens(g, "g")
    beta = _as_tokens(beta, "beta", heads_dim=False)
    a, keep = _activations(q, k, v, g, beta, A_log, dt_bias, None, -5.0, host=True)
    n = (cu_seqlens.numel() - 1 if cu_seqlens is not None
         else n_seqs if n_seqs is not None else (dense_b if dense_b is not None else 1))
    lib = _native.lib()
    need = int(lib.kda_chunk_fwd_host_workspace_bytes(ctypes.byref(a), _ptr(cu_seqlens), n,
                                                      int(segment_tokens), int(groups)))
    del keep
    if need == 0:
        raise _native.KdaError(_native.KDA_ERR_INVALID_ARGUMENT, lib.kda_last_error().decode())
    return need


def kda_chunk_fwd_noalloc(q, k, v, g, beta, *, out, A_log=None, dt_bias=None, scale=None,
                          lower_bound=-5.0, cu_seqlens=None, n_seqs=None, initial_state=None,
                          final_state=None, state_cache=None, state_indices=None,
                          has_initial_state=None, groups: int = 0, stream=None):
    """Chunked prefill through ``kda_chunk_fwd_noalloc``: for callers that
    cannot allocate device memory.  The library's fixed 64 MiB scratch array
    replaces the workspace; the caller passes every input and output
    (``out`` and, if wanted, ``final_state``), so with contiguous A_log /
    dt_bias this wrapper allocates nothing on the device either.  Calls that
    overlap on the GPU race on the shared scratch.  Returns (out, final_state)."""
    dense_b = q.shape[0] if q.dim() == 4 else None
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    v, g = _as_tokens(v, "v"), _as_tokens(g, "g")
    beta = _as_tokens(beta, "beta", heads_dim=False)
    a, keep = _activations(q, k, v, g, beta, A_log, dt_bias, scale, lower_bound)
    if cu_seqlens is not None:
        n = cu_seqlens.numel() - 1
    else:
        n = n_seqs if n_seqs is not None else (dense_b if dense_b is not None else 1)
    slot_stride, n_slots = 0, 0
    if state_cache is not None:
        slot_stride, n_slots = state_cache.stride(0), state_cache.shape[0]
    a.state_bf16 = _state_bf16(initial_state, final_state, state_cache)
    rc = _native.lib().kda_chunk_fwd_noalloc(
        ctypes.byref(a), _ptr(out), _ptr(cu_seqlens), n, _ptr(initial_state), _ptr(final_state),
        _ptr(state_cache), slot_stride, n_slots, _ptr(state_indices), _ptr(has_initial_state),
        int(groups), _stream_handle(stream))
    _native.check(rc)
    del keep
    return out, final_state


def _window_call(verify, q, k, v, g, beta, state_pool, query_start, slots, window, *, A_log,
                 dt_bias, scale, lower_bound, out, corr, kg, work_counter, stream,
                 num_accepted_tokens=None, conv_weight=None, conv_state=None, conv_dim_first=False):
    a, keep = _activations(_as_tokens(q, "q"), _as_tokens(k, "k"), _as_tokens(v, "v"),
                           _as_tokens(g, "g"), _as_tokens(beta, "beta", heads_dim=False),
                           A_log, dt_bias, scale, lower_bound)
    T, hv = a.t_total, a.hv
    table = slots.dim() == 2
    n_req = slots.shape[0] if table else slots.numel()
    if query_start.dtype != torch.int32 or slots.dtype != torch.int32:
        raise TypeError("query_start and slots must have dtype torch.int32.")
    if table and verify:
        raise ValueError("kda_verify takes one slot per request.")
    if table and slots.stride(1) != 1:
        raise ValueError("a [n_req, steps] slot table must have contiguous rows.")
    if num_accepted_tokens is not None:
        if num_accepted_tokens.dtype != torch.int32 or num_accepted_tokens.numel() != n_req:
            raise ValueError("num_accepted_tokens must be int32 with one entry per request.")
    a.state_bf16 = _state_bf16(state_pool)
    if tuple(state_pool.shape[1:]) != (hv, D, D) or state_pool[0].stride() != (D * D, D, 1):
        raise ValueError("state_pool must be [slots, Hv, 128, 128] with contiguous rows.")
    if out is None:
        out = torch.empty((T, hv, D), dtype=q.dtype, device=q.device)
    lib = _native.lib()
    if verify:
        if corr is None:
            corr = torch.empty((n_req, hv, window, D), dtype=torch.float32, device=q.device)
        if kg is None:
            kg = torch.empty((n_req, hv, window, 2 * D), dtype=q.dtype, device=q.device)
        if work_counter is None:
            work_counter = torch.zeros(1, dtype=torch.int32, device=q.device)
        cv, cv_keep = _conv(conv_weight, conv_state, conv_dim_first, a.hqk, hv,
                            num_accepted=num_accepted_tokens)
        if cv is not None:
            if num_accepted_tokens is None:
                raise ValueError("verify with a conv needs num_accepted_tokens.")
            rc = lib.kda_verify_ex(ctypes.byref(a), _ptr(out), _ptr(state_pool), state_pool.stride(0),
                                   state_pool.shape[0], _ptr(query_start), _ptr(slots), n_req, window,
                                   _ptr(corr), _ptr(kg), _ptr(work_counter), ctypes.byref(cv),
                                   _stream_handle(stream))
            del cv_keep
        else:
            rc = lib.kda_verify(ctypes.byref(a), _ptr(out), _ptr(state_pool), state_pool.stride(0),
                                state_pool.shape[0], _ptr(query_start), _ptr(slots), n_req, window,
                                _ptr(corr), _ptr(kg), _ptr(work_counter), _stream_handle(stream))
    elif table:
        rc = lib.kda_decode_steps(ctypes.byref(a), _ptr(out), _ptr(state_pool), state_pool.stride(0),
                                  state_pool.shape[0], _ptr(query_start), _ptr(slots),
                                  slots.stride(0), _ptr(num_accepted_tokens), n_req, window,
                                  _stream_handle(stream))
    else:
        rc = lib.kda_decode(ctypes.byref(a), _ptr(out), _ptr(state_pool), state_pool.stride(0),
                            state_pool.shape[0], _ptr(query_start), _ptr(slots), n_req, window,
                            _stream_handle(stream))
    _native.check(rc)
    del keep
    return out, corr, kg


def kda_decode(q, k, v, g, beta, state_pool, query_start, slots, window, *, A_log=None,
               dt_bias=None, scale=None, lower_bound=-5.0, out=None, stream=None):
    """In-place decode: request b runs tokens query_start[b]..query_start[b+1]-1
    (at most ``window``) on pool row slots[b] (negative = padding).  Returns out."""
    return _window_call(False, q, k, v, g, beta, state_pool, query_start, slots, window,
                        A_log=A_log, dt_bias=dt_bias, scale=scale, lower_bound=lower_bound,
                        out=out, corr=None, kg=None, work_counter=None, stream=stream)[0]


def kda_decode_steps(q, k, v, g, beta, state_pool, query_start, state_indices, window, *,
                     num_accepted_tokens=None, A_log=None, dt_bias=None, scale=None,
                     lower_bound=-5.0, out=None, stream=None):
    """Decode with a [n_req, steps] int32 slot table (steps >= window):
    request b starts from pool row state_indices[b, num_accepted_tokens[b] - 1]
    (column 0 without counts) and the state after its token t is stored to
    row state_indices[b, t] (negative = no store; a negative start row makes
    b padding).  Returns out."""
    if state_indices.dim() != 2:
        raise ValueError("state_indices must be a [n_req, steps] table.")
    return _window_call(False, q, k, v, g, beta, state_pool, query_start, state_indices, window,
                        A_log=A_log, dt_bias=dt_bias, scale=scale, lower_bound=lower_bound,
                        out=out, corr=None, kg=None, work_counter=None, stream=stream,
                        num_accepted_tokens=num_accepted_tokens)[0]


def kda_verify(q, k, v, g, beta, state_pool, query_start, slots, window, *, A_log=None,
               dt_bias=None, scale=None, lower_bound=-5.0, out=None, corr=None, kg=None,
               work_counter=None, stream=None, conv_weight=None, conv_state=None,
               num_accepted_tokens=None, conv_dim_first=False):
    """Speculative verify (state read only).  Returns (out, corr, kg).

    With ``conv_weight`` [C, 4] and ``conv_state`` bf16 [slots, positions >=
    window + 2, C] (``conv_dim_first``: [slots, C, positions]) and
    ``num_accepted_tokens`` [n_req], q, k, v are the raw projection bands:
    they pass the width-4 conv + SiLU after the history at positions
    accepted-1 .. accepted+1 of row slots[b], and the conv state is rolled."""
    return _window_call(True, q, k, v, g, beta, state_pool, query_start, slots, window,
                        A_log=A_log, dt_bias=dt_bias, scale=scale, lower_bound=lower_bound,
                        out=out, corr=corr, kg=kg, work_counter=work_counter, stream=stream,
                        num_accepted_tokens=num_accepted_tokens, conv_weight=conv_weight,
                        conv_state=conv_state, conv_dim_first=conv_dim_first)


def kda_commit(state_pool, slots, num_accepted, corr, kg, window, *, A_log=None, dt_bias=None,
               lower_bound=-5.0, stream=None):
    """Speculative-decode commit: rebuild pool rows slots[b] in place as the
    state after request b's first num_accepted[b] verified tokens, from the
    corr / kg records of :func:`kda_verify` (same pool, window and gate
    parameters).  Returns the pool."""
    if slots.dtype != torch.int32 or num_accepted.dtype != torch.int32:
        raise TypeError("slots and num_accepted must have dtype torch.int32.")
    state_bf16 = _state_bf16(state_pool)
    hv = state_pool.shape[1]
    if tuple(state_pool.shape[1:]) != (hv, D, D) or state_pool[0].stride() != (D * D, D, 1):
        raise ValueError("state_pool must be [slots, Hv, 128, 128] with contiguous rows.")
    n_req = slots.numel()
    if num_accepted.numel() != n_req:
        raise ValueError("num_accepted must have one entry per request.")
    if tuple(corr.shape) != (n_req, hv, window, D) or corr.dtype != torch.float32 or not corr.is_contiguous():
        raise ValueError("corr must be a contiguous float32 [n_req, Hv, window, 128] tensor.")
    if (tuple(kg.shape) != (n_req, hv, window, 2 * D) or kg.dtype not in (torch.bfloat16, torch.float16)
            or not kg.is_contiguous()):
        raise ValueError("kg must be a contiguous bfloat16 / float16 [n_req, Hv, window, 256] tensor.")
    keep = []
    if A_log is not None:
        A_log = A_log.detach().float().contiguous()
        dt_bias = dt_bias.detach().float().contiguous()
        keep = [A_log, dt_bias]
    rc = _native.lib().kda_commit_ex(_ptr(state_pool), state_pool.stride(0), state_pool.shape[0],
                                     _ptr(slots), _ptr(num_accepted), n_req, hv, window, _ptr(corr),
                                     _ptr(kg), _ptr(A_log), _ptr(dt_bias), float(lower_bound), state_bf16,
                                     int(kg.dtype == torch.float16), _stream_handle(stream))
    _native.check(rc)
    del keep
    return state_pool


def kda_device_status(stream=None, clear: bool = True) -> int:
    """Synchronise and read the device error word (0 = clean)."""
    return int(_native.lib().kda_device_status(_stream_handle(stream), int(clear)))


def kda_selftest_wait_timeout(limit_us: int = 1000, stream=None) -> None:
    """Launch the bounded-wait self-test: one CTA waits on a barrier nothing
    arrives at and gives up after ``limit_us`` microseconds, setting the
    timeout bit that ``kda_device_status`` then reports."""
    _native.check(_native.lib().kda_selftest_wait_timeout(int(limit_us), _stream_handle(stream)))
