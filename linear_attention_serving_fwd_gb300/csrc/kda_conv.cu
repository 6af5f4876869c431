// Conv state updates, launched after the kernels that read the history
// (stream order keeps every read ahead of the write of its row).
//  * prefill (kda_chunk_fwd with a conv): sequence n's row ends holding its
//    last three raw inputs at positions 0..2 (a shorter sequence keeps the
//    tail of its history in front of them);
//  * verify: the rolled state of the verify page's conv path, positions
//    0, 1 = the two newest history inputs (read at accepted-1 .. accepted+1)
//    and 2 + t = raw input t of the window.
// One thread per (sequence or request, channel).
// A prefill given a conv scratch buffer also convolves every (token, channel)
// once, in its own pass, before the prologue (kda_conv_prefill_kernel).
#include "kda_conv.cuh"

namespace kda {

constexpr int CONV_THREADS = 256;

__global__ void __launch_bounds__(CONV_THREADS) kda_conv_prefill_state_kernel(ChunkParams p) {
  const int n = blockIdx.y;
  const int64_t C = (2 * (int64_t)p.hqk + p.hv) * D;
  const int64_t ch = (int64_t)blockIdx.x * CONV_THREADS + threadIdx.x;
  if (ch >= C) return;
  const ConvParams& cv = p.conv;
  const int row = cv.idx[n];
  if (row < 0) return;
  if (row >= cv.rows) {
    if (ch == 0) set_error(p.err, ERR_INDEX);
    return;
  }
  const int bos = p.cu_seqlens ? p.cu_seqlens[n] : n * p.dense_len;
  const int eos = p.cu_seqlens ? p.cu_seqlens[n + 1] : (n + 1) * p.dense_len;
  const int len = eos - bos;
  if (len < 0) return;  // flagged by the chunk index kernel
  __nv_bfloat16* st = cv.state + (int64_t)row * cv.row_st + ch * cv.ch_st;
  const bool init = !cv.has_init || cv.has_init[n];
  __nv_bfloat16 h[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) h[i] = init ? st[i * cv.pos_st] : __float2bfloat16(0.f);
  int64_t ts;
  const __nv_bfloat16* src = conv_source(p, ch, ts);
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int t = len - 3 + i;  // the input three, two, one back from the end
    st[i * cv.pos_st] = t >= 0 ? src[(int64_t)(bos + t) * ts] : h[i + len];
  }
}

__global__ void __launch_bounds__(CONV_THREADS) kda_conv_roll_kernel(WindowParams p) {
  const int b = blockIdx.y;
  const int64_t C = (2 * (int64_t)p.hqk + p.hv) * D;
  const int64_t ch = (int64_t)blockIdx.x * CONV_THREADS + threadIdx.x;
  if (ch >= C) return;
  const ConvParams& cv = p.conv;
  const int64_t slot = p.slots[b];
  const int qs = p.query_start[b], qlen = p.query_start[b + 1] - qs;
  const int first = cv.accepted[b] - 1;
  // the items the window kernel treated as padding or flagged keep their row
  if (slot < 0 || slot >= p.n_slots || slot >= cv.rows || qlen <= 0 || qlen > p.window || first < 0 ||
      first + 3 > cv.positions)
    return;
  __nv_bfloat16* st = cv.state + slot * cv.row_st + ch * cv.ch_st;
  const __nv_bfloat16 h1 = st[(first + 1) * cv.pos_st], h2 = st[(first + 2) * cv.pos_st];
  int64_t ts;
  const __nv_bfloat16* src = conv_source(p, ch, ts);
  st[0] = h1;
  st[cv.pos_st] = h2;
  for (int t = 0; t < qlen; ++t) st[(2 + t) * cv.pos_st] = src[(int64_t)(qs + t) * ts];
}

// The conv + SiLU of the prefill's raw q, k, v bands into p.conv_out, one
// thread per (channel pair, run of CONV_RUN tokens of the flattened batch):
// the run's raw inputs (and the three before it) are loaded first, then each
// token's taps read its own sequence's inputs, and before the sequence's
// first token the history at positions 0..2 of its conv row (zeros without
// one), as each prologue item reads its halo rows.  The arithmetic is the
// prologue's (conv_silu: the same per-tap roundings in the same order), so
// both paths give the same bf16 outputs.
constexpr int CONV_RUN = 32;

__global__ void __launch_bounds__(CONV_THREADS) kda_conv_prefill_kernel(ChunkParams p) {
  const int64_t qk = (int64_t)p.hqk * D, C = 2 * qk + (int64_t)p.hv * D;
  const int64_t ch = 2 * ((int64_t)blockIdx.x * CONV_THREADS + threadIdx.x);  // channels ch, ch + 1
  if (ch >= C) return;
  const int T = p.t_total;
  const int t0 = blockIdx.y * CONV_RUN, t1 = min(t0 + CONV_RUN, T);
  if (t0 >= T) return;
  const ConvParams& cv = p.conv;
  int64_t ts;
  const __nv_bfloat16* src = conv_source(p, ch, ts);
  __nv_bfloat162 raw[CONV_RUN + 3];  // tokens t0 - 3 .. t0 + CONV_RUN - 1
#pragma unroll
  for (int i = 0; i < CONV_RUN + 3; ++i) {
    const int t = t0 - 3 + i;
    raw[i] = (t >= 0 && t < t1) ? *reinterpret_cast<const __nv_bfloat162*>(src + (int64_t)t * ts)
                                : __float2bfloat162_rn(0.f);
  }
  // the sequence holding token t0 (the last whose start is <= t0)
  int n;
  if (p.cu_seqlens) {
    int lo = 0, hi = p.n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.cu_seqlens[mid] <= t0) lo = mid; else hi = mid - 1;
    }
    n = lo;
  } else {
    n = t0 / p.dense_len;
  }
  auto seq_bounds = [&](int m, int& b, int& e) {
    b = p.cu_seqlens ? p.cu_seqlens[m] : m * p.dense_len;
    e = p.cu_seqlens ? p.cu_seqlens[m + 1] : (m + 1) * p.dense_len;
  };
  auto history = [&](int m, __nv_bfloat162 h[3]) {
    const int row = cv.idx[m];
    const bool init = row >= 0 && row < cv.rows && (!cv.has_init || cv.has_init[m]);
    const __nv_bfloat16* st = cv.state + (int64_t)row * cv.row_st + ch * cv.ch_st;
#pragma unroll
    for (int i = 0; i < 3; ++i)
      h[i] = init ? __halves2bfloat162(st[i * cv.pos_st], st[i * cv.pos_st + cv.ch_st]) : __float2bfloat162_rn(0.f);
  };
  int bos, eos;
  seq_bounds(n, bos, eos);
  __nv_bfloat162 h[3];
  history(n, h);
  __nv_bfloat16* dst;
  int64_t ds;
  if (ch < qk) {
    dst = p.conv_out + ch;
    ds = qk;
  } else if (ch < 2 * qk) {
    dst = p.conv_out + (int64_t)T * qk + (ch - qk);
    ds = qk;
  } else {
    dst = p.conv_out + 2 * (int64_t)T * qk + (ch - 2 * qk);
    ds = (int64_t)p.hv * D;
  }
  const float4 w0 = conv_taps(cv, ch), w1 = conv_taps(cv, ch + 1);
  // channel-pair taps: bf16 pairs (each product a bf16 pair multiply, the
  // exact product rounded to bf16) or fp32 pairs (an fma chain)
  const float2 wf[4] = {make_float2(w0.x, w1.x), make_float2(w0.y, w1.y), make_float2(w0.z, w1.z),
                        make_float2(w0.w, w1.w)};
  __nv_bfloat162 wb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) wb[j] = __floats2bfloat162_rn(wf[j].x, wf[j].y);  // exact: bf16 taps
  const bool f32 = cv.w_f32 != 0;
  // SiLU of the conv sum over inputs x0 (oldest) .. x3 of the two channels
  auto conv2 = [&](__nv_bfloat162 x0, __nv_bfloat162 x1, __nv_bfloat162 x2, __nv_bfloat162 x3) {
    const __nv_bfloat162 xs[4] = {x0, x1, x2, x3};
    float2 acc;
    if (f32) {
      acc = fmul2(__bfloat1622float2(xs[0]), wf[0]);
#pragma unroll
      for (int j = 1; j < 4; ++j) acc = ffma2(__bfloat1622float2(xs[j]), wf[j], acc);
    } else {
      acc = __bfloat1622float2(__hmul2(xs[0], wb[0]));
#pragma unroll
      for (int j = 1; j < 4; ++j) acc = fadd2(acc, __bfloat1622float2(__hmul2(xs[j], wb[j])));
    }
    return __floats2bfloat162_rn(silu(acc.x), silu(acc.y));
  };
  if (t0 - 3 >= bos && t1 <= eos) {
    // the run and the three inputs before it lie in one sequence (almost
    // every run): no history, no boundary
#pragma unroll
    for (int i = 0; i < CONV_RUN; ++i)
      if (t0 + i < t1)
        *reinterpret_cast<__nv_bfloat162*>(dst + (int64_t)(t0 + i) * ds) =
            conv2(raw[i], raw[i + 1], raw[i + 2], raw[i + 3]);
    return;
  }
  for (int i = 0; i < CONV_RUN; ++i) {
    const int t = t0 + i;
    if (t >= t1) break;
    if (t >= eos) {  // a new sequence (skipping empty ones) starts at t
      while (n + 1 < p.n_seqs && t >= eos) {
        ++n;
        seq_bounds(n, bos, eos);
      }
      history(n, h);
    }
    __nv_bfloat162 x[4];  // inputs of tokens t - 3 .. t
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tt = t - 3 + j;
      const int hp = tt - bos + 3;  // before the sequence: its history position
      // (the few runs that meet a sequence boundary re-read their inputs,
      // just loaded and cached, so that raw[] keeps static indices)
      x[j] = (tt >= bos && tt >= 0) ? *reinterpret_cast<const __nv_bfloat162*>(src + (int64_t)tt * ts)
                       : (hp >= 0 ? h[hp < 3 ? hp : 2] : __float2bfloat162_rn(0.f));
    }
    *reinterpret_cast<__nv_bfloat162*>(dst + (int64_t)t * ds) = conv2(x[0], x[1], x[2], x[3]);
  }
}

int launch_conv_prefill(const ChunkParams& p, cudaStream_t stream) {
  const int64_t C = (2 * (int64_t)p.hqk + p.hv) * D;
  trace_begin("kda_conv_prefill", stream);
  kda_conv_prefill_kernel<<<dim3((unsigned)((C / 2 + CONV_THREADS - 1) / CONV_THREADS),
                                 (unsigned)((p.t_total + CONV_RUN - 1) / CONV_RUN)),
                            CONV_THREADS, 0, stream>>>(p);
  trace_end(stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_conv_prefill_state(const ChunkParams& p, cudaStream_t stream) {
  const int64_t C = (2 * (int64_t)p.hqk + p.hv) * D;
  trace_begin("kda_conv_state", stream);
  kda_conv_prefill_state_kernel<<<dim3((unsigned)((C + CONV_THREADS - 1) / CONV_THREADS), p.n_seqs),
                                  CONV_THREADS, 0, stream>>>(p);
  trace_end(stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_conv_roll(const WindowParams& p, cudaStream_t stream) {
  const int64_t C = (2 * (int64_t)p.hqk + p.hv) * D;
  trace_begin("kda_conv_roll", stream);
  kda_conv_roll_kernel<<<dim3((unsigned)((C + CONV_THREADS - 1) / CONV_THREADS), p.n_req), CONV_THREADS,
                         0, stream>>>(p);
  trace_end(stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace kda
