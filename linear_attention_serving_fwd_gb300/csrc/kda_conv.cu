// Conv state updates, launched after the kernels that read the history
// (stream order keeps every read ahead of the write of its row).
//  * prefill (kda_chunk_fwd with a conv): sequence n's row ends holding its
//    last three raw inputs at positions 0..2 (a shorter sequence keeps the
//    tail of its history in front of them);
//  * verify: the rolled state of the verify page's conv path, positions
//    0, 1 = the two newest history inputs (read at accepted-1 .. accepted+1)
//    and 2 + t = raw input t of the window.
// One thread per (sequence or request, channel).
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
