// Decode (in place) and speculative verify (read only) over a paged fp32
// state cache, window Q <= 8 tokens per request.
//
// Design (memory bound: each (request, head) moves its 64 KB V-first state
// once in, and for decode once out):
//  * persistent grid, one CTA per SM, 256 threads = 8 warps;
//  * two 64 KB state buffers filled by 1-D bulk async copies (TMA engine)
//    completing on mbarriers, plus two small buffers for the window's q/k/v/g
//    rows; the state of the item two ahead streams in while this one runs;
//  * warp w owns state rows v = 16w..16w+15 (rows of S^T), lane L owns key
//    channels 4L..4L+3, so a warp reads one 512-byte row per instruction
//    (bank-conflict free) and the state lives in 64 registers per thread;
//  * per token, the two row dot products (with exp(gate) * k^ and with
//    exp(gate) * q~) are reduced across the warp by one recursive-halving
//    reduce-scatter (31 shuffles for 32 sums), after which lane L < 16 holds
//    row L's correction U and lane L + 16 its output.
// Token order inside the window follows the recurrence exactly:
//   S <- diag(e^gate) S;  U = beta (v - S^T k^);  S <- S + k^ U^T;  o = S^T q~
// computed as U = beta (v - S_old^T (e^gate * k^)),
//             o = S_old^T (e^gate * q~) + U (k^ . q~),  S = e^gate * S_old + k^ U^T.
// Verify (the vLLM kimi_k3 CuTeDSL verify page, KdaTcVerify) additionally
// writes corr = U_t and kg = (raw k_t, raw g_t) and never writes the state;
// its persistent scheduler takes tickets from a caller-zeroed counter and the
// taker of the last ticket resets it.
#include "kda_params.cuh"

namespace kda {



constexpr int WIN_THREADS = 256;
constexpr int STATE_BYTES = D * D * 4;           // 65536
constexpr int ROW_BYTES = D * 2;                 // one bf16 row of 128
constexpr int IN_BYTES = MAX_WINDOW * 4 * ROW_BYTES;  // q, k, v, g rows per token
constexpr int WIN_SMEM = 2 * STATE_BYTES + 2 * IN_BYTES + 64;

struct ItemInfo {
  int request, head, qs, qlen;
  int64_t slot;
  bool work;   // state is loaded and tokens processed
  bool zero;   // padding request: write zero outputs
  bool bad;    // out-of-range slot or window length (reported, treated as padding)
};

__device__ __forceinline__ ItemInfo item_info(const WindowParams& p, int item) {
  ItemInfo r;
  r.request = item / p.hv;
  r.head = item - r.request * p.hv;
  r.qs = p.query_start[r.request];
  r.qlen = p.query_start[r.request + 1] - r.qs;
  r.slot = p.slots[r.request];
  bool bad_len = r.qlen < 0 || r.qlen > p.window;
  bool bad_slot = r.slot >= p.n_slots;
  r.work = !bad_len && !bad_slot && r.slot >= 0 && r.qlen > 0;
  r.zero = !bad_len && r.qlen > 0 && !r.work;
  r.bad = bad_len || bad_slot;
  return r;
}

// Issue the bulk copies of an item: the state into sbuf (on sbar) or the
// window's q/k/v/g rows into ibuf (on ibar).  Called by one thread.
__device__ __forceinline__ void issue_state(const WindowParams& p, const ItemInfo& it,
                                            float* sbuf, uint64_t* sbar) {
  const float* src = p.pool + it.slot * p.slot_stride + (int64_t)it.head * D * D;
  mbar_arrive_expect_tx(sbar, STATE_BYTES);
  // two 32 KB pieces keep each copy well inside one bulk transaction
  bulk_g2s(sbuf, src, STATE_BYTES / 2, sbar);
  bulk_g2s(sbuf + D * D / 2, src + D * D / 2, STATE_BYTES / 2, sbar);
}

__device__ __forceinline__ void issue_inputs(const WindowParams& p, const ItemInfo& it,
                                             __nv_bfloat16* ibuf, uint64_t* ibar) {
  const int hq = it.head / (p.hv / p.hqk);
  mbar_arrive_expect_tx(ibar, it.qlen * 4 * ROW_BYTES);
  for (int t = 0; t < it.qlen; ++t) {
    const int64_t tok = it.qs + t;
    __nv_bfloat16* dst = ibuf + t * 4 * D;
    bulk_g2s(dst + 0 * D, p.q + tok * p.q_st + hq * p.q_sh, ROW_BYTES, ibar);
    bulk_g2s(dst + 1 * D, p.k + tok * p.k_st + hq * p.k_sh, ROW_BYTES, ibar);
    bulk_g2s(dst + 2 * D, p.v + tok * p.v_st + it.head * p.v_sh, ROW_BYTES, ibar);
    bulk_g2s(dst + 3 * D, p.g + tok * p.g_st + it.head * p.g_sh, ROW_BYTES, ibar);
  }
}

// Recursive-halving reduce-scatter of 32 per-lane partial sums: on return
// lane L holds the warp-wide sum of value index L.
__device__ __forceinline__ float reduce_scatter32(float (&x)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int m = 0; m < s; ++m) {
      float send = up ? x[m] : x[m + s];
      float keep = up ? x[m + s] : x[m];
      x[m] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return x[0];
}

template <bool VERIFY>
__device__ void run_item(const WindowParams& p, const ItemInfo& it, float (&S)[16][4],
                         const __nv_bfloat16* ibuf, int warp, int lane) {
  const int h = it.head;
  const float a = p.has_gate ? __expf(p.A_log[h]) : 0.f;
  float dtb[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.has_gate) {
    float4 d4 = *reinterpret_cast<const float4*>(p.dt_bias + h * D + 4 * lane);
    dtb[0] = d4.x; dtb[1] = d4.y; dtb[2] = d4.z; dtb[3] = d4.w;
  }
  const int row_l = lane & 15;
  const int vrow = 16 * warp + row_l;
  for (int t = 0; t < it.qlen; ++t) {
    const int64_t tok = it.qs + t;
    const __nv_bfloat16* rowp = ibuf + t * 4 * D;
    float qv[4], kv[4], gv[4];
    load_bf16x4(rowp + 0 * D + 4 * lane, qv);
    load_bf16x4(rowp + 1 * D + 4 * lane, kv);
    load_bf16x4(rowp + 3 * D + 4 * lane, gv);
    const float vval = bf2f(rowp[2 * D + vrow]);
    const float blog = bf2f(p.beta[tok * p.b_st + h * p.b_sh]);
    const float sq = warp_sum(qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3]);
    const float sk = warp_sum(kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3]);
    const float rq = rsqrtf(sq + 1e-6f) * p.scale;
    const float rk = rsqrtf(sk + 1e-6f);
    float kh[4], dec[4], pk[4], pq[4];
    float kq = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float qh = qv[j] * rq;
      kh[j] = kv[j] * rk;
      const float gate = p.has_gate ? p.lower_bound * sigmoidf_(a * (gv[j] + dtb[j])) : gv[j];
      dec[j] = __expf(gate);
      pk[j] = dec[j] * kh[j];
      pq[j] = dec[j] * qh;
      kq += kh[j] * qh;
    }
    kq = warp_sum(kq);
    const float beta = sigmoidf_(blog);
    float part[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      part[i] = S[i][0] * pk[0] + S[i][1] * pk[1] + S[i][2] * pk[2] + S[i][3] * pk[3];
      part[16 + i] = S[i][0] * pq[0] + S[i][1] * pq[1] + S[i][2] * pq[2] + S[i][3] * pq[3];
    }
    const float mine = reduce_scatter32(part, lane);
    const float U = beta * (vval - mine);              // meaningful on lanes < 16
    const float Urow = __shfl_sync(0xffffffffu, U, row_l);
    if (lane >= 16) {
      const float o = mine + Urow * kq;
      p.out[(tok * p.hv + h) * D + vrow] = __float2bfloat16_rn(o);
    } else if (VERIFY) {
      p.corr[(((int64_t)it.request * p.hv + h) * p.window + t) * D + vrow] = U;
    }
    if (VERIFY && warp == 0) {
      // kg record: raw k (its query/key head) then raw g, as loaded
      __nv_bfloat16* dst = p.kg + (((int64_t)it.request * p.hv + h) * p.window + t) * 2 * D;
      *reinterpret_cast<uint2*>(dst + 4 * lane) =
          *reinterpret_cast<const uint2*>(rowp + 1 * D + 4 * lane);
      *reinterpret_cast<uint2*>(dst + D + 4 * lane) =
          *reinterpret_cast<const uint2*>(rowp + 3 * D + 4 * lane);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float Ui = __shfl_sync(0xffffffffu, U, i);
#pragma unroll
      for (int j = 0; j < 4; ++j) S[i][j] = fmaf(S[i][j], dec[j], kh[j] * Ui);
    }
  }
}

template <bool VERIFY>
__global__ void __launch_bounds__(WIN_THREADS, 1) kda_window_kernel(const WindowParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* sbuf[2] = {reinterpret_cast<float*>(smem_raw),
                    reinterpret_cast<float*>(smem_raw + STATE_BYTES)};
  __nv_bfloat16* ibuf[2] = {
      reinterpret_cast<__nv_bfloat16*>(smem_raw + 2 * STATE_BYTES),
      reinterpret_cast<__nv_bfloat16*>(smem_raw + 2 * STATE_BYTES + IN_BYTES)};
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + 2 * STATE_BYTES + 2 * IN_BYTES);
  uint64_t* sbar = bars;      // [2]
  uint64_t* ibar = bars + 2;  // [2]
  __shared__ int s_next;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = p.n_req * p.hv;
  const int ctas = gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Scheduling.  Decode: static stride.  Verify: tickets (first item is the
  // CTA's own; ticket t names item t + ctas).
  auto take = [&](void) -> int {
    int t = atomicAdd(p.counter, 1);
    if (t == items - 1) atomicExch(p.counter, 0);
    return t + ctas;
  };
  int cur = blockIdx.x;
  int nxt;
  if (tid == 0) s_next = VERIFY ? take() : cur + ctas;
  __syncthreads();
  nxt = s_next;
  __syncthreads();

  // prefetch the first two items
  if (tid == 0) {
    int its[2] = {cur, nxt};
    for (int b = 0; b < 2; ++b) {
      if (its[b] < items) {
        ItemInfo ii = item_info(p, its[b]);
        if (ii.work) {
          issue_state(p, ii, sbuf[b], &sbar[b]);
          issue_inputs(p, ii, ibuf[b], &ibar[b]);
        }
      }
    }
  }
  uint32_t sphase[2] = {0u, 0u}, iphase[2] = {0u, 0u};
  int b = 0;
  while (cur < items) {
    // the item after next (its ticket is taken while this item runs)
    int nn = items;
    if (tid == 0) {
      if (nxt < items) s_next = VERIFY ? take() : nxt + ctas;
      else s_next = items;
    }
    const ItemInfo it = item_info(p, cur);
    bool ok = true;
    float S[16][4];
    if (it.work) {
      ok = mbar_wait_bounded(&sbar[b], sphase[b], p.err);
      ok = ok && mbar_wait_bounded(&ibar[b], iphase[b], p.err);
      sphase[b] ^= 1u;
      iphase[b] ^= 1u;
      if (ok) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float4 x = *reinterpret_cast<const float4*>(sbuf[b] + (16 * warp + i) * D + 4 * lane);
          S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
        }
      }
    }
    // all threads: state buffer b read (or unused); the ticket is published
    if (__syncthreads_or(!ok)) {
      // a copy never landed (error word set): wait, bounded, for the copies
      // still in flight into the other buffer before leaving
      if (tid == 0 && nxt < items && item_info(p, nxt).work) {
        mbar_wait_bounded(&sbar[b ^ 1], sphase[b ^ 1], p.err);
        mbar_wait_bounded(&ibar[b ^ 1], iphase[b ^ 1], p.err);
      }
      return;
    }
    nn = s_next;
    const ItemInfo it2 = nn < items ? item_info(p, nn) : ItemInfo{};
    if (tid == 0 && nn < items && it2.work) issue_state(p, it2, sbuf[b], &sbar[b]);
    if (it.work) {
      run_item<VERIFY>(p, it, S, ibuf[b], warp, lane);
      if (!VERIFY) {
        float* dst = p.pool + it.slot * p.slot_stride + (int64_t)it.head * D * D;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          *reinterpret_cast<float4*>(dst + (16 * warp + i) * D + 4 * lane) =
              make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
      }
    } else if (it.zero) {
      for (int e = tid; e < it.qlen * D; e += WIN_THREADS) {
        const int t = e / D, c = e - t * D;
        p.out[((int64_t)(it.qs + t) * p.hv + it.head) * D + c] = __float2bfloat16_rn(0.f);
      }
    }
    if (tid == 0 && it.bad) set_error(p.err, ERR_INDEX);
    __syncthreads();  // input buffer b consumed
    if (tid == 0 && nn < items && it2.work) issue_inputs(p, it2, ibuf[b], &ibar[b]);
    cur = nxt;
    nxt = nn;
    b ^= 1;
  }
}

// Host-side launchers (called from the API layer after validation).
int launch_window(const WindowParams& p, bool verify, cudaStream_t stream) {
  static int num_sms = 0;
  if (num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(kda_window_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         WIN_SMEM);
    cudaFuncSetAttribute(kda_window_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         WIN_SMEM);
  }
  const int items = p.n_req * p.hv;
  if (items == 0) return 0;
  const int grid = items < num_sms ? items : num_sms;
  trace_begin(verify ? "kda_verify_window" : "kda_decode_window", stream);
  if (verify)
    kda_window_kernel<true><<<grid, WIN_THREADS, WIN_SMEM, stream>>>(p);
  else
    kda_window_kernel<false><<<grid, WIN_THREADS, WIN_SMEM, stream>>>(p);
  trace_end(stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace kda
