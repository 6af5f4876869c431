// Speculative-decode commit: rebuild a request's state after its accepted
// prefix from the records kda_verify wrote (the vLLM kimi_k3 verify page's
// corr / kg records, KdaTcVerify), in place in the state pool.
//
// With the window's tokens t = 1..a accepted, the recurrence unrolls to
//   S_a = diag(e^{L_a}) S_0 + sum_{t <= a} diag(e^{L_a - L_t}) k^_t U_t^T
// (K x V; L_t = gate cumsum per key channel, k^_t = k_t / |k_t|, U_t the
// recorded correction), so the state moves once in and once out and the
// window's tokens need no recomputation of their corrections.
//
// Design (memory bound, like decode): persistent grid, one CTA (16 warps)
// per SM; each (request, head) item's 64 KB state and its records arrive by
// bulk copies on mbarriers, two items in flight; warp t prepares token t's
// k^_t and gate, 128 threads form e^{L_a} and the weights e^{L_a - L_t} k^_t,
// and every thread applies the rank-a update to its 4 rows x 8 channels in
// registers; the new state goes back through a staging buffer and two bulk
// stores.
#include "kda_params.cuh"

namespace kda {

constexpr int CM_THREADS = 512;
constexpr int CM_STATE = D * D * 4;  // 65536

struct __align__(128) CommitSmem {
  float state[2][D * D];
  float sout[D * D];
  float corr[2][MAX_WINDOW * D];
  __nv_bfloat16 kg[2][MAX_WINDOW * 2 * D];
  float w[MAX_WINDOW][D];     // k^_t, then e^{L_a - L_t} k^_t
  float gate[MAX_WINDOW][D];
  float ela[D];               // e^{L_a}
  uint64_t sbar[2], rbar[2];
};
static_assert(sizeof(CommitSmem) <= 227 * 1024, "commit kernel shared memory");

struct CommitItem {
  int request, head, a;
  int64_t slot;
  bool work;  // rows to rebuild
  bool bad;   // out-of-range slot or accepted count (reported, skipped)
};

__device__ __forceinline__ CommitItem commit_item(const CommitParams& p, int item) {
  CommitItem r;
  r.request = item / p.hv;
  r.head = item - r.request * p.hv;
  r.slot = p.slots[r.request];
  r.a = p.accepted[r.request];
  r.bad = r.a < 0 || r.a > p.window || r.slot >= p.n_slots;
  r.work = !r.bad && r.slot >= 0 && r.a > 0;
  return r;
}

// A state row's bytes (fp32 or bf16 elements).
template <bool SBF16>
__device__ __forceinline__ unsigned char* cm_state_row(const CommitParams& p, int64_t slot, int head) {
  return static_cast<unsigned char*>(p.pool) + (slot * p.slot_stride + (int64_t)head * D * D) * (SBF16 ? 2 : 4);
}

template <bool SBF16>
__device__ __forceinline__ void commit_issue_state(const CommitParams& p, const CommitItem& it, float* sbuf,
                                                   uint64_t* bar) {
  constexpr int bytes = SBF16 ? CM_STATE / 2 : CM_STATE;
  const unsigned char* src = cm_state_row<SBF16>(p, it.slot, it.head);
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(sbuf, src, bytes / 2, bar);
  bulk_g2s(reinterpret_cast<unsigned char*>(sbuf) + bytes / 2, src + bytes / 2, bytes / 2, bar);
}

__device__ __forceinline__ void commit_issue_records(const CommitParams& p, const CommitItem& it, float* cbuf,
                                                     __nv_bfloat16* kbuf, uint64_t* bar) {
  const int64_t row = ((int64_t)it.request * p.hv + it.head) * p.window;
  mbar_arrive_expect_tx(bar, it.a * (D * 4 + 2 * D * 2));
  bulk_g2s(cbuf, p.corr + row * D, it.a * D * 4, bar);
  bulk_g2s(kbuf, p.kg + row * 2 * D, it.a * 2 * D * 2, bar);
}

// thread (warp w, lane L): state rows 8w + 4 (L / 16) + i, key channels
// 4 (L % 16) + 64 j .. + 3 (as in the window kernel)
__device__ __forceinline__ int cm_row(int warp, int lane, int i) { return 8 * warp + 4 * (lane >> 4) + i; }
__device__ __forceinline__ int cm_chan(int lane, int j) { return 4 * (lane & 15) + 64 * j; }

template <bool SBF16>
__global__ void __launch_bounds__(CM_THREADS, 1) kda_commit_kernel(const CommitParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  CommitSmem& s = *reinterpret_cast<CommitSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = p.n_req * p.hv, stride = gridDim.x;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.sbar[i], 1);
      mbar_init(&s.rbar[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  int cur = blockIdx.x, nxt = cur + stride;
  CommitItem it = cur < items ? commit_item(p, cur) : CommitItem{};
  CommitItem itn = nxt < items ? commit_item(p, nxt) : CommitItem{};
  if (tid == 0) {
    if (it.work) {
      commit_issue_state<SBF16>(p, it, s.state[0], &s.sbar[0]);
      commit_issue_records(p, it, s.corr[0], s.kg[0], &s.rbar[0]);
    }
    if (itn.work) {
      commit_issue_state<SBF16>(p, itn, s.state[1], &s.sbar[1]);
      commit_issue_records(p, itn, s.corr[1], s.kg[1], &s.rbar[1]);
    }
  }
  uint32_t sphase[2] = {0u, 0u}, rphase[2] = {0u, 0u};
  int b = 0;
  bool stored = false;  // a bulk state store is in flight from sout (thread 0)
  while (cur < items) {
    const int nn = nxt + stride;
    const CommitItem it2 = nn < items ? commit_item(p, nn) : CommitItem{};
    bool ok = true;
    float2 S[4][4];
    if (it.work) {
      ok = mbar_wait_bounded(&s.sbar[b], sphase[b], p.err);
      ok = mbar_wait_bounded(&s.rbar[b], rphase[b], p.err) && ok;
      sphase[b] ^= 1u;
      rphase[b] ^= 1u;
      if (ok) {
        if (warp < it.a) {
          // token t = warp: k^_t and the gate, lane = 4 channels
          const __nv_bfloat16* kr = s.kg[b] + warp * 2 * D;
          float kv[4], gv[4];
          if (p.kg_fp16) {
            load_act4<true>(kr + 4 * lane, kv);
            load_act4<true>(kr + D + 4 * lane, gv);
          } else {
            load_act4<false>(kr + 4 * lane, kv);
            load_act4<false>(kr + D + 4 * lane, gv);
          }
          const float rk = rsqrtf(warp_sum(kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3]) +
                                  1e-6f);
          float4 dt = make_float4(0.f, 0.f, 0.f, 0.f);
          float a_h = 0.f;
          if (p.has_gate) {
            dt = *reinterpret_cast<const float4*>(p.dt_bias + it.head * D + 4 * lane);
            a_h = __expf(p.A_log[it.head]);
          }
          const float dtv[4] = {dt.x, dt.y, dt.z, dt.w};
          float gt[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            gt[j] = p.has_gate ? p.lower_bound * sigmoidf_(a_h * (gv[j] + dtv[j])) : gv[j];
          *reinterpret_cast<float4*>(&s.w[warp][4 * lane]) =
              make_float4(kv[0] * rk, kv[1] * rk, kv[2] * rk, kv[3] * rk);
          *reinterpret_cast<float4*>(&s.gate[warp][4 * lane]) = make_float4(gt[0], gt[1], gt[2], gt[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float4 x4;
            if constexpr (SBF16) {
              float v[4];
              load_bf16x4(reinterpret_cast<const __nv_bfloat16*>(s.state[b]) + cm_row(warp, lane, i) * D +
                              cm_chan(lane, j), v);
              x4 = make_float4(v[0], v[1], v[2], v[3]);
            } else {
              x4 = *reinterpret_cast<const float4*>(s.state[b] + cm_row(warp, lane, i) * D + cm_chan(lane, j));
            }
            S[i][2 * j] = make_float2(x4.x, x4.y);
            S[i][2 * j + 1] = make_float2(x4.z, x4.w);
          }
      }
    }
    if (__syncthreads_or(!ok)) {
      // a copy never landed (error word set): wait, bounded, for the copies
      // into the other buffer and for the last state store before leaving
      if (tid == 0 && itn.work) {
        mbar_wait_bounded(&s.sbar[b ^ 1], sphase[b ^ 1], p.err);
        mbar_wait_bounded(&s.rbar[b ^ 1], rphase[b ^ 1], p.err);
      }
      if (tid == 0) bulk_wait<0>();
      return;
    }
    // state buffer b is in registers: the item after next may stream into it
    if (tid == 0 && it2.work) commit_issue_state<SBF16>(p, it2, s.state[b], &s.sbar[b]);
    if (it.work) {
      if (tid < D) {
        // channel k = tid: L_t, e^{L_a} and the weights e^{L_a - L_t} k^_t
        float L[MAX_WINDOW];
        float acc = 0.f;
#pragma unroll
        for (int t = 0; t < MAX_WINDOW; ++t) {
          if (t < it.a) acc += s.gate[t][tid];
          L[t] = acc;
        }
        s.ela[tid] = __expf(acc);
#pragma unroll
        for (int t = 0; t < MAX_WINDOW; ++t)
          if (t < it.a) s.w[t][tid] *= __expf(acc - L[t]);
      }
      __syncthreads();
      // S_a = e^{L_a} S_0 + sum_t (e^{L_a - L_t} k^_t) U_t^T, per row i (value v)
      float2 e2[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float4 e4 = *reinterpret_cast<const float4*>(&s.ela[cm_chan(lane, j)]);
        e2[2 * j] = make_float2(e4.x, e4.y);
        e2[2 * j + 1] = make_float2(e4.z, e4.w);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) S[i][jj] = fmul2(S[i][jj], e2[jj]);
      for (int t = 0; t < it.a; ++t) {
        float2 w2[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float4 w4 = *reinterpret_cast<const float4*>(&s.w[t][cm_chan(lane, j)]);
          w2[2 * j] = make_float2(w4.x, w4.y);
          w2[2 * j + 1] = make_float2(w4.z, w4.w);
        }
        const float4 u4 = *reinterpret_cast<const float4*>(&s.corr[b][t * D + cm_row(warp, lane, 0)]);
        const float u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 uu = make_float2(u[i], u[i]);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) S[i][jj] = ffma2(w2[jj], uu, S[i][jj]);
        }
      }
      // sout is free once the previous item's bulk store has read it
      if (tid == 0 && stored) bulk_wait_read<0>();
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int o = cm_row(warp, lane, i) * D + cm_chan(lane, j);
          if constexpr (SBF16) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(S[i][2 * j].x, S[i][2 * j].y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(S[i][2 * j + 1].x, S[i][2 * j + 1].y);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(s.sout) + o) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
          } else {
            *reinterpret_cast<float4*>(s.sout + o) =
                make_float4(S[i][2 * j].x, S[i][2 * j].y, S[i][2 * j + 1].x, S[i][2 * j + 1].y);
          }
        }
      fence_proxy_async_smem();
    }
    if (tid == 0 && it.bad) set_error(p.err, ERR_INDEX);
    __syncthreads();  // records of buffer b consumed, sout written
    if (tid == 0) {
      if (it.work) {
        constexpr int bytes = SBF16 ? CM_STATE / 2 : CM_STATE;
        unsigned char* dst = cm_state_row<SBF16>(p, it.slot, it.head);
        const unsigned char* src = reinterpret_cast<const unsigned char*>(s.sout);
        bulk_s2g(dst, src, bytes / 2);
        bulk_s2g(dst + bytes / 2, src + bytes / 2, bytes / 2);
        bulk_commit();
        stored = true;
      }
      if (it2.work) commit_issue_records(p, it2, s.corr[b], s.kg[b], &s.rbar[b]);
    }
    cur = nxt;
    nxt = nn;
    it = itn;
    itn = it2;
    b ^= 1;
  }
  if (tid == 0) bulk_wait<0>();  // the last state store has landed
}

int launch_commit(const CommitParams& p, cudaStream_t stream) {
  static int sms[64] = {0};
  static uint64_t done = 0;
  int dev = 0;
  once_per_device(done, [&](int d) {
    cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d);
    cudaFuncSetAttribute(kda_commit_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(CommitSmem));
    cudaFuncSetAttribute(kda_commit_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(CommitSmem));
  });
  cudaGetDevice(&dev);
  const int num_sms = sms[dev & 63] > 0 ? sms[dev & 63] : 152;
  const int items = p.n_req * p.hv;
  if (items == 0) return 0;
  const int grid = items < num_sms ? items : num_sms;
  trace_begin("kda_commit", stream);
  if (p.state_bf16)
    kda_commit_kernel<true><<<grid, CM_THREADS, sizeof(CommitSmem), stream>>>(p);
  else
    kda_commit_kernel<false><<<grid, CM_THREADS, sizeof(CommitSmem), stream>>>(p);
  trace_end(stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace kda
