// Decode (in place) and speculative verify (read only) over a paged fp32 or
// bf16 state cache, window Q <= 8 tokens per request.
//
// Design (memory bound: each (request, head) moves its 64 KB V-first state
// once in, and for decode once out):
//  * persistent grid; every state and q/k/v/g row arrives by 1-D bulk async
//    copies (TMA engine) completing on mbarriers, and the next item's
//    per-token scalars (beta, A_log, dt_bias) are loaded a step ahead;
//  * two layouts by the state rows WR a thread holds (rows of S^T, 8 key
//    channels each, so the state lives in 8 WR registers per thread and a
//    row's dot products reduce over the 16 lanes of a half warp):
//    - WR = 8 (verify, decode of windows longer than one token, and
//      one-token decode on bf16 states): 256 threads, two CTAs per SM, one
//      64 KB state buffer each; the next item's state streams in while one
//      runs (for one-token bf16 decode the buffer holds two states and the
//      one two items ahead streams in), and the other CTA's work hides each
//      item's latency chain; decode stores the new state from registers;
//    - WR = 4 (one-token decode on fp32 states, which only moves bytes): 512 threads,
//      one CTA per SM, two state buffers (the state two items ahead streams
//      in) and a third for the write-back, which leaves by two bulk stores
//      so no thread waits on it;
//  * with a [request, step] slot table decode reads the row of the last
//    accepted token and also stores the state after each earlier token of
//    the window, from registers;
//  * per item, warp t < qlen first turns token t's raw rows into the vectors
//    every warp needs (L2-normalised k^ and q~, exp(gate), their products)
//    in shared memory, once;
//  * per token, the 2 WR dot products of a half warp (its rows with
//    exp(gate) * k^ and with exp(gate) * q~) are reduced by one
//    recursive-halving reduce-scatter, after which a lane (WR = 8) or lane
//    pair (WR = 4) holds one row's correction U or output; products use
//    packed fp32x2 FMAs.
// Token order inside the window follows the recurrence exactly:
//   S <- diag(e^gate) S;  U = beta (v - S^T k^);  S <- S + k^ U^T;  o = S^T q~
// computed as U = beta (v - S_old^T (e^gate * k^)),
//             o = S_old^T (e^gate * q~) + U (k^ . q~),  S = e^gate * S_old + k^ U^T.
// Verify with a conv (the verify page's conv path): q, k, v are the raw
// projection bands; each token's rows are first convolved (width 4, SiLU)
// with the history at the accepted column, by two warps (half the channels
// each), the outputs replace the raw rows, and a small kernel afterwards
// rolls the conv state.
// Verify (the vLLM kimi_k3 CuTeDSL verify page, KdaTcVerify) additionally
// writes corr = U_t and kg = (raw k_t, raw g_t) and never writes the state;
// its persistent scheduler takes tickets from a caller-zeroed counter and the
// taker of the last ticket resets it.
#include "kda_conv.cuh"
#include "kda_params.cuh"

namespace kda {

// Two thread layouts, by the state rows WR a thread holds (8 key channels
// each): WR = 8, 256 threads, two CTAs per SM with one state buffer each;
// WR = 4, 512 threads, one CTA per SM with two state buffers and a
// write-back staging buffer (one-token decode on fp32 states, where the
// kernel only moves bytes and wants the most of them in flight).
template <int WR>
__host__ __device__ constexpr int win_threads() { return 2048 / WR; }
constexpr int STATE_BYTES = D * D * 4;                // 65536
constexpr int ROW_BYTES = D * 2;                      // one bf16 row of 128

// Verify with a staged conv (token-major conv state, bf16 taps): each item's
// taps (3 bands x 128 channels x 4) and the three history positions of its
// 3 bands, per input buffer.
constexpr int CONV_TAPS_BYTES = 3 * 1024;
constexpr int CONV_STAGE_BYTES = CONV_TAPS_BYTES + 9 * 256;

struct __align__(128) WinSmem {
  float state[D * D];  // the next item's state streams in while this one runs
  __nv_bfloat16 in[2][MAX_WINDOW * 4 * D];
  float tp[MAX_WINDOW][D];    // e^gate * k^
  float tr[MAX_WINDOW][D];    // e^gate * q~
  float tdec[MAX_WINDOW][D];  // e^gate
  float tkh[MAX_WINDOW][D];   // k^
  float tbeta[MAX_WINDOW];
  float tkq[MAX_WINDOW];      // k^ . q~
  float cc[4][4], dd[4][4];   // windowed solve: coupling scalars c_tj, d_tj
  uint64_t sbar[2], ibar[2];
  int next;
};

// Past the block: WR = 8, the two conv staging areas; WR = 4, the second
// state buffer and the write-back staging buffer.
constexpr int EXTRA_WR8 = 2 * CONV_STAGE_BYTES;
constexpr int EXTRA_WR4 = 2 * STATE_BYTES;
// two WR = 8 CTAs (each with its 1 KB reserve) share an SM's 228 KB
static_assert(2 * (sizeof(WinSmem) + EXTRA_WR8 + 1024) <= 228 * 1024, "two window CTAs per SM");
static_assert(sizeof(WinSmem) + EXTRA_WR4 <= 227 * 1024, "a WR = 4 window CTA fits");

struct ItemInfo {
  int request, head, qs, qlen;
  int64_t slot;   // the row the state is read from
  int64_t wslot;  // decode: the row the state after the last token goes to (< 0: none)
  bool work;  // state is loaded and tokens processed
  bool zero;  // padding request: write zero outputs
  bool bad;   // out-of-range slot or window length (reported, treated as padding)
};

__device__ __forceinline__ ItemInfo item_info(const WindowParams& p, int item) {
  ItemInfo r;
  r.request = item / p.hv;
  r.head = item - r.request * p.hv;
  r.qs = p.query_start[r.request];
  r.qlen = p.query_start[r.request + 1] - r.qs;
  const bool bad_len = r.qlen < 0 || r.qlen > p.window;
  bool bad_slot;
  if (p.step_slots) {
    // slot table: read the column of the last accepted token, write a row
    // per token (window <= step_stride, so columns t < qlen exist)
    const int32_t* row = p.step_slots + (int64_t)r.request * p.step_stride;
    const int col = p.n_accepted ? p.n_accepted[r.request] - 1 : 0;
    const bool bad_col = col < 0 || col >= p.step_stride;
    r.slot = bad_col ? -1 : row[col];
    r.wslot = (!bad_len && r.qlen > 0) ? row[r.qlen - 1] : -1;
    bad_slot = bad_col || r.slot >= p.n_slots;
    if (!bad_len)
      for (int t = 0; t < r.qlen; ++t) bad_slot |= row[t] >= p.n_slots;
  } else {
    r.slot = p.slots[r.request];
    r.wslot = r.slot;
    bad_slot = r.slot >= p.n_slots;
  }
  if (p.conv.state && r.slot >= 0 && !bad_len && r.qlen > 0) {
    // verify with a conv: its history sits at positions accepted-1 .. +1
    const int first = p.conv.accepted[r.request] - 1;
    bad_slot |= first < 0 || first + 3 > p.conv.positions || r.slot >= p.conv.rows;
  }
  r.work = !bad_len && !bad_slot && r.slot >= 0 && r.qlen > 0;
  r.zero = !bad_len && r.qlen > 0 && !r.work;
  r.bad = bad_len || bad_slot;
  return r;
}

// A state row's bytes: fp32 or bf16 elements.
template <bool SBF16>
__device__ __forceinline__ unsigned char* state_row(const WindowParams& p, int64_t slot, int head) {
  return static_cast<unsigned char*>(p.pool) + (slot * p.slot_stride + (int64_t)head * D * D) * (SBF16 ? 2 : 4);
}

// Bulk copy of an item's state into sbuf on sbar (one thread).
template <bool SBF16>
__device__ __forceinline__ void issue_state(const WindowParams& p, const ItemInfo& it, float* sbuf,
                                            uint64_t* sbar) {
  constexpr int bytes = SBF16 ? STATE_BYTES / 2 : STATE_BYTES;
  const unsigned char* src = state_row<SBF16>(p, it.slot, it.head);
  mbar_arrive_expect_tx(sbar, bytes);
  bulk_g2s(sbuf, src, bytes / 2, sbar);
  bulk_g2s(reinterpret_cast<unsigned char*>(sbuf) + bytes / 2, src + bytes / 2, bytes / 2, sbar);
}

// Four state values of row ``row``, channels ``chan``.. from a staged state
// (fp32, or bf16 widened).
template <bool SBF16>
__device__ __forceinline__ float4 state_ld4(const float* sbuf, int row, int chan) {
  if constexpr (SBF16) {
    float v[4];
    load_bf16x4(reinterpret_cast<const __nv_bfloat16*>(sbuf) + row * D + chan, v);
    return make_float4(v[0], v[1], v[2], v[3]);
  } else {
    return *reinterpret_cast<const float4*>(sbuf + row * D + chan);
  }
}
template <bool SBF16>
__device__ __forceinline__ void state_st4(void* base, int row, int chan, float4 x) {
  if constexpr (SBF16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + row * D + chan) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + row * D + chan) = x;
  }
}

// The window's q/k/v/g rows, one bulk copy per lane of the calling warp (and,
// for a staged conv, the item's taps and history into ``stage``).
__device__ __forceinline__ void issue_inputs(const WindowParams& p, const ItemInfo& it,
                                             __nv_bfloat16* ibuf, uint64_t* ibar, int lane,
                                             unsigned char* stage = nullptr) {
  const int hq = it.head / (p.hv / p.hqk);
  const bool conv = stage != nullptr;
  constexpr int tap_bytes = D * 8;  // bf16 taps
  if (lane == 0) mbar_arrive_expect_tx(ibar, it.qlen * 4 * ROW_BYTES + (conv ? 3 * tap_bytes + 9 * 256 : 0));
  __syncwarp();
  if (conv && lane < 12) {
    int64_t ch[3];
    conv_channels(p.hqk, p.hv, it.head, 0, ch);
    if (lane < 3) {
      const unsigned char* w = static_cast<const unsigned char*>(p.conv.w) + ch[lane] * (tap_bytes / D);
      bulk_g2s(stage + lane * 1024, w, tap_bytes, ibar);
    } else {
      const int x = (lane - 3) / 3, i = (lane - 3) % 3;
      const int first = p.conv.accepted[it.request] - 1;
      const __nv_bfloat16* h = p.conv.state + it.slot * p.conv.row_st + (int64_t)(first + i) * p.conv.pos_st + ch[x];
      bulk_g2s(stage + CONV_TAPS_BYTES + (x * 3 + i) * 256, h, 256, ibar);
    }
  }
  if (lane < 4 * it.qlen) {
    const int t = lane >> 2, which = lane & 3;
    const int64_t tok = it.qs + t;
    const __nv_bfloat16* src;
    if (which == 0) src = p.q + tok * p.q_st + hq * p.q_sh;
    else if (which == 1) src = p.k + tok * p.k_st + hq * p.k_sh;
    else if (which == 2) src = p.v + tok * p.v_st + it.head * p.v_sh;
    else src = p.g + tok * p.g_st + it.head * p.g_sh;
    bulk_g2s(ibuf + (t * 4 + which) * D, src, ROW_BYTES, ibar);
  }
}

// Token ``t = warp``'s scalars, loaded a step before their use: beta (lane 0),
// dt_bias for the lane's 4 channels and A_log of the head.
struct TokenScalars {
  float4 dt;
  float alog;
  __nv_bfloat16 beta;
};
__device__ __forceinline__ TokenScalars load_token_scalars(const WindowParams& p, const ItemInfo& it, int t,
                                                           int lane) {
  TokenScalars r;
  r.dt = make_float4(0.f, 0.f, 0.f, 0.f);
  r.alog = 0.f;
  r.beta = __float2bfloat16(0.f);
  if (it.work && t < it.qlen) {
    if (p.has_gate) {
      r.dt = *reinterpret_cast<const float4*>(p.dt_bias + it.head * D + 4 * lane);
      r.alog = p.A_log[it.head];
    }
    r.beta = p.beta[(it.qs + t) * p.b_st + it.head * p.b_sh];
  }
  return r;
}

// Token t's per-channel vectors, computed by one warp (lane = 4 channels).
template <bool FP16>
__device__ __forceinline__ void token_vectors(const WindowParams& p, WinSmem& s, const TokenScalars& ts,
                                              const __nv_bfloat16* rowp, int t, int lane) {
  float qv[4], kv[4], gv[4];
  load_act4<FP16>(rowp + 0 * D + 4 * lane, qv);
  load_act4<FP16>(rowp + 1 * D + 4 * lane, kv);
  load_act4<FP16>(rowp + 3 * D + 4 * lane, gv);
  const float sq = warp_sum(qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3]);
  const float sk = warp_sum(kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3]);
  const float rq = rsqrtf(sq + 1e-6f) * p.scale, rk = rsqrtf(sk + 1e-6f);
  const float a = p.has_gate ? __expf(ts.alog) : 0.f;
  const float dt[4] = {ts.dt.x, ts.dt.y, ts.dt.z, ts.dt.w};
  float kh[4], dec[4], pk[4], pq[4], kq = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float qh = qv[j] * rq;
    kh[j] = kv[j] * rk;
    const float gate = p.has_gate ? p.lower_bound * sigmoidf_(a * (gv[j] + dt[j])) : gv[j];
    dec[j] = __expf(gate);
    pk[j] = dec[j] * kh[j];
    pq[j] = dec[j] * qh;
    kq += kh[j] * qh;
  }
  kq = warp_sum(kq);
  *reinterpret_cast<float4*>(&s.tp[t][4 * lane]) = make_float4(pk[0], pk[1], pk[2], pk[3]);
  *reinterpret_cast<float4*>(&s.tr[t][4 * lane]) = make_float4(pq[0], pq[1], pq[2], pq[3]);
  *reinterpret_cast<float4*>(&s.tdec[t][4 * lane]) = make_float4(dec[0], dec[1], dec[2], dec[3]);
  *reinterpret_cast<float4*>(&s.tkh[t][4 * lane]) = make_float4(kh[0], kh[1], kh[2], kh[3]);
  if (lane == 0) {
    s.tkq[t] = kq;
    s.tbeta[t] = sigmoidf_(act_f<FP16>(ts.beta));
  }
}

// Verify with a conv: the conv + SiLU outputs of token t for channels c, c+1
// of each band (q and k of the head's q/k head, v of the head), from the
// window's raw rows and, for the taps before the window, the history at
// positions accepted-1 .. accepted+1 of the slot's conv row; rounded to bf16
// (the convolved rows replace the raw bf16 rows).  The 2 qlen units (token,
// half of the 128 channels) are spread over the CTA's warps.
__device__ __forceinline__ void conv_unit(const WindowParams& p, const ItemInfo& it,
                                          const __nv_bfloat16* ibuf, const unsigned char* stage, int t,
                                          int c, uint32_t (&y)[3]) {
  const ConvParams& cv = p.conv;
  const int first = cv.accepted[it.request] - 1;
  int64_t ch[3];
  conv_channels(p.hqk, p.hv, it.head, c, ch);
  const __nv_bfloat16* hist = cv.state + it.slot * cv.row_st;
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    float2 win[4];  // tap j reads token t - 3 + j
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tt = t - 3 + j;
      if (tt >= 0) {
        win[j] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(ibuf + (tt * 4 + x) * D + c));
      } else if (cv.bulk) {  // staged history position first + 3 + tt
        win[j] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(
            reinterpret_cast<const __nv_bfloat16*>(stage + CONV_TAPS_BYTES + (x * 3 + 3 + tt) * 256) + c));
      } else {
        const __nv_bfloat16* h = hist + (int64_t)(first + 3 + tt) * cv.pos_st;
        win[j] = make_float2(bf2f(h[ch[x] * cv.ch_st]), bf2f(h[(ch[x] + 1) * cv.ch_st]));
      }
    }
    float ye[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float4 w;
      if (cv.bulk) {  // staged bf16 taps
        float t4[4];
        load_bf16x4(reinterpret_cast<const __nv_bfloat16*>(stage + x * 1024 + (c + e) * 8), t4);
        w = make_float4(t4[0], t4[1], t4[2], t4[3]);
      } else {
        w = conv_taps(cv, ch[x] + e);
      }
      ye[e] = conv_silu(cv.w_f32, w, e ? win[0].y : win[0].x, e ? win[1].y : win[1].x,
                        e ? win[2].y : win[2].x, e ? win[3].y : win[3].x);
    }
    const __nv_bfloat162 yy = __floats2bfloat162_rn(ye[0], ye[1]);
    y[x] = *reinterpret_cast<const uint32_t*>(&yy);
  }
}

// Thread (warp w, lane L) holds state rows v = 2 WR w + WR (L / 16) + i, i < WR,
// at key channels 4 (L % 16) + 64 j .. + 3, j < 2, as float2 pairs S[i][jj]
// (jj = 2 j, 2 j + 1): each row's dot products reduce over the 16 lanes of
// a half warp, and a half warp's 16-byte accesses to a row are contiguous.
template <int WR>
__device__ __forceinline__ int win_row(int warp, int lane, int i) { return 2 * WR * warp + WR * (lane >> 4) + i; }
__device__ __forceinline__ int win_chan(int lane, int j) { return 4 * (lane & 15) + 64 * j; }

__device__ __forceinline__ void load_pairs(const float* vec, int lane, float2 (&v)[4]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float4 x4 = *reinterpret_cast<const float4*>(vec + win_chan(lane, j));
    v[2 * j] = make_float2(x4.x, x4.y);
    v[2 * j + 1] = make_float2(x4.z, x4.w);
  }
}

template <bool VERIFY, bool SBF16, bool FP16, int WR>
__device__ __forceinline__ void run_tokens(const WindowParams& p, WinSmem& s, const ItemInfo& it,
                                           float2 (&S)[WR][4], const __nv_bfloat16* ibuf, int warp,
                                           int lane) {
  const int h = it.head;
  // the 2 WR sums of a half warp are reduce-scattered over its 16 lanes by
  // L halvings (lane bits 3, 2, ..), then the last 4 - L lane bits summed
  constexpr int L = WR == 8 ? 4 : 3;
  constexpr int SH = 4 - L;
  const int e = (lane & 15) >> SH;           // the sum this lane ends with
  const int ei = e & (WR - 1);               // its row; e < WR: row . (e^gate k^), else row . (e^gate q~)
  const bool lead = (lane & ((1 << SH) - 1)) == 0;
  const int my_row = win_row<WR>(warp, lane, ei);
  const int half = lane & 16;
  for (int t = 0; t < it.qlen; ++t) {
    const int64_t tok = it.qs + t;
    float2 pv[4], rv[4];
    load_pairs(s.tp[t], lane, pv);
    load_pairs(s.tr[t], lane, rv);
    const float beta = s.tbeta[t], kq = s.tkq[t];
    // x[i]: row i . (e^gate k^), x[WR + i]: row i . (e^gate q~), over this lane's 8 channels
    float x[2 * WR];
#pragma unroll
    for (int i = 0; i < WR; ++i) {
      float2 a = fmul2(S[i][0], pv[0]), bq = fmul2(S[i][0], rv[0]);
#pragma unroll
      for (int jj = 1; jj < 4; ++jj) {
        a = ffma2(S[i][jj], pv[jj], a);
        bq = ffma2(S[i][jj], rv[jj], bq);
      }
      x[i] = a.x + a.y;
      x[WR + i] = bq.x + bq.y;
    }
#pragma unroll
    for (int lvl = 0; lvl < L; ++lvl) {
      const int m = 8 >> lvl, n = WR >> lvl;
      const bool up = (lane & m) != 0;
#pragma unroll
      for (int q = 0; q < WR; ++q) {
        if (q < n) {
          const float send = up ? x[q] : x[q + n], keep = up ? x[q + n] : x[q];
          x[q] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
    }
    if (SH) x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
    const float mine = x[0];
    // sums e < WR: U of row e; e >= WR: the output of row e - WR
    const float vval = act_f<FP16>(ibuf[t * 4 * D + 2 * D + my_row]);
    const float U = beta * (vval - mine);
    const float Urow = __shfl_sync(0xffffffffu, U, half | (ei << SH));
    if (lead) {
      if (e >= WR) {
        p.out[(tok * p.hv + h) * D + my_row] = act_from_f(mine + Urow * kq, FP16);
      } else if (VERIFY) {
        p.corr[(((int64_t)it.request * p.hv + h) * p.window + t) * D + my_row] = U;
      }
    }
    if (VERIFY && warp == 0) {
      __nv_bfloat16* dst = p.kg + (((int64_t)it.request * p.hv + h) * p.window + t) * 2 * D;
      const __nv_bfloat16* rowp = ibuf + t * 4 * D;
      *reinterpret_cast<uint2*>(dst + 4 * lane) = *reinterpret_cast<const uint2*>(rowp + 1 * D + 4 * lane);
      *reinterpret_cast<uint2*>(dst + D + 4 * lane) = *reinterpret_cast<const uint2*>(rowp + 3 * D + 4 * lane);
    }
    float2 dv[4], kv[4];
    load_pairs(s.tdec[t], lane, dv);
    load_pairs(s.tkh[t], lane, kv);
#pragma unroll
    for (int i = 0; i < WR; ++i) {
      const float Ui = __shfl_sync(0xffffffffu, U, half | (i << SH));
      const float2 uu = make_float2(Ui, Ui);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) S[i][jj] = ffma2(S[i][jj], dv[jj], fmul2(kv[jj], uu));
    }
    if constexpr (SBF16) {
      // a bf16 state is stored after every token: the next token starts
      // from the rounded state, as repeated single-token decode would
#pragma unroll
      for (int i = 0; i < WR; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float4 r = round_bf16x4(make_float4(S[i][2 * j].x, S[i][2 * j].y, S[i][2 * j + 1].x,
                                                    S[i][2 * j + 1].y));
          S[i][2 * j] = make_float2(r.x, r.y);
          S[i][2 * j + 1] = make_float2(r.z, r.w);
        }
    }
    if (!VERIFY && p.step_slots && t + 1 < it.qlen) {
      // slot table: the state after token t, unless its row is the last
      // token's (written after the window) or disabled
      const int64_t row = p.step_slots[(int64_t)it.request * p.step_stride + t];
      if (row >= 0 && row != it.wslot) {
        void* dst = state_row<SBF16>(p, row, h);
#pragma unroll
        for (int i = 0; i < WR; ++i)
#pragma unroll
          for (int j = 0; j < 2; ++j)
            state_st4<SBF16>(dst, win_row<WR>(warp, lane, i), win_chan(lane, j),
                             make_float4(S[i][2 * j].x, S[i][2 * j].y, S[i][2 * j + 1].x, S[i][2 * j + 1].y));
      }
    }
  }
}

// Step (1) of the windowed solve, run by warp t < Q for token t: k^_t, q~_t,
// e^{gate_t} and beta_t into shared memory, and verify's kg record.
template <bool FP16>
__device__ __forceinline__ void window_vectors(const WindowParams& p, WinSmem& s, const ItemInfo& it,
                                               const __nv_bfloat16* ibuf, const TokenScalars& ts, int warp,
                                               int lane) {
  constexpr int QW = 4;
  const int h = it.head;
  float* z = &s.tp[0][0];
  float* khat = z;
  float* qtil = z + QW * D;
  float* dec = z + 2 * QW * D;
  const int c0 = 4 * lane;
  const __nv_bfloat16* rowp = ibuf + warp * 4 * D;
  float qv[4], kv[4], gv[4];
  load_act4<FP16>(rowp + 0 * D + c0, qv);
  load_act4<FP16>(rowp + 1 * D + c0, kv);
  load_act4<FP16>(rowp + 3 * D + c0, gv);
  const float sq = warp_sum(qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3]);
  const float sk = warp_sum(kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3]);
  const float rq = rsqrtf(sq + 1e-6f) * p.scale, rk = rsqrtf(sk + 1e-6f);
  const float a = p.has_gate ? __expf(ts.alog) : 0.f;
  const float dt[4] = {ts.dt.x, ts.dt.y, ts.dt.z, ts.dt.w};
  float dv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float gate = p.has_gate ? p.lower_bound * sigmoidf_(a * (gv[j] + dt[j])) : gv[j];
    dv[j] = __expf(gate);
  }
  *reinterpret_cast<float4*>(khat + warp * D + c0) = make_float4(kv[0] * rk, kv[1] * rk, kv[2] * rk, kv[3] * rk);
  *reinterpret_cast<float4*>(qtil + warp * D + c0) = make_float4(qv[0] * rq, qv[1] * rq, qv[2] * rq, qv[3] * rq);
  *reinterpret_cast<float4*>(dec + warp * D + c0) = make_float4(dv[0], dv[1], dv[2], dv[3]);
  if (lane == 0) s.tbeta[warp] = sigmoidf_(act_f<FP16>(ts.beta));
  {  // verify's kg record
    __nv_bfloat16* dst = p.kg + (((int64_t)it.request * p.hv + h) * p.window + warp) * 2 * D;
    *reinterpret_cast<uint2*>(dst + c0) = *reinterpret_cast<const uint2*>(rowp + 1 * D + c0);
    *reinterpret_cast<uint2*>(dst + D + c0) = *reinterpret_cast<const uint2*>(rowp + 3 * D + c0);
  }
}

// Windowed solve of a 2..4-token window on an fp32 state (the verify page's
// probes and coupling scalars, KdaTcVerify steps 2-4), replacing the token
// loop: with P_t = prod_{i <= t} e^{gate_i} and r_{j,t} = k^_j prod_{i=j+1..t}
// e^{gate_i} (per channel, every factor <= 1),
//   U_t = beta_t (v_t - S0^T (P_t k^_t) - sum_{j<t} (r_{j,t} . k^_t) U_j)
//   o_t = S0^T (P_t q~_t) + sum_{j<=t} (r_{j,t} . q~_t) U_j
//   S   = P_{Q-1} * S0 + sum_j r_{j,Q-1} U_j^T
// so the state is read once for all 2Q probes and updated once.  Every
// thread takes part (it holds the state rows of the token loop's layout).
template <bool FP16, int WR>
__device__ __forceinline__ void window_solve(const WindowParams& p, WinSmem& s, const ItemInfo& it,
                                             const float2 (&S)[WR][4], const __nv_bfloat16* ibuf,
                                             const TokenScalars& ts, int tid, int warp, int lane,
                                             bool vectors_done) {
  constexpr int QW = 4;
  const int Q = it.qlen, h = it.head;
  float* z = &s.tp[0][0];  // tp, tr, tdec, tkh: 16 KB of contiguous scratch
  float* khat = z;
  float* qtil = z + QW * D;
  float* dec = z + 2 * QW * D;
  float* kG = z + 3 * QW * D;
  float* qG = z + 4 * QW * D;
  float* pb = z;           // S0^T kG_t, over khat once the couplings are done
  float* pa = z + QW * D;  // S0^T qG_t, over qtil
  const int c0 = 4 * lane;
  // (1) vectors: done by the caller unless a conv rewrote the rows after
  // the state was loaded
  if (!vectors_done) {
    if (warp < Q) window_vectors<FP16>(p, s, it, ibuf, ts, warp, lane);
    __syncthreads();
  }
  // (2) warp j: P_j k^_j, P_j q~_j (zero for j >= Q), the chain r_{j,t}
  // and its couplings with tokens t >= j
  if (warp < QW) {
    const int j = warp;
    if (j < Q) {
      float4 P = make_float4(1.f, 1.f, 1.f, 1.f);
      for (int i = 0; i <= j; ++i) {
        const float4 d4 = *reinterpret_cast<const float4*>(dec + i * D + c0);
        P = make_float4(P.x * d4.x, P.y * d4.y, P.z * d4.z, P.w * d4.w);
      }
      const float4 kj = *reinterpret_cast<const float4*>(khat + j * D + c0);
      const float4 qj = *reinterpret_cast<const float4*>(qtil + j * D + c0);
      *reinterpret_cast<float4*>(kG + j * D + c0) = make_float4(kj.x * P.x, kj.y * P.y, kj.z * P.z, kj.w * P.w);
      *reinterpret_cast<float4*>(qG + j * D + c0) = make_float4(qj.x * P.x, qj.y * P.y, qj.z * P.z, qj.w * P.w);
      float4 r = kj;
      float dsum[QW], csum[QW];
#pragma unroll
      for (int t = 0; t < QW; ++t) {
        dsum[t] = 0.f;
        csum[t] = 0.f;
        if (t >= j && t < Q) {
          if (t > j) {
            const float4 d4 = *reinterpret_cast<const float4*>(dec + t * D + c0);
            r = make_float4(r.x * d4.x, r.y * d4.y, r.z * d4.z, r.w * d4.w);
          }
          const float4 qt = *reinterpret_cast<const float4*>(qtil + t * D + c0);
          const float4 kt = *reinterpret_cast<const float4*>(khat + t * D + c0);
          dsum[t] = r.x * qt.x + r.y * qt.y + r.z * qt.z + r.w * qt.w;
          csum[t] = r.x * kt.x + r.y * kt.y + r.z * kt.z + r.w * kt.w;
        }
      }
      // reduce-scatter of the 8 sums over the warp (halving by lane bits
      // 4, 3, 2, then bits 1 and 0 summed): lanes with bits 1..0 clear end
      // with entry 4 b4 + 2 b3 + b2 of (d_0..d_3, c_0..c_3)
      float y[8] = {dsum[0], dsum[1], dsum[2], dsum[3], csum[0], csum[1], csum[2], csum[3]};
#pragma unroll
      for (int lvl = 0; lvl < 3; ++lvl) {
        const int m = 16 >> lvl, n = 4 >> lvl;
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < n) {
            const float send = up ? y[q] : y[q + n], keep = up ? y[q + n] : y[q];
            y[q] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
      }
      y[0] += __shfl_xor_sync(0xffffffffu, y[0], 2);
      y[0] += __shfl_xor_sync(0xffffffffu, y[0], 1);
      if ((lane & 3) == 0) {
        const int e = 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
        if (e < 4)
          s.dd[e][j] = y[0];
        else
          s.cc[e - 4][j] = y[0];
      }
    } else {
      *reinterpret_cast<float4*>(kG + j * D + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(qG + j * D + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();
  // (3) probes, keys then queries, TP = 16 / WR tokens at a time: this
  // thread's WR rows x 8 channels against those tokens' vectors;
  // x[TP i + u] = row i . vec_{t0+u}, reduce-scattered over the half warp's
  // 16 lanes (halving by lane bits 3, 2, 1, 0) so that lane e of the half
  // ends with x[e]: row e / TP, token t0 + e % TP
  constexpr int TP = 16 / WR;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float* vecs = half == 0 ? kG : qG;
#pragma unroll
    for (int t0 = 0; t0 < QW; t0 += TP) {
      float x[16];
#pragma unroll
      for (int u = 0; u < TP; ++u) {
        float2 w2[4];
        load_pairs(vecs + (t0 + u) * D, lane, w2);
#pragma unroll
        for (int i = 0; i < WR; ++i) {
          float2 acc = fmul2(S[i][0], w2[0]);
#pragma unroll
          for (int jj = 1; jj < 4; ++jj) acc = ffma2(S[i][jj], w2[jj], acc);
          x[TP * i + u] = acc.x + acc.y;
        }
      }
#pragma unroll
      for (int lvl = 0; lvl < 4; ++lvl) {
        const int m = 8 >> lvl;
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (q < m) {
            const float send = up ? x[q] : x[q + m], keep = up ? x[q + m] : x[q];
            x[q] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
      }
      const int e = lane & 15;
      (half == 0 ? pb : pa)[(t0 + e % TP) * D + win_row<WR>(warp, lane, e / TP)] = x[0];
    }
  }
  __syncthreads();
  // (4) thread v < 128: forward substitution for row v, outputs, records
  if (tid < D) {
    const int v = tid;
    float u[QW];
#pragma unroll
    for (int t = 0; t < QW; ++t) {
      u[t] = 0.f;
      if (t < Q) {
        float acc = act_f<FP16>(ibuf[t * 4 * D + 2 * D + v]) - pb[t * D + v];
#pragma unroll
        for (int j = 0; j < t; ++j) acc -= s.cc[t][j] * u[j];
        u[t] = s.tbeta[t] * acc;
        float o = pa[t * D + v];
#pragma unroll
        for (int j = 0; j <= t; ++j) o += s.dd[t][j] * u[j];
        p.out[((int64_t)(it.qs + t) * p.hv + h) * D + v] = act_from_f(o, FP16);
        p.corr[(((int64_t)it.request * p.hv + h) * p.window + t) * D + v] = u[t];
      }
    }
  }
}

// The staging area of input buffer b for a verify with a staged conv, else
// none.
__device__ __forceinline__ unsigned char* conv_stage(const WindowParams& p, unsigned char* extra, int b) {
  return (p.conv.state && p.conv.bulk) ? extra + b * CONV_STAGE_BYTES : nullptr;
}

// WR = 8: one fp32 state buffer, the next item's state streams in while an
// item runs; a bf16 state is half the size, so for one-token windows (which
// wait on bytes, not on compute) the buffer holds two and the state two
// items ahead streams in.  The new state is stored from registers.
// WR = 4 (decode only): two state buffers, the state two items ahead streams
// in, and the new state leaves through a staging buffer by two bulk stores,
// so no thread waits on its write.
template <bool VERIFY, bool SBF16, bool FP16, int WR, int NBUF>
__global__ void __launch_bounds__(win_threads<WR>(), WR == 8 ? 2 : 1) kda_window_kernel(const WindowParams p) {
  static_assert(WR == 8 || (WR == 4 && !VERIFY), "verify runs the WR = 8 layout");
  static_assert((WR == 4 && NBUF == 2) || (WR == 8 && (NBUF == 1 || SBF16)), "state buffers of the layout");
  constexpr int THREADS = win_threads<WR>();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  WinSmem& s = *reinterpret_cast<WinSmem*>(smem_raw);
  unsigned char* const extra = smem_raw + sizeof(WinSmem);
  auto state_buf = [&](int k) -> float* {
    if (WR == 8) return s.state + k * (D * D / 2);  // bf16: two states in the buffer
    return k == 0 ? s.state : reinterpret_cast<float*>(extra);
  };
  float* const sout = reinterpret_cast<float*>(extra + STATE_BYTES);  // WR = 4
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = p.n_req * p.hv;
  const int ctas = gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.sbar[i], 1);
      mbar_init(&s.ibar[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Scheduling.  Decode: static stride.  Verify: tickets (the first item is
  // the CTA's own; ticket t names item t + ctas; the last ticket resets).
  auto take = [&](void) -> int {
    const int t = atomicAdd(p.counter, 1);
    if (t == items - 1) atomicExch(p.counter, 0);
    return t + ctas;
  };
  int cur = blockIdx.x;
  if (tid == 0) s.next = VERIFY ? take() : cur + ctas;
  __syncthreads();
  int nxt = s.next;
  __syncthreads();

  if (warp == 0) {
    const int its[2] = {cur, nxt};
    for (int b = 0; b < 2; ++b) {
      if (its[b] < items) {
        const ItemInfo ii = item_info(p, its[b]);
        if (ii.work) {
          if (b < NBUF && lane == 0) issue_state<SBF16>(p, ii, state_buf(b), &s.sbar[b]);
          issue_inputs(p, ii, s.in[b], &s.ibar[b], lane, conv_stage(p, extra, b));
        }
      }
    }
  }
  ItemInfo it = cur < items ? item_info(p, cur) : ItemInfo{};
  ItemInfo itn = nxt < items ? item_info(p, nxt) : ItemInfo{};
  TokenScalars ts = load_token_scalars(p, it, warp, lane);
  uint32_t sphase[2] = {0u, 0u}, iphase[2] = {0u, 0u};
  int b = 0, sb = 0;  // input buffer, state buffer
  bool stored = false;  // WR = 4: a bulk state store is in flight from sout
  while (cur < items) {
    // verify's ticket is drawn here and resolved at the end of the item: a
    // comparison on it here would hold warp 0, and the barrier below every
    // warp, for the atomic's round trip
    int ticket = 0;
    if (VERIFY && tid == 0 && nxt < items) ticket = atomicAdd(p.counter, 1);
    // decode's static stride names the item after next here, so its
    // metadata loads run under the state wait (with two state buffers its
    // state is issued right after the barrier below)
    int nn = items;
    ItemInfo it2 = ItemInfo{};
    if (!VERIFY) {
      nn = nxt < items ? nxt + ctas : items;
      if (nn < items) it2 = item_info(p, nn);
    }
    bool ok = true;
    const bool conv = VERIFY && !FP16 && p.conv.state != nullptr;  // conv: bf16 activations only
    // verify of 2..4 tokens on an fp32 state: the windowed solve (measured
    // faster than the token loop there; for decode, whose update and
    // write-back follow, the token loop measured faster)
    const bool windowed = VERIFY && !SBF16 && it.qlen >= 2 && it.qlen <= 4;
    float2 S[WR][4];
    uint32_t yc[2][3];  // verify with a conv: this warp's units' bf16 outputs
    if (it.work) {
      ok = mbar_wait_bounded(&s.sbar[sb], sphase[sb], p.err);
      ok = mbar_wait_bounded(&s.ibar[b], iphase[b], p.err) && ok;
      sphase[sb] ^= 1u;
      iphase[b] ^= 1u;
      if (ok) {
        if (conv) {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int u = warp + 8 * k;  // unit: token u / 2, channels 64 (u % 2) + 2 lane ..
            if (u < 2 * it.qlen)
              conv_unit(p, it, s.in[b], extra + b * CONV_STAGE_BYTES, u >> 1, 64 * (u & 1) + 2 * lane, yc[k]);
          }
        } else if (warp < it.qlen) {
          // token t's vectors by warp t, beside the other warps' state loads
          if (!windowed) token_vectors<FP16>(p, s, ts, s.in[b] + warp * 4 * D, warp, lane);
          else if constexpr (VERIFY) window_vectors<FP16>(p, s, it, s.in[b], ts, warp, lane);
        }
        const float* sbuf = state_buf(sb);
#pragma unroll
        for (int i = 0; i < WR; ++i)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float4 x4 = state_ld4<SBF16>(sbuf, win_row<WR>(warp, lane, i), win_chan(lane, j));
            S[i][2 * j] = make_float2(x4.x, x4.y);
            S[i][2 * j + 1] = make_float2(x4.z, x4.w);
          }
      }
    }
    // the state buffer read, token vectors written
    if (__syncthreads_or(!ok)) {
      // a copy never landed (error word set): wait, bounded, for the copies
      // still in flight (the next item's inputs, and with two state buffers
      // its state), then leave
      if (tid == 0 && itn.work) {
        mbar_wait_bounded(&s.ibar[b ^ 1], iphase[b ^ 1], p.err);
        if (NBUF == 2) mbar_wait_bounded(&s.sbar[sb ^ 1], sphase[sb ^ 1], p.err);
      }
      if (WR == 4 && tid == 0) bulk_wait<0>();
      return;
    }
    // the freed state buffer takes the state of the item after this one (one
    // buffer) or of the item after that (two buffers)
    if (tid == 0) {
      const ItemInfo& ahead = NBUF == 2 ? it2 : itn;
      if (ahead.work) issue_state<SBF16>(p, ahead, state_buf(sb), &s.sbar[sb]);
    }
    if (conv && it.work) {
      // every raw row has been read: the conv outputs replace them, then
      // the token vectors come from the convolved rows
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int u = warp + 8 * k;
        if (u < 2 * it.qlen)
#pragma unroll
          for (int x = 0; x < 3; ++x)
            *reinterpret_cast<uint32_t*>(s.in[b] + ((u >> 1) * 4 + x) * D + 64 * (u & 1) + 2 * lane) = yc[k][x];
      }
      __syncthreads();
      if (!windowed) {
        if (warp < it.qlen) token_vectors<FP16>(p, s, ts, s.in[b] + warp * 4 * D, warp, lane);
        __syncthreads();
      }
    }
    // the next item's scalars, used a step from now
    const TokenScalars ts_next = load_token_scalars(p, itn, warp, lane);
    if (it.work) {
      bool solved = false;
      if constexpr (VERIFY) {
        if (windowed) {
          window_solve<FP16, WR>(p, s, it, S, s.in[b], ts, tid, warp, lane, !conv);
          solved = true;
        }
      }
      if (!solved) run_tokens<VERIFY, SBF16, FP16, WR>(p, s, it, S, s.in[b], warp, lane);
      if (!VERIFY && it.wslot >= 0) {
        // the state after the last token: WR = 8 straight from registers,
        // each half warp storing 256 contiguous bytes of a row per
        // instruction; WR = 4 into sout, once the previous item's bulk store
        // has read it (issued a whole item ago)
        void* dst = state_row<SBF16>(p, it.wslot, it.head);
        if (WR == 4) {
          if (tid == 0 && stored) bulk_wait_read<0>();
          __syncthreads();
          dst = sout;
        }
#pragma unroll
        for (int i = 0; i < WR; ++i)
#pragma unroll
          for (int j = 0; j < 2; ++j)
            state_st4<SBF16>(dst, win_row<WR>(warp, lane, i), win_chan(lane, j),
                             make_float4(S[i][2 * j].x, S[i][2 * j].y, S[i][2 * j + 1].x, S[i][2 * j + 1].y));
        if (WR == 4) fence_proxy_async_smem();
      }
    } else if (it.zero) {
      for (int e = tid; e < it.qlen * D; e += THREADS) {
        const int t = e / D, c = e - t * D;
        p.out[((int64_t)(it.qs + t) * p.hv + it.head) * D + c] = __float2bfloat16_rn(0.f);
      }
    }
    if (tid == 0 && it.bad) set_error(p.err, ERR_INDEX);
    if (VERIFY && tid == 0) {
      int v = items;
      if (nxt < items) {
        if (ticket == items - 1) atomicExch(p.counter, 0);
        v = ticket + ctas;
      }
      s.next = v;
    }
    __syncthreads();  // input buffer b and the token vectors consumed, sout written, the ticket published
    if (VERIFY) {
      nn = s.next;
      it2 = nn < items ? item_info(p, nn) : ItemInfo{};
    }
    if (WR == 4 && !VERIFY && tid == 0 && it.work && it.wslot >= 0) {
      constexpr int bytes = SBF16 ? STATE_BYTES / 2 : STATE_BYTES;
      unsigned char* dst = state_row<SBF16>(p, it.wslot, it.head);
      const unsigned char* src = reinterpret_cast<const unsigned char*>(sout);
      bulk_s2g(dst, src, bytes / 2);
      bulk_s2g(dst + bytes / 2, src + bytes / 2, bytes / 2);
      bulk_commit();
      stored = true;
    }
    // verify: the last warp, which no window of up to four tokens gives a
    // token, so that its wait on the item's metadata delays no token warp
    if (warp == (VERIFY ? THREADS / 32 - 1 : 1) && nn < items && it2.work) issue_inputs(p, it2, s.in[b], &s.ibar[b], lane, conv_stage(p, extra, b));
    ts = ts_next;
    cur = nxt;
    nxt = nn;
    it = itn;
    itn = it2;
    b ^= 1;
    if (NBUF == 2) sb ^= 1;
  }
  if (WR == 4 && tid == 0) bulk_wait<0>();  // the last state store has landed
}

// Host-side launcher (called from the API layer after validation).
template <bool VERIFY, bool SBF16, bool FP16, int WR, int NBUF = (WR == 4 ? 2 : 1)>
static void launch_window_t(const WindowParams& p, int num_sms, cudaStream_t stream) {
  constexpr int smem = (int)sizeof(WinSmem) + (WR == 8 ? EXTRA_WR8 : EXTRA_WR4);
  static uint64_t done = 0;
  once_per_device(done, [](int) {
    cudaFuncSetAttribute(kda_window_kernel<VERIFY, SBF16, FP16, WR, NBUF>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(kda_window_kernel<VERIFY, SBF16, FP16, WR, NBUF>,
                         cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  });
  const int items = p.n_req * p.hv;
  const int slots = (WR == 8 ? 2 : 1) * num_sms;  // resident CTAs
  const int grid = items < slots ? items : slots;
  kda_window_kernel<VERIFY, SBF16, FP16, WR, NBUF><<<grid, win_threads<WR>(), smem, stream>>>(p);
}

int launch_window(const WindowParams& p, bool verify, cudaStream_t stream) {
  static int sms[64] = {0};
  static uint64_t done = 0;
  once_per_device(done, [&](int d) { cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d); });
  int dev = 0;
  cudaGetDevice(&dev);
  const int num_sms = sms[dev & 63] > 0 ? sms[dev & 63] : 152;
  const int items = p.n_req * p.hv;
  if (items == 0) return 0;
  // decode of one token per request moves the state with almost no
  // compute: fp32 states run the WR = 4 layout, which keeps the most bytes
  // in flight; bf16 states (half the bytes) run two CTAs per SM with two
  // states in each CTA's buffer (0.157 -> 0.136 ms for 8192 items).  Longer
  // windows and verify overlap two CTAs' compute with one buffer each (WR = 8).
  const int variant = (verify ? 4 : 0) + (p.state_bf16 ? 2 : 0) + (p.in_fp16 ? 1 : 0);
  const bool one = !verify && p.window == 1;
  trace_begin(verify ? "kda_verify_window" : "kda_decode_window", stream);
  switch (one ? 8 + variant : variant) {
    case 0: launch_window_t<false, false, false, 8>(p, num_sms, stream); break;
    case 1: launch_window_t<false, false, true, 8>(p, num_sms, stream); break;
    case 2: launch_window_t<false, true, false, 8>(p, num_sms, stream); break;
    case 3: launch_window_t<false, true, true, 8>(p, num_sms, stream); break;
    case 4: launch_window_t<true, false, false, 8>(p, num_sms, stream); break;
    case 5: launch_window_t<true, false, true, 8>(p, num_sms, stream); break;
    case 6: launch_window_t<true, true, false, 8>(p, num_sms, stream); break;
    case 7: launch_window_t<true, true, true, 8>(p, num_sms, stream); break;
    case 8: launch_window_t<false, false, false, 4>(p, num_sms, stream); break;
    case 9: launch_window_t<false, false, true, 4>(p, num_sms, stream); break;
    case 10: launch_window_t<false, true, false, 8, 2>(p, num_sms, stream); break;
    default: launch_window_t<false, true, true, 8, 2>(p, num_sms, stream); break;
  }
  trace_end(stream);
  // verify with a conv: every history has been read, roll the conv state
  if (verify && p.conv.state && launch_conv_roll(p, stream) != 0) return -1;
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace kda
