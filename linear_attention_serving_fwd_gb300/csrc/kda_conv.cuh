// Width-4 depthwise causal conv + SiLU over the raw q/k/v projection bands,
// in the precision of the vLLM kimi_k3 verify page's conv path (KdaTcVerify,
// step 2): with bf16 taps each product is rounded to bf16 and the four are
// added in fp32 in tap order; with fp32 taps the sum is an fp32 fma chain;
// the SiLU output is rounded to bf16 by the caller.
//   y_t = SiLU(w_0 x_{t-3} + w_1 x_{t-2} + w_2 x_{t-1} + w_3 x_t)
#pragma once

#include "kda_params.cuh"

namespace kda {

__device__ __forceinline__ float4 conv_taps(const ConvParams& cv, int64_t ch) {
  if (cv.w_f32) return *reinterpret_cast<const float4*>(static_cast<const float*>(cv.w) + ch * 4);
  float t[4];
  load_bf16x4(static_cast<const __nv_bfloat16*>(cv.w) + ch * 4, t);
  return make_float4(t[0], t[1], t[2], t[3]);
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// SiLU in fp32 (a fast divide: for acc below about -88 the denominator is
// inf and the result -0, the value rounded to bf16 anyway).
__device__ __forceinline__ float silu(float acc) { return __fdividef(acc, 1.f + __expf(-acc)); }

// SiLU of the conv sum over x0 (oldest) .. x3 (current), in fp32.
__device__ __forceinline__ float conv_silu(bool f32, float4 w, float x0, float x1, float x2, float x3) {
  float acc;
  if (f32) {
    acc = fmaf(x0, w.x, 0.f);
    acc = fmaf(x1, w.y, acc);
    acc = fmaf(x2, w.z, acc);
    acc = fmaf(x3, w.w, acc);
  } else {  // bf16 x bf16 products are exact in fp32 before the rounding
    acc = bf16_round(x0 * w.x);
    acc = acc + bf16_round(x1 * w.y);
    acc = acc + bf16_round(x2 * w.z);
    acc = acc + bf16_round(x3 * w.w);
  }
  return silu(acc);
}

// Two consecutive outputs of one channel from five window values x[0..4]
// (x[0] oldest: the first output reads x[0..3], the second x[1..4]),
// rounded to a bf16 pair.  With bf16 taps the products are bf16 pair
// multiplies (each the exact product rounded to bf16) summed as fp32 pairs
// in tap order; with fp32 taps an fp32 pair fma chain.
__device__ __forceinline__ __nv_bfloat162 conv_silu2(bool f32, float4 w, const __nv_bfloat16* x) {
  float2 acc;
  if (f32) {
    float xf[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) xf[i] = __bfloat162float(x[i]);
    acc = fmul2(make_float2(xf[0], xf[1]), make_float2(w.x, w.x));
    acc = ffma2(make_float2(xf[1], xf[2]), make_float2(w.y, w.y), acc);
    acc = ffma2(make_float2(xf[2], xf[3]), make_float2(w.z, w.z), acc);
    acc = ffma2(make_float2(xf[3], xf[4]), make_float2(w.w, w.w), acc);
  } else {
    const float wt[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 pr = __hmul2(__halves2bfloat162(x[j], x[j + 1]), __float2bfloat162_rn(wt[j]));
      const float2 pf = __bfloat1622float2(pr);
      acc = j == 0 ? pf : fadd2(acc, pf);
    }
  }
  return __floats2bfloat162_rn(silu(acc.x), silu(acc.y));
}

// Raw projection channel ch of token 0, and its token stride, for the q / k
// / v bands of a parameter block with q, k, v pointers and strides.
template <class P>
__device__ __forceinline__ const __nv_bfloat16* conv_source(const P& p, int64_t ch, int64_t& tok_stride) {
  const int64_t qk = (int64_t)p.hqk * D;
  if (ch < qk) {
    tok_stride = p.q_st;
    return p.q + (ch / D) * p.q_sh + ch % D;
  }
  if (ch < 2 * qk) {
    ch -= qk;
    tok_stride = p.k_st;
    return p.k + (ch / D) * p.k_sh + ch % D;
  }
  ch -= 2 * qk;
  tok_stride = p.v_st;
  return p.v + (ch / D) * p.v_sh + ch % D;
}

// The three channels of (v-head h, column c): q and k of h's q/k head, v of h.
__device__ __forceinline__ void conv_channels(int hqk, int hv, int h, int c, int64_t ch[3]) {
  const int hq = h / (hv / hqk);
  ch[0] = (int64_t)hq * D + c;
  ch[1] = (int64_t)hqk * D + (int64_t)hq * D + c;
  ch[2] = 2 * (int64_t)hqk * D + (int64_t)h * D + c;
}

}  // namespace kda
