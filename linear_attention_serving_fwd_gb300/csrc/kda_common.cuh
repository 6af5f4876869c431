// Shared device helpers for the KDA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int D = 128;      // head dimension, K = V
constexpr int CHUNK = 64;   // prefill chunk length
constexpr int MAX_WINDOW = 8;

// Error bits of the per-device error word.
constexpr unsigned ERR_INDEX = 1u;    // bad slot / length seen by a kernel
constexpr unsigned ERR_TIMEOUT = 2u;  // a bounded wait expired
constexpr unsigned ERR_RANGE = 4u;    // a prefill without gate parameters met a log decay outside [-10.5, 0]

// Bounded waits: every mbarrier / flag spin gives up after WAIT_NS of wall
// time (read from %globaltimer every 64 rounds) or WAIT_CAP rounds, far
// beyond any legitimate wait.
constexpr uint32_t WAIT_CAP = 1u << 26;
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Kernels report through a pointer to the library's per-device error word
// (passed in their parameters; see the API layer).
__device__ __forceinline__ void set_error(unsigned* err, unsigned bits) { atomicOr(err, bits); }

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Activations are 16-bit storage read through __nv_bfloat16 pointers: bf16,
// or fp16 bits when the call's activations are fp16.
template <bool FP16>
__device__ __forceinline__ float act_f(__nv_bfloat16 x) {
  if constexpr (FP16) {
    return __half2float(*reinterpret_cast<const __half*>(&x));
  } else {
    return __bfloat162float(x);
  }
}
__device__ __forceinline__ float act_f(__nv_bfloat16 x, bool fp16) {
  return fp16 ? act_f<true>(x) : act_f<false>(x);
}
// two fp32 values rounded to the activation type, as 32 bits
template <bool FP16>
__device__ __forceinline__ uint32_t act_pack2(float a, float b) {
  if constexpr (FP16) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}
__device__ __forceinline__ __nv_bfloat16 act_from_f(float x, bool fp16) {
  if (fp16) {
    const __half h = __float2half_rn(x);
    return *reinterpret_cast<const __nv_bfloat16*>(&h);
  }
  return __float2bfloat16_rn(x);
}

// Four consecutive bf16 (8 bytes, 8-byte aligned) to fp32.
__device__ __forceinline__ void load_bf16x4(const __nv_bfloat16* p, float out[4]) {
  uint2 raw = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  out[0] = fa.x; out[1] = fa.y; out[2] = fb.x; out[3] = fb.y;
}
// Two consecutive activations (4 bytes, 4-byte aligned) to fp32.
template <bool FP16>
__device__ __forceinline__ float2 act_f2(const __nv_bfloat16* p) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  if constexpr (FP16) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  } else {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
}

// Four consecutive activations (8 bytes, 8-byte aligned) to fp32.
template <bool FP16>
__device__ __forceinline__ void load_act4(const __nv_bfloat16* p, float out[4]) {
  if constexpr (FP16) {
    uint2 raw = *reinterpret_cast<const uint2*>(p);
    const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    out[0] = fa.x; out[1] = fa.y; out[2] = fb.x; out[3] = fb.y;
  } else {
    load_bf16x4(p, out);
  }
}

// Four fp32 values rounded to bf16 and back (a bf16 state's storage).
__device__ __forceinline__ float4 round_bf16x4(float4 x) {
  const float2 a = __bfloat1622float2(__floats2bfloat162_rn(x.x, x.y));
  const float2 b = __bfloat1622float2(__floats2bfloat162_rn(x.z, x.w));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* p, const float v[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 raw;
  raw.x = *reinterpret_cast<uint32_t*>(&a);
  raw.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = raw;
}

// packed fp32x2 helpers
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ar = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long br = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long cr = *reinterpret_cast<unsigned long long*>(&c);
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(ar), "l"(br), "l"(cr));
  return *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  unsigned long long ar = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long br = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ar), "l"(br));
  return *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long ar = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long br = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ar), "l"(br));
  return *reinterpret_cast<float2*>(&r);
}

// logistic function with the fast (2-ulp) divide; exp(-x) = inf gives 0
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// barrier among ``count`` threads (whole warps) on hardware barrier ``id``
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier among ``count`` threads on hardware barrier ``id`` that also
// returns whether any of them passed ``pred`` true: a uniform decision.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n"
      ".reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n"
      "}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
  return x;
}

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy (TMA) wrappers.  Addresses are shared-state-space
// 32-bit addresses obtained with __cvta_generic_to_shared.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Test (and briefly wait for) the completion of ``phase``: the thread may be
// suspended until the phase completes or about 0.1 ms pass, so waiting
// threads park instead of spinning.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase), "r"(100000u)
      : "memory");
  return ok != 0;
}

// Bring ``bytes`` (a multiple of 16, 16-byte aligned) at ``src`` into L2
// without waiting.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Non-blocking test of ``phase``: the fast path before a parking wait.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

// Wait for ``phase`` of ``bar`` to complete, at most WAIT_CAP rounds.  On
// expiry sets ERR_TIMEOUT and returns false; the caller must stop using the
// guarded buffer.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase, unsigned* err) {
  if (mbar_test_wait(bar, phase)) return true;
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < WAIT_CAP; ++i) {
    if (mbar_try_wait(bar, phase)) return true;
    const uint64_t t = globaltimer_ns();
    if (t0 == 0) t0 = t;
    else if (t - t0 > WAIT_NS) break;
  }
  set_error(err, ERR_TIMEOUT);
  return false;
}

// 1-D bulk copy global -> shared, completing ``bytes`` of tx on ``bar``.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy shared -> global (bulk async-group completion).
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(dst), "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// 16-byte asynchronous copy global -> shared (Ampere-style cp.async);
// src_bytes = 0 fills the destination with zeros without reading.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (bulk copies, tensor cores) and order async-proxy results before generic
// reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace kda
