// tcgen05 (5th-generation tensor core) building blocks for sm_103a, written
// as inline PTX: TMEM allocation, shared-memory matrix descriptors for the
// canonical K-major and MN-major no-swizzle layouts and the 128-byte
// swizzled K-major one, kind::f16 / kind::tf32 MMAs with fp32 accumulation
// in TMEM, commit to an mbarrier, and TMEM loads.
//
// Operand layout used throughout (K-major, no swizzle).  A matrix of R rows
// (M or N) by K 16-bit elements is stored as core matrices of 8 rows x 16
// bytes (8 elements):
//     byte(row, k) = (k / 8) * (R * 16) + (row / 8) * 128 + (row % 8) * 16 + (k % 8) * 2
// i.e. consecutive K groups of 8 are R*16 bytes apart (the descriptor's
// leading-dimension offset) and consecutive 8-row groups 128 bytes apart (its
// stride-dimension offset).  One MMA instruction consumes K = 16, two K groups.
#pragma once

#include <stdint.h>

#include "kda_common.cuh"

namespace kda {
namespace tc {

// byte offset of element (row, k) in a K-major no-swizzle operand of R rows
__host__ __device__ __forceinline__ uint32_t kmajor_offset(uint32_t row, uint32_t k, uint32_t R) {
  return (k >> 3) * (R * 16u) + (row >> 3) * 128u + (row & 7u) * 16u + (k & 7u) * 2u;
}

// Shared-memory matrix descriptor (sm_100 family format): start address,
// leading-dimension byte offset (between K groups), stride-dimension byte
// offset (between 8-row groups), fixed version bits 46-47 = 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  return d;  // base offset 0, lbo mode 0, layout type 0 (no swizzle)
}

// Instruction descriptor of kind::f16 with fp32 accumulation, both operands
// K-major.  ab_bf16 selects bf16 (1) or fp16 (0) for A and B alike.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, uint32_t ab_bf16) {
  return (1u << 4)                 // D format: f32
         | (ab_bf16 << 7)          // A format: f16 = 0, bf16 = 1
         | (ab_bf16 << 10)         // B format
         | ((N >> 3) << 17)        // N / 8
         | ((M >> 4) << 24);       // M / 16
}

// kind::tf32 with fp32 accumulation, both operands K-major (fp32 storage;
// the MMA reads the tf32 part).  One instruction consumes K = 8 (32 bytes).
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// byte offset of element (row, k) of a K-major no-swizzle fp32 operand
__host__ __device__ __forceinline__ uint32_t kmajor_offset32(uint32_t row, uint32_t k, uint32_t R) {
  return (k >> 2) * (R * 16u) + (row >> 3) * 128u + (row & 7u) * 16u + (k & 3u) * 4u;
}

// 128-byte-swizzled K-major fp32 operand of R rows (R % 8 == 0): K blocks of
// 32 elements (128 bytes per row) are R * 128 bytes apart; inside a block,
// rows are 128 bytes apart and the 16-byte chunk c of row r sits at chunk
// c ^ (r % 8).  The block base must be 1024-byte aligned.  A warp storing 32
// consecutive k of one row covers one 128-byte line: bank-conflict free.
__host__ __device__ __forceinline__ uint32_t sw128_offset32(uint32_t row, uint32_t k, uint32_t R) {
  const uint32_t kin = k & 31u;
  return (k >> 5) * (R * 128u) + (row >> 3) * 1024u + (row & 7u) * 128u +
         ((((kin >> 2) ^ (row & 7u)) & 7u) << 4) + (kin & 3u) * 4u;
}

// descriptor of a 128-byte-swizzled K-major operand (8-row groups 1024 bytes apart)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                  // leading offset: unused for swizzled K-major
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;                  // SWIZZLE_128B
  return d;
}

// round an fp32 value to tf32 (nearest, ties away), kept in fp32 storage
__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
// The same rounding on the integer pipe, for finite x below 2^128 - 2^115:
// tf32 keeps 10 of fp32's 23 fraction bits, so adding half of the dropped
// 13-bit field (0x1000) to the sign-magnitude pattern rounds the magnitude
// half up (ties away from zero; a carry correctly bumps the exponent), and
// the mask clears the dropped bits.
__device__ __forceinline__ float to_tf32_int(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// --- TMEM allocation (one full warp executes these) -----------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(smem_dst)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// --- ordering --------------------------------------------------------------
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// --- MMA -------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T, M x N x 16 per instruction.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on ``bar`` when every MMA this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// byte offset of element (row, k) in a K-major no-swizzle operand whose K
// groups are ``lbo`` bytes apart (lbo = R * 16 packs them; a padded lbo keeps
// column-wise stores from different K groups off the same banks)
__host__ __device__ __forceinline__ uint32_t kmajor_offset_lbo(uint32_t row, uint32_t k,
                                                              uint32_t lbo) {
  return (k >> 3) * lbo + (row >> 3) * 128u + (row & 7u) * 16u + (k & 7u) * 2u;
}

// A run of STEPS kind::f16 instructions whose descriptors advance by fixed
// byte steps (a_step, b_step; multiples of 16): the descriptors are built
// once and only their start-address fields move, which keeps the issuing
// thread's work per instruction to two adds.
template <int STEPS>
__device__ __forceinline__ void mma_run(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t a_step,
                                        uint32_t b_step, uint32_t idesc, bool accumulate_first) {
#pragma unroll
  for (int s = 0; s < STEPS; ++s)
    mma_f16(d_tmem, ad + (uint64_t)((s * a_step) >> 4), bd + (uint64_t)((s * b_step) >> 4), idesc,
            (s > 0 || accumulate_first) ? 1u : 0u);
}

// One K-major x K-major product over K elements (K % 16 == 0): A has M rows
// at a_saddr, B has N rows at b_saddr, both in the layout above (B's K groups
// b_lbo bytes apart; 0 = packed, N * 16).
__device__ __forceinline__ void mma_kloop(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr,
                                          uint32_t M, uint32_t N, uint32_t K, uint32_t ab_bf16,
                                          bool accumulate_first, uint32_t b_lbo_bytes = 0) {
  const uint32_t idesc = idesc_f16(M, N, ab_bf16);
  const uint32_t a_lbo = M * 16u, b_lbo = b_lbo_bytes ? b_lbo_bytes : N * 16u;
  for (uint32_t s = 0; s < K / 16u; ++s) {
    const uint64_t ad = smem_desc(a_saddr + s * 2u * a_lbo, a_lbo, 128u);
    const uint64_t bd = smem_desc(b_saddr + s * 2u * b_lbo, b_lbo, 128u);
    mma_f16(d_tmem, ad, bd, idesc, (s > 0 || accumulate_first) ? 1u : 0u);
  }
}

// K-major A times MN-major B over K elements (K % 16 == 0).  B's layout:
//     byte(n, k) = (n / 8) * b_sbo + (k / 8) * b_lbo + (k % 8) * 16 + (n % 8) * 2
// (8 consecutive n contiguous), selected by bit 16 of the instruction
// descriptor; each instruction advances B by two 8-row K groups.
__device__ __forceinline__ void mma_kloop_bmn(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr,
                                              uint32_t M, uint32_t N, uint32_t K, uint32_t b_lbo,
                                              uint32_t b_sbo, bool accumulate_first) {
  const uint32_t idesc = idesc_f16(M, N, 0) | (1u << 16);
  const uint32_t a_lbo = M * 16u;
  for (uint32_t s = 0; s < K / 16u; ++s) {
    const uint64_t ad = smem_desc(a_saddr + s * 2u * a_lbo, a_lbo, 128u);
    const uint64_t bd = smem_desc(b_saddr + s * 2u * b_lbo, b_lbo, b_sbo);
    mma_f16(d_tmem, ad, bd, idesc, (s > 0 || accumulate_first) ? 1u : 0u);
  }
}

// byte offset of element (n, k) of an MN-major 16-bit operand (layout above)
__host__ __device__ __forceinline__ uint32_t mnmajor_offset(uint32_t n, uint32_t k, uint32_t lbo,
                                                           uint32_t sbo) {
  return (n >> 3) * sbo + (k >> 3) * lbo + (k & 7u) * 16u + (n & 7u) * 2u;
}

// Same for fp32 operands on kind::tf32 (K in elements, K % 8 == 0).
__device__ __forceinline__ void mma_kloop_tf32(uint32_t d_tmem, uint32_t a_saddr,
                                               uint32_t b_saddr, uint32_t M, uint32_t N,
                                               uint32_t K, bool accumulate_first) {
  const uint32_t idesc = idesc_tf32(M, N);
  const uint32_t a_lbo = M * 16u, b_lbo = N * 16u;
  for (uint32_t s = 0; s < K / 8u; ++s) {
    const uint64_t ad = smem_desc(a_saddr + s * 2u * a_lbo, a_lbo, 128u);
    const uint64_t bd = smem_desc(b_saddr + s * 2u * b_lbo, b_lbo, 128u);
    mma_tf32(d_tmem, ad, bd, idesc, (s > 0 || accumulate_first) ? 1u : 0u);
  }
}

// kind::tf32 over K elements with both operands 128-byte-swizzled K-major:
// four K = 8 steps per 128-byte block (start address + 32 bytes each), then
// the next block (+ rows * 128 bytes).
__device__ __forceinline__ void mma_kloop_tf32_sw128(uint32_t d_tmem, uint32_t a_saddr,
                                                     uint32_t b_saddr, uint32_t M, uint32_t N,
                                                     uint32_t K, bool accumulate_first) {
  const uint32_t idesc = idesc_tf32(M, N);
  for (uint32_t s = 0; s < K / 8u; ++s) {
    const uint32_t kb = s >> 2, kk = s & 3u;
    const uint64_t ad = smem_desc_sw128(a_saddr + kb * M * 128u + kk * 32u);
    const uint64_t bd = smem_desc_sw128(b_saddr + kb * N * 128u + kk * 32u);
    mma_tf32(d_tmem, ad, bd, idesc, (s > 0 || accumulate_first) ? 1u : 0u);
  }
}

// --- TMEM -> registers -------------------------------------------------------
// tcgen05.ld writes its registers asynchronously: they hold the data only
// after tcgen05.wait::ld.  The wait is a separate asm statement with no
// register operands, so on its own nothing keeps the compiler from moving a
// use of the loaded registers above it.  tmem_regs ties them to the wait: an
// empty volatile asm that reads and writes every register, placed after the
// wait (volatile asm statements keep their order), on which every later use
// depends.
__device__ __forceinline__ void tmem_regs(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]));
}
__device__ __forceinline__ void tmem_regs(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]));
  asm volatile(""
               : "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                 "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (taddr.lane + i), columns taddr.col .. +31.  The warp may only touch
// its own 32-lane sub-partition (warp id % 4).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  tmem_regs(r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tmem_ld32 without the wait: issue several, then tmem_wait_ld() once and
// tmem_regs() on each array before using any of them.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  tmem_regs(r);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

}  // namespace tc

// Programmatic dependent launch.  griddep_launch_dependents: this CTA lets the
// next kernel of the stream (launched with programmatic stream serialization)
// be scheduled once every CTA of this grid has said so or exited.
// griddep_wait: wait until the kernels this one depends on have completed and
// their memory is visible (returns at once without a programmatic launch).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace kda
