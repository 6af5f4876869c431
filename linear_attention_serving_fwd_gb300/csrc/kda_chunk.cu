// Chunked KDA prefill (chunk = 64) on tcgen05 tensor cores.
//
// Split as the vLLM kimi_k3 AMD kda_chunk page splits it: a prologue that is
// parallel over (chunk, head) - gate, beta, L2 norms, gate cumsum, both
// intra-chunk passes and the WY/UT solve - and a walk that is serial over the
// chunks of a (sequence, head) and fused with the output, plus the chunk-group
// parallel scan of _chunk_groups for long chains.
//
// Per chunk of rows r = 0..63 (Lam = in-chunk cumsum of the gate, C = 63):
//   A_kk[r,i] = beta_r sum_c k^_rc k^_ic e^{Lam_rc - Lam_ic}  (i < r)
//   A_qk[r,i] = sum_c q~_rc k^_ic e^{Lam_rc - Lam_ic}          (i <= r)
//   T  = (I + A_kk)^{-1} diag(beta)
//   Kg = e^{Lam} * k^,  qg = e^{Lam} * q~,  kg = e^{Lam_C - Lam} * k^,  d = e^{Lam_C}
// With w = T Kg and U = T v - w S the chunk step is
//   o = qg S + A_qk U,   S' = diag(d) S + kg^T U,
// which the walk evaluates in transition form, S kept in fp32:
//   S' = d * S + P S + R v,      P = -kg^T w  (K x K),  R = kg^T T  (K x C)
//   o  = qg' S + o_intra,        qg' = qg - A_qk w,  o_intra = A_qk T v
// so that only the product P S (K = 128) lies on the chunk-to-chunk chain.
// The prologue emits, per (chunk, head), the walk's tensor-core operands in
// their shared-memory layout (fp16, K-major, no swizzle):
//   P (128 x 128), R (128 x 64), d (fp32, 128), qg' (64 x 128),
//   o_intra (bf16, four blocks of [64 r][32 v], each row's four 16-byte
//   chunks rotated by r / 2: oi_offset) and v^T in four blocks of 32 value
//   columns.
//
// Precision: A_kk / A_qk use kind::tf32 (their operands carry exponent
// factors up to e^{8 |gate|}, outside fp16 range); every other product uses
// fp16 operands (11-bit significands, the tf32 class of rounding) with fp32
// accumulation, and the state stays fp32.  Operand magnitudes: T, w, kg, Kg,
// qg are bounded by 1 (scale); U and S scale with v and the initial state.
//
// The exponent differences of A_kk / A_qk are factored around m_R = Lam at
// the middle row 16 R + 7 of the row's own 16-row sub-chunk R:
//   e^{Lam_r - Lam_i} = (e^{Lam_r - m_R}) (e^{m_R - Lam_i})      (i <= 16 R + 15)
// The first factor stays within e^{+-84} as long as any 8 consecutive gates
// sum above -84 (lower_bound >= -10.5); the second is at most e^{84} and
// below 1 for every i before the middle row.  Kg, qg and kg take their
// exponentials directly (e^{Lam_i}, e^{Lam_C - Lam_i}, both at most 1).
#include <cuda.h>  // CUtensorMap (types only; the encoder comes via the runtime)
#include <cudaTypedefs.h>

#include "kda_conv.cuh"
#include "kda_params.cuh"
#include "kda_tc.cuh"

namespace kda {

// Per-(chunk, head) workspace record, bytes.  v^T is one K-major operand of
// 128 rows (value columns) by K = 64 (tokens): K groups 2048 bytes apart, so
// that a product over all 128 columns takes it whole and one over 32 columns
// takes, from each K group, the 512 bytes of its rows.
constexpr uint32_t VB_ROWS_BYTES = 32 * 16;         // 32 value rows of one K group
constexpr uint32_t VB_BYTES = VB_ROWS_BYTES * 64 / 8;  // a 32-column block, packed: 4096
constexpr uint32_t CH_P = 0;                        // fp16 128 x 128, rows k, K = k'
constexpr uint32_t CH_R = CH_P + 128 * 128 * 2;     // fp16 128 x 64,  rows k, K = r
constexpr uint32_t CH_D = CH_R + 128 * 64 * 2;      // fp32 128
constexpr uint32_t CH_QG = CH_D + 128 * 4;          // fp16 64 x 128,  rows r, K = k'
constexpr uint32_t OI_BLOCK = 64 * 32 * 2;          // bf16 o_intra block [64 r][32 v]
constexpr uint32_t CH_OI = CH_QG + 64 * 128 * 2;    // 4 o_intra blocks, one per 32 columns
constexpr uint32_t CH_V16 = CH_OI + 4 * OI_BLOCK;   // fp16 v^T, [128 v][64 r] K-major
constexpr uint32_t V16_BYTES = 128 * 64 * 2;
constexpr uint32_t CH_BYTES = CH_V16 + V16_BYTES;   // 98816
static_assert(CH_BYTES % 128 == 0, "records are whole 128-byte lines (the pipelined walk drops them from L2)");
constexpr uint32_t CH_A_BYTES = CH_QG - CH_P;       // P, R, d: the chain's part (49664)
constexpr uint32_t QG_BYTES = CH_OI - CH_QG;        // qg' (16384)

// Byte offset of the 16-byte chunk j (value columns 8 j .. 8 j + 7) of row r
// in an o_intra block: rows are 64 bytes apart and row r's chunks are
// rotated by r / 2, so that 16 rows stored or loaded at once spread over the
// shared-memory banks (2-way instead of 8-way).
__host__ __device__ constexpr uint32_t oi_offset(int r, int j) {
  return (uint32_t)(r * 64 + 16 * ((j + (r >> 1)) & 3));
}

__device__ __forceinline__ int seq_bos(const ChunkParams& p, int n) {
  return p.cu_seqlens ? p.cu_seqlens[n] : n * p.dense_len;
}
__device__ __forceinline__ int seq_eos(const ChunkParams& p, int n) {
  return p.cu_seqlens ? p.cu_seqlens[n + 1] : (n + 1) * p.dense_len;
}

// Chunk tables.  With cu_seqlens they are built on the device by
// kda_chunk_index_kernel; dense sequences of dense_len tokens have them in
// closed form (ceil(dense_len / 64) chunks each), and that launch is skipped.
__device__ __forceinline__ int dense_chunks(const ChunkParams& p) { return (p.dense_len + CHUNK - 1) / CHUNK; }
__device__ __forceinline__ int num_chunks_of(const ChunkParams& p) {
  return p.cu_seqlens ? *p.n_chunks : p.n_seqs * dense_chunks(p);
}
__device__ __forceinline__ int chunk_off_of(const ChunkParams& p, int n) {
  return p.cu_seqlens ? p.chunk_off[n] : n * dense_chunks(p);
}
__device__ __forceinline__ int chunk_seq_of(const ChunkParams& p, int c) {
  return p.cu_seqlens ? p.chunk_seq[c] : c / dense_chunks(p);
}
__device__ __forceinline__ int chunk_j_of(const ChunkParams& p, int c) {
  return p.cu_seqlens ? p.chunk_j[c] : c % dense_chunks(p);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Bounded mbarrier wait that also gives up once another thread of the CTA has
// raised the abort flag.  ``limit_ns`` of wall time (WAIT_NS in the kernels;
// the self-test below passes a short one).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t phase, volatile int* abort,
                                              unsigned* err, uint64_t limit_ns = WAIT_NS) {
  if (mbar_test_wait(bar, phase)) return true;  // already complete: no parking round trip
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < WAIT_CAP; ++i) {
    if (mbar_try_wait(bar, phase)) return true;
    if (*abort) return false;
    const uint64_t t = globaltimer_ns();
    if (t0 == 0) t0 = t;
    else if (t - t0 > limit_ns) break;
  }
  set_error(err, ERR_TIMEOUT);
  *abort = 1;
  return false;
}

// --------------------------------------------------------------------------
// Self-test of the bounded-wait abort path (no fault, no trap): one CTA of
// four warps holds TMEM as the chunk kernels do and waits, with the chunk
// kernels' wait_or_abort, on an mbarrier that nothing ever arrives at.  The
// first thread whose wait passes ``limit_ns`` sets ERR_TIMEOUT and raises
// the CTA's abort flag; the other threads see the flag and stop; warp 0
// frees the TMEM and the CTA returns.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1) kda_wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem;
  __shared__ int abort;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    tc::tmem_alloc(&tmem, 32);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    abort = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  wait_or_abort(&bar, 0, &abort, err, limit_ns);  // phase 0 never completes
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, 32);
}

int launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t stream) {
  kda_wait_selftest_kernel<<<1, 128, 0, stream>>>(err, limit_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// --------------------------------------------------------------------------
// Chunk index builder: chunk_off[n] = first global chunk of sequence n,
// chunk_seq / chunk_j name each chunk.  One block.
// --------------------------------------------------------------------------
__global__ void kda_chunk_index_kernel(ChunkParams p) {
  if (threadIdx.x == 0) {
    int off = 0;
    bool bad = p.cu_seqlens && p.cu_seqlens[0] != 0;
    for (int n = 0; n < p.n_seqs; ++n) {
      p.chunk_off[n] = off;
      int len = seq_eos(p, n) - seq_bos(p, n);
      if (len < 0) { bad = true; len = 0; }
      int nc = (len + CHUNK - 1) / CHUNK;
      if (off + nc > p.max_chunks) { bad = true; nc = p.max_chunks - off; }
      off += nc;
    }
    if (p.cu_seqlens && p.cu_seqlens[p.n_seqs] != p.t_total) bad = true;
    p.chunk_off[p.n_seqs] = off;
    *p.n_chunks = off;
    if (bad) set_error(p.err, ERR_INDEX);
  }
  __syncthreads();
  for (int n = threadIdx.x >> 5; n < p.n_seqs; n += blockDim.x >> 5) {
    const int c0 = p.chunk_off[n], c1 = p.chunk_off[n + 1];
    for (int c = c0 + (threadIdx.x & 31); c < c1; c += 32) {
      p.chunk_seq[c] = n;
      p.chunk_j[c] = c - c0;
    }
  }
}

// --------------------------------------------------------------------------
// Prologue: persistent, one CTA (512 threads, 16 warps) per SM looping over
// (chunk, head) items; while an item runs its inverse and last two products,
// the next item's q, k, g, v rows stream into the part of the operand region
// those steps leave free.
//
// Phase 1 is channel-owner: thread (c, R) holds channel c of the 16 rows of
// sub-chunk R and writes every operand that needs the gate cumsum straight
// into its MMA layout (tf32 128-byte-swizzled K-major, which a warp's 32
// consecutive channels of one row fill without bank conflicts):
//   X   = [k^ e^{Lam - m} ; q~ e^{Lam - m}]          128 rows (m = m_R of the row)
//   Y_R = k^_i e^{m_R - Lam_i},  i = 0 .. 16R + 15   16 (R + 1) rows
// The four Y_R are stacked into one 160-row operand (Y_R from row 8R(R+1)),
// so one kind::tf32 product D = X Y^T (N = 160) holds, in the rows of
// sub-chunk R and columns 8R(R+1).., A_kk (rows 0..63) and A_qk (rows
// 64..127) against every column of sub-chunks 0..R.
//
// The inverse of L = I + A_kk (unit lower triangular) is built by recursive
// doubling: the four diagonal 16 x 16 blocks by forward substitution, then
//   L^{-1}_{ba} = - L^{-1}_{bb} A_{ba} L^{-1}_{aa}
// for the two 16-row pairs and then for the two 32-row halves.
// --------------------------------------------------------------------------
constexpr int PRO_THREADS = 512;
// The thread that issues an item's record stores (and owns their bulk group):
// its warp has no work in the inverse's rounds, where the pipelined launch
// waits for the stores to land.
constexpr int REC_THREAD = 256;
constexpr int LDT = 68;  // row stride (floats) of the 64 x 64 fp32 matrices (16-byte rows)
constexpr int LDW = 34;  // row stride of the 32 x 32 fp32 temporary (8-byte column pairs)
constexpr int YROWS = 160;  // rows of the stacked Y operand

// first row of Y_R in the stacked operand = its first TMEM accumulator column
__host__ __device__ constexpr uint32_t d_col(int R) { return 8u * (uint32_t)(R * (R + 1)); }

// After the A_kk / A_qk MMAs the X / Y region holds (byte offsets):
constexpr uint32_t P_LI = 0;         // fp32 [64][LDT]  = L^{-1}
constexpr uint32_t P_A = 17408;      // fp32 [64][LDT]  = beta-scaled strictly lower A_kk
constexpr uint32_t P_W = 34816;      // fp32 [32][LDW]  temporary product
constexpr uint32_t P_A3 = 17408;     // fp16 [128][128] = [[T, 0], [-A_qk T, I]], over A and W
constexpr uint32_t P_A2 = 50176;     // fp16 [128][64]  = [A_qk ; 0]
constexpr uint32_t P_B2 = 66560;     // fp16 [64][64]   = T^T
constexpr uint32_t P_TILES = 75776;  // bf16 tiles of the next item (below)
// Record staging in the last round.  P is written while qg' and o_intra
// still read A3, so its two 16 KB halves go where L^{-1} and A2 were; qg' and
// o_intra follow over A3 once every product is done.
constexpr uint32_t ST_P0 = 0;        // P record bytes [0, 16384)
constexpr uint32_t ST_P1 = 50176;    // P record bytes [16384, 32768)
constexpr uint32_t ST_QG = 16384;    // qg' then o_intra (32 KB)
static_assert(P_LI + 64 * LDT * 4 <= P_A && P_A + 64 * LDT * 4 <= P_W, "prologue carve");
static_assert(P_W + 32 * LDW * 4 <= P_A3 + 32768 && P_A3 + 32768 <= P_A2, "A3 covers A and W");
static_assert(P_A2 + 16384 <= P_B2 && P_B2 + 8192 <= P_TILES, "prologue carve");
static_assert(ST_P0 + 16384 <= P_A3 && P_A3 + 32768 <= ST_P1 && ST_P1 + 16384 <= P_TILES,
              "P staging stays clear of A3, which the last products read");
static_assert(ST_P0 + 16384 <= ST_QG && ST_QG + 32768 <= ST_P1, "record staging");

struct __align__(1024) ProSmem {
  // X (tf32, 128 x 128) at XY, Y_0 .. Y_3 stacked (tf32 [YROWS][128]) at
  // XY + 65536; the carve P_* above once the MMAs have read them
  unsigned char XY[65536 + 81920];
  unsigned char B3[32768];  // fp16 [c][K]: K 0..63 = Kg rows, 64..127 = qg rows
  unsigned char KG[16384];  // fp16 kg^T, K-major [k][r]
  unsigned char VT[16384];  // fp16 v^T, K-major [v][r] (K groups 2048 bytes apart)
  float qtot[8][128];       // gate sum of each 8-row half sub-chunk
  float ssk[2][64];         // |k_r|^2 partial per group of 64 channels
  float ssq[2][64];
  float beta[64];
  // the next item's scalars, fetched during this item's inverse by threads
  // that have no part in it: sigmoid(beta) per row (0 past its length),
  // a_h dt_bias per channel pair and a_h = e^{A_log} of its head
  float beta_n[64];
  float2 adt_n[64];
  float ah_n;
  int4 meta[2];             // (chunk, head, first token, rows) of this and the next item
  uint64_t bar;
  uint64_t bar2;            // the P product of the last round, ahead of the others
  uint64_t tbar;            // tile loads
  uint32_t tmem;
  int next_t;               // the next item
  int abort;
};
// The tiles: q, k, v, each HALO rows (the three tokens before the chunk,
// which a conv reads) then the chunk's 64 rows, then g (64 rows).
constexpr int HALO = 3;
constexpr int TILE_QKV = (HALO + CHUNK) * D;  // elements of a q / k / v tile (17,152 bytes)
static_assert(P_TILES + (3 * TILE_QKV + CHUNK * D) * 2 <= sizeof(ProSmem::XY), "carve fits");
static_assert((P_TILES + HALO * D * 2) % 128 == 0 && (TILE_QKV * 2) % 128 == 0, "TMA tile alignment");
// row r (from -HALO) of band x (0 q, 1 k, 2 v) / row r of g
__device__ __forceinline__ int tile_row(int x, int r) { return x * TILE_QKV + (HALO + r) * D; }
__device__ __forceinline__ int g_row(int r) { return 3 * TILE_QKV + r * D; }

// Item t of the prologue: t = chunk * Hv + head; in the pipelined launch
// (walk_ctas > 0, dense sequences) level-major instead, t = (j * n_seqs + n)
// * Hv + head for in-sequence chunk j, so that every chain's chunk j is
// produced before any chain's chunk j + 1 is started.
__device__ __forceinline__ int4 item_meta(const ChunkParams& p, int t) {
  int c, h;
  if (p.walk_ctas > 0) {
    const int chains = p.n_seqs * p.hv, j = t / chains, r = t - j * chains, n = r / p.hv;
    h = r - n * p.hv;
    c = chunk_off_of(p, n) + j;
  } else {
    c = t / p.hv;
    h = t - c * p.hv;
  }
  const int n = chunk_seq_of(p, c);
  const int bos = seq_bos(p, n) + chunk_j_of(p, c) * CHUNK;
  return make_int4(c, h, bos, min(CHUNK, seq_eos(p, n) - bos));
}

// Tensor maps of q, k (dims 128 x Hqk x T) and g, v (128 x Hv x T), bf16,
// box 128 x 1 x 64: one tiled TMA load brings a (chunk, head) tile.
struct TileMaps {
  CUtensorMap q, k, g, v;
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// One item's q, k, v, g rows (bf16, 64 x 128 each) into ``tiles`` with four
// tiled TMA loads completing on ``bar`` (one thread).  With a conv the q, k,
// v boxes start three tokens early (HALO rows: the conv's history inside a
// sequence; at a sequence start the conv phase replaces them).  Tokens
// before 0 or past T arrive as zeros; rows past the sequence end hold the
// next sequence's tokens and readers mask them.
template <bool CONV>
__device__ __forceinline__ void load_tiles(const ChunkParams& p, const TileMaps& maps, int4 m,
                                           __nv_bfloat16* tiles, uint64_t* bar) {
  const int h = m.y, bos = m.z, hq = h / (p.hv / p.hqk);
  constexpr int halo = CONV ? HALO : 0;
  mbar_arrive_expect_tx(bar, (uint32_t)((3 * (CHUNK + halo) + CHUNK) * D * 2));
  tma_load_3d(tiles + tile_row(0, -halo), &maps.q, 0, hq, bos - halo, bar);
  tma_load_3d(tiles + tile_row(1, -halo), &maps.k, 0, hq, bos - halo, bar);
  tma_load_3d(tiles + tile_row(2, -halo), &maps.v, 0, h, bos - halo, bar);
  tma_load_3d(tiles + g_row(0), &maps.g, 0, h, bos, bar);
}

// Width-4 conv + SiLU of the item's q, k, v tiles, in place (conv mode).
// Thread (channel c, sub-chunk Rq) computes rows 16 Rq .. +15 of the three
// bands from the raw rows 16 Rq - 3 .. 16 Rq + 15; at a sequence's first
// chunk the HALO rows are first replaced by the conv state's history
// (zeros without one).  Ends with a barrier.
__device__ __forceinline__ void conv_tiles(const ChunkParams& p, __nv_bfloat16* tiles, int c_glob, int h,
                                        int tid) {
  const ConvParams& cv = p.conv;
  const int c = tid & 127, Rq = tid >> 7;
  int64_t ch[3];
  conv_channels(p.hqk, p.hv, h, c, ch);
  if (chunk_j_of(p, c_glob) == 0 && Rq < 3) {
    const int n = chunk_seq_of(p, c_glob);
    const int row = cv.idx[n];
    const bool init = row >= 0 && row < cv.rows && (!cv.has_init || cv.has_init[n]);
    const int64_t chx = Rq == 0 ? ch[0] : (Rq == 1 ? ch[1] : ch[2]);
    const __nv_bfloat16* src = cv.state + (int64_t)row * cv.row_st + chx * cv.ch_st;
#pragma unroll
    for (int i = 0; i < HALO; ++i)
      tiles[tile_row(Rq, i - HALO) + c] = init ? src[i * cv.pos_st] : __float2bfloat16(0.f);
  }
  __syncthreads();
  __nv_bfloat162 y[3][8];  // outputs, rows in pairs
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    const float4 w = conv_taps(cv, ch[x]);
    const __nv_bfloat16* col = tiles + tile_row(x, 16 * Rq - HALO) + c;
    __nv_bfloat16 win[16 + HALO];  // rows 16 Rq - 3 .. 16 Rq + 15
#pragma unroll
    for (int i = 0; i < 16 + HALO; ++i) win[i] = col[i * D];
#pragma unroll
    for (int i = 0; i < 16; i += 2) y[x][i >> 1] = conv_silu2(cv.w_f32, w, win + i);
  }
  __syncthreads();  // every raw row read
#pragma unroll
  for (int x = 0; x < 3; ++x)
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      tiles[tile_row(x, 16 * Rq + i) + c] = y[x][i >> 1].x;
      tiles[tile_row(x, 16 * Rq + i + 1) + c] = y[x][i >> 1].y;
    }
  __syncthreads();
}

// The item's raw per-row beta (threads 0..63), dt_bias of channel tid % 128
// and A_log: loaded early, consumed at the item's start.
// Threads 320..447 of the prologue: item m's per-item scalars into shared
// memory (the ProSmem fields beta_n, adt_n, ah_n).  They run it while the
// others invert, so its global loads' latency is on no one's path.
template <bool FP16>
__device__ __forceinline__ void fetch_scalars(const ChunkParams& p, float* beta_n, float2* adt_n, float* ah_n,
                                              int4 m, int tid) {
  const int h = m.y, bos = m.z, len = m.w;
  const int u = tid - 320;
  if (u >= 0 && u < 64) {
    beta_n[u] = u < len ? sigmoidf_(act_f<FP16>(p.beta[(int64_t)(bos + u) * p.b_st + h * p.b_sh])) : 0.f;
  } else if (u >= 64 && u < 128) {
    const int cp = u - 64;
    float ah = 0.f;
    float2 adt = make_float2(0.f, 0.f);
    if (p.has_gate) {
      ah = __expf(p.A_log[h]);
      const float2 dt = *reinterpret_cast<const float2*>(p.dt_bias + h * D + 2 * cp);
      adt = make_float2(ah * dt.x, ah * dt.y);
    }
    adt_n[cp] = adt;
    if (cp == 0) *ah_n = ah;
  }
}

// Per-phase cycle accounting of the prologue, compiled in only with
// -DKDA_PHASE_TIMING (the package's ``phase_timing`` module builds and runs
// that copy): thread 0 of each CTA adds the clock64 cycles between the
// barriers that close the phases of every item, and at exit adds its sums
// and item count to g_phase_cycles / g_phase_items.  Every phase ends with a
// barrier of all threads, so these are the phases' wall times on the SM.
#ifdef KDA_PHASE_TIMING
constexpr int N_PHASES = 12;
__device__ unsigned long long g_phase_cycles[N_PHASES];
__device__ unsigned long long g_phase_items;
#define PH_BEGIN()                                       \
  __shared__ unsigned long long ph_acc[N_PHASES];        \
  long long ph_t = clock64();                            \
  int ph_items = 0;                                      \
  if (tid == 0)                                          \
    for (int i_ = 0; i_ < N_PHASES; ++i_) ph_acc[i_] = 0
#define PH(i)                                            \
  do {                                                   \
    if (tid == 0) {                                      \
      const long long n_ = clock64();                    \
      ph_acc[i] += (unsigned long long)(n_ - ph_t);      \
      ph_t = n_;                                         \
    }                                                    \
  } while (0)
#define PH_ITEM() (++ph_items)
#define PH_END()                                                                  \
  do {                                                                            \
    if (tid == 0) {                                                               \
      for (int i_ = 0; i_ < N_PHASES; ++i_) atomicAdd(&g_phase_cycles[i_], ph_acc[i_]); \
      atomicAdd(&g_phase_items, (unsigned long long)ph_items);                    \
    }                                                                             \
  } while (0)
#else
#define PH_BEGIN() \
  do {             \
  } while (0)
#define PH(i) \
  do {        \
  } while (0)
#define PH_ITEM() ((void)0)
#define PH_END() \
  do {           \
  } while (0)
#endif

// The ready flag of a record: set once the record's stores have completed,
// with release semantics at GPU scope (the bulk stores are ordered before it
// by the proxy fence).  The walk acquires it before loading the record.
__device__ __forceinline__ void publish_ready(unsigned* flag) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(1u) : "memory");
}

// The prologue's items first, first + stride, ... on one CTA (smem_raw: a
// ProSmem).  With p.ready set, each item's ready flag is raised once its
// record has landed: at the next item's first barrier, or at the end.
template <bool CONV, bool FP16>
__device__ __forceinline__ void prologue_items(const ChunkParams& p, const TileMaps& maps, int first,
                                               int stride, unsigned char* smem_raw) {
  ProSmem& s = *reinterpret_cast<ProSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = num_chunks_of(p) * p.hv;
  if (first >= n_items) return;
  __nv_bfloat16* tiles = reinterpret_cast<__nv_bfloat16*>(s.XY + P_TILES);
  PH_BEGIN();

  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&s.bar, 1);
    mbar_init(&s.bar2, 1);
    mbar_init(&s.tbar, 1);
    fence_mbar_init();
    s.abort = 0;
    // items first, first + stride, ...; or, with p.item_counter, whichever
    // item is next when this CTA asks (an SM that runs slower takes fewer;
    // each CTA holds one drawn item beyond its next)
    const int t0 = p.item_counter ? (int)atomicAdd(p.item_counter, 1u) : first;
    s.next_t = t0;
    if (t0 < n_items) {
      s.meta[0] = item_meta(p, t0);
      load_tiles<CONV>(p, maps, s.meta[0], tiles, &s.tbar);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem;
  int t = s.next_t;
  // thread 32 draws the item after next one item ahead, so that the counter's
  // round trip never delays the next item's tile loads
  int t_ahead = 0;
  if (tid == 32) t_ahead = p.item_counter ? (int)atomicAdd(p.item_counter, 1u) : t + stride;
  if (t < n_items) fetch_scalars<FP16>(p, s.beta_n, s.adt_n, &s.ah_n, s.meta[0], tid);
  __syncthreads();
  uint32_t bar_phase = 0, bar2_phase = 0, tile_phase = 0, tiles_issued = t < n_items ? 1 : 0;
  int cur = 0;
  int pending = -1;  // REC_THREAD: the record whose stores are in flight (pipelined launch)
  for (; t < n_items; cur ^= 1) {
    // this CTA's last item: the walk may start its setup on the SMs that
    // finish first (it waits for this grid before reading any record)
    if (!p.item_counter && t + stride >= n_items) griddep_launch_dependents();
    const int4 meta = s.meta[cur];
    const int c_glob = meta.x, h = meta.y, len = meta.w;
    const float a_h = s.ah_n;
    if (tid < 64) s.beta[tid] = s.beta_n[tid];
    unsigned char* wsb = reinterpret_cast<unsigned char*>(p.ch) + ((size_t)c_glob * p.hv + h) * CH_BYTES;
    // ---- phase 0: this item's tiles (issued during the previous item) -------
    wait_or_abort(&s.tbar, tile_phase, &s.abort, p.err);
    tile_phase ^= 1u;
    __syncthreads();
    if constexpr (CONV) conv_tiles(p, tiles, c_glob, h, tid);
    PH_ITEM();
    PH(0);

    // ---- phase 1: thread = (channel pair: channels c, c + 1 with c = 2 cp;
    // rows 8 hs .. 8 hs + 7, half hs % 2 of sub-chunk Rq = hs / 2) ------------
    const int cp = tid & 63, hs = tid >> 6, Rq = hs >> 1;
    const int c = 2 * cp;
    float2 lam[8], kv[8], qv[8];  // per row, the two channels
    {
      float2 acc = make_float2(0.f, 0.f);
      bool gate_bad = false;
      uint32_t vw[2][4];  // v of channels c and c + 1 as fp16 pairs along rows
      const float2 ah2 = make_float2(a_h, a_h), adt2 = s.adt_n[cp];
      const float2 zero2 = make_float2(0.f, 0.f);
      // rows at or past ``len`` belong to the next sequence
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        float2 vv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = 8 * hs + i + e;
          const bool in = r < len;
          qv[i + e] = in ? act_f2<FP16>(tiles + tile_row(0, r) + c) : zero2;
          kv[i + e] = in ? act_f2<FP16>(tiles + tile_row(1, r) + c) : zero2;
          float2 g = in ? act_f2<FP16>(tiles + g_row(r) + c) : zero2;
          if (p.has_gate) {  // lower_bound * sigmoid(a (g + dt_bias)), both channels
            const float2 t = ffma2(ah2, g, adt2);
            const float2 den = fadd2(make_float2(__expf(-t.x), __expf(-t.y)), make_float2(1.f, 1.f));
            g = in ? make_float2(__fdividef(p.lower_bound, den.x), __fdividef(p.lower_bound, den.y)) : zero2;
          } else {  // g is the log decay itself: it must lie in [-10.5, 0]
            gate_bad |= !(g.x >= -10.5f && g.x <= 0.f && g.y >= -10.5f && g.y <= 0.f);
          }
          acc = fadd2(acc, g);
          lam[i + e] = acc;
          vv[e] = in ? act_f2<FP16>(tiles + tile_row(2, r) + c) : zero2;
        }
        vw[0][i >> 1] = pack_half2(vv[0].x, vv[1].x);
        vw[1][i >> 1] = pack_half2(vv[0].y, vv[1].y);
      }
      // a raw log decay outside [-10.5, 0] (or NaN) leaves the exponent range
      // the factored A_kk / A_qk operands are built for: report it
      if (!p.has_gate && __any_sync(0xffffffffu, gate_bad) && lane == 0) set_error(p.err, ERR_RANGE);
      // v^T of the two channels: the record, and VT for the o_intra product
      // (made here only for the 32-column walk); they share a layout
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t o = tc::kmajor_offset(c + e, 8 * hs, 128);
        const uint4 v4 = make_uint4(vw[e][0], vw[e][1], vw[e][2], vw[e][3]);
        *reinterpret_cast<uint4*>(wsb + CH_V16 + o) = v4;
        if (!p.rec128) *reinterpret_cast<uint4*>(s.VT + o) = v4;
      }
      *reinterpret_cast<float2*>(&s.qtot[hs][c]) = acc;
      // row norms: the 8 per-row partials reduce-scatter over the warp's 64
      // channels (halving by lane bits 4, 3, 2; bits 1, 0 summed): lanes with
      // bits 1..0 clear hold row 4 b4 + 2 b3 + b2; the two channel halves
      // meet in shared memory
      float pk[8], pq[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pk[i] = kv[i].x * kv[i].x + kv[i].y * kv[i].y;
        pq[i] = qv[i].x * qv[i].x + qv[i].y * qv[i].y;
      }
#pragma unroll
      for (int lvl = 0; lvl < 3; ++lvl) {
        const int m = 16 >> lvl, n = 4 >> lvl;
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < n) {
            const float sk = up ? pk[q] : pk[q + n], kk = up ? pk[q + n] : pk[q];
            const float sq = up ? pq[q] : pq[q + n], qq = up ? pq[q + n] : pq[q];
            pk[q] = kk + __shfl_xor_sync(0xffffffffu, sk, m);
            pq[q] = qq + __shfl_xor_sync(0xffffffffu, sq, m);
          }
        }
      }
#pragma unroll
      for (int m = 2; m >= 1; m >>= 1) {
        pk[0] += __shfl_xor_sync(0xffffffffu, pk[0], m);
        pq[0] += __shfl_xor_sync(0xffffffffu, pq[0], m);
      }
      if ((lane & 3) == 0) {
        const int row = 8 * hs + 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
        s.ssk[cp >> 5][row] = pk[0];
        s.ssq[cp >> 5][row] = pq[0];
      }
      // the last item's record stores have read the staging area, which the
      // X / Y build below overwrites
      if (tid == REC_THREAD) bulk_wait_read<0>();
    }
    __syncthreads();
    PH(1);
    float2 mR;  // Lam at row 16 Rq + 7, the sub-chunk's reference
    float2 dr[8], eL0, eC7;  // the rows' decays e^{Lam_i - Lam_{i-1}}; e^{Lam_0}, e^{Lam_C - Lam_7}
    {
      // Every thread reads what it needs straight from the half-sub-chunk
      // gate totals and the norm partials: its rows' offset (the totals of
      // the halves before), the references m_R = Lam at row 16 R + 7 (the
      // totals of halves 0 .. 2R), Lam_C (all eight) and its rows' norms.
      float2 run = make_float2(0.f, 0.f), off = run, mref[4];
#pragma unroll
      for (int h2 = 0; h2 < 8; ++h2) {
        if (h2 == hs) off = run;
        run = fadd2(run, *reinterpret_cast<const float2*>(&s.qtot[h2][c]));
        if ((h2 & 1) == 0) mref[h2 >> 1] = run;
      }
      const float2 lamC = run;
#pragma unroll
      for (int i = 0; i < 8; ++i) lam[i] = fadd2(lam[i], off);
      mR = Rq == 0 ? mref[0] : (Rq == 1 ? mref[1] : (Rq == 2 ? mref[2] : mref[3]));
      if (hs == 7)
        *reinterpret_cast<float2*>(wsb + CH_D + 4 * c) = make_float2(__expf(lamC.x), __expf(lamC.y));
      // normalised keys and queries: lane l of the warp forms 1/|k_r| (l & 8
      // clear) or scale/|q_r| (l & 8 set) of row r = 8 hs + (l & 7) from the
      // two channel halves' partial sums; shuffles hand the warp's 8 rows to
      // every lane
      {
        const int rr = 8 * hs + (lane & 7);
        const bool isq = (lane & 8) != 0;
        const float sum = isq ? s.ssq[0][rr] + s.ssq[1][rr] : s.ssk[0][rr] + s.ssk[1][rr];
        const float nrm = isq ? rsqrtf(sum + 1e-6f) * p.scale : rsqrtf(sum + 1e-6f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float rr_k = __shfl_sync(0xffffffffu, nrm, i), rr_q = __shfl_sync(0xffffffffu, nrm, 8 + i);
          kv[i] = fmul2(kv[i], make_float2(rr_k, rr_k));
          qv[i] = fmul2(qv[i], make_float2(rr_q, rr_q));
        }
      }
      // X and Y first (8-byte pairs of tf32 along the channels): the A_kk /
      // A_qk product starts on them while the B3 / KG operands are built
      auto tf32x2 = [](float2 v) {
        return make_uint2(__float_as_uint(tc::to_tf32_int(v.x)), __float_as_uint(tc::to_tf32_int(v.y)));
      };
      // Every exponential below is e^{Lam_i - x} or e^{x - Lam_i} for this
      // thread's 8 consecutive rows i, so each follows from one anchor by
      // the rows' decays dr_i = e^{Lam_i - Lam_{i-1}}: 4 exponentials a
      // channel per row become 1.  The products telescope exactly over the
      // (rounded) Lam, so they differ from the direct exponentials only by
      // a few roundings, far below the tf32 / fp16 operands they scale.
      dr[0] = make_float2(1.f, 1.f);
#pragma unroll
      for (int i = 1; i < 8; ++i) dr[i] = make_float2(__expf(lam[i].x - lam[i - 1].x), __expf(lam[i].y - lam[i - 1].y));
      eL0 = make_float2(__expf(lam[0].x), __expf(lam[0].y));                     // e^{Lam_0}
      eC7 = make_float2(__expf(lamC.x - lam[7].x), __expf(lamC.y - lam[7].y));   // e^{Lam_C - Lam_7}
      {  // X = [k^; q~] e^{Lam - m}, rows upward from e^{Lam_0 - m} (within e^{+-84})
        float2 E = make_float2(__expf(lam[0].x - mR.x), __expf(lam[0].y - mR.y));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 8 * hs + i;
          if (i > 0) E = fmul2(E, dr[i]);
          *reinterpret_cast<uint2*>(s.XY + tc::sw128_offset32(r, c, 128)) = tf32x2(fmul2(kv[i], E));
          *reinterpret_cast<uint2*>(s.XY + tc::sw128_offset32(64 + r, c, 128)) = tf32x2(fmul2(qv[i], E));
        }
      }
      {  // Y_R2 = k^ e^{m_R2 - Lam} for this sub-chunk and the later ones
         // (R2 >= Rq), rows downward from e^{m_R2 - Lam_7}.  Each factor is
         // one exponential's worth: at most e^{84}, and flushed to zero only
         // where the term it scales is below e^{-87} (a product through
         // e^{m_R2 - m_Rq}, which spans 16 rows, could underflow while the
         // term itself does not)
        float2 yf[4];
#pragma unroll
        for (int R2 = 0; R2 < 4; ++R2)
          yf[R2] = R2 >= Rq ? make_float2(__expf(mref[R2].x - lam[7].x), __expf(mref[R2].y - lam[7].y))
                            : make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 7; i >= 0; --i) {
          const int r = 8 * hs + i;
#pragma unroll
          for (int R2 = 0; R2 < 4; ++R2)
            if (R2 >= Rq) {
              if (i < 7) yf[R2] = fmul2(yf[R2], dr[i + 1]);
              *reinterpret_cast<uint2*>(s.XY + 65536 + tc::sw128_offset32(d_col(R2) + r, c, YROWS)) =
                  tf32x2(fmul2(kv[i], yf[R2]));
            }
        }
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      PH(3);

      // ---- phase 2: A_kk / A_qk, one kind::tf32 product (N = 160) ------------
      if (tid == 0) {
        tc::mma_kloop_tf32_sw128(tmem, smem_u32(s.XY), smem_u32(s.XY + 65536), 128, YROWS, 128, false);
        tc::mma_commit(&s.bar);
      }
      // meanwhile: Kg = k^ e^{Lam}, qg = q~ e^{Lam}, kg = k^ e^{Lam_C - Lam}
      // (each factor at most 1: an underflow only drops a term below e^{-87})
      uint32_t Kgx[2][4], qgx[2][4], kgw[2][4];  // per channel, fp16 pairs along rows
      {  // e^{Lam}: rows upward from e^{Lam_0}
        float2 eL = eL0;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          if (i > 0) eL = fmul2(eL, dr[i]);
          const float2 Kg0 = fmul2(kv[i], eL), qg0 = fmul2(qv[i], eL);
          eL = fmul2(eL, dr[i + 1]);
          const float2 Kg1 = fmul2(kv[i + 1], eL), qg1 = fmul2(qv[i + 1], eL);
          Kgx[0][i >> 1] = pack_half2(Kg0.x, Kg1.x);
          Kgx[1][i >> 1] = pack_half2(Kg0.y, Kg1.y);
          qgx[0][i >> 1] = pack_half2(qg0.x, qg1.x);
          qgx[1][i >> 1] = pack_half2(qg0.y, qg1.y);
        }
      }
      {  // e^{Lam_C - Lam}: rows downward from e^{Lam_C - Lam_7}
        float2 eC = eC7;
#pragma unroll
        for (int i = 6; i >= 0; i -= 2) {
          if (i < 6) eC = fmul2(eC, dr[i + 2]);
          const float2 kg1 = fmul2(kv[i + 1], eC);
          eC = fmul2(eC, dr[i + 1]);
          const float2 kg0 = fmul2(kv[i], eC);
          kgw[0][i >> 1] = pack_half2(kg0.x, kg1.x);
          kgw[1][i >> 1] = pack_half2(kg0.y, kg1.y);
        }
      }
      // B3 [c][K]: Kg row i at K = i, qg row r at K = 64 + r; KG [k = c][K = r]
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int ch = c + e, r0 = 8 * hs;
        *reinterpret_cast<uint4*>(s.B3 + tc::kmajor_offset(ch, r0, 128)) =
            make_uint4(Kgx[e][0], Kgx[e][1], Kgx[e][2], Kgx[e][3]);
        *reinterpret_cast<uint4*>(s.B3 + tc::kmajor_offset(ch, 64 + r0, 128)) =
            make_uint4(qgx[e][0], qgx[e][1], qgx[e][2], qgx[e][3]);
        *reinterpret_cast<uint4*>(s.KG + tc::kmajor_offset(ch, r0, 128)) =
            make_uint4(kgw[e][0], kgw[e][1], kgw[e][2], kgw[e][3]);
      }
      fence_proxy_async_smem();
    }
    // the next item (thread 32; every thread reads it after phase 5's barrier)
    int t_next = 0;
    if (tid == 32) {
      t_next = t_ahead;
      t_ahead = p.item_counter ? (int)atomicAdd(p.item_counter, 1u) : t_next + stride;
      s.next_t = t_next;
      if (t_next < n_items) s.meta[cur ^ 1] = item_meta(p, t_next);
    }
    wait_or_abort(&s.bar, bar_phase, &s.abort, p.err);
    bar_phase ^= 1u;
    tc::fence_after_sync();
    // the product has read Y: the next item's rows stream in over it (the
    // carve below stays under P_TILES)
    if (tid == 32 && t_next < n_items) load_tiles<CONV>(p, maps, s.meta[cur ^ 1], tiles, &s.tbar);
    PH(4);

    float* Af = reinterpret_cast<float*>(s.XY + P_A);
    float* Li = reinterpret_cast<float*>(s.XY + P_LI);
    float* Wt = reinterpret_cast<float*>(s.XY + P_W);
    unsigned char* A2 = s.XY + P_A2;
    unsigned char* A3 = s.XY + P_A3;
    unsigned char* B2 = s.XY + P_B2;
    {
      // warp = (TMEM sub-partition sp, 16-column group cg); rows 0..63 of the
      // accumulators are A_kk, rows 64..127 A_qk
      const int sp = warp & 3, cg = warp >> 2;
      const int r = 32 * (sp & 1) + lane, Rr = r >> 4, Rlo = 2 * (sp & 1);
      float a0[16], a1[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) { a0[t] = 0.f; a1[t] = 0.f; }
      if (cg <= Rlo) tc::tmem_ld16(tc::tmem_addr(tmem, 32 * sp, d_col(Rlo) + 16 * cg), a0);
      if (cg <= Rlo + 1) tc::tmem_ld16(tc::tmem_addr(tmem, 32 * sp, d_col(Rlo + 1) + 16 * cg), a1);
      const bool hi = Rr != Rlo, live = cg <= Rr;
      if (sp < 2) {
        const float b = s.beta[r];
        float av[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const int col = 16 * cg + t;
          av[t] = (live && col < r) ? b * (hi ? a1[t] : a0[t]) : 0.f;
        }
#pragma unroll
        for (int t = 0; t < 16; t += 4)
          *reinterpret_cast<float4*>(&Af[r * LDT + 16 * cg + t]) =
              make_float4(av[t], av[t + 1], av[t + 2], av[t + 3]);
      } else {
        uint32_t hv[8];
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          const int col = 16 * cg + t;
          const float x0 = (live && col <= r) ? (hi ? a1[t] : a0[t]) : 0.f;
          const float x1 = (live && col + 1 <= r) ? (hi ? a1[t + 1] : a0[t + 1]) : 0.f;
          hv[t >> 1] = pack_half2(x0, x1);
        }
#pragma unroll
        for (int g8 = 0; g8 < 2; ++g8)
          *reinterpret_cast<uint4*>(A2 + tc::kmajor_offset(r, 16 * cg + 8 * g8, 128)) =
              make_uint4(hv[4 * g8], hv[4 * g8 + 1], hv[4 * g8 + 2], hv[4 * g8 + 3]);
      }
      // A2 rows 64..127 are zero; L^{-1} above its diagonal blocks is zero
      *reinterpret_cast<uint4*>(A2 + tc::kmajor_offset(64 + (tid & 63), 8 * (tid >> 6), 128)) =
          make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = tid + u * PRO_THREADS, rr = e >> 6, cc = e & 63;
        if ((cc >> 4) > (rr >> 4)) Li[rr * LDT + cc] = 0.f;
      }
    }
    __syncthreads();
    PH(5);

    t_next = s.next_t;
    const bool has_next = t_next < n_items;
    // the next item's scalars (its tiles are already on their way), by
    // threads that skip the inverse
    if (has_next) {
      tiles_issued += 1;
      fetch_scalars<FP16>(p, s.beta_n, s.adt_n, &s.ah_n, s.meta[cur ^ 1], tid);
    }
    // The inverse below runs on threads 0..255, which synchronise among
    // themselves (barrier 1) until its last round; threads 256.. go straight
    // to that round's barrier.  In the pipelined launch the record thread
    // (256) meanwhile waits for the last item's stores to land and raises its
    // flag, off the working threads' path.
    if (tid == REC_THREAD && pending >= 0) {
      bulk_wait<0>();
      publish_ready(p.ready + pending);
      pending = -1;
    }

    // ---- phase 3: L^{-1} by recursive doubling ---------------------------------
    if (tid < 64) {
      // diagonal 16 x 16 blocks, thread = (block R, column jc), forward substitution
      const int b0 = 16 * (tid >> 4), jc = tid & 15;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float s0 = (i == jc) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
        for (int m = 0; m + 1 < i; m += 2) {
          s0 -= Af[(b0 + i) * LDT + b0 + m] * x[m];
          s1 -= Af[(b0 + i) * LDT + b0 + m + 1] * x[m + 1];
        }
        if (i & 1) s0 -= Af[(b0 + i) * LDT + b0 + i - 1] * x[i - 1];
        x[i] = (i < jc) ? 0.f : s0 + s1;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) Li[(b0 + i) * LDT + b0 + jc] = x[i];
    }
    if (tid < 256) named_bar_sync(1, 256);
    PH(6);
    // 16-row pairs (a, b) = (2P, 2P + 1): thread (P, row i, column pair jp)
    // of the first 256 threads computes two entries
    if (tid < 256) {
      // W = A_ba L^{-1}_aa
      const int P = tid >> 7, i = (tid >> 3) & 15, j0 = 2 * (tid & 7);
      const int a0 = 32 * P, b0 = 32 * P + 16;
      float2 r = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 16; m += 4) {
        const float4 x = *reinterpret_cast<const float4*>(&Af[(b0 + i) * LDT + a0 + m]);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          r = ffma2(make_float2(xs[u], xs[u]), *reinterpret_cast<const float2*>(&Li[(a0 + m + u) * LDT + a0 + j0]), r);
      }
      *reinterpret_cast<float2*>(&Wt[(16 * P + i) * LDW + j0]) = r;
    }
    if (tid < 256) named_bar_sync(1, 256);
    if (tid < 256) {
      // L^{-1}_ba = - L^{-1}_bb W
      const int P = tid >> 7, i = (tid >> 3) & 15, j0 = 2 * (tid & 7);
      const int a0 = 32 * P, b0 = 32 * P + 16;
      float2 r = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 16; m += 4) {
        const float4 x = *reinterpret_cast<const float4*>(&Li[(b0 + i) * LDT + b0 + m]);
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          r = ffma2(make_float2(xs[u], xs[u]), *reinterpret_cast<const float2*>(&Wt[(16 * P + m + u) * LDW + j0]), r);
      }
      *reinterpret_cast<float2*>(&Li[(b0 + i) * LDT + a0 + j0]) = make_float2(-r.x, -r.y);
    }
    if (tid < 256) named_bar_sync(1, 256);
    PH(7);
    // 32-row halves: thread (row pair rp, column pair cp) of the first 256
    // threads computes a 2 x 2 tile; the left factor's rows are 16-byte
    // broadcasts, the right factor's column pairs 8-byte loads
    if (tid < 256) {
      // W = A_{[32,64) [0,32)} L^{-1}_{[0,32) [0,32)}
      const int i0 = 2 * (tid >> 4), j0 = 2 * (tid & 15);
      float2 r0 = make_float2(0.f, 0.f), r1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 32; m += 4) {
        const float4 x = *reinterpret_cast<const float4*>(&Af[(32 + i0) * LDT + m]);
        const float4 z = *reinterpret_cast<const float4*>(&Af[(33 + i0) * LDT + m]);
        const float xs[4] = {x.x, x.y, x.z, x.w}, zs[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 c2 = *reinterpret_cast<const float2*>(&Li[(m + u) * LDT + j0]);
          r0 = ffma2(make_float2(xs[u], xs[u]), c2, r0);
          r1 = ffma2(make_float2(zs[u], zs[u]), c2, r1);
        }
      }
      *reinterpret_cast<float2*>(&Wt[i0 * LDW + j0]) = r0;
      *reinterpret_cast<float2*>(&Wt[(i0 + 1) * LDW + j0]) = r1;
    }
    if (tid < 256) named_bar_sync(1, 256);
    if (tid < 256) {
      // L^{-1}_{[32,64) [0,32)} = - L^{-1}_{[32,64) [32,64)} W
      const int i0 = 2 * (tid >> 4), j0 = 2 * (tid & 15);
      float2 r0 = make_float2(0.f, 0.f), r1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 32; m += 4) {
        const float4 x = *reinterpret_cast<const float4*>(&Li[(32 + i0) * LDT + 32 + m]);
        const float4 z = *reinterpret_cast<const float4*>(&Li[(33 + i0) * LDT + 32 + m]);
        const float xs[4] = {x.x, x.y, x.z, x.w}, zs[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 c2 = *reinterpret_cast<const float2*>(&Wt[(m + u) * LDW + j0]);
          r0 = ffma2(make_float2(xs[u], xs[u]), c2, r0);
          r1 = ffma2(make_float2(zs[u], zs[u]), c2, r1);
        }
      }
      *reinterpret_cast<float2*>(&Li[(32 + i0) * LDT + j0]) = make_float2(-r0.x, -r0.y);
      *reinterpret_cast<float2*>(&Li[(33 + i0) * LDT + j0]) = make_float2(-r1.x, -r1.y);
    }
    __syncthreads();
    PH(8);

    // ---- phase 4: T^T = (L^{-1} diag(beta))^T into B2 (the B operand of
    // A_qk T and of R = kg^T T) and the identity block of A3's rows 64..;
    // thread = (row r, K group g of 8)
    {
      const int r = tid & 63, g = tid >> 6;
      const float br = s.beta[r];
      uint32_t bv[4], iv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i0 = 8 * g + 2 * u;
        bv[u] = pack_half2(Li[i0 * LDT + r] * br, Li[(i0 + 1) * LDT + r] * br);
        iv[u] = pack_half2(i0 == r ? 1.f : 0.f, i0 + 1 == r ? 1.f : 0.f);
      }
      *reinterpret_cast<uint4*>(A3 + tc::kmajor_offset(64 + r, 64 + 8 * g, 128)) =
          make_uint4(iv[0], iv[1], iv[2], iv[3]);
      *reinterpret_cast<uint4*>(B2 + tc::kmajor_offset(r, 8 * g, 64)) =
          make_uint4(bv[0], bv[1], bv[2], bv[3]);
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    PH(9);

    // ---- phase 5: A_qk T (fp16 MMA) into columns 0..63 and R = kg^T T
    // (A = kg^T) into columns 128..191.  Then -A_qk T goes to A3's rows 64..
    // (beside the identity block) and R, as the A operand of P = -R Kg, over
    // kg^T (its last reader was this product); R leaves for the record from
    // there with the item's other records.
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_kloop(tmem, smem_u32(A2), smem_u32(B2), 128, 64, 64, 0, false);
      tc::mma_kloop(tmem + 128, smem_u32(s.KG), smem_u32(B2), 128, 64, 64, 0, false);
      tc::mma_commit(&s.bar);
    }
    wait_or_abort(&s.bar, bar_phase, &s.abort, p.err);
    bar_phase ^= 1u;
    tc::fence_after_sync();
    {
      const int sp = warp & 3, cq = warp >> 2;
      float b[16];
      tc::tmem_ld16(tc::tmem_addr(tmem, 32 * sp, 128 + 16 * cq), b);
      uint32_t rv[8];
#pragma unroll
      for (int t = 0; t < 16; t += 2) rv[t >> 1] = pack_half2(b[t], b[t + 1]);
      const int k = 32 * sp + lane;
#pragma unroll
      for (int g8 = 0; g8 < 2; ++g8)
        *reinterpret_cast<uint4*>(s.KG + tc::kmajor_offset(k, 16 * cq + 8 * g8, 128)) =
            make_uint4(rv[4 * g8], rv[4 * g8 + 1], rv[4 * g8 + 2], rv[4 * g8 + 3]);
      if (sp < 2) {
        const int r = 32 * sp + lane;
        float a[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, 32 * sp, 16 * cq), a);
        uint32_t neg[8];
#pragma unroll
        for (int t = 0; t < 16; t += 2) neg[t >> 1] = pack_half2(-a[t], -a[t + 1]);
#pragma unroll
        for (int g8 = 0; g8 < 2; ++g8)
          *reinterpret_cast<uint4*>(A3 + tc::kmajor_offset(64 + r, 16 * cq + 8 * g8, 128)) =
              make_uint4(neg[4 * g8], neg[4 * g8 + 1], neg[4 * g8 + 2], neg[4 * g8 + 3]);
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    PH(10);

    // ---- phase 6, one round of three products (A3r = A3's rows 64..,
    // M = 64: row r at TMEM lane r % 16 + 32 (r / 16)):
    //   qg'      = A3r [Kg ; qg] = qg - A_qk T Kg            -> columns 0..127
    //   P'       = R Kg  (P = -P' = -kg^T T Kg = -kg^T w)      -> columns 128..255
    //   -o_intra = A3r[:, 0..63] v = -A_qk T v                -> columns 256..383
    // For the 128-column walk (the pipelined launch, or its own launch) the
    // walk forms o_intra itself: the record carries -qg' and -A_qk T (A3r's
    // first 64 columns) instead of qg' and o_intra, and the third product is
    // not made.
    const bool piped = p.rec128 != 0;
    if (tid == 0) {
      tc::fence_after_sync();
      // P' first, on a barrier of its own: its epilogue runs while the
      // tensor core works on qg' and o_intra
      tc::mma_kloop(tmem + 128, smem_u32(s.KG), smem_u32(s.B3), 128, 128, 64, 0, false);
      tc::mma_commit(&s.bar2);
      const uint64_t a3r = tc::smem_desc(smem_u32(A3) + 1024, 2048, 128);
      tc::mma_run<8>(tmem, a3r, tc::smem_desc(smem_u32(s.B3), 2048, 128), 4096, 4096,
                     tc::idesc_f16(64, 128, 0), false);
      if (!piped)
        tc::mma_run<4>(tmem + 256, a3r, tc::smem_desc(smem_u32(s.VT), 2048, 128), 4096, 4096,
                       tc::idesc_f16(64, 128, 0), false);
      tc::mma_commit(&s.bar);
    }
    wait_or_abort(&s.bar2, bar2_phase, &s.abort, p.err);
    bar2_phase ^= 1u;
    tc::fence_after_sync();
    {
      // P (all 128 lanes), then qg' and o_intra (lanes 0..15 of each
      // sub-partition hold rows 16 sp + lane) into the staging area in their
      // record layouts; warp = (sp, 32-column block cq)
      const int sp = warp & 3, cq = warp >> 2;
      float a[32];
      tc::tmem_ld32(tc::tmem_addr(tmem, 32 * sp, 128 + 32 * cq), a);
      {
        const int k = 32 * sp + lane;
        uint32_t hv[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) hv[t >> 1] = pack_half2(-a[t], -a[t + 1]);
        // columns 32 cq .. are K groups 4 cq .., record bytes 8192 cq ..
        unsigned char* pst = s.XY + (cq < 2 ? ST_P0 : ST_P1 - 16384u);
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8)
          *reinterpret_cast<uint4*>(pst + tc::kmajor_offset(k, 32 * cq + 8 * g8, 128)) =
              make_uint4(hv[4 * g8], hv[4 * g8 + 1], hv[4 * g8 + 2], hv[4 * g8 + 3]);
      }
      wait_or_abort(&s.bar, bar_phase, &s.abort, p.err);
      bar_phase ^= 1u;
      tc::fence_after_sync();
      const int r = 16 * sp + (lane & 15);
      if (piped) {
        // -A_qk T (A3's rows 64.., K groups 0..7) after -qg' in B3, packed to a
        // 64-row K-major operand: thread = (K group tid / 64, row tid % 64)
        const int kg = tid >> 6, rr = tid & 63;
        *reinterpret_cast<uint4*>(s.B3 + QG_BYTES + kg * 1024 + rr * 16) =
            *reinterpret_cast<const uint4*>(A3 + 1024 + kg * 2048 + rr * 16);
      }
      tc::tmem_ld32(tc::tmem_addr(tmem, 32 * sp, 32 * cq), a);
      if (lane < 16) {
        // qg' (pipelined: -qg', staged in B3, which the products have read,
        // since ST_QG lies over A3)
        const float sg = piped ? -1.f : 1.f;
        unsigned char* qst = piped ? s.B3 : s.XY + ST_QG;
        uint32_t hv[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) hv[t >> 1] = pack_half2(sg * a[t], sg * a[t + 1]);
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8)
          *reinterpret_cast<uint4*>(qst + tc::kmajor_offset(r, 32 * cq + 8 * g8, 64)) =
              make_uint4(hv[4 * g8], hv[4 * g8 + 1], hv[4 * g8 + 2], hv[4 * g8 + 3]);
      }
      if (!piped) tc::tmem_ld32(tc::tmem_addr(tmem, 32 * sp, 256 + 32 * cq), a);
      if (!piped && lane < 16) {
        uint32_t ov[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(-a[t], -a[t + 1]);
          ov[t >> 1] = *reinterpret_cast<uint32_t*>(&b2);
        }
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8)
          *reinterpret_cast<uint4*>(s.XY + ST_QG + (CH_OI - CH_QG) + cq * OI_BLOCK + oi_offset(r, g8)) =
              make_uint4(ov[4 * g8], ov[4 * g8 + 1], ov[4 * g8 + 2], ov[4 * g8 + 3]);
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    // the item's P, R, qg' and o_intra records leave by four bulk stores;
    // their shared-memory reads finish before the next item's X / Y build
    // writes over the staging area (and its Kg build over R)
    if (tid == REC_THREAD) {
      bulk_s2g(wsb + CH_P, s.XY + ST_P0, 16384);
      bulk_s2g(wsb + CH_P + 16384, s.XY + ST_P1, 16384);
      bulk_s2g(wsb + CH_R, s.KG, 128 * 64 * 2);
      if (piped) {
        bulk_s2g(wsb + CH_QG, s.B3, QG_BYTES + 64 * 64 * 2);  // -qg', -A_qk T
      } else {
        bulk_s2g(wsb + CH_QG, s.XY + ST_QG, CH_V16 - CH_QG);
      }
      bulk_commit();
      if (p.ready) pending = c_glob * p.hv + h;
    }
    PH(11);
    t = t_next;
  }  // items
  PH_END();
  // after an abort, leave no tile load in flight: wait (bounded) for the last
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0 && s.abort) mbar_wait_bounded(&s.tbar, (tiles_issued - 1) & 1, p.err);
  if (tid == REC_THREAD) {
    bulk_wait<0>();  // every record store has landed
    if (pending >= 0 && !s.abort) publish_ready(p.ready + pending);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <bool CONV, bool FP16>
__global__ void __launch_bounds__(PRO_THREADS, 1)
    kda_prologue_kernel(ChunkParams p, const __grid_constant__ TileMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  prologue_items<CONV, FP16>(p, maps, blockIdx.x, gridDim.x, smem_raw);
}

// --------------------------------------------------------------------------
// Inter-chunk walk on tcgen05, transition form.  One CTA per (block of 32
// value columns, head, sequence x group); thread k of warps 0-3 holds state
// row k in fp32 and TMEM lane k (warps 4-7 the same rows' other 16 of the
// block's 32 columns).  Per chunk c:
//   Y_c = P_c S_c,  RV_c = R_c v_c  (TMEM),   S_{c+1} = d_c * S_c + Y_c + RV_c
//   o_c = qg'_c S_c + o_intra_c   (M = 64: row r at lane r % 16 + 32 (r / 16))
// Warps 0-7 keep the chain; P S, the one product on it, is issued as two
// K halves into two accumulators by threads 0 and 32, which halves its issue
// time, and both halves and R v complete on one barrier; warp 13 issues
// qg' S and the next chunk's R v once that barrier has fired, so that they
// run while the chain threads work, not beside P S; warps 8-11 add o_intra
// and write the output rows; warp 12 streams the records in (chain part
// triple buffered, output part double buffered).
// mode 1 is the group scan's pass one: B_g from a zero state (blocks 0..3)
// and M_g from the identity (blocks 4..7, no R v), no output.
// --------------------------------------------------------------------------
constexpr int WALK_THREADS = 448;
constexpr int CHAIN_THREADS = 256;
constexpr int NB = 32;
constexpr uint32_t S16_LBO = 128, S16_SBO = 2048;  // S^T block, MN-major [v][k]
constexpr uint32_t S16_BYTES = 8192;
constexpr uint32_t B_BYTES = QG_BYTES + OI_BLOCK;  // qg' and this block's o_intra

struct __align__(1024) WalkSmem {
  unsigned char a[3][CH_A_BYTES];   // P, R, d of a chunk
  unsigned char va[3][VB_BYTES];    // this block's v^T, fp16 [v][r] (K groups packed)
  unsigned char b[2][B_BYTES];      // qg' and o_intra of a chunk
  unsigned char s16[3][S16_BYTES];  // fp16 S of the chunk being entered
  uint64_t fullA[3], emptyA[3], fullB[2];
  uint64_t bar_y[2], bar_o[2], o_done[2], s_free[3];
  int issuedA[3], issuedB[2];
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(WalkSmem) <= 227 * 1024, "walk shared memory");

// Element offset of sequence n's head-h initial / final state in
// init_base(p) / final_base(p) (the paged cache, or h0 / hT), or -1 for none.
// Elements are fp32, or bf16 with p.state_bf16.
__device__ __forceinline__ int64_t initial_state_off(const ChunkParams& p, int n, int h) {
  if (p.cache) {
    const int64_t slot = p.state_indices[n];
    if (slot < 0) return -1;
    if (slot >= p.n_slots) { set_error(p.err, ERR_INDEX); return -1; }
    if (p.has_init && !p.has_init[n]) return -1;
    return slot * p.slot_stride + (int64_t)h * D * D;
  }
  return p.h0 ? ((int64_t)n * p.hv + h) * D * D : -1;
}
__device__ __forceinline__ int64_t final_state_off(const ChunkParams& p, int n, int h) {
  if (p.cache) {
    const int64_t slot = p.state_indices[n];
    if (slot < 0 || slot >= p.n_slots) return -1;
    return slot * p.slot_stride + (int64_t)h * D * D;
  }
  return p.hT ? ((int64_t)n * p.hv + h) * D * D : -1;
}
__device__ __forceinline__ const void* init_base(const ChunkParams& p) { return p.cache ? p.cache : p.h0; }
__device__ __forceinline__ void* final_base(const ChunkParams& p) { return p.cache ? p.cache : p.hT; }
__device__ __forceinline__ float state_load(const ChunkParams& p, const void* base, int64_t i) {
  return p.state_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i])
                      : static_cast<const float*>(base)[i];
}
__device__ __forceinline__ void state_store(const ChunkParams& p, void* base, int64_t i, float x) {
  if (p.state_bf16)
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
  else
    static_cast<float*>(base)[i] = x;
}

__device__ __forceinline__ void group_range(const ChunkParams& p, int n, int gidx, int& c0, int& c1) {
  const int base = chunk_off_of(p, n), nc = chunk_off_of(p, n + 1) - base;
  const int per = (nc + p.groups - 1) / p.groups;
  c0 = base + min(nc, gidx * per);
  c1 = base + min(nc, (gidx + 1) * per);
}

__global__ void __launch_bounds__(WALK_THREADS, 1) kda_walk_kernel(ChunkParams p, int mode) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  WalkSmem& s = *reinterpret_cast<WalkSmem*>(smem_raw);
  const int cb = blockIdx.x, h = blockIdx.y;
  const int n = blockIdx.z / p.groups, gidx = blockIdx.z % p.groups;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool ident = mode == 1 && cb >= D / NB;
  const bool outp = mode == 0;
  const int vblk = cb % (D / NB), col0 = vblk * NB;
  int c0, c1;
  group_range(p, n, gidx, c0, c1);
  const int nch = c1 - c0;
  const int64_t plane = (((int64_t)n * p.hv + h) * p.groups + gidx) * D * D;
  const unsigned char* wsb = reinterpret_cast<const unsigned char*>(p.ch);

  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, 256);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) {
      mbar_init(&s.fullA[i], 1);
      mbar_init(&s.emptyA[i], ident ? 2 : 3);  // the chain's two P S halves and warp 9's R v
      mbar_init(&s.s_free[i], 1);
      s.issuedA[i] = 0;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.fullB[i], 1);
      mbar_init(&s.bar_y[i], ident ? 2 : 3);  // the two P S halves and R v
      mbar_init(&s.bar_o[i], 1);
      mbar_init(&s.o_done[i], 4);  // the four output warps
      s.issuedB[i] = 0;
    }
    fence_mbar_init();
    s.abort = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem;
  const uint32_t T_Y = 0, T_RV = 128, T_O = 192;  // Y half j, buffer b at T_Y + 64 j + 32 b

  if (warp < 8) {
    // ---------------- chain: state row k, columns 16 ch ..; threads 0 and 32
    // issue the two halves of P S
    const int k = tid & 127, ch = tid >> 7;
    const int half = tid == 0 ? 0 : (tid == 32 ? 1 : -1);
    float S[16];
    {
      // pass two of a group scan starts from the composed state (fp32),
      // written by the kernel before this one; a serial walk from the
      // sequence's initial state (state dtype), which no kernel of this call
      // writes, so it is read before the wait
      const float* gsrc = (mode == 0 && p.groups > 1) ? p.gS + plane : nullptr;
      if (gsrc) griddep_wait();
      const int64_t ioff = (mode == 0 && p.groups == 1) ? initial_state_off(p, n, h) : -1;
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        const int col = col0 + 16 * ch + v;
        float x = 0.f;
        if (mode == 1) x = (ident && k == col) ? 1.f : 0.f;
        else if (gsrc) x = gsrc[(int64_t)col * D + k];
        else if (ioff >= 0) x = state_load(p, init_base(p), ioff + (int64_t)col * D + k);
        S[v] = x;
      }
      if (!gsrc) griddep_wait();
    }
    // fp16 S^T block: thread (k, ch) writes its 16 columns as two 8-column chunks
    auto write_s16 = [&](int sb) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        *reinterpret_cast<uint4*>(s.s16[sb] + tc::mnmajor_offset(16 * ch + 8 * j, k, S16_LBO, S16_SBO)) =
            make_uint4(pack_half2(S[8 * j], S[8 * j + 1]), pack_half2(S[8 * j + 2], S[8 * j + 3]),
                       pack_half2(S[8 * j + 4], S[8 * j + 5]), pack_half2(S[8 * j + 6], S[8 * j + 7]));
    };
    auto issue_ps = [&](int it) {  // Y_half[it & 1] = P_it[:, half] S16[it % 3][half, :]
      // K = 64 half * 64 ..: 8 K groups of P (2048 bytes each), 8 of S16 (128 bytes)
      tc::mma_kloop_bmn(tmem + T_Y + 64 * half + 32 * (it & 1),
                        smem_u32(s.a[it % 3] + CH_P) + half * 8 * 2048,
                        smem_u32(s.s16[it % 3]) + half * 8 * S16_LBO, 128, 32, 64, S16_LBO, S16_SBO, false);
      tc::mma_commit(&s.bar_y[it & 1]);
    };
    // A failed wait sets ``fail``; the chain stops only at a barrier, all
    // 128 threads together.
    // mid-prefill snapshot of this sequence: after in-sequence chunk ck_j
    int ck_j = -1;
    int64_t ck_off = 0;
    if (mode == 0 && p.ckpt) {
      const int o = p.ckpt_off[n];
      const int len = seq_eos(p, n) - seq_bos(p, n);
      const int64_t row = p.ckpt_idx ? (int64_t)p.ckpt_idx[n] : (int64_t)n;
      if (o > 0 && o % CHUNK == 0 && o <= len && row >= 0) {
        if (row < p.ckpt_rows) {
          ck_j = o / CHUNK - 1;
          ck_off = row * p.ckpt_stride + (int64_t)h * D * D;
        } else if (tid == 0) {
          set_error(p.err, ERR_INDEX);
        }
      }
    }
    const int seq_c0 = chunk_off_of(p, n);
    float dcur = 0.f;
    bool fail = false;
    if (nch > 0) {
      fail = !wait_or_abort(&s.fullA[0], 0, &s.abort, p.err);
      if (!fail) dcur = reinterpret_cast<const float*>(s.a[0] + CH_D)[k];
      write_s16(0);
      fence_proxy_async_smem();
      tc::fence_before_sync();
      fail = named_bar_or(1, CHAIN_THREADS, fail);
      if (half >= 0 && !fail) {
        tc::fence_after_sync();
        issue_ps(0);
      }
    }
    for (int it = 0; !fail && it < nch; ++it) {
      const int yb = it & 1, ab = (it + 1) % 3;
      const bool more = it + 1 < nch;
      float dnext = 0.f;
      // while P S runs: the next record's d, and the S16 buffer it will take
      // (last read by the output product of chunk it - 2)
      if (more) {
        fail = !wait_or_abort(&s.fullA[ab], ((it + 1) / 3) & 1, &s.abort, p.err);
        if (!fail) dnext = reinterpret_cast<const float*>(s.a[ab] + CH_D)[k];
        if (!fail && outp && it >= 2)
          fail = !wait_or_abort(&s.s_free[ab], ((it - 2) / 3) & 1, &s.abort, p.err);
      }
      if (!fail) fail = !wait_or_abort(&s.bar_y[yb], (it >> 1) & 1, &s.abort, p.err);
      if (!fail) {
        tc::fence_after_sync();
        uint32_t y0[16], y1[16], y2[16];
        const uint32_t lanes = tc::tmem_addr(tmem, 32 * (warp & 3), 16 * ch + 32 * yb);
        tc::tmem_ld16_async(lanes + T_Y, y0);
        tc::tmem_ld16_async(lanes + T_Y + 64, y1);
        if (!ident) tc::tmem_ld16_async(lanes + T_RV, y2);
        tc::tmem_wait_ld();
        tc::tmem_regs(y0);
        tc::tmem_regs(y1);
        if (!ident) tc::tmem_regs(y2);
#pragma unroll
        for (int v = 0; v < 16; ++v)
          S[v] = fmaf(dcur, S[v], __uint_as_float(y0[v]) + __uint_as_float(y1[v]) +
                                      (ident ? 0.f : __uint_as_float(y2[v])));
        if (c0 + it - seq_c0 == ck_j)  // S now holds the state after the snapshot's chunk
#pragma unroll
          for (int v = 0; v < 16; ++v) state_store(p, p.ckpt, ck_off + (int64_t)(col0 + 16 * ch + v) * D + k, S[v]);
        if (more) {
          write_s16(ab);
          fence_proxy_async_smem();
        }
      }
      tc::fence_before_sync();
      fail = named_bar_or(1, CHAIN_THREADS, fail);  // Y, RV read; S16 holds S_{it+1}
      if (fail) break;
      if (half >= 0) {
        tc::fence_after_sync();
        tc::mma_commit(&s.emptyA[it % 3]);  // chunk it's P and d
        if (more) issue_ps(it + 1);
      }
      dcur = dnext;
    }
    // end state of this column block, V-first rows col0..: the group scan's
    // operators (fp32), or the sequence's final state (state dtype)
    if (!s.abort) {
      if (mode == 1) {
        float* dst = (ident ? p.gM : p.gB) + plane;
#pragma unroll
        for (int v = 0; v < 16; ++v) dst[(int64_t)(col0 + 16 * ch + v) * D + k] = S[v];
      } else if (p.groups == 1) {
        const int64_t fo = final_state_off(p, n, h);
        if (fo >= 0)
#pragma unroll
          for (int v = 0; v < 16; ++v) state_store(p, final_base(p), fo + (int64_t)(col0 + 16 * ch + v) * D + k, S[v]);
      }
    }
  } else if (warp < 12) {
    // ---------------- output rows: O[b] lanes 16 q .. 16 q + 15 --------------
    griddep_wait();
    const int q = warp - 8, r = 16 * q + (lane & 15);
    for (int it = 0; outp && it < nch; ++it) {
      const int ob = it & 1;
      if (!wait_or_abort(&s.bar_o[ob], (it >> 1) & 1, &s.abort, p.err)) break;
      tc::fence_after_sync();
      float o[32];
      tc::tmem_ld32(tc::tmem_addr(tmem, 32 * q, T_O + 32 * ob), o);
      uint4 oi[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) oi[j] = *reinterpret_cast<const uint4*>(s.b[ob] + QG_BYTES + oi_offset(r, j));
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.o_done[ob]);  // O[ob] and b[ob] read
      // every chunk of this walk belongs to sequence n
      const int bos = seq_bos(p, n) + (c0 + it - chunk_off_of(p, n)) * CHUNK;
      const int len = min(CHUNK, seq_eos(p, n) - bos);
      if (lane < 16 && r < len) {
        __nv_bfloat16* dst = p.out + ((int64_t)(bos + r) * p.hv + h) * D + col0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat162* ib = reinterpret_cast<const __nv_bfloat162*>(&oi[j]);
          uint4 w;
          uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(ib[u]);
            const float a0 = o[8 * j + 2 * u] + f.x, a1 = o[8 * j + 2 * u + 1] + f.y;
            wp[u] = p.in_fp16 ? act_pack2<true>(a0, a1) : act_pack2<false>(a0, a1);
          }
          *reinterpret_cast<uint4*>(dst + 8 * j) = w;
        }
      }
    }
  } else if (warp == 12) {
    // ---------------- loaders: lane 0 the chain's part, lane 16 the output's;
    // each also warms L2 with the record it will load LOOKAHEAD chunks later.
    // The records come from the kernel before this one, which may still be
    // finishing under a programmatic launch.
    griddep_wait();
    constexpr int LOOKAHEAD = 4;
    if (lane == 0) {
      for (int it = 0; it < nch; ++it) {
        const unsigned char* src = wsb + ((size_t)(c0 + it) * p.hv + h) * CH_BYTES;
        if (it == 0)
          for (int j = 1; j < LOOKAHEAD && j < nch; ++j)
            bulk_prefetch_l2(wsb + ((size_t)(c0 + j) * p.hv + h) * CH_BYTES, CH_A_BYTES);
        if (it + LOOKAHEAD < nch)
          bulk_prefetch_l2(wsb + ((size_t)(c0 + it + LOOKAHEAD) * p.hv + h) * CH_BYTES, CH_A_BYTES);
        const int ab = it % 3;
        if (it >= 3 && !wait_or_abort(&s.emptyA[ab], ((it / 3) - 1) & 1, &s.abort, p.err)) break;
        mbar_arrive_expect_tx(&s.fullA[ab], CH_A_BYTES + (ident ? 0u : VB_BYTES));
        bulk_g2s(s.a[ab], src + CH_P, 32768, &s.fullA[ab]);
        bulk_g2s(s.a[ab] + 32768, src + CH_P + 32768, CH_A_BYTES - 32768, &s.fullA[ab]);
        if (!ident)  // the block's 32 rows of each of the 8 K groups
          for (int kg = 0; kg < 8; ++kg)
            bulk_g2s(s.va[ab] + kg * VB_ROWS_BYTES, src + CH_V16 + kg * 2048 + vblk * VB_ROWS_BYTES,
                     VB_ROWS_BYTES, &s.fullA[ab]);
        s.issuedA[ab] += 1;
      }
    } else if (lane == 16 && outp) {
      for (int it = 0; it < nch; ++it) {
        const unsigned char* src = wsb + ((size_t)(c0 + it) * p.hv + h) * CH_BYTES;
        if (it + LOOKAHEAD < nch)
          bulk_prefetch_l2(wsb + ((size_t)(c0 + it + LOOKAHEAD) * p.hv + h) * CH_BYTES + CH_QG,
                           CH_BYTES - CH_QG);
        const int bb = it & 1;
        if (it >= 2 && !wait_or_abort(&s.o_done[bb], ((it >> 1) - 1) & 1, &s.abort, p.err)) break;
        mbar_arrive_expect_tx(&s.fullB[bb], B_BYTES);
        bulk_g2s(s.b[bb], src + CH_QG, QG_BYTES, &s.fullB[bb]);
        bulk_g2s(s.b[bb] + QG_BYTES, src + CH_OI + vblk * OI_BLOCK, OI_BLOCK, &s.fullB[bb]);
        s.issuedB[bb] += 1;
      }
    }
  } else if (!ident) {
    // ---------------- R v one chunk ahead, and qg' S ----------------
    griddep_wait();
    if (lane == 0) {
      auto issue_rv = [&](int it) {  // RV[it & 1] = R_it v_it
        const int ab = it % 3;
        if (!wait_or_abort(&s.fullA[ab], (it / 3) & 1, &s.abort, p.err)) return false;
        tc::fence_after_sync();
        tc::mma_kloop(tmem + T_RV + 32 * (it & 1), smem_u32(s.a[ab] + CH_R), smem_u32(s.va[ab]), 128, 32,
                      64, 0, false);
        tc::mma_commit(&s.bar_y[it & 1]);
        return true;
      };
      bool go = nch > 0 && issue_rv(0);
      for (int it = 0; go && it < nch; ++it) {
        const int ob = it & 1, sb = it % 3;
        // chunk it's P S and R v are done: S16[sb] holds S_it and the chain
        // has read RV of chunk it - 1
        if (!wait_or_abort(&s.bar_y[ob], (it >> 1) & 1, &s.abort, p.err)) break;
        if (outp) {
          if (!wait_or_abort(&s.fullB[ob], (it >> 1) & 1, &s.abort, p.err)) break;
          if (it >= 2 && !wait_or_abort(&s.o_done[ob], ((it >> 1) - 1) & 1, &s.abort, p.err)) break;
          tc::fence_after_sync();
          tc::mma_kloop_bmn(tmem + T_O + 32 * ob, smem_u32(s.b[ob]), smem_u32(s.s16[sb]), 64, 32, 128,
                            S16_LBO, S16_SBO, false);
          tc::mma_commit(&s.bar_o[ob]);
          tc::mma_commit(&s.s_free[sb]);
        }
        if (it + 1 < nch && !issue_rv(it + 1)) break;
        tc::mma_commit(&s.emptyA[sb]);  // chunk it's R and v
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0 && s.abort) {
    // leave no bulk copy in flight: wait (bounded) for the last load of each buffer
    for (int i = 0; i < 3; ++i)
      if (s.issuedA[i] > 0) mbar_wait_bounded(&s.fullA[i], (s.issuedA[i] - 1) & 1, p.err);
    for (int i = 0; i < 2; ++i)
      if (s.issuedB[i] > 0) mbar_wait_bounded(&s.fullB[i], (s.issuedB[i] - 1) & 1, p.err);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// --------------------------------------------------------------------------
// Pipelined launch: one cooperative kernel whose first walk_ctas CTAs each
// walk one (sequence, head) chain over all 128 value columns, while the
// other CTAs run the prologue in level-major item order (chunk j of every
// chain before chunk j + 1 of any) and raise a ready flag per record.  A
// walk CTA loads chunk c's record once its flag is up, so a chain's walk
// runs behind the prologue instead of after it.  Prologue CTAs never wait
// on a walk CTA, and a cooperative launch keeps every CTA resident, so each
// flag a walk CTA waits for is eventually raised.
//
// Walk CTA (512 threads), per chunk c of the chain:
//   Y = P_c S_c (two K halves, R_c v_c added to half 0),  S_{c+1} = d_c * S_c + Y
//   o_c = -[(-qg'_c) S_c + (-A_qk T)_c v_c]               (M = 64)
// (the record of this launch carries -qg' and -A_qk T; o_intra = A_qk T v
// is formed here, off the chain)
// warps 0-7    the chain: thread (k, ch) holds state row k, value columns
//              64 ch .. 64 ch + 63 in fp32 (TMEM lane k); threads 0 and 32
//              issue the two K halves of P S, thread 0 also R v.
// warps 8-11   the output: rows 16 q .. 16 q + 15 (TMEM lanes 32 q ..) to out.
// warp 12      lane 0 waits for each record's flag, then loads P, R, d, v^T
//              (A, double buffered) and -qg', -A_qk T (B).
// warp 13      lane 0 issues chunk c's output products once its P S has
//              completed (its fp16 S is then written).
// TMEM: Y half 0 at column 0, half 1 at 128, the output at 256 and 384.
// --------------------------------------------------------------------------
constexpr int PIPE_MAX_CHAINS = 48;      // walk CTAs at most
constexpr int PIPE_MIN_PROLOGUE = 64;    // prologue CTAs at least
constexpr uint32_t WA_BYTES = CH_A_BYTES + V16_BYTES;  // P, R, d, then v^T
constexpr uint32_t S16F_BYTES = 128 * 128 * 2;         // fp16 S, MN-major [v][k]

constexpr uint32_t WB_BYTES = QG_BYTES + 64 * 64 * 2;  // -qg', then -A_qk T (K-major, K groups 1024 B apart)

struct __align__(1024) Walk128Smem {
  unsigned char a[2][WA_BYTES];
  unsigned char b[WB_BYTES];
  unsigned char s16[2][S16F_BYTES];
  uint64_t fullA[2], emptyA[2], fullB, freeB, bar_y[2], bar_o[2], o_done[2], s_free[2];
  int issuedA[2], issuedB;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(Walk128Smem) <= 227 * 1024, "pipelined walk shared memory");
static_assert(WA_BYTES % 16 == 0 && CH_A_BYTES % 16 == 0, "bulk copy alignment");

// Drop one 128-byte line from L2 without writing it back (its contents
// become undefined): for records that no one reads again.
__device__ __forceinline__ void discard_l2(const void* line) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait for a record's ready flag (bounded, like wait_or_abort): on expiry
// sets ERR_TIMEOUT and raises the CTA's abort flag.
__device__ __forceinline__ bool wait_ready_or_abort(const unsigned* flag, volatile int* abort, unsigned* err) {
  if (ld_acquire_gpu(flag)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < WAIT_CAP; ++i) {
    __nanosleep(64);
    if (ld_acquire_gpu(flag)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > WAIT_NS) break;
  }
  set_error(err, ERR_TIMEOUT);
  *abort = 1;
  return false;
}

// Measurement build only: cycles of the pipelined walk's chain (thread 0)
// per activity, summed over chunks and walk CTAs: [0] waiting for the next
// record and S16 buffer, [1] waiting for P S, [2] the state update and S16
// write, [3] barrier and issue; the loader's [4] ready-flag and [5] buffer
// waits; [6] chunk steps.
#ifdef KDA_PHASE_TIMING
constexpr int N_WALK_CTR = 6;
__device__ unsigned long long g_walk_cycles[N_WALK_CTR + 1];
#define WK_MARK(t) const long long t = clock64()
#define WK_ADD(acc, t)                                                  \
  do {                                                                  \
    const long long n_ = clock64();                                     \
    acc += (unsigned long long)(n_ - t);                                \
  } while (0)
#else
#define WK_MARK(t) \
  do {             \
  } while (0)
#define WK_ADD(acc, t) \
  do {                 \
  } while (0)
#endif

__device__ __forceinline__ void walk_chain128(const ChunkParams& p, int chain, unsigned char* smem_raw) {
  Walk128Smem& s = *reinterpret_cast<Walk128Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = chain / p.hv, h = chain - n * p.hv;
  const int c0 = chunk_off_of(p, n), nch = chunk_off_of(p, n + 1) - c0;
  const unsigned char* wsb = reinterpret_cast<const unsigned char*>(p.ch);
  const unsigned* ready = p.ready ? p.ready + (size_t)c0 * p.hv + h : nullptr;  // chunk it's flag: ready[it * Hv]

  if (warp == 0) {
    tc::tmem_alloc(&s.tmem, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.fullA[i], 1);
      mbar_init(&s.emptyA[i], 3);  // threads 0, 32 and warp 13's lane 0, once their products have read A
      mbar_init(&s.bar_y[i], 2);   // the two P S halves (R v with half 0)
      mbar_init(&s.bar_o[i], 1);
      mbar_init(&s.o_done[i], 4);  // the four output warps
      mbar_init(&s.s_free[i], 1);
      s.issuedA[i] = 0;
    }
    mbar_init(&s.fullB, 1);
    mbar_init(&s.freeB, 1);
    s.issuedB = 0;
    fence_mbar_init();
    s.abort = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem;
  constexpr uint32_t T_Y = 0, T_O = 256;

  if (warp < 8) {
    // ---------------- chain ----------------
    const int k = tid & 127, ch = tid >> 7;
    const int half = tid == 0 ? 0 : (tid == 32 ? 1 : -1);
    float S[64];
    {
      const int64_t ioff = initial_state_off(p, n, h);
#pragma unroll
      for (int v = 0; v < 64; ++v)
        S[v] = ioff >= 0 ? state_load(p, init_base(p), ioff + (int64_t)(64 * ch + v) * D + k) : 0.f;
    }
    auto write_s16 = [&](int sb) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(s.s16[sb] + tc::mnmajor_offset(64 * ch + 8 * j, k, S16_LBO, S16_SBO)) =
            make_uint4(pack_half2(S[8 * j], S[8 * j + 1]), pack_half2(S[8 * j + 2], S[8 * j + 3]),
                       pack_half2(S[8 * j + 4], S[8 * j + 5]), pack_half2(S[8 * j + 6], S[8 * j + 7]));
    };
    // chunk it's products from A[it & 1] and S16[it & 1]: Y half = P[:, half] S[half, :]
    auto issue = [&](int it) {
      const int b = it & 1;
      tc::mma_kloop_bmn(tmem + T_Y + 128 * half, smem_u32(s.a[b] + CH_P) + half * 8 * 2048,
                        smem_u32(s.s16[b]) + half * 8 * S16_LBO, 128, 128, 64, S16_LBO, S16_SBO, false);
      if (half == 0)
        tc::mma_kloop(tmem + T_Y, smem_u32(s.a[b] + CH_R), smem_u32(s.a[b] + CH_A_BYTES), 128, 128, 64, 0, true);
      tc::mma_commit(&s.bar_y[b]);
      tc::mma_commit(&s.emptyA[b]);
    };
    // mid-prefill snapshot of this sequence: the state after in-sequence chunk ck_j
    int ck_j = -1;
    int64_t ck_off = 0;
    if (p.ckpt) {
      const int o = p.ckpt_off[n];
      const int len = seq_eos(p, n) - seq_bos(p, n);
      const int64_t row = p.ckpt_idx ? (int64_t)p.ckpt_idx[n] : (int64_t)n;
      if (o > 0 && o % CHUNK == 0 && o <= len && row >= 0) {
        if (row < p.ckpt_rows) {
          ck_j = o / CHUNK - 1;
          ck_off = row * p.ckpt_stride + (int64_t)h * D * D;
        } else if (tid == 0) {
          set_error(p.err, ERR_INDEX);
        }
      }
    }
    float dcur = 0.f;
    bool fail = false;
    if (nch > 0) {
      fail = !wait_or_abort(&s.fullA[0], 0, &s.abort, p.err);
      if (!fail) dcur = reinterpret_cast<const float*>(s.a[0] + CH_D)[k];
      write_s16(0);
      fence_proxy_async_smem();
      tc::fence_before_sync();
      fail = named_bar_or(1, CHAIN_THREADS, fail);
      if (half >= 0 && !fail) {
        tc::fence_after_sync();
        issue(0);
      }
    }
#ifdef KDA_PHASE_TIMING
    unsigned long long wk[4] = {0, 0, 0, 0};
#endif
    for (int it = 0; !fail && it < nch; ++it) {
      const int b = it & 1, nb = b ^ 1;
      const bool more = it + 1 < nch;
      float dnext = 0.f;
      WK_MARK(wk0);
      // while P S runs: the next record (its d) and the S16 buffer the next
      // state goes to, last read by the output product of chunk it - 1
      if (more) {
        fail = !wait_or_abort(&s.fullA[nb], ((it + 1) >> 1) & 1, &s.abort, p.err);
        if (!fail) dnext = reinterpret_cast<const float*>(s.a[nb] + CH_D)[k];
        if (!fail && it >= 1) fail = !wait_or_abort(&s.s_free[nb], ((it - 1) >> 1) & 1, &s.abort, p.err);
      }
      WK_ADD(wk[0], wk0);
      WK_MARK(wk1);
      if (!fail) fail = !wait_or_abort(&s.bar_y[b], (it >> 1) & 1, &s.abort, p.err);
      WK_ADD(wk[1], wk1);
      WK_MARK(wk2);
      if (!fail) {
        tc::fence_after_sync();
        const uint32_t lanes = tc::tmem_addr(tmem, 32 * (warp & 3), 64 * ch);
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          uint32_t y0[16], y1[16];
          tc::tmem_ld16_async(lanes + T_Y + 16 * pc, y0);
          tc::tmem_ld16_async(lanes + T_Y + 128 + 16 * pc, y1);
          tc::tmem_wait_ld();
          tc::tmem_regs(y0);
          tc::tmem_regs(y1);
#pragma unroll
          for (int v = 0; v < 16; ++v)
            S[16 * pc + v] = fmaf(dcur, S[16 * pc + v], __uint_as_float(y0[v]) + __uint_as_float(y1[v]));
        }
        if (it == ck_j)  // S now holds the state after the snapshot's chunk
#pragma unroll
          for (int v = 0; v < 64; ++v) state_store(p, p.ckpt, ck_off + (int64_t)(64 * ch + v) * D + k, S[v]);
        if (more) {
          write_s16(nb);
          fence_proxy_async_smem();
        }
      }
      WK_ADD(wk[2], wk2);
      WK_MARK(wk3);
      tc::fence_before_sync();
      fail = named_bar_or(1, CHAIN_THREADS, fail);  // Y read; S16[nb] holds S_{it+1}
      if (fail) break;
      if (half >= 0 && more) {
        tc::fence_after_sync();
        issue(it + 1);
      }
      WK_ADD(wk[3], wk3);
      dcur = dnext;
    }
#ifdef KDA_PHASE_TIMING
    if (tid == 0) {
      for (int i = 0; i < 4; ++i) atomicAdd(&g_walk_cycles[i], wk[i]);
      atomicAdd(&g_walk_cycles[N_WALK_CTR], (unsigned long long)nch);
    }
#endif
    if (!s.abort) {
      const int64_t fo = final_state_off(p, n, h);
      if (fo >= 0)
#pragma unroll
        for (int v = 0; v < 64; ++v) state_store(p, final_base(p), fo + (int64_t)(64 * ch + v) * D + k, S[v]);
    }
  } else if (warp < 12) {
    // ---------------- output rows 16 q .. 16 q + 15 ----------------
    const int q = warp - 8, r = 16 * q + (lane & 15);
    for (int it = 0; it < nch; ++it) {
      const int ob = it & 1;
      if (!wait_or_abort(&s.bar_o[ob], (it >> 1) & 1, &s.abort, p.err)) break;
      tc::fence_after_sync();
      const int bos = seq_bos(p, n) + it * CHUNK;
      const int len = min(CHUNK, seq_eos(p, n) - bos);
      __nv_bfloat16* dst = p.out + ((int64_t)(bos + r) * p.hv + h) * D;
#pragma unroll
      for (int jb = 0; jb < 4; ++jb) {
        float o[32];
        tc::tmem_ld32(tc::tmem_addr(tmem, 32 * q, T_O + 128 * ob + 32 * jb), o);
        if (lane < 16 && r < len) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 w;
            uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // the accumulator holds -o
              const float a0 = -o[8 * j + 2 * u], a1 = -o[8 * j + 2 * u + 1];
              wp[u] = p.in_fp16 ? act_pack2<true>(a0, a1) : act_pack2<false>(a0, a1);
            }
            *reinterpret_cast<uint4*>(dst + 32 * jb + 8 * j) = w;
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.o_done[ob]);  // O[ob] read
    }
  } else if (warp == 12) {
    // ---------------- loader: lane 0 waits and loads; in the pipelined
    // launch the whole warp then drops from L2 the record of two chunks
    // back, which every reader has finished with (chunk it - 2's A buffer
    // is empty and chunk it - 1's B load was allowed), so that a record that
    // lives a few microseconds is never written back to HBM
#ifdef KDA_PHASE_TIMING
    unsigned long long wf = 0, wb = 0;
#endif
    for (int it = 0; it < nch; ++it) {
      const int b = it & 1;
      int go = 1;
      if (lane == 0) {
        WK_MARK(wl0);
        if (p.ready) {  // pipelined: this record's flag
          if (!wait_ready_or_abort(ready + (size_t)it * p.hv, &s.abort, p.err)) go = 0;
          asm volatile("fence.proxy.async.global;" ::: "memory");  // the bulk loads below read it
        } else if (it == 0) {
          griddep_wait();  // a launch of its own: the prologue before it has finished
        }
        WK_ADD(wf, wl0);
        const unsigned char* src = wsb + ((size_t)(c0 + it) * p.hv + h) * CH_BYTES;
        WK_MARK(wl1);
        if (go && it >= 2 && !wait_or_abort(&s.emptyA[b], ((it >> 1) - 1) & 1, &s.abort, p.err)) go = 0;
        WK_ADD(wb, wl1);
        if (go) {
          mbar_arrive_expect_tx(&s.fullA[b], WA_BYTES);
          bulk_g2s(s.a[b], src + CH_P, 32768, &s.fullA[b]);
          bulk_g2s(s.a[b] + 32768, src + CH_P + 32768, CH_A_BYTES - 32768, &s.fullA[b]);
          bulk_g2s(s.a[b] + CH_A_BYTES, src + CH_V16, V16_BYTES, &s.fullA[b]);
          s.issuedA[b] += 1;
        }
        if (go && it >= 1 && !wait_or_abort(&s.freeB, (it - 1) & 1, &s.abort, p.err)) go = 0;
        if (go) {
          mbar_arrive_expect_tx(&s.fullB, WB_BYTES);
          bulk_g2s(s.b, src + CH_QG, WB_BYTES, &s.fullB);  // -qg' and -A_qk T are adjacent
          s.issuedB += 1;
        }
      }
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      // only whole lines of this record: the record area must be 128-byte
      // aligned (the workspace need only be 16-byte aligned), or a line
      // would reach into another chain's record
      if (p.ready && it >= 2 && (reinterpret_cast<uintptr_t>(wsb) & 127u) == 0) {
        const unsigned char* old = wsb + ((size_t)(c0 + it - 2) * p.hv + h) * CH_BYTES;
        for (uint32_t off = 128u * lane; off < CH_BYTES; off += 32u * 128u) discard_l2(old + off);
      }
    }
#ifdef KDA_PHASE_TIMING
    if (lane == 0) {
      atomicAdd(&g_walk_cycles[4], wf);
      atomicAdd(&g_walk_cycles[5], wb);
    }
#endif
  } else if (warp == 13) {
    // ---------------- qg' S ----------------
    if (lane == 0) {
      for (int it = 0; it < nch; ++it) {
        const int b = it & 1;
        // chunk it's P S has completed, so S16[b] holds S_it
        if (!wait_or_abort(&s.bar_y[b], (it >> 1) & 1, &s.abort, p.err)) break;
        if (!wait_or_abort(&s.fullB, it & 1, &s.abort, p.err)) break;
        if (it >= 2 && !wait_or_abort(&s.o_done[b], ((it >> 1) - 1) & 1, &s.abort, p.err)) break;
        tc::fence_after_sync();
        // -o = (-qg') S + (-A_qk T) v; v^T sits in chunk it's A buffer
        tc::mma_kloop_bmn(tmem + T_O + 128 * b, smem_u32(s.b), smem_u32(s.s16[b]), 64, 128, 128, S16_LBO,
                          S16_SBO, false);
        tc::mma_kloop(tmem + T_O + 128 * b, smem_u32(s.b + QG_BYTES), smem_u32(s.a[b] + CH_A_BYTES), 64, 128,
                      64, 0, true);
        tc::mma_commit(&s.bar_o[b]);
        tc::mma_commit(&s.s_free[b]);
        tc::mma_commit(&s.freeB);
        tc::mma_commit(&s.emptyA[b]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0 && s.abort) {
    // leave no bulk copy in flight: wait (bounded) for the last load of each buffer
    for (int i = 0; i < 2; ++i)
      if (s.issuedA[i] > 0) mbar_wait_bounded(&s.fullA[i], (s.issuedA[i] - 1) & 1, p.err);
    if (s.issuedB > 0) mbar_wait_bounded(&s.fullB, (s.issuedB - 1) & 1, p.err);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// Measurement build only: each CTA's span in the pipelined kernel, as
// %globaltimer ns at start and end and SM cycles in between (thread 0).
#ifdef KDA_PHASE_TIMING
constexpr int MAX_SPAN_CTAS = 256;
__device__ unsigned long long g_cta_span[MAX_SPAN_CTAS][4];
#endif

template <bool CONV, bool FP16>
__global__ void __launch_bounds__(PRO_THREADS, 1)
    kda_pipelined_kernel(ChunkParams p, const __grid_constant__ TileMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
#ifdef KDA_PHASE_TIMING
  const unsigned long long g0 = globaltimer_ns();
  const long long c0 = clock64();
#endif
  if ((int)blockIdx.x < p.walk_ctas)
    walk_chain128(p, blockIdx.x, smem_raw);
  else
    prologue_items<CONV, FP16>(p, maps, blockIdx.x - p.walk_ctas, gridDim.x - p.walk_ctas, smem_raw);
#ifdef KDA_PHASE_TIMING
  if (threadIdx.x == 0 && blockIdx.x < MAX_SPAN_CTAS) {
    g_cta_span[blockIdx.x][0] = g0;
    g_cta_span[blockIdx.x][1] = globaltimer_ns();
    g_cta_span[blockIdx.x][2] = (unsigned long long)(clock64() - c0);
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_cta_span[blockIdx.x][3] = smid;
  }
#endif
}
constexpr size_t PIPE_SMEM = sizeof(Walk128Smem) > sizeof(ProSmem) ? sizeof(Walk128Smem) : sizeof(ProSmem);

// The 128-column walk as a launch of its own after the prologue (one CTA per
// (sequence, head) chain), for calls with more chains than the pipelined
// launch takes: it needs a quarter of the 32-column walk's CTAs for about
// the same time per chunk.  Launched programmatically; the loader waits for
// the prologue before its first record load.
__global__ void __launch_bounds__(PRO_THREADS, 1) kda_walk128_kernel(ChunkParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  walk_chain128(p, blockIdx.x, smem_raw);
}

// --------------------------------------------------------------------------
// Group composition: S_{g+1}^T = S_g^T M_g^T + B_g^T serially over groups,
// recording each group's incoming state; the last one is the final state.
// One CTA (256 threads) per (value block of 32 rows, head, sequence).
// --------------------------------------------------------------------------
constexpr int COMPOSE_THREADS = 256;

__global__ void __launch_bounds__(COMPOSE_THREADS, 1) kda_compose_kernel(ChunkParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  float* St = reinterpret_cast<float*>(smem_raw);  // [32][128] rows v0..v0+31 of S^T
  float* Mt = St + NB * D;                         // [128][128]
  const int vb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x;
  const int v0 = vb * NB;
  const int64_t ioff = initial_state_off(p, n, h);
  for (int e = tid; e < NB * D; e += COMPOSE_THREADS)
    St[e] = ioff >= 0 ? state_load(p, init_base(p), ioff + (int64_t)v0 * D + e) : 0.f;
  __syncthreads();
  for (int gi = 0; gi < p.groups; ++gi) {
    const int64_t plane = (((int64_t)n * p.hv + h) * p.groups + gi) * D * D;
    for (int e = tid; e < NB * D; e += COMPOSE_THREADS) p.gS[plane + (int64_t)v0 * D + e] = St[e];
    for (int e = tid; e < D * D; e += COMPOSE_THREADS) Mt[e] = p.gM[plane + e];
    __syncthreads();
    const int v = tid >> 3, kq = tid & 7;
    float acc[16];
#pragma unroll
    for (int j2 = 0; j2 < 16; ++j2) acc[j2] = p.gB[plane + (int64_t)(v0 + v) * D + kq + 8 * j2];
    for (int m = 0; m < D; ++m) {
      const float sv = St[v * D + m];
#pragma unroll
      for (int j2 = 0; j2 < 16; ++j2) acc[j2] = fmaf(sv, Mt[m * D + kq + 8 * j2], acc[j2]);
    }
    __syncthreads();
#pragma unroll
    for (int j2 = 0; j2 < 16; ++j2) St[v * D + kq + 8 * j2] = acc[j2];
    __syncthreads();
  }
  const int64_t fo = final_state_off(p, n, h);
  if (fo >= 0)
    for (int e = tid; e < NB * D; e += COMPOSE_THREADS) state_store(p, final_base(p), fo + (int64_t)v0 * D + e, St[e]);
}

// --------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------
static size_t int_words(int n_seqs, int max_chunks) {
  size_t ints = 4 + (size_t)(n_seqs + 1) + 2 * (size_t)max_chunks;
  return (ints + 63) & ~(size_t)63;  // keep the record area 256-byte aligned
}

size_t chunk_workspace_floats(int n_seqs, int t_total, int hv, int groups, int* max_chunks_out) {
  const int max_chunks = t_total / CHUNK + n_seqs;
  if (max_chunks_out) *max_chunks_out = max_chunks;
  size_t words = int_words(n_seqs, max_chunks);
  words += (size_t)max_chunks * hv * (CH_BYTES / 4);
  if (groups > 1) words += 3 * (size_t)n_seqs * hv * groups * D * D;
  words += (size_t)max_chunks * hv + 1;  // the pipelined launch's ready flags and item counter
  return words;  // 4-byte words
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda)
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// rows of ``heads`` x 128 bf16 per token: dims (128, heads, T), box (128, 1, rows)
static bool encode_rows(CUtensorMap* map, const void* base, int heads, int T, int64_t st_head,
                        int64_t st_tok, bool fp16, int rows = CHUNK) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)st_head * 2, (cuuint64_t)st_tok * 2};
  const cuuint32_t box[3] = {(cuuint32_t)D, 1u, (cuuint32_t)rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Does the pipelined launch beat the two launches?  Estimated step times (us)
// from measured GB300 rates: a prologue item takes about T_ITEM on its SM, a
// chunk step of the 32-column walk T_STEP32 and of the pipelined 128-column
// walk T_STEP128.  Two launches: the prologue's waves, then the walk's
// chains.  Pipelined: the prologue's waves on the SMs the chains leave, or
// one item and a whole chain, whichever is longer.
static bool pipeline_pays(int items, int chains, int chunks_per_chain, int sms) {
  constexpr double T_ITEM = 10.0, T_STEP32 = 1.06, T_STEP128 = 1.3;
  auto waves = [](long work, long width) { return (double)((work + width - 1) / width); };
  const double two = waves(items, sms) * T_ITEM + waves(4L * chains, sms) * chunks_per_chain * T_STEP32;
  const double pro = waves(items, sms - chains) * T_ITEM, walk = T_ITEM + chunks_per_chain * T_STEP128;
  return (pro > walk ? pro : walk) < two;
}

int launch_chunk(ChunkParams p, void* workspace, cudaStream_t stream) {
  static uint64_t attrs_done = 0;
  once_per_device(attrs_done, [](int) {
    cudaFuncSetAttribute(kda_prologue_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(ProSmem));
    cudaFuncSetAttribute(kda_prologue_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(ProSmem));
    cudaFuncSetAttribute(kda_prologue_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(ProSmem));
    cudaFuncSetAttribute(kda_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(WalkSmem));
    cudaFuncSetAttribute(kda_compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)((NB * D + D * D) * sizeof(float)));
    cudaFuncSetAttribute(kda_pipelined_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)PIPE_SMEM);
    cudaFuncSetAttribute(kda_pipelined_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)PIPE_SMEM);
    cudaFuncSetAttribute(kda_pipelined_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)PIPE_SMEM);
    cudaFuncSetAttribute(kda_walk128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(Walk128Smem));
  });
  int max_chunks = 0;
  chunk_workspace_floats(p.n_seqs, p.t_total, p.hv, p.groups, &max_chunks);
  int32_t* iw = reinterpret_cast<int32_t*>(workspace);
  p.max_chunks = max_chunks;
  p.n_chunks = iw;
  p.chunk_off = iw + 4;
  p.chunk_seq = p.chunk_off + (p.n_seqs + 1);
  p.chunk_j = p.chunk_seq + max_chunks;
  float* fw = reinterpret_cast<float*>(iw + int_words(p.n_seqs, max_chunks));
  p.ch = fw;
  fw += (size_t)max_chunks * p.hv * (CH_BYTES / 4);
  if (p.groups > 1) {
    const size_t plane = (size_t)p.n_seqs * p.hv * p.groups * D * D;
    p.gM = fw;
    p.gB = fw + plane;
    p.gS = fw + 2 * plane;
    fw += 3 * plane;
  }
  unsigned* ready_flags = reinterpret_cast<unsigned*>(fw);
  const int items = max_chunks * p.hv;
  const int sms = p.sm_count > 0 ? p.sm_count : 152;
  const int chains = p.n_seqs * p.hv;
  const bool can_pipe = p.groups == 1 && !p.cu_seqlens && chains <= PIPE_MAX_CHAINS &&
                        sms - chains >= PIPE_MIN_PROLOGUE;
  if (p.pipeline == 2 && !can_pipe) {
    set_last_error(KDA_ERR_INVALID_ARGUMENT,
                   "kda_chunk_fwd: groups = -1 (pipelined launch) needs dense sequences (no cu_seqlens) and at "
                   "most 48 (sequence, head) chains.");
    return -2;
  }
  // a serial walk in a launch of its own: the 128-column walk (one CTA per
  // chain) once the 32-column walk's four CTAs per chain would not fit on
  // the SMs in one wave
  const bool walk128 = p.groups == 1 && 4L * chains > sms;
  if (p.cu_seqlens) {  // dense sequences have closed-form chunk tables
    trace_begin("kda_chunk_index", stream);
    kda_chunk_index_kernel<<<1, 256, 0, stream>>>(p);
    trace_end(stream);
  }
  // a conv with a scratch buffer: convolve every (token, channel) once, then
  // run the plain prologue on the convolved bands (pp); the conv state update
  // below still reads the raw bands of p
  ChunkParams pp = p;
  if (p.conv.state && p.conv_out) {
    if (launch_conv_prefill(p, stream) != 0) return -1;
    const int64_t qk = (int64_t)p.hqk * D;
    pp.q = p.conv_out;
    pp.k = p.conv_out + (int64_t)p.t_total * qk;
    pp.v = p.conv_out + 2 * (int64_t)p.t_total * qk;
    pp.q_st = pp.k_st = qk;
    pp.v_st = (int64_t)p.hv * D;
    pp.q_sh = pp.k_sh = pp.v_sh = D;
    pp.conv.state = nullptr;
  }
  TileMaps maps;
  const int qkv_rows = CHUNK + (pp.conv.state ? HALO : 0);
  const bool f16 = pp.in_fp16 != 0;
  if (!encode_rows(&maps.q, pp.q, pp.hqk, pp.t_total, pp.q_sh, pp.q_st, f16, qkv_rows) ||
      !encode_rows(&maps.k, pp.k, pp.hqk, pp.t_total, pp.k_sh, pp.k_st, f16, qkv_rows) ||
      !encode_rows(&maps.g, pp.g, pp.hv, pp.t_total, pp.g_sh, pp.g_st, f16) ||
      !encode_rows(&maps.v, pp.v, pp.hv, pp.t_total, pp.v_sh, pp.v_st, f16, qkv_rows)) {
    set_last_error(KDA_ERR_INVALID_ARGUMENT,
                   "kda_chunk_fwd: q/k/v/g layout cannot be described by a TMA tensor map "
                   "(strides must be positive multiples of 8 elements below 2^39 bytes).");
    return -2;
  }
  const int cps = p.dense_len > 0 ? (p.dense_len + CHUNK - 1) / CHUNK : 0;  // chunks per dense sequence
  const bool pipe = p.pipeline == 2 || (p.pipeline == 1 && can_pipe && pipeline_pays(chains * cps, chains, cps, sms));
  pp.rec128 = (pipe || walk128) ? 1 : 0;
  if (pipe) {
    const int grid = chains + (items < sms - chains ? items : sms - chains);
    pp.walk_ctas = chains;
    pp.ready = ready_flags;
    pp.item_counter = ready_flags + items;
    if (cudaMemsetAsync(ready_flags, 0, (size_t)(items + 1) * sizeof(unsigned), stream) != cudaSuccess) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(PRO_THREADS);
    cfg.dynamicSmemBytes = PIPE_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: each awaited flag gets raised
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    trace_begin("kda_pipelined", stream);
    cudaError_t e;
    if (pp.conv.state)
      e = cudaLaunchKernelEx(&cfg, kda_pipelined_kernel<true, false>, pp, maps);
    else if (pp.in_fp16)
      e = cudaLaunchKernelEx(&cfg, kda_pipelined_kernel<false, true>, pp, maps);
    else
      e = cudaLaunchKernelEx(&cfg, kda_pipelined_kernel<false, false>, pp, maps);
    trace_end(stream);
    if (e == cudaSuccess) {
      if (p.conv.state && launch_conv_prefill_state(p, stream) != 0) return -1;
      return cudaGetLastError() == cudaSuccess ? 0 : -1;
    }
    // not all CTAs could be resident at once (e.g. SMs held back): two launches
    if (e != cudaErrorCooperativeLaunchTooLarge || p.pipeline == 2) return -1;
    (void)cudaGetLastError();
    pp.walk_ctas = 0;
    pp.ready = nullptr;
    pp.item_counter = nullptr;
    pp.rec128 = walk128 ? 1 : 0;
  }
  trace_begin("kda_prologue", stream);
  const int grid = items < sms ? items : sms;
  if (pp.conv.state)  // bf16 activations only (checked by the API layer)
    kda_prologue_kernel<true, false><<<grid, PRO_THREADS, sizeof(ProSmem), stream>>>(pp, maps);
  else if (pp.in_fp16)
    kda_prologue_kernel<false, true><<<grid, PRO_THREADS, sizeof(ProSmem), stream>>>(pp, maps);
  else
    kda_prologue_kernel<false, false><<<grid, PRO_THREADS, sizeof(ProSmem), stream>>>(pp, maps);
  trace_end(stream);
  // the conv history of every sequence has been read: roll the conv state
  if (p.conv.state && launch_conv_prefill_state(p, stream) != 0) return -1;
  // the walks are launched programmatically: a walk CTA sets up (TMEM,
  // barriers, its initial state) while the kernel before it finishes, and
  // waits for that kernel before its first read of what it wrote
  auto launch_walk = [&](dim3 grid, int mode) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(WALK_THREADS);
    cfg.dynamicSmemBytes = sizeof(WalkSmem);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kda_walk_kernel, p, mode);
  };
  if (p.groups > 1) {
    trace_begin("kda_walk_pass1", stream);
    if (launch_walk(dim3(2 * D / NB, p.hv, p.n_seqs * p.groups), 1) != cudaSuccess) return -1;
    trace_end(stream);
    trace_begin("kda_group_compose", stream);
    kda_compose_kernel<<<dim3(D / NB, p.hv, p.n_seqs), COMPOSE_THREADS,
                         (NB * D + D * D) * sizeof(float), stream>>>(p);
    trace_end(stream);
  }
  if (pp.rec128) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(chains);
    cfg.blockDim = dim3(PRO_THREADS);
    cfg.dynamicSmemBytes = sizeof(Walk128Smem);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    trace_begin("kda_walk128", stream);
    if (cudaLaunchKernelEx(&cfg, kda_walk128_kernel, p) != cudaSuccess) return -1;
    trace_end(stream);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
  }
  trace_begin("kda_walk", stream);
  if (launch_walk(dim3(D / NB, p.hv, p.n_seqs * p.groups), 0) != cudaSuccess) return -1;
  trace_end(stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace kda

#ifdef KDA_PHASE_TIMING
// Measurement build only: copy the prologue's per-phase cycle sums (n of
// them, at most 12) and its item count to ``out[0..n]`` (out[n] = items),
// optionally clearing them.  Not part of the regular library's ABI.
// The pipelined kernel's per-CTA spans of its last launch: for CTA i,
// out[4 i .. 4 i + 3] = start ns, end ns, SM cycles, SM id (at most n CTAs).
extern "C" int kda_cta_spans(unsigned long long* out, int32_t n) {
  if (!out || n < 1 || n > kda::MAX_SPAN_CTAS) return KDA_ERR_INVALID_ARGUMENT;
  if (cudaDeviceSynchronize() != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(out, kda::g_cta_span, (size_t)n * 4 * sizeof(unsigned long long)) != cudaSuccess)
    return KDA_ERR_CUDA;
  return KDA_OK;
}

// The pipelined walk's counters (n of them, at most 6, then the chunk steps
// at out[n]), optionally clearing them.
extern "C" int kda_walk_cycles(unsigned long long* out, int32_t n, int32_t reset) {
  if (!out || n < 1 || n > kda::N_WALK_CTR) return KDA_ERR_INVALID_ARGUMENT;
  if (cudaDeviceSynchronize() != cudaSuccess) return KDA_ERR_CUDA;
  unsigned long long all[kda::N_WALK_CTR + 1];
  if (cudaMemcpyFromSymbol(all, kda::g_walk_cycles, sizeof(all)) != cudaSuccess) return KDA_ERR_CUDA;
  for (int i = 0; i < n; ++i) out[i] = all[i];
  out[n] = all[kda::N_WALK_CTR];
  if (reset) {
    const unsigned long long zero[kda::N_WALK_CTR + 1] = {};
    if (cudaMemcpyToSymbol(kda::g_walk_cycles, zero, sizeof(zero)) != cudaSuccess) return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

extern "C" int kda_phase_cycles(unsigned long long* out, int32_t n, int32_t reset) {
  if (!out || n < 1 || n > kda::N_PHASES) return KDA_ERR_INVALID_ARGUMENT;
  if (cudaDeviceSynchronize() != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(out, kda::g_phase_cycles, n * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMemcpyFromSymbol(out + n, kda::g_phase_items, sizeof(unsigned long long)) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (reset) {
    const unsigned long long zero[kda::N_PHASES + 1] = {};
    if (cudaMemcpyToSymbol(kda::g_phase_cycles, zero, kda::N_PHASES * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMemcpyToSymbol(kda::g_phase_items, zero, sizeof(unsigned long long)) != cudaSuccess)
      return KDA_ERR_CUDA;
  }
  return KDA_OK;
}
#endif
