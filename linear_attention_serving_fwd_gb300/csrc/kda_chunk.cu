// Chunked KDA prefill (chunk = 64), as the vLLM kimi_k3 AMD kda_chunk page
// splits it: a prologue that is parallel over chunks (gate, beta, L2 norms,
// gate cumsum, both intra-chunk passes, the WY/UT solve) and a walk that is
// serial over chunks per (sequence, head) and fused with the output, plus
// the chunk-group parallel scan of _chunk_groups for long chains.
//
// Per chunk of rows r = 0..63 (Lam = in-chunk cumsum of the gate):
//   A_kk[r,i] = beta_r sum_c k^_rc k^_ic e^{Lam_rc - Lam_ic}   (i < r)
//   A_qk[r,i] = sum_c q~_rc k^_ic e^{Lam_rc - Lam_ic}           (i <= r)
//   (I + A_kk) w = diag(beta) (e^{Lam} * k^),  (I + A_kk) u = diag(beta) v
//   qg = e^{Lam} * q~,  kg = e^{Lam_C - Lam} * k^,  d = e^{Lam_C}
// and the walk, with S the K x V state:
//   U = u - w S,  o = qg S + A_qk U,  S <- diag(d) S + kg^T U.
// The exponent differences are factored per 16-row sub-chunk I around
// ref_I = Lam at the middle row 16 I + 7 of I: below the block the row factor
// e^{Lam_r - ref_I} is <= 1 and the column factor e^{ref_I - Lam_i} is at most
// e^{8 |gate|max}; so factors stay inside fp32 (and bf16) range as long as
// any 8 consecutive gates sum to more than -88 (a lower_bound >= -11).
#include "kda_params.cuh"

namespace kda {

// Floats of per-(chunk, head) prologue output in the workspace.
constexpr int CH_W = 0;
constexpr int CH_U = CH_W + CHUNK * D;
constexpr int CH_QG = CH_U + CHUNK * D;
constexpr int CH_KG = CH_QG + CHUNK * D;
constexpr int CH_AQK = CH_KG + CHUNK * D;
constexpr int CH_D = CH_AQK + CHUNK * CHUNK;
constexpr int CH_FLOATS = CH_D + D;



__device__ __forceinline__ int seq_bos(const ChunkParams& p, int n) {
  return p.cu_seqlens ? p.cu_seqlens[n] : n * p.dense_len;
}
__device__ __forceinline__ int seq_eos(const ChunkParams& p, int n) {
  return p.cu_seqlens ? p.cu_seqlens[n + 1] : (n + 1) * p.dense_len;
}

// --------------------------------------------------------------------------
// Chunk index builder: chunk_off[n] = first global chunk of sequence n,
// chunk_seq/chunk_j name each chunk.  One block.
// --------------------------------------------------------------------------
__global__ void kda_chunk_index_kernel(ChunkParams p) {
  __shared__ int s_total;
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
    s_total = off;
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
// Prologue + intra-chunk solve, one CTA (256 threads) per (chunk, head).
// --------------------------------------------------------------------------
constexpr int PRO_THREADS = 256;
constexpr int LDA = D + 4;  // padded row stride (floats) for the [64][128] tiles

struct ProSmem {
  float kh[CHUNK][LDA];
  float qh[CHUNK][LDA];
  float lam[CHUNK][LDA];
  float Y[16][LDA];
  float Akk[CHUNK][CHUNK + 1];
  float Aqk[CHUNK][CHUNK + 1];
  float beta[CHUNK];
  float ref[D];
};

__global__ void __launch_bounds__(PRO_THREADS, 1) kda_prologue_kernel(ChunkParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ProSmem& s = *reinterpret_cast<ProSmem*>(smem_raw);
  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= *p.n_chunks) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = p.chunk_seq[c], j = p.chunk_j[c];
  const int bos = seq_bos(p, n) + j * CHUNK;
  const int len = min(CHUNK, seq_eos(p, n) - bos);
  const int hq = h / (p.hv / p.hqk);
  const float a = p.has_gate ? __expf(p.A_log[h]) : 0.f;

  // 1. loads and the gate
  for (int e = tid; e < CHUNK * D; e += PRO_THREADS) {
    const int r = e >> 7, ch = e & (D - 1);
    float qv = 0.f, kv = 0.f, gate = 0.f;
    if (r < len) {
      const int64_t tok = bos + r;
      qv = bf2f(p.q[tok * p.q_st + hq * p.q_sh + ch]);
      kv = bf2f(p.k[tok * p.k_st + hq * p.k_sh + ch]);
      const float gv = bf2f(p.g[tok * p.g_st + h * p.g_sh + ch]);
      gate = p.has_gate ? p.lower_bound * sigmoidf_(a * (gv + p.dt_bias[h * D + ch])) : gv;
    }
    s.qh[r][ch] = qv;
    s.kh[r][ch] = kv;
    s.lam[r][ch] = gate;
  }
  if (tid < CHUNK) {
    s.beta[tid] = tid < len ? sigmoidf_(bf2f(p.beta[(int64_t)(bos + tid) * p.b_st + h * p.b_sh])) : 0.f;
  }
  __syncthreads();
  // 2. L2 norms (warp per row) and 3. gate cumsum (thread per channel)
  for (int r = warp; r < CHUNK; r += PRO_THREADS / 32) {
    float sq = 0.f, sk = 0.f;
    for (int ch = lane; ch < D; ch += 32) {
      sq += s.qh[r][ch] * s.qh[r][ch];
      sk += s.kh[r][ch] * s.kh[r][ch];
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float rq = rsqrtf(sq + 1e-6f) * p.scale, rk = rsqrtf(sk + 1e-6f);
    for (int ch = lane; ch < D; ch += 32) {
      s.qh[r][ch] *= rq;
      s.kh[r][ch] *= rk;
    }
  }
  if (tid < D) {
    float acc = 0.f;
    for (int r = 0; r < CHUNK; ++r) {
      acc += s.lam[r][tid];
      s.lam[r][tid] = acc;
    }
  }
  __syncthreads();

  // 4. A_kk and A_qk, one 16-column block I at a time
  for (int I = 0; I < 4; ++I) {
    if (tid < D) s.ref[tid] = s.lam[16 * I + 7][tid];
    __syncthreads();
    for (int e = tid; e < 16 * D; e += PRO_THREADS) {
      const int i = e >> 7, ch = e & (D - 1);
      s.Y[i][ch] = s.kh[16 * I + i][ch] * __expf(s.ref[ch] - s.lam[16 * I + i][ch]);
    }
    __syncthreads();
    const int r = tid >> 2, part = tid & 3;
    float ak[16], aq[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ak[i] = aq[i] = 0.f;
    if (r >= 16 * I) {
      for (int cc = 0; cc < 32; ++cc) {
        const int ch = part + 4 * cc;
        const float f = __expf(s.lam[r][ch] - s.ref[ch]);
        const float xk = s.kh[r][ch] * f, xq = s.qh[r][ch] * f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          ak[i] = fmaf(xk, s.Y[i][ch], ak[i]);
          aq[i] = fmaf(xq, s.Y[i][ch], aq[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      ak[i] += __shfl_xor_sync(0xffffffffu, ak[i], 1);
      ak[i] += __shfl_xor_sync(0xffffffffu, ak[i], 2);
      aq[i] += __shfl_xor_sync(0xffffffffu, aq[i], 1);
      aq[i] += __shfl_xor_sync(0xffffffffu, aq[i], 2);
    }
    if (part == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int col = 16 * I + i;
        s.Akk[r][col] = (col < r) ? s.beta[r] * ak[i] : 0.f;
        s.Aqk[r][col] = (col <= r) ? aq[i] : 0.f;
      }
    }
    __syncthreads();
  }

  // 5. forward substitution: thread ch < 128 solves column ch of w, thread
  //    128 + ch column ch of u; rows depend only on earlier rows of the same
  //    column.
  float* ws = p.ch + ((int64_t)c * p.hv + h) * CH_FLOATS;
  {
    const int ch = tid & (D - 1);
    const bool is_u = tid >= D;
    float col[CHUNK];
#pragma unroll
    for (int r = 0; r < CHUNK; ++r) {
      float rhs;
      if (is_u) {
        rhs = r < len ? bf2f(p.v[(int64_t)(bos + r) * p.v_st + h * p.v_sh + ch]) : 0.f;
      } else {
        rhs = __expf(s.lam[r][ch]) * s.kh[r][ch];
      }
      float acc = s.beta[r] * rhs;
#pragma unroll
      for (int i = 0; i < r; ++i) acc = fmaf(-s.Akk[r][i], col[i], acc);
      col[r] = acc;
    }
    float* dst = ws + (is_u ? CH_U : CH_W);
#pragma unroll
    for (int r = 0; r < CHUNK; ++r) dst[r * D + ch] = col[r];
  }
  // 6. qg, kg, d, A_qk
  for (int e = tid; e < CHUNK * D; e += PRO_THREADS) {
    const int r = e >> 7, ch = e & (D - 1);
    const float lc = s.lam[CHUNK - 1][ch];
    ws[CH_QG + e] = __expf(s.lam[r][ch]) * s.qh[r][ch];
    ws[CH_KG + e] = __expf(lc - s.lam[r][ch]) * s.kh[r][ch];
  }
  for (int e = tid; e < CHUNK * CHUNK; e += PRO_THREADS) ws[CH_AQK + e] = s.Aqk[e >> 6][e & 63];
  if (tid < D) ws[CH_D + tid] = __expf(s.lam[CHUNK - 1][tid]);
}

// --------------------------------------------------------------------------
// Inter-chunk walk.  One CTA per (column block of 32, head, sequence x group).
// mode 0: outputs (+ final state when groups == 1), state from the initial
//         state (group 0) or the composed incoming state;
// mode 1: pass one of the group scan: zero start with u for the 4 value
//         blocks -> B_g, identity start with u = 0 for blocks 4..7 -> M_g.
// --------------------------------------------------------------------------
constexpr int WALK_THREADS = 256;
constexpr int NB = 32;  // state columns per CTA

struct WalkSmem {
  float w[CHUNK][D];
  float qg[CHUNK][D];
  float kg[CHUNK][D];
  float aqk[CHUNK][CHUNK];
  float u[CHUNK][NB];
  float U[CHUNK][NB];
  float S[D][NB];
  float d[D];
};

__device__ __forceinline__ const float* initial_state(const ChunkParams& p, int n, int h) {
  if (p.cache) {
    const int64_t slot = p.state_indices[n];
    if (slot < 0) return nullptr;
    if (slot >= p.n_slots) { set_error(p.err, ERR_INDEX); return nullptr; }
    if (p.has_init && !p.has_init[n]) return nullptr;
    return p.cache + slot * p.slot_stride + (int64_t)h * D * D;
  }
  return p.h0 ? p.h0 + ((int64_t)n * p.hv + h) * D * D : nullptr;
}

__device__ __forceinline__ float* final_state(const ChunkParams& p, int n, int h) {
  if (p.cache) {
    const int64_t slot = p.state_indices[n];
    if (slot < 0 || slot >= p.n_slots) return nullptr;
    return p.cache + slot * p.slot_stride + (int64_t)h * D * D;
  }
  return p.hT ? p.hT + ((int64_t)n * p.hv + h) * D * D : nullptr;
}

__device__ __forceinline__ void group_range(const ChunkParams& p, int n, int gidx, int& c0, int& c1) {
  const int base = p.chunk_off[n], nc = p.chunk_off[n + 1] - base;
  const int per = (nc + p.groups - 1) / p.groups;
  c0 = base + min(nc, gidx * per);
  c1 = base + min(nc, (gidx + 1) * per);
}

__global__ void __launch_bounds__(WALK_THREADS, 1) kda_walk_kernel(ChunkParams p, int mode) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  WalkSmem& s = *reinterpret_cast<WalkSmem*>(smem_raw);
  const int cb = blockIdx.x, h = blockIdx.y;
  const int n = blockIdx.z / p.groups, gidx = blockIdx.z % p.groups;
  const int tid = threadIdx.x;
  const bool ident = mode == 1 && cb >= D / NB;   // M_g columns
  const int col0 = (cb % (D / NB)) * NB;          // first value (or identity) column
  int c0, c1;
  group_range(p, n, gidx, c0, c1);
  const int64_t plane = (((int64_t)n * p.hv + h) * p.groups + gidx) * D * D;

  // incoming state columns col0..col0+31, stored S[k][v]
  {
    const float* src = nullptr;
    if (mode == 0) src = (p.groups > 1) ? p.gS + plane : initial_state(p, n, h);
    for (int e = tid; e < D * NB; e += WALK_THREADS) {
      const int v = e >> 7, k = e & (D - 1);
      float x = 0.f;
      if (mode == 1) x = (ident && k == col0 + v) ? 1.f : 0.f;
      else if (src) x = src[(int64_t)(col0 + v) * D + k];
      s.S[k][v] = x;
    }
  }
  __syncthreads();
  const int lv = tid & 31;        // state column within the block
  const int rg = tid >> 5;        // row group (8 warps)
  for (int c = c0; c < c1; ++c) {
    const float* ws = p.ch + ((int64_t)c * p.hv + h) * CH_FLOATS;
    const int n_ = p.chunk_seq[c];
    const int bos = seq_bos(p, n_) + p.chunk_j[c] * CHUNK;
    const int len = min(CHUNK, seq_eos(p, n_) - bos);
    for (int e = tid; e < CHUNK * D / 4; e += WALK_THREADS) {
      reinterpret_cast<float4*>(&s.w[0][0])[e] = reinterpret_cast<const float4*>(ws + CH_W)[e];
      reinterpret_cast<float4*>(&s.kg[0][0])[e] = reinterpret_cast<const float4*>(ws + CH_KG)[e];
      if (mode == 0)
        reinterpret_cast<float4*>(&s.qg[0][0])[e] = reinterpret_cast<const float4*>(ws + CH_QG)[e];
    }
    if (mode == 0)
      for (int e = tid; e < CHUNK * CHUNK / 4; e += WALK_THREADS)
        reinterpret_cast<float4*>(&s.aqk[0][0])[e] = reinterpret_cast<const float4*>(ws + CH_AQK)[e];
    for (int e = tid; e < CHUNK * NB; e += WALK_THREADS) {
      const int r = e >> 5, v = e & 31;
      s.u[r][v] = ident ? 0.f : ws[CH_U + r * D + col0 + v];
    }
    if (tid < D) s.d[tid] = ws[CH_D + tid];
    __syncthreads();
    // U = u - w S and the inter-chunk part of o (8 rows per thread)
    float accU[8], accO[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) accU[i] = accO[i] = 0.f;
    for (int k = 0; k < D; k += 4) {
      const float s0 = s.S[k][lv], s1 = s.S[k + 1][lv], s2 = s.S[k + 2][lv], s3 = s.S[k + 3][lv];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        const float4 w4 = *reinterpret_cast<const float4*>(&s.w[r][k]);
        accU[i] += w4.x * s0 + w4.y * s1 + w4.z * s2 + w4.w * s3;
        if (mode == 0) {
          const float4 q4 = *reinterpret_cast<const float4*>(&s.qg[r][k]);
          accO[i] += q4.x * s0 + q4.y * s1 + q4.z * s2 + q4.w * s3;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) s.U[rg * 8 + i][lv] = s.u[rg * 8 + i][lv] - accU[i];
    __syncthreads();
    if (mode == 0) {
      for (int i2 = 0; i2 < CHUNK; ++i2) {
        const float ui = s.U[i2][lv];
#pragma unroll
        for (int i = 0; i < 8; ++i) accO[i] = fmaf(s.aqk[rg * 8 + i][i2], ui, accO[i]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        if (r < len)
          p.out[((int64_t)(bos + r) * p.hv + h) * D + col0 + lv] = __float2bfloat16_rn(accO[i]);
      }
    }
    // S <- diag(d) S + kg^T U (16 state rows per thread)
    float accS[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) accS[i] = s.d[rg * 16 + i] * s.S[rg * 16 + i][lv];
    for (int r = 0; r < CHUNK; ++r) {
      const float ur = s.U[r][lv];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(&s.kg[r][rg * 16 + i]);
        accS[i] = fmaf(k4.x, ur, accS[i]);
        accS[i + 1] = fmaf(k4.y, ur, accS[i + 1]);
        accS[i + 2] = fmaf(k4.z, ur, accS[i + 2]);
        accS[i + 3] = fmaf(k4.w, ur, accS[i + 3]);
      }
    }
    __syncthreads();  // everyone done reading S, U, chunk tiles
#pragma unroll
    for (int i = 0; i < 16; ++i) s.S[rg * 16 + i][lv] = accS[i];
    __syncthreads();
  }
  // end state of this column block, V-first rows col0..col0+31
  float* dst = nullptr;
  if (mode == 1) dst = (ident ? p.gM : p.gB) + plane;
  else if (p.groups == 1) dst = final_state(p, n, h);
  if (dst)
    for (int e = tid; e < D * NB; e += WALK_THREADS) {
      const int v = e >> 7, k = e & (D - 1);
      dst[(int64_t)(col0 + v) * D + k] = s.S[k][v];
    }
}

// --------------------------------------------------------------------------
// Group composition: S_{g+1}^T = S_g^T M_g^T + B_g^T serially over groups,
// recording each group's incoming state; the last one is the final state.
// One CTA (256 threads) per (value block of 32 rows, head, sequence).
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(WALK_THREADS, 1) kda_compose_kernel(ChunkParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* St = reinterpret_cast<float*>(smem_raw);  // [32][128] rows v0..v0+31 of S^T
  float* Mt = St + NB * D;                         // [128][128]
  const int vb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x;
  const int v0 = vb * NB;
  const float* src = initial_state(p, n, h);
  for (int e = tid; e < NB * D; e += WALK_THREADS)
    St[e] = src ? src[(int64_t)v0 * D + e] : 0.f;
  __syncthreads();
  for (int gi = 0; gi < p.groups; ++gi) {
    const int64_t plane = (((int64_t)n * p.hv + h) * p.groups + gi) * D * D;
    for (int e = tid; e < NB * D; e += WALK_THREADS) p.gS[plane + (int64_t)v0 * D + e] = St[e];
    for (int e = tid; e < D * D; e += WALK_THREADS) Mt[e] = p.gM[plane + e];
    __syncthreads();
    // thread: row v = tid >> 3, 16 columns k = (tid & 7) + 8 j
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
  float* dst = final_state(p, n, h);
  if (dst)
    for (int e = tid; e < NB * D; e += WALK_THREADS) dst[(int64_t)v0 * D + e] = St[e];
}

// --------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------
size_t chunk_workspace_floats(int n_seqs, int t_total, int hv, int groups, int* max_chunks_out) {
  const int max_chunks = t_total / CHUNK + n_seqs;
  if (max_chunks_out) *max_chunks_out = max_chunks;
  size_t ints = 4 + (size_t)(n_seqs + 1) + 2 * (size_t)max_chunks;
  ints = (ints + 3) & ~(size_t)3;  // keep the float area 16-byte aligned
  size_t floats = (size_t)max_chunks * hv * CH_FLOATS;
  if (groups > 1) floats += 3 * (size_t)n_seqs * hv * groups * D * D;
  return ints + floats;  // in 4-byte words
}

int launch_chunk(ChunkParams p, void* workspace, cudaStream_t stream) {
  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(kda_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(ProSmem));
    cudaFuncSetAttribute(kda_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(WalkSmem));
    cudaFuncSetAttribute(kda_compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)((NB * D + D * D) * sizeof(float)));
    attrs = true;
  }
  int max_chunks = 0;
  chunk_workspace_floats(p.n_seqs, p.t_total, p.hv, p.groups, &max_chunks);
  int32_t* iw = reinterpret_cast<int32_t*>(workspace);
  p.max_chunks = max_chunks;
  p.n_chunks = iw;
  p.chunk_off = iw + 4;
  p.chunk_seq = p.chunk_off + (p.n_seqs + 1);
  p.chunk_j = p.chunk_seq + max_chunks;
  size_t ints = 4 + (size_t)(p.n_seqs + 1) + 2 * (size_t)max_chunks;
  ints = (ints + 3) & ~(size_t)3;
  float* fw = reinterpret_cast<float*>(iw + ints);
  p.ch = fw;
  fw += (size_t)max_chunks * p.hv * CH_FLOATS;
  if (p.groups > 1) {
    const size_t plane = (size_t)p.n_seqs * p.hv * p.groups * D * D;
    p.gM = fw;
    p.gB = fw + plane;
    p.gS = fw + 2 * plane;
  }
  trace_begin("kda_chunk_index", stream);
  kda_chunk_index_kernel<<<1, 256, 0, stream>>>(p);
  trace_end(stream);
  trace_begin("kda_prologue", stream);
  kda_prologue_kernel<<<dim3(max_chunks, p.hv), PRO_THREADS, sizeof(ProSmem), stream>>>(p);
  trace_end(stream);
  if (p.groups > 1) {
    trace_begin("kda_walk_pass1", stream);
    kda_walk_kernel<<<dim3(2 * D / NB, p.hv, p.n_seqs * p.groups), WALK_THREADS,
                      sizeof(WalkSmem), stream>>>(p, 1);
    trace_end(stream);
    trace_begin("kda_group_compose", stream);
    kda_compose_kernel<<<dim3(D / NB, p.hv, p.n_seqs), WALK_THREADS,
                         (NB * D + D * D) * sizeof(float), stream>>>(p);
    trace_end(stream);
  }
  trace_begin("kda_walk", stream);
  kda_walk_kernel<<<dim3(D / NB, p.hv, p.n_seqs * p.groups), WALK_THREADS, sizeof(WalkSmem),
                    stream>>>(p, 0);
  trace_end(stream);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace kda
