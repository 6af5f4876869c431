// Kernel parameter blocks shared by the API layer and the kernels.
#pragma once

#include <mutex>

#include "kda_common.cuh"

namespace kda {

// Width-4 depthwise conv + SiLU over the raw q/k/v projection bands
// (state == nullptr: off).  Channel ch of C = (2 Hqk + Hv) * 128 numbers the
// q band, then k, then v (band offset + head * 128 + c).
struct ConvParams {
  const void* w;               // [C, 4] taps, bf16 or fp32 (w_f32)
  int w_f32;
  __nv_bfloat16* state;        // element (row, pos, ch) at row*row_st + pos*pos_st + ch*ch_st
  int64_t row_st, pos_st, ch_st, rows;
  int positions;
  const int32_t* idx;          // prefill: [N] state row per sequence (< 0: zero history, no update)
  const uint8_t* has_init;     // prefill: [N] or null (all rows hold a history)
  const int32_t* accepted;     // verify: [n_req]; history at positions accepted-1 .. accepted+1
  int bulk;                    // verify: token-major state and 16-byte rows: taps and history
                               // are staged into shared memory by bulk copies with the inputs
};

struct WindowParams {
  const __nv_bfloat16 *q, *k, *v, *g, *beta;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh, g_st, g_sh, b_st, b_sh;
  const float* A_log;
  const float* dt_bias;
  float scale, lower_bound;
  int has_gate;
  __nv_bfloat16* out;  // [T, Hv, 128], activation dtype
  void* pool;          // [n_slots, Hv, 128, 128] fp32 or bf16 (read only for verify)
  int64_t slot_stride;
  int64_t n_slots;
  const int32_t* query_start;
  const int32_t* slots;
  // decode with a [n_req, step_stride] slot table (slots unused): the state
  // is read from row step_slots[b][n_accepted[b] - 1] (column 0 without
  // n_accepted) and the state after token t goes to row step_slots[b][t]
  const int32_t* step_slots;
  int64_t step_stride;
  const int32_t* n_accepted;
  int n_req, window, hqk, hv;
  ConvParams conv;       // verify only
  int in_fp16, state_bf16;  // activation / state dtypes
  float* corr;          // verify: [n_req, Hv, window, 128]
  __nv_bfloat16* kg;    // verify: [n_req, Hv, window, 256]
  int32_t* counter;     // verify: ticket counter
  unsigned* err;        // device error word
};

struct CommitParams {
  void* pool;                  // [n_slots, Hv, 128, 128] fp32 or bf16, rewritten in place
  int64_t slot_stride, n_slots;
  const int32_t* slots;        // [n_req]
  const int32_t* accepted;     // [n_req] accepted prefix length a
  const float* corr;           // [n_req, Hv, window, 128] U_t from kda_verify
  const __nv_bfloat16* kg;     // [n_req, Hv, window, 256] raw k_t, raw g_t from kda_verify
  int state_bf16, kg_fp16;
  const float* A_log;
  const float* dt_bias;
  float lower_bound;
  int has_gate;
  int n_req, hv, window;
  unsigned* err;
};

struct ChunkParams {
  const __nv_bfloat16 *q, *k, *v, *g, *beta;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh, g_st, g_sh, b_st, b_sh;
  const float* A_log;
  const float* dt_bias;
  float scale, lower_bound;
  int has_gate;
  int t_total, hqk, hv, n_seqs;
  int dense_len;               // > 0: dense sequences of this length (no cu_seqlens)
  const int32_t* cu_seqlens;   // [N+1] or null
  __nv_bfloat16* out;          // activation dtype
  int in_fp16, state_bf16;     // activation / state dtypes
  const void* h0;              // [N, Hv, 128, 128] state dtype, or null
  void* hT;                    // [N, Hv, 128, 128] or null
  void* cache;                 // paged cache or null
  int64_t slot_stride, n_slots;
  const int32_t* state_indices;
  const uint8_t* has_init;
  int max_chunks;
  int groups;
  int sm_count;         // SMs of the device: the persistent prologue's grid
  // pipelined launch: CTAs 0 .. walk_ctas - 1 walk one chain each (all 128
  // value columns) while the others run the prologue in level-major order;
  // ready[c * Hv + h] is raised once record (c, h) has landed.  0 / null in
  // the two-launch path.
  int walk_ctas;
  unsigned* ready;
  unsigned* item_counter;  // pipelined launch: prologue CTAs take their next item from it (zeroed)
  int pipeline;         // host: 0 two launches, 1 the library chooses, 2 pipelined (groups = -1)
  int rec128;           // records for the 128-column walk: -qg' and -A_qk T in place of qg' and o_intra
  // workspace carve
  int32_t* chunk_off;   // [N+1]
  int32_t* chunk_seq;   // [max_chunks]
  int32_t* chunk_j;     // [max_chunks]
  int32_t* n_chunks;    // [1]
  float* ch;            // per-(chunk, head) records, CH_BYTES each
  float* gM;            // [N, Hv, G, 128, 128]  M_g^T
  float* gB;            // [N, Hv, G, 128, 128]  B_g^T
  float* gS;            // [N, Hv, G, 128, 128]  incoming state of each group (V-first)
  // mid-prefill snapshots: the state after ckpt_off[n] tokens of sequence n
  // (a positive multiple of CHUNK, at most its length) goes to row
  // ckpt_idx[n] (or n) of ckpt; others are skipped
  void* ckpt;                   // state dtype
  int64_t ckpt_stride, ckpt_rows;
  const int32_t* ckpt_off;
  const int32_t* ckpt_idx;
  ConvParams conv;
  __nv_bfloat16* conv_out;     // prefill with a conv: the convolved q, k, v bands ([T, Hqk, 128]
                               // twice, then [T, Hv, 128]), or null (each prologue item
                               // convolves its own tiles)
  unsigned* err;        // device error word
};

// Kernel tracing (kda_trace_* in the API layer): when enabled, CUDA events
// are recorded on the launching stream around each kernel; off by default,
// then these are one predictable branch each.
void trace_begin(const char* name, cudaStream_t stream);
void trace_end(cudaStream_t stream);

// Set the thread-local text that kda_last_error() returns.
void set_last_error(int code, const char* msg);

// Host: per-device set-up (kernel attributes, SM counts, symbol addresses)
// runs once per device under one library-wide lock, so that threads making
// their first calls at the same time do not race.  ``done`` has one bit per
// device (devices 0..63).  Returns false without running ``fn`` when no
// device is current.
std::mutex& host_mutex();
template <class F>
inline bool once_per_device(uint64_t& done, F&& fn) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(host_mutex());
  if (!(done & (1ull << dev))) {
    fn(dev);
    done |= 1ull << dev;
  }
  return true;
}

// Launchers (kernels' translation units); return 0 or -1 (see cudaGetLastError).
int launch_window(const WindowParams& p, bool verify, cudaStream_t stream);
int launch_commit(const CommitParams& p, cudaStream_t stream);
int launch_conv_prefill_state(const ChunkParams& p, cudaStream_t stream);
int launch_conv_prefill(const ChunkParams& p, cudaStream_t stream);
int launch_conv_roll(const WindowParams& p, cudaStream_t stream);
size_t chunk_workspace_floats(int n_seqs, int t_total, int hv, int groups, int* max_chunks_out);
int launch_chunk(ChunkParams p, void* workspace, cudaStream_t stream);
int launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t stream);

}  // namespace kda
