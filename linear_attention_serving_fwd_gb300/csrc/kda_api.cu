// Host side of the C ABI declared in include/kda.h: argument validation
// (the shape, dtype and pairing rules of the MATE chunk_kda /
// gated_delta_rule_decode validation and of the vLLM fused_kda_chunk cache
// rules), the per-device error word, and the kernel launches.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kda_params.cuh"

namespace {

thread_local std::string g_last_error;

// One error word per device that loads the library.  Host code passes its
// device address (cudaGetSymbolAddress) to every kernel.
__device__ unsigned int g_error_word = 0u;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return KDA_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The error word's device address, resolved once per device (under the
// library lock).  The address stays valid for the life of the device's
// primary context: a cudaDeviceReset inside the process after the first
// call is not supported.
unsigned* error_word_ptr() {
  static unsigned* ptrs[64] = {nullptr};
  static uint64_t done = 0;
  int dev = -1;
  const bool have = kda::once_per_device(done, [&](int d) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) ptrs[d] = static_cast<unsigned*>(p);
    else cudaGetLastError();
  });
  if (!have || cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(kda::host_mutex());
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rules shared by all entry points.
int check_activations(const kda_activations* x, bool need_rows_aligned) {
  if (!x) return fail(KDA_ERR_INVALID_ARGUMENT, "activations must not be NULL.");
  if (x->dtype != KDA_DTYPE_BF16 && x->dtype != KDA_DTYPE_FP16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "q/k/v/g/beta dtype must be bfloat16 or float16 (got %d).",
                x->dtype);
  if (x->state_bf16 != 0 && x->state_bf16 != 1)
    return fail(KDA_ERR_INVALID_ARGUMENT, "state_bf16 must be 0 (fp32 states) or 1 (bf16 states).");
  if (x->hqk <= 0 || x->hv <= 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "head counts must be positive (hqk=%d, hv=%d).", x->hqk, x->hv);
  if (x->hv % x->hqk != 0)
    return fail(KDA_ERR_INVALID_ARGUMENT,
                "GVA requires v/g heads to be divisible by q/k heads (hv=%d, hqk=%d).", x->hv, x->hqk);
  if (x->t_total < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "t_total must be >= 0.");
  if ((x->A_log == nullptr) != (x->dt_bias == nullptr))
    return fail(KDA_ERR_INVALID_ARGUMENT, "A_log and dt_bias must be provided together.");
  if (x->use_qk_l2norm != 1)
    return fail(KDA_ERR_INVALID_ARGUMENT,
                "use_qk_l2norm must be 1: only the in-kernel q/k L2 norm is built.");
  if (x->A_log && !(x->lower_bound <= 0.f && x->lower_bound >= -10.5f))
    return fail(KDA_ERR_INVALID_ARGUMENT,
                "lower_bound must lie in [-10.5, 0] (got %g).", (double)x->lower_bound);
  if (x->t_total > 0) {
    if (!x->q || !x->k || !x->v || !x->g || !x->beta)
      return fail(KDA_ERR_INVALID_ARGUMENT, "q, k, v, g and beta must not be NULL.");
    const void* rows[4] = {x->q, x->k, x->v, x->g};
    const int64_t st[8] = {x->q_stride_tok, x->q_stride_head, x->k_stride_tok, x->k_stride_head,
                           x->v_stride_tok, x->v_stride_head, x->g_stride_tok, x->g_stride_head};
    for (int i = 0; i < 8; ++i)
      if (st[i] < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "strides must be non-negative.");
    if (x->beta_stride_tok < 0 || x->beta_stride_head < 0)
      return fail(KDA_ERR_INVALID_ARGUMENT, "strides must be non-negative.");
    if (need_rows_aligned) {
      for (int i = 0; i < 4; ++i)
        if (!aligned16(rows[i]))
          return fail(KDA_ERR_INVALID_ARGUMENT, "q, k, v and g must be 16-byte aligned.");
      for (int i = 0; i < 8; ++i)
        if (st[i] % 8 != 0)
          return fail(KDA_ERR_INVALID_ARGUMENT,
                      "q/k/v/g token and head strides must be multiples of 8 elements.");
    }
    if (x->A_log && !aligned16(x->dt_bias))
      return fail(KDA_ERR_INVALID_ARGUMENT, "dt_bias must be 16-byte aligned.");
  }
  return KDA_OK;
}

void fill_common(const kda_activations* x, const __nv_bfloat16*& q, const __nv_bfloat16*& k,
                 const __nv_bfloat16*& v, const __nv_bfloat16*& g, const __nv_bfloat16*& b) {
  q = static_cast<const __nv_bfloat16*>(x->q);
  k = static_cast<const __nv_bfloat16*>(x->k);
  v = static_cast<const __nv_bfloat16*>(x->v);
  g = static_cast<const __nv_bfloat16*>(x->g);
  b = static_cast<const __nv_bfloat16*>(x->beta);
}

// Rows of states (fp32, or bf16 with ``bf16``): the stride counts elements
// and keeps rows 16-byte aligned for the bulk copies.
int check_pool(const void* pool, int64_t slot_stride, int64_t n_slots, int hv, bool bf16, const char* name,
               const char* stride_name = "slot_stride") {
  if (!pool) return fail(KDA_ERR_INVALID_ARGUMENT, "%s must not be NULL.", name);
  if (!aligned16(pool)) return fail(KDA_ERR_INVALID_ARGUMENT, "%s must be 16-byte aligned.", name);
  if (n_slots <= 0) return fail(KDA_ERR_INVALID_ARGUMENT, "%s must contain at least one slot.", name);
  const int64_t unit = bf16 ? 8 : 4;
  if (slot_stride % unit != 0 || slot_stride < (int64_t)hv * kda::D * kda::D)
    return fail(KDA_ERR_INVALID_ARGUMENT,
                "%s must be a multiple of %lld elements and >= Hv*128*128 (got %lld).", stride_name,
                (long long)unit, (long long)slot_stride);
  return KDA_OK;
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();  // no device here: size for a full GB300
    return 152;
  }
  return sms;
}

// Chunk groups per sequence for the parallel scan (the vLLM kda_chunk page's
// _chunk_groups rule, fitted to this walk): the walk runs one CTA per SM and
// is latency bound, so splitting a chain only pays while pass one's grid
// (8 column blocks per sequence, head and group) still fits on the SMs, and
// while groups stay at least 8 chunks long.  G = 2 is depth-neutral, so the
// split starts at G = 4.
int choose_groups(int32_t n_seqs, int32_t t_total, int32_t hv, int32_t requested) {
  if (requested > 0) return requested < 64 ? requested : 64;
  if (requested == -1) return 1;  // the pipelined launch walks each chain serially
  const int sms = device_sm_count();
  const long pass1 = 8L * n_seqs * hv;
  const long chunks = ((long)t_total + kda::CHUNK - 1) / kda::CHUNK;
  const long avg = chunks / (n_seqs > 0 ? n_seqs : 1);
  int g = 1;
  while (g < 64 && pass1 * 2 * g <= sms && avg / (2 * g) >= 8) g *= 2;
  return g >= 4 ? g : 1;
}

// --- kernel tracing --------------------------------------------------------
struct TraceRec {
  std::string name;
  cudaEvent_t start, stop;
};
struct TraceTotal {
  std::string name;
  double ms;
  int launches;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace_pending;
std::vector<TraceTotal> g_trace_totals;
std::vector<cudaEvent_t> g_trace_free;

cudaEvent_t trace_event() {
  if (!g_trace_free.empty()) {
    cudaEvent_t e = g_trace_free.back();
    g_trace_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void trace_drain() {  // caller holds the lock
  for (auto& r : g_trace_pending) {
    float ms = 0.f;
    cudaEventSynchronize(r.stop);
    cudaEventElapsedTime(&ms, r.start, r.stop);
    bool found = false;
    for (auto& t : g_trace_totals)
      if (t.name == r.name) { t.ms += ms; t.launches += 1; found = true; break; }
    if (!found) g_trace_totals.push_back({r.name, (double)ms, 1});
    g_trace_free.push_back(r.start);
    g_trace_free.push_back(r.stop);
  }
  g_trace_pending.clear();
}

}  // namespace

namespace kda {
std::mutex& host_mutex() {
  static std::mutex m;
  return m;
}

void set_last_error(int code, const char* msg) {
  (void)code;
  g_last_error = msg;
}

void trace_begin(const char* name, cudaStream_t stream) {
  if (!g_trace_on) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  TraceRec r{name, trace_event(), trace_event()};
  cudaEventRecord(r.start, stream);
  g_trace_pending.push_back(r);
}
void trace_end(cudaStream_t stream) {
  if (!g_trace_on) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_pending.empty()) cudaEventRecord(g_trace_pending.back().stop, stream);
}
}  // namespace kda

extern "C" {

int kda_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  trace_drain();
  g_trace_totals.clear();
  g_trace_on = on != 0;
  return KDA_OK;
}

int kda_trace_read(int32_t index, char* name, int32_t name_cap, double* total_ms,
                   int32_t* launches) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  trace_drain();
  const int n = (int)g_trace_totals.size();
  if (index >= 0 && index < n) {
    const TraceTotal& t = g_trace_totals[index];
    if (name && name_cap > 0) {
      strncpy(name, t.name.c_str(), (size_t)name_cap - 1);
      name[name_cap - 1] = 0;
    }
    if (total_ms) *total_ms = t.ms;
    if (launches) *launches = t.launches;
  }
  return n;
}

const char* kda_version(void) { return "kda-gb300 0.1 sm_103a"; }

const char* kda_last_error(void) { return g_last_error.c_str(); }
const char* kda_last_error_message(void) { return g_last_error.c_str(); }

size_t kda_conv_scratch_bytes(int32_t t_total, int32_t hqk, int32_t hv) {
  if (t_total < 0 || hqk <= 0 || hv <= 0) return 0;
  return (size_t)t_total * (2 * (size_t)hqk + hv) * kda::D * 2;
}

size_t kda_chunk_workspace_bytes(int32_t n_seqs, int32_t t_total, int32_t hv, int32_t groups) {
  if (n_seqs <= 0 || t_total < 0 || hv <= 0) return 0;
  const int G = choose_groups(n_seqs, t_total, hv, groups);
  return 4 * kda::chunk_workspace_floats(n_seqs, t_total, hv, G, nullptr);
}

// Host rules of a kda_conv; fills cp (state == nullptr when conv is NULL).
static int check_conv(const kda_conv* conv, const kda_activations* x, bool verify, int32_t window,
                      int64_t n_slots, kda::ConvParams& cp) {
  memset(&cp, 0, sizeof(cp));
  if (!conv) return KDA_OK;
  if (x->dtype != KDA_DTYPE_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "the conv path takes bfloat16 activations (the conv state is bf16).");
  if (!conv->weight || !conv->state)
    return fail(KDA_ERR_INVALID_ARGUMENT, "conv weight and state must not be NULL.");
  if (!aligned16(conv->weight)) return fail(KDA_ERR_INVALID_ARGUMENT, "conv weight must be 16-byte aligned.");
  if (conv->weight_f32 != 0 && conv->weight_f32 != 1)
    return fail(KDA_ERR_INVALID_ARGUMENT, "conv weight_f32 must be 0 (bf16 taps) or 1 (fp32 taps).");
  if (conv->rows <= 0 || conv->row_stride <= 0 || conv->pos_stride <= 0 || conv->chan_stride <= 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "conv state rows and strides must be positive.");
  const int need = verify ? window + 2 : 3;
  if (conv->positions < need)
    return fail(KDA_ERR_INVALID_ARGUMENT, "conv state needs at least %d positions (got %d).", need,
                conv->positions);
  if (verify) {
    if (!conv->num_accepted) return fail(KDA_ERR_INVALID_ARGUMENT, "verify with a conv needs num_accepted.");
    if (conv->rows < n_slots)
      return fail(KDA_ERR_INVALID_ARGUMENT, "conv state needs a row per state slot (%lld < %lld).",
                  (long long)conv->rows, (long long)n_slots);
    if (conv->scratch) return fail(KDA_ERR_INVALID_ARGUMENT, "verify takes no conv scratch.");
  } else if (!conv->state_indices) {
    return fail(KDA_ERR_INVALID_ARGUMENT, "prefill with a conv needs conv state_indices.");
  } else if (conv->scratch) {
    const size_t need_s = kda_conv_scratch_bytes(x->t_total, x->hqk, x->hv);
    if (conv->scratch_bytes < need_s)
      return fail(KDA_ERR_INVALID_ARGUMENT, "conv scratch needs %zu bytes (got %zu).", need_s,
                  conv->scratch_bytes);
    if (!aligned16(conv->scratch)) return fail(KDA_ERR_INVALID_ARGUMENT, "conv scratch must be 16-byte aligned.");
  }
  cp.w = conv->weight;
  cp.w_f32 = conv->weight_f32;
  cp.state = static_cast<__nv_bfloat16*>(conv->state);
  cp.row_st = conv->row_stride;
  cp.pos_st = conv->pos_stride;
  cp.ch_st = conv->chan_stride;
  cp.rows = conv->rows;
  cp.positions = conv->positions;
  cp.idx = conv->state_indices;
  cp.has_init = conv->has_initial_state;
  cp.accepted = conv->num_accepted;
  // staged by bulk copies (verify): bf16 taps and a token-major state with
  // 16-byte aligned rows and positions
  cp.bulk = verify && !conv->weight_f32 && aligned16(conv->weight) && conv->chan_stride == 1 &&
            conv->pos_stride % 8 == 0 && conv->row_stride % 8 == 0 && aligned16(conv->state);
  return KDA_OK;
}

static int chunk_common(const kda_activations* x, void* out, const int32_t* cu_seqlens, int32_t n_seqs,
                        const void* initial_state, void* final_state, void* state_cache,
                        int64_t slot_stride, int64_t n_slots, const int32_t* state_indices,
                        const uint8_t* has_initial_state, void* checkpoint_state,
                        int64_t checkpoint_row_stride, int64_t checkpoint_rows,
                        const int32_t* checkpoint_offsets, const int32_t* checkpoint_state_indices,
                        const kda_conv* conv, int32_t groups, void* workspace, size_t workspace_bytes,
                        void* stream) {
  int rc = check_activations(x, true);
  if (rc) return rc;
  kda::ConvParams cp;
  rc = check_conv(conv, x, false, 0, 0, cp);
  if (rc) return rc;
  if (n_seqs <= 0) return fail(KDA_ERR_INVALID_ARGUMENT, "n_seqs must be >= 1.");
  if (!cu_seqlens && x->t_total % n_seqs != 0)
    return fail(KDA_ERR_INVALID_ARGUMENT,
                "dense mode (no cu_seqlens) needs t_total divisible by n_seqs.");
  if (x->t_total > 0 && !out) return fail(KDA_ERR_INVALID_ARGUMENT, "out must not be NULL.");
  if (state_cache) {
    if (initial_state || final_state)
      return fail(KDA_ERR_INVALID_ARGUMENT, "state_cache replaces initial_state/final_state.");
    if (!state_indices) return fail(KDA_ERR_INVALID_ARGUMENT, "state_cache needs state_indices.");
    rc = check_pool(state_cache, slot_stride, n_slots, x->hv, x->state_bf16, "state_cache");
    if (rc) return rc;
  }
  if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
    return fail(KDA_ERR_INVALID_ARGUMENT, "states must be 16-byte aligned.");
  if (checkpoint_state) {
    if (!checkpoint_offsets)
      return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoint_state needs checkpoint_offsets.");
    rc = check_pool(checkpoint_state, checkpoint_row_stride, checkpoint_rows, x->hv, x->state_bf16,
                    "checkpoint_state",
                    "checkpoint_row_stride");
    if (rc) return rc;
    if (!checkpoint_state_indices && checkpoint_rows < n_seqs)
      return fail(KDA_ERR_INVALID_ARGUMENT,
                  "checkpoint_state without checkpoint_state_indices needs a row per sequence "
                  "(%lld < %d).", (long long)checkpoint_rows, n_seqs);
  } else if (checkpoint_offsets || checkpoint_state_indices) {
    return fail(KDA_ERR_INVALID_ARGUMENT, "checkpoint offsets or indices given without checkpoint_state.");
  }
  const int G = choose_groups(n_seqs, x->t_total, x->hv, groups);
  const size_t need = 4 * kda::chunk_workspace_floats(n_seqs, x->t_total, x->hv, G, nullptr);
  if (!workspace || workspace_bytes < need)
    return fail(KDA_ERR_INVALID_ARGUMENT, "workspace needs %zu bytes (got %zu).", need,
                workspace ? workspace_bytes : (size_t)0);
  if (!aligned16(workspace)) return fail(KDA_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned.");
  unsigned* err = error_word_ptr();
  if (!err) return fail(KDA_ERR_CUDA, "cannot resolve the device error word.");

  kda::ChunkParams p;
  memset(&p, 0, sizeof(p));
  fill_common(x, p.q, p.k, p.v, p.g, p.beta);
  p.q_st = x->q_stride_tok; p.q_sh = x->q_stride_head;
  p.k_st = x->k_stride_tok; p.k_sh = x->k_stride_head;
  p.v_st = x->v_stride_tok; p.v_sh = x->v_stride_head;
  p.g_st = x->g_stride_tok; p.g_sh = x->g_stride_head;
  p.b_st = x->beta_stride_tok; p.b_sh = x->beta_stride_head;
  p.A_log = x->A_log; p.dt_bias = x->dt_bias; p.has_gate = x->A_log != nullptr;
  p.scale = x->scale; p.lower_bound = x->lower_bound;
  p.t_total = x->t_total; p.hqk = x->hqk; p.hv = x->hv; p.n_seqs = n_seqs;
  p.dense_len = cu_seqlens ? 0 : x->t_total / n_seqs;
  p.cu_seqlens = cu_seqlens;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.in_fp16 = x->dtype == KDA_DTYPE_FP16; p.state_bf16 = x->state_bf16;
  p.h0 = initial_state; p.hT = final_state; p.cache = state_cache;
  p.slot_stride = slot_stride; p.n_slots = n_slots;
  p.state_indices = state_indices; p.has_init = has_initial_state;
  p.groups = G;
  p.pipeline = groups == -1 ? 2 : (groups <= 0 && G == 1 ? 1 : 0);
  p.sm_count = device_sm_count();
  p.ckpt = checkpoint_state; p.ckpt_stride = checkpoint_row_stride; p.ckpt_rows = checkpoint_rows;
  p.ckpt_off = checkpoint_offsets; p.ckpt_idx = checkpoint_state_indices;
  p.conv = cp;
  p.conv_out = conv ? static_cast<__nv_bfloat16*>(conv->scratch) : nullptr;
  p.err = err;
  const int lrc = kda::launch_chunk(p, workspace, static_cast<cudaStream_t>(stream));
  if (lrc == -2) return KDA_ERR_INVALID_ARGUMENT;  // message set by the launcher
  if (lrc != 0) return cuda_fail(cudaGetLastError(), "kda_chunk_fwd launch");
  return ok();
}

int kda_chunk_fwd(const kda_activations* x, void* out, const int32_t* cu_seqlens, int32_t n_seqs,
                  const void* initial_state, void* final_state, void* state_cache,
                  int64_t slot_stride, int64_t n_slots, const int32_t* state_indices,
                  const uint8_t* has_initial_state, int32_t groups, void* workspace,
                  size_t workspace_bytes, void* stream) {
  return chunk_common(x, out, cu_seqlens, n_seqs, initial_state, final_state, state_cache, slot_stride,
                      n_slots, state_indices, has_initial_state, nullptr, 0, 0, nullptr, nullptr, nullptr,
                      groups, workspace, workspace_bytes, stream);
}

int kda_chunk_fwd_ex(const kda_activations* x, void* out, const int32_t* cu_seqlens, int32_t n_seqs,
                     const void* initial_state, void* final_state, void* state_cache,
                     int64_t slot_stride, int64_t n_slots, const int32_t* state_indices,
                     const uint8_t* has_initial_state, void* checkpoint_state,
                     int64_t checkpoint_row_stride, int64_t checkpoint_rows,
                     const int32_t* checkpoint_offsets, const int32_t* checkpoint_state_indices,
                     const kda_conv* conv, int32_t groups, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return chunk_common(x, out, cu_seqlens, n_seqs, initial_state, final_state, state_cache, slot_stride,
                      n_slots, state_indices, has_initial_state, checkpoint_state, checkpoint_row_stride,
                      checkpoint_rows, checkpoint_offsets, checkpoint_state_indices, conv, groups, workspace,
                      workspace_bytes, stream);
}

// --- prefill from host memory ---------------------------------------------
// Chunked prefill in the serving sense: each sequence is cut into segments of
// L tokens (a multiple of the 64-token chunk, so the kernels' chunks are the
// ones an uncut prefill forms), and call j runs segment j of every sequence
// still active as one varlen prefill, the fp32 state carried from call to
// call in a state-cache table in the workspace.  Three streams: copy-in
// (host to device mirrors), compute, copy-out; call j computes while call
// j + 1's rows arrive and call j - 1's outputs leave.
namespace {

constexpr size_t HOST_ALIGN = 256;
size_t align_up(size_t n) { return (n + HOST_ALIGN - 1) / HOST_ALIGN * HOST_ALIGN; }

struct HostPlan {
  int n_calls = 0;
  std::vector<int64_t> bnd;                // call j covers tokens bnd[j] .. bnd[j+1] of each sequence
  bool dense = false;                      // n_seqs sequences of t_total / n_seqs tokens
  std::vector<int64_t> start, len;         // per sequence, host rows
  std::vector<int32_t> call_n, call_rows;  // per call: sequences, tokens
  std::vector<int64_t> call_row;           // per call: first row in the device mirrors
  std::vector<uint8_t> call_dense;         // the call's pieces are equally long
  std::vector<int64_t> call_meta;          // per call: int32 offset of its cu_seqlens, then indices
  std::vector<size_t> call_ws;             // per call: chunk workspace bytes
  size_t meta_ints = 0;
  // the table block, staged page-locked on the host and moved by one copy:
  // call tables (int32), A_log, dt_bias, beta of every call (call-major)
  size_t tab_alog = 0, tab_dt = 0, tab_beta = 0, tab_bytes = 0;
  size_t off_q = 0, off_k = 0, off_v = 0, off_g = 0, off_o = 0, off_cache = 0, off_tab = 0, off_ws = 0,
         total = 0;
};

// Validates a host-memory prefill and lays out its calls and workspace.
int plan_host(const kda_activations* x, const int32_t* cu, int32_t n_seqs, int32_t segment,
              int32_t groups, HostPlan& P) {
  int rc = check_activations(x, false);
  if (rc) return rc;
  if (x->state_bf16 != 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "the host-memory prefill carries fp32 states only (state_bf16 = 0).");
  if (n_seqs <= 0) return fail(KDA_ERR_INVALID_ARGUMENT, "n_seqs must be >= 1.");
  if (segment > 0 && segment % kda::CHUNK != 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "segment_tokens must be a positive multiple of %d (got %d).",
                kda::CHUNK, segment);
  const int64_t T = x->t_total, hqk = x->hqk, hv = x->hv, D = kda::D;
  if (T > 0) {
    if ((hqk > 1 && (x->q_stride_head != D || x->k_stride_head != D)) ||
        (hv > 1 && (x->v_stride_head != D || x->g_stride_head != D)) || (hv > 1 && x->beta_stride_head != 1))
      return fail(KDA_ERR_INVALID_ARGUMENT,
                  "host rows need contiguous heads (q/k/v/g head stride 128, beta head stride 1).");
    if (x->q_stride_tok < hqk * D || x->k_stride_tok < hqk * D || x->v_stride_tok < hv * D ||
        x->g_stride_tok < hv * D || x->beta_stride_tok < hv)
      return fail(KDA_ERR_INVALID_ARGUMENT, "host token strides must cover a token's heads.");
  }
  P.start.assign(n_seqs, 0);
  P.len.assign(n_seqs, 0);
  P.dense = cu == nullptr;
  if (cu) {
    if (cu[0] != 0 || cu[n_seqs] != T)
      return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must run from 0 to t_total.");
    for (int b = 0; b < n_seqs; ++b) {
      if (cu[b + 1] < cu[b]) return fail(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must be non-decreasing.");
      P.start[b] = cu[b];
      P.len[b] = cu[b + 1] - cu[b];
    }
  } else {
    if (T % n_seqs != 0)
      return fail(KDA_ERR_INVALID_ARGUMENT, "dense mode (no cu_seqlens) needs t_total divisible by n_seqs.");
    for (int b = 0; b < n_seqs; ++b) {
      P.start[b] = (T / n_seqs) * b;
      P.len[b] = T / n_seqs;
    }
  }
  int64_t max_len = 0;
  for (int64_t l : P.len) max_len = l > max_len ? l : max_len;
  // Segment boundaries.  Given a length: uniform.  By default: shrinking
  // towards the end, so that the last call's prefill and output copy, the
  // part no later copy hides, are short, while each call's prefill still
  // fits under the next call's copy-in (a prefill segment here runs about
  // twice as fast as the host link delivers its rows): from the end 256,
  // 256, 512, 1024, ... doubling up to 4096 tokens, the first segment taking
  // the rest.  (B=2 x 4096 tokens, H=16 on GB300: 1.13 ms a step as one
  // segment, 0.89 in four of 1024.)
  P.bnd.assign(1, 0);
  if (segment > 0) {
    for (int64_t b = segment; b - segment < max_len; b += segment) P.bnd.push_back(b);
  } else if (max_len > 0) {
    std::vector<int64_t> tail;  // segment lengths from the end
    int64_t covered = 0, next = 256;
    while (covered < max_len) {
      tail.push_back(next);
      covered += next;
      if (tail.size() >= 2) next = std::min<int64_t>(2 * next, 4096);
    }
    for (size_t i = tail.size(); i-- > 0;) P.bnd.push_back(P.bnd.back() + tail[i]);
    // the first segment shrinks to what the sequence leaves, in whole chunks
    const int64_t over = (P.bnd.back() - max_len) / kda::CHUNK * kda::CHUNK;
    for (size_t i = 1; i < P.bnd.size(); ++i) P.bnd[i] -= over;
  }
  P.n_calls = (int)P.bnd.size() - 1;
  int64_t row = 0;
  for (int j = 0; j < P.n_calls; ++j) {
    int32_t n = 0, rows = 0;
    int64_t first = -1;
    bool eq = true;
    for (int b = 0; b < n_seqs; ++b) {
      if (P.len[b] <= P.bnd[j]) continue;
      const int64_t piece = std::min<int64_t>(P.bnd[j + 1], P.len[b]) - P.bnd[j];
      if (first < 0) first = piece;
      eq &= piece == first;
      ++n;
      rows += (int32_t)piece;
    }
    P.call_n.push_back(n);
    P.call_rows.push_back(rows);
    P.call_row.push_back(row);
    P.call_dense.push_back(eq);
    P.call_meta.push_back((int64_t)P.meta_ints);
    P.meta_ints += 2 * (size_t)n + 1;
    const int G = choose_groups(n, rows, x->hv, groups);
    P.call_ws.push_back(4 * kda::chunk_workspace_floats(n, rows, x->hv, G, nullptr));
    row += rows;
  }
  const size_t es = 2;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
  P.off_q = take(T * hqk * D * es);
  P.off_k = take(T * hqk * D * es);
  P.off_v = take(T * hv * D * es);
  P.off_g = take(T * hv * D * es);
  P.off_o = take(T * hv * D * es);
  P.off_cache = take((size_t)n_seqs * hv * D * D * 4);
  P.tab_alog = align_up(P.meta_ints * 4);
  P.tab_dt = align_up(P.tab_alog + (x->A_log ? hv * 4 : 0));
  P.tab_beta = align_up(P.tab_dt + (x->A_log ? hv * D * 4 : 0));
  P.tab_bytes = P.tab_beta + T * hv * es;
  P.off_tab = take(P.tab_bytes);
  size_t ws = 0;
  for (size_t w : P.call_ws) ws = w > ws ? w : ws;
  P.off_ws = take(ws);
  P.total = o;
  return KDA_OK;
}

struct HostCtx {
  std::mutex mu;
  bool ready = false;
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> ev;
  unsigned char* meta = nullptr;  // page-locked staging of the table block
  size_t meta_cap = 0;            // bytes
  cudaEvent_t meta_done = nullptr;
  bool meta_used = false;
};
HostCtx g_host_ctx[64];

int host_ctx_ready(HostCtx& c, size_t events, size_t meta_bytes) {
  cudaError_t e = cudaSuccess;
  if (!c.ready) {
    if ((e = cudaStreamCreateWithFlags(&c.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&c.s_comp, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&c.s_out, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c.meta_done, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e, "host prefill streams");
    c.ready = true;
  }
  while (c.ev.size() < events) {
    cudaEvent_t ev = nullptr;
    if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e, "host prefill events");
    c.ev.push_back(ev);
  }
  // the previous call's tables have left the staging buffer
  if (c.meta_used && (e = cudaEventSynchronize(c.meta_done)) != cudaSuccess)
    return cuda_fail(e, "host prefill tables");
  if (meta_bytes > c.meta_cap) {
    if (c.meta) cudaFreeHost(c.meta);
    c.meta = nullptr;
    c.meta_cap = 0;
    const size_t cap = meta_bytes < 4096 ? 4096 : 2 * meta_bytes;
    if ((e = cudaHostAlloc(reinterpret_cast<void**>(&c.meta), cap, cudaHostAllocDefault)) != cudaSuccess)
      return cuda_fail(e, "host prefill tables");
    c.meta_cap = cap;
  }
  return KDA_OK;
}

// rows x row_bytes from a strided source to a packed destination
cudaError_t copy_rows(void* dst, const void* src, size_t row_bytes, size_t src_pitch, size_t rows,
                      cudaMemcpyKind kind, cudaStream_t s) {
  if (rows == 0 || row_bytes == 0) return cudaSuccess;
  if (src_pitch == row_bytes) return cudaMemcpyAsync(dst, src, row_bytes * rows, kind, s);
  return cudaMemcpy2DAsync(dst, row_bytes, src, src_pitch, row_bytes, rows, kind, s);
}

}  // namespace

size_t kda_chunk_fwd_host_workspace_bytes(const kda_activations* x, const int32_t* cu_seqlens,
                                          int32_t n_seqs, int32_t segment_tokens, int32_t groups) {
  HostPlan P;
  if (plan_host(x, cu_seqlens, n_seqs, segment_tokens, groups, P) != KDA_OK) return 0;
  return P.total + HOST_ALIGN;
}

int kda_chunk_fwd_host(const kda_activations* x, void* out, const int32_t* cu_seqlens, int32_t n_seqs,
                       const float* initial_state, float* final_state, int32_t segment_tokens,
                       int32_t groups, void* workspace, size_t workspace_bytes, void* stream) {
  HostPlan P;
  int rc = plan_host(x, cu_seqlens, n_seqs, segment_tokens, groups, P);
  if (rc) return rc;
  if (x->t_total > 0 && !out) return fail(KDA_ERR_INVALID_ARGUMENT, "out must not be NULL.");
  if (!workspace || workspace_bytes < P.total + HOST_ALIGN)
    return fail(KDA_ERR_INVALID_ARGUMENT, "workspace needs %zu bytes (got %zu).", P.total + HOST_ALIGN,
                workspace ? workspace_bytes : (size_t)0);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(KDA_ERR_CUDA, "device ordinal %d out of range.", dev);
  HostCtx& c = g_host_ctx[dev];
  std::lock_guard<std::mutex> lock(c.mu);
  rc = host_ctx_ready(c, 2 * (size_t)P.n_calls + 3, P.tab_bytes);
  if (rc) return rc;
  const int64_t hqk = x->hqk, hv = x->hv, D = kda::D, es = 2;
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(workspace) + HOST_ALIGN - 1) / HOST_ALIGN * HOST_ALIGN);
  float* cache = reinterpret_cast<float*>(base + P.off_cache);
  const size_t state_bytes = (size_t)n_seqs * hv * D * D * 4;
  // the call tables: cu_seqlens of the packed call, then its sequences' cache rows
  for (int j = 0; j < P.n_calls; ++j) {
    int32_t* cu = reinterpret_cast<int32_t*>(c.meta) + P.call_meta[j];
    int32_t* idx = cu + P.call_n[j] + 1;
    int n = 0, acc = 0;
    cu[0] = 0;
    for (int b = 0; b < n_seqs; ++b) {
      if (P.len[b] <= P.bnd[j]) continue;
      acc += (int)(std::min<int64_t>(P.bnd[j + 1], P.len[b]) - P.bnd[j]);
      idx[n] = b;
      cu[++n] = acc;
    }
  }
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  cudaEvent_t ev_start = c.ev[0], ev_end = c.ev[1], ev_init = c.ev[2];
  auto step = [&](cudaError_t r, const char* what) {
    if (r != cudaSuccess && rc == KDA_OK) rc = cuda_fail(r, what);
    return rc == KDA_OK;
  };
  step(cudaEventRecord(ev_start, user), "cudaEventRecord");
  for (cudaStream_t s : {c.s_in, c.s_comp, c.s_out}) step(cudaStreamWaitEvent(s, ev_start, 0), "cudaStreamWaitEvent");
  if (rc) return rc;
  // the gate parameters and every call's beta rows (call-major) join the
  // tables: each copy costs the copy engine a few microseconds on top of
  // its bytes, so the small ones travel as one
  if (x->A_log) {
    memcpy(c.meta + P.tab_alog, x->A_log, hv * 4);
    memcpy(c.meta + P.tab_dt, x->dt_bias, hv * D * 4);
  }
  {
    const size_t rb = hv * es, pitch = x->beta_stride_tok * es;
    unsigned char* dst = c.meta + P.tab_beta;
    for (int j = 0; j < P.n_calls; ++j)
      for (int b = 0; b < n_seqs; ++b) {
        if (P.len[b] <= P.bnd[j]) continue;
        const int64_t piece = std::min<int64_t>(P.bnd[j + 1], P.len[b]) - P.bnd[j];
        const unsigned char* src = static_cast<const unsigned char*>(x->beta) + (P.start[b] + P.bnd[j]) * pitch;
        if (pitch == rb) {
          memcpy(dst, src, piece * rb);
          dst += piece * rb;
        } else {
          for (int64_t r = 0; r < piece; ++r, dst += rb) memcpy(dst, src + r * pitch, rb);
        }
      }
  }
  if (P.tab_bytes)
    step(cudaMemcpyAsync(base + P.off_tab, c.meta, P.tab_bytes, cudaMemcpyHostToDevice, c.s_in), "tables");
  step(cudaEventRecord(c.meta_done, c.s_in), "cudaEventRecord");
  c.meta_used = true;
  if (initial_state)
    step(cudaMemcpyAsync(cache, initial_state, state_bytes, cudaMemcpyHostToDevice, c.s_in), "initial_state");
  else
    step(cudaMemsetAsync(cache, 0, state_bytes, c.s_in), "zero initial state");

  struct Band { const void* host; int64_t tok_stride, width; size_t off; };
  const Band bands[4] = {{x->q, x->q_stride_tok, hqk * D, P.off_q}, {x->k, x->k_stride_tok, hqk * D, P.off_k},
                         {x->v, x->v_stride_tok, hv * D, P.off_v}, {x->g, x->g_stride_tok, hv * D, P.off_g}};
  const int64_t out_row = hv * D * es;
  for (int j = 0; j < P.n_calls && rc == KDA_OK; ++j) {
    cudaEvent_t ev_in = c.ev[3 + 2 * j], ev_comp = c.ev[4 + 2 * j];
    const int64_t jL = P.bnd[j], jR = P.bnd[j + 1];
    const int64_t piece0 = std::min<int64_t>(jR, P.len[0]) - jL;
    // copy in (q, k, v, g; beta came with the tables): a dense call's pieces
    // are evenly spaced, one 2-D copy per band
    for (const Band& bd : bands) {
      const size_t rb = bd.width * es, pitch = bd.tok_stride * es;
      unsigned char* dst = base + bd.off + P.call_row[j] * rb;
      if (P.dense && pitch == rb && (size_t)P.len[0] * rb < ((size_t)1 << 31)) {
        const size_t w = piece0 * rb;
        step(cudaMemcpy2DAsync(dst, w, static_cast<const unsigned char*>(bd.host) + jL * rb, P.len[0] * rb, w,
                               P.call_n[j], cudaMemcpyHostToDevice, c.s_in), "copy in");
        continue;
      }
      for (int b = 0; b < n_seqs; ++b) {
        if (P.len[b] <= jL) continue;
        const int64_t piece = std::min<int64_t>(jR, P.len[b]) - jL;
        step(copy_rows(dst, static_cast<const unsigned char*>(bd.host) + (P.start[b] + jL) * pitch, rb, pitch,
                       piece, cudaMemcpyHostToDevice, c.s_in), "copy in");
        dst += piece * rb;
      }
    }
    step(cudaEventRecord(ev_in, c.s_in), "cudaEventRecord");
    step(cudaStreamWaitEvent(c.s_comp, ev_in, 0), "cudaStreamWaitEvent");
    if (rc) break;
    // compute: the packed call against the cache rows of its sequences
    kda_activations xd = *x;
    xd.q = base + P.off_q + P.call_row[j] * hqk * D * es;
    xd.k = base + P.off_k + P.call_row[j] * hqk * D * es;
    xd.v = base + P.off_v + P.call_row[j] * hv * D * es;
    xd.g = base + P.off_g + P.call_row[j] * hv * D * es;
    xd.beta = base + P.off_tab + P.tab_beta + P.call_row[j] * hv * es;
    xd.q_stride_tok = xd.k_stride_tok = hqk * D;
    xd.v_stride_tok = xd.g_stride_tok = hv * D;
    xd.q_stride_head = xd.k_stride_head = xd.v_stride_head = xd.g_stride_head = D;
    xd.beta_stride_tok = hv;
    xd.beta_stride_head = 1;
    xd.A_log = x->A_log ? reinterpret_cast<const float*>(base + P.off_tab + P.tab_alog) : nullptr;
    xd.dt_bias = x->A_log ? reinterpret_cast<const float*>(base + P.off_tab + P.tab_dt) : nullptr;
    xd.t_total = P.call_rows[j];
    const int32_t* mcu = reinterpret_cast<const int32_t*>(base + P.off_tab) + P.call_meta[j];
    unsigned char* out_dev = base + P.off_o + P.call_row[j] * out_row;
    rc = chunk_common(&xd, out_dev, P.call_dense[j] ? nullptr : mcu, P.call_n[j], nullptr, nullptr, cache,
                      hv * D * D, n_seqs, mcu + P.call_n[j] + 1, nullptr, nullptr, 0, 0, nullptr, nullptr,
                      nullptr, groups, base + P.off_ws, P.call_ws[j], c.s_comp);
    step(cudaEventRecord(ev_comp, c.s_comp), "cudaEventRecord");
    step(cudaStreamWaitEvent(c.s_out, ev_comp, 0), "cudaStreamWaitEvent");
    if (rc) break;
    // copy out: the call's output rows back to their tokens
    if (P.dense && (size_t)P.len[0] * out_row < ((size_t)1 << 31)) {
      const size_t w = piece0 * out_row;
      step(cudaMemcpy2DAsync(static_cast<unsigned char*>(out) + jL * out_row, P.len[0] * out_row, out_dev, w, w,
                             P.call_n[j], cudaMemcpyDeviceToHost, c.s_out), "copy out");
      continue;
    }
    for (int b = 0; b < n_seqs; ++b) {
      if (P.len[b] <= jL) continue;
      const int64_t piece = std::min<int64_t>(jR, P.len[b]) - jL;
      step(cudaMemcpyAsync(static_cast<unsigned char*>(out) + (P.start[b] + jL) * out_row, out_dev,
                           piece * out_row, cudaMemcpyDeviceToHost, c.s_out), "copy out");
      out_dev += piece * out_row;
    }
  }
  // join: copy-out after every copy-in and compute, the caller's stream after copy-out
  const int keep = rc;
  rc = KDA_OK;
  step(cudaEventRecord(ev_init, c.s_in), "cudaEventRecord");
  step(cudaStreamWaitEvent(c.s_out, ev_init, 0), "cudaStreamWaitEvent");
  if (keep == KDA_OK && final_state)
    step(cudaMemcpyAsync(final_state, cache, state_bytes, cudaMemcpyDeviceToHost, c.s_out), "final_state");
  step(cudaEventRecord(ev_end, c.s_comp), "cudaEventRecord");
  step(cudaStreamWaitEvent(c.s_out, ev_end, 0), "cudaStreamWaitEvent");
  step(cudaEventRecord(ev_end, c.s_out), "cudaEventRecord");
  step(cudaStreamWaitEvent(user, ev_end, 0), "cudaStreamWaitEvent");
  if (keep != KDA_OK) return keep;
  return rc == KDA_OK ? ok() : rc;
}

static int window_common(const kda_activations* x, void* out, const void* pool, int64_t slot_stride,
                         int64_t n_slots, const int32_t* query_start, const int32_t* slots,
                         int32_t n_req, int32_t window, bool verify, float* corr, void* kg,
                         int32_t* counter, void* stream, const int32_t* step_slots = nullptr,
                         int64_t step_stride = 0, const int32_t* n_accepted = nullptr,
                         const kda_conv* conv = nullptr) {
  int rc = check_activations(x, true);
  if (rc) return rc;
  kda::ConvParams cp;
  rc = check_conv(conv, x, true, window, n_slots, cp);
  if (rc) return rc;
  if (window < 1 || window > kda::MAX_WINDOW)
    return fail(KDA_ERR_INVALID_ARGUMENT, "window must satisfy 1 <= window <= 8 (got %d).", window);
  if (n_req < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "n_req must be >= 0.");
  if (step_slots && step_stride < window)
    return fail(KDA_ERR_INVALID_ARGUMENT,
                "state_indices needs at least window = %d columns, got %lld.", window,
                (long long)step_stride);
  if (n_req == 0) return ok();
  if (!query_start || !(slots || step_slots))
    return fail(KDA_ERR_INVALID_ARGUMENT, "query_start and state_indices must not be NULL.");
  if (x->t_total > 0 && !out) return fail(KDA_ERR_INVALID_ARGUMENT, "out must not be NULL.");
  rc = check_pool(pool, slot_stride, n_slots, x->hv, x->state_bf16, "state_pool");
  if (rc) return rc;
  if (verify && (!corr || !kg || !counter))
    return fail(KDA_ERR_INVALID_ARGUMENT, "verify needs corr, kg and work_counter.");
  if ((int64_t)n_req * x->hv > 0x7fffffff)
    return fail(KDA_ERR_INVALID_ARGUMENT, "n_req * Hv exceeds 2^31.");
  unsigned* err = error_word_ptr();
  if (!err) return fail(KDA_ERR_CUDA, "cannot resolve the device error word.");
  kda::WindowParams p;
  memset(&p, 0, sizeof(p));
  fill_common(x, p.q, p.k, p.v, p.g, p.beta);
  p.q_st = x->q_stride_tok; p.q_sh = x->q_stride_head;
  p.k_st = x->k_stride_tok; p.k_sh = x->k_stride_head;
  p.v_st = x->v_stride_tok; p.v_sh = x->v_stride_head;
  p.g_st = x->g_stride_tok; p.g_sh = x->g_stride_head;
  p.b_st = x->beta_stride_tok; p.b_sh = x->beta_stride_head;
  p.A_log = x->A_log; p.dt_bias = x->dt_bias; p.has_gate = x->A_log != nullptr;
  p.scale = x->scale; p.lower_bound = x->lower_bound;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.pool = const_cast<void*>(pool);
  p.in_fp16 = x->dtype == KDA_DTYPE_FP16; p.state_bf16 = x->state_bf16;
  p.slot_stride = slot_stride; p.n_slots = n_slots;
  p.query_start = query_start; p.slots = slots;
  p.step_slots = step_slots; p.step_stride = step_stride; p.n_accepted = n_accepted;
  p.conv = cp;
  p.n_req = n_req; p.window = window; p.hqk = x->hqk; p.hv = x->hv;
  p.corr = corr; p.kg = static_cast<__nv_bfloat16*>(kg); p.counter = counter;
  p.err = err;
  if (kda::launch_window(p, verify, static_cast<cudaStream_t>(stream)) != 0)
    return cuda_fail(cudaGetLastError(), verify ? "kda_verify launch" : "kda_decode launch");
  return ok();
}

int kda_decode(const kda_activations* x, void* out, void* state_pool, int64_t slot_stride,
               int64_t n_slots, const int32_t* query_start, const int32_t* slots, int32_t n_req,
               int32_t window, void* stream) {
  return window_common(x, out, state_pool, slot_stride, n_slots, query_start, slots, n_req,
                       window, false, nullptr, nullptr, nullptr, stream);
}

int kda_decode_steps(const kda_activations* x, void* out, void* state_pool, int64_t slot_stride,
                     int64_t n_slots, const int32_t* query_start, const int32_t* state_indices,
                     int64_t indices_stride, const int32_t* num_accepted_tokens, int32_t n_req,
                     int32_t window, void* stream) {
  if (!state_indices && n_req > 0)
    return fail(KDA_ERR_INVALID_ARGUMENT, "query_start and state_indices must not be NULL.");
  return window_common(x, out, state_pool, slot_stride, n_slots, query_start, nullptr, n_req, window,
                       false, nullptr, nullptr, nullptr, stream, state_indices, indices_stride,
                       num_accepted_tokens);
}

int kda_verify(const kda_activations* x, void* out, const void* state_pool, int64_t slot_stride,
               int64_t n_slots, const int32_t* query_start, const int32_t* slots, int32_t n_req,
               int32_t window, float* corr, void* kg, int32_t* work_counter, void* stream) {
  return window_common(x, out, state_pool, slot_stride, n_slots, query_start, slots, n_req,
                       window, true, corr, kg, work_counter, stream);
}

int kda_verify_ex(const kda_activations* x, void* out, const void* state_pool, int64_t slot_stride,
                  int64_t n_slots, const int32_t* query_start, const int32_t* slots, int32_t n_req,
                  int32_t window, float* corr, void* kg, int32_t* work_counter, const kda_conv* conv,
                  void* stream) {
  return window_common(x, out, state_pool, slot_stride, n_slots, query_start, slots, n_req, window, true,
                       corr, kg, work_counter, stream, nullptr, 0, nullptr, conv);
}

int kda_commit(float* state_pool, int64_t slot_stride, int64_t n_slots, const int32_t* slots,
               const int32_t* num_accepted, int32_t n_req, int32_t hv, int32_t window,
               const float* corr, const void* kg, const float* A_log, const float* dt_bias,
               float lower_bound, void* stream) {
  return kda_commit_ex(state_pool, slot_stride, n_slots, slots, num_accepted, n_req, hv, window, corr, kg,
                       A_log, dt_bias, lower_bound, 0, 0, stream);
}

int kda_commit_ex(void* state_pool, int64_t slot_stride, int64_t n_slots, const int32_t* slots,
                  const int32_t* num_accepted, int32_t n_req, int32_t hv, int32_t window,
                  const float* corr, const void* kg, const float* A_log, const float* dt_bias,
                  float lower_bound, int32_t state_bf16, int32_t kg_fp16, void* stream) {
  if ((state_bf16 != 0 && state_bf16 != 1) || (kg_fp16 != 0 && kg_fp16 != 1))
    return fail(KDA_ERR_INVALID_ARGUMENT, "state_bf16 and kg_fp16 must be 0 or 1.");
  if (window < 1 || window > kda::MAX_WINDOW)
    return fail(KDA_ERR_INVALID_ARGUMENT, "window must satisfy 1 <= window <= 8 (got %d).", window);
  if (n_req < 0) return fail(KDA_ERR_INVALID_ARGUMENT, "n_req must be >= 0.");
  if (hv <= 0) return fail(KDA_ERR_INVALID_ARGUMENT, "hv must be positive (got %d).", hv);
  if (n_req == 0) return ok();
  if (!slots || !num_accepted)
    return fail(KDA_ERR_INVALID_ARGUMENT, "slots and num_accepted must not be NULL.");
  if (!corr || !kg) return fail(KDA_ERR_INVALID_ARGUMENT, "corr and kg must not be NULL.");
  if (!aligned16(corr) || !aligned16(kg))
    return fail(KDA_ERR_INVALID_ARGUMENT, "corr and kg must be 16-byte aligned.");
  if ((A_log == nullptr) != (dt_bias == nullptr))
    return fail(KDA_ERR_INVALID_ARGUMENT, "A_log and dt_bias must be provided together.");
  if (A_log && !aligned16(dt_bias)) return fail(KDA_ERR_INVALID_ARGUMENT, "dt_bias must be 16-byte aligned.");
  if (A_log && !(lower_bound <= 0.f && lower_bound >= -10.5f))
    return fail(KDA_ERR_INVALID_ARGUMENT, "lower_bound must lie in [-10.5, 0] (got %g).", (double)lower_bound);
  int rc = check_pool(state_pool, slot_stride, n_slots, hv, state_bf16, "state_pool");
  if (rc) return rc;
  if ((int64_t)n_req * hv > 0x7fffffff)
    return fail(KDA_ERR_INVALID_ARGUMENT, "n_req * Hv exceeds 2^31.");
  unsigned* err = error_word_ptr();
  if (!err) return fail(KDA_ERR_CUDA, "cannot resolve the device error word.");
  kda::CommitParams p;
  memset(&p, 0, sizeof(p));
  p.pool = state_pool; p.slot_stride = slot_stride; p.n_slots = n_slots;
  p.state_bf16 = state_bf16; p.kg_fp16 = kg_fp16;
  p.slots = slots; p.accepted = num_accepted;
  p.corr = corr; p.kg = static_cast<const __nv_bfloat16*>(kg);
  p.A_log = A_log; p.dt_bias = dt_bias; p.lower_bound = lower_bound; p.has_gate = A_log != nullptr;
  p.n_req = n_req; p.hv = hv; p.window = window;
  p.err = err;
  if (kda::launch_commit(p, static_cast<cudaStream_t>(stream)) != 0)
    return cuda_fail(cudaGetLastError(), "kda_commit launch");
  return ok();
}

int kda_device_status(void* stream, int32_t clear) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kda_device_status sync");
  unsigned word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "kda_device_status read");
  if (clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "kda_device_status clear");
  }
  if (word & kda::ERR_TIMEOUT) return fail(KDA_ERR_DEVICE_TIMEOUT, "a bounded device wait expired.");
  if (word & kda::ERR_INDEX)
    return fail(KDA_ERR_DEVICE_INDEX, "a kernel met an out-of-range slot or sequence length.");
  if (word & kda::ERR_RANGE)
    return fail(KDA_ERR_DEVICE_RANGE,
                "a prefill without gate parameters met a raw log decay outside [-10.5, 0].");
  return ok();
}

int kda_selftest_wait_timeout(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(KDA_ERR_INVALID_ARGUMENT, "limit_us must lie in [1, 1000000] (got %u).", limit_us);
  unsigned* err = error_word_ptr();
  if (!err) return fail(KDA_ERR_CUDA, "the device error word could not be resolved.");
  if (kda::launch_wait_selftest(err, (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream)) != 0)
    return cuda_fail(cudaGetLastError(), "kda_selftest_wait_timeout launch");
  return ok();
}

}  // extern "C"
