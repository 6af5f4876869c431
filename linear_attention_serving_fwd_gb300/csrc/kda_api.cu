// Host side of the C ABI declared in include/kda.h: argument validation
// (the shape, dtype and pairing rules of the MATE chunk_kda /
// gated_delta_rule_decode validation and of the vLLM fused_kda_chunk cache
// rules), the per-device error word, and the kernel launches.
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

unsigned* error_word_ptr() {
  static unsigned* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  }
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
  } else if (!conv->state_indices) {
    return fail(KDA_ERR_INVALID_ARGUMENT, "prefill with a conv needs conv state_indices.");
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
  p.sm_count = device_sm_count();
  p.ckpt = checkpoint_state; p.ckpt_stride = checkpoint_row_stride; p.ckpt_rows = checkpoint_rows;
  p.ckpt_off = checkpoint_offsets; p.ckpt_idx = checkpoint_state_indices;
  p.conv = cp;
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
  return ok();
}

}  // extern "C"
