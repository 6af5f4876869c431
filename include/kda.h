/*
 * kda.h - C ABI of the GB300 (sm_103a) Kimi Delta Attention forward path.
 *
 * The operation (all three entry points): the gated delta rule with
 * per-channel decay, head dimension K = V = 128, value heads Hv a multiple of
 * query/key heads Hqk (value head h reads query/key head h / (Hv/Hqk)):
 *
 *   gate_t = lower_bound * sigmoid(exp(A_log[h]) * (g_t + dt_bias[h]))   [K]
 *   beta_t = sigmoid(b_t)
 *   k^_t = k_t / sqrt(|k_t|^2 + 1e-6),  q~_t = scale * q_t / sqrt(|q_t|^2 + 1e-6)
 *   S_t  = (I - beta_t k^_t k^_t^T) diag(exp(gate_t)) S_{t-1} + beta_t k^_t v_t^T
 *   o_t  = S_t^T q~_t
 *
 * as the MATE kda module defines it (chunk_kda docstring: gate parameters
 * A_log [Hv] and dt_bias [Hv, 128], lower_bound default -5, in-kernel q/k L2
 * norm, scale default 128^-0.5, beta given as logits) and as the vLLM
 * kimi_k3 CuTeDSL verify page's windowed solve (KdaTcVerify.kernel, steps
 * 2-4) unrolls it.  Without A_log/dt_bias the gate input g is the log decay
 * and lower_bound is unused.
 *
 * Layouts.  Activations are token-major: q, k [T_tot, Hqk, 128];
 * v, g [T_tot, Hv, 128]; beta [T_tot, Hv], with explicit token and head
 * strides in elements and the last dimension contiguous (g and beta may be
 * column slices of a fused projection, as the vLLM kimi_k3 AMD kda_chunk page
 * notes for fused_kda_prologue).  Outputs o are [T_tot, Hv, 128] contiguous.
 * Recurrent states are fp32 (or bf16, kda_activations.state_bf16) and
 * V-first: [.., Hv, V=128, K=128] with K contiguous (the decode page's default state_v_first layout, the verify
 * page's [slots, H, V, K] state and fused_kda_chunk's final state).  A paged
 * cache is [slots, Hv, 128, 128] with a caller-chosen slot stride (in state
 * elements, 16-byte rows: a multiple of 4 for fp32, 8 for bf16,
 * >= Hv*128*128).
 *
 * Ownership.  Every pointer is caller-owned device memory unless stated; the
 * library allocates no device memory and never synchronises inside an entry
 * point.  Work is enqueued on ``stream`` (a cudaStream_t; NULL = legacy
 * default stream).  The library keeps one device-resident error word per
 * device, set by kernels that meet a bad index or an expired wait; read it
 * with kda_device_status().
 *
 * Errors.  Every entry point returns a kda_status.  Host-side validation
 * failures return before any launch and leave all outputs untouched; the
 * message is available from kda_last_error() (thread-local).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARGUMENT = 1, /* shape / pointer / size rule broken */
  KDA_ERR_UNSUPPORTED_DTYPE = 2, /* a dtype outside bf16/fp16 activations */
  KDA_ERR_CUDA = 3,              /* a CUDA runtime call or launch failed */
  KDA_ERR_DEVICE_TIMEOUT = 4,    /* a bounded device wait expired */
  KDA_ERR_DEVICE_INDEX = 5,      /* a kernel met a bad slot / length */
  KDA_ERR_DEVICE_RANGE = 6       /* a prefill without gate parameters met a raw
                                    log decay outside [-10.5, 0]: its outputs
                                    and states are not valid */
} kda_status;

enum { KDA_DTYPE_BF16 = 0, KDA_DTYPE_FP16 = 1 };

/* The activations of one call (token-major; strides in elements). */
typedef struct kda_activations {
  const void* q;    int64_t q_stride_tok, q_stride_head;       /* [T, Hqk, 128] */
  const void* k;    int64_t k_stride_tok, k_stride_head;       /* [T, Hqk, 128] */
  const void* v;    int64_t v_stride_tok, v_stride_head;       /* [T, Hv, 128]  */
  const void* g;    int64_t g_stride_tok, g_stride_head;       /* [T, Hv, 128]  */
  const void* beta; int64_t beta_stride_tok, beta_stride_head; /* [T, Hv] logits */
  const float* A_log;   /* [Hv] fp32, or NULL (then dt_bias must be NULL)      */
  const float* dt_bias; /* [Hv, 128] fp32 contiguous, or NULL                   */
  int32_t dtype;        /* KDA_DTYPE_BF16 or KDA_DTYPE_FP16: q, k, v, g, beta and
                           the output o all have this type                      */
  int32_t t_total;      /* total tokens T                                        */
  int32_t hqk, hv;      /* heads; hv % hqk == 0                                  */
  int32_t use_qk_l2norm;/* must be 1: the in-kernel L2 norm of q and k          */
  float scale;          /* q scale applied after the norm (128^-0.5 usual)       */
  float lower_bound;    /* gate lower bound in [-10.5, 0] (-5 usual); unused
                           without A_log                                        */
  int32_t state_bf16;   /* 0: every recurrent state of the call (initial, final,
                           cache, pool, snapshots) is fp32; 1: bf16, widened to
                           fp32 for arithmetic.  Prefill rounds the final state
                           (and snapshots) once; decode and verify round the
                           carried state after every token, as repeated
                           single-token decode would (the MATE decode page's
                           bf16 state).  Strides then count bf16 elements and
                           must be multiples of 8 (16-byte rows).              */
} kda_activations;

/*
 * kda_conv - the width-4 depthwise causal conv + SiLU that kda_chunk_fwd_ex
 * and kda_verify_ex can apply to q, k and v first: the conv arguments of
 * the vLLM kimi_k3 AMD kda_chunk page's fused_kda_prologue (conv_weight,
 * conv_state, conv_state_indices, conv_has_initial_state) and the conv path
 * of the verify page's KdaTcVerify.  q, k and v (kda_activations) are then
 * the raw bands of the QKV projection.  Channels number the q band, then k,
 * then v: C = (2*Hqk + Hv)*128, channel = band offset + head*128 + c.  Per
 * channel, with history inputs h0, h1, h2 (oldest first) before the inputs
 * x_t:  y_t = SiLU(w0 x_{t-3} + w1 x_{t-2} + w2 x_{t-1} + w3 x_t), rounded
 * to bf16; with bf16 taps each product is rounded to bf16 and the four are
 * summed in fp32 in tap order, with fp32 taps the sum is an fp32 fma chain
 * (the verify page's "stock kernel's order").
 *
 *   weight        [C, 4] contiguous, 16-byte aligned: bf16, or fp32 when
 *                 weight_f32 = 1 (the stock conv1d parameter)
 *   state         bf16 conv state; element (row, position, channel) at
 *                 state[row*row_stride + position*pos_stride +
 *                 channel*chan_stride] (token major [rows, positions, C] or
 *                 channel major [rows, C, positions], the verify page's
 *                 conv_dim_first), updated in place by the call
 *   rows, positions  its extent; prefill needs positions >= 3, verify
 *                 positions >= window + 2
 *   state_indices prefill: device int32 [n_seqs], the row of each sequence
 *                 (negative: zero history and no update; >= rows sets
 *                 KDA_ERR_DEVICE_INDEX, zero history, no update)
 *   has_initial_state prefill: device uint8 [n_seqs] or NULL (= all true);
 *                 0 starts that sequence from a zero history
 *   num_accepted  verify: device int32 [n_req]; request b's history is at
 *                 positions num_accepted[b]-1 .. num_accepted[b]+1 of row
 *                 slots[b] (the verify page's accepted tokens)
 *   scratch, scratch_bytes  prefill: device memory of at least
 *                 kda_conv_scratch_bytes(t_total, Hqk, Hv) bytes, 16-byte
 *                 aligned, or NULL.  With it the conv runs once per (token,
 *                 channel) in a pass of its own that writes the convolved
 *                 bands there, and the prefill reads them; without it each
 *                 (chunk, head) item of the prefill convolves its own rows
 *                 (so under GVA every v-head of a q/k head convolves the q/k
 *                 rows again).  The results are the same.  Verify: must be
 *                 NULL.
 * Prefill reads the history at positions 0..2 and leaves sequence n's last
 * three raw inputs there (a sequence shorter than three keeps the tail of
 * its history in front).  Verify leaves the rolled state: positions 0 and 1
 * = the two newest history inputs, position 2 + t = raw input t of the
 * window; an out-of-range num_accepted sets KDA_ERR_DEVICE_INDEX and the
 * request is treated as padding.  The conv-state update runs as its own
 * launch after every history has been read.
 */
typedef struct kda_conv {
  const void* weight;
  int32_t weight_f32;
  void* state;
  int64_t row_stride, pos_stride, chan_stride;
  int64_t rows;
  int32_t positions;
  const int32_t* state_indices;
  const uint8_t* has_initial_state;
  const int32_t* num_accepted;
  void* scratch;
  size_t scratch_bytes;
} kda_conv;

/* kda_conv_scratch_bytes - the conv scratch a prefill of t_total tokens with
 * Hqk q/k heads and Hv v heads can take: (2*Hqk + Hv)*128 bf16 values a
 * token.  Returns 0 on invalid sizes. */
size_t kda_conv_scratch_bytes(int32_t t_total, int32_t hqk, int32_t hv);

/*
 * kda_chunk_workspace_bytes - device scratch needed by kda_chunk_fwd.
 *   n_seqs  number of sequences; t_total total tokens; hv value heads;
 *   groups  chunk groups per sequence for the parallel scan (the same value
 *           later passed to kda_chunk_fwd; <= 0 lets the library choose).
 * The size covers the worst case chunk count t_total/64 + n_seqs and the
 * chunk-group scan buffers.  Returns 0 on invalid sizes.
 */
size_t kda_chunk_workspace_bytes(int32_t n_seqs, int32_t t_total, int32_t hv, int32_t groups);

/*
 * kda_chunk_fwd - chunked prefill (chunk = 64): the MATE chunk_kda contract
 * with fp32 or bf16 states, and the vLLM kimi_k3 AMD fused_kda_prologue +
 * fused_kda_chunk pair (including the paged-cache form and the chunk-group
 * parallel scan of _chunk_groups / _kda_group_workspace).
 *
 *   x              activations (see kda_activations)
 *   out            [T, Hv, 128] bf16 contiguous, written
 *   cu_seqlens     device int32 [n_seqs + 1] token offsets (0, .., T), or
 *                  NULL for n_seqs dense sequences of T / n_seqs tokens
 *   n_seqs         number of sequences (>= 1)
 *   initial_state  [n_seqs, Hv, 128, 128] state dtype, or NULL (zero start)
 *   final_state    [n_seqs, Hv, 128, 128] state dtype, or NULL (not returned)
 *   state_cache    [slots, Hv, 128, 128] paged cache (state dtype), or NULL.  When
 *                  given, sequence n starts from row state_indices[n] (zero
 *                  when has_initial_state[n] == 0) and its final state is
 *                  written back to that row; initial_state and final_state
 *                  must then be NULL.  A negative row skips the state I/O of
 *                  that sequence (zero start, final state dropped).
 *   slot_stride    elements between cache rows (16-byte rows, >= Hv*16384)
 *   n_slots        rows in the cache; a row >= n_slots sets
 *                  KDA_ERR_DEVICE_INDEX in the device error word and is skipped
 *   state_indices  device int32 [n_seqs]
 *   has_initial_state device uint8 [n_seqs] or NULL (= all true)
 *   groups         chunk groups per sequence (vLLM _chunk_groups): 1 walks
 *                  each chain serially, in a launch after the prologue's;
 *                  G > 1 runs the exact group scan (pass one per group,
 *                  serial composition of the transfer operators, pass two);
 *                  -1 runs the pipelined launch: one cooperative kernel in
 *                  which one CTA per (sequence, head) chain walks all 128
 *                  value columns while the other SMs run the prologue, the
 *                  walk taking each chunk as soon as its record is ready
 *                  (dense sequences only, at most 48 chains;
 *                  KDA_ERR_INVALID_ARGUMENT otherwise); 0 (or any other
 *                  value <= 0) lets the library choose among the three
 *   workspace      device scratch of >= kda_chunk_workspace_bytes(.., groups)
 *                  bytes, 16-byte aligned; contents need not be initialised
 *   stream         cudaStream_t
 * cu_seqlens must start at 0, be non-decreasing and end at T; a violation
 * found on the device sets KDA_ERR_DEVICE_INDEX.  The gate's 16-token
 * sub-chunk factorisation needs any 8 consecutive per-token log decays to
 * sum above -87, inside fp32's exponent range: always true for
 * lower_bound >= -10.5, which is enforced.  Without A_log / dt_bias every raw
 * g must lie in [-10.5, 0]; a value outside it (or NaN) sets
 * KDA_ERR_DEVICE_RANGE, and that call's outputs and states are not valid.
 */
int kda_chunk_fwd(const kda_activations* x, void* out, const int32_t* cu_seqlens,
                  int32_t n_seqs, const void* initial_state, void* final_state,
                  void* state_cache, int64_t slot_stride, int64_t n_slots,
                  const int32_t* state_indices, const uint8_t* has_initial_state,
                  int32_t groups, void* workspace, size_t workspace_bytes, void* stream);

/* Checkpoint offsets of kda_chunk_fwd_ex must be multiples of this (the
 * prefill's chunk length): the walk snapshots states at chunk boundaries. */
#define KDA_CHECKPOINT_ALIGNMENT 64

/*
 * kda_chunk_fwd_ex - kda_chunk_fwd plus mid-prefill state snapshots (the
 * vLLM kda_chunk page's fused_kda_chunk checkpoint_state /
 * checkpoint_offsets / checkpoint_state_indices).  All other arguments as
 * kda_chunk_fwd.
 *   checkpoint_state      [rows, Hv, 128, 128] (state dtype) destination, or NULL (no
 *                         snapshots; the offsets and indices must then be NULL).
 *                         Without indices it is a staging buffer with a row per
 *                         sequence; with them it may be the paged state cache.
 *   checkpoint_row_stride elements between rows (16-byte rows, >= Hv*16384)
 *   checkpoint_rows       rows in checkpoint_state; a destination row >= rows
 *                         sets KDA_ERR_DEVICE_INDEX and is skipped
 *   checkpoint_offsets    device int32 [n_seqs]: sequence n's state after
 *                         checkpoint_offsets[n] of its tokens is written to its
 *                         row.  0 disables the snapshot; an offset that is not a
 *                         positive multiple of KDA_CHECKPOINT_ALIGNMENT or
 *                         exceeds the sequence's length is skipped silently, so
 *                         callers filter rather than rely on the store.
 *   checkpoint_state_indices device int32 [n_seqs] destination rows, or NULL
 *                         (row n); a negative row disables that sequence's
 *                         snapshot
 *   conv                  the conv applied to q, k, v first (see kda_conv),
 *                         or NULL
 * Writing a snapshot row that the same call also uses as a state cache row
 * of another sequence is a race.
 */
int kda_chunk_fwd_ex(const kda_activations* x, void* out, const int32_t* cu_seqlens,
                     int32_t n_seqs, const void* initial_state, void* final_state,
                     void* state_cache, int64_t slot_stride, int64_t n_slots,
                     const int32_t* state_indices, const uint8_t* has_initial_state,
                     void* checkpoint_state, int64_t checkpoint_row_stride,
                     int64_t checkpoint_rows, const int32_t* checkpoint_offsets,
                     const int32_t* checkpoint_state_indices, const kda_conv* conv,
                     int32_t groups, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kda_chunk_fwd_noalloc - kda_chunk_fwd for callers that cannot allocate
 * device memory.  The paper has no counterpart; this is a deployment aid.
 *
 * Who needs it: a runtime that reserves all device memory up front, or that
 * records work into CUDA graphs and forbids cudaMalloc afterwards; a plugin
 * whose host owns the allocator; code that must not synchronise (cudaMalloc
 * may).  Such callers cannot provide the prefill's workspace.
 *
 * Same arguments and results as kda_chunk_fwd, without workspace and
 * workspace_bytes.  The scratch is one fixed 64 MiB array inside the library,
 * held by every GPU that loads the library until the process exits.  A call
 * whose kda_chunk_workspace_bytes(n_seqs, T, Hv, groups) exceeds 64 MiB is
 * rejected with KDA_ERR_INVALID_ARGUMENT before any launch.  The first call
 * on a device resolves the array's device address (cudaGetSymbolAddress), so
 * make that first call before any stream capture.  All calls share the one
 * array and it keeps the last call's contents; nothing in it needs to start
 * at zero.  Calls that overlap on the GPU (other streams, other threads) race
 * on it: serialise them.  Allocates nothing (no cudaMalloc / cudaFree).
 */
int kda_chunk_fwd_noalloc(const kda_activations* x, void* out, const int32_t* cu_seqlens,
                          int32_t n_seqs, const void* initial_state, void* final_state,
                          void* state_cache, int64_t slot_stride, int64_t n_slots,
                          const int32_t* state_indices, const uint8_t* has_initial_state,
                          int32_t groups, void* stream);

/*
 * kda_chunk_fwd_host - kda_chunk_fwd on activations, output and states in
 * HOST memory: the library moves them and overlaps the moves with the
 * prefill.  The paper has no counterpart; it is the serving form of chunked
 * prefill (the MATE chunk_kda contract cut into segments).
 *
 * Each sequence is cut into segments of segment_tokens tokens (the last one
 * shorter); call j runs segment j of every sequence still active as one
 * varlen prefill on device mirrors in the workspace, the fp32 state carried
 * from call to call.  Segments are multiples of the 64-token chunk, so the
 * chunks are those of an uncut prefill.  Three library streams copy the
 * rows in, compute and copy the outputs out, so call j computes while call
 * j + 1's rows arrive and call j - 1's outputs leave; the work is ordered
 * after earlier work on ``stream`` and ``stream`` waits for all of it.
 *
 *   x               q, k, v, g, beta, A_log, dt_bias are host pointers
 *                   (page-locked memory lets the copies overlap; pageable
 *                   memory works, without overlap).  Heads contiguous within
 *                   a token (q/k/v/g head stride 128, beta head stride 1);
 *                   any token stride that covers a token's heads.
 *                   state_bf16 must be 0.
 *   out             host [T, Hv, 128] contiguous, x->dtype, written
 *   cu_seqlens      host int32 [n_seqs + 1] (0 .. T, non-decreasing), or
 *                   NULL for n_seqs dense sequences of T / n_seqs tokens
 *   initial_state   host fp32 [n_seqs, Hv, 128, 128], or NULL (zero start)
 *   final_state     host fp32 [n_seqs, Hv, 128, 128], or NULL (dropped)
 *   segment_tokens  a positive multiple of 64: segments of that length; or
 *                   <= 0: segments shrinking towards the end (from the end
 *                   256, 256, 512, 1024, .. doubling up to 4096 tokens, the
 *                   first taking the rest), so the last call, which no copy
 *                   hides, is short
 *   groups          as kda_chunk_fwd, per call
 *   workspace       device memory of at least
 *                   kda_chunk_fwd_host_workspace_bytes(..) bytes: the
 *                   mirrors of the inputs and the output, the carried states
 *                   and each call's prefill scratch
 *   stream          cudaStream_t
 * The host buffers must stay valid, and the workspace untouched, until
 * ``stream`` reaches the end of this call's work.  Calls on one device share
 * the library streams and one page-locked buffer, in which a call stages its
 * call tables, A_log, dt_bias and beta rows for a single copy; a call reuses
 * it only after the previous call's block reached the device (it waits on
 * the host for that); not for stream capture.  Device-side rules and error
 * words as kda_chunk_fwd.
 */
int kda_chunk_fwd_host(const kda_activations* x, void* out, const int32_t* cu_seqlens, int32_t n_seqs,
                       const float* initial_state, float* final_state, int32_t segment_tokens,
                       int32_t groups, void* workspace, size_t workspace_bytes, void* stream);

/* kda_chunk_fwd_host_workspace_bytes - the workspace kda_chunk_fwd_host needs
 * for these arguments (the same x, cu_seqlens, n_seqs, segment_tokens and
 * groups); 0 when they are invalid (kda_last_error says why). */
size_t kda_chunk_fwd_host_workspace_bytes(const kda_activations* x, const int32_t* cu_seqlens,
                                          int32_t n_seqs, int32_t segment_tokens, int32_t groups);

/*
 * kda_decode - in-place decode of a short window (1 <= window <= 8 tokens per
 * request) on a paged state cache: the MATE gated_delta_rule_decode
 * contract for fp32 or bf16 V-first states with in-kernel gate, lower bound, beta
 * sigmoid and q/k L2 norm, continuous batching by slot.
 *
 *   x            activations; x->t_total = query_start[n_req]
 *   out          [T, Hv, 128] bf16, written (zero for padding requests)
 *   state_pool   [n_slots, Hv, 128, 128] (state dtype), read and updated in place:
 *                request b's row state_indices[b] ends holding the state
 *                after all of its tokens
 *   slot_stride  elements between rows (16-byte rows, >= Hv*16384)
 *   query_start  device int32 [n_req + 1]; request b owns tokens
 *                query_start[b] .. query_start[b+1]-1, at most ``window``
 *   slots        device int32 [n_req]; a negative slot is a padding entry
 *                (zero output, no state traffic); a slot >= n_slots or a
 *                request longer than ``window`` sets KDA_ERR_DEVICE_INDEX
 *                and is treated as padding
 * Requests must use distinct slots (two requests on one row race).
 */
int kda_decode(const kda_activations* x, void* out, void* state_pool,
               int64_t slot_stride, int64_t n_slots, const int32_t* query_start,
               const int32_t* slots, int32_t n_req, int32_t window, void* stream);

/*
 * kda_decode_steps - kda_decode with a [request, step] slot table and
 * accepted-token counts: the MATE gated_delta_rule_decode contract for
 * [B, T] state_indices with num_accepted_tokens (speculative, multi-token
 * in-place decode).  The page names these arguments and their shape rules;
 * the reading taken of their meaning is:
 *   state_indices        device int32 [n_req, indices_stride], indices_stride
 *                        >= window.  Request b reads its initial state from
 *                        row state_indices[b][c], c = num_accepted_tokens[b]-1
 *                        (c = 0 when num_accepted_tokens is NULL), and the
 *                        state after its token t is written to row
 *                        state_indices[b][t], t < its length.  A negative row
 *                        at column c makes b a padding request (zero output,
 *                        no state traffic); a negative row at column t skips
 *                        that store.  A row >= n_slots at column c or at any
 *                        column t < length, or c outside [0, indices_stride),
 *                        sets KDA_ERR_DEVICE_INDEX and b is treated as padding.
 *   num_accepted_tokens  device int32 [n_req] or NULL
 * All other arguments as kda_decode.  Columns that repeat a row are written
 * in token order, so the row ends holding the later token's state; with
 * every column of b equal to one slot this is kda_decode.  Rows must not be
 * shared between requests; the read row may be one of the request's own
 * write rows (it is read before any store).
 */
int kda_decode_steps(const kda_activations* x, void* out, void* state_pool, int64_t slot_stride,
                     int64_t n_slots, const int32_t* query_start, const int32_t* state_indices,
                     int64_t indices_stride, const int32_t* num_accepted_tokens, int32_t n_req,
                     int32_t window, void* stream);

/*
 * kda_verify - windowed speculative verify (1 <= window <= 8): the vLLM
 * kimi_k3 CuTeDSL KdaTcVerify contract with fp32 or bf16 states.  Same inputs and
 * outputs ``out`` as kda_decode, but the state pool is only read, and per
 * request b, value head h and window position t < qlen it records
 *   corr [n_req, Hv, window, 128] fp32 : the correction U_t (the delta-rule
 *        term beta_t (v_t - S_{t-1}^T k^_t) of token t)
 *   kg   [n_req, Hv, window, 256] activation dtype : raw k_t (its
 *        query/key head) then raw g_t, as loaded
 * from which the accepted prefix's state can be rebuilt.  Entries t >= qlen
 * and padding requests are not written.
 *   work_counter  device int32[1], zero on entry; the launch's persistent
 *                 scheduler takes tickets from it and leaves it zero.
 */
int kda_verify(const kda_activations* x, void* out, const void* state_pool,
               int64_t slot_stride, int64_t n_slots, const int32_t* query_start,
               const int32_t* slots, int32_t n_req, int32_t window, float* corr,
               void* kg, int32_t* work_counter, void* stream);

/*
 * kda_verify_ex - kda_verify with the conv path of the verify page
 * (KdaTcVerify with conv): q, k and v are the raw projection bands, each
 * request's tokens are convolved (width 4, SiLU, see kda_conv) after the
 * history at positions num_accepted[b]-1 .. num_accepted[b]+1 of conv row
 * slots[b] (conv->rows >= n_slots, conv->positions >= window + 2,
 * conv->num_accepted required), the recurrence runs on the convolved
 * values, the kg record holds the convolved k, and the conv state is left
 * rolled.  conv NULL: exactly kda_verify.  The SSM state pool is still only
 * read.
 */
int kda_verify_ex(const kda_activations* x, void* out, const void* state_pool,
                  int64_t slot_stride, int64_t n_slots, const int32_t* query_start,
                  const int32_t* slots, int32_t n_req, int32_t window, float* corr,
                  void* kg, int32_t* work_counter, const kda_conv* conv, void* stream);

/*
 * kda_commit - speculative-decode commit: rebuild each request's state after
 * its accepted prefix from the records kda_verify wrote, in place.  The
 * vLLM kimi_k3 verify page (KdaTcVerify) writes the corr and kg records so
 * that the accepted prefix's state can be rebuilt; with tokens t = 1..a of
 * request b accepted, the recurrence unrolls to
 *   S_a = diag(e^{L_a}) S_0 + sum_{t <= a} diag(e^{L_a - L_t}) k^_t U_t^T
 * (L_t the per-channel cumsum of gate_t, k^_t = k_t / sqrt(|k_t|^2 + 1e-6)).
 *   state_pool, slot_stride, n_slots : the pool kda_verify read (fp32
 *                  V-first rows, as in kda_decode); row slots[b] holds S_0
 *                  on entry and S_a on return
 *   slots          device int32[n_req]; negative = padding (skipped); a slot
 *                  >= n_slots sets KDA_ERR_DEVICE_INDEX and is skipped
 *   num_accepted   device int32[n_req], a in [0, window]; a = 0 leaves the
 *                  row untouched; a outside the range sets
 *                  KDA_ERR_DEVICE_INDEX and is skipped.  a must not exceed
 *                  the request's verified token count (records past it are
 *                  not defined).
 *   hv, window     value heads and the window kda_verify ran with
 *   corr, kg       kda_verify's records [n_req, hv, window, 128] fp32 and
 *                  [n_req, hv, window, 256] bf16, 16-byte aligned
 *   A_log, dt_bias, lower_bound : the gate parameters kda_verify used (both
 *                  NULL: raw g is the log decay)
 *   stream         cudaStream_t
 * Returns KDA_OK or an error status; nothing is allocated.
 */
int kda_commit(float* state_pool, int64_t slot_stride, int64_t n_slots, const int32_t* slots,
               const int32_t* num_accepted, int32_t n_req, int32_t hv, int32_t window,
               const float* corr, const void* kg, const float* A_log, const float* dt_bias,
               float lower_bound, void* stream);

/*
 * kda_commit_ex - kda_commit for the dtype variants of kda_verify: the pool
 * holds bf16 rows when state_bf16 = 1 (S_0 widened, S_a computed in fp32
 * and rounded once), and the kg record holds fp16 raw k and g when
 * kg_fp16 = 1 (a verify with KDA_DTYPE_FP16 activations).  slot_stride is
 * then in bf16 elements (a multiple of 8).  state_bf16 = kg_fp16 = 0 is
 * kda_commit.
 */
int kda_commit_ex(void* state_pool, int64_t slot_stride, int64_t n_slots, const int32_t* slots,
                  const int32_t* num_accepted, int32_t n_req, int32_t hv, int32_t window,
                  const float* corr, const void* kg, const float* A_log, const float* dt_bias,
                  float lower_bound, int32_t state_bf16, int32_t kg_fp16, void* stream);

/* Thread-local text of the last error returned on this thread ("" if none).
 * kda_last_error_message is the same function under the name the serving
 * contract uses; kda_last_error is kept for existing callers. */
const char* kda_last_error_message(void);
const char* kda_last_error(void);

/*
 * kda_device_status - synchronise ``stream``, read this device's error word
 * and return KDA_OK, KDA_ERR_DEVICE_INDEX, KDA_ERR_DEVICE_RANGE or
 * KDA_ERR_DEVICE_TIMEOUT (the most severe seen since the last clear, in the
 * order timeout, index, range).  clear != 0 resets the word.
 */
int kda_device_status(void* stream, int32_t clear);

/*
 * kda_selftest_wait_timeout - test aid for the bounded device waits; the
 * pages have no counterpart.  Launches one CTA on ``stream`` that holds
 * tensor memory as the chunk kernels do and waits, with their bounded
 * mbarrier wait, on a barrier that nothing arrives at.  After ``limit_us``
 * microseconds (1 .. 1,000,000) of wall time the wait gives up: the kernel
 * sets the timeout bit of the device error word, frees its tensor memory
 * and returns, so the context stays usable.  kda_device_status then returns
 * KDA_ERR_DEVICE_TIMEOUT.  Nothing faults or traps.  Returns KDA_OK once
 * launched, KDA_ERR_INVALID_ARGUMENT for a limit out of range.
 */
int kda_selftest_wait_timeout(uint32_t limit_us, void* stream);

/*
 * Kernel tracing (off by default).  kda_trace_enable(1) clears the totals and
 * starts recording a CUDA event pair around every kernel the library
 * launches, on the launching stream; kda_trace_enable(0) stops.
 * kda_trace_read(i, ..) synchronises on the recorded events, fills entry i
 * (kernel name, total milliseconds, launch count; any out pointer may be
 * NULL) and returns the number of entries.  Host-thread safe; not meant
 * for use inside CUDA graph capture.
 */
int kda_trace_enable(int32_t on);
int kda_trace_read(int32_t index, char* name, int32_t name_cap, double* total_ms,
                   int32_t* launches);

/* Library version, e.g. "kda-gb300 0.1 sm_103a". */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
