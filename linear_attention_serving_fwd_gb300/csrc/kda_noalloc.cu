// kda_chunk_fwd_noalloc: the chunked prefill for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace.  A runtime inside a
// CUDA-graph-only or pre-reserved memory plan may forbid cudaMalloc after
// start-up.  A plugin host may own the caching allocator.  Code on a path that
// must not synchronise cannot call cudaMalloc either, because cudaMalloc can
// synchronise the device.  For them this file keeps the prefill's scratch in
// one fixed device array, compiled into the library.  Every GPU that loads
// the library holds the array until the process exits.  The caller still
// passes inputs and outputs; only the workspace comes from here.
#include <cstdio>
#include <mutex>

#include "kda_params.cuh"

namespace {

// Largest workspace the fixed scratch serves: 64 MiB per device.
constexpr size_t kNoallocScratchBytes = size_t(64) << 20;

// The scratch itself.  In host code this name is only a host-side stand-in
// for the symbol, not a device address: the address a kernel needs comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_chunk_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[64] = {nullptr};  // resolved device address, per device

// Resolve the scratch address for the current device once.  The first call
// on a device does this set-up, so that first call should come before any
// stream capture.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    kda::set_last_error(KDA_ERR_CUDA, "kda_chunk_fwd_noalloc: cudaGetDevice failed");
    return KDA_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) {
    kda::set_last_error(KDA_ERR_INVALID_ARGUMENT, "kda_chunk_fwd_noalloc: device index beyond 63");
    return KDA_ERR_INVALID_ARGUMENT;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_chunk_scratch);
    if (e != cudaSuccess || p == nullptr) {
      kda::set_last_error(KDA_ERR_CUDA,
                          "kda_chunk_fwd_noalloc: cudaGetSymbolAddress of the scratch failed");
      return KDA_ERR_CUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return KDA_OK;
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const kda_activations* x, void* out,
                                     const int32_t* cu_seqlens, int32_t n_seqs,
                                     const void* initial_state, void* final_state,
                                     void* state_cache, int64_t slot_stride, int64_t n_slots,
                                     const int32_t* state_indices,
                                     const uint8_t* has_initial_state, int32_t groups,
                                     void* stream) {
  if (!x) {
    kda::set_last_error(KDA_ERR_INVALID_ARGUMENT, "activations must not be NULL.");
    return KDA_ERR_INVALID_ARGUMENT;
  }
  const size_t need = kda_chunk_workspace_bytes(n_seqs, x->t_total, x->hv, groups);
  if (need == 0)  // invalid sizes: let the full validation report which rule broke
    return kda_chunk_fwd(x, out, cu_seqlens, n_seqs, initial_state, final_state, state_cache,
                         slot_stride, n_slots, state_indices, has_initial_state, groups, nullptr,
                         0, stream);
  if (need > kNoallocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "kda_chunk_fwd_noalloc needs %zu bytes of scratch for this call; its fixed "
             "scratch holds %zu bytes (64 MiB). Use kda_chunk_fwd with a workspace.",
             need, kNoallocScratchBytes);
    kda::set_last_error(KDA_ERR_INVALID_ARGUMENT, msg);
    return KDA_ERR_INVALID_ARGUMENT;
  }
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != KDA_OK) return rc;
  // The prefill needs no part of its workspace to start at zero: every word
  // its kernels read is written earlier in the same call (chunk table, then
  // per-chunk operands, then group planes).  So the last call's contents may
  // stay.  Calls that overlap on the GPU share this one array and race.
  return kda_chunk_fwd(x, out, cu_seqlens, n_seqs, initial_state, final_state, state_cache,
                       slot_stride, n_slots, state_indices, has_initial_state, groups, scratch,
                       kNoallocScratchBytes, stream);
}
