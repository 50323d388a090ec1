// kda_fwd_noalloc: the forward pass with its scratch in a static device array.
//
// For callers that cannot allocate device memory (no cudaMalloc, no allocator
// handle to hand the library a workspace).  The scratch that kda_fwd normally
// takes from the caller's workspace lives here instead, in one file-scope
// __device__ array of KDA_NOALLOC_SCRATCH_BYTES bytes; every GPU that loads
// the library holds it until the process exits.  Nothing in this file
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.

#include <stdio.h>

#include <mutex>

#include "kda_internal.cuh"

namespace {

// The static scratch.  In host code this name is only a host-side stand-in for
// the symbol, not a device address: the address kernels need comes from
// cudaGetSymbolAddress, looked up once per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};

// Device address of the scratch on the current device (looked up on the first
// call per device, with that device current).  Returns nullptr on failure and
// leaves a message for kda_last_error().
void* scratch_address() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    kda::set_last_error("kda_fwd_noalloc: no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      char buf[256];
      snprintf(buf, sizeof(buf), "kda_fwd_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      kda::set_last_error(buf);
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" kda_status kda_fwd_noalloc(const kda_fwd_params* p, void* stream) {
  kda_status s = kda_fwd_check(p);
  if (s != KDA_OK) return s;
  const size_t need = kda_fwd_workspace_size(p);
  if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "kda_fwd_noalloc: these sizes need %zu bytes of scratch, the static scratch holds %zu "
             "(use kda_fwd with a caller-provided workspace)",
             need, (size_t)KDA_NOALLOC_SCRATCH_BYTES);
    kda::set_last_error(buf);
    return KDA_ERR_WORKSPACE;
  }
  void* ptr = scratch_address();
  if (ptr == nullptr) return KDA_ERR_CUDA;
  // Same pass as kda_fwd, with the workspace replaced, run stage after stage on the
  // caller's stream (bit-identical to kda_fwd's schedule).  Running the stages in series
  // keeps this entry point free of the library's internal streams and events, so that its
  // only first-use set-up is the address lookup above.  Every scratch element a kernel reads
  // is written earlier in the same call, so nothing needs clearing.
  kda_fwd_params q = *p;
  q.workspace = ptr;
  q.workspace_bytes = KDA_NOALLOC_SCRATCH_BYTES;
  const int32_t nst = kda_fwd_num_stages(&q);
  for (int32_t i = 0; i < nst; ++i) {
    s = kda_fwd_stage(&q, stream, i);
    if (s != KDA_OK) return s;
  }
  return KDA_OK;
}
