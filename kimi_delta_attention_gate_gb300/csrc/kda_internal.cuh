// Internal declarations shared by the host layer and the kernels of the GB300 KDA library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kMaxK = 256;
constexpr int kMaxV = 256;

// Resolved launch plan: how tokens map to sequences and chunks, and where each
// intermediate lives in the caller's workspace.
struct Plan {
  int B, T, H, HV, K, V, C, N, G;
  int64_t ntok;             // B * T (flattened token axis)
  int64_t tok_end;          // one past the last token any sequence covers (cu_seqlens[N] with
                            // varlen, else ntok); rows [tok_end, ntok) of o are set to zero
  int64_t nct;              // total chunks over all sequences
  int nc_per_seq;           // chunks per sequence when there is no cu_seqlens
  bool varlen;
  size_t off_chunk_table;   // int64 [N + 1] chunk offsets (varlen only)
  size_t off_inter;         // per chunk-head intermediates
  size_t inter_block_bytes; // bytes per (chunk, value head)
  bool tensor_core;         // bf16 tensor-core kernels (else the fp32 CUDA-core kernels)
  int nseg;                 // chunk-range segments of the pipelined tensor-core schedule
  size_t off_state;         // fp32 [N][HV][K][V] states carried between segments (nseg > 1)
  size_t total_bytes;
};

// Arguments every kernel of the forward pass receives (by value).
struct FwdArgs {
  Plan plan;
  int dtype, gate_mode, qk_l2norm, beta_sigmoid, allow_neg_eigval, state_v_first;
  float lower_bound, scale;
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const float* A_log;
  const float* dt_bias;
  const float* h0;
  const int64_t* cu_seqlens;
  void* o;
  float* final_state;
  float* h_out;             // per-chunk states (optional)
  char* ws;                 // workspace base
  unsigned int* status;     // device status word
  int64_t c_begin, c_end;   // global chunk range of this launch (tensor-core kernels)
};

// ---------------------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float sigmoid_exact(float x) { return 1.0f / (1.0f + expf(-x)); }

// log(1 + e^x); above 20 the correction log1p(e^-x) < 2.1e-9 is below fp32 resolution of x.
__device__ __forceinline__ float softplus_exact(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

// Activated log-decay gate of one element ("FLA-KDA engineering notes", section 2):
//   PLAIN  -exp(A_log) softplus(x)     SAFE  lower_bound sigmoid(exp(A_log) x)
// with x = g + dt_bias; `a` is exp(A_log) (1 when A_log is absent in SAFE mode).
__device__ __forceinline__ float gate_exact(int mode, float graw, float a, float dt, float lb) {
  const float x = graw + dt;
  if (mode == KDA_GATE_PLAIN) return -a * softplus_exact(x);
  if (mode == KDA_GATE_SAFE) return lb * sigmoid_exact(a * x);
  return graw;
}

__device__ __forceinline__ void flag_status(unsigned int* status, unsigned int bits) {
  atomicOr(status, bits);
}

// Sequence and position of global chunk `c`.  Returns false (and flags the status
// word) if the device-side sequence table is inconsistent with the plan.
__device__ __forceinline__ bool locate_chunk(const FwdArgs& a, int64_t c, int& n, int64_t& t0,
                                             int& L) {
  const Plan& p = a.plan;
  int64_t bos, eos, ci;
  if (!p.varlen) {
    n = (int)((uint32_t)c / (uint32_t)p.nc_per_seq);  // chunk indexes fit in 32 bits
    ci = c - (int64_t)n * p.nc_per_seq;
    bos = (int64_t)n * p.T;
    eos = bos + p.T;
  } else {
    const int64_t* cs = reinterpret_cast<const int64_t*>(a.ws + p.off_chunk_table);
    int lo = 0, hi = p.N;  // find n with cs[n] <= c < cs[n+1]
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (cs[mid] <= c) lo = mid; else hi = mid;
    }
    n = lo;
    ci = c - cs[n];
    bos = a.cu_seqlens[n];
    eos = a.cu_seqlens[n + 1];
  }
  t0 = bos + ci * p.C;
  int64_t len = eos - t0;
  if (ci < 0 || t0 < 0 || len <= 0 || eos > p.ntok) {
    flag_status(a.status, KDA_DEV_BAD_SEQLENS);
    return false;
  }
  L = (int)(len < p.C ? len : p.C);
  return true;
}

// Token range of sequence n; false (flagged) if inconsistent.
__device__ __forceinline__ bool seq_range(const FwdArgs& a, int n, int64_t& bos, int64_t& eos,
                                         int64_t& c_first) {
  const Plan& p = a.plan;
  if (!p.varlen) {
    bos = (int64_t)n * p.T;
    eos = bos + p.T;
    c_first = (int64_t)n * p.nc_per_seq;
    return true;
  }
  bos = a.cu_seqlens[n];
  eos = a.cu_seqlens[n + 1];
  c_first = reinterpret_cast<const int64_t*>(a.ws + p.off_chunk_table)[n];
  if (bos < 0 || eos < bos || eos > p.ntok || c_first < 0 ||
      c_first + (eos - bos + p.C - 1) / p.C > p.nct) {
    flag_status(a.status, KDA_DEV_BAD_SEQLENS);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------------------------------
// Launchers (each returns the cudaError_t of its launch)
// ---------------------------------------------------------------------------------------
// Sets the message kda_last_error() returns on the calling thread.
void set_last_error(const char* msg);

// Sets rows [tok_end, ntok) of o to zero (cudaMemsetAsync; no-op without such rows).
cudaError_t zero_uncovered_rows(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_chunk_table(const FwdArgs& a, cudaStream_t s);
size_t simt_inter_block_bytes(int C, int K, int V);
cudaError_t launch_simt_intra(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_simt_recur(const FwdArgs& a, cudaStream_t s);

// token-recurrent forward (decode / short prefill)
size_t recurrent_smem_bytes(int K);
cudaError_t launch_recurrent(const FwdArgs& a, cudaStream_t s);

// bf16 tensor-core path (K = V = 128, chunk 64)
bool tc_eligible(const Plan& p, int dtype);
size_t tc_inter_block_bytes();
cudaError_t launch_tc_intra(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_tc_recur(const FwdArgs& a, cudaStream_t s);

}  // namespace kda
