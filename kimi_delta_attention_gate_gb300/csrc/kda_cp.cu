// Affine state maps for context parallelism: S_out = P S_in + R per map (fp32).
//
// A shard of tokens acts on the state entering it as an affine map ("Reading Notes:
// Implementation Notes for KDA in FLA", forward step 4, is affine in the state); the
// ranks of a sequence-sharded pass chain those maps.  One CTA per (map, 32-column tile of
// V): the S_in tile is staged in shared memory, each warp owns rows of P and every lane one
// column of the tile.
#include <stdio.h>

#include "kda_cp.h"
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kCpThreads = 256;
constexpr int kCpTile = 32;

__global__ void __launch_bounds__(kCpThreads)
    state_affine_kernel(const float* __restrict__ P, const float* __restrict__ R,
                        const float* __restrict__ S_in, float* __restrict__ S_out, int K, int V,
                        int v_first) {
  __shared__ float tile[kMaxK][kCpTile + 1];  // S_in[j][v0 + c]
  const int64_t i = blockIdx.x;
  const int v0 = blockIdx.y * kCpTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t st = (size_t)K * V;
  // element (row j of K, column v of V) of a state stored [K][V], or [V][K] when v_first
  auto at = [&](int j, int v) -> size_t {
    return v_first ? (size_t)v * K + j : (size_t)j * V + v;
  };
  for (int e = tid; e < K * kCpTile; e += kCpThreads) {
    // [K][V]: consecutive threads take consecutive columns; [V][K]: consecutive rows
    const int j = v_first ? e % K : e / kCpTile, c = v_first ? e / K : e % kCpTile;
    const int v = v0 + c;
    tile[j][c] = (S_in != nullptr && v < V) ? S_in[i * st + at(j, v)] : 0.f;
  }
  __syncthreads();
  const int v = v0 + lane;
  const float* Pi = P + i * (size_t)K * K;
  for (int k = warp; k < K; k += kCpThreads / 32) {
    float acc = 0.f;
    const float* prow = Pi + (size_t)k * K;
    for (int j = 0; j < K; ++j) acc = fmaf(__ldg(prow + j), tile[j][lane], acc);
    if (v < V) {
      const size_t o = i * st + at(k, v);
      S_out[o] = acc + R[o];
    }
  }
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace kda

extern "C" kda_status kda_state_affine_apply(const float* P, const float* R, const float* S_in,
                                             float* S_out, int64_t nmaps, int32_t K, int32_t V,
                                             int32_t state_v_first, void* stream) {
  using namespace kda;
  char buf[256];
  if (K < 1 || K > kMaxK || V < 1 || V > kMaxV || nmaps < 0) {
    snprintf(buf, sizeof(buf), "kda_state_affine_apply: need 1 <= K, V <= 256 and nmaps >= 0 "
             "(got K=%d, V=%d, nmaps=%lld)", K, V, (long long)nmaps);
    set_last_error(buf);
    return KDA_ERR_SHAPE;
  }
  if (state_v_first != 0 && state_v_first != 1) {
    set_last_error("kda_state_affine_apply: state_v_first must be 0 or 1");
    return KDA_ERR_INVALID_ARG;
  }
  if (nmaps == 0) {
    set_last_error("");
    return KDA_OK;
  }
  if (P == nullptr || R == nullptr || S_out == nullptr || !aligned4(P) || !aligned4(R) ||
      !aligned4(S_out) || (S_in != nullptr && !aligned4(S_in))) {
    set_last_error("kda_state_affine_apply: P, R and S_out are required and every pointer "
                   "must be 4-byte aligned");
    return KDA_ERR_INVALID_ARG;
  }
  if ((const void*)S_out == (const void*)P || (const void*)S_out == (const void*)R ||
      (const void*)S_out == (const void*)S_in) {
    set_last_error("kda_state_affine_apply: S_out must not alias P, R or S_in");
    return KDA_ERR_INVALID_ARG;
  }
  if (nmaps > 0x7fffffffLL) {
    set_last_error("kda_state_affine_apply: nmaps must fit in 31 bits");
    return KDA_ERR_SHAPE;
  }
  const dim3 grid((unsigned)nmaps, (unsigned)((V + kCpTile - 1) / kCpTile));
  state_affine_kernel<<<grid, kCpThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      P, R, S_in, S_out, K, V, state_v_first);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(buf, sizeof(buf), "kda_state_affine_apply: launch failed: %s", cudaGetErrorString(e));
    set_last_error(buf);
    return KDA_ERR_CUDA;
  }
  set_last_error("");
  return KDA_OK;
}
