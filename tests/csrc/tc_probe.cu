// Test-only probe of the tcgen05 primitives in tc_common.cuh: one CTA places bf16
// A [M x K] and B [N x K] in shared memory (K-major or MN-major, 128-byte swizzle),
// runs D = (+/-)A * B^T as a chain of K/16 tcgen05.mma, and dumps all 128 TMEM lanes
// x N columns.  The host side is plain test scaffolding (it allocates freely).
#include <cuda_bf16.h>
#include <stdint.h>
#include <stdio.h>

#include "tc_common.cuh"

using namespace kda::tc;

struct ProbeArgs {
  int M, N, K, a_mn, b_mn, neg_a, a_tmem;  // a_tmem: A read from tensor memory
  const uint16_t* A;  // logical [M][K]
  const uint16_t* B;  // logical [N][K]
  float* out;         // [128][N]
  int* err;
};

__device__ uint32_t operand_offset(int mn_major, int rows, int K, int r, int k) {
  // K-major: panels of 64 K-columns, each panel holds all `rows` rows.
  // MN-major: panels of 64 rows (MN elements), each panel holds all K rows.
  if (!mn_major) return (uint32_t)(k / 64) * (uint32_t)(rows * 128) + sw128_offset(r, k % 64);
  return (uint32_t)(r / 64) * (uint32_t)(K * 128) + sw128_offset(k, r % 64);
}

__global__ void __launch_bounds__(128) tc_probe_kernel(ProbeArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;          // 32 KB
  unsigned char* sB = smem + 32768;  // 64 KB
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < a.M * a.K; i += blockDim.x) {
    const int m = i / a.K, k = i % a.K;
    *(uint16_t*)(sA + operand_offset(a.a_mn, a.M, a.K, m, k)) = a.A[i];
  }
  for (int i = tid; i < a.N * a.K; i += blockDim.x) {
    const int n = i / a.K, k = i % a.K;
    *(uint16_t*)(sB + operand_offset(a.b_mn, a.N, a.K, n, k)) = a.B[i];
  }
  fence_async_smem();
  if (warp == 0) {
    tmem_alloc(&tbase, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  if (a.a_tmem) {  // row m of A -> lane m, columns 256 + k/2 (bf16 pairs, lower k low)
    const int m = 32 * warp + lane;
    for (int k0 = 0; k0 < a.K; k0 += 16) {
      uint32_t r[8];
      for (int j = 0; j < 8; ++j) {
        const int k = k0 + 2 * j;
        const uint32_t lo = m < a.M ? a.A[m * a.K + k] : 0u, hi = m < a.M ? a.A[m * a.K + k + 1] : 0u;
        r[j] = lo | (hi << 16);
      }
      tmem_st8(tmem_addr(tmem, 32 * warp, 256 + k0 / 2), r);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16(a.M, a.N, a.a_mn, a.b_mn, a.neg_a);
    for (int ks = 0; ks < a.K / 16; ++ks) {
      uint64_t ad, bd;
      if (!a.a_mn)
        ad = sdesc_sw128(smem_u32(sA) + (ks / 4) * (a.M * 128) + (ks % 4) * 32, 16, 1024);
      else
        ad = sdesc_sw128(smem_u32(sA) + ks * 2048, a.K * 128, 1024);
      if (!a.b_mn)
        bd = sdesc_sw128(smem_u32(sB) + (ks / 4) * (a.N * 128) + (ks % 4) * 32, 16, 1024);
      else
        bd = sdesc_sw128(smem_u32(sB) + ks * 2048, a.K * 128, 1024);
      if (a.a_tmem)
        mma_bf16_ts(tmem, tmem + 256 + ks * 8, bd, idesc, ks > 0);
      else
        mma_bf16(tmem, ad, bd, idesc, ks > 0);
    }
    mma_commit(&bar);
  }
  __syncwarp();
  bool ok = mbar_wait(&bar, 0, 1000000000ull);
  tc_fence_after();
  if (!ok) {
    if (lane == 0) atomicExch(a.err, 1);
  } else {
    for (int c = 0; c < a.N; c += 16) {
      uint32_t r[16];
      tmem_ld16(tmem_addr(tmem, 32 * warp, c), r);
      tmem_wait_ld();
      for (int j = 0; j < 16; ++j) a.out[(32 * warp + lane) * a.N + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

extern "C" int tc_probe_run(int M, int N, int K, int a_mn, int b_mn, int neg_a, int a_tmem,
                            const uint16_t* hA, const uint16_t* hB, float* hOut) {
  if (M > 128 || N > 256 || K > 128 || K % 16 || (a_mn && M % 64) || (b_mn && N % 64 && N != 32) ||
      (a_tmem && (M != 128 || a_mn)))
    return -1;
  uint16_t *dA, *dB;
  float* dO;
  int* dE;
  cudaMalloc(&dA, M * K * 2);
  cudaMalloc(&dB, N * K * 2);
  cudaMalloc(&dO, 128 * N * 4);
  cudaMalloc(&dE, 4);
  cudaMemcpy(dA, hA, M * K * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dB, hB, N * K * 2, cudaMemcpyHostToDevice);
  cudaMemset(dO, 0, 128 * N * 4);
  cudaMemset(dE, 0, 4);
  ProbeArgs a{M, N, K, a_mn, b_mn, neg_a, a_tmem, dA, dB, dO, dE};
  const int smem = 1024 + 32768 + 65536;
  cudaFuncSetAttribute(tc_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  tc_probe_kernel<<<1, 128, smem>>>(a);
  cudaError_t e = cudaDeviceSynchronize();
  int err = 0;
  cudaMemcpy(&err, dE, 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(hOut, dO, 128 * N * 4, cudaMemcpyDeviceToHost);
  cudaFree(dA); cudaFree(dB); cudaFree(dO); cudaFree(dE);
  if (e != cudaSuccess) {
    fprintf(stderr, "probe: %s\n", cudaGetErrorString(e));
    return -2;
  }
  return err ? -3 : 0;
}
