// Tensor-core form of the backward's state stage (K = V = 128, chunk 64): the state before
// every chunk and V_new, recomputed chunk after chunk as in "Reading Notes: Implementation
// Notes for KDA in FLA", backward-propagation step 2 (the forward's step 4 rerun):
//   V_new = U - W S,   S <- Diag(e^gamma_C) S + Kg^T V_new.
// One CTA per (sequence, value head) holds all V = 128 columns, in transposed form so that
// the MMA M dimension is v (as the forward's recurrence kernel):
//   V_new^T = U^T + S^T (-W)^T            G1: 8 K-steps over the 128 channels
//   S^T    <- S^T Diag(e^gamma_C) + V_new^T Kg   G2: 4 K-steps over the 64 tokens
// with S^T in tensor memory in fp32.  The gradients need fp32-accurate states, so every
// product takes both operands as bf16 high and low parts (x = hi + lo to ~2^-16) and
// accumulates hi*hi + hi*lo + lo*hi in fp32: three MMAs per K-step.  -W and Kg^T come as
// hi / lo tiles written by the recompute stage (kTileNegW, kTileKgT), U and e^gamma_C from
// the workspace block; the A operands (S^T, V_new^T hi / lo) are written to tensor memory by
// the epilogue warps.  Warps 0-15: epilogue (thread v = 32 q + lane of TMEM lane quadrant
// q = warp % 4 owns row v; the four warps of a quadrant split the columns); warp 16: one
// thread issues the MMAs; warp 17: one thread issues the bulk copies.  Every wait is bounded
// and reports KDA_DEV_TIMEOUT through the status word.

#include <stdint.h>

#include "kda_bwd.cuh"
#include "kda_internal.cuh"
#include "tc_common.cuh"

namespace kda {
namespace bwd {
namespace {

using namespace tc;

// shared memory: two chunk slots, each [tiles 64 KB | U fp32 [64][128] 32 KB | e^gamma_C 512 B]
constexpr uint32_t SS_TILES = 0;
constexpr uint32_t SS_U = 65536;
constexpr uint32_t SS_D = 98304;
constexpr uint32_t SS_BYTES = 98304 + 512;
constexpr uint32_t SS_SLOT = 99328;                  // 1024-byte multiple
constexpr uint32_t SS_BAR = 2 * SS_SLOT;             // full[2], freed[2], bar_v, bar_s, bar_vn, bar_st
constexpr uint32_t SS_TMEM = SS_BAR + 64;
constexpr uint32_t SS_SMEM = SS_TMEM + 16 + 1024;    // + alignment slack
// tensor-memory columns
constexpr uint32_t TS_VN = 0;     // V_new^T fp32 [128 v x 64 tokens]
constexpr uint32_t TS_S = 64;     // S^T fp32 [128 v x 128 channels]
constexpr uint32_t TS_SA = 192;   // S^T bf16 pairs: hi 192..255, lo 256..319
constexpr uint32_t TS_VA = 320;   // V_new^T bf16 pairs: hi 320..351, lo 352..383
constexpr int kEpi = 16;          // epilogue warps
constexpr int kStThreads = 32 * kEpi + 64;

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}
// hi / lo bf16 pair words of x0, x1 (hi = x rounded, lo = x - hi rounded)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
  lo = pack_bf16x2(x0 - h0, x1 - h1);
}

__global__ void __launch_bounds__(kStThreads, 1) states_tc_kernel(const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  const Plan& p = a.p;
  const int HV = p.HV, V = p.V, K = p.K;
  const int hv = (int)(blockIdx.x % HV);
  const int n = (int)(blockIdx.x / HV);
  int64_t bos, eos, cfirst;
  if (!seq_range(a, n, bos, eos, cfirst)) {
    if (threadIdx.x == 0) atomicOr(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const int64_t nch = (eos - bos + p.C - 1) / p.C;
  if (nch == 0) return;  // nothing recorded for an empty sequence
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + SS_BAR);
  uint64_t* freed = full + 2;
  uint64_t* bar_v = full + 4;   // G1 done: V_new^T complete
  uint64_t* bar_s = full + 5;   // G2 done: the next state complete
  uint64_t* bar_vn = full + 6;  // epilogue: V_new^T hi / lo written
  uint64_t* bar_st = full + 7;  // epilogue: S^T hi / lo, the rescaled S^T and U^T written
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + SS_TMEM);
  if (warp == kEpi) {
    tmem_alloc(sTmem, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&full[i], 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_vn, kEpi);
    mbar_init(bar_st, kEpi);
    fence_mbar_init();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  bool ok = true;
  auto slot = [&](int64_t ci) { return sm + (uint32_t)(ci & 1) * SS_SLOT; };
  auto par = [](int64_t ci) { return (uint32_t)((ci >> 1) & 1); };

  if (warp == kEpi + 1) {
    // ------------------------------- copy warp ---------------------------------------
    if (lane == 0) {
      auto issue = [&](int64_t ci) {  // chunk ci -> its slot: tiles, U, e^gamma_C
        const int64_t c = cfirst + ci;
        uint8_t* dst = slot(ci);
        const float* blk = block_ptr(a, c, hv);
        mbar_arrive_expect_tx(&full[ci & 1], SS_BYTES);
        bulk_g2s(dst + SS_TILES, tile_ptr(a, c, hv), (uint32_t)kTileBytes, &full[ci & 1]);
        bulk_g2s(dst + SS_U, blk + p.blk.u, 32768u, &full[ci & 1]);
        bulk_g2s(dst + SS_D, blk + p.blk.decay, 512u, &full[ci & 1]);
      };
      int64_t issued = 0;
      issue(0);
      issued = 1;
      if (nch > 1) {
        issue(1);
        issued = 2;
      }
      for (int64_t ci = 0; ci + 2 < nch; ++ci) {  // chunk ci + 2 once G2 of chunk ci is done
        if (!mbar_wait(&freed[ci & 1], par(ci))) { ok = false; break; }
        issue(ci + 2);
        issued = ci + 3;
      }
      if (!ok) {
        atomicOr(a.status, KDA_DEV_TIMEOUT);
        for (int64_t c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
          mbar_wait(&full[c & 1], par(c), 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kEpi) {
    // -------------------------------- MMA warp ---------------------------------------
    if (lane == 0) {
      for (int64_t ci = 0; ci < nch && ok; ++ci) {
        const uint32_t tb = smem_u32(slot(ci) + SS_TILES);
        const uint32_t w_hi = tb + (uint32_t)kTileNegW, w_lo = w_hi + (uint32_t)kTileLo;
        const uint32_t k_hi = tb + (uint32_t)kTileKgT, k_lo = k_hi + (uint32_t)kTileLo;
        if (!mbar_wait(&full[ci & 1], par(ci))) { ok = false; break; }
        // G1 needs S^T hi / lo, the rescaled S^T and U^T of this chunk
        if (!mbar_wait_spin(bar_st, (uint32_t)(ci & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks) {  // channels 16 ks .. 16 ks + 15
          const uint32_t boff = (uint32_t)(ks >> 2) * 8192u + (uint32_t)(ks & 3) * 32u;
          const uint32_t idesc = idesc_bf16(128, 64);
          mma_bf16_ts(tmem + TS_VN, tmem + TS_SA + 8 * ks, sdesc_sw128(w_hi + boff, 16, 1024), idesc, 1);
          mma_bf16_ts(tmem + TS_VN, tmem + TS_SA + 8 * ks, sdesc_sw128(w_lo + boff, 16, 1024), idesc, 1);
          mma_bf16_ts(tmem + TS_VN, tmem + TS_SA + 64 + 8 * ks, sdesc_sw128(w_hi + boff, 16, 1024), idesc, 1);
        }
        mma_commit(bar_v);
        // G2 needs V_new^T hi / lo
        if (!mbar_wait_spin(bar_vn, (uint32_t)(ci & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {  // tokens 16 ks .. 16 ks + 15
          const uint32_t boff = (uint32_t)ks * 32u;
          const uint32_t idesc = idesc_bf16(128, 128);
          mma_bf16_ts(tmem + TS_S, tmem + TS_VA + 8 * ks, sdesc_sw128(k_hi + boff, 16, 1024), idesc, 1);
          mma_bf16_ts(tmem + TS_S, tmem + TS_VA + 8 * ks, sdesc_sw128(k_lo + boff, 16, 1024), idesc, 1);
          mma_bf16_ts(tmem + TS_S, tmem + TS_VA + 32 + 8 * ks, sdesc_sw128(k_hi + boff, 16, 1024), idesc, 1);
        }
        mma_commit(bar_s);
        mma_commit(&freed[ci & 1]);  // the slot's last reader
      }
      if (!ok) atomicOr(a.status, KDA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue warps -------------------------------------
    const int q4 = warp & 3, part = warp >> 2;  // part: channels 32 part ..; tokens 16 part ..
    const int v = 32 * q4 + lane;
    const uint32_t lb = tmem_addr(tmem, 32 * q4, 0);
    auto arrive = [&](uint64_t* bar) {  // one arrival per warp, after the warp's writes
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    float S[32];  // S^T[v][32 part + j]: this thread's part of the state before the chunk
    {
      const size_t sbase = ((size_t)n * HV + hv) * (size_t)K * V;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int k = 32 * part + j;
        S[j] = a.h0 == nullptr ? 0.f
                               : a.h0[sbase + (a.state_v_first ? (size_t)v * K + k : (size_t)k * V + v)];
      }
    }
    // U^T of chunk ci into the V_new^T accumulator (G1 adds S^T (-W)^T to it)
    auto write_u = [&](int64_t ci) -> bool {
      const bool w = mbar_wait(&full[ci & 1], par(ci));
      const float* u = reinterpret_cast<const float*>(slot(ci) + SS_U);
      uint32_t r[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(u[(16 * part + x) * 128 + v]);
      tmem_st16(lb + TS_VN + 16 * part, r);
      return w;
    };
    // S^T of chunk ci as hi / lo A operands, S^T Diag(e^gamma_C) into the accumulator; then
    // G1 of chunk ci may start (its U^T was written before)
    auto publish = [&](int64_t ci) -> bool {
      const bool w = mbar_wait(&full[ci & 1], par(ci));
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) split2(S[2 * j], S[2 * j + 1], hi[j], lo[j]);
      tmem_st16(lb + TS_SA + 16 * part, hi);
      tmem_st16(lb + TS_SA + 64 + 16 * part, lo);
      const float* d = reinterpret_cast<const float*>(slot(ci) + SS_D) + 32 * part;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sc[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) sc[x] = __float_as_uint(S[16 * h + x] * d[16 * h + x]);
        tmem_st16(lb + TS_S + 32 * part + 16 * h, sc);
      }
      tmem_wait_st();
      tc_fence_before();
      arrive(bar_st);
      return w;
    };
    auto store_state = [&](int64_t ci) {  // the state before chunk ci, [K][V] in the workspace
      float* hs = state_ptr(a, p.off_h, cfirst + ci, hv);
#pragma unroll
      for (int j = 0; j < 32; ++j) hs[(size_t)(32 * part + j) * V + v] = S[j];
    };
    ok = write_u(0) && ok;
    ok = publish(0) && ok;
    store_state(0);
    for (int64_t ci = 0; ci < nch && ok; ++ci) {
      // V_new^T of chunk ci -> hi / lo A operands of G2; out to the workspace
      bool w = mbar_wait(&bar_v[0], (uint32_t)(ci & 1));
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(lb + TS_VN + 16 * part, r);
      tmem_wait_ld();
      {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          split2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]), hi[j], lo[j]);
        tmem_st8(lb + TS_VA + 8 * part, hi);
        tmem_st8(lb + TS_VA + 32 + 8 * part, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      arrive(bar_vn);
      {
        float* vn = block_ptr(a, cfirst + ci, hv) + p.blk.vn;
#pragma unroll
        for (int x = 0; x < 16; ++x) vn[(size_t)(16 * part + x) * V + v] = __uint_as_float(r[x]);
      }
      if (ci + 1 < nch) w = write_u(ci + 1) && w;  // G1 of chunk ci is done with the accumulator
      // the state after chunk ci
      w = mbar_wait(&bar_s[0], (uint32_t)(ci & 1)) && w;
      tc_fence_after();
      {
        uint32_t r0[16], r1[16];
        tmem_ld16(lb + TS_S + 32 * part, r0);
        tmem_ld16(lb + TS_S + 32 * part + 16, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          S[j] = __uint_as_float(r0[j]);
          S[16 + j] = __uint_as_float(r1[j]);
        }
      }
      if (ci + 1 < nch) {
        w = publish(ci + 1) && w;
        store_state(ci + 1);
      }
      if (!w) ok = false;
    }
    if (!ok) atomicOr(a.status, KDA_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kEpi) tmem_dealloc(tmem, 512);
}

}  // namespace

// The state stage on the tensor cores: one CTA per (sequence, value head).
cudaError_t run_states_tc(const Args& a, cudaStream_t st) {
  const unsigned grid = (unsigned)((int64_t)a.p.N * a.p.HV);
  if (grid == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(states_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SS_SMEM);
  if (e != cudaSuccess) return e;
  states_tc_kernel<<<grid, kStThreads, SS_SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace bwd
}  // namespace kda
