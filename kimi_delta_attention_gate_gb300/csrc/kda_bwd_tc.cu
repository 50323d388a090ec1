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

#include <cudaTypedefs.h>
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

// ======================================================================================
// The state-gradient stage (backward-propagation steps 3-4) on the tensor cores, chunks in
// reverse, with dS' (the gradient of the state after the chunk) in tensor memory:
//   dV_new^T = dO^T Aqk + dS'^T Kg^T                      -> dV_new
//   dS^T     = dS'^T Diag(e^gamma_C) + dO^T Qg + dV_new^T (-W)   (the next chunk's dS')
// dO (bf16 input, exact) is the MN-major A operand of the two products that do not depend
// on the chain, loaded by TMA; the chain's A operands (dS'^T, dV_new^T) are hi / lo pairs in
// tensor memory; B operands are the hi / lo tiles (-W and Kg^T read as MN-major operands,
// Aqk and Qg written for this stage).  Shared memory: the dO / Aqk / e^gamma_C part of a
// chunk is double-buffered; Kg^T and the Qg / -W pair are single-buffered and refilled as
// soon as the chunk's G1 (Kg^T) or G2 (Qg, -W) has read them.
// ======================================================================================
constexpr uint32_t DA_DO = 0;          // dO tile [64 tokens x 128 v] bf16, two MN panels
constexpr uint32_t DA_AQK = 16384;     // Aqk hi, lo (8 KB each)
constexpr uint32_t DA_D = 32768;       // e^gamma_C fp32 [128]
constexpr uint32_t DA_BYTES = 32768 + 512;
constexpr uint32_t DA_SLOT = 33792;
constexpr uint32_t DS_KG = 2 * DA_SLOT;        // Kg^T hi, lo (16 KB each)
constexpr uint32_t DS_QW = DS_KG + 32768;      // Qg hi, lo, then -W hi, lo (16 KB each)
constexpr uint32_t DS_BAR = DS_QW + 65536;     // 12 barriers
constexpr uint32_t DS_TMEM = DS_BAR + 96;
constexpr uint32_t DS_SMEM = DS_TMEM + 16 + 1024;
constexpr uint32_t TD_DV = 0;     // dV_new^T fp32 [128 v x 64 tokens]
constexpr uint32_t TD_DS = 64;    // dS^T fp32 [128 v x 128 channels]
constexpr uint32_t TD_DSA = 192;  // dS'^T bf16 pairs: hi 192..255, lo 256..319
constexpr uint32_t TD_DVA = 320;  // dV_new^T bf16 pairs: hi 320..351, lo 352..383

__global__ void __launch_bounds__(kStThreads, 1)
    dstate_tc_kernel(const Args a, const __grid_constant__ CUtensorMap domap) {
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
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t sbase = ((size_t)n * HV + hv) * (size_t)K * V;
  if (nch == 0) {  // an empty sequence: dh0 is the incoming gradient itself
    if (a.dh0 != nullptr)
      for (int e = tid; e < K * V; e += blockDim.x)
        a.dh0[sbase + e] = a.d_final_state != nullptr ? a.d_final_state[sbase + e] : 0.f;
    return;
  }
  uint64_t* fullA = reinterpret_cast<uint64_t*>(sm + DS_BAR);  // [2]
  uint64_t* freedA = fullA + 2;                               // [2]
  uint64_t* fullKG = fullA + 4;
  uint64_t* freedKG = fullA + 5;
  uint64_t* fullQW = fullA + 6;
  uint64_t* freedQW = fullA + 7;
  uint64_t* bar_dv = fullA + 8;    // G1 done: dV_new^T complete
  uint64_t* bar_ds = fullA + 9;    // G2 done: the next dS'^T complete
  uint64_t* bar_dvn = fullA + 10;  // epilogue: dV_new^T hi / lo written
  uint64_t* bar_st = fullA + 11;   // epilogue: dS'^T hi / lo and dS'^T e^gamma_C written
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + DS_TMEM);
  if (warp == kEpi) {
    tmem_alloc(sTmem, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&fullA[i], 1);
    mbar_init(bar_dv, 1);
    mbar_init(bar_ds, 1);
    mbar_init(bar_dvn, kEpi);
    mbar_init(bar_st, kEpi);
    fence_mbar_init();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  bool ok = true;
  // iteration it processes chunk nch - 1 - it
  auto chunk_of = [&](int64_t it) { return nch - 1 - it; };
  auto slotA = [&](int64_t it) { return sm + (uint32_t)(it & 1) * DA_SLOT; };
  auto parA = [](int64_t it) { return (uint32_t)((it >> 1) & 1); };
  auto par1 = [](int64_t it) { return (uint32_t)(it & 1); };

  if (warp == kEpi + 1) {
    // ------------------------------- copy warp ---------------------------------------
    if (lane == 0) {
      const CUtensorMap* dmap = &domap;
      auto issueA = [&](int64_t it) {  // dO tile, Aqk hi / lo, e^gamma_C of iteration it
        const int64_t cl = chunk_of(it), c = cfirst + cl;
        uint8_t* dst = slotA(it);
        mbar_arrive_expect_tx(&fullA[it & 1], DA_BYTES);
        const int32_t t0 = (int32_t)(bos + cl * p.C);
        tma_load_3d(dst + DA_DO, dmap, 0, hv, t0, &fullA[it & 1]);
        tma_load_3d(dst + DA_DO + 8192, dmap, 64, hv, t0, &fullA[it & 1]);
        bulk_g2s(dst + DA_AQK, tile_ptr(a, c, hv) + kTileAqk, 16384u, &fullA[it & 1]);
        bulk_g2s(dst + DA_D, block_ptr(a, c, hv) + p.blk.decay, 512u, &fullA[it & 1]);
      };
      auto issueKG = [&](int64_t it) {
        mbar_arrive_expect_tx(fullKG, 32768u);
        bulk_g2s(sm + DS_KG, tile_ptr(a, cfirst + chunk_of(it), hv) + kTileKgT, 32768u, fullKG);
      };
      auto issueQW = [&](int64_t it) {
        const char* t = tile_ptr(a, cfirst + chunk_of(it), hv);
        mbar_arrive_expect_tx(fullQW, 65536u);
        bulk_g2s(sm + DS_QW, t + kTileQg, 32768u, fullQW);
        bulk_g2s(sm + DS_QW + 32768, t + kTileNegW, 32768u, fullQW);
      };
      int64_t a_issued = 1, kg_issued = 1, qw_issued = 1;
      issueA(0);
      if (nch > 1) {
        issueA(1);
        a_issued = 2;
      }
      issueKG(0);
      issueQW(0);
      for (int64_t it = 0; it + 1 < nch; ++it) {
        if (!mbar_wait(freedKG, par1(it))) { ok = false; break; }   // G1 of it has read Kg^T
        issueKG(it + 1);
        kg_issued = it + 2;
        if (!mbar_wait(freedQW, par1(it))) { ok = false; break; }   // G2 of it has read Qg, -W
        issueQW(it + 1);
        qw_issued = it + 2;
        if (it + 2 < nch) {                                          // and its dO / Aqk slot
          if (!mbar_wait(&freedA[it & 1], parA(it))) { ok = false; break; }
          issueA(it + 2);
          a_issued = it + 3;
        }
      }
      if (!ok) {
        atomicOr(a.status, KDA_DEV_TIMEOUT);
        // the copies in flight must land before the CTA's shared memory is released
        for (int64_t it = a_issued > 2 ? a_issued - 2 : 0; it < a_issued; ++it)
          mbar_wait(&fullA[it & 1], parA(it), 100000000ull);
        mbar_wait(fullKG, par1(kg_issued - 1), 100000000ull);
        mbar_wait(fullQW, par1(qw_issued - 1), 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kEpi) {
    // -------------------------------- MMA warp ---------------------------------------
    if (lane == 0) {
      const uint32_t kg_hi = smem_u32(sm + DS_KG), kg_lo = kg_hi + 16384u;
      const uint32_t qg_hi = smem_u32(sm + DS_QW), qg_lo = qg_hi + 16384u;
      const uint32_t nw_hi = qg_hi + 32768u, nw_lo = qg_hi + 49152u;
      // dO^T Aqk of iteration it into the dV_new^T accumulator (its first product): wait for
      // the slot, zero the dO rows past the chunk's end (another sequence's tokens)
      auto issue_doaqk = [&](int64_t it) -> bool {
        if (!mbar_wait(&fullA[it & 1], parA(it))) return false;
        uint8_t* sl = slotA(it);
        const int64_t t0 = bos + chunk_of(it) * p.C;
        const int L = (int)((eos - t0) < p.C ? (eos - t0) : p.C);
        if (L < p.C) {
          for (int e = L * 8; e < p.C * 8; ++e) {  // 8 16-byte pieces per 128-byte row
            *reinterpret_cast<uint4*>(sl + DA_DO + (uint32_t)e * 16u) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sl + DA_DO + 8192u + (uint32_t)e * 16u) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        }
        tc_fence_after();
        const uint32_t dob = smem_u32(sl + DA_DO), aqb = smem_u32(sl + DA_AQK);
        const uint32_t idesc = idesc_bf16(128, 64, true, true);
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {  // tokens t' 16 ks .. 16 ks + 15
          const uint64_t ad = sdesc_sw128(dob + ks * 2048, 8192, 1024);
          mma_bf16(tmem + TD_DV, ad, sdesc_sw128(aqb + ks * 2048, 8192, 1024), idesc, ks > 0);
          mma_bf16(tmem + TD_DV, ad, sdesc_sw128(aqb + 8192 + ks * 2048, 8192, 1024), idesc, 1);
        }
        return true;
      };
      if (!issue_doaqk(0)) ok = false;
      for (int64_t it = 0; it < nch && ok; ++it) {
        const uint32_t dob = smem_u32(slotA(it) + DA_DO);
        if (!mbar_wait(fullKG, par1(it))) { ok = false; break; }
        // G1: needs dS'^T hi / lo (and the rescaled dS'^T already in the accumulator)
        if (!mbar_wait_spin(bar_st, par1(it))) { ok = false; break; }
        tc_fence_after();
        {
          const uint32_t idesc = idesc_bf16(128, 64, false, true);
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks) {  // channels 16 ks .. 16 ks + 15 (rows of Kg^T)
            const uint32_t bo = (uint32_t)ks * 2048u;
            mma_bf16_ts(tmem + TD_DV, tmem + TD_DSA + 8 * ks, sdesc_sw128(kg_hi + bo, 8192, 1024), idesc, 1);
            mma_bf16_ts(tmem + TD_DV, tmem + TD_DSA + 8 * ks, sdesc_sw128(kg_lo + bo, 8192, 1024), idesc, 1);
            mma_bf16_ts(tmem + TD_DV, tmem + TD_DSA + 64 + 8 * ks, sdesc_sw128(kg_hi + bo, 8192, 1024), idesc, 1);
          }
        }
        mma_commit(bar_dv);
        mma_commit(freedKG);
        // dO^T Qg into the dS^T accumulator while the epilogue turns dV_new^T into operands
        if (!mbar_wait(fullQW, par1(it))) { ok = false; break; }
        tc_fence_after();
        {
          const uint32_t idesc = idesc_bf16(128, 128, true, true);
#pragma unroll 1
          for (int ks = 0; ks < 4; ++ks) {  // tokens 16 ks .. 16 ks + 15
            const uint64_t ad = sdesc_sw128(dob + ks * 2048, 8192, 1024);
            mma_bf16(tmem + TD_DS, ad, sdesc_sw128(qg_hi + ks * 2048, 8192, 1024), idesc, 1);
            mma_bf16(tmem + TD_DS, ad, sdesc_sw128(qg_lo + ks * 2048, 8192, 1024), idesc, 1);
          }
        }
        // G2: needs dV_new^T hi / lo
        if (!mbar_wait_spin(bar_dvn, par1(it))) { ok = false; break; }
        tc_fence_after();
        {
          const uint32_t idesc = idesc_bf16(128, 128, false, true);
#pragma unroll 1
          for (int ks = 0; ks < 4; ++ks) {  // tokens 16 ks .. 16 ks + 15 (rows of -W)
            const uint32_t bo = (uint32_t)ks * 2048u;
            mma_bf16_ts(tmem + TD_DS, tmem + TD_DVA + 8 * ks, sdesc_sw128(nw_hi + bo, 8192, 1024), idesc, 1);
            mma_bf16_ts(tmem + TD_DS, tmem + TD_DVA + 8 * ks, sdesc_sw128(nw_lo + bo, 8192, 1024), idesc, 1);
            mma_bf16_ts(tmem + TD_DS, tmem + TD_DVA + 32 + 8 * ks, sdesc_sw128(nw_hi + bo, 8192, 1024), idesc, 1);
          }
        }
        mma_commit(bar_ds);
        mma_commit(freedQW);
        mma_commit(&freedA[it & 1]);
        if (it + 1 < nch && !issue_doaqk(it + 1)) { ok = false; break; }
      }
      if (!ok) atomicOr(a.status, KDA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue warps -------------------------------------
    const int q4 = warp & 3, part = warp >> 2;  // part: channels 32 part ..; tokens 16 part ..
    const int v = 32 * q4 + lane;
    const uint32_t lb = tmem_addr(tmem, 32 * q4, 0);
    auto arrive = [&](uint64_t* bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    auto sidx = [&](int k) -> size_t {  // element (channel k, column v) of an external state
      return sbase + (a.state_v_first ? (size_t)v * K + k : (size_t)k * V + v);
    };
    float D[32];  // dS'^T[v][32 part + j]: the gradient of the state after the chunk
#pragma unroll
    for (int j = 0; j < 32; ++j)
      D[j] = a.d_final_state == nullptr ? 0.f : a.d_final_state[sidx(32 * part + j)];
    for (int64_t it = 0; it < nch && ok; ++it) {
      const int64_t c = cfirst + chunk_of(it);
      // dS'^T as hi / lo A operands of G1 and dS'^T Diag(e^gamma_C) into the accumulator
      bool w = mbar_wait(&fullA[it & 1], parA(it));
      {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) split2(D[2 * j], D[2 * j + 1], hi[j], lo[j]);
        tmem_st16(lb + TD_DSA + 16 * part, hi);
        tmem_st16(lb + TD_DSA + 64 + 16 * part, lo);
        const float* dc = reinterpret_cast<const float*>(slotA(it) + DA_D) + 32 * part;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t sc[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) sc[x] = __float_as_uint(D[16 * h + x] * dc[16 * h + x]);
          tmem_st16(lb + TD_DS + 32 * part + 16 * h, sc);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      arrive(bar_st);
      {  // dS' of this chunk out to the workspace, [K][V]
        float* hd = state_ptr(a, p.off_dh, c, hv);
#pragma unroll
        for (int j = 0; j < 32; ++j) hd[(size_t)(32 * part + j) * V + v] = D[j];
      }
      // dV_new^T -> hi / lo A operands of G2; out to the workspace
      w = mbar_wait(bar_dv, par1(it)) && w;
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(lb + TD_DV + 16 * part, r);
      tmem_wait_ld();
      {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          split2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]), hi[j], lo[j]);
        tmem_st8(lb + TD_DVA + 8 * part, hi);
        tmem_st8(lb + TD_DVA + 32 + 8 * part, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      arrive(bar_dvn);
      {
        float* dvn = block_ptr(a, c, hv) + p.blk.dvn;
#pragma unroll
        for (int x = 0; x < 16; ++x) dvn[(size_t)(16 * part + x) * V + v] = __uint_as_float(r[x]);
      }
      // the gradient of the state before this chunk: the previous chunk's dS'
      w = mbar_wait(bar_ds, par1(it)) && w;
      tc_fence_after();
      {
        uint32_t r0[16], r1[16];
        tmem_ld16(lb + TD_DS + 32 * part, r0);
        tmem_ld16(lb + TD_DS + 32 * part + 16, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          D[j] = __uint_as_float(r0[j]);
          D[16 + j] = __uint_as_float(r1[j]);
        }
      }
      if (!w) ok = false;
    }
    if (ok && a.dh0 != nullptr) {
#pragma unroll
      for (int j = 0; j < 32; ++j) a.dh0[sidx(32 * part + j)] = D[j];
    }
    if (!ok) atomicOr(a.status, KDA_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kEpi) tmem_dealloc(tmem, 512);
}

// ======================================================================================
// The gradient stage's products over v (backward-propagation step 5) on the tensor cores,
// one CTA per (chunk, value head), M = 64 tokens:
//   dQg = dO S^T, dW = -dV_new S^T            (steps 0, 1: B = S, A = dV_new)
//   dKg = V_new dS'^T, dAqk = dO V_new^T       (steps 2, 3: B = dS', A = V_new)
// each over the 128 columns of v in two 64-column halves (h = step % 2).  The fp32 rows of
// a step's B and A operands (the workspace's states, V_new, dV_new) arrive in a staging
// buffer by TMA while the previous step's MMAs and epilogue run; every thread then splits
// its share of them into bf16 hi / lo parts in the swizzled K-major layout, TMA brings the dO
// panel (an exact bf16 input), and one thread issues the MMAs (two per K-step with dO as A,
// three otherwise).  The diagonal of S dS'^T is summed while dS' is split (S read from the
// workspace directly).  Outputs go to the block's dq, y, dk, aqk and dkg slots, where the
// gradient stage reads them.
// ======================================================================================
constexpr uint32_t VP_B = 0;          // B tile (S or dS') hi, lo: [128 rows k][64 v], 16 KB each
constexpr uint32_t VP_A = 32768;      // A tile (dV_new or V_new) hi, lo: [64 rows t][64 v], 8 KB each
constexpr uint32_t VP_DO = 49152;     // dO panel [64 t][64 v] bf16
constexpr uint32_t VP_SB = 57344;     // fp32 staging of the B rows [128][64]
constexpr uint32_t VP_SA = 90112;     // fp32 staging of the A rows [64][64]
constexpr uint32_t VP_RED = 106496;   // [128][8] partial sums of diag(S dS'^T)
constexpr uint32_t VP_BAR = 110592;   // bar_do, bar_mma, bar_stg
constexpr uint32_t VP_TMEM = VP_BAR + 32;
constexpr uint32_t VP_SMEM = VP_TMEM + 16 + 1024;
constexpr uint32_t VP_STAGE_BYTES = 49152;
constexpr int kVpThreads = 256;

// hi / lo parts of eight consecutive fp32 values into the 16-byte chunks at `off` of a tile's
// high part and at `off + lo` of its low part
__device__ __forceinline__ void put8(uint8_t* tile, uint32_t off, uint32_t lo_off, const float4& x0,
                                     const float4& x1) {
  uint4 h, l;
  split2(x0.x, x0.y, h.x, l.x);
  split2(x0.z, x0.w, h.y, l.y);
  split2(x1.x, x1.y, h.z, l.z);
  split2(x1.z, x1.w, h.w, l.w);
  *reinterpret_cast<uint4*>(tile + off) = h;
  *reinterpret_cast<uint4*>(tile + off + lo_off) = l;
}

__global__ void __launch_bounds__(kVpThreads, 2)
    vprod_tc_kernel(const Args a, const __grid_constant__ CUtensorMap domap,
                    const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap dsmap,
                    const __grid_constant__ CUtensorMap vnmap, const __grid_constant__ CUtensorMap dvnmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  const Plan& p = a.p;
  const int64_t c = blockIdx.x;
  const int hv = blockIdx.y;
  const int K = p.K, V = p.V, C = p.C;
  int n, L;
  int64_t t0;
  if (!locate(a, c, n, t0, L)) {
    if (threadIdx.x == 0) atomicOr(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar_do = reinterpret_cast<uint64_t*>(sm + VP_BAR);
  uint64_t* bar_mma = bar_do + 1;
  uint64_t* bar_stg = bar_do + 2;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + VP_TMEM);
  float* sRed = reinterpret_cast<float*>(sm + VP_RED);
  const float* sSB = reinterpret_cast<const float*>(sm + VP_SB);
  const float* sSA = reinterpret_cast<const float*>(sm + VP_SA);
  if (warp == 0) {
    tmem_alloc(sTmem, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_do, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_stg, 1);
    fence_mbar_init();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  bool ok = true;
  float* blk = block_ptr(a, c, hv);
  const float* S = state_ptr(a, p.off_h, c, hv);
  const int32_t zc = (int32_t)(c * p.HV + hv);  // (chunk, value head) coordinate of the maps
  // staging of step st: B rows (S, dS') and A rows (dV_new, V_new) of v half st % 2
  auto issue_stage = [&](int st) {
    const int32_t v0 = 64 * (st & 1);
    mbar_arrive_expect_tx(bar_stg, VP_STAGE_BYTES);
    tma_load_3d(sm + VP_SB, st < 2 ? &smap : &dsmap, v0, 0, zc, bar_stg);
    tma_load_3d(sm + VP_SA, st < 2 ? &dvnmap : &vnmap, v0, 0, zc, bar_stg);
  };
  float dgc[4] = {0.f, 0.f, 0.f, 0.f};  // partials of diag(S dS'^T): rows (tid >> 3) + 32 i
  int do_open = -1, mma_open = -1, stg_open = -1;  // (thread 0) issued, not yet seen done
  const uint32_t b_hi = smem_u32(sm + VP_B), b_lo = b_hi + 16384u;
  const uint32_t a_hi = smem_u32(sm + VP_A), a_lo = a_hi + 8192u;
  const uint32_t do_b = smem_u32(sm + VP_DO);
  if (tid == 0) {
    issue_stage(0);
    stg_open = 0;
  }
  for (int step = 0; step < 4 && ok; ++step) {
    const int pair = step >> 1, h = step & 1;  // pair 0: B = S, A = dV_new; pair 1: dS', V_new
    const int v0 = 64 * h;
    if (tid == 0) {
      mbar_arrive_expect_tx(bar_do, 8192u);
      tma_load_3d(sm + VP_DO, &domap, v0, hv, (int32_t)t0, bar_do);
      do_open = step;
    }
    // items: B (row r = (tid >> 3) + 32 i, columns v0 + 8 g ..), A (row t likewise), g = tid & 7
    const int g = tid & 7, r_lo = tid >> 3;
    float4 sd[4][2];  // S at the B items, for the diagonal (dS' steps)
    if (pair == 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float* src = S + (size_t)(r_lo + 32 * i) * V + v0 + 8 * g;
        sd[i][0] = *reinterpret_cast<const float4*>(src);
        sd[i][1] = *reinterpret_cast<const float4*>(src + 4);
      }
    }
    if (!mbar_wait(bar_stg, (uint32_t)(step & 1))) ok = false;
    else if (tid == 0) stg_open = -1;
    if (ok) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = r_lo + 32 * i;
        const float4 x0 = *reinterpret_cast<const float4*>(sSB + r * 64 + 8 * g);
        const float4 x1 = *reinterpret_cast<const float4*>(sSB + r * 64 + 8 * g + 4);
        put8(sm + VP_B, swz128((uint32_t)r, (uint32_t)(8 * g)), 16384u, x0, x1);
        if (pair == 1) {
          const float4 y0 = sd[i][0], y1 = sd[i][1];
          dgc[i] = fmaf(x0.x, y0.x, fmaf(x0.y, y0.y, fmaf(x0.z, y0.z, fmaf(x0.w, y0.w, dgc[i]))));
          dgc[i] = fmaf(x1.x, y1.x, fmaf(x1.y, y1.y, fmaf(x1.z, y1.z, fmaf(x1.w, y1.w, dgc[i]))));
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = r_lo + 32 * i;
        const float4 x0 = *reinterpret_cast<const float4*>(sSA + t * 64 + 8 * g);
        const float4 x1 = *reinterpret_cast<const float4*>(sSA + t * 64 + 8 * g + 4);
        put8(sm + VP_A, swz128((uint32_t)t, (uint32_t)(8 * g)), 8192u, x0, x1);
      }
    }
    // the dO panel; rows past the chunk's end (another sequence's tokens) become zero
    if (ok) {
      if (!mbar_wait(bar_do, (uint32_t)(step & 1))) ok = false;
      else if (tid == 0) do_open = -1;
    }
    if (ok && L < C) {
      for (int e = tid; e < (C - L) * 8; e += kVpThreads)
        *reinterpret_cast<uint4*>(sm + VP_DO + (uint32_t)(L * 8 + e) * 16u) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    ok = named_bar_and(1, kVpThreads, ok);  // operand tiles written, staging free
    if (tid == 0 && ok) {
      if (step < 3) {  // the next step's rows arrive while this step's MMAs run
        issue_stage(step + 1);
        stg_open = step + 1;
      }
      tc_fence_after();
#pragma unroll 1
      for (int ks = 0; ks < 4; ++ks) {  // v0 + 16 ks .. + 15
        const uint32_t o = (uint32_t)ks * 32u;
        const uint32_t acc = (h > 0 || ks > 0) ? 1u : 0u;
        const uint64_t dA = sdesc_sw128(do_b + o, 16, 1024);
        const uint64_t Ah = sdesc_sw128(a_hi + o, 16, 1024), Al = sdesc_sw128(a_lo + o, 16, 1024);
        const uint64_t Bh = sdesc_sw128(b_hi + o, 16, 1024), Bl = sdesc_sw128(b_lo + o, 16, 1024);
        if (pair == 0) {
          const uint32_t id = idesc_bf16(64, 128), idn = idesc_bf16(64, 128, false, false, true);
          mma_bf16(tmem + 0, dA, Bh, id, acc);        // dQg = dO S^T
          mma_bf16(tmem + 0, dA, Bl, id, 1);
          mma_bf16(tmem + 128, Ah, Bh, idn, acc);     // dW = -dV_new S^T
          mma_bf16(tmem + 128, Ah, Bl, idn, 1);
          mma_bf16(tmem + 128, Al, Bh, idn, 1);
        } else {
          const uint32_t id = idesc_bf16(64, 128), id64 = idesc_bf16(64, 64);
          mma_bf16(tmem + 0, Ah, Bh, id, acc);        // dKg = V_new dS'^T
          mma_bf16(tmem + 0, Ah, Bl, id, 1);
          mma_bf16(tmem + 0, Al, Bh, id, 1);
          mma_bf16(tmem + 128, dA, Ah, id64, acc);    // dAqk = dO V_new^T (B = the A tile)
          mma_bf16(tmem + 128, dA, Al, id64, 1);
        }
      }
      mma_commit(bar_mma);
      mma_open = step;
    }
    if (ok) {
      if (!mbar_wait(bar_mma, (uint32_t)(step & 1))) ok = false;
      else if (tid == 0) mma_open = -1;
      ok = named_bar_and(1, kVpThreads, ok);
    }
    tc_fence_after();
    if (h == 1 && ok) {
      // epilogue of the pair: row t = 16 q + lane (lanes 0-15 of TMEM quadrant q = warp % 4
      // hold the M = 64 rows); warp / 4 picks the column half
      const int q = warp & 3, half = warp >> 2, t = 16 * q + lane;
      const uint32_t lb = tmem_addr(tmem, 32 * q, 0);
      float* out0 = blk + (pair == 0 ? p.blk.dq : p.blk.dk);
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t r[16];
        tmem_ld16(lb + 64 * half + 16 * j, r);
        tmem_wait_ld();
        if (lane < 16) {
          float4* d = reinterpret_cast<float4*>(out0 + (size_t)t * K + 64 * half + 16 * j);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            d[x] = make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                               __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
        }
      }
      if (pair == 0) {  // dW into the y slot
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t r[16];
          tmem_ld16(lb + 128 + 64 * half + 16 * j, r);
          tmem_wait_ld();
          if (lane < 16) {
            float4* d = reinterpret_cast<float4*>(blk + p.blk.y + (size_t)t * K + 64 * half + 16 * j);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              d[x] = make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                                 __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
          }
        }
      } else {  // dAqk, masked to j <= t < L, into the aqk slot
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
          uint32_t r[16];
          tmem_ld16(lb + 128 + 32 * half + 16 * j, r);
          tmem_wait_ld();
          if (lane < 16) {
            const int jb = 32 * half + 16 * j;
            float* d = blk + p.blk.aqk + (size_t)t * C + jb;
#pragma unroll
            for (int x = 0; x < 16; ++x) d[x] = (t < L && jb + x <= t) ? __uint_as_float(r[x]) : 0.f;
          }
        }
      }
      tc_fence_before();
      __syncthreads();  // the accumulators are read before the next pair's MMAs overwrite them
    }
  }
  if (ok) {  // diag(S dS'^T): the eight threads of each channel
#pragma unroll
    for (int i = 0; i < 4; ++i) sRed[(size_t)((tid >> 3) + 32 * i) * 8 + (tid & 7)] = dgc[i];
    __syncthreads();
    if (tid < K) {
      float d = 0.f;
#pragma unroll
      for (int x = 0; x < 8; ++x) d += sRed[(size_t)tid * 8 + x];
      blk[p.blk.dkg + tid] = d;
    }
  } else if (tid == 0) {
    atomicOr(a.status, KDA_DEV_TIMEOUT);
    // copies or an MMA group still in flight must end before shared and tensor memory go
    if (stg_open >= 0) mbar_wait(bar_stg, (uint32_t)(stg_open & 1), 100000000ull);
    if (do_open >= 0) mbar_wait(bar_do, (uint32_t)(do_open & 1), 100000000ull);
    if (mma_open >= 0) mbar_wait(bar_mma, (uint32_t)(mma_open & 1), 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// Driver entry point for tensor-map encoding, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

namespace {
// dO as [64 tokens x 64 v] boxes with 128-byte swizzle (one row of 128 bytes per token)
bool make_do_map(const Args& a, CUtensorMap& m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)a.p.V, (cuuint64_t)a.p.HV, (cuuint64_t)a.p.ntok};
  const cuuint64_t strides[2] = {(cuuint64_t)a.p.V * 2, (cuuint64_t)a.p.HV * a.p.V * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.d_o), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// fp32 rows of the workspace as [z][rows][cols] with z = chunk * HV + value head, rows
// `row_stride` floats apart, z `z_stride` floats apart: [rows x 64] boxes, no swizzle
bool make_rows_map(const Args& a, CUtensorMap& m, size_t off_bytes, int rows, int cols,
                   size_t row_stride, size_t z_stride, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)(a.p.nct * a.p.HV)};
  const cuuint64_t strides[2] = {(cuuint64_t)(row_stride * 4), (cuuint64_t)(z_stride * 4)};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.ws + off_bytes, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

// The state-gradient stage on the tensor cores (bf16 dO): one CTA per (sequence, value head).
cudaError_t run_dstate_tc(const Args& a, cudaStream_t st) {
  const unsigned grid = (unsigned)((int64_t)a.p.N * a.p.HV);
  if (grid == 0) return cudaSuccess;
  if (tmap_encoder() == nullptr) return cudaErrorNotSupported;
  CUtensorMap domap;  // MN-major A operand panels of dO^T
  if (!make_do_map(a, domap)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dstate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)DS_SMEM);
  if (e != cudaSuccess) return e;
  dstate_tc_kernel<<<grid, kStThreads, DS_SMEM, st>>>(a, domap);
  return cudaGetLastError();
}

// The gradient stage's products over v on the tensor cores (bf16 dO): one CTA per
// (chunk, value head).
cudaError_t run_vprod_tc(const Args& a, cudaStream_t st) {
  if (a.p.nct == 0 || a.p.HV == 0) return cudaSuccess;
  if (tmap_encoder() == nullptr) return cudaErrorNotSupported;
  CUtensorMap domap;  // K-major A operand panels of dO
  if (!make_do_map(a, domap)) return cudaErrorInvalidValue;
  // the states (S before, dS' after each chunk: [K][V] per (chunk, value head)) and the
  // V_new, dV_new rows of each block ([C][V])
  const Plan& p = a.p;
  const size_t kv = (size_t)p.K * p.V, blk0 = p.off_blocks;
  CUtensorMap smap, dsmap, vnmap, dvnmap;
  if (!make_rows_map(a, smap, p.off_h, p.K, p.V, p.V, kv, 128) ||
      !make_rows_map(a, dsmap, p.off_dh, p.K, p.V, p.V, kv, 128) ||
      !make_rows_map(a, vnmap, blk0 + 4 * p.blk.vn, p.C, p.V, p.V, p.blk.floats, 64) ||
      !make_rows_map(a, dvnmap, blk0 + 4 * p.blk.dvn, p.C, p.V, p.V, p.blk.floats, 64))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(vprod_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)VP_SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)a.p.nct, (unsigned)a.p.HV);
  vprod_tc_kernel<<<grid, kVpThreads, VP_SMEM, st>>>(a, domap, smap, dsmap, vnmap, dvnmap);
  return cudaGetLastError();
}

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
