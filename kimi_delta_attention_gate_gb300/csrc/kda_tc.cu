// bf16 tensor-core path of the KDA chunk forward (K = V = 128, chunk 64).
//
// Two kernels exchange, per (chunk, value head), one packed block laid out exactly
// as the recurrence kernel's shared-memory MMA operands (128-byte-swizzled panels):
//
//   tc_intra  one CTA per (chunk, value head), all chunks in parallel.
//             "Reading Notes: Implementation Notes for KDA in FLA", forward steps 1-3:
//             gate activation + chunk-local cumsum (log2 units), q/k L2 norm, beta
//             sigmoid; Aqk and Akk by tcgen05 MMAs; A = (I + Akk)^-1 by blocked
//             forward substitution; W = A Diag(beta) (e^Gamma . K) by a tcgen05 MMA;
//             Qg, Kg^T, e^gamma_C.
//   tc_recur  one CTA per (sequence, value head), chunks in order.
//             Steps 4-5 in transposed form so that the MMA M dimension is the V tile:
//               V_new^T = V^T T^T - S^T W^T          (T = A Diag(beta))
//               O^T     = S^T Qg^T + V_new^T Aqk^T
//               S^T     = S^T Diag(e^gamma_C) + V_new^T Kg
//             S^T stays in tensor memory in fp32 and is rounded to bf16 only as an MMA
//             operand.
//
// Exponent range (FLA-KDA engineering notes, section 3): the decay inside a chunk
// reaches 2^-461 at lower_bound = -5, so (Q e^Gamma)(K e^-Gamma)^T cannot be formed
// over a whole chunk.  Each 16-row block I uses its own reference r_I = Gamma just
// before the block: the query side q_i 2^(Gamma_i - r_I) <= 1 and the key side
// k_j 2^(r_I - Gamma_j), which is <= 1 for earlier blocks and at most 2^115 inside the
// block at lower_bound = -5 (16 tokens x 5 nat), within the fp32/bf16 exponent range.
// A block whose in-block decay could exceed 2^120 (tested as either 8-row half exceeding
// 2^60, which never happens for the safe gate at lower_bound = -5: 8 tokens x 5 nat is
// 2^57.7; possible for the plain or pre-gated gate) takes its diagonal 16 x 16 entries
// from an exact element-wise evaluation instead.
#include <cudaTypedefs.h>
#include <stdio.h>

#include "kda_internal.cuh"
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int TC_C = 64;
constexpr int TC_K = 128;
constexpr int TC_V = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kGuardLog2 = 120.0f;

// Packed block (bytes).  All panels 1024-byte aligned within the block.
//   B1 = [-W; Qg]   [128 rows x 128 ch]: panel p (16 KB) holds channels 64p..64p+63,
//                   rows 0-63 = -W (tokens), rows 64-127 = Qg (tokens)
//   B2 = [Aqk; Kg^T] [192 rows x 64 tokens]: rows 0-63 = Aqk, 64-191 = Kg^T (channels)
//   T  = A Diag(beta) [64 x 64];  D = e^gamma_C fp32 [128]
constexpr uint32_t OFF_B1 = 0;
constexpr uint32_t OFF_B2 = 32768;
constexpr uint32_t OFF_T = 57344;
constexpr uint32_t OFF_D = 65536;
constexpr uint32_t BLOCK_BYTES = 66048;

// First 1024-byte-aligned byte of the dynamic shared memory.  The offset is added to the
// shared array itself, not to an integer copy of its address, so that every access made
// through the result compiles to a 32-bit shared-memory access rather than a generic one.
__device__ __forceinline__ uint8_t* align1024(uint8_t* smem) {
  return smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}
__device__ __forceinline__ void sts_u32(uint8_t* base, uint32_t off, uint32_t v) {
  *reinterpret_cast<uint32_t*>(base + off) = v;
}
__device__ __forceinline__ void sts_v4(uint8_t* base, uint32_t off, uint32_t a, uint32_t b,
                                       uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(base + off) = make_uint4(a, b, c, d);
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sigmoid through ex2 / rcp (hardware approximations): absolute error ~1e-7, far below
// bf16 resolution
__device__ __forceinline__ float sigmoid_fast(float x) {
  return rcp_approx(1.0f + ex2(-x * kLog2e));
}
__device__ __forceinline__ float softplus_fast(float x) {
  return x > 20.0f ? x : log1pf(ex2(x * kLog2e));
}
// Packed fp32 pair arithmetic (one instruction for both channels of a pair; each half is
// rounded exactly as the scalar operation would be)
__device__ __forceinline__ uint64_t u64_of(float2 v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 f2_of(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(u64_of(a)), "l"(u64_of(b)));
  return f2_of(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(u64_of(a)), "l"(u64_of(b)));
  return f2_of(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(u64_of(a)), "l"(u64_of(b)), "l"(u64_of(c)));
  return f2_of(r);
}
__device__ __forceinline__ float2 bf_pair(uint32_t v) { return make_float2(bf_lo(v), bf_hi(v)); }
__device__ __forceinline__ uint32_t pack2(float2 v) { return pack_bf16x2(v.x, v.y); }

template <int GATE>
__device__ __forceinline__ float gate_fast(float x, float a, float lb) {
  if (GATE == KDA_GATE_PLAIN) return -a * softplus_fast(x);
  if (GATE == KDA_GATE_SAFE) return lb * sigmoid_fast(a * x);
  return x;
}

// ======================================================================================
// tc_intra
// ======================================================================================
// One CTA (256 threads, two resident per SM) per (chunk, value head).  The chunk's q, k
// and g tiles arrive by TMA in the 128-byte-swizzled panel layout of the MMA operands and
// are transformed in place: q, k -> [Qs; Ks] (A operand of the Aqk/Akk MMA) and g -> X =
// e^Gamma . K (MN-major B operand of the W MMA).  The packed block goes straight from
// registers to global memory.
constexpr uint32_t P_QK = 0;        // 2 K-panels x 128 rows, 16 KB each: row block b holds the
                                    // queries of tokens 16b..16b+15 in rows 32b..32b+15 and
                                    // their keys in rows 32b+16..32b+31;
                                    // after the Aqk/Akk MMA: T (A operand of the W MMA)
constexpr uint32_t P_X = 32768;     // 2 MN-panels x [64 tokens x 64 ch], 8 KB each: g, then X
constexpr uint32_t P_KA = 49152;    // [Ka_0; Ka_1; Ka_2; Ka_3] B operand: 160 rows, 2 panels x
                                    // 20 KB; after the Aqk/Akk MMA: fp32 solve scratch
constexpr uint32_t KA_PANEL = 20480;
constexpr uint32_t P_DIAG = P_KA + 2 * KA_PANEL;  // fp32 [4][2][16][16] exact diagonal blocks;
                                                  // later solve scratch Y [32][32]
constexpr uint32_t P_BETA = P_DIAG + 8192;        // fp32 [64]
constexpr uint32_t P_BSUM = P_BETA + 256;         // fp32 [8][128] half-block sums of the gate
constexpr uint32_t P_NORM = P_BSUM + 4096;        // fp32 [64 rows][2]: q (with scale), k multipliers
constexpr uint32_t P_DT = P_NORM + 512;           // fp32 [128] dt_bias row
constexpr uint32_t P_FLAG = P_DT + 512;
constexpr uint32_t P_BAR = P_FLAG + 16;  // [0] g + dt_bias loads, [1] MMA completions, [2] q, k loads
constexpr uint32_t P_TMEM = P_BAR + 32;
constexpr uint32_t P_END = P_TMEM + 16;
constexpr uint32_t P_SMEM = P_END + 1024;
// Ka_I (16(I+1) rows) starts at row 8 I (I+1) of the B operand; its accumulator D_I at the
// same TMEM column: 0, 16, 48, 96
__host__ __device__ constexpr uint32_t ka_row(int I) { return 8u * (uint32_t)(I * (I + 1)); }
// Rows of token t's query and key in the [Qs; Ks] operand (one TMEM lane quadrant per block)
__host__ __device__ constexpr uint32_t q_row(int t) { return 32u * (uint32_t)(t >> 4) + (uint32_t)(t & 15); }
__host__ __device__ constexpr uint32_t k_row(int t) { return q_row(t) + 16u; }
constexpr int SOLVE_LD = 65;

__device__ __forceinline__ uint2 lds_u64(const uint8_t* base, uint32_t off) {
  return *reinterpret_cast<const uint2*>(base + off);
}
__device__ __forceinline__ void sts_u64(uint8_t* base, uint32_t off, uint32_t a, uint32_t b) {
  *reinterpret_cast<uint2*>(base + off) = make_uint2(a, b);
}
__device__ __forceinline__ uint32_t lds_u32(const uint8_t* base, uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(base + off);
}

// Exact diagonal 16 x 16 block of Aqk and Akk0 for row block rg (every exponent
// Gamma_i - Gamma_j <= 0): partial sums over this thread's two channels, from the raw
// q / k tiles (read before they are transformed in place) and the gate cumsums gs[0..15],
// gs[16..31] of the two channels; out of line so that it costs the common path no
// instruction-cache space.
__device__ __noinline__ void guard_diagonal(const uint8_t* qk_pan, uint32_t cc, int rg, int L,
                                            const float* gs, const float* sNorm, float* dq) {
  float* dk = dq + 256;
  for (int i = 0; i < 16; ++i) {
    const int rowi = 16 * rg + i;
    const uint32_t qv = rowi < L ? lds_u32(qk_pan, sw128_offset(q_row(rowi), cc)) : 0u;
    const uint32_t kiv = rowi < L ? lds_u32(qk_pan, sw128_offset(k_row(rowi), cc)) : 0u;
    const float qn = sNorm[2 * rowi], kni = sNorm[2 * rowi + 1];
    const float qi0 = bf_lo(qv) * qn, qi1 = bf_hi(qv) * qn;
    const float ki0 = bf_lo(kiv) * kni, ki1 = bf_hi(kiv) * kni;
    for (int j = 0; j <= i; ++j) {
      const int rowj = 16 * rg + j;
      const uint32_t kv = rowj < L ? lds_u32(qk_pan, sw128_offset(k_row(rowj), cc)) : 0u;
      const float knj = sNorm[2 * rowj + 1];
      const float kj0 = bf_lo(kv) * knj, kj1 = bf_hi(kv) * knj;
      const float e0 = ex2(gs[i] - gs[j]), e1 = ex2(gs[16 + i] - gs[16 + j]);
      atomicAdd(&dq[i * 16 + j], qi0 * kj0 * e0 + qi1 * kj1 * e1);
      atomicAdd(&dk[i * 16 + j], ki0 * kj0 * e0 + ki1 * kj1 * e1);
    }
  }
}

template <int GATE>
__global__ void __launch_bounds__(256, 2)
    tc_intra_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap gmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const Plan& p = a.plan;
  const int64_t c = a.c_begin + blockIdx.x;
  const int hv = blockIdx.y;
  const int h = hv / p.G;
  int n, L;
  int64_t t0;
  // A launch of the next chunk range that was made dependent on this one programmatically
  // may start its CTAs once every CTA of this grid has started (this grid's last wave then
  // shares the SMs with that grid's first); no CTA of either reads what the other writes.
  // Without such a launch the instruction does nothing.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!locate_chunk(a, c, n, t0, L)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* sBeta = reinterpret_cast<float*>(sm + P_BETA);
  float* sBsum = reinterpret_cast<float*>(sm + P_BSUM);
  float* sNorm = reinterpret_cast<float*>(sm + P_NORM);
  float* sDiag = reinterpret_cast<float*>(sm + P_DIAG);
  float* sDt = reinterpret_cast<float*>(sm + P_DT);
  int* sFlag = reinterpret_cast<int*>(sm + P_FLAG);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + P_BAR);
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + P_TMEM);
  uint8_t* blk = reinterpret_cast<uint8_t*>(a.ws) + p.off_inter +
                 ((size_t)c * p.HV + hv) * p.inter_block_bytes;
  const bool has_dt = a.dt_bias != nullptr && GATE != KDA_GATE_PREGATED;

  if (warp == 0) {
    tmem_alloc(sTmem, 256);
    tmem_relinquish();
  }
  if (tid == 32) {  // tile loads: g -> 2 panels and the dt_bias row first (the gate phase
                    // needs only them), then q, k -> [Qs; Ks] row blocks on their own barrier
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    fence_mbar_init();
    sFlag[0] = 0;
    const int32_t tt = (int32_t)t0;
    mbar_arrive_expect_tx(&bars[0], 16384u + (has_dt ? TC_K * 4u : 0u));
    tma_load_3d(sm + P_X, &gmap, 0, hv, tt, &bars[0]);
    tma_load_3d(sm + P_X + 8192, &gmap, 64, hv, tt, &bars[0]);
    if (has_dt) bulk_g2s(sDt, a.dt_bias + (size_t)hv * TC_K, TC_K * 4, &bars[0]);
    mbar_arrive_expect_tx(&bars[2], 32768u);
#pragma unroll
    for (int pn = 0; pn < 2; ++pn)  // 16-token boxes: queries and keys of each row block
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint8_t* dst = sm + P_QK + pn * 16384 + b * 4096;
        tma_load_3d(dst, &qmap, 64 * pn, h, tt + 16 * b, &bars[2]);
        tma_load_3d(dst + 2048, &kmap, 64 * pn, h, tt + 16 * b, &bars[2]);
      }
  }
  for (int i = tid; i < 4 * 2 * 256; i += 256) sDiag[i] = 0.f;  // exact diagonal blocks
  // beta is read here and published to shared memory only after the tile wait, so that
  // its load latency overlaps the TMA loads
  const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(a.beta);
  __nv_bfloat16 beta_raw = __float2bfloat16_rn(0.f);
  if (tid < L && tid < TC_C) beta_raw = gb[(t0 + tid) * p.HV + hv];
  const float lb = a.lower_bound;
  const float aexp = (GATE != KDA_GATE_PREGATED && a.A_log != nullptr) ? expf(a.A_log[hv]) : 1.f;
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  if (!mbar_wait(&bars[0], 0)) flag_status(a.status, KDA_DEV_TIMEOUT);
  // A short chunk: its q, k and g rows past L (the next sequence's tokens or the copy's fill)
  // become zero once, so that no later load needs a row mask.
  if (L < TC_C) {
    for (int e = tid; e < (TC_C - L) * 16; e += 256) {  // g: 2 panels x 8 pieces per token
      const int t = L + (e >> 4), pn = (e >> 3) & 1, ch = e & 7;
      sts_v4(sm + P_X + pn * 8192, (uint32_t)t * 128 + ch * 16, 0u, 0u, 0u, 0u);
    }
    __syncthreads();
  }

  // ---- element-wise phases: thread = 8-row half block hb (of 16-row block rg) x channels
  // c0..c0+3 (pairs A = c0, c0+1 and B = c0+2, c0+3); warp hb holds all 128 channels of its
  // rows, so that row norms reduce inside the warp ----
  const int hb = tid >> 5, rg = hb >> 1, c0 = 4 * lane;
  const uint32_t pan = (uint32_t)(c0 >> 6);  // panel of these channels
  const uint32_t cc = (uint32_t)(c0 & 63);
  uint8_t* qk_pan = sm + P_QK + pan * 16384;
  uint8_t* x_pan = sm + P_X + pan * 8192;
  float2 dtA = make_float2(0.f, 0.f), dtB = make_float2(0.f, 0.f);
  if (has_dt) {
    const float4 d4 = *reinterpret_cast<const float4*>(sDt + c0);
    dtA = make_float2(d4.x, d4.y);
    dtB = make_float2(d4.z, d4.w);
  }
  // gate + in-half-block cumsum (log2 units); G <= 0 for every non-positive gate
  float2 GA[8], GB[8];
  float2 accA = make_float2(0.f, 0.f), accB = make_float2(0.f, 0.f);
  float span = 0.f;
  const float zsc = -kLog2e * aexp;  // safe gate: 2^(zsc (g + dt)) = e^(-aexp (g + dt))
  const float2 zsc2 = make_float2(zsc, zsc), lb2 = make_float2(lb, lb);
  const float2 one2 = make_float2(1.f, 1.f), l2e2 = make_float2(kLog2e, kLog2e);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int row = 8 * hb + r;
    float2 gpA = make_float2(0.f, 0.f), gpB = make_float2(0.f, 0.f);
    if (row < L) {
      const uint2 gv = lds_u64(x_pan, sw128_offset(row, cc));
      if (GATE == KDA_GATE_SAFE) {  // lb sigmoid(a x) on the two channel pairs
        const float2 zA = mul2(add2(bf_pair(gv.x), dtA), zsc2);
        const float2 zB = mul2(add2(bf_pair(gv.y), dtB), zsc2);
        const float2 dA = add2(make_float2(ex2(zA.x), ex2(zA.y)), one2);
        const float2 dB = add2(make_float2(ex2(zB.x), ex2(zB.y)), one2);
        gpA = mul2(make_float2(rcp_approx(dA.x), rcp_approx(dA.y)), lb2);
        gpB = mul2(make_float2(rcp_approx(dB.x), rcp_approx(dB.y)), lb2);
      } else {
        gpA.x = gate_fast<GATE>(bf_lo(gv.x) + dtA.x, aexp, lb);
        gpA.y = gate_fast<GATE>(bf_hi(gv.x) + dtA.y, aexp, lb);
        gpB.x = gate_fast<GATE>(bf_lo(gv.y) + dtB.x, aexp, lb);
        gpB.y = gate_fast<GATE>(bf_hi(gv.y) + dtB.y, aexp, lb);
      }
    }
    accA = fma2(gpA, l2e2, accA);
    accB = fma2(gpB, l2e2, accB);
    GA[r] = accA;
    GB[r] = accB;
    if (GATE == KDA_GATE_PREGATED)
      span = fmaxf(span, fmaxf(fmaxf(fabsf(accA.x), fabsf(accA.y)), fmaxf(fabsf(accB.x), fabsf(accB.y))));
  }
  // a gate that is never positive makes the cumsum monotone: its last value is the span
  if (GATE != KDA_GATE_PREGATED)
    span = fmaxf(fmaxf(fabsf(accA.x), fabsf(accA.y)), fmaxf(fabsf(accB.x), fabsf(accB.y)));
  *reinterpret_cast<float4*>(sBsum + hb * 128 + c0) = make_float4(accA.x, accA.y, accB.x, accB.y);
  // both halves within 2^60 keep the block's in-block decay within 2^120
  if (span > 0.5f * kGuardLog2) atomicOr(sFlag, 1 << rg);
  if (tid < TC_C) {
    float b = __bfloat162float(beta_raw);
    if (a.beta_sigmoid && tid < L) b = (a.allow_neg_eigval ? 2.f : 1.f) * sigmoid_fast(b);
    sBeta[tid] = b;
  }
  if (!mbar_wait(&bars[2], 0)) flag_status(a.status, KDA_DEV_TIMEOUT);
  if (L < TC_C) {  // q, k: 2 panels x (query row, key row) x 8 pieces per token
    for (int e = tid; e < (TC_C - L) * 32; e += 256) {
      const int t = L + (e >> 5), pn = (e >> 4) & 1, rk = (e >> 3) & 1, ch = e & 7;
      sts_v4(sm + P_QK + pn * 16384, (rk ? k_row(t) : q_row(t)) * 128 + ch * 16, 0u, 0u, 0u, 0u);
    }
    __syncthreads();
  }
  // row sums of squares of q and k over all 128 channels inside the warp: a butterfly that
  // halves the rows each lane carries (lane bits 16, 8, 4), then sums over lane bits 2 and 1;
  // lane 4m ends with row 8 hb + m and publishes its multipliers
  {
    float sq[8], sk[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int row = 8 * hb + r;
      const uint2 qv = lds_u64(qk_pan, sw128_offset(q_row(row), cc));
      const uint2 kv = lds_u64(qk_pan, sw128_offset(k_row(row), cc));
      const float2 qa = bf_pair(qv.x), qb = bf_pair(qv.y), ka = bf_pair(kv.x), kb = bf_pair(kv.y);
      sq[r] = fmaf(qa.x, qa.x, fmaf(qa.y, qa.y, fmaf(qb.x, qb.x, qb.y * qb.y)));
      sk[r] = fmaf(ka.x, ka.x, fmaf(ka.y, ka.y, fmaf(kb.x, kb.x, kb.y * kb.y)));
    }
#pragma unroll
    for (int hw = 4; hw >= 1; hw >>= 1) {  // keep rows [hw, 2hw) if the lane bit is set
      const bool up = (lane & (4 * hw)) != 0;
#pragma unroll
      for (int x = 0; x < hw; ++x) {
        const float qs = up ? sq[x] : sq[x + hw], ks = up ? sk[x] : sk[x + hw];
        const float qk_ = up ? sq[x + hw] : sq[x], kk_ = up ? sk[x + hw] : sk[x];
        sq[x] = qk_ + __shfl_xor_sync(0xffffffffu, qs, 4 * hw);
        sk[x] = kk_ + __shfl_xor_sync(0xffffffffu, ks, 4 * hw);
      }
    }
#pragma unroll
    for (int o = 2; o >= 1; o >>= 1) {
      sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], o);
      sk[0] += __shfl_xor_sync(0xffffffffu, sk[0], o);
    }
    if ((lane & 3) == 0) {
      const int row = 8 * hb + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
      float qn = a.scale, kn = 1.f;
      if (a.qk_l2norm) {
        qn *= rsqrtf(sq[0] + 1e-6f);
        kn = rsqrtf(sk[0] + 1e-6f);
      }
      *reinterpret_cast<float2*>(sNorm + 2 * row) = make_float2(qn, kn);
    }
  }
  __syncthreads();  // half-block sums, exact-diagonal flags, row multipliers

  // ---- carries, factors, operand tiles ----
  // block references r_I = Gamma just before block I and gamma_C, summed from the half-block
  // sums; G made relative to the start of block rg
  float4 rI[4], gl;
  {
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f), cy = run;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      if ((x & 1) == 0) rI[x >> 1] = run;
      const float4 h4 = *reinterpret_cast<const float4*>(sBsum + x * 128 + c0);
      if (x == hb - 1 && (hb & 1)) cy = h4;
      run = make_float4(run.x + h4.x, run.y + h4.y, run.z + h4.z, run.w + h4.w);
    }
    gl = run;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      GA[r] = add2(GA[r], make_float2(cy.x, cy.y));
      GB[r] = add2(GB[r], make_float2(cy.z, cy.w));
    }
  }
  // r_b by selects (a run-time index would move rI to local memory)
  const float4 rb = rg == 0 ? rI[0] : (rg == 1 ? rI[1] : (rg == 2 ? rI[2] : rI[3]));
  const bool guard = (sFlag[0] >> rg) & 1;
  const float2 erbA = make_float2(ex2(rb.x), ex2(rb.y)), erbB = make_float2(ex2(rb.z), ex2(rb.w));
  const float2 ekgA = make_float2(ex2(gl.x - rb.x), ex2(gl.y - rb.y));
  const float2 ekgB = make_float2(ex2(gl.z - rb.z), ex2(gl.w - rb.w));
  if (hb == 0)
    *reinterpret_cast<float4*>(blk + OFF_D + 4 * c0) =
        make_float4(ex2(gl.x), ex2(gl.y), ex2(gl.z), ex2(gl.w));
  float2 FA[4], FB[4];  // 2^(r_I - r_b) for the blocks I > rg that see this block's keys
#pragma unroll
  for (int I = 0; I < 4; ++I) {
    FA[I] = (I > rg) ? make_float2(ex2(rI[I].x - rb.x), ex2(rI[I].y - rb.y)) : one2;
    FB[I] = (I > rg) ? make_float2(ex2(rI[I].z - rb.z), ex2(rI[I].w - rb.w)) : one2;
  }
  if (sFlag[0] != 0) {  // some block needs its diagonal entries evaluated exactly
    // the gate cumsums of (block, channel pair) go to a scratch row in the (not yet written)
    // Ka tile; then thread (block tid / 64, pair tid % 64) evaluates its 16 x 16 partial sums
    // out of line
    const int p0 = 2 * lane;  // pairs p0 (A) and p0 + 1 (B) of this thread
    float* gsA = reinterpret_cast<float*>(sm + P_KA) + (rg * 64 + p0) * 33;
    float* gsB = gsA + 33;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int ri = 8 * (hb & 1) + r;
      gsA[ri] = GA[r].x;
      gsA[16 + ri] = GA[r].y;
      gsB[ri] = GB[r].x;
      gsB[16 + ri] = GB[r].y;
    }
    __syncthreads();
    const int grg = tid >> 6, gp = tid & 63;
    if ((sFlag[0] >> grg) & 1)
      guard_diagonal(sm + P_QK + (uint32_t)((2 * gp) >> 6) * 16384, (uint32_t)((2 * gp) & 63), grg,
                     L, reinterpret_cast<float*>(sm + P_KA) + (grg * 64 + gp) * 33, sNorm,
                     sDiag + grg * 512);
    __syncthreads();
  }
  // Kg^T (row = channel, 8 consecutive tokens per thread) is packed two tokens per register
  // and written as one 16-byte piece per channel after the loop
  uint32_t kt[4][4];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int row = 8 * hb + r;
    const uint32_t oq = sw128_offset(q_row(row), cc), ok = sw128_offset(k_row(row), cc);
    const uint2 qv = lds_u64(qk_pan, oq), kv = lds_u64(qk_pan, ok);
    const float2 nrm = *reinterpret_cast<const float2*>(sNorm + 2 * row);  // (qn, kn)
    const float2 qn2 = make_float2(nrm.x, nrm.x), kn2 = make_float2(nrm.y, nrm.y);
    const float2 kfA = mul2(bf_pair(kv.x), kn2), kfB = mul2(bf_pair(kv.y), kn2);
    const float2 PA = make_float2(ex2(GA[r].x), ex2(GA[r].y));  // 2^(Gamma - r_b) <= 1
    const float2 PB = make_float2(ex2(GB[r].x), ex2(GB[r].y));
    const float2 qsA = mul2(mul2(bf_pair(qv.x), qn2), PA), qsB = mul2(mul2(bf_pair(qv.y), qn2), PB);
    const float2 ksA = mul2(kfA, PA), ksB = mul2(kfB, PB);
    sts_u64(qk_pan, oq, pack2(qsA), pack2(qsB));  // Qs
    sts_u64(qk_pan, ok, pack2(ksA), pack2(ksB));  // Ks
    // Qg (rows 64-127 of B1) and X share 2^Gamma = P 2^r_b
    sts_u64(blk + OFF_B1 + pan * 16384, sw128_offset(64 + row, cc), pack2(mul2(qsA, erbA)),
            pack2(mul2(qsB, erbB)));
    sts_u64(x_pan, sw128_offset(row, cc), pack2(mul2(ksA, erbA)), pack2(mul2(ksB, erbB)));
    float2 kgA, kgB;
    if (!guard) {
      // 2^(r_b - Gamma) <= 2^120
      const float2 keA = mul2(kfA, make_float2(ex2(-GA[r].x), ex2(-GA[r].y)));
      const float2 keB = mul2(kfB, make_float2(ex2(-GB[r].x), ex2(-GB[r].y)));
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        if (I < rg) continue;
        sts_u64(sm + P_KA + pan * KA_PANEL, sw128_offset(ka_row(I) + row, cc),
                pack2(mul2(keA, FA[I])), pack2(mul2(keB, FB[I])));  // F[rg] = 1 exactly
      }
      kgA = mul2(keA, ekgA);
      kgB = mul2(keB, ekgB);
    } else {
      // every exponent below is <= 0; the diagonal block is evaluated exactly above
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        if (I < rg) continue;
        float2 vA = make_float2(0.f, 0.f), vB = vA;
        if (I > rg) {
          vA = make_float2(kfA.x * ex2(rI[I].x - rb.x - GA[r].x), kfA.y * ex2(rI[I].y - rb.y - GA[r].y));
          vB = make_float2(kfB.x * ex2(rI[I].z - rb.z - GB[r].x), kfB.y * ex2(rI[I].w - rb.w - GB[r].y));
        }
        sts_u64(sm + P_KA + pan * KA_PANEL, sw128_offset(ka_row(I) + row, cc), pack2(vA), pack2(vB));
      }
      kgA = make_float2(kfA.x * ex2(gl.x - rb.x - GA[r].x), kfA.y * ex2(gl.y - rb.y - GA[r].y));
      kgB = make_float2(kfB.x * ex2(gl.z - rb.z - GB[r].x), kfB.y * ex2(gl.w - rb.w - GB[r].y));
    }
    const float kg[4] = {kgA.x, kgA.y, kgB.x, kgB.y};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      if (r & 1)
        kt[x][r >> 1] = pack_bf16x2(__uint_as_float(kt[x][r >> 1]), kg[x]);
      else  // hold the even row's value until its odd partner is computed
        kt[x][r >> 1] = __float_as_uint(kg[x]);
    }
  }
#pragma unroll
  for (int x = 0; x < 4; ++x)
    sts_v4(blk + OFF_B2, sw128_offset(64 + c0 + x, 8 * hb), kt[x][0], kt[x][1], kt[x][2], kt[x][3]);
  fence_async_smem();
  __syncthreads();

  // ---- Aqk / Akk in one MMA: D = [Qs;Ks] [Ka_0;..;Ka_3]^T, M=128, N=160, K=128 ----
  if (tid == 0) {
    tc_fence_after();
    const uint32_t abase = smem_u32(sm + P_QK), bbase = smem_u32(sm + P_KA);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_bf16(tmem, sdesc_sw128(abase + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
               sdesc_sw128(bbase + (ks >> 2) * KA_PANEL + (ks & 3) * 32, 16, 1024),
               idesc_bf16(128, 160), ks > 0);
    mma_commit(&bars[1]);
  }
  __syncwarp();
  if (!mbar_wait(&bars[1], 0)) flag_status(a.status, KDA_DEV_TIMEOUT);
  tc_fence_after();

  // ---- epilogue A: TMEM lane quadrant b holds row block b: queries in lanes 0-15, keys
  // in lanes 16-31.  Row i of block b uses the 16(b+1) columns of D_b, in 16-column pieces
  // shared by the quadrant's two warps ----
  float* sL = reinterpret_cast<float*>(sm + P_KA);  // beta Akk0 [64][65]; Ka no longer needed
  float* sX = sL + 64 * SOLVE_LD;                   // (I + beta Akk0)^-1 [64][65]
  {
    const int bq = warp & 3, hh = warp >> 2;
    const bool isk = lane >= 16;
    const int i = 16 * bq + (lane & 15);
    const bool diag_exact = (sFlag[0] >> bq) & 1;
    const float bi = sBeta[i];
    const float* dg = sDiag + bq * 512 + (isk ? 256 : 0) + (lane & 15) * 16;
    for (int pc = hh; pc <= bq; pc += 2) {
      const int jb = 16 * pc;  // first key index of the piece
      uint32_t r[16];
      tmem_ld16(tmem_addr(tmem, 32 * bq, ka_row(bq) + jb), r);
      tmem_wait_ld();
      float vals[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) vals[x] = __uint_as_float(r[x]);
      if (pc == bq) {  // the diagonal piece (warp-uniform): exact entries, lower triangle
        if (diag_exact) {
#pragma unroll
          for (int x = 0; x < 16; ++x) vals[x] = dg[x];
        }
        const int li = lane & 15;
#pragma unroll
        for (int x = 0; x < 16; ++x) vals[x] = (isk ? (x < li) : (x <= li)) ? vals[x] : 0.f;
      }
      if (!isk) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf)
          sts_v4(blk + OFF_B2, sw128_offset(i, jb + 8 * hlf),
                 pack_bf16x2(vals[8 * hlf + 0], vals[8 * hlf + 1]),
                 pack_bf16x2(vals[8 * hlf + 2], vals[8 * hlf + 3]),
                 pack_bf16x2(vals[8 * hlf + 4], vals[8 * hlf + 5]),
                 pack_bf16x2(vals[8 * hlf + 6], vals[8 * hlf + 7]));
      } else {
#pragma unroll
        for (int x = 0; x < 16; ++x) sL[i * SOLVE_LD + jb + x] = bi * vals[x];
      }
    }
    if (!isk && hh == 0) {  // Aqk columns past the row's block are zero
      for (int j0 = 16 * (bq + 1); j0 < TC_C; j0 += 8)
        sts_v4(blk + OFF_B2, sw128_offset(i, j0), 0u, 0u, 0u, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---- solve X = (I + beta Akk0)^-1 by recursive halving (16 -> 32 -> 64), fp32 ----
  float* sY = sDiag;  // scratch
  if (tid < 64) {     // level 1: the four 16 x 16 diagonal blocks, one column per thread,
                      // right-looking so that each step adds one FMA to the dependent chain
    const int b = tid >> 4, col = tid & 15, base = 16 * b;
    float x[16], sacc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) sacc[i] = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      x[m] = (m == col) ? 1.f : ((m > col) ? -sacc[m] : 0.f);
#pragma unroll
      for (int i = m + 1; i < 16; ++i)
        sacc[i] = fmaf(sL[(base + i) * SOLVE_LD + base + m], x[m], sacc[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sX[(base + i) * SOLVE_LD + base + col] = x[i];
  } else if (tid < 128) {  // the upper-right 16 x 16 of each 32 x 32 diagonal block is zero
    const int e = tid - 64;  // 64 threads x 8 entries
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const int f = 8 * e + x, pr = f >> 8, i = (f >> 4) & 15, j = f & 15;
      sX[(32 * pr + i) * SOLVE_LD + 32 * pr + 16 + j] = 0.f;
    }
  }
  __syncthreads();
  {  // level 2: X_{2p+1,2p} = -X_{2p+1,2p+1} (L_{2p+1,2p} X_{2p,2p}), p = 0, 1
    for (int e = tid; e < 512; e += 256) {
      const int pr = e >> 8, i = (e >> 4) & 15, j = e & 15;
      const int rb = 32 * pr + 16, cb = 32 * pr;
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        s = fmaf(sL[(rb + i) * SOLVE_LD + cb + m], sX[(cb + m) * SOLVE_LD + cb + j], s);
      sY[e] = s;
    }
    __syncthreads();
    for (int e = tid; e < 512; e += 256) {
      const int pr = e >> 8, i = (e >> 4) & 15, j = e & 15;
      const int rb = 32 * pr + 16, cb = 32 * pr;
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        s = fmaf(sX[(rb + i) * SOLVE_LD + rb + m], sY[pr * 256 + m * 16 + j], s);
      sX[(rb + i) * SOLVE_LD + cb + j] = -s;
    }
    __syncthreads();
  }
  // level 3: X_{B,A} = -X_BB (L_BA X_AA), A = rows / columns 0..31, B = 32..63, as two
  // tcgen05 MMA rounds (M = 64 with rows 32..63 kept, N = 32, K = 32).  Each fp32 operand is
  // split into bf16 hi + lo parts and a b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi is accumulated
  // in fp32 (relative error ~2^-16, far below the bf16 rounding of T).  Operand tiles live in
  // the dead [Qs; Ks] tile: A hi / lo (K-major, 64 rows) and B hi / lo (MN-major, 32 rows).
  {
    uint8_t* tA = sm + P_QK;          // [2][64 rows x 128 B]: hi, lo
    uint8_t* tB = sm + P_QK + 16384;  // [2][32 rows x 128 B]: hi, lo
    const uint32_t la = tmem + 0, lb = tmem + 32;  // first / second MMA round accumulators
    // 4 consecutive fp32 values -> hi / lo bf16 quads at byte offset `off` of two tiles
    auto put4 = [&](uint8_t* hi_tile, uint32_t tile_bytes, uint32_t off, const float* v) {
      const uint32_t h0 = pack_bf16x2(v[0], v[1]), h1 = pack_bf16x2(v[2], v[3]);
      const uint32_t l0 = pack_bf16x2(v[0] - bf_lo(h0), v[1] - bf_hi(h0));
      const uint32_t l1 = pack_bf16x2(v[2] - bf_lo(h1), v[3] - bf_hi(h1));
      *reinterpret_cast<uint2*>(hi_tile + off) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(hi_tile + tile_bytes + off) = make_uint2(l0, l1);
    };
    auto issue_round = [&](uint32_t acc) {  // 2 K steps x 3 hi / lo products
      tc_fence_after();
      const uint32_t ab = smem_u32(tA), bb = smem_u32(tB);
      int n = 0;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int t = 0; t < 3; ++t) {
          const uint32_t ao = (t == 2) ? 8192u : 0u, bo = (t == 1) ? 4096u : 0u;
          mma_bf16(acc, sdesc_sw128(ab + ao + ks * 32, 16, 1024),
                   sdesc_sw128(bb + bo + ks * 2048, 4096, 1024),
                   idesc_bf16(64, 32, false, true), n++ > 0);
        }
      mma_commit(&bars[1]);
    };
    // D rows 32..63 sit in lanes 0-15 of quadrants 2, 3 (M = 64 layout); warp halves split
    // the 32 columns
    const bool epi = (warp & 2) && lane < 16;
    const int er = 16 * ((warp & 3) - 2) + lane;  // row - 32
    const int ec = 16 * (warp >> 2);              // first column
    {  // first MMA round's operands: A = L[32..63][0..31], B = X_AA
      const int i = tid >> 3, m0 = (tid & 7) * 4;
      float v[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) v[x] = sL[(32 + i) * SOLVE_LD + m0 + x];
      put4(tA, 8192, sw128_offset(32 + i, m0), v);
#pragma unroll
      for (int x = 0; x < 4; ++x) v[x] = sX[i * SOLVE_LD + m0 + x];
      put4(tB, 4096, sw128_offset(i, m0), v);
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) issue_round(la);
    __syncwarp();
    if (!mbar_wait(&bars[1], 1)) flag_status(a.status, KDA_DEV_TIMEOUT);
    tc_fence_after();
    {  // second MMA round's operands: B = Y = L_BA X_AA (from TMEM), A = X[32..63][32..63]
      uint32_t r[16];
      tmem_ld16(tmem_addr(la, 32 * (warp & 3), ec), r);
      tmem_wait_ld();
      if (epi) {
#pragma unroll
        for (int x = 0; x < 16; x += 4) {
          const float v[4] = {__uint_as_float(r[x]), __uint_as_float(r[x + 1]),
                              __uint_as_float(r[x + 2]), __uint_as_float(r[x + 3])};
          put4(tB, 4096, sw128_offset(er, ec + x), v);
        }
      }
      const int i = tid >> 3, m0 = (tid & 7) * 4;
      float v[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) v[x] = sX[(32 + i) * SOLVE_LD + 32 + m0 + x];
      put4(tA, 8192, sw128_offset(32 + i, m0), v);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) issue_round(lb);
    __syncwarp();
    if (!mbar_wait(&bars[1], 0)) flag_status(a.status, KDA_DEV_TIMEOUT);
    tc_fence_after();
    {  // X_BA = -(X_BB Y)
      uint32_t r[16];
      tmem_ld16(tmem_addr(lb, 32 * (warp & 3), ec), r);
      tmem_wait_ld();
      if (epi) {
#pragma unroll
        for (int x = 0; x < 16; ++x) sX[(32 + er) * SOLVE_LD + ec + x] = -__uint_as_float(r[x]);
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  // T = X Diag(beta), bf16: A operand of the W MMA (over the dead [Qs; Ks] tile) and block
  {
    const int i = tid >> 2, j0 = (tid & 3) * 16;
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      float t[8];
      const float4 b0 = *reinterpret_cast<const float4*>(sBeta + j0 + 8 * hlf);
      const float4 b1 = *reinterpret_cast<const float4*>(sBeta + j0 + 8 * hlf + 4);
      const float bj[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int j = j0 + 8 * hlf + x;
        t[x] = (j <= i) ? sX[i * SOLVE_LD + j] * bj[x] : 0.f;
      }
      const uint32_t w0 = pack_bf16x2(t[0], t[1]), w1 = pack_bf16x2(t[2], t[3]);
      const uint32_t w2 = pack_bf16x2(t[4], t[5]), w3 = pack_bf16x2(t[6], t[7]);
      const uint32_t off = sw128_offset(i, j0 + 8 * hlf);
      sts_v4(sm + P_QK, off, w0, w1, w2, w3);
      sts_v4(blk + OFF_T, off, w0, w1, w2, w3);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- W = T X: M=64 tokens, N=128 channels, K=64 (X MN-major; row i of W in TMEM
  // lane 32(i/16)+i%16) ----
  if (tid == 0) {
    tc_fence_after();
    const uint32_t abase = smem_u32(sm + P_QK), bbase = smem_u32(sm + P_X);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(tmem, sdesc_sw128(abase + ks * 32, 16, 1024),
               sdesc_sw128(bbase + ks * 2048, 8192, 1024), idesc_bf16(64, 128, false, true),
               ks > 0);
    mma_commit(&bars[1]);
  }
  __syncwarp();
  if (!mbar_wait(&bars[1], 1)) flag_status(a.status, KDA_DEV_TIMEOUT);
  tc_fence_after();
  {
    const int q4 = warp & 3, hh = warp >> 2;
    const int i = 16 * q4 + (lane & 15);
    uint8_t* wp = blk + OFF_B1 + hh * 16384;  // rows 0-63 of panel hh
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t r[16];
      tmem_ld16(tmem_addr(tmem, 32 * q4, 64 * hh + 16 * c4), r);
      tmem_wait_ld();
      if (lane < 16) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf)
          sts_v4(wp, sw128_offset(i, 16 * c4 + 8 * hlf),  // -W (rows 0-63 of B1)
                 pack_bf16x2(-__uint_as_float(r[8 * hlf + 0]), -__uint_as_float(r[8 * hlf + 1])),
                 pack_bf16x2(-__uint_as_float(r[8 * hlf + 2]), -__uint_as_float(r[8 * hlf + 3])),
                 pack_bf16x2(-__uint_as_float(r[8 * hlf + 4]), -__uint_as_float(r[8 * hlf + 5])),
                 pack_bf16x2(-__uint_as_float(r[8 * hlf + 6]), -__uint_as_float(r[8 * hlf + 7])));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ======================================================================================
// tc_recur
// ======================================================================================
// One CTA per (sequence, value head) holds the whole V = 128.  Warps 0-15 are epilogue
// warps (thread v = 32q + lane of TMEM lane quadrant q = warp % 4 owns row v of every
// transposed tile; the four warps of a quadrant split its columns); in warp 16 one thread
// issues every MMA, in warp 17 one thread every bulk / tensor copy and L2 prefetch (issuing
// a chunk's copies takes ~1,000 cycles, which must not delay the next MMA), and the roles
// meet on mbarriers.  The fp32 state S^T lives in tensor memory as an MMA accumulator; the bf16
// copies of S^T and V_new^T that serve as A operands are written to tensor memory too, so
// no operand goes through shared memory except the packed block and the v tile.
// An MMA instruction (M = 128, K = 16) costs at least ~94 cycles whatever N up to 128
// (~107 at N = 192, measured), so the chunk's products are merged into as few
// instructions as the tensor-memory layout [V_new^T | O^T | S^T] (64 + 64 + 128 columns)
// allows.  Per chunk (M = 128 rows of v in every MMA):
//   U      V_new^T = V^T T^T                       A = v tile (smem)  4 MMAs, N = 64
//   G1+O1  [V_new^T | O^T] += S^T [-W; Qg]^T       A = S^T (TMEM)     8 MMAs, N = 128
//   G2+O2  [O^T | S^T] += V_new^T [Aqk; Kg^T]^T    A = V_new^T (TMEM) 4 MMAs, N = 192
// where O^T was cleared and S^T scaled to S^T Diag(e^gamma_C) by the epilogue beforehand.
// G1+O1 -> G2+O2 -> G1+O1 is the dependent chain; U runs in its shadow.  O^T is drained
// through a shared-memory staging tile written back by one TMA store.  Packed blocks and
// v tiles are prefetched into L2 four chunks ahead and copied into shared memory one chunk
// ahead.
constexpr uint32_t SL_T = 57344;                     // within a slot (same offsets as the block)
constexpr uint32_t SL_D = 65536;
constexpr uint32_t SL_V = 66560;                     // v tile [64 tokens x 128 v], 2 MN panels
constexpr uint32_t SLOT = 82944;
constexpr uint32_t R_RING = 0;                       // 2 slots
constexpr uint32_t R_STG = 2 * SLOT;                 // O staging [2][64 tokens x 128 v] bf16
constexpr uint32_t R_BAR = R_STG + 32768;  // full[2], bar_v, bar_s, bar_vn, bar_st, freed[2]
constexpr uint32_t R_TMEM = R_BAR + 64;
constexpr uint32_t R_END = R_TMEM + 16;
constexpr uint32_t R_SMEM = R_END + 1024;
// tensor-memory columns
constexpr uint32_t TM_VN = 0;    // V_new^T fp32 [128 v x 64 tokens]
constexpr uint32_t TM_O = 64;    // O^T fp32 [128 v x 64 tokens]
constexpr uint32_t TM_S = 128;   // S^T fp32 [128 v x 128 ch]
constexpr uint32_t TM_SA = 256;  // S^T bf16 pairs (A operand), 64 columns
constexpr uint32_t TM_VA = 320;  // V_new^T bf16 pairs (A operand), 32 columns
constexpr int kPrefetch = 4;     // chunks whose loads are prefetched into L2 ahead
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kMmaWarp = kEpiWarps, kCopyWarp = kEpiWarps + 1;
constexpr int kRecThreads = kEpiThreads + 64;  // + MMA warp + copy warp

template <bool SAVE_STATES>  // SAVE_STATES: write the state before every chunk to h_out
__global__ void __launch_bounds__(kRecThreads, 1)
    tc_recur_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap omap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const Plan& p = a.plan;
  const int HV = p.HV;
  const int hv = (int)(blockIdx.x % HV);
  const int n = (int)(blockIdx.x / HV);
  int64_t bos, eos, cfirst;
  if (!seq_range(a, n, bos, eos, cfirst)) return;
  // the part of the sequence inside this launch's chunk range [c_begin, c_end)
  const int64_t nch_seq = (eos - bos + TC_C - 1) / TC_C;
  const int64_t lo = cfirst > a.c_begin ? cfirst : a.c_begin;
  const int64_t hi = cfirst + nch_seq < a.c_end ? cfirst + nch_seq : a.c_end;
  bool mine = lo < hi;
  if (nch_seq == 0)  // an empty sequence: one launch passes its initial state through
    mine = (a.c_begin <= cfirst && cfirst < a.c_end) || (cfirst == a.c_end && a.c_end == p.nct);
  if (!mine) return;
  const bool seq_start = nch_seq == 0 || lo == cfirst;
  const bool seq_end = nch_seq == 0 || hi == cfirst + nch_seq;
  const int64_t nch = nch_seq == 0 ? 0 : hi - lo;
  if (nch_seq > 0) {
    bos += (lo - cfirst) * TC_C;
    cfirst = lo;
  }
  float* carry = reinterpret_cast<float*>(a.ws + p.off_state);  // states between segments
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + R_BAR);
  uint64_t* bar_v = full + 2;   // G1+O1 done: V_new^T complete
  uint64_t* bar_s = full + 3;   // G2+O2 done: O^T and the next chunk's S^T complete
  uint64_t* bar_vn = full + 4;  // epilogue: bf16 V_new^T written
  uint64_t* bar_st = full + 5;  // epilogue: O^T read and cleared, bf16 S^T written
  uint64_t* freed = full + 6;   // [2]: G2+O2 of the slot's chunk done, the slot may be refilled
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + R_TMEM);
  if (warp == kMmaWarp) {
    tmem_alloc(sTmem, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&full[i], 1);
    mbar_init(&freed[0], 1);
    mbar_init(&freed[1], 1);
    mbar_init(bar_vn, kEpiWarps);
    mbar_init(bar_st, kEpiWarps);
    fence_mbar_init();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  bool ok = true;

  const uint8_t* blocks = reinterpret_cast<const uint8_t*>(a.ws) + p.off_inter;
  if (warp == kCopyWarp) {
    // ----------------------------------- copy warp ------------------------------------
    if (lane == 0) {
      const CUtensorMap* vmap_ptr = &vmap;  // generic address of the kernel parameter
      auto issue = [&](int64_t ci, int st) {  // chunk ci -> slot st: block + 2 v halves
        const int64_t cg = cfirst + ci;
        uint8_t* dst = sm + R_RING + st * SLOT;
        const uint8_t* src = blocks + ((size_t)cg * HV + hv) * p.inter_block_bytes;
        mbar_arrive_expect_tx(&full[st], BLOCK_BYTES + 16384);
        bulk_g2s(dst, src, BLOCK_BYTES, &full[st]);  // one large copy: per-SM bulk-copy
                                                     // throughput grows with copy size
        tma_load_3d(dst + SL_V, vmap_ptr, 0, hv, (int32_t)(bos + ci * TC_C), &full[st]);
        tma_load_3d(dst + SL_V + 8192, vmap_ptr, 64, hv, (int32_t)(bos + ci * TC_C), &full[st]);
      };
      auto prefetch = [&](int64_t ci) {
        const int64_t cg = cfirst + ci;
        bulk_prefetch_l2(blocks + ((size_t)cg * HV + hv) * p.inter_block_bytes, BLOCK_BYTES);
        tma_prefetch_3d(vmap_ptr, 0, hv, (int32_t)(bos + ci * TC_C));
        tma_prefetch_3d(vmap_ptr, 64, hv, (int32_t)(bos + ci * TC_C));
      };
      // Slot s holds chunks s, s+2, ...: chunk ci+2 is copied in as soon as G2+O2 of chunk ci
      // (the last reader of the slot) completes, a whole chunk before U of chunk ci+2 needs it.
      // freed[s] completes once per chunk of slot s and chunk ci+2 cannot complete before this
      // thread has seen chunk ci's phase, so the parity waits never fall two phases behind.
      int64_t issued = 0;
      if (nch > 0) {
        issue(0, 0);
        issued = 1;
        if (nch > 1) {
          issue(1, 1);
          issued = 2;
        }
        for (int64_t d = 2; d < 2 + kPrefetch && d < nch; ++d) prefetch(d);
      }
      for (int64_t ci = 0; ci + 2 < nch; ++ci) {
        const int s = (int)(ci & 1);
        if (!mbar_wait(&freed[s], (uint32_t)((ci >> 1) & 1))) { ok = false; break; }
        issue(ci + 2, s);
        issued = ci + 3;
        if (ci + 2 + kPrefetch < nch) prefetch(ci + 2 + kPrefetch);
      }
      if (!ok) {
        flag_status(a.status, KDA_DEV_TIMEOUT);
        // the copies in flight must land before the CTA's shared memory is released
        for (int64_t c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
          mbar_wait(&full[c & 1], (uint32_t)((c >> 1) & 1), 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------ MMA warp ------------------------------------
    if (lane == 0) {
      // wait for chunk ci's data, clear v rows past the chunk end, issue U^T into TM_VN
      auto issue_u = [&](int64_t ci) -> bool {
        const int st = (int)(ci & 1);
        if (!mbar_wait(&full[st], (uint32_t)((ci >> 1) & 1))) return false;
        uint8_t* slot = sm + R_RING + st * SLOT;
        const int64_t t0 = bos + ci * TC_C;
        const int L = (int)((eos - t0) < TC_C ? (eos - t0) : TC_C);
        if (L < TC_C) {  // those rows belong to another sequence or to padding
          for (int e = L * 8; e < TC_C * 8; ++e) {
            sts_v4(slot + SL_V, (uint32_t)e * 16u, 0u, 0u, 0u, 0u);
            sts_v4(slot + SL_V + 8192, (uint32_t)e * 16u, 0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        }
        tc_fence_after();
        const uint32_t vb = smem_u32(slot + SL_V), tb = smem_u32(slot + SL_T);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_VN, sdesc_sw128(vb + ks * 2048, 8192, 1024),
                   sdesc_sw128(tb + ks * 32, 16, 1024), idesc_bf16(128, 64, true), ks > 0);
        return true;
      };
      if (nch > 0 && !issue_u(0)) ok = false;
      for (int64_t ci = 0; ci < nch && ok; ++ci) {
        const int s = (int)(ci & 1);
        uint8_t* slot = sm + R_RING + s * SLOT;
        const uint32_t b1 = smem_u32(slot + OFF_B1), b2 = smem_u32(slot + OFF_B2);
        // G1+O1 need the bf16 S^T of this chunk and a cleared O^T
        if (!mbar_wait_spin(bar_st, (uint32_t)(ci & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_ts(tmem + TM_VN, tmem + TM_SA + 8 * ks,
                      sdesc_sw128(b1 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                      idesc_bf16(128, 128), 1);
        mma_commit(bar_v);
        // G2+O2 need the bf16 V_new^T of this chunk
        if (!mbar_wait_spin(bar_vn, (uint32_t)(ci & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_ts(tmem + TM_O, tmem + TM_VA + 8 * ks, sdesc_sw128(b2 + ks * 32, 16, 1024),
                      idesc_bf16(128, 192), 1);
        mma_commit(bar_s);
        mma_commit(&freed[s]);  // the slot's last reader
        if (ci + 1 < nch && !issue_u(ci + 1)) { ok = false; break; }
      }
      if (!ok) flag_status(a.status, KDA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // --------------------------------- epilogue warps ---------------------------------
    const int q4 = warp & 3, part = warp >> 2;  // part: S^T columns 32 part..; tokens 16 part..
    const int v = 32 * q4 + lane;
    const uint32_t lane_base = tmem_addr(tmem, 32 * q4, 0);
    const size_t sbase = ((size_t)n * HV + hv) * (size_t)TC_K * TC_V;
    float* sout = seq_end ? a.final_state : carry;
    // state element (channel 32 part + j, column v): [K][V] in the carry buffer, [K][V] or
    // [V][K] (state_v_first) in h0 / final_state
    auto sloc = [&](int j, bool external) -> size_t {  // offset within one K x V state
      return (external && a.state_v_first) ? (size_t)v * TC_K + 32 * part + j
                                           : (size_t)(32 * part + j) * TC_V + v;
    };
    auto sidx = [&](int j, bool external) -> size_t { return sbase + sloc(j, external); };
    auto arrive = [&](uint64_t* bar) {  // one arrival per warp, after the warp's writes
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    auto slot_of = [&](int64_t ci) { return sm + R_RING + (int)(ci & 1) * SLOT; };
    // the state before chunk ci, when the caller asked for the per-chunk states
    auto save_chunk_state = [&](const float (&S)[32], int64_t ci) {
      if (!SAVE_STATES) return;
      float* hc = a.h_out + ((size_t)(cfirst + ci) * HV + hv) * (size_t)TC_K * TC_V;
#pragma unroll
      for (int j = 0; j < 32; ++j) hc[sloc(j, true)] = S[j];
    };
    // bf16 copy of 32 state columns into the A operand of G1+O1; releases G1+O1
    auto publish_state = [&](const float (&S)[32]) {
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(S[2 * j], S[2 * j + 1]);
      tmem_st16(lane_base + TM_SA + 16 * part, pk);
      tmem_wait_st();
      tc_fence_before();
      arrive(bar_st);
    };
    // S^T Diag(e^gamma_C) of chunk ci into the accumulator (before G2+O2 of chunk ci)
    auto rescale_state = [&](const float (&S)[32], int64_t ci) -> bool {
      const bool w = mbar_wait(&full[ci & 1], (uint32_t)((ci >> 1) & 1));
      const float4* dec = reinterpret_cast<const float4*>(slot_of(ci) + SL_D) + 8 * part;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sc[16];
#pragma unroll
        for (int x4 = 0; x4 < 4; ++x4) {
          const float4 d = dec[4 * h + x4];
          const int j = 16 * h + 4 * x4;
          sc[4 * x4 + 0] = __float_as_uint(S[j + 0] * d.x);
          sc[4 * x4 + 1] = __float_as_uint(S[j + 1] * d.y);
          sc[4 * x4 + 2] = __float_as_uint(S[j + 2] * d.z);
          sc[4 * x4 + 3] = __float_as_uint(S[j + 3] * d.w);
        }
        tmem_st16(lane_base + TM_S + 32 * part + 16 * h, sc);
      }
      tmem_wait_st();
      return w;
    };
    __nv_bfloat16* go = static_cast<__nv_bfloat16*>(a.o);
    const CUtensorMap* omap_ptr = &omap;
    // O of chunk ci (this thread: 16 tokens of column v) through staging tile ci & 1: one TMA
    // store for a full chunk, 16-byte stores of the valid rows otherwise.  The tile was last
    // read by the store of chunk ci-2, which the first barrier confirms.
    auto store_o = [&](int64_t ci, const uint32_t (&ro)[16], bool good) -> bool {
      const int64_t t0 = bos + ci * TC_C;
      const int L = (int)((eos - t0) < TC_C ? (eos - t0) : TC_C);
      uint8_t* stg = sm + R_STG + (uint32_t)(ci & 1) * 16384u;
      if (tid == 0) bulk_wait_read1();
      good = named_bar_and(1, kEpiThreads, good);
#pragma unroll
      for (int x = 0; x < 16; ++x)
        *reinterpret_cast<__nv_bfloat16*>(stg + (16 * part + x) * 256 + v * 2) =
            __float2bfloat16_rn(__uint_as_float(ro[x]));
      fence_async_smem();
      good = named_bar_and(1, kEpiThreads, good);
      if (L == TC_C) {
        if (tid == 0) {
          tma_store_3d(omap_ptr, 0, hv, (int32_t)t0, stg);
          bulk_commit();
        }
      } else {
        for (int e = tid; e < L * 16; e += kEpiThreads) {
          const int row = e >> 4, c16 = e & 15;
          reinterpret_cast<uint4*>(go + ((t0 + row) * HV + hv) * (int64_t)TC_V)[c16] =
              reinterpret_cast<const uint4*>(stg + row * 256)[c16];
        }
      }
      return good;
    };

    {  // initial state -> bf16 A operand and the accumulator (scaled for chunk 0); O^T = 0
      float S[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        S[j] = !seq_start ? carry[sidx(j, false)] : (a.h0 != nullptr) ? a.h0[sidx(j, true)] : 0.f;
      if (nch == 0 && sout != nullptr) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sout[sidx(j, seq_end)] = S[j];
      }
      tmem_st16_zero(lane_base + TM_O + 16 * part);
      if (nch > 0) save_chunk_state(S, 0);
      publish_state(S);
      if (nch > 0 && !rescale_state(S, 0)) ok = false;
    }

    for (int64_t ci = 0; ci < nch; ++ci) {
      // V_new^T -> bf16 A operand of G2+O2 (this warp: tokens 16 part .. +15)
      bool w = mbar_wait(bar_v, (uint32_t)(ci & 1));
      tc_fence_after();
      {
        uint32_t r[16], pk[8];
        tmem_ld16(lane_base + TM_VN + 16 * part, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        tmem_st8(lane_base + TM_VA + 8 * part, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      arrive(bar_vn);
      // S^T of chunk ci+1 and O^T of chunk ci in one tensor-memory round trip; O^T cleared,
      // then G1+O1 of chunk ci+1 released before the output and the rescale are handled
      w = mbar_wait(bar_s, (uint32_t)(ci & 1)) && w;
      tc_fence_after();
      uint32_t ro[16];
      {
        uint32_t r0[16], r1[16];
        tmem_ld16(lane_base + TM_S + 32 * part, r0);
        tmem_ld16(lane_base + TM_S + 32 * part + 16, r1);
        tmem_ld16(lane_base + TM_O + 16 * part, ro);
        tmem_wait_ld();
        tmem_st16_zero(lane_base + TM_O + 16 * part);
        float S[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          S[j] = __uint_as_float(r0[j]);
          S[16 + j] = __uint_as_float(r1[j]);
        }
        if (ci + 1 < nch) {
          save_chunk_state(S, ci + 1);
          publish_state(S);
          w = rescale_state(S, ci + 1) && w;
        } else {
          tmem_wait_st();
          if (sout != nullptr) {
#pragma unroll
            for (int j = 0; j < 32; ++j) sout[sidx(j, seq_end)] = S[j];
          }
        }
      }
      if (!store_o(ci, ro, w)) { ok = false; break; }
    }
    if (!ok) flag_status(a.status, KDA_DEV_TIMEOUT);
    if (tid == 0) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// Driver entry point for tensor-map encoding, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool tc_eligible(const Plan& p, int dtype) {
  return dtype == KDA_BF16 && p.K == TC_K && p.V == TC_V && p.C == TC_C && p.ntok > 0;
}

size_t tc_inter_block_bytes() { return BLOCK_BYTES; }

cudaError_t launch_tc_intra(const FwdArgs& a, cudaStream_t s, bool overlap_previous) {
  const Plan& p = a.plan;
  if (a.c_end <= a.c_begin) return cudaSuccess;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  // q, k tiles: [16 tokens x 64 channels] boxes, g tiles: [64 tokens x 64 channels] boxes,
  // all with 128-byte swizzle (MMA operand layout)
  CUtensorMap qmap, kmap, gmap;
  const cuuint64_t qdims[3] = {(cuuint64_t)TC_K, (cuuint64_t)p.H, (cuuint64_t)p.ntok};
  const cuuint64_t qstr[2] = {(cuuint64_t)TC_K * 2, (cuuint64_t)p.H * TC_K * 2};
  const cuuint64_t gdims[3] = {(cuuint64_t)TC_K, (cuuint64_t)p.HV, (cuuint64_t)p.ntok};
  const cuuint64_t gstr[2] = {(cuuint64_t)TC_K * 2, (cuuint64_t)p.HV * TC_K * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t box16[3] = {64, 1, 16};  // q / k: one 16-token row block per box
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), qdims, qstr,
                   box16, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  r = enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k), qdims, qstr, box16,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  r = enc(&gmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.g), gdims, gstr, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)(a.c_end - a.c_begin), (unsigned)p.HV);
  // overlap_previous: the kernel may start while the work enqueued before it on `s` (the
  // previous chunk range's intra-chunk kernel, which triggers at its start) is still running
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = P_SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  cudaError_t e;
#define KDA_LAUNCH_INTRA(G)                                                                  \
  e = cudaFuncSetAttribute(tc_intra_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)P_SMEM);                                                     \
  if (e != cudaSuccess) return e;                                                            \
  e = cudaLaunchKernelEx(&cfg, tc_intra_kernel<G>, a, qmap, kmap, gmap);                     \
  if (e != cudaSuccess) return e;
  if (a.gate_mode == KDA_GATE_SAFE) {
    KDA_LAUNCH_INTRA(KDA_GATE_SAFE)
  } else if (a.gate_mode == KDA_GATE_PLAIN) {
    KDA_LAUNCH_INTRA(KDA_GATE_PLAIN)
  } else {
    KDA_LAUNCH_INTRA(KDA_GATE_PREGATED)
  }
#undef KDA_LAUNCH_INTRA
  return cudaGetLastError();
}

cudaError_t launch_tc_intra(const FwdArgs& a, cudaStream_t s) { return launch_tc_intra(a, s, false); }

cudaError_t launch_tc_recur(const FwdArgs& a, cudaStream_t s) {
  const Plan& p = a.plan;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  // v tiles: [64 tokens x 64 channels] boxes with 128-byte swizzle (MMA operand)
  // o tiles: [64 tokens x 128 channels] boxes, plain row-major (output staging)
  CUtensorMap vmap, omap;
  const cuuint64_t dims[3] = {(cuuint64_t)TC_V, (cuuint64_t)p.HV, (cuuint64_t)p.ntok};
  const cuuint64_t strides[2] = {(cuuint64_t)TC_V * 2, (cuuint64_t)p.HV * TC_V * 2};
  const cuuint32_t vbox[3] = {64, 1, 64};
  const cuuint32_t obox[3] = {128, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.v), dims, strides,
                   vbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  r = enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.o, dims, strides, obox, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((size_t)p.HV * p.N));
  auto kern = a.h_out != nullptr ? tc_recur_kernel<true> : tc_recur_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)R_SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, kRecThreads, R_SMEM, s>>>(a, vmap, omap);
  return cudaGetLastError();
}

}  // namespace kda
