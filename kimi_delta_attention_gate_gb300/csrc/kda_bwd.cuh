// Backward pass of the chunk-parallel KDA forward: fp32 CUDA-core stage bodies, written once
// for the GPU kernels (kda_bwd.cu) and for a host build that the tests run under
// AddressSanitizer.
//
// The stages follow the backward-propagation section of "Reading Notes: Implementation
// Notes for KDA in FLA" (chunk_kda_bwd), with C the chunk size, Gamma the chunk-local cumsum
// of the log decay g', gamma_C its last row, Q = scale * q / |q|, K = k / |k|:
//   prep    per (chunk, value head): g', Gamma, Q, K, beta, Aqk (lower), the strictly lower
//           P_ij = sum_k K_ik K_jk e^(Gamma_ik - Gamma_jk), e^gamma_C, Qg = e^Gamma Q,
//           Kg = e^(gamma_C - Gamma) K, and W = A Diag(beta) e^Gamma K, U = A Diag(beta) V
//           with A = (I + Diag(beta) P)^-1 by forward substitution (the recompute, step 1)
//   states  per (sequence, value head, 32-column V tile), chunks in order: the state S
//           before every chunk and V_new = U - W S (the recompute of the states, step 2)
//   dstate  per (sequence, value head, V tile), chunks in reverse, with dS' the gradient of
//           the state after a chunk: dV_new = Aqk^T dO + Kg dS' and
//           dS = Qg^T dO - W^T dV_new + Diag(e^gamma_C) dS' (steps 3-4)
//   grads   per (chunk, value head): dAqk = (dO V_new^T) masked lower, dQg = dO S^T,
//           dW = -dV_new S^T, dKg = V_new dS'^T; X = A^T dV_new and Y = A^T dW by back
//           substitution; dv = beta X, dbeta from X, Y and dAkk = -(A^T dA A^T) masked
//           strictly lower with A^T dA = X (beta V)^T + Y (beta e^Gamma K)^T; the
//           e^(Gamma_i - Gamma_j) terms of Aqk and P; the reverse cumsum of dGamma; the
//           backward of the gate activation, of the L2 norm and of the beta sigmoid
//           (steps 5-7).
// Every exponent is Gamma_i - Gamma_j with i >= j, Gamma_i, or gamma_C - Gamma_i: never
// positive while the log decay is non-positive, as in the forward's CUDA-core path.
//
// Execution model.  A stage body is a sequence of phases separated by block-wide barriers.
// Inside a phase each thread takes the elements tid, tid + nthr, ... of the phase's work
// ranges and keeps nothing across a barrier except in memory; control flow outside the
// phases is the same for every thread.  On the GPU a phase is one thread's share followed
// by __syncthreads(); the host build runs every thread's share of a phase, in a shuffled
// thread order, before the next phase, so that the host tests run the index arithmetic,
// barriers and work split of the GPU kernels.
#pragma once

#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "kda_bwd.h"

#if defined(__CUDACC__)
#define KDA_HD __host__ __device__ __forceinline__
#define KDA_BODY __device__ __forceinline__
#define KDA_UNROLL _Pragma("unroll")
#define KDA_UNROLL4 _Pragma("unroll 4")
#else
#define KDA_HD inline
#define KDA_BODY inline
#define KDA_UNROLL
#define KDA_UNROLL4
#endif

namespace kda {
namespace bwd {

constexpr int kThreads = 256;  // threads per block of every stage
constexpr int kBV = 32;        // V columns per block of the two state stages
constexpr float kL2Eps = 1e-6f;

// Operand tiles of the tensor-core state stages, per (chunk, value head), for K = V = 128 and
// C = 64, as bf16 high and low parts (x = hi + lo to ~2^-16), each part in the 128-byte-
// swizzled panel layout of the tensor cores' shared-memory operands: -W [64 tokens][128
// channels] (two 64-channel panels) and Kg^T [128 channels][64 tokens] (one panel) for both
// stages; Aqk [64 tokens][64 tokens] and Qg [64 tokens][128 channels] (two panels) for the
// state-gradient stage when it runs on the tensor cores too.
constexpr size_t kTileBytes = 65536;     // -W and Kg^T
constexpr size_t kTileBytesDs = 114688;  // + Aqk and Qg
constexpr size_t kTileNegW = 0;       // hi at +0, lo at +16384
constexpr size_t kTileKgT = 32768;    // hi at +32768, lo at +49152
constexpr size_t kTileLo = 16384;
constexpr size_t kTileAqk = 65536;    // hi at +65536, lo at +73728
constexpr size_t kTileAqkLo = 8192;
constexpr size_t kTileQg = 81920;     // hi at +81920, lo at +98304

// Float offsets of one (chunk, value head) block of the workspace.
struct Block {
  size_t gam, qn, kn, qg, kg, w, y, dq, dk, dgam, dkg;  // [C][K]
  size_t u, vn, dvn, x;                                  // [C][V]
  size_t aqk, p, ati;                                    // [C][C]
  size_t qf, kf, kb;                                     // [C][K] block-referenced rows
  size_t beta, decay, flag;                              // [C], [K], [4]
  size_t floats;                                         // a multiple of 64 (256 bytes)
};

KDA_HD Block block_layout(int C, int K, int V) {
  const size_t ck = (size_t)C * K, cv = (size_t)C * V, cc = (size_t)C * C;
  Block b;
  size_t o = 0;
  b.gam = o; o += ck;   // Gamma
  b.qn = o; o += ck;    // Q
  b.kn = o; o += ck;    // K
  b.qg = o; o += ck;    // Qg
  b.kg = o; o += ck;    // Kg
  b.w = o; o += ck;     // W
  b.y = o; o += ck;     // dW, then Y = A^T dW
  b.dq = o; o += ck;    // gradient of Q
  b.dk = o; o += ck;    // gradient of K
  b.dgam = o; o += ck;  // gradient of Gamma
  b.dkg = o; o += ck;   // dKg * Kg (the gamma_C part of the Kg gradient)
  b.u = o; o += cv;     // U
  b.vn = o; o += cv;    // V_new
  b.dvn = o; o += cv;   // dV_new
  b.x = o; o += cv;     // X = A^T dV_new
  b.aqk = o; o += cc;   // Aqk
  b.p = o; o += cc;     // P (strictly lower, without beta)
  b.ati = o; o += cc;   // A^T, A = (I + Diag(beta) P)^-1 (rows and columns >= L zero)
  b.qf = o; o += ck;    // Q e^(Gamma - rho_B), B the row's 16-row block (from prep)
  b.kf = o; o += ck;    // K e^(Gamma - rho_B)
  b.kb = o; o += ck;    // K e^(rho_B - Gamma)
  b.beta = o; o += C;
  b.decay = o; o += K;  // e^gamma_C
  b.flag = o; o += 4;   // > 0: some block-referenced exponent out of range (from prep)
  b.floats = (o + 63) / 64 * 64;
  return b;
}

// Resolved sizes and workspace layout of one backward call.
struct Plan {
  int B, T, H, HV, K, V, C, N, G;
  int64_t ntok, nct;
  int64_t cov_lo, cov_hi;  // the tokens the sequences cover: [cov_lo, cov_hi)
  int nc_per_seq, varlen;
  size_t off_table;   // int64 [N + 1] chunk offsets (varlen only)
  size_t off_blocks;  // [nct][HV] blocks
  size_t off_h;       // fp32 [nct][HV][K][V]: the state before every chunk
  size_t off_dh;      // fp32 [nct][HV][K][V]: the gradient of the state after every chunk
  int tc_states;      // the state stage runs on the tensor cores (K = V = 128, C = 64)
  int tc_dstate;      // and the state-gradient stage too (bf16 inputs as well)
  int tc_vprod;       // the gradient stage's V-reduced products run as their own tensor-core
                      // stage (same shapes): dQg, dW, dKg into the dq, y, dk slots, dAqk into
                      // the aqk slot, diag(S dS'^T) into the first K floats of the dkg slot
  size_t tile_bytes;  // operand tiles per (chunk, value head): kTileBytes or kTileBytesDs
  size_t off_tiles;   // [nct][HV] operand tiles of those stages
  size_t total_bytes;
  Block blk;
};

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Plan of a checked parameter set (host only).
inline Plan make_plan(const kda_fwd_params* f) {
  Plan p;
  memset(&p, 0, sizeof p);
  p.B = f->B; p.T = f->T; p.H = f->H; p.HV = f->HV; p.K = f->K; p.V = f->V;
  p.C = f->chunk_size; p.N = f->N; p.G = f->HV / f->H;
  p.ntok = (int64_t)f->B * f->T;
  p.varlen = f->cu_seqlens != nullptr || f->cu_seqlens_host != nullptr;
  p.nc_per_seq = (f->T + p.C - 1) / p.C;
  if (p.varlen) {
    int64_t nct = 0;
    for (int n = 0; n < f->N; ++n)
      nct += (f->cu_seqlens_host[n + 1] - f->cu_seqlens_host[n] + p.C - 1) / p.C;
    p.nct = nct;
    p.cov_lo = f->cu_seqlens_host[0];
    p.cov_hi = f->cu_seqlens_host[f->N];
  } else {
    p.nct = (int64_t)f->B * p.nc_per_seq;
    p.cov_lo = 0;
    p.cov_hi = p.ntok;
  }
  p.blk = block_layout(p.C, p.K, p.V);
  size_t off = 256;
  p.off_table = off;
  if (p.varlen) off += round256(sizeof(int64_t) * (size_t)(p.N + 1));
  p.off_blocks = off;
  off += round256(sizeof(float) * p.blk.floats * (size_t)p.nct * p.HV);
  const size_t states = sizeof(float) * (size_t)p.nct * p.HV * p.K * p.V;
  p.off_h = off;
  off += round256(states);
  p.off_dh = off;
  off += round256(states);
  p.tc_states = p.K == 128 && p.V == 128 && p.C == 64;
  p.tc_dstate = p.tc_states && f->in_dtype == KDA_BF16;
  p.tc_vprod = p.tc_dstate;
  if (p.tc_states) {
    p.tile_bytes = p.tc_dstate ? kTileBytesDs : kTileBytes;
    off = (off + 1023) / 1024 * 1024;
    p.off_tiles = off;
    off += p.tile_bytes * (size_t)p.nct * p.HV;
  }
  p.total_bytes = off;
  return p;
}

// The parts of the outputs that must read zero before the stages run: what atomics
// accumulate into (dA_log, ddt_bias and, with grouped heads, dq and dk) and the rows of the
// tokens no sequence covers.  Every other output element is written exactly once by the
// stages.  Entries: (output, first float, floats); returns their number (at most 14).
enum ZeroOut { kZeroDq, kZeroDk, kZeroDv, kZeroDg, kZeroDbeta, kZeroDAlog, kZeroDdt };
struct ZeroRange { int out; size_t first, count; };
inline int zero_ranges(const Plan& p, ZeroRange* z) {
  int n = 0;
  const size_t lo = (size_t)p.cov_lo, hi = (size_t)p.cov_hi, nt = (size_t)p.ntok;
  const size_t row[5] = {(size_t)p.H * p.K, (size_t)p.H * p.K, (size_t)p.HV * p.V,
                         (size_t)p.HV * p.K, (size_t)p.HV};
  for (int o = kZeroDq; o <= kZeroDbeta; ++o) {
    if (p.G > 1 && (o == kZeroDq || o == kZeroDk)) {
      z[n++] = {o, 0, nt * row[o]};
      continue;
    }
    if (lo > 0) z[n++] = {o, 0, lo * row[o]};
    if (hi < nt) z[n++] = {o, hi * row[o], (nt - hi) * row[o]};
  }
  z[n++] = {kZeroDAlog, 0, (size_t)p.HV};
  z[n++] = {kZeroDdt, 0, (size_t)p.HV * p.K};
  return n;
}

// Arguments of every stage (passed by value to the kernels).
struct Args {
  Plan p;
  int dtype, gate_mode, qk_l2norm, beta_sigmoid, allow_neg_eigval, state_v_first;
  float lower_bound, scale;
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const void* d_o;
  const float* A_log;
  const float* dt_bias;
  const float* h0;
  const float* d_final_state;
  const int64_t* cu_seqlens;
  float* dq;
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  float* dA_log;
  float* ddt_bias;
  float* dh0;
  char* ws;
  unsigned int* status;
};

// Grid sizes (blocks) of the stages.
inline int64_t chunk_blocks(const Plan& p) { return p.nct * p.HV; }
inline int64_t state_blocks(const Plan& p) {
  return (int64_t)p.N * p.HV * ((p.V + kBV - 1) / kBV);
}
// Dynamic shared memory (bytes) of the stages.
// prep: the Gamma, q and k tiles ([C][K + 1] each) in the first phases; beta P and the
// substitution's columns afterwards; then the exponent-range flag
KDA_HD size_t prep_region(const Plan& p) {
  const size_t C = (size_t)p.C;
  const size_t NB = (C + 15) / 16;
  const size_t early = 3 * C * (size_t)(p.K + 1) + (NB + NB * (NB - 1) / 2) * (size_t)p.K;
  const size_t late = C * C + C * (C + 4) + C * (size_t)(p.K + p.V);
  return early > late ? early : late;
}
inline size_t prep_smem(const Plan& p) { return sizeof(float) * (prep_region(p) + 4); }
inline size_t states_smem(const Plan& p) {
  const size_t K4 = (size_t)((p.K + 3) & ~3), C = (size_t)p.C;
  return sizeof(float) * (K4 * kBV + 2 * C * kBV + C * (K4 + 4) + C * K4 + K4);
}
KDA_HD bool dstate_stages_qw(int C, int K);
inline size_t dstate_smem(const Plan& p) {
  const size_t K4 = (size_t)((p.K + 3) & ~3), C = (size_t)p.C;
  const size_t base = K4 * kBV + 2 * C * kBV + C * (C + 4) + C * (K4 + 4) + K4;
  return sizeof(float) * (base + (dstate_stages_qw(p.C, p.K) ? 2 * C * K4 : 0));
}
// floats of the gradient stage's staging / scratch region: the back substitution's column
// half, the 32-column slices of the products, the row-norm partials
// The gradient stage's product slices: 32 columns of v per slice, rows 36 floats apart.
constexpr int kGradSliceW = 32, kGradSliceLd = 36;
// Scratch of the gradient stage once its product slices are done (behind beta P and A^T dA).
inline size_t grads_scratch(const Plan& p) {
  const size_t C = (size_t)p.C;
  size_t s = C * ((p.V + p.K + 1) / 2);
  s = s > 2 * C * 68 ? s : 2 * C * 68;                          // 64-column A^T dA slices
  const size_t ng = (size_t)((p.K + 3) / 4), l2 = 2 * ng * (2 * C + 1) + 4 * C;
  s = s > l2 ? s : l2;                                          // L2-norm backward sums
  s = s > 4 * (size_t)p.K ? s : 4 * (size_t)p.K;                // gate backward half sums
  // dP transposed, then the block-referenced key rows beyond the C x C of beta P's region
  const size_t kb_rows_in_ak = (C * C) / (size_t)p.K;
  const size_t kb_tail = C > kb_rows_in_ak ? (C - kb_rows_in_ak) * (size_t)p.K : 0;
  s = s > C * (C + 4) + kb_tail ? s : C * (C + 4) + kb_tail;
  return s;
}
// The region the product slices are staged in, and that beta P, A^T dA and the scratch take
// over afterwards.
inline size_t grads_region(const Plan& p) {
  const size_t C = (size_t)p.C, K4 = (size_t)((p.K + 3) & ~3);
  const size_t slices = (2 * K4 + 3 * C) * kGradSliceLd;
  const size_t after = C * C + C * (C + 1) + grads_scratch(p);
  return slices > after ? slices : after;
}
inline size_t grads_smem(const Plan& p) {
  return sizeof(float) * ((size_t)p.C * (p.C + 4) + 2 * (size_t)p.C + kThreads + 12 +
                          (size_t)((p.K + 3) & ~3) + grads_region(p));
}

// ---- element helpers ------------------------------------------------------------------

KDA_HD float bits_to_f32(uint32_t u) {
#if defined(__CUDA_ARCH__)
  return __uint_as_float(u);
#else
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
#endif
}

// Element i of an input tensor (bf16 widens exactly to fp32).
KDA_HD float ld_in(const void* base, int dtype, size_t i) {
  return dtype == KDA_F32 ? static_cast<const float*>(base)[i]
                          : bits_to_f32((uint32_t) static_cast<const uint16_t*>(base)[i] << 16);
}

// e^x through the hardware base-2 exponential on the GPU (a few ulp; every backward gradient
// is checked to 1e-4 relative), the C library's expf on the host
KDA_HD float fexp(float x) {
#if defined(__CUDA_ARCH__)
  return __expf(x);
#else
  return expf(x);
#endif
}
// fp32 -> bf16 bits, rounded to nearest even (finite inputs)
KDA_HD uint16_t bf16_bits_rn(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
KDA_HD float bf16_to_f32(uint16_t h) {
  const uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}
// Byte offset of element (row, col < 64) in a 128-byte-swizzled panel: rows of 128 bytes in
// groups of eight, the eight 16-byte chunks of row r permuted by chunk ^ (r % 8).
KDA_HD uint32_t swz128(uint32_t row, uint32_t col) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((((col >> 3) ^ (row & 7u)) & 7u) << 4) +
         ((col & 7u) << 1);
}
// Eight consecutive elements x[0..7] as bf16 hi + lo: one 16-byte chunk at byte offset `off`
// of a tile's high part and one at the same offset of its low part.  On the GPU two elements
// round in one instruction (cvt.rn.bf16x2.f32, round to nearest even as bf16_bits_rn: the same
// bits for every finite value); the element with the lower index sits in the lower half.
KDA_HD void put_hilo8(char* tile, size_t off, const float (&x)[8], size_t lo_off = kTileLo) {
#if defined(__CUDA_ARCH__)
  uint32_t h[4], l[4];
  KDA_UNROLL
  for (int j = 0; j < 4; ++j) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(x[2 * j + 1]), "f"(x[2 * j]));
    const float r0 = x[2 * j] - __uint_as_float(h[j] << 16);
    const float r1 = x[2 * j + 1] - __uint_as_float(h[j] & 0xFFFF0000u);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l[j]) : "f"(r1), "f"(r0));
  }
  *reinterpret_cast<uint4*>(tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(tile + off + lo_off) = make_uint4(l[0], l[1], l[2], l[3]);
#else
  uint16_t hi[8], lo[8];
  for (int j = 0; j < 8; ++j) {
    hi[j] = bf16_bits_rn(x[j]);
    lo[j] = bf16_bits_rn(x[j] - bf16_to_f32(hi[j]));
  }
  memcpy(tile + off, hi, 16);
  memcpy(tile + off + lo_off, lo, 16);
#endif
}

// Four consecutive elements as bf16 hi + lo: the 8-byte half of a 16-byte chunk at `off` (its
// first or second half: the column's bit 2 in swz128), the same in the low part.
KDA_HD void put_hilo4(char* tile, size_t off, const float (&x)[4], size_t lo_off = kTileLo) {
#if defined(__CUDA_ARCH__)
  uint32_t h[2], l[2];
  KDA_UNROLL
  for (int j = 0; j < 2; ++j) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(x[2 * j + 1]), "f"(x[2 * j]));
    const float r0 = x[2 * j] - __uint_as_float(h[j] << 16);
    const float r1 = x[2 * j + 1] - __uint_as_float(h[j] & 0xFFFF0000u);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l[j]) : "f"(r1), "f"(r0));
  }
  *reinterpret_cast<uint2*>(tile + off) = make_uint2(h[0], h[1]);
  *reinterpret_cast<uint2*>(tile + off + lo_off) = make_uint2(l[0], l[1]);
#else
  uint16_t hi[4], lo[4];
  for (int j = 0; j < 4; ++j) {
    hi[j] = bf16_bits_rn(x[j]);
    lo[j] = bf16_bits_rn(x[j] - bf16_to_f32(hi[j]));
  }
  memcpy(tile + off, hi, 8);
  memcpy(tile + off + lo_off, lo, 8);
#endif
}

KDA_HD float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
// The sigmoid's derivative s(x) (1 - s(x)) = t / (1 + t)^2 with t = e^-|x| <= 1: one
// exponential, and no cancellation once s(x) rounds to 1 (|x| beyond about 17 in fp32).
KDA_HD float dsigmoid_f(float x) {
  const float t = fexp(-fabsf(x)), d = 1.0f + t;
  return t / (d * d);
}
// log(1 + e^x); above 20 the correction log1p(e^-x) < 2.1e-9 is below fp32 resolution of x.
KDA_HD float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

// The activated log decay of one element ("FLA-KDA engineering notes", section 2), with
// x = g + dt_bias and `a` = exp(A_log) (1 without A_log in the safe gate).
KDA_HD float gate_f(int mode, float graw, float a, float dt, float lb) {
  const float x = graw + dt;
  if (mode == KDA_GATE_PLAIN) return -a * softplus_f(x);
  if (mode == KDA_GATE_SAFE) return lb * sigmoid_f(a * x);
  return graw;
}

KDA_HD float* block_ptr(const Args& a, int64_t c, int hv) {
  return reinterpret_cast<float*>(a.ws + a.p.off_blocks) +
         ((size_t)c * a.p.HV + hv) * a.p.blk.floats;
}

// The tensor-core state stage's operand tiles of (chunk c, value head hv) (tc_states only).
KDA_HD char* tile_ptr(const Args& a, int64_t c, int hv) {
  return a.ws + a.p.off_tiles + ((size_t)c * a.p.HV + hv) * a.p.tile_bytes;
}

KDA_HD float* state_ptr(const Args& a, size_t off, int64_t c, int hv) {
  return reinterpret_cast<float*>(a.ws + off) + ((size_t)c * a.p.HV + hv) * (size_t)a.p.K * a.p.V;
}

// Sequence n, first token t0 and length L of global chunk c; false if the device-side chunk
// table disagrees with the plan.
KDA_HD bool locate(const Args& a, int64_t c, int& n, int64_t& t0, int& L) {
  const Plan& p = a.p;
  int64_t bos, eos, ci;
  if (!p.varlen) {
    n = (int)(c / p.nc_per_seq);
    ci = c - (int64_t)n * p.nc_per_seq;
    bos = (int64_t)n * p.T;
    eos = bos + p.T;
  } else {
    const int64_t* cs = reinterpret_cast<const int64_t*>(a.ws + p.off_table);
    int lo = 0, hi = p.N;  // n with cs[n] <= c < cs[n + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cs[mid] <= c) lo = mid; else hi = mid;
    }
    n = lo;
    ci = c - cs[n];
    bos = a.cu_seqlens[n];
    eos = a.cu_seqlens[n + 1];
  }
  t0 = bos + ci * p.C;
  const int64_t len = eos - t0;
  if (ci < 0 || t0 < 0 || len <= 0 || eos > p.ntok) return false;
  L = (int)(len < p.C ? len : p.C);
  return true;
}

// Token range and first global chunk of sequence n; false if inconsistent.
KDA_HD bool seq_range(const Args& a, int n, int64_t& bos, int64_t& eos, int64_t& cfirst) {
  const Plan& p = a.p;
  if (!p.varlen) {
    bos = (int64_t)n * p.T;
    eos = bos + p.T;
    cfirst = (int64_t)n * p.nc_per_seq;
    return true;
  }
  bos = a.cu_seqlens[n];
  eos = a.cu_seqlens[n + 1];
  cfirst = reinterpret_cast<const int64_t*>(a.ws + p.off_table)[n];
  return bos >= 0 && eos >= bos && eos <= p.ntok && cfirst >= 0 &&
         cfirst + (eos - bos + p.C - 1) / p.C <= p.nct;
}

// ---- small vector helpers (16-byte loads on the GPU, plain element accesses on the host) ---

struct F4 { float x, y, z, w; };
// four consecutive floats from a 16-byte aligned address (a 16-byte shared load on the GPU)
KDA_HD F4 ld4(const float* p) {
#if defined(__CUDA_ARCH__)
  const float4 v = *reinterpret_cast<const float4*>(p);
  return {v.x, v.y, v.z, v.w};
#else
  return {p[0], p[1], p[2], p[3]};
#endif
}
KDA_HD void st4(float* p, const float (&v)[4]) {
#if defined(__CUDA_ARCH__)
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
#else
  p[0] = v[0]; p[1] = v[1]; p[2] = v[2]; p[3] = v[3];
#endif
}
KDA_HD float f4at(const F4& v, int i) { return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w)); }

KDA_HD int pad4(int x) { return (x + 3) & ~3; }

// Four consecutive elements off..off+3 of a row (fp32 workspace or an input tensor), zero
// past `len`; `vec`: the row length is a multiple of 4, so that the four are one aligned
// 16-byte (fp32) or 8-byte (bf16) load.  A plain (coherent) load: workspace rows are read in
// the kernel that wrote them.
KDA_HD F4 ld4w(const float* row, int off, int len, bool vec) {
  if (vec) {
#if defined(__CUDA_ARCH__)
    const float4 v = *reinterpret_cast<const float4*>(row + off);
    return {v.x, v.y, v.z, v.w};
#else
    return {row[off], row[off + 1], row[off + 2], row[off + 3]};
#endif
  }
  return {off < len ? row[off] : 0.f, off + 1 < len ? row[off + 1] : 0.f,
          off + 2 < len ? row[off + 2] : 0.f, off + 3 < len ? row[off + 3] : 0.f};
}
// The same for an input tensor (read-only for the whole pass: the read-only data path).
KDA_HD F4 ld4i(const void* base, int dtype, size_t row, int off, int len, bool vec) {
  if (vec) {
#if defined(__CUDA_ARCH__)
    if (dtype == KDA_F32) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + row + off));
      return {v.x, v.y, v.z, v.w};
    }
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + row + off));
    return {__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
            __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u)};
#endif
  }
  return {off < len ? ld_in(base, dtype, row + off) : 0.f,
          off + 1 < len ? ld_in(base, dtype, row + off + 1) : 0.f,
          off + 2 < len ? ld_in(base, dtype, row + off + 2) : 0.f,
          off + 3 < len ? ld_in(base, dtype, row + off + 3) : 0.f};
}
// Four consecutive shared-memory floats p[0..3], those at or past `avail` read as zero; one
// 16-byte load when all four exist and `vec` (the address is 16-byte aligned).
KDA_HD F4 lds4m(const float* p, int avail, bool vec) {
  if (vec && avail >= 4) return ld4(p);
  return {avail > 0 ? p[0] : 0.f, avail > 1 ? p[1] : 0.f, avail > 2 ? p[2] : 0.f, avail > 3 ? p[3] : 0.f};
}
// The store counterpart (shared or global memory): p[0..3] = v, those at or past `avail`
// left alone; one 16-byte store when all four exist and `vec`.
KDA_HD void sts4m(float* p, const float (&v)[4], int avail, bool vec) {
  if (vec && avail >= 4) {
    st4(p, v);
    return;
  }
  for (int x = 0; x < 4 && x < avail; ++x) p[x] = v[x];
}
KDA_HD float dot4(const F4& a, const F4& b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// Elements e = tid, tid + nthr, ... < n, NB at a time: first every load of the NB elements
// (ld(e) returns what an element needs), then the rest (st(e, loaded)).  The workspace arrays
// an element reads and writes are distinct in fact but not provably so, which would keep the
// compiler from moving one element's loads above the previous element's stores: each element
// would wait out a full memory latency.  Grouping the loads lets NB of them overlap.
template <int NB, class Ld, class St>
KDA_BODY void batched(int tid, int nthr, int n, Ld ld, St st) {
  using T = decltype(ld(0));
  for (int e0 = tid; e0 < n; e0 += NB * nthr) {
    T v[NB];
    KDA_UNROLL
    for (int u = 0; u < NB; ++u) {
      const int e = e0 + u * nthr;
      v[u] = e < n ? ld(e) : T{};
    }
    KDA_UNROLL
    for (int u = 0; u < NB; ++u) {
      const int e = e0 + u * nthr;
      if (e < n) st(e, v[u]);
    }
  }
}

// ---- prep: per (chunk c, value head hv) ------------------------------------------------

// SC, SK, SV: the chunk size and head dimensions as compile-time constants (0: the plan's),
// so that the index arithmetic of the common shape folds into shifts and multiplies.
template <int SC = 0, int SK = 0, int SV = 0, class Exec>
KDA_BODY void prep_body(Exec& ex, const Args& a, int64_t c, int hv, float* smem) {
  const Plan& p = a.p;
  const int C = SC ? SC : p.C, K = SK ? SK : p.K, V = SV ? SV : p.V;
  const int H = p.H, HV = p.HV, h = hv / p.G;
  int n, L;
  int64_t t0;
  if (!locate(a, c, n, t0, L)) {
    ex.flag(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  float* blk = block_ptr(a, c, hv);
  const Block& b = p.blk;
  float* Gam = blk + b.gam;
  float* Qn = blk + b.qn;
  float* Kn = blk + b.kn;
  float* Qg = blk + b.qg;
  float* Kg = blk + b.kg;
  float* W = blk + b.w;
  float* U = blk + b.u;
  float* Aqk = blk + b.aqk;
  float* P = blk + b.p;
  float* Be = blk + b.beta;
  float* Dc = blk + b.decay;
  const bool has_alog = a.A_log != nullptr && a.gate_mode != KDA_GATE_PREGATED;
  const float a_exp = has_alog ? expf(a.A_log[hv]) : 1.0f;
  float* sFlag = smem + prep_region(p);  // > 0: an exponent out of range
  // Gamma, q and k of the chunk stay in shared memory through the element-wise phases (rows
  // K + 1 floats apart: both row- and column-wise walks are free of bank conflicts); their
  // final values also go to the workspace, where the gradient stage reads them
  const bool vecK = (K & 3) == 0, vecV = (V & 3) == 0;  // rows of 16-byte (fp32) / 8-byte (bf16) pieces
  const int ldq = K + 1;
  float* sGam = smem;                   // [C][ldq]
  float* sQn = sGam + (size_t)C * ldq;  // [C][ldq]
  float* sKn = sQn + (size_t)C * ldq;   // [C][ldq]
  float* sRho = sKn + (size_t)C * ldq;  // [NB][K] Gamma at each 16-row block's middle row
  float* sF = sRho + (size_t)((C + 15) / 16) * K;  // [NB (NB - 1) / 2][K] e^(rho_I - rho_B), B < I

  // gate activation, q and k rows, beta; rows i >= L are zero
  ex.phase([&](int tid, int nthr) {
    if (tid == 0) sFlag[0] = 0.f;
    const bool has_dt = a.dt_bias != nullptr && a.gate_mode != KDA_GATE_PREGATED;
    // four channels per element: one 8-byte (bf16) or 16-byte (fp32) load per input row piece
    struct GQK { F4 g, q, k; };
    const int q4 = (K + 3) / 4;
    batched<4>(tid, nthr, C * q4, [&](int e) {
      const int i = e / q4, c4 = 4 * (e - (e / q4) * q4);
      GQK v{{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (i < L) {
        const size_t tok = (size_t)(t0 + i);
        v.g = ld4i(a.g, a.dtype, (tok * HV + hv) * K, c4, K, vecK);
        v.q = ld4i(a.q, a.dtype, (tok * H + h) * K, c4, K, vecK);
        v.k = ld4i(a.k, a.dtype, (tok * H + h) * K, c4, K, vecK);
      }
      return v;
    }, [&](int e, const GQK& v) {
      const int i = e / q4, c4 = 4 * (e - (e / q4) * q4);
      const F4 dt = has_dt ? ld4w(a.dt_bias + (size_t)hv * K, c4, K, vecK) : F4{0.f, 0.f, 0.f, 0.f};
      KDA_UNROLL
      for (int x = 0; x < 4; ++x) {
        if (c4 + x >= K) break;
        const size_t o = (size_t)i * ldq + c4 + x;
        sGam[o] = i < L ? gate_f(a.gate_mode, f4at(v.g, x), a_exp, f4at(dt, x), a.lower_bound) : 0.f;
        sQn[o] = f4at(v.q, x);
        sKn[o] = f4at(v.k, x);
      }
    });
    for (int i = tid; i < C; i += nthr) {
      float bv = 0.f;
      if (i < L) {
        bv = ld_in(a.beta, a.dtype, (size_t)(t0 + i) * HV + hv);
        if (a.beta_sigmoid) bv = (a.allow_neg_eigval ? 2.f : 1.f) * sigmoid_f(bv);
      }
      Be[i] = bv;
    }
  });
  // chunk-local cumsum (one thread per channel); L2 norm and scale of the rows (one thread
  // per row of q or k)
  ex.phase([&](int tid, int nthr) {
    for (int kk = tid; kk < K; kk += nthr) {
      float acc = 0.f;
      for (int i = 0; i < L; ++i) {
        acc += sGam[(size_t)i * ldq + kk];
        sGam[(size_t)i * ldq + kk] = acc;
      }
    }
    for (int r = tid; r < 2 * C; r += nthr) {
      const int i = r < C ? r : r - C;
      if (i >= L) continue;
      float* row = (r < C ? sQn : sKn) + (size_t)i * ldq;
      float mul = 1.f;
      if (a.qk_l2norm) {
        float ss = 0.f, ss2 = 0.f;
        int kk = 0;
        KDA_UNROLL4
        for (; kk + 1 < K; kk += 2) {
          ss = fmaf(row[kk], row[kk], ss);
          ss2 = fmaf(row[kk + 1], row[kk + 1], ss2);
        }
        if (kk < K) ss = fmaf(row[kk], row[kk], ss);
        mul = 1.0f / sqrtf((ss + ss2) + kL2Eps);
      }
      if (r < C) mul *= a.scale;
      KDA_UNROLL4
      for (int kk = 0; kk < K; ++kk) row[kk] *= mul;
    }
  });
  // e^gamma_C; Qg, Kg; the right-hand side of W; the block references rho_B (Gamma at the
  // middle row of each 16-row block)
  const int NB = (L + 15) >> 4;
  auto mid_row = [&](int B) { return (16 * B + 7) < L - 1 ? 16 * B + 7 : L - 1; };
  ex.phase([&](int tid, int nthr) {
    for (int kk = tid; kk < K; kk += nthr) Dc[kk] = expf(sGam[(size_t)(L - 1) * ldq + kk]);
    for (int e = tid; e < C * K; e += nthr) {  // the final Gamma, Q and K rows to the workspace
      const int i = e / K, kk = e - (e / K) * K;
      const size_t o = (size_t)i * ldq + kk;
      Gam[e] = sGam[o];
      Qn[e] = sQn[o];
      Kn[e] = sKn[o];
    }
    for (int u = tid; u < NB * K; u += nthr) {
      const int B = u / K;
      sRho[u] = sGam[(size_t)mid_row(B) * ldq + (u - B * K)];
    }
    // Kg's rows are read only by the CUDA-core state stages: on the GPU with both state stages
    // on the tensor cores (which read its operand tile) nothing reads them
    const bool kg_rows = !(Exec::kTensorCores && p.tc_states && p.tc_dstate);
    struct Row { float gi, gl, q, k, be; };
    batched<4>(tid, nthr, C * K, [&](int e) {
      const int i = e / K, kk = e - (e / K) * K;
      Row r{0.f, 0.f, 0.f, 0.f, 0.f};
      if (i < L) {
        const size_t o = (size_t)i * ldq + kk;
        r = Row{sGam[o], sGam[(size_t)(L - 1) * ldq + kk], sQn[o], sKn[o], Be[i]};
      }
      return r;
    }, [&](int e, const Row& r) {
      float qg = 0.f, kg = 0.f, w = 0.f;
      if (e / K < L) {
        const float eg = fexp(r.gi);
        qg = r.q * eg;
        kg = r.k * fexp(r.gl - r.gi);
        w = r.be * eg * r.k;
      }
      Qg[e] = qg;
      if (kg_rows) Kg[e] = kg;
      W[e] = w;
    });
    if (p.tc_states) {  // the state stages' Kg^T and Qg operand tiles (K = 128, C = 64), formed
                        // from shared memory exactly as Kg and Qg above (the same bits)
      char* tile = tile_ptr(a, c, hv);
      const int c8 = C / 8;
      for (int u = tid; u < K * c8; u += nthr) {  // Kg^T: row = channel, 8 tokens per piece
        const int kk = u / c8, tb = 8 * (u - (u / c8) * c8);
        const float gl = sGam[(size_t)(L - 1) * ldq + kk];
        float x[8];
        KDA_UNROLL
        for (int j = 0; j < 8; ++j) {
          const size_t o = (size_t)(tb + j) * ldq + kk;
          x[j] = tb + j < L ? sKn[o] * fexp(gl - sGam[o]) : 0.f;
        }
        put_hilo8(tile, kTileKgT + swz128((uint32_t)kk, (uint32_t)tb), x);
      }
      if (p.tc_dstate) {
        const int k4 = K / 4;
        for (int u = tid; u < C * k4; u += nthr) {  // Qg: row = token, 4 channels per half piece
          const int i = u / k4, k0 = 4 * (u - (u / k4) * k4);
          float x[4];
          KDA_UNROLL
          for (int j = 0; j < 4; ++j) {
            const size_t o = (size_t)i * ldq + k0 + j;
            x[j] = i < L ? sQn[o] * fexp(sGam[o]) : 0.f;
          }
          put_hilo4(tile, kTileQg + (size_t)(k0 >> 6) * 8192 + swz128((uint32_t)i, (uint32_t)(k0 & 63)), x);
        }
      }
    }
  });
  float* QFw = blk + b.qf;
  float* KFw = blk + b.kf;
  float* KBw = blk + b.kb;
  // The block-referenced operands of Aqk and P, in place in shared memory: QF = Q e^(Gamma -
  // rho_B), KF = K e^(Gamma - rho_B) and KB = K e^(rho_B - Gamma) (B the row's block), and
  // F_IB = e^(rho_I - rho_B) for B < I, so that Aqk[i][j] = sum_k QF_i KB_j F_IB and P[i][j] =
  // sum_k KF_i KB_j F_IB with I, B the blocks of i, j need no exponential per (i, j, k).  Any
  // exponent beyond 60 (QF, KB, F, or the product KB F = K e^(rho_I - Gamma_j)) sends the
  // chunk to the direct evaluation.  The three go to the workspace too, with the range flag.
  ex.phase([&](int tid, int nthr) {
    for (int u = tid; u < (NB * (NB - 1) / 2) * K; u += nthr) {
      const int pr = u / K, kk = u - pr * K;
      const int I = pr >= 3 ? (pr >= 6 ? 4 : 3) : (pr >= 1 ? 2 : 1);  // pr = I (I - 1) / 2 + B
      const int B = pr - I * (I - 1) / 2;
      const float d = sRho[(size_t)I * K + kk] - sRho[(size_t)B * K + kk];
      if (d > 60.f) ex.atomic_add(sFlag, 1.f);
      sF[u] = fexp(d);
    }
    for (int e = tid; e < L * K; e += nthr) {
      const int i = e / K, kk = e - (e / K) * K, B = i >> 4;
      const size_t o = (size_t)i * ldq + kk;
      const float g = sGam[o], rho = sRho[(size_t)B * K + kk];
      bool bad = g - rho > 60.f;
      for (int I = B; I < NB; ++I) bad = bad || sRho[(size_t)I * K + kk] - g > 60.f;
      if (bad) ex.atomic_add(sFlag, 1.f);
      const float f = fexp(g - rho), kv = sKn[o];
      const float qf = sQn[o] * f, kf = kv * f, kb = kv * fexp(rho - g);
      sQn[o] = qf;
      sKn[o] = kf;
      sGam[o] = kb;
      // the same rows for the gradient stage's e^(Gamma_i - Gamma_j) sums
      QFw[e] = qf;
      KFw[e] = kf;
      KBw[e] = kb;
    }
    for (int e = L * K + tid; e < C * K; e += nthr) QFw[e] = KFw[e] = KBw[e] = 0.f;
  });
  const int CB = C / 4;
  if (sFlag[0] == 0.f) {
    // Aqk (j <= i) and P (j < i) in 4 x 4 blocks: rows i of one 16-row block I, keys j of
    // block B, over the channels of the shared-memory operands.  Aqk's fp32 rows are read only by
    // the CUDA-core state-gradient stage; with it and the v products on the tensor cores the
    // slot receives dAqk instead, and Aqk leaves only as the operand tile.
    const bool aqk_rows = !(Exec::kTensorCores && p.tc_dstate && p.tc_vprod);
    ex.phase([&](int tid, int nthr) {
      for (int u = tid; u < CB * CB; u += nthr) {
        const int ib = u / CB, jb = u - (u / CB) * CB;
        float aq[4][4] = {}, ak[4][4] = {};
        if (jb <= ib && 4 * ib < L) {
          const int I = ib >> 2, B = jb >> 2;
          const float* fr = sF + (size_t)(B < I ? I * (I - 1) / 2 + B : 0) * K;
          const float* qr = sQn + (size_t)(4 * ib) * ldq;
          const float* kr = sKn + (size_t)(4 * ib) * ldq;
          const float* br = sGam + (size_t)(4 * jb) * ldq;
          KDA_UNROLL4
          for (int kk = 0; kk < K; ++kk) {
            const float f = B < I ? fr[kk] : 1.f;
            float qf[4], kf[4], kb[4];
            KDA_UNROLL
            for (int y = 0; y < 4; ++y) {
              qf[y] = qr[(size_t)y * ldq + kk];
              kf[y] = kr[(size_t)y * ldq + kk];
              kb[y] = br[(size_t)y * ldq + kk] * f;
            }
            KDA_UNROLL
            for (int y = 0; y < 4; ++y)
              KDA_UNROLL
              for (int x = 0; x < 4; ++x) {
                aq[y][x] = fmaf(qf[y], kb[x], aq[y][x]);
                ak[y][x] = fmaf(kf[y], kb[x], ak[y][x]);
              }
          }
        }
        for (int y = 0; y < 4; ++y) {
          float row[4];
          for (int x = 0; x < 4; ++x) {
            const int i = 4 * ib + y, j = 4 * jb + x;
            const size_t e = (size_t)i * C + j;
            row[x] = (i < L && j <= i) ? aq[y][x] : 0.f;
            if (aqk_rows) Aqk[e] = row[x];
            P[e] = (i < L && j < i) ? ak[y][x] : 0.f;
          }
          if (p.tc_dstate)  // the state-gradient stage's Aqk operand tile
            put_hilo4(tile_ptr(a, c, hv), kTileAqk + swz128((uint32_t)(4 * ib + y), (uint32_t)(4 * jb)),
                      row, kTileAqkLo);
        }
      }
    });
  } else {
    // exact path: every e^(Gamma_i - Gamma_j) evaluated directly
    ex.phase([&](int tid, int nthr) {
      for (int e = tid; e < C * C; e += nthr) {
        const int i = e / C, j = e - (e / C) * C;
        float sq = 0.f, sk = 0.f;
        if (i < L && j <= i) {
          const float* gi = Gam + (size_t)i * K;
          const float* gj = Gam + (size_t)j * K;
          const float* qi = Qn + (size_t)i * K;
          const float* ki = Kn + (size_t)i * K;
          const float* kj = Kn + (size_t)j * K;
          for (int kk = 0; kk < K; ++kk) {
            const float kd = kj[kk] * expf(gi[kk] - gj[kk]);
            sq = fmaf(qi[kk], kd, sq);
            sk = fmaf(ki[kk], kd, sk);
          }
        }
        Aqk[e] = sq;
        P[e] = j < i ? sk : 0.f;
      }
    });
  }
  // A = (I + Diag(beta) P)^-1 by forward substitution on the identity's columns, blocked by 16
  // rows; then W = A (beta e^Gamma K) and U = A (beta V) as one dense product over the
  // right-hand sides in shared memory; A^T goes to the workspace for the gradient stage
  const int ldA = C + 4;              // 16-byte rows; the transposed walk is a 4-way conflict
  float* sP = smem;                   // [C][C] beta_i P_ij
  float* sA = sP + (size_t)C * C;     // [C][ldA] the identity, then A
  float* sX = sA + (size_t)C * ldA;   // [C][K + V] the right-hand sides of W and U
  const int nrhs = K + V;
  ex.phase([&](int tid, int nthr) {
    if (tid == 0) blk[b.flag] = sFlag[0];
    batched<8>(tid, nthr, C * C, [&](int e) { return Be[e / C] * P[e]; }, [&](int e, float v) { sP[e] = v; });
    for (int e = tid; e < C * ldA; e += nthr) {
      const int i = e / ldA, cc = e - (e / ldA) * ldA;
      sA[e] = cc == i ? 1.f : 0.f;
    }
    if (vecK && (nrhs & 3) == 0) {  // W's rows by 16-byte asynchronous copies
      const int q = K / 4;
      for (int e = tid; e < C * q; e += nthr) {
        const int i = e / q, x4 = 4 * (e - (e / q) * q);
        ex.copy16(sX + (size_t)i * nrhs + x4, W + (size_t)i * K + x4);
      }
    } else {
      batched<8>(tid, nthr, C * K, [&](int e) { return W[e]; }, [&](int e, float v) {
        sX[(size_t)(e / K) * nrhs + (e - (e / K) * K)] = v;
      });
    }
    const int v4 = (V + 3) / 4;
    batched<4>(tid, nthr, C * v4, [&](int e) {  // beta V, four columns of v per element
      const int i = e / v4, c4 = 4 * (e - (e / v4) * v4);
      return i < L ? ld4i(a.v, a.dtype, ((size_t)(t0 + i) * HV + hv) * V, c4, V, vecV)
                   : F4{0.f, 0.f, 0.f, 0.f};
    }, [&](int e, const F4& x) {
      const int i = e / v4, c4 = 4 * (e - (e / v4) * v4);
      const float bt = i < L ? Be[i] : 0.f;
      for (int y = 0; y < 4 && c4 + y < V; ++y) sX[(size_t)i * nrhs + K + c4 + y] = bt * f4at(x, y);
    });
    ex.copy_wait();
  });
  // each block's rows solved within the block (one thread per column), then the later rows
  // updated with the block's solution in 4 x 4 tiles (every thread)
  for (int J = 0; J * 16 < L; ++J) {
    const int j0 = 16 * J, jend = j0 + 16 < L ? j0 + 16 : L;
    ex.phase([&](int tid, int nthr) {
      for (int col = tid; col < jend; col += nthr) {  // A is lower triangular: columns < jend
        for (int i = j0 + 1; i < jend; ++i) {
          const float* pr = sP + (size_t)i * C;
          float x = sA[(size_t)i * ldA + col];
          for (int j = j0; j < i; ++j) x = fmaf(-pr[j], sA[(size_t)j * ldA + col], x);
          sA[(size_t)i * ldA + col] = x;
        }
      }
    });
    if (jend >= L) break;
    ex.phase([&](int tid, int nthr) {
      const int nr4 = (L - jend + 3) / 4, nc4 = jend / 4;  // columns >= jend are still zero
      for (int u = tid; u < nr4 * nc4; u += nthr) {
        const int i0 = jend + 4 * (u / nc4), c0 = 4 * (u - (u / nc4) * nc4);
        float acc[4][4];
        KDA_UNROLL
        for (int y = 0; y < 4; ++y) {
          const F4 v = ld4(sA + (size_t)(i0 + y) * ldA + c0);
          KDA_UNROLL
          for (int x = 0; x < 4; ++x) acc[y][x] = f4at(v, x);
        }
        for (int j = j0; j < jend; ++j) {
          float pv[4];
          KDA_UNROLL
          for (int y = 0; y < 4; ++y) pv[y] = i0 + y < L ? sP[(size_t)(i0 + y) * C + j] : 0.f;
          const F4 xv = ld4(sA + (size_t)j * ldA + c0);
          KDA_UNROLL
          for (int y = 0; y < 4; ++y)
            KDA_UNROLL
            for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(-pv[y], f4at(xv, x), acc[y][x]);
        }
        KDA_UNROLL
        for (int y = 0; y < 4; ++y)
          if (i0 + y < L) st4(sA + (size_t)(i0 + y) * ldA + c0, acc[y]);
      }
    });
  }
  // W's fp32 rows are read only by the CUDA-core state stages (both state stages on the tensor
  // cores read the -W operand tile)
  const bool w_rows = !(Exec::kTensorCores && p.tc_states && p.tc_dstate);
  // [W | U] = A [beta e^Gamma K | beta V]: 4 x 4 tiles of (rows i, columns), sums over j <= i;
  // a warp's lanes share the row tile (the A words are broadcasts) and take consecutive column
  // quads; thread t pairs row tiles t' and CB - 1 - t' (long and short sums)
  ex.phase([&](int tid, int nthr) {
    const int nc4 = (nrhs + 3) / 4, CB4 = C / 4;
    const bool vec = (nrhs & 3) == 0;
    for (int u = tid; u < CB4 * nc4; u += nthr) {
      const int t = u / nc4, c0 = 4 * (u - t * nc4);
      const int ib = t < CB4 / 2 ? t : (CB4 + CB4 / 2 - 1 - t);
      const int r0 = 4 * ib;
      float acc[4][4];
      KDA_UNROLL
      for (int y = 0; y < 4; ++y)
        KDA_UNROLL
        for (int x = 0; x < 4; ++x) acc[y][x] = 0.f;
      const int jend = r0 + 4 < L ? r0 + 4 : L;
      KDA_UNROLL4
      for (int j = 0; j < jend; ++j) {
        float av[4];
        KDA_UNROLL
        for (int y = 0; y < 4; ++y) av[y] = r0 + y < L ? sA[(size_t)(r0 + y) * ldA + j] : 0.f;
        const F4 xv = lds4m(sX + (size_t)j * nrhs + c0, nrhs - c0, vec);
        KDA_UNROLL
        for (int y = 0; y < 4; ++y)
          KDA_UNROLL
          for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(av[y], f4at(xv, x), acc[y][x]);
      }
      const bool whole = c0 + 4 <= nrhs;
      KDA_UNROLL
      for (int y = 0; y < 4; ++y) {
        const size_t i = (size_t)(r0 + y);
        if (whole && c0 + 4 <= K && vecK) {
          if (w_rows) st4(W + i * K + c0, acc[y]);
          if (p.tc_states) {  // the state stage's -W operand tile
            const float nw[4] = {-acc[y][0], -acc[y][1], -acc[y][2], -acc[y][3]};
            put_hilo4(tile_ptr(a, c, hv), kTileNegW + (size_t)(c0 >> 6) * 8192 +
                                              swz128((uint32_t)i, (uint32_t)(c0 & 63)), nw);
          }
        } else if (whole && c0 >= K && vecV && ((c0 - K) & 3) == 0) {
          st4(U + i * V + (c0 - K), acc[y]);
        } else {
          for (int x = 0; x < 4 && c0 + x < nrhs; ++x) {
            const int col = c0 + x;
            if (col < K) W[i * K + col] = acc[y][x];
            else U[i * V + col - K] = acc[y][x];
          }
        }
      }
    }
  });
  ex.phase([&](int tid, int nthr) {
    float* ATi = blk + b.ati;  // ATi[c][i] = A[i][c]
    for (int e = tid; e < C * C; e += nthr) {
      const int cc = e / C, i = e - (e / C) * C;
      ATi[e] = (i < L && cc < L) ? sA[(size_t)i * ldA + cc] : 0.f;
    }
    // the state-gradient stage's Aqk tile was written with Aqk, except by the exact path
    if (p.tc_dstate && sFlag[0] != 0.f) {
      char* tile = tile_ptr(a, c, hv);
      const int c8 = C / 8;
      for (int u = tid; u < C * c8; u += nthr) {  // row = token, 8 tokens per piece
        const int i = u / c8, j0 = 8 * (u - (u / c8) * c8);
        const float* src = Aqk + (size_t)i * C + j0;
        const F4 x0 = ld4w(src, 0, 8, true), x1 = ld4w(src, 4, 8, true);
        const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        put_hilo8(tile, kTileAqk + swz128((uint32_t)i, (uint32_t)j0), x, kTileAqkLo);
      }
    }
  });
}

// ---- states: per (sequence, value head, V tile), chunks in order ------------------------
//
// Per chunk, W, Kg and the U tile are staged in shared memory once; V_new = U - W S is then
// computed in 2 x 4 register blocks (two rows, i and i + C/2, of four adjacent columns) and
// S <- Diag(e^gamma_C) S + Kg^T V_new in 4 x 4 blocks (four channels of four columns), every
// operand read as 16 bytes from shared memory.  K is padded to K4 (a multiple of 4) with zero
// rows, and W's rows are K4 + 4 floats apart so that the rows a warp reads fall in different
// banks.


template <class Exec>
KDA_BODY void states_body(Exec& ex, const Args& a, int64_t bid, float* smem) {
  const Plan& p = a.p;
  const int C = p.C, K = p.K, V = p.V, HV = p.HV;
  const int K4 = pad4(K), ldw = K4 + 4, half = C / 2;
  const int nvt = (V + kBV - 1) / kBV;
  const int vt = (int)(bid % nvt);
  const int hv = (int)((bid / nvt) % HV);
  const int n = (int)(bid / ((int64_t)nvt * HV));
  int64_t bos, eos, cfirst;
  if (!seq_range(a, n, bos, eos, cfirst)) {
    ex.flag(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Block& b = p.blk;
  float* sS = smem;                          // [K4][kBV] the state tile
  float* sVn = sS + (size_t)K4 * kBV;        // [C][kBV] V_new tile
  float* sW = sVn + (size_t)C * kBV;         // [C][ldw] W
  float* sKg = sW + (size_t)C * ldw;         // [C][K4] Kg
  float* sU = sKg + (size_t)C * K4;          // [C][kBV] U tile
  float* sD = sU + (size_t)C * kBV;          // [K4] e^gamma_C
  const int c0 = vt * kBV;
  const int nc = V - c0 < kBV ? V - c0 : kBV;  // columns of this tile
  const size_t sbase = ((size_t)n * HV + hv) * (size_t)K * V;
  ex.phase([&](int tid, int nthr) {
    for (int e = tid; e < K4 * kBV; e += nthr) {
      const int kk = e / kBV, cl = e - (e / kBV) * kBV;
      float s = 0.f;
      if (kk < K && cl < nc && a.h0 != nullptr)
        s = a.h0[sbase + (a.state_v_first ? (size_t)(c0 + cl) * K + kk : (size_t)kk * V + c0 + cl)];
      sS[e] = s;
    }
  });
  const int64_t nch = (eos - bos + C - 1) / C;
  for (int64_t ci = 0; ci < nch; ++ci) {
    const int64_t c = cfirst + ci;
    const int64_t rem = eos - (bos + ci * C);
    const int L = (int)(rem < C ? rem : C);
    const float* blk = block_ptr(a, c, hv);
    const float* W = blk + b.w;
    const float* U = blk + b.u;
    const float* Kg = blk + b.kg;
    const float* Dc = blk + b.decay;
    float* Vn = block_ptr(a, c, hv) + b.vn;
    float* hS = state_ptr(a, p.off_h, c, hv);
    // stage W, Kg, U, e^gamma_C (16-byte asynchronous copies where the rows allow them; the
    // rows past L of the workspace blocks are zero); the state before this chunk goes out
    ex.phase([&](int tid, int nthr) {
      if ((K & 3) == 0) {
        const int q = K4 / 4;
        for (int e = tid; e < C * q; e += nthr) {
          const int i = e / q, k4 = 4 * (e - (e / q) * q);
          ex.copy16(sW + (size_t)i * ldw + k4, W + (size_t)i * K + k4);
          ex.copy16(sKg + (size_t)i * K4 + k4, Kg + (size_t)i * K + k4);
        }
        for (int e = tid; e < q; e += nthr) ex.copy16(sD + 4 * e, Dc + 4 * e);
      } else {
        for (int e = tid; e < C * K4; e += nthr) {
          const int i = e / K4, kk = e - (e / K4) * K4;
          sW[(size_t)i * ldw + kk] = kk < K ? W[(size_t)i * K + kk] : 0.f;
          sKg[e] = kk < K ? Kg[(size_t)i * K + kk] : 0.f;
        }
        for (int kk = tid; kk < K4; kk += nthr) sD[kk] = kk < K ? Dc[kk] : 0.f;
      }
      if ((V & 3) == 0 && nc == kBV) {
        for (int e = tid; e < C * (kBV / 4); e += nthr) {
          const int i = e / (kBV / 4), x4 = 4 * (e - (e / (kBV / 4)) * (kBV / 4));
          ex.copy16(sU + (size_t)i * kBV + x4, U + (size_t)i * V + c0 + x4);
        }
      } else {
        for (int e = tid; e < C * kBV; e += nthr) {
          const int i = e / kBV, cl = e - (e / kBV) * kBV;
          sU[e] = cl < nc ? U[(size_t)i * V + c0 + cl] : 0.f;
        }
      }
      for (int e = tid; e < K * kBV; e += nthr) {
        const int kk = e / kBV, cl = e - (e / kBV) * kBV;
        if (cl < nc) hS[(size_t)kk * V + c0 + cl] = sS[e];
      }
      ex.copy_wait();
    });
    // V_new = U - W S: rows i and i + C/2, columns 4 g .. 4 g + 3
    ex.phase([&](int tid, int nthr) {
      for (int u = tid; u < half * (kBV / 4); u += nthr) {
        const int i0 = u / (kBV / 4), g = u - (u / (kBV / 4)) * (kBV / 4), i1 = i0 + half;
        float acc[2][4];
        {
          const F4 u0 = ld4(sU + (size_t)i0 * kBV + 4 * g), u1 = ld4(sU + (size_t)i1 * kBV + 4 * g);
          for (int x = 0; x < 4; ++x) { acc[0][x] = f4at(u0, x); acc[1][x] = f4at(u1, x); }
        }
        for (int kk = 0; kk < K4; kk += 4) {
          const F4 w0 = ld4(sW + (size_t)i0 * ldw + kk), w1 = ld4(sW + (size_t)i1 * ldw + kk);
          for (int y = 0; y < 4; ++y) {
            const F4 s = ld4(sS + (size_t)(kk + y) * kBV + 4 * g);
            const float a0 = f4at(w0, y), a1 = f4at(w1, y);
            for (int x = 0; x < 4; ++x) {
              acc[0][x] = fmaf(-a0, f4at(s, x), acc[0][x]);
              acc[1][x] = fmaf(-a1, f4at(s, x), acc[1][x]);
            }
          }
        }
        st4(sVn + (size_t)i0 * kBV + 4 * g, acc[0]);
        st4(sVn + (size_t)i1 * kBV + 4 * g, acc[1]);
        for (int r = 0; r < 2; ++r) {
          const int i = r == 0 ? i0 : i1;
          for (int x = 0; x < 4; ++x)
            if (4 * g + x < nc) Vn[(size_t)i * V + c0 + 4 * g + x] = acc[r][x];
        }
      }
    });
    // S <- Diag(e^gamma_C) S + Kg^T V_new: channels 4 q .. 4 q + 3, columns 4 g .. 4 g + 3
    ex.phase([&](int tid, int nthr) {
      for (int u = tid; u < (K4 / 4) * (kBV / 4); u += nthr) {
        const int q4 = u / (kBV / 4), g = u - (u / (kBV / 4)) * (kBV / 4);
        float acc[4][4];
        for (int y = 0; y < 4; ++y) {
          const F4 s = ld4(sS + (size_t)(4 * q4 + y) * kBV + 4 * g);
          const float d = sD[4 * q4 + y];
          for (int x = 0; x < 4; ++x) acc[y][x] = f4at(s, x) * d;
        }
        for (int i = 0; i < L; ++i) {
          const F4 kg = ld4(sKg + (size_t)i * K4 + 4 * q4), vn = ld4(sVn + (size_t)i * kBV + 4 * g);
          for (int y = 0; y < 4; ++y)
            for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(f4at(kg, y), f4at(vn, x), acc[y][x]);
        }
        for (int y = 0; y < 4; ++y) st4(sS + (size_t)(4 * q4 + y) * kBV + 4 * g, acc[y]);
      }
    });
  }
}

// ---- dstate: per (sequence, value head, V tile), chunks in reverse -----------------------
//
// Per chunk, Aqk, Kg, Qg, W and the dO tile are staged in shared memory once (Qg
// and W are read from the workspace directly when K is too large for all of them to fit);
// dV_new = Aqk^T dO + Kg dS' is computed in 2 x 4 register blocks and
// dS = Diag(e^gamma_C) dS' + Qg^T dO - W^T dV_new in 4 x 4 blocks.

// Whether dstate stages Qg and W in shared memory (everything fits in 200 KB).
KDA_HD bool dstate_stages_qw(int C, int K) {
  const size_t K4 = (size_t)pad4(K);
  const size_t base = K4 * kBV + 2 * (size_t)C * kBV + (size_t)C * (C + 4) + (size_t)C * (K4 + 4) + K4;
  return sizeof(float) * (base + 2 * (size_t)C * K4) <= 200u * 1024u;
}

template <class Exec>
KDA_BODY void dstate_body(Exec& ex, const Args& a, int64_t bid, float* smem) {
  const Plan& p = a.p;
  const int C = p.C, K = p.K, V = p.V, HV = p.HV;
  const int K4 = pad4(K), ldk = K4 + 4, lda = C + 4, half = C / 2;
  const bool stage_qw = dstate_stages_qw(C, K);
  const int nvt = (V + kBV - 1) / kBV;
  const int vt = (int)(bid % nvt);
  const int hv = (int)((bid / nvt) % HV);
  const int n = (int)(bid / ((int64_t)nvt * HV));
  int64_t bos, eos, cfirst;
  if (!seq_range(a, n, bos, eos, cfirst)) {
    ex.flag(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Block& b = p.blk;
  float* sD = smem;                          // [K4][kBV] gradient of the state after the chunk
  float* sDv = sD + (size_t)K4 * kBV;        // [C][kBV] dV_new
  float* sDo = sDv + (size_t)C * kBV;        // [C][kBV] dO
  float* sAt = sDo + (size_t)C * kBV;        // [C][lda] Aqk (row j, column i)
  float* sKg = sAt + (size_t)C * lda;        // [C][ldk] Kg
  float* sDc = sKg + (size_t)C * ldk;        // [K4] e^gamma_C
  float* sQg = sDc + K4;                     // [C][K4] Qg (if staged)
  float* sW = sQg + (size_t)C * K4;          // [C][K4] W (if staged)
  const int c0 = vt * kBV;
  const int nc = V - c0 < kBV ? V - c0 : kBV;
  const size_t sbase = ((size_t)n * HV + hv) * (size_t)K * V;
  ex.phase([&](int tid, int nthr) {
    for (int e = tid; e < K4 * kBV; e += nthr) {
      const int kk = e / kBV, cl = e - (e / kBV) * kBV;
      float d = 0.f;
      if (kk < K && cl < nc && a.d_final_state != nullptr)
        d = a.d_final_state[sbase + (a.state_v_first ? (size_t)(c0 + cl) * K + kk
                                                     : (size_t)kk * V + c0 + cl)];
      sD[e] = d;
    }
  });
  const int64_t nch = (eos - bos + C - 1) / C;
  for (int64_t ci = nch - 1; ci >= 0; --ci) {
    const int64_t c = cfirst + ci;
    const int64_t t0 = bos + ci * C;
    const int64_t rem = eos - t0;
    const int L = (int)(rem < C ? rem : C);
    const float* blk = block_ptr(a, c, hv);
    const float* Aqk = blk + b.aqk;
    const float* Kg = blk + b.kg;
    const float* Qg = blk + b.qg;
    const float* W = blk + b.w;
    const float* Dc = blk + b.decay;
    float* dVn = block_ptr(a, c, hv) + b.dvn;
    float* hD = state_ptr(a, p.off_dh, c, hv);
    // dS' of this chunk goes out; stage the dO tile, Aqk^T, Kg (Qg, W) and e^gamma_C
    ex.phase([&](int tid, int nthr) {
      for (int e = tid; e < K * kBV; e += nthr) {
        const int kk = e / kBV, cl = e - (e / kBV) * kBV;
        if (cl < nc) hD[(size_t)kk * V + c0 + cl] = sD[e];
      }
      for (int e = tid; e < C * kBV; e += nthr) {
        const int i = e / kBV, cl = e - (e / kBV) * kBV;
        sDo[e] = (i < L && cl < nc)
                     ? ld_in(a.d_o, a.dtype, ((size_t)(t0 + i) * HV + hv) * V + c0 + cl) : 0.f;
      }
      // Aqk row-major (row j, column i; zero above the diagonal and past L in the workspace)
      for (int e = tid; e < C * (C / 4); e += nthr) {
        const int j = e / (C / 4), i4 = 4 * (e - (e / (C / 4)) * (C / 4));
        ex.copy16(sAt + (size_t)j * lda + i4, Aqk + (size_t)j * C + i4);
      }
      if ((K & 3) == 0) {
        const int q = K4 / 4;
        for (int e = tid; e < C * q; e += nthr) {
          const int i = e / q, k4 = 4 * (e - (e / q) * q);
          ex.copy16(sKg + (size_t)i * ldk + k4, Kg + (size_t)i * K + k4);
          if (stage_qw) {
            ex.copy16(sQg + (size_t)i * K4 + k4, Qg + (size_t)i * K + k4);
            ex.copy16(sW + (size_t)i * K4 + k4, W + (size_t)i * K + k4);
          }
        }
        for (int e = tid; e < q; e += nthr) ex.copy16(sDc + 4 * e, Dc + 4 * e);
      } else {
        for (int e = tid; e < C * K4; e += nthr) {
          const int i = e / K4, kk = e - (e / K4) * K4;
          const bool in = kk < K;
          sKg[(size_t)i * ldk + kk] = in ? Kg[(size_t)i * K + kk] : 0.f;
          if (stage_qw) {
            sQg[e] = in ? Qg[(size_t)i * K + kk] : 0.f;
            sW[e] = in ? W[(size_t)i * K + kk] : 0.f;
          }
        }
        for (int kk = tid; kk < K4; kk += nthr) sDc[kk] = kk < K ? Dc[kk] : 0.f;
      }
      ex.copy_wait();
    });
    // dV_new = Aqk^T dO + Kg dS': rows i and i + C/2, columns 4 g .. 4 g + 3
    ex.phase([&](int tid, int nthr) {
      for (int u = tid; u < half * (kBV / 4); u += nthr) {
        const int i0 = u / (kBV / 4), g = u - (u / (kBV / 4)) * (kBV / 4), i1 = i0 + half;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int j = i0; j < L; ++j) {  // Aqk[j][i] is zero for j < i
          const F4 d = ld4(sDo + (size_t)j * kBV + 4 * g);
          const float a0 = sAt[(size_t)j * lda + i0], a1 = sAt[(size_t)j * lda + i1];
          for (int x = 0; x < 4; ++x) {
            acc[0][x] = fmaf(a0, f4at(d, x), acc[0][x]);
            acc[1][x] = fmaf(a1, f4at(d, x), acc[1][x]);
          }
        }
        for (int kk = 0; kk < K4; kk += 4) {
          const F4 k0 = ld4(sKg + (size_t)i0 * ldk + kk), k1 = ld4(sKg + (size_t)i1 * ldk + kk);
          for (int y = 0; y < 4; ++y) {
            const F4 s = ld4(sD + (size_t)(kk + y) * kBV + 4 * g);
            const float a0 = f4at(k0, y), a1 = f4at(k1, y);
            for (int x = 0; x < 4; ++x) {
              acc[0][x] = fmaf(a0, f4at(s, x), acc[0][x]);
              acc[1][x] = fmaf(a1, f4at(s, x), acc[1][x]);
            }
          }
        }
        st4(sDv + (size_t)i0 * kBV + 4 * g, acc[0]);
        st4(sDv + (size_t)i1 * kBV + 4 * g, acc[1]);
        for (int r = 0; r < 2; ++r) {
          const int i = r == 0 ? i0 : i1;
          for (int x = 0; x < 4; ++x)
            if (4 * g + x < nc) dVn[(size_t)i * V + c0 + 4 * g + x] = acc[r][x];
        }
      }
    });
    // dS = Diag(e^gamma_C) dS' + Qg^T dO - W^T dV_new: channels 4 q .. 4 q + 3, columns 4 g ..
    ex.phase([&](int tid, int nthr) {
      for (int u = tid; u < (K4 / 4) * (kBV / 4); u += nthr) {
        const int q4 = u / (kBV / 4), g = u - (u / (kBV / 4)) * (kBV / 4);
        float acc[4][4];
        for (int y = 0; y < 4; ++y) {
          const F4 s = ld4(sD + (size_t)(4 * q4 + y) * kBV + 4 * g);
          const float d = sDc[4 * q4 + y];
          for (int x = 0; x < 4; ++x) acc[y][x] = f4at(s, x) * d;
        }
        for (int i = 0; i < L; ++i) {
          float qg[4], w[4];
          if (stage_qw) {
            const F4 q = ld4(sQg + (size_t)i * K4 + 4 * q4), ww = ld4(sW + (size_t)i * K4 + 4 * q4);
            for (int y = 0; y < 4; ++y) { qg[y] = f4at(q, y); w[y] = f4at(ww, y); }
          } else {
            for (int y = 0; y < 4; ++y) {
              const int kk = 4 * q4 + y;
              qg[y] = kk < K ? Qg[(size_t)i * K + kk] : 0.f;
              w[y] = kk < K ? W[(size_t)i * K + kk] : 0.f;
            }
          }
          const F4 o = ld4(sDo + (size_t)i * kBV + 4 * g), dv = ld4(sDv + (size_t)i * kBV + 4 * g);
          for (int y = 0; y < 4; ++y)
            for (int x = 0; x < 4; ++x)
              acc[y][x] = fmaf(qg[y], f4at(o, x), fmaf(-w[y], f4at(dv, x), acc[y][x]));
        }
        for (int y = 0; y < 4; ++y) st4(sD + (size_t)(4 * q4 + y) * kBV + 4 * g, acc[y]);
      }
    });
  }
  if (a.dh0 != nullptr) {
    ex.phase([&](int tid, int nthr) {
      for (int e = tid; e < K * kBV; e += nthr) {
        const int kk = e / kBV, cl = e - (e / kBV) * kBV;
        if (cl < nc)
          a.dh0[sbase + (a.state_v_first ? (size_t)(c0 + cl) * K + kk : (size_t)kk * V + c0 + cl)] =
              sD[e];
      }
    });
  }
}

// ---- vprod: per (chunk c, value head hv), when tc_vprod -------------------------------
//
// The gradient stage's products over v (backward-propagation step 5): dQg = dO S^T,
// dW = -dV_new S^T, dKg = V_new dS'^T, dAqk = dO V_new^T (masked to j <= i < L) and the
// diagonal of S dS'^T, written to the block for the gradient stage.  On the GPU a tensor-core
// kernel (kda_bwd_tc.cu) computes them; this body, one output element per thread and step,
// is their plain statement, which the host emulation runs in its place.
template <class Exec>
KDA_BODY void vprod_body(Exec& ex, const Args& a, int64_t c, int hv, float* /*smem*/) {
  const Plan& p = a.p;
  const int C = p.C, K = p.K, V = p.V, HV = p.HV;
  int n, L;
  int64_t t0;
  if (!locate(a, c, n, t0, L)) {
    ex.flag(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Block& b = p.blk;
  float* blk = block_ptr(a, c, hv);
  const float* Vn = blk + b.vn;
  const float* dVn = blk + b.dvn;
  const float* S = state_ptr(a, p.off_h, c, hv);
  const float* dSp = state_ptr(a, p.off_dh, c, hv);
  auto dO = [&](int i, int v) {
    return i < L ? ld_in(a.d_o, a.dtype, ((size_t)(t0 + i) * HV + hv) * V + v) : 0.f;
  };
  ex.phase([&](int tid, int nthr) {
    for (int e = tid; e < C * K; e += nthr) {
      const int i = e / K, kk = e - (e / K) * K;
      float q = 0.f, w = 0.f, kg = 0.f;
      for (int v = 0; v < V; ++v) {
        const float s = S[(size_t)kk * V + v];
        q = fmaf(dO(i, v), s, q);
        w = fmaf(-dVn[(size_t)i * V + v], s, w);
        kg = fmaf(Vn[(size_t)i * V + v], dSp[(size_t)kk * V + v], kg);
      }
      blk[b.dq + e] = q;
      blk[b.y + e] = w;
      blk[b.dk + e] = kg;
    }
    for (int e = tid; e < C * C; e += nthr) {
      const int i = e / C, j = e - (e / C) * C;
      float d = 0.f;
      if (i < L && j <= i)
        for (int v = 0; v < V; ++v) d = fmaf(dO(i, v), Vn[(size_t)j * V + v], d);
      blk[b.aqk + e] = d;
    }
    for (int kk = tid; kk < K; kk += nthr) {
      float d = 0.f;
      for (int v = 0; v < V; ++v) d = fmaf(S[(size_t)kk * V + v], dSp[(size_t)kk * V + v], d);
      blk[b.dkg + kk] = d;
    }
  });
}

// ---- grads: per (chunk c, value head hv) -----------------------------------------------
//
// The chunk's dense products (dAqk = dO V_new^T, dQg = dO S^T, dW = -dV_new S^T,
// dKg = V_new dS'^T, A^T dA = X (beta V)^T + Y (beta e^Gamma K)^T) run in 4 x 4 register
// blocks over 16-byte loads.  The e^(Gamma_i - Gamma_j)-weighted sums of the Aqk and P
// gradients take every exponent from a per-16-row-block reference rho (Gamma at the block's
// middle row): e^(Gamma_r - Gamma_j) = e^(Gamma_r - rho_R) e^(rho_R - Gamma_j), so that one
// exponential serves a whole block instead of one per (row, channel, j) -- unless some
// exponent could leave [-inf, 60] (an in-block decay beyond 60 nat on either side of the
// middle row), in which case the chunk evaluates every e^(Gamma_i - Gamma_j) directly.


// SC, SK, SV: the chunk size and head dimensions as compile-time constants (0: the plan's),
// so that the index arithmetic of the common shape folds into shifts and multiplies.
template <int SC = 0, int SK = 0, int SV = 0, class Exec>
KDA_BODY void grads_body(Exec& ex, const Args& a, int64_t c, int hv, float* smem) {
  const Plan& p = a.p;
  const int C = SC ? SC : p.C, K = SK ? SK : p.K, V = SV ? SV : p.V;
  const int HV = p.HV;
  int n, L;
  int64_t t0;
  if (!locate(a, c, n, t0, L)) {
    ex.flag(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Block& b = p.blk;
  float* blk = block_ptr(a, c, hv);
  const float* Gam = blk + b.gam;
  const float* Qn = blk + b.qn;
  const float* Kn = blk + b.kn;
  const float* Qg = blk + b.qg;
  const float* Vn = blk + b.vn;
  const float* dVn = blk + b.dvn;
  const float* P = blk + b.p;
  const float* Be = blk + b.beta;
  const float* ATi = blk + b.ati;
  float* Y = blk + b.y;
  float* X = blk + b.x;
  float* dQ = blk + b.dq;
  float* dK = blk + b.dk;
  float* dGam = blk + b.dgam;
  float* dKG = blk + b.dkg;
  float* EK = blk + b.w;   // e^Gamma K (the W slot: W is not needed any more)
  const float* QF = blk + b.qf;  // the recompute stage's block-referenced rows
  const float* KF = blk + b.kf;
  const float* KB = blk + b.kb;
  const float* S = state_ptr(a, p.off_h, c, hv);
  const float* dSp = state_ptr(a, p.off_dh, c, hv);
  const int ldz = C + 1;                      // padded rows: the row-per-thread substitution
  const int lda = C + 4;                      // rows of the transposed tiles (16-byte aligned)
  float* sdAt = smem;                         // [C][lda] dAqk transposed: sdAt[j][i] = dAqk[i][j]
  float* sB = sdAt + (size_t)C * lda;         // [C] beta
  float* sDB = sB + C;                        // [C] gradient of beta (the value)
  float* sRed = sDB + C;                      // [kThreads] partial sums of dA_log
  float* sFlag = sRed + kThreads;             // [4] > 0: some block exponent out of range
  float* sTc = sFlag + 4;                     // [8] the tensor-core product's barrier
  float* sDgc = sFlag + 12;                   // [K4] diagonal of S dS'^T
  float* sRg = sDgc + pad4(K);                // the product slices' staging, then:
  float* sAt = sRg;                           // [C][C] A^T: sAt[j][i] = A[i][j]
  float* sAk = sRg;                           // the same region, for the key rows later
  float* sZ = sAk + (size_t)C * C;            // [C][ldz] A^T dA, then A^T dA A^T, then dP
  float* sT = sZ + (size_t)C * ldz;           // scratch (grads_scratch floats)
  float* sXY = sT;                            // [C][(V + K + 1) / 2] back substitution columns
  float* sZt = sT;                            // [C][lda] dP transposed (the scratch is free then)
  const int ncol = V + K, half_cols = (ncol + 1) / 2;
  const int K4 = pad4(K), CB = C / 4;
  const bool vecV = (V & 3) == 0, vecK = (K & 3) == 0;
  // rows of the inputs dO and v (only rows < L exist)
  auto in_row = [&](int i) { return ((size_t)(t0 + i) * HV + hv) * V; };

  // beta; the accumulators of the tiled products start at zero, or (products over v done by
  // their own stage) take that stage's dAqk and diag(S dS'^T)
  ex.phase([&](int tid, int nthr) {
    if (p.tc_vprod) {
      const float* dAqk = blk + b.aqk;  // rows read whole, written transposed
      batched<8>(tid, nthr, C * C, [&](int e) { return dAqk[e]; }, [&](int e, float v) {
        const int i = e / C, j = e - (e / C) * C;
        sdAt[(size_t)j * lda + i] = v;
      });
      for (int e = tid; e < C * (lda - C); e += nthr) {
        const int j = e / (lda - C), x = e - (e / (lda - C)) * (lda - C);
        sdAt[(size_t)j * lda + C + x] = 0.f;
      }
      for (int kk = tid; kk < K4; kk += nthr) sDgc[kk] = kk < K ? dKG[kk] : 0.f;
    } else {
      for (int e = tid; e < C * lda; e += nthr) sdAt[e] = 0.f;
      for (int kk = tid; kk < K4; kk += nthr) sDgc[kk] = 0.f;
    }
    for (int i = tid; i < C; i += nthr) sB[i] = Be[i];
    if (tid == 0) sFlag[0] = 0.f;
  });
  // The products over v in 32-column slices staged in shared memory (16-byte asynchronous
  // copies where the rows allow them): dAqk = dO V_new^T (into sdAt), dQg = dO S^T,
  // dW = -dV_new S^T, dKg = V_new dS'^T (partial sums in the dQ, Y, dK slots of the block,
  // read back and added per slice) and the diagonal of S dS'^T (gamma_C's gradient, sDgc).
  // Rows are 36 floats (nine 16-byte units) apart and a warp's lanes take consecutive rows, so
  // that the lanes' 16-byte loads fall in distinct banks.
  constexpr int SW = kGradSliceW, SL = kGradSliceLd;
  float* sS = sRg;                            // [K4][SL] S slice
  float* sDs = sS + (size_t)K4 * SL;          // [K4][SL] dS' slice
  float* sDv = sDs + (size_t)K4 * SL;         // [C][SL] dV_new slice
  float* sVn = sDv + (size_t)C * SL;          // [C][SL] V_new slice
  float* sDo = sVn + (size_t)C * SL;          // [C][SL] dO slice
  const int nvt = p.tc_vprod ? 0 : (V + SW - 1) / SW;
  for (int t = 0; t < nvt; ++t) {
    const int v0 = SW * t, w = V - v0 < SW ? V - v0 : SW;
    const bool async = vecV && w == SW;
    ex.phase([&](int tid, int nthr) {
      for (int e = tid; e < (2 * K4 + 2 * C) * (SW / 4); e += nthr) {  // 4-column pieces
        const int row = e / (SW / 4), c4 = 4 * (e - (e / (SW / 4)) * (SW / 4));
        const float* src;
        float* dst;
        if (row < K4) { src = row < K ? S + (size_t)row * V : nullptr; dst = sS + (size_t)row * SL; }
        else if (row < 2 * K4) {
          const int k = row - K4;
          src = k < K ? dSp + (size_t)k * V : nullptr;
          dst = sDs + (size_t)k * SL;
        } else if (row < 2 * K4 + C) {
          const int i = row - 2 * K4;
          src = dVn + (size_t)i * V;
          dst = sDv + (size_t)i * SL;
        } else {
          const int i = row - 2 * K4 - C;
          src = Vn + (size_t)i * V;
          dst = sVn + (size_t)i * SL;
        }
        if (src == nullptr) {
          const float z[4] = {0.f, 0.f, 0.f, 0.f};
          st4(dst + c4, z);
        } else if (async) {
          ex.copy16(dst + c4, src + v0 + c4);
        } else {
          const F4 x = ld4w(src, v0 + c4, V, false);
          const float y[4] = {x.x, x.y, x.z, x.w};
          st4(dst + c4, y);
        }
      }
      for (int e = tid; e < C * (SW / 4); e += nthr) {
        const int i = e / (SW / 4), c4 = 4 * (e - (e / (SW / 4)) * (SW / 4));
        const F4 x = i < L ? ld4i(a.d_o, a.dtype, in_row(i), v0 + c4, V, async)
                           : F4{0.f, 0.f, 0.f, 0.f};
        const float y[4] = {x.x, x.y, x.z, x.w};
        st4(sDo + (size_t)i * SL + c4, y);
      }
      ex.copy_wait();
    });
    ex.phase([&](int tid, int nthr) {
      // unit (ib, kb): rows 4 ib .. 4 ib + 3, channels kb + nkb x (x = 0..3)
      const int nkb = K4 / 4;
      for (int u = tid; u < CB * nkb; u += nthr) {
        const int ib = u / nkb, kb = u - (u / nkb) * nkb;
        float aq[4][4], aw[4][4], ak[4][4];
        for (int y = 0; y < 4; ++y)
          for (int x = 0; x < 4; ++x) {
            const int i = 4 * ib + y, kk = kb + nkb * x;
            const bool rd = t > 0 && kk < K;
            const size_t e = (size_t)i * K + kk;
            aq[y][x] = rd ? dQ[e] : 0.f;
            aw[y][x] = rd ? Y[e] : 0.f;
            ak[y][x] = rd ? dK[e] : 0.f;
          }
        for (int c = 0; c < SW; c += 4) {  // dQg and dW (both against S)
          F4 o[4], dv[4], s[4];
          for (int y = 0; y < 4; ++y) {
            o[y] = ld4(sDo + (size_t)(4 * ib + y) * SL + c);
            dv[y] = ld4(sDv + (size_t)(4 * ib + y) * SL + c);
            s[y] = ld4(sS + (size_t)(kb + nkb * y) * SL + c);
          }
          for (int y = 0; y < 4; ++y)
            for (int x = 0; x < 4; ++x) {
              aq[y][x] += dot4(o[y], s[x]);
              aw[y][x] -= dot4(dv[y], s[x]);
            }
        }
        for (int c = 0; c < SW; c += 4) {  // dKg
          F4 vn[4], ds[4];
          for (int y = 0; y < 4; ++y) {
            vn[y] = ld4(sVn + (size_t)(4 * ib + y) * SL + c);
            ds[y] = ld4(sDs + (size_t)(kb + nkb * y) * SL + c);
          }
          for (int y = 0; y < 4; ++y)
            for (int x = 0; x < 4; ++x) ak[y][x] += dot4(vn[y], ds[x]);
        }
        for (int y = 0; y < 4; ++y)
          for (int x = 0; x < 4; ++x) {
            const int i = 4 * ib + y, kk = kb + nkb * x;
            if (kk >= K) continue;
            const size_t e = (size_t)i * K + kk;
            dQ[e] = aq[y][x];
            Y[e] = aw[y][x];
            dK[e] = ak[y][x];
          }
      }
      for (int u = tid; u < CB * CB; u += nthr) {  // dAqk: rows 4 ib .., keys jb + CB x
        const int ib = u / CB, jb = u - (u / CB) * CB;
        float acc[4][4];
        for (int y = 0; y < 4; ++y)
          for (int x = 0; x < 4; ++x) acc[y][x] = sdAt[(size_t)(jb + CB * x) * lda + 4 * ib + y];
        for (int c = 0; c < SW; c += 4) {
          F4 o[4], vn[4];
          for (int y = 0; y < 4; ++y) {
            o[y] = ld4(sDo + (size_t)(4 * ib + y) * SL + c);
            vn[y] = ld4(sVn + (size_t)(jb + CB * y) * SL + c);
          }
          for (int y = 0; y < 4; ++y)
            for (int x = 0; x < 4; ++x) acc[y][x] += dot4(o[y], vn[x]);
        }
        for (int y = 0; y < 4; ++y)
          for (int x = 0; x < 4; ++x) {
            const int i = 4 * ib + y, j = jb + CB * x;
            sdAt[(size_t)j * lda + i] = (i < L && j <= i) ? acc[y][x] : 0.f;
          }
      }
      for (int kk = tid; kk < K; kk += nthr) {  // diagonal of S dS'^T
        float d = 0.f;
        for (int c = 0; c < SW; c += 4) d += dot4(ld4(sS + (size_t)kk * SL + c), ld4(sDs + (size_t)kk * SL + c));
        sDgc[kk] += d;
      }
    });
  }
  // the direct terms of dQg, dW, dKg; e^Gamma K for the A^T dA product
  // element: four consecutive channels of a row (one 16-byte load per array when K % 4 == 0).
  // Kg = Kn e^(Gamma_L-1 - Gamma) is formed again here exactly as the recompute stage forms
  // it (the same operands and operations, so the same bits) instead of being read back.
  struct Direct { F4 gi, dqg, dkg, qg, kn; };
  ex.phase([&](int tid, int nthr) {
    batched<8>(tid, nthr, C * C, [&](int e) { return ATi[e]; }, [&](int e, float v) { sAt[e] = v; });
    const int q4 = (K + 3) / 4;
    batched<3>(tid, nthr, C * q4, [&](int e) {
      const int i = e / q4, c4 = 4 * (e - (e / q4) * q4);
      const F4 z{0.f, 0.f, 0.f, 0.f};
      Direct d{z, z, z, z, z};
      if (i < L) {
        const size_t r = (size_t)i * K;
        d = Direct{ld4w(Gam + r, c4, K, vecK), ld4w(dQ + r, c4, K, vecK), ld4w(dK + r, c4, K, vecK),
                   ld4w(Qg + r, c4, K, vecK), ld4w(Kn + r, c4, K, vecK)};
      }
      return d;
    }, [&](int e, const Direct& d) {
      const int i = e / q4, c4 = 4 * (e - (e / q4) * q4);
      const F4 gl = ld4w(Gam + (size_t)(L - 1) * K, c4, K, vecK);  // cached: the same row for all
      float dq[4], dk[4], dg[4], dkg_kg[4], ekv[4];
      KDA_UNROLL
      for (int x = 0; x < 4; ++x) {
        dq[x] = dk[x] = dg[x] = dkg_kg[x] = ekv[x] = 0.f;
        if (i < L) {
          const float gi = f4at(d.gi, x), dqg = f4at(d.dqg, x), dkg = f4at(d.dkg, x);
          const float eg = fexp(gi), egl = fexp(f4at(gl, x) - gi);
          dq[x] = dqg * eg;
          dk[x] = dkg * egl;
          dkg_kg[x] = dkg * (f4at(d.kn, x) * egl);
          dg[x] = dqg * f4at(d.qg, x) - dkg_kg[x];
          ekv[x] = eg * f4at(d.kn, x);
        }
      }
      const size_t o = (size_t)i * K + c4;
      if (i >= L) sts4m(Y + o, dq, K - c4, vecK);  // rows past the chunk's end: zero
      sts4m(dQ + o, dq, K - c4, vecK);
      sts4m(dK + o, dk, K - c4, vecK);
      sts4m(dGam + o, dg, K - c4, vecK);
      sts4m(dKG + o, dkg_kg, K - c4, vecK);
      sts4m(EK + o, ekv, K - c4, vecK);
    });
  });
  // X = A^T dV_new, Y = A^T dW with A^T from the recompute stage (sAt): dense products over
  // the rows j >= i (A^T is upper triangular), in two halves of the V + K columns staged in
  // shared memory, 4 x 4 tiles of (rows, columns); a warp's lanes share the row tile (the A^T
  // words are broadcasts) and take consecutive column quads.  Thread t takes row tiles t' and
  // CB - 1 - t' of its two items, so that the long and short sums pair up.
  for (int part = 0; part < 2; ++part) {
    const int cbeg = part == 0 ? 0 : half_cols, cnt = part == 0 ? half_cols : ncol - half_cols;
    ex.phase([&](int tid, int nthr) {
      const bool onv = cbeg + cnt <= V, ony = cbeg >= V;
      const int s0 = onv ? cbeg : cbeg - V;  // first source column
      if (((onv && vecV) || (ony && vecK)) && (cnt & 3) == 0 && (s0 & 3) == 0) {
        // whole rows of one array: 16-byte asynchronous copies (dV_new rows >= L are zero)
        const int q = cnt / 4;
        for (int e = tid; e < C * q; e += nthr) {
          const int i = e / q, x4 = 4 * (e - (e / q) * q);
          float* dst = sXY + (size_t)i * cnt + x4;
          if (onv && i >= L) {
            const float z[4] = {0.f, 0.f, 0.f, 0.f};
            st4(dst, z);
          } else {
            ex.copy16(dst, onv ? dVn + (size_t)i * V + s0 + x4 : Y + (size_t)i * K + s0 + x4);
          }
        }
        ex.copy_wait();
      } else {
        batched<8>(tid, nthr, C * cnt, [&](int e) {
          const int i = e / cnt, col = cbeg + (e - (e / cnt) * cnt);
          return col < V ? (i < L ? dVn[(size_t)i * V + col] : 0.f) : Y[(size_t)i * K + col - V];
        }, [&](int e, float v) { sXY[e] = v; });
      }
    });
    ex.phase([&](int tid, int nthr) {
      const int nc4 = (cnt + 3) / 4;
      const bool vec = (cnt & 3) == 0;  // 16-byte rows: one load per four columns
      for (int u = tid; u < CB * nc4; u += nthr) {
        const int t = u / nc4, c0 = 4 * (u - t * nc4);
        const int ib = t < CB / 2 ? t : (CB + CB / 2 - 1 - t);
        const int r0 = 4 * ib;  // rows >= L come out zero (A^T's rows >= L are zero)
        float acc[4][4];
        KDA_UNROLL
        for (int y = 0; y < 4; ++y)
          KDA_UNROLL
          for (int x = 0; x < 4; ++x) acc[y][x] = 0.f;
        KDA_UNROLL4
        for (int j = r0; j < L; ++j) {
          float av[4];
          KDA_UNROLL
          for (int y = 0; y < 4; ++y) av[y] = sAt[(size_t)(r0 + y) * C + j];
          const F4 xv = lds4m(sXY + (size_t)j * cnt + c0, cnt - c0, vec);
          KDA_UNROLL
          for (int y = 0; y < 4; ++y)
            KDA_UNROLL
            for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(av[y], f4at(xv, x), acc[y][x]);
        }
        // X and dv = beta X; Y and its direct terms dK += beta Y e^Gamma, dGamma += beta Y
        // e^Gamma K (rows < L)
        const int col0 = cbeg + c0;
        const bool whole = c0 + 4 <= cnt;
        if (whole && col0 + 4 <= V && vecV && (col0 & 3) == 0) {
          KDA_UNROLL
          for (int y = 0; y < 4; ++y) {
            const size_t i = (size_t)(r0 + y);
            st4(X + i * V + col0, acc[y]);
            if (r0 + y < L) {
              const float bi = sB[r0 + y];
              const float d[4] = {bi * acc[y][0], bi * acc[y][1], bi * acc[y][2], bi * acc[y][3]};
              st4(a.dv + ((size_t)(t0 + i) * HV + hv) * V + col0, d);
            }
          }
        } else if (whole && col0 >= V && vecK && ((col0 - V) & 3) == 0) {
          const int k0 = col0 - V;
          F4 gv[4], dkv[4], ekv[4], dgv[4];
          KDA_UNROLL
          for (int y = 0; y < 4; ++y) {
            const size_t o = (size_t)(r0 + y < L ? r0 + y : 0) * K;
            gv[y] = ld4w(Gam + o, k0, K, true); dkv[y] = ld4w(dK + o, k0, K, true);
            ekv[y] = ld4w(EK + o, k0, K, true); dgv[y] = ld4w(dGam + o, k0, K, true);
          }
          KDA_UNROLL
          for (int y = 0; y < 4; ++y) {
            const size_t i = (size_t)(r0 + y);
            st4(Y + i * K + k0, acc[y]);
            if (r0 + y < L) {
              const float bi = sB[r0 + y];
              float nk[4], ng4[4];
              KDA_UNROLL
              for (int x = 0; x < 4; ++x) {
                const float t = bi * acc[y][x];
                nk[x] = f4at(dkv[y], x) + t * fexp(f4at(gv[y], x));
                ng4[x] = f4at(dgv[y], x) + t * f4at(ekv[y], x);
              }
              st4(dK + i * K + k0, nk);
              st4(dGam + i * K + k0, ng4);
            }
          }
        } else {
          for (int y = 0; y < 4; ++y) {
            const size_t i = (size_t)(r0 + y);
            for (int x = 0; x < 4 && c0 + x < cnt; ++x) {
              const int col = col0 + x;
              const float v = acc[y][x];
              if (col < V) {
                X[i * V + col] = v;
                if (r0 + y < L) a.dv[((size_t)(t0 + i) * HV + hv) * V + col] = sB[r0 + y] * v;
              } else {
                const size_t e = i * K + (col - V);
                Y[e] = v;
                if (r0 + y < L) {
                  const float t = sB[r0 + y] * v;
                  dK[e] += t * fexp(Gam[e]);
                  dGam[e] += t * EK[e];
                }
              }
            }
          }
        }
      }
    });
  }
  // A^T dA = X (beta V)^T + Y (beta e^Gamma K)^T over 64-column slices of v, then of k, staged
  // in shared memory and accumulated in sZ (lower blocks with the diagonal: its entries,
  // without beta, are the WY part of dbeta)
  if constexpr (Exec::kTensorCores && SC == 64 && SK == 128 && SV == 128) {
    // on the tensor cores: bf16 hi / lo operand tiles per 64-column slice in the scratch,
    // the accumulator in tensor memory, then sZ
    ex.zprod(sZ, ldz, sT, sTc, X, Y, a.v, in_row(0), (size_t)HV * V, a.dtype, EK, L, a.status);
  } else {
    constexpr int ZW = 64, SLZ = 68;    // slice width; padded rows (17 16-byte units apart)
    float* sA = sT;                     // [C][SLZ] X (or Y) slice
    float* sBt = sA + (size_t)C * SLZ;  // [C][SLZ] v (or e^Gamma K) slice
    const int ntv = (V + ZW - 1) / ZW, ntk = (K + ZW - 1) / ZW;
    for (int t = 0; t < ntv + ntk; ++t) {
      const bool onv = t < ntv;
      const int o0 = ZW * (onv ? t : t - ntv), len = onv ? V : K;
      const int w = len - o0 < ZW ? len - o0 : ZW;
      const bool async = (onv ? vecV : vecK) && w == ZW;
      ex.phase([&](int tid, int nthr) {
        for (int e = tid; e < C * (ZW / 4); e += nthr) {
          const int i = e / (ZW / 4), c4 = 4 * (e - (e / (ZW / 4)) * (ZW / 4));
          const float* ar = (onv ? X + (size_t)i * V : Y + (size_t)i * K);
          if (async) {
            ex.copy16(sA + (size_t)i * SLZ + c4, ar + o0 + c4);
          } else {
            const F4 x = ld4w(ar, o0 + c4, len, false);
            const float y[4] = {x.x, x.y, x.z, x.w};
            st4(sA + (size_t)i * SLZ + c4, y);
          }
          F4 bx;
          if (onv) {
            bx = i < L ? ld4i(a.v, a.dtype, in_row(i), o0 + c4, V, async) : F4{0.f, 0.f, 0.f, 0.f};
          } else {
            bx = ld4w(EK + (size_t)i * K, o0 + c4, K, async);
          }
          const float y[4] = {bx.x, bx.y, bx.z, bx.w};
          st4(sBt + (size_t)i * SLZ + c4, y);
        }
        ex.copy_wait();
      });
      ex.phase([&](int tid, int nthr) {
        for (int u = tid; u < CB * CB; u += nthr) {  // rows 4 ib .., columns jb + CB x
          const int ib = u / CB, jb = u - (u / CB) * CB;
          float acc[4][4];
          for (int y = 0; y < 4; ++y)
            for (int x = 0; x < 4; ++x)
              acc[y][x] = t > 0 ? sZ[(size_t)(4 * ib + y) * ldz + jb + CB * x] : 0.f;
          for (int c = 0; c < ZW; c += 4) {
            F4 xr[4], br[4];
            for (int y = 0; y < 4; ++y) {
              xr[y] = ld4(sA + (size_t)(4 * ib + y) * SLZ + c);
              br[y] = ld4(sBt + (size_t)(jb + CB * y) * SLZ + c);
            }
            for (int y = 0; y < 4; ++y)
              for (int x = 0; x < 4; ++x) acc[y][x] += dot4(xr[y], br[x]);
          }
          for (int y = 0; y < 4; ++y)
            for (int x = 0; x < 4; ++x) sZ[(size_t)(4 * ib + y) * ldz + jb + CB * x] = acc[y][x];
        }
      });
    }
  }
  // the diagonal is the WY part of dbeta; A^T dA = beta_j (...) strictly below it
  ex.phase([&](int tid, int nthr) {
    for (int e = tid; e < C * C; e += nthr) {
      const int i = e / C, j = e - (e / C) * C;
      float* z = sZ + (size_t)i * ldz + j;
      if (j == i) {
        sDB[i] = i < L ? *z : 0.f;
        *z = 0.f;
      } else {
        *z = (i < L && j < i) ? sB[j] * *z : 0.f;
      }
    }
  });
  // dAkk = -(A^T dA A^T) masked strictly lower: M[r][i] = sum_j Z[r][j] A[i][j] for i < r with
  // Z = A^T dA (sZ, strictly lower) and A lower triangular, so j < min(r, i + 1); 4 x 4 tiles
  // of (rows r, columns i), a warp's lanes taking consecutive column tiles of one row tile
  // (the Z words are broadcasts, the A^T rows 16-byte loads), into sM.  Then dP = beta dAkk
  // (into sZ) and dbeta += rowsum(dAkk P).
  float* sM = sT;  // [C][ldz]
  ex.phase([&](int tid, int nthr) {
    for (int u = tid; u < CB * CB; u += nthr) {
      const int rb = u / CB, ib = u - rb * CB;
      if (ib > rb || 4 * rb >= L) continue;
      float acc[4][4];
      KDA_UNROLL
      for (int y = 0; y < 4; ++y)
        KDA_UNROLL
        for (int x = 0; x < 4; ++x) acc[y][x] = 0.f;
      const int jend = 4 * ib + 4 < L ? 4 * ib + 4 : L;
      KDA_UNROLL4
      for (int j = 0; j < jend; ++j) {
        float zv[4];
        KDA_UNROLL
        for (int y = 0; y < 4; ++y) zv[y] = sZ[(size_t)(4 * rb + y) * ldz + j];
        const F4 av = ld4(sAt + (size_t)j * C + 4 * ib);  // A[4 ib ..][j]
        KDA_UNROLL
        for (int y = 0; y < 4; ++y)
          KDA_UNROLL
          for (int x = 0; x < 4; ++x) acc[y][x] = fmaf(zv[y], f4at(av, x), acc[y][x]);
      }
      KDA_UNROLL
      for (int y = 0; y < 4; ++y)
        KDA_UNROLL
        for (int x = 0; x < 4; ++x) sM[(size_t)(4 * rb + y) * ldz + 4 * ib + x] = acc[y][x];
    }
  });
  // (row r, one of nq column pieces) per thread; the pieces' dbeta sums meet in sRed and are
  // added at the start of the next phase
  const int nq = kThreads / C > 0 ? kThreads / C : 1, qw = (C + nq - 1) / nq;
  ex.phase([&](int tid, int nthr) {
    for (int u = tid; u < nq * C; u += nthr) {
      const int r = u / nq, q = u - (u / nq) * nq;
      float db = 0.f;
      if (r < L) {
        float* z = sZ + (size_t)r * ldz;
        const float* m = sM + (size_t)r * ldz;
        const int ib = q * qw, ie = ib + qw < r ? ib + qw : r;
        for (int i = ib; i < ie; ++i) {
          const float d = -m[i];
          db = fmaf(d, P[(size_t)r * C + i], db);
          z[i] = sB[r] * d;
        }
      }
      sRed[u] = db;
    }
  });
  // the recompute stage's rows K_j e^(rho_B - Gamma_j) (B the block of j) in shared memory:
  // rows below kbA in beta P's dead region, the rest after dP^T; its range flag; dP transposed
  const int kbA = (C * C) / K;
  auto kb_row = [&](int j) -> float* {
    return j < kbA ? sAk + (size_t)j * K : sT + (size_t)C * lda + (size_t)(j - kbA) * K;
  };
  ex.phase([&](int tid, int nthr) {
    for (int r = tid; r < L; r += nthr) {
      float db = 0.f;
      for (int q = 0; q < nq; ++q) db += sRed[(size_t)r * nq + q];
      sDB[r] += db;
    }
    for (int e = tid; e < C * C; e += nthr) {
      const int i = e / C, j = e - (e / C) * C;
      sZt[(size_t)j * lda + i] = sZ[(size_t)i * ldz + j];
    }
    // the recompute stage's K e^(rho_B - Gamma) rows and its range flag
    if (tid == 0) sFlag[0] = blk[b.flag];
    if (vecK) {
      const int q = K / 4;
      for (int e = tid; e < C * q; e += nthr) {
        const int j = e / q, x4 = 4 * (e - (e / q) * q);
        ex.copy16(kb_row(j) + x4, KB + (size_t)j * K + x4);
      }
      ex.copy_wait();
    } else {
      for (int e = tid; e < C * K; e += nthr) {
        const int j = e / K, kk = e - (e / K) * K;
        kb_row(j)[kk] = KB[e];
      }
    }
  });
  if (sFlag[0] == 0.f) {
    // the e^(Gamma_i - Gamma_j) terms of Aqk and P, one thread per (8-row half H of a 16-row
    // block R, four channels k), for the rows r of H:
    //   s1 = sum_{j<=r} dAqk[r][j] K_j e^(G_r - G_j)   s2 = sum_{j<r} dP[r][j] K_j e^(G_r - G_j)
    //   s3 = sum_{i>=r} dAqk[i][r] Q_i e^(G_i - G_r)   s4 = sum_{i>r} dP[i][r] K_i e^(G_i - G_r)
    // with e^(G_r - G_j) = e^(G_r - rho_R) e^(rho_R - rho_B) e^(rho_B - G_j) (B the block of j)
    // and e^(G_i - G_r) = e^(G_i - rho_I) e^(rho_I - rho_R) e^(rho_R - G_r) (I the block of i).
    // A warp's lanes share (R, H) and take consecutive channel quads, so that every dAqk and
    // dP value a lane loads is one broadcast word serving four channels.
    ex.phase([&](int tid, int nthr) {
      const int NB = (L + 15) >> 4, q4 = (K + 3) / 4;
      for (int u = tid; u < NB * 2 * q4; u += nthr) {
        const int rh = u / q4, k0 = 4 * (u - rh * q4);
        const int R = rh >> 1, r0 = 16 * R + 8 * (rh & 1);
        if (r0 >= L) continue;
        const int nr = L - r0 < 8 ? L - r0 : 8;  // rows r0 .. r0 + nr - 1
        auto mid = [&](int blk_) { return (16 * blk_ + 7) < L - 1 ? 16 * blk_ + 7 : L - 1; };
        const F4 rho = ld4w(Gam + (size_t)mid(R) * K, k0, K, vecK);
        float s[8][4], t[8][4];
KDA_UNROLL
        for (int y = 0; y < 8; ++y)
KDA_UNROLL
          for (int x = 0; x < 4; ++x) { s[y][x] = 0.f; t[y][x] = 0.f; }
        const int jend = r0 + nr;  // j <= r for the rows of this half
        for (int B = 0; B <= R; ++B) {
          F4 fb{1.f, 1.f, 1.f, 1.f};
          if (B < R) {
            const F4 gb = ld4w(Gam + (size_t)mid(B) * K, k0, K, vecK);
            fb = F4{fexp(rho.x - gb.x), fexp(rho.y - gb.y), fexp(rho.z - gb.z), fexp(rho.w - gb.w)};
          }
          const int j1 = 16 * B + 16 < jend ? 16 * B + 16 : jend;
          KDA_UNROLL4
          for (int j = 16 * B; j < j1; ++j) {
            const F4 kv = lds4m(kb_row(j) + k0, K - k0, vecK);
            const float ke[4] = {kv.x * fb.x, kv.y * fb.y, kv.z * fb.z, kv.w * fb.w};
            const float* da = sdAt + (size_t)j * lda + r0;  // dAqk[r0 ..][j], zero for r < j
            const float* dz = sZt + (size_t)j * lda + r0;   // dP[r0 ..][j], zero for r <= j
            const F4 a0 = ld4(da), a1 = ld4(da + 4), z0 = ld4(dz), z1 = ld4(dz + 4);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float zv[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
KDA_UNROLL
            for (int y = 0; y < 8; ++y)
KDA_UNROLL
              for (int x = 0; x < 4; ++x) {
                s[y][x] = fmaf(av[y], ke[x], s[y][x]);
                t[y][x] = fmaf(zv[y], ke[x], t[y][x]);
              }
          }
        }
        // rows of this half: e^(G_r - rho_R) applied, then dQ += s1, dK += s2,
        // dGamma += Q s1 + K s2 (the elements belong to this thread alone)
KDA_UNROLL
        for (int y0 = 0; y0 < 8; y0 += 2) {
          F4 gr[2], qv[2], kv[2], dq[2], dk[2], dg[2];
KDA_UNROLL
          for (int y = 0; y < 2; ++y) {
            const size_t o = (size_t)(r0 + (y0 + y < nr ? y0 + y : 0)) * K;
            gr[y] = ld4w(Gam + o, k0, K, vecK);
            qv[y] = ld4w(Qn + o, k0, K, vecK); kv[y] = ld4w(Kn + o, k0, K, vecK);
            dq[y] = ld4w(dQ + o, k0, K, vecK); dk[y] = ld4w(dK + o, k0, K, vecK);
            dg[y] = ld4w(dGam + o, k0, K, vecK);
          }
KDA_UNROLL
          for (int y = 0; y < 2; ++y) {
            if (y0 + y >= nr) continue;
            const size_t o = (size_t)(r0 + y0 + y) * K + k0;
            float nq[4], nk[4], ng4[4];
KDA_UNROLL
            for (int x = 0; x < 4; ++x) {
              const float f = fexp(f4at(gr[y], x) - f4at(rho, x));
              const float a1 = s[y0 + y][x] * f, a2 = t[y0 + y][x] * f;
              nq[x] = f4at(dq[y], x) + a1;
              nk[x] = f4at(dk[y], x) + a2;
              ng4[x] = f4at(dg[y], x) + (f4at(qv[y], x) * a1 + f4at(kv[y], x) * a2);
            }
            sts4m(dQ + o, nq, K - k0, vecK);
            sts4m(dK + o, nk, K - k0, vecK);
            sts4m(dGam + o, ng4, K - k0, vecK);
          }
        }
      }
    });
    // s3 + s4 (their factors are the same) over slices of C channels, whose rows Q e^(G -
    // rho_I) and K e^(G - rho_I) are first copied into shared memory (into the key rows'
    // region and dP's row-major tile, both dead by now): one thread per (4-row group, channel
    // quad of the slice), summing the rows i of every block I >= R, each scaled by
    // e^(rho_I - rho_R), then dK += s34 e^(rho_R - G_r), dGamma -= K s34 e^(rho_R - G_r)
    float* sQFs = sAk;  // [C][C]
    float* sKFs = sZ;   // [C][C] (of C x ldz)
    const int NBs = (L + 15) >> 4;
    auto mid_s = [&](int blk_) { return (16 * blk_ + 7) < L - 1 ? 16 * blk_ + 7 : L - 1; };
    for (int c0 = 0; c0 < K; c0 += C) {
      const int W = K - c0 < C ? K - c0 : C, wq = (W + 3) / 4;
      ex.phase([&](int tid, int nthr) {
        if (vecK) {
          for (int e = tid; e < C * wq; e += nthr) {
            const int i = e / wq, x4 = 4 * (e - (e / wq) * wq);
            ex.copy16(sQFs + (size_t)i * C + x4, QF + (size_t)i * K + c0 + x4);
            ex.copy16(sKFs + (size_t)i * C + x4, KF + (size_t)i * K + c0 + x4);
          }
          ex.copy_wait();
        } else {
          for (int e = tid; e < C * 4 * wq; e += nthr) {
            const int i = e / (4 * wq), x = e - (e / (4 * wq)) * (4 * wq);
            sQFs[(size_t)i * C + x] = x < W ? QF[(size_t)i * K + c0 + x] : 0.f;
            sKFs[(size_t)i * C + x] = x < W ? KF[(size_t)i * K + c0 + x] : 0.f;
          }
        }
      });
      ex.phase([&](int tid, int nthr) {
        for (int u = tid; u < (C / 4) * wq; u += nthr) {
          const int g4 = u / wq, xq = 4 * (u - (u / wq) * wq);
          const int r0 = 4 * g4, R = r0 >> 4, k0 = c0 + xq;
          if (r0 >= L) continue;
          const int nr = L - r0 < 4 ? L - r0 : 4;
          const F4 rho = ld4w(Gam + (size_t)mid_s(R) * K, k0, K, vecK);
          float sv[4][4];
KDA_UNROLL
          for (int y = 0; y < 4; ++y)
KDA_UNROLL
            for (int x = 0; x < 4; ++x) sv[y][x] = 0.f;
          for (int I = R; I < NBs; ++I) {
            F4 fi{1.f, 1.f, 1.f, 1.f};
            if (I > R) {
              const F4 gi = ld4w(Gam + (size_t)mid_s(I) * K, k0, K, vecK);
              fi = F4{fexp(gi.x - rho.x), fexp(gi.y - rho.y), fexp(gi.z - rho.z), fexp(gi.w - rho.w)};
            }
            const int ib = 16 * I > r0 ? 16 * I : r0, iend = 16 * I + 16 < L ? 16 * I + 16 : L;
            KDA_UNROLL4
            for (int i = ib; i < iend; ++i) {
              const F4 qf = ld4(sQFs + (size_t)i * C + xq), kf = ld4(sKFs + (size_t)i * C + xq);
              const float qe[4] = {qf.x * fi.x, qf.y * fi.y, qf.z * fi.z, qf.w * fi.w};
              const float ke[4] = {kf.x * fi.x, kf.y * fi.y, kf.z * fi.z, kf.w * fi.w};
KDA_UNROLL
              for (int y = 0; y < 4; ++y) {
                const float dav = sdAt[(size_t)(r0 + y) * lda + i];  // dAqk[i][r], zero for i < r
                const float dzv = sZt[(size_t)(r0 + y) * lda + i];   // dP[i][r], zero for i <= r
KDA_UNROLL
                for (int x = 0; x < 4; ++x) sv[y][x] = fmaf(dav, qe[x], fmaf(dzv, ke[x], sv[y][x]));
              }
            }
          }
          F4 gr[4], kv[4], dk[4], dg[4];
KDA_UNROLL
          for (int y = 0; y < 4; ++y) {
            const size_t o = (size_t)(r0 + (y < nr ? y : 0)) * K;
            gr[y] = ld4w(Gam + o, k0, K, vecK);
            kv[y] = ld4w(Kn + o, k0, K, vecK); dk[y] = ld4w(dK + o, k0, K, vecK);
            dg[y] = ld4w(dGam + o, k0, K, vecK);
          }
KDA_UNROLL
          for (int y = 0; y < 4; ++y) {
            if (y >= nr) continue;
            const size_t o = (size_t)(r0 + y) * K + k0;
            float nk[4], ng4[4];
KDA_UNROLL
            for (int x = 0; x < 4; ++x) {
              const float s34 = sv[y][x] * fexp(f4at(rho, x) - f4at(gr[y], x));
              nk[x] = f4at(dk[y], x) + s34;
              ng4[x] = f4at(dg[y], x) - f4at(kv[y], x) * s34;
            }
            sts4m(dK + o, nk, K - k0, vecK);
            sts4m(dGam + o, ng4, K - k0, vecK);
          }
        }
      });
    }
  } else {
    // exact fallback: every e^(Gamma_i - Gamma_j) evaluated directly, one thread per (row
    // r, channel k): r as the row index i (dQ, dK) and as the column index j (dK)
    ex.phase([&](int tid, int nthr) {
      for (int e = tid; e < C * K; e += nthr) {
        const int r = e / K, kk = e - (e / K) * K;
        if (r >= L) continue;
        const float gr = Gam[e];
        float s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f;
        for (int j = 0; j <= r; ++j) {
          const float kd = Kn[(size_t)j * K + kk] * expf(gr - Gam[(size_t)j * K + kk]);
          s1 = fmaf(sdAt[(size_t)j * lda + r], kd, s1);
          if (j < r) s2 = fmaf(sZ[(size_t)r * ldz + j], kd, s2);
        }
        for (int i = r; i < L; ++i) {
          const float ed = expf(Gam[(size_t)i * K + kk] - gr);
          s3 = fmaf(sdAt[(size_t)r * lda + i], Qn[(size_t)i * K + kk] * ed, s3);
          if (i > r) s4 = fmaf(sZ[(size_t)i * ldz + r], Kn[(size_t)i * K + kk] * ed, s4);
        }
        dQ[e] += s1;
        dK[e] += s2 + s3 + s4;
        dGam[e] += Qn[e] * s1 + Kn[e] * (s2 - s3 - s4);
      }
    });
  }
  // hand-over to the gate stage (through the X slot, dead by now): dbeta's WY and dAkk parts
  // and diag(S dS'^T)
  ex.phase([&](int tid, int nthr) {
    for (int i = tid; i < C; i += nthr) X[i] = sDB[i];
    for (int kk = tid; kk < K; kk += nthr) X[C + kk] = sDgc[kk];
  });
}

// ---- gate: per (chunk c, value head hv), after grads -----------------------------------
//
// The reverse cumsum of dGamma with the gamma_C terms, the gate activation's backward (dg,
// dA_log, ddt_bias), dbeta with the sigmoid's backward, and the L2-norm backward of q and k
// (dq, dk): element-wise phases over the gradient stage's dGamma, dK, dQ rows, in a kernel of
// their own so that their small shared memory and registers allow more blocks per SM.

inline size_t gate_scratch(const Plan& p) {
  const size_t C = (size_t)p.C, ng = (size_t)((p.K + 3) / 4);
  const size_t l2 = 2 * ng * (2 * C + 1) + 4 * C, half = 4 * (size_t)p.K;
  return l2 > half ? l2 : half;
}
inline size_t gate_smem(const Plan& p) {
  return sizeof(float) * ((size_t)p.C + (size_t)((p.K + 3) & ~3) + kThreads + gate_scratch(p));
}

template <int SC = 0, int SK = 0, int SV = 0, class Exec>
KDA_BODY void gate_body(Exec& ex, const Args& a, int64_t c, int hv, float* smem) {
  const Plan& p = a.p;
  const int C = SC ? SC : p.C, K = SK ? SK : p.K;
  const int H = p.H, HV = p.HV, h = hv / p.G;
  int n, L;
  int64_t t0;
  if (!locate(a, c, n, t0, L)) {
    ex.flag(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Block& b = p.blk;
  float* blk = block_ptr(a, c, hv);
  const float* dGam = blk + b.dgam;
  const float* dKG = blk + b.dkg;
  const float* Dc = blk + b.decay;
  const float* dQ = blk + b.dq;
  const float* dK = blk + b.dk;
  const float* X = blk + b.x;  // the gradient stage's hand-over
  float* sDB = smem;                      // [C] gradient of beta (the value)
  float* sDgc = sDB + C;                  // [K4] diagonal of S dS'^T
  float* sRed = sDgc + pad4(K);           // [kThreads] partial sums of dA_log
  float* sT = sRed + kThreads;            // scratch (gate_scratch floats)
  const bool has_alog = a.A_log != nullptr && a.gate_mode != KDA_GATE_PREGATED;
  const float a_exp = has_alog ? expf(a.A_log[hv]) : 1.0f;
  const bool vecK = (K & 3) == 0;
  ex.phase([&](int tid, int nthr) {
    for (int i = tid; i < C; i += nthr) sDB[i] = X[i];
    for (int kk = tid; kk < K; kk += nthr) sDgc[kk] = X[C + kk];
  });
  // reverse cumsum of dGamma (plus the gamma_C terms on the last row) and the gate backward,
  // with each channel's rows in two halves: first every half's sums of dGamma and of the
  // gamma_C terms, then each half's reverse cumsum from the total of the rows above it
  const int hrows = (L + 1) / 2;
  float* sHalf = sT;          // [2][K] sum of dGamma over the half's rows
  float* sKgh = sT + 2 * K;   // [2][K] sum of the gamma_C terms over the half's rows
  ex.phase([&](int tid, int nthr) {
    for (int u = tid; u < 2 * K; u += nthr) {
      const int hf = u / K, kk = u - (u / K) * K;
      const int i0 = hf * hrows, i1 = hf == 0 ? hrows : L;
      float sg = 0.f, sk = 0.f;
      for (int ib = i0; ib < i1; ib += 8) {  // eight rows' loads at a time
        float g8[8], k8[8];
        KDA_UNROLL
        for (int x = 0; x < 8; ++x) {
          const int i = ib + x < i1 ? ib + x : i0;
          g8[x] = dGam[(size_t)i * K + kk];
          k8[x] = dKG[(size_t)i * K + kk];
        }
        KDA_UNROLL
        for (int x = 0; x < 8; ++x)
          if (ib + x < i1) {
            sg += g8[x];
            sk += k8[x];
          }
      }
      sHalf[u] = sg;
      sKgh[u] = sk;
    }
  });
  ex.phase([&](int tid, int nthr) {
    const bool gated = a.gate_mode == KDA_GATE_PLAIN || a.gate_mode == KDA_GATE_SAFE;
    float alog_part = 0.f;
    for (int u = tid; u < 2 * K; u += nthr) {
      const int hf = u / K, kk = u - (u / K) * K;
      const int i0 = hf * hrows, i1 = hf == 0 ? hrows : L;
      if (i1 <= i0) continue;
      const float dgc = sDgc[kk] * Dc[kk] + (sKgh[kk] + sKgh[K + kk]);
      const float dt = (a.dt_bias != nullptr && a.gate_mode != KDA_GATE_PREGATED)
                           ? a.dt_bias[(size_t)hv * K + kk] : 0.f;
      float run = hf == 0 ? dgc + sHalf[K + kk] : dgc, dt_part = 0.f;
      for (int ie = i1 - 1; ie >= i0; ie -= 8) {  // eight rows at a time, loads first
        float dgm[8], gx[8];
        KDA_UNROLL
        for (int x = 0; x < 8; ++x) {
          const int i = ie - x;
          dgm[x] = i >= i0 ? dGam[(size_t)i * K + kk] : 0.f;
          gx[x] = (i >= i0 && gated) ? ld_in(a.g, a.dtype, ((size_t)(t0 + i) * HV + hv) * K + kk) : 0.f;
        }
        KDA_UNROLL
        for (int x = 0; x < 8; ++x) {
          const int i = ie - x;
          if (i < i0) continue;
          run += dgm[x];
          float dx = run;
          if (a.gate_mode == KDA_GATE_PLAIN) {
            const float xx = gx[x] + dt;
            dx = run * (-a_exp) * sigmoid_f(xx);
            alog_part = fmaf(run * (-a_exp), softplus_f(xx), alog_part);
          } else if (a.gate_mode == KDA_GATE_SAFE) {
            const float xx = gx[x] + dt;
            const float ds = run * a.lower_bound * dsigmoid_f(a_exp * xx);
            dx = ds * a_exp;
            alog_part = fmaf(ds * a_exp, xx, alog_part);
          }
          a.dg[((size_t)(t0 + i) * HV + hv) * K + kk] = dx;
          dt_part += dx;
        }
      }
      if (a.ddt_bias != nullptr) ex.atomic_add(a.ddt_bias + (size_t)hv * K + kk, dt_part);
    }
    sRed[tid] = alog_part;
  });
  // dA_log; dbeta; the L2-norm backward of q and k: sums (x^2, x d) over four-channel pieces
  // of every row, then per row, then every element with its row's factors
  const int ng = (K + 3) / 4, ldp = 2 * C + 1;  // padded: both access orders conflict-free
  float* sSS = sT;                              // [ng][ldp] sum x^2 of a piece
  float* sSD = sSS + (size_t)ng * ldp;          // [ng][ldp] sum x d of a piece
  float* sRowF = sSD + (size_t)ng * ldp;        // [2C][2]: 1 / |x|, sum x d / |x|
  struct XD { F4 x, d; };
  // piece u: row r (the q rows, then the k rows), channels 4 (u % ng) ..
  auto load_piece = [&](int u) {
    const int r = u / ng, c4 = 4 * (u - (u / ng) * ng), i = r < C ? r : r - C;
    XD v{{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (i < L) {
      v.d = ld4w((r < C ? dQ : dK) + (size_t)i * K, c4, K, vecK);
      if (a.qk_l2norm) v.x = ld4i(r < C ? a.q : a.k, a.dtype, ((size_t)(t0 + i) * H + h) * K, c4, K, vecK);
    }
    return v;
  };
  ex.phase([&](int tid, int nthr) {
    if (tid < 8 && a.dA_log != nullptr && has_alog) {  // eight partial sums, eight atomics
      float s = 0.f;
      for (int t = tid; t < nthr; t += 8) s += sRed[t];
      ex.atomic_add(a.dA_log + hv, s);
    }
    if (a.qk_l2norm) {
      batched<4>(tid, nthr, 2 * C * ng, load_piece, [&](int u, const XD& v) {
        const int r = u / ng, g = u - (u / ng) * ng;
        const float mul = r < C ? a.scale : 1.f;  // Q = scale * q / |q|
        sSS[(size_t)g * ldp + r] = dot4(v.x, v.x);
        sSD[(size_t)g * ldp + r] = dot4(v.x, F4{mul * v.d.x, mul * v.d.y, mul * v.d.z, mul * v.d.w});
      });
    }
    for (int i = tid; i < L; i += nthr) {
      float db = sDB[i];
      if (a.beta_sigmoid) {
        db *= (a.allow_neg_eigval ? 2.f : 1.f) *
              dsigmoid_f(ld_in(a.beta, a.dtype, (size_t)(t0 + i) * HV + hv));
      }
      a.dbeta[(size_t)(t0 + i) * HV + hv] = db;
    }
  });
  if (a.qk_l2norm) {
    ex.phase([&](int tid, int nthr) {
      for (int r = tid; r < 2 * C; r += nthr) {
        float ss = 0.f, sd = 0.f;
        for (int g = 0; g < ng; ++g) {
          ss += sSS[(size_t)g * ldp + r];
          sd += sSD[(size_t)g * ldp + r];
        }
        const float inv = 1.0f / sqrtf(ss + kL2Eps);
        sRowF[2 * r] = inv;
        sRowF[2 * r + 1] = inv * sd;
      }
    });
  }
  ex.phase([&](int tid, int nthr) {
    batched<4>(tid, nthr, 2 * C * ng, load_piece, [&](int u, const XD& v) {
      const int r = u / ng, c4 = 4 * (u - (u / ng) * ng), i = r < C ? r : r - C;
      if (i >= L) return;
      const float mul = r < C ? a.scale : 1.f;
      float* dst = (r < C ? a.dq : a.dk) + ((size_t)(t0 + i) * H + h) * K;
      const float inv = a.qk_l2norm ? sRowF[2 * r] : 0.f, t = a.qk_l2norm ? sRowF[2 * r + 1] : 0.f;
      float val[4];
      KDA_UNROLL
      for (int x = 0; x < 4; ++x) {
        const float d = mul * f4at(v.d, x);
        val[x] = a.qk_l2norm ? (d - f4at(v.x, x) * inv * t) * inv : d;
      }
      if (p.G == 1) {
        sts4m(dst + c4, val, K - c4, vecK);
      } else {
        KDA_UNROLL
        for (int x = 0; x < 4; ++x)
          if (c4 + x < K) ex.atomic_add(dst + c4 + x, val[x]);
      }
    });
  });
}

}  // namespace bwd
}  // namespace kda
