// Token-recurrent KDA forward: the method's recurrence taken one token at a time, with the
// state read from memory at the start and written back at the end.  This is the decode /
// short-prefill counterpart of the chunk path ("Reading Notes: Implementation Notes for
// KDA in FLA", section 1: fused_recurrent_kda next to chunk_kda), for one or a few tokens
// per sequence where the chunk form has nothing to amortise.
//
// Per token t of a sequence, for value head hv (q/k head hv / G):
//   alpha = exp(g'_t)                          g' the activated gate (section 2)
//   S <- Diag(alpha) S ;  p = S^T k ;  S <- S + beta k (v - p)^T ;  o_t = scale S^T q
// with q, k L2-normalised over K and beta = sigmoid(logit) (x2 with allow_neg_eigval) when
// the flags ask for it.
//
// Three kernels.  For K = V = 128 with the [K][V] state layout, the decode shape
// (recurrent_k128_bulk_kernel), the state moves in and out of shared memory by one bulk copy
// each.  Otherwise, for K <= 128 (recurrent_reg_kernel) the state lives in registers: one CTA
// per (sequence, value head, 64 columns of V), each column held by 4 adjacent lanes that own
// its K rows r = 4j + sub (32 fp32 values each), so that every reduction over K is two
// shuffles and a token costs one block barrier.  For larger K (recurrent_kernel) one CTA per
// (sequence, value head, 32 columns of V); 8 warps split the K rows of the 32-column state
// tile, which stays in shared memory in fp32.

#include "kda_internal.cuh"
#include "tc_common.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;  // V columns per CTA

__device__ __forceinline__ float warp_sum_all(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(const FwdArgs a) {
  extern __shared__ float smem[];
  const Plan& p = a.plan;
  const int K = p.K, V = p.V, HV = p.HV, H = p.H;
  const int nvt = (V + kTile - 1) / kTile;
  float* sS = smem;                       // [K][kTile] state tile
  float* sQ = sS + (size_t)K * kTile;     // [K] normalised, scaled query
  float* sK = sQ + K;                     // [K] normalised key
  float* sA = sK + K;                     // [K] decay alpha
  float* sRed = sA + K;                   // [kWarps][kTile] cross-warp partial sums
  float* sMisc = sRed + kWarps * kTile;   // [2 * kWarps] norm partials, [2] beta / flags

  const int vt = (int)(blockIdx.x % nvt);
  const int hv = (int)((blockIdx.x / nvt) % HV);
  const int n = (int)(blockIdx.x / ((unsigned)nvt * HV));
  const int h = hv / p.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int col = vt * kTile + lane;
  const bool cv = col < V;
  int64_t bos, eos;  // token range of sequence n
  if (p.varlen) {
    bos = a.cu_seqlens[n];
    eos = a.cu_seqlens[n + 1];
  } else {
    bos = (int64_t)n * p.T;
    eos = bos + p.T;
  }
  if (bos < 0 || eos < bos || eos > p.ntok) {
    if (tid == 0) flag_status(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Tin* gq = static_cast<const Tin*>(a.q);
  const Tin* gk = static_cast<const Tin*>(a.k);
  const Tin* gv = static_cast<const Tin*>(a.v);
  const Tin* gg = static_cast<const Tin*>(a.g);
  const Tin* gb = static_cast<const Tin*>(a.beta);
  Tin* go = static_cast<Tin*>(a.o);
  const size_t state_base = ((size_t)n * HV + hv) * (size_t)K * V;
  auto sidx = [&](int kk) {
    return state_base + (a.state_v_first ? (size_t)col * K + kk : (size_t)kk * V + col);
  };
  for (int kk = warp; kk < K; kk += kWarps)
    sS[kk * kTile + lane] = (a.h0 != nullptr && cv) ? a.h0[sidx(kk)] : 0.f;
  const float a_exp = (a.gate_mode != KDA_GATE_PREGATED && a.A_log != nullptr) ? expf(a.A_log[hv]) : 1.f;

  for (int64_t t = bos; t < eos; ++t) {
    // per-token vectors over K (thread i < K holds element i)
    float qi = 0.f, ki = 0.f;
    if (tid < K) {
      qi = to_f32(gq[(t * H + h) * (int64_t)K + tid]);
      ki = to_f32(gk[(t * H + h) * (int64_t)K + tid]);
      const float gi = to_f32(gg[(t * HV + hv) * (int64_t)K + tid]);
      const float dt = (a.dt_bias != nullptr && a.gate_mode != KDA_GATE_PREGATED)
                           ? a.dt_bias[(size_t)hv * K + tid] : 0.f;
      sA[tid] = expf(gate_exact(a.gate_mode, gi, a_exp, dt, a.lower_bound));
    }
    if (a.qk_l2norm) {
      const float sq = warp_sum_all(qi * qi), sk = warp_sum_all(ki * ki);
      if (lane == 0) {
        sMisc[warp] = sq;
        sMisc[kWarps + warp] = sk;
      }
    }
    if (tid == 0) {
      float b = to_f32(gb[t * HV + hv]);
      if (a.beta_sigmoid) b = (a.allow_neg_eigval ? 2.f : 1.f) * sigmoid_exact(b);
      sMisc[2 * kWarps] = b;
    }
    __syncthreads();
    if (tid < K) {
      float qn = a.scale, kn = 1.f;
      if (a.qk_l2norm) {
        float sq = 0.f, sk = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          sq += sMisc[w];
          sk += sMisc[kWarps + w];
        }
        qn *= rsqrtf(sq + 1e-6f);
        kn = rsqrtf(sk + 1e-6f);
      }
      sQ[tid] = qi * qn;
      sK[tid] = ki * kn;
    }
    __syncthreads();
    // S <- Diag(alpha) S and this warp's part of p = S^T k
    float pacc = 0.f;
    for (int kk = warp; kk < K; kk += kWarps) {
      const float s = sS[kk * kTile + lane] * sA[kk];
      sS[kk * kTile + lane] = s;
      pacc = fmaf(s, sK[kk], pacc);
    }
    sRed[warp * kTile + lane] = pacc;
    __syncthreads();
    float pv = 0.f;
    for (int w = 0; w < kWarps; ++w) pv += sRed[w * kTile + lane];
    const float vv = cv ? to_f32(gv[(t * HV + hv) * (int64_t)V + col]) : 0.f;
    const float u = sMisc[2 * kWarps] * (vv - pv);
    __syncthreads();  // sRed is rewritten below
    // S <- S + k u^T and this warp's part of o = scale S^T q (scale folded into sQ)
    float oacc = 0.f;
    for (int kk = warp; kk < K; kk += kWarps) {
      const float s = fmaf(sK[kk], u, sS[kk * kTile + lane]);
      sS[kk * kTile + lane] = s;
      oacc = fmaf(s, sQ[kk], oacc);
    }
    sRed[warp * kTile + lane] = oacc;
    __syncthreads();
    if (warp == 0 && cv) {
      float o = 0.f;
      for (int w = 0; w < kWarps; ++w) o += sRed[w * kTile + lane];
      go[(t * HV + hv) * (int64_t)V + col] = from_f32<Tin>(o);
    }
    __syncthreads();  // the next token rewrites sQ, sK, sA, sRed
  }
  if (a.final_state != nullptr && cv)
    for (int kk = warp; kk < K; kk += kWarps) a.final_state[sidx(kk)] = sS[kk * kTile + lane];
}

constexpr int kColLanes = 4;                   // lanes per V column
constexpr int kRegRows = 32;                   // K rows per lane (K <= kColLanes * kRegRows)
constexpr int kRegCols = kThreads / kColLanes;  // V columns per CTA

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 2) recurrent_reg_kernel(const FwdArgs a) {
  __shared__ float sQ[kColLanes * kRegRows], sK[kColLanes * kRegRows];  // raw q, k
  __shared__ float sA[kColLanes * kRegRows];                            // decay
  __shared__ float sPart[2][kWarps];                                       // sums of squares
  __shared__ float sBeta;
  const Plan& p = a.plan;
  const int K = p.K, V = p.V, HV = p.HV, H = p.H;
  const bool v_first = a.state_v_first;
  const int nvt = (V + kRegCols - 1) / kRegCols;
  const int vt = (int)(blockIdx.x % nvt);
  const int hv = (int)((blockIdx.x / nvt) % HV);
  const int n = (int)(blockIdx.x / ((unsigned)nvt * HV));
  const int h = hv / p.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane & (kColLanes - 1);  // rows kColLanes j + sub
  const int col = vt * kRegCols + warp * (32 / kColLanes) + lane / kColLanes;
  const bool cv = col < V;
  int64_t bos, eos;
  if (p.varlen) {
    bos = a.cu_seqlens[n];
    eos = a.cu_seqlens[n + 1];
  } else {
    bos = (int64_t)n * p.T;
    eos = bos + p.T;
  }
  if (bos < 0 || eos < bos || eos > p.ntok) {
    if (tid == 0) flag_status(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Tin* gq = static_cast<const Tin*>(a.q);
  const Tin* gk = static_cast<const Tin*>(a.k);
  const Tin* gv = static_cast<const Tin*>(a.v);
  const Tin* gg = static_cast<const Tin*>(a.g);
  const Tin* gb = static_cast<const Tin*>(a.beta);
  Tin* go = static_cast<Tin*>(a.o);
  const size_t state_base = ((size_t)n * HV + hv) * (size_t)K * V;
  auto sidx = [&](int r) {
    return state_base + (v_first ? (size_t)col * K + r : (size_t)r * V + col);
  };
  float S[kRegRows];
#pragma unroll
  for (int j = 0; j < kRegRows; ++j) {
    const int r = kColLanes * j + sub;
    S[j] = (a.h0 != nullptr && cv && r < K) ? a.h0[sidx(r)] : 0.f;
  }
  const float a_exp = (a.gate_mode != KDA_GATE_PREGATED && a.A_log != nullptr) ? expf(a.A_log[hv]) : 1.f;

  for (int64_t t = bos; t < eos; ++t) {
    // the token's q, k, decay and beta (thread r < K holds row r; rows past K stay 0)
    float qi = 0.f, ki = 0.f, ai = 1.f;
    if (tid < K) {
      qi = to_f32(gq[(t * H + h) * (int64_t)K + tid]);
      ki = to_f32(gk[(t * H + h) * (int64_t)K + tid]);
      const float gi = to_f32(gg[(t * HV + hv) * (int64_t)K + tid]);
      const float dt = (a.dt_bias != nullptr && a.gate_mode != KDA_GATE_PREGATED)
                           ? a.dt_bias[(size_t)hv * K + tid] : 0.f;
      ai = expf(gate_exact(a.gate_mode, gi, a_exp, dt, a.lower_bound));
    }
    if (tid < kColLanes * kRegRows) {
      sQ[tid] = qi;
      sK[tid] = ki;
      sA[tid] = ai;
    }
    const float vv = cv ? to_f32(gv[(t * HV + hv) * (int64_t)V + col]) : 0.f;
    if (a.qk_l2norm) {
      const float sq = warp_sum_all(qi * qi), sk = warp_sum_all(ki * ki);
      if (lane == 0) {
        sPart[0][warp] = sq;
        sPart[1][warp] = sk;
      }
    }
    if (tid == 0) {
      float b = to_f32(gb[t * HV + hv]);
      if (a.beta_sigmoid) b = (a.allow_neg_eigval ? 2.f : 1.f) * sigmoid_exact(b);
      sBeta = b;
    }
    __syncthreads();
    float qn = a.scale, kn = 1.f;
    if (a.qk_l2norm) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        sq += sPart[0][w];
        sk += sPart[1][w];
      }
      qn *= rsqrtf(sq + 1e-6f);
      kn = rsqrtf(sk + 1e-6f);
    }
    // S <- Diag(alpha) S and this lane's part of S^T k
    float pp = 0.f;
#pragma unroll
    for (int j = 0; j < kRegRows; ++j) {
      const int r = kColLanes * j + sub;
      S[j] *= sA[r];
      pp = fmaf(S[j], sK[r], pp);
    }
    pp += __shfl_xor_sync(0xffffffffu, pp, 1);
    pp += __shfl_xor_sync(0xffffffffu, pp, 2);
    const float ku = kn * (sBeta * (vv - kn * pp));  // S <- S + k_hat u^T, k_hat = kn k
    float oo = 0.f;
#pragma unroll
    for (int j = 0; j < kRegRows; ++j) {
      const int r = kColLanes * j + sub;
      S[j] = fmaf(sK[r], ku, S[j]);
      oo = fmaf(S[j], sQ[r], oo);
    }
    oo += __shfl_xor_sync(0xffffffffu, oo, 1);
    oo += __shfl_xor_sync(0xffffffffu, oo, 2);
    if (sub == 0 && cv) go[(t * HV + hv) * (int64_t)V + col] = from_f32<Tin>(qn * oo);
    __syncthreads();  // the next token rewrites the shared vectors
  }
  if (a.final_state != nullptr && cv) {
#pragma unroll
    for (int j = 0; j < kRegRows; ++j) {
      const int r = kColLanes * j + sub;
      if (r < K) a.final_state[sidx(r)] = S[j];
    }
  }
}

// K = V = 128 with the [K][V] state layout, the state in shared memory: one CTA per (sequence,
// value head) whose 64 KB state arrives by one bulk copy and leaves by one, so that the load /
// store units only carry the token's vectors; thread t owns column v = t % 128 over the rows of
// half t / 128, and a token is two passes over the state (S <- Diag(alpha) S with S^T k; then
// S <- S + k u^T with S^T q), the halves' column sums meeting in shared memory.  64 KB + 3 KB of
// shared memory: three CTAs per SM.
constexpr uint32_t kBulkStateBytes = 128 * 128 * 4;
constexpr int kBulkThreads = 512, kBulkSplit = kBulkThreads / 128, kBulkRows = 128 / kBulkSplit;
constexpr size_t kBulkSmem =
    kBulkStateBytes + sizeof(float) * (4 * 128 + 2 * kBulkSplit * 128 + 2 * kWarps + 4) + 16;
template <typename Tin>
__global__ void __launch_bounds__(kBulkThreads) recurrent_k128_bulk_kernel(const FwdArgs a) {
  constexpr int K = 128, V = 128;
  extern __shared__ __align__(16) float rsm[];
  float* sS = rsm;              // [K][V]
  float* sQ = sS + K * V;       // [K] q, k as loaded; alpha; v
  float* sK = sQ + K;
  float* sA = sK + K;
  float* sV = sA + K;
  float* sP = sV + V;                   // [kBulkSplit][V] partial sums of S^T k
  float* sO = sP + kBulkSplit * V;      // [kBulkSplit][V] partial sums of S^T q
  float* sPart = sO + kBulkSplit * V;   // [2][kWarps]
  float* sBeta = sPart + 2 * kWarps;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sBeta + 4);
  const Plan& p = a.plan;
  const int HV = p.HV, H = p.H;
  const int hv = (int)(blockIdx.x % HV);
  const int n = (int)(blockIdx.x / HV);
  const int h = hv / p.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v = tid & (V - 1), hf = tid >> 7;  // hf: this thread's group of kBulkRows rows
  int64_t bos, eos;
  if (p.varlen) {
    bos = a.cu_seqlens[n];
    eos = a.cu_seqlens[n + 1];
  } else {
    bos = (int64_t)n * p.T;
    eos = bos + p.T;
  }
  if (bos < 0 || eos < bos || eos > p.ntok) {
    if (tid == 0) flag_status(a.status, KDA_DEV_BAD_SEQLENS);
    return;
  }
  const Tin* gq = static_cast<const Tin*>(a.q);
  const Tin* gk = static_cast<const Tin*>(a.k);
  const Tin* gv = static_cast<const Tin*>(a.v);
  const Tin* gg = static_cast<const Tin*>(a.g);
  const Tin* gb = static_cast<const Tin*>(a.beta);
  Tin* go = static_cast<Tin*>(a.o);
  const size_t sbase = ((size_t)n * HV + hv) * (size_t)K * V;
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  bool pending = a.h0 != nullptr;  // the state's bulk copy has not been waited for yet
  if (pending) {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(bar, kBulkStateBytes);
      tc::bulk_g2s(sS, a.h0 + sbase, kBulkStateBytes, bar);
    }
  } else {
    for (int e = tid; e < K * V / 4; e += kBulkThreads)
      reinterpret_cast<float4*>(sS)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  bool ok = true;
  const float a_exp = (a.gate_mode != KDA_GATE_PREGATED && a.A_log != nullptr) ? expf(a.A_log[hv]) : 1.f;
  for (int64_t t = bos; t < eos; ++t) {
    if (tid < K) {
      const float qi = to_f32(gq[(t * H + h) * (int64_t)K + tid]);
      const float ki = to_f32(gk[(t * H + h) * (int64_t)K + tid]);
      const float gi = to_f32(gg[(t * HV + hv) * (int64_t)K + tid]);
      const float dt = (a.dt_bias != nullptr && a.gate_mode != KDA_GATE_PREGATED)
                           ? a.dt_bias[(size_t)hv * K + tid] : 0.f;
      sQ[tid] = qi;
      sK[tid] = ki;
      sA[tid] = expf(gate_exact(a.gate_mode, gi, a_exp, dt, a.lower_bound));
      sV[tid] = to_f32(gv[(t * HV + hv) * (int64_t)V + tid]);
      if (a.qk_l2norm) {
        const float sq = warp_sum_all(qi * qi), sk = warp_sum_all(ki * ki);
        if (lane == 0) {
          sPart[warp] = sq;
          sPart[kWarps + warp] = sk;
        }
      }
    }
    if (tid == 0) {
      float b = to_f32(gb[t * HV + hv]);
      if (a.beta_sigmoid) b = (a.allow_neg_eigval ? 2.f : 1.f) * sigmoid_exact(b);
      sBeta[0] = b;
    }
    if (pending) {  // the first token's vectors were loaded while the state arrived
      if (!tc::mbar_wait(bar, 0)) ok = false;
      pending = false;
    }
    __syncthreads();
    float qn = a.scale, kn = 1.f;
    if (a.qk_l2norm) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int w = 0; w < K / 32; ++w) {
        sq += sPart[w];
        sk += sPart[kWarps + w];
      }
      qn *= rsqrtf(sq + 1e-6f);
      kn = rsqrtf(sk + 1e-6f);
    }
    // S <- Diag(alpha) S and this half's rows of S^T k
    float acc = 0.f;
    const int r0 = kBulkRows * hf;
    float* col = sS + (size_t)r0 * V + v;
#pragma unroll 8
    for (int r = 0; r < kBulkRows; ++r) {
      const float s_ = col[(size_t)r * V] * sA[r0 + r];
      col[(size_t)r * V] = s_;
      acc = fmaf(s_, sK[r0 + r], acc);
    }
    sP[hf * V + v] = acc;
    __syncthreads();
    // u = kn beta (v - kn S^T k); S <- S + k u^T (k_hat u^T with k_hat = kn k); S^T q
    float pk = 0.f;
#pragma unroll
    for (int x = 0; x < kBulkSplit; ++x) pk += sP[x * V + v];
    const float u = kn * (sBeta[0] * (sV[v] - kn * pk));
    acc = 0.f;
#pragma unroll 8
    for (int r = 0; r < kBulkRows; ++r) {
      const float s_ = fmaf(sK[r0 + r], u, col[(size_t)r * V]);
      col[(size_t)r * V] = s_;
      acc = fmaf(s_, sQ[r0 + r], acc);
    }
    sO[hf * V + v] = acc;
    __syncthreads();
    if (tid < V) {
      float o = 0.f;
#pragma unroll
      for (int x = 0; x < kBulkSplit; ++x) o += sO[x * V + tid];
      go[(t * HV + hv) * (int64_t)V + tid] = from_f32<Tin>(qn * o);
    }
    __syncthreads();  // the next token rewrites the shared vectors
  }
  if (pending && !tc::mbar_wait(bar, 0)) ok = false;  // no token: the state passes through
  ok = __syncthreads_and(ok) != 0;
  if (!ok) {
    if (tid == 0) {
      flag_status(a.status, KDA_DEV_TIMEOUT);
      tc::mbar_wait(bar, 0, 100000000ull);  // the copy in flight lands before the CTA leaves
    }
    return;
  }
  if (a.final_state != nullptr) {
    tc::fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::bulk_s2g(a.final_state + sbase, sS, kBulkStateBytes);
      tc::bulk_commit();
      tc::bulk_wait_read0();
    }
  }
}

}  // namespace

size_t recurrent_smem_bytes(int K) {
  return sizeof(float) * ((size_t)K * kTile + 3 * (size_t)K + kWarps * kTile + 2 * kWarps + 2);
}

cudaError_t launch_recurrent(const FwdArgs& a, cudaStream_t s) {
  const Plan& p = a.plan;
  if (p.K <= kColLanes * kRegRows) {  // state in registers
    const int nvr = (p.V + kRegCols - 1) / kRegCols;
    const size_t blocks = (size_t)p.N * p.HV * nvr;
    if (blocks == 0) return cudaSuccess;
    if (p.K == 128 && p.V == 128 && !a.state_v_first) {  // the state by bulk copies
      const unsigned nb = (unsigned)((size_t)p.N * p.HV);
      cudaError_t e;
      if (a.dtype == KDA_BF16) {
        e = cudaFuncSetAttribute(recurrent_k128_bulk_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmem);
        if (e != cudaSuccess) return e;
        recurrent_k128_bulk_kernel<__nv_bfloat16><<<nb, kBulkThreads, kBulkSmem, s>>>(a);
      } else {
        e = cudaFuncSetAttribute(recurrent_k128_bulk_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmem);
        if (e != cudaSuccess) return e;
        recurrent_k128_bulk_kernel<float><<<nb, kBulkThreads, kBulkSmem, s>>>(a);
      }
      return cudaGetLastError();
    }
    if (a.dtype == KDA_BF16)
      recurrent_reg_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(a);
    else
      recurrent_reg_kernel<float><<<(unsigned)blocks, kThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
  const int nvt = (p.V + kTile - 1) / kTile;
  const size_t blocks = (size_t)p.N * p.HV * nvt;
  if (blocks == 0) return cudaSuccess;
  const size_t smem = recurrent_smem_bytes(p.K);
  cudaError_t e;
  if (a.dtype == KDA_BF16) {
    e = cudaFuncSetAttribute(recurrent_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    recurrent_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(recurrent_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    recurrent_kernel<float><<<(unsigned)blocks, kThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kda
