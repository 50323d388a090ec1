// fp32 CUDA-core path of the KDA chunk forward (used for fp32 inputs).
//
// Two kernels, following the chunk-parallel form of "Reading Notes: Implementation
// Notes for KDA in FLA" (forward pass):
//   simt_intra  one CTA per (chunk, value head), all chunks in parallel:
//               step 1 gate + chunk-local cumsum, step 2 Aqk / Akk with (I + Akk)^-1
//               applied by forward substitution, step 3 U, W, Qg, Kg.
//   simt_recur  one CTA per (sequence, value head, 32-wide V tile), chunks in order:
//               step 4 V_new = U - W S, S <- Diag(e^gamma_C) S + Kg^T V_new,
//               step 5 O = Qg S + Aqk V_new.
// Everything is fp32 with accurate expf; the intra-chunk decay factors are
// evaluated as exp(Gamma_i - Gamma_j) per element (exponent <= 0 on every
// unmasked entry), so no exponent-range trick is needed here.

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kIntraThreads = 256;
constexpr int kRecThreads = 256;
constexpr int kRecWarps = kRecThreads / 32;
constexpr int kBV = 32;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Float offsets of the intermediates inside one (chunk, value head) block.
struct InterView {
  float* qg;     // [C][K]  scale * q * e^Gamma
  float* kg;     // [C][K]  k * e^(gamma_C - Gamma)
  float* w;      // [C][K]  A Diag(beta) (e^Gamma * k)
  float* u;      // [C][V]  A Diag(beta) v
  float* aqk;    // [C][C]  scale * q k^T decayed, lower with diagonal
  float* decay;  // [K]     e^gamma_C
  __device__ InterView(const FwdArgs& a, int64_t c, int hv) {
    const Plan& p = a.plan;
    float* blk = reinterpret_cast<float*>(a.ws + p.off_inter) +
                 ((size_t)c * p.HV + hv) * (p.inter_block_bytes / sizeof(float));
    const size_t ck = (size_t)p.C * p.K;
    qg = blk; kg = blk + ck; w = blk + 2 * ck; u = blk + 3 * ck;
    aqk = u + (size_t)p.C * p.V;
    decay = aqk + (size_t)p.C * p.C;
  }
};

size_t intra_smem_bytes(int C, int K, int V) {
  const int KP = K + 1, XP = (K > V ? K : V) + 1;
  return sizeof(float) * ((size_t)C * XP + 2 * (size_t)C * KP + (size_t)C * C + C);
}

template <typename Tin>
__global__ void __launch_bounds__(kIntraThreads) simt_intra_kernel(const FwdArgs a) {
  extern __shared__ float smem[];
  const Plan& p = a.plan;
  const int C = p.C, K = p.K, V = p.V, HV = p.HV, H = p.H;
  const int KP = K + 1;                  // padded strides: column-wise access is conflict-free
  const int XP = (K > V ? K : V) + 1;
  float* sG = smem;                      // [C][XP]  gate -> Gamma; later beta*v -> U
  float* sQ = sG + (size_t)C * XP;       // [C][KP]  q (normed, scaled); later W
  float* sK = sQ + (size_t)C * KP;       // [C][KP]  k (normed)
  float* sA = sK + (size_t)C * KP;       // [C][C]   Akk0, strictly lower
  float* sB = sA + (size_t)C * C;        // [C]      beta

  const int64_t c = blockIdx.x;
  const int hv = blockIdx.y;
  const int h = hv / p.G;
  int n, L;
  int64_t t0;
  if (!locate_chunk(a, c, n, t0, L)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Tin* gq = static_cast<const Tin*>(a.q);
  const Tin* gk = static_cast<const Tin*>(a.k);
  const Tin* gv = static_cast<const Tin*>(a.v);
  const Tin* gg = static_cast<const Tin*>(a.g);
  const Tin* gb = static_cast<const Tin*>(a.beta);

  const bool has_alog = a.A_log != nullptr && a.gate_mode != KDA_GATE_PREGATED;
  const float a_exp = has_alog ? expf(a.A_log[hv]) : 1.0f;

  // Load: gate activation of g, q and k rows; padded rows (i >= L) are zero.
  for (int e = tid; e < C * K; e += kIntraThreads) {
    const int i = e / K, kk = e - (e / K) * K;
    float gval = 0.f, qv = 0.f, kv = 0.f;
    if (i < L) {
      const int64_t tok = t0 + i;
      const float dt = a.dt_bias ? a.dt_bias[(size_t)hv * K + kk] : 0.f;
      gval = gate_exact(a.gate_mode, to_f32(gg[(tok * HV + hv) * K + kk]), a_exp, dt,
                        a.lower_bound);
      qv = to_f32(gq[(tok * H + h) * K + kk]);
      kv = to_f32(gk[(tok * H + h) * K + kk]);
    }
    sG[i * XP + kk] = gval;
    sQ[i * KP + kk] = qv;
    sK[i * KP + kk] = kv;
  }
  for (int i = tid; i < C; i += kIntraThreads) {
    float b = 0.f;
    if (i < L) {
      b = to_f32(gb[(t0 + i) * HV + hv]);
      if (a.beta_sigmoid) b = (a.allow_neg_eigval ? 2.f : 1.f) * sigmoid_exact(b);
    }
    sB[i] = b;
  }
  __syncthreads();

  // Step 1: chunk-local cumsum of the log decay (one thread per channel).
  for (int kk = tid; kk < K; kk += kIntraThreads) {
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      acc += sG[i * XP + kk];
      sG[i * XP + kk] = acc;
    }
  }
  // L2 norm of q and k rows (one warp per row); scale folds into q.
  for (int r = warp; r < 2 * C; r += kIntraThreads / 32) {
    float* row = r < C ? sQ + r * KP : sK + (r - C) * KP;
    float mul = 1.f;
    if (a.qk_l2norm) {
      float ss = 0.f;
      for (int kk = lane; kk < K; kk += 32) ss += row[kk] * row[kk];
      ss = warp_sum(ss);
      mul = 1.0f / sqrtf(ss + 1e-6f);
    }
    if (r < C) mul *= a.scale;
    for (int kk = lane; kk < K; kk += 32) row[kk] *= mul;
  }
  __syncthreads();

  // Step 2: Aqk (lower with diagonal) and Akk0 = Diag(beta) (k k^T decayed, strictly lower).
  InterView out(a, c, hv);
  for (int e = tid; e < C * C; e += kIntraThreads) {
    const int i = e / C, j = e - (e / C) * C;
    float aqk = 0.f, akk = 0.f;
    if (i < L && j <= i) {
      const float* gi = sG + i * XP;
      const float* gj = sG + j * XP;
      const float* qi = sQ + i * KP;
      const float* ki = sK + i * KP;
      const float* kj = sK + j * KP;
      for (int kk = 0; kk < K; ++kk) {
        const float kd = kj[kk] * expf(gi[kk] - gj[kk]);
        aqk = fmaf(qi[kk], kd, aqk);
        akk = fmaf(ki[kk], kd, akk);
      }
      akk = (j < i) ? akk * sB[i] : 0.f;
    }
    out.aqk[e] = aqk;
    sA[e] = akk;
  }
  for (int kk = tid; kk < K; kk += kIntraThreads) out.decay[kk] = expf(sG[(L - 1) * XP + kk]);
  __syncthreads();

  // Step 3 (elementwise part): Qg, Kg to global; W's right-hand side Diag(beta) e^Gamma k into sQ.
  for (int e = tid; e < C * K; e += kIntraThreads) {
    const int i = e / K, kk = e - (e / K) * K;
    float qg = 0.f, kg = 0.f, rhs = 0.f;
    if (i < L) {
      const float gi = sG[i * XP + kk];
      const float eg = expf(gi);
      const float kv = sK[i * KP + kk];
      qg = sQ[i * KP + kk] * eg;
      kg = kv * expf(sG[(L - 1) * XP + kk] - gi);
      rhs = sB[i] * eg * kv;
    }
    out.qg[e] = qg;
    out.kg[e] = kg;
    sQ[i * KP + kk] = rhs;
  }
  __syncthreads();
  // U's right-hand side Diag(beta) v into sG (Gamma is no longer needed).
  for (int e = tid; e < C * V; e += kIntraThreads) {
    const int i = e / V, cc = e - (e / V) * V;
    float x = 0.f;
    if (i < L) x = sB[i] * to_f32(gv[((t0 + i) * HV + hv) * V + cc]);
    sG[i * XP + cc] = x;
  }
  __syncthreads();

  // Step 2/3: apply A = (I + Akk0)^-1 by forward substitution, one thread per column of [W | U].
  for (int col = tid; col < K + V; col += kIntraThreads) {
    float* X = col < K ? sQ + col : sG + (col - K);
    const int stride = col < K ? KP : XP;
    for (int i = 1; i < L; ++i) {
      float x = X[i * stride];
      const float* arow = sA + i * C;
      for (int j = 0; j < i; ++j) x = fmaf(-arow[j], X[j * stride], x);
      X[i * stride] = x;
    }
  }
  __syncthreads();
  for (int e = tid; e < C * K; e += kIntraThreads) {
    const int i = e / K, kk = e - (e / K) * K;
    out.w[e] = sQ[i * KP + kk];
  }
  for (int e = tid; e < C * V; e += kIntraThreads) {
    const int i = e / V, cc = e - (e / V) * V;
    out.u[e] = sG[i * XP + cc];
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kRecThreads) simt_recur_kernel(const FwdArgs a) {
  extern __shared__ float smem[];
  const Plan& p = a.plan;
  const int C = p.C, K = p.K, V = p.V, HV = p.HV;
  float* sS = smem;                     // [K][kBV]  state tile, fp32
  float* sVn = sS + (size_t)K * kBV;    // [C][kBV]  V_new tile
  const int nvt = (V + kBV - 1) / kBV;
  const int vt = (int)(blockIdx.x % nvt);
  const int hv = (int)((blockIdx.x / nvt) % HV);
  const int n = (int)(blockIdx.x / ((unsigned)nvt * HV));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int col = vt * kBV + lane;
  const bool cv = col < V;
  int64_t bos, eos, cfirst;
  if (!seq_range(a, n, bos, eos, cfirst)) return;
  Tin* go = static_cast<Tin*>(a.o);
  const size_t state_base = ((size_t)n * HV + hv) * (size_t)K * V;

  for (int kk = warp; kk < K; kk += kRecWarps) {
    const size_t si = a.state_v_first ? (size_t)col * K + kk : (size_t)kk * V + col;
    sS[kk * kBV + lane] = (a.h0 != nullptr && cv) ? a.h0[state_base + si] : 0.f;
  }
  __syncthreads();

  const int64_t nch = (eos - bos + C - 1) / C;
  for (int64_t ci = 0; ci < nch; ++ci) {
    const int64_t t0 = bos + ci * C;
    const int L = (int)((eos - t0) < C ? (eos - t0) : C);
    InterView in(a, cfirst + ci, hv);
    if (a.h_out != nullptr && cv) {  // the state before this chunk
      float* hc = a.h_out + ((size_t)(cfirst + ci) * HV + hv) * (size_t)K * V;
      for (int kk = warp; kk < K; kk += kRecWarps)
        hc[a.state_v_first ? (size_t)col * K + kk : (size_t)kk * V + col] = sS[kk * kBV + lane];
    }
    float preg[64 / kRecWarps];
    // Step 4, first half and step 5, first half: both read S_{t-1}.
#pragma unroll
    for (int r = 0; r < 64 / kRecWarps; ++r) {
      const int i = warp + kRecWarps * r;
      preg[r] = 0.f;
      if (i < L) {
        float vn = cv ? in.u[(size_t)i * V + col] : 0.f;
        float pq = 0.f;
        const float* wr = in.w + (size_t)i * K;
        const float* qr = in.qg + (size_t)i * K;
        for (int kk = 0; kk < K; ++kk) {
          const float s = sS[kk * kBV + lane];
          vn = fmaf(-__ldg(wr + kk), s, vn);
          pq = fmaf(__ldg(qr + kk), s, pq);
        }
        sVn[i * kBV + lane] = vn;
        preg[r] = pq;
      }
    }
    __syncthreads();
    // Step 5: O = Qg S_{t-1} + Aqk V_new.
#pragma unroll
    for (int r = 0; r < 64 / kRecWarps; ++r) {
      const int i = warp + kRecWarps * r;
      if (i < L) {
        float ov = preg[r];
        const float* ar = in.aqk + (size_t)i * C;
        for (int j = 0; j <= i; ++j) ov = fmaf(__ldg(ar + j), sVn[j * kBV + lane], ov);
        if (cv) go[((t0 + i) * HV + hv) * (int64_t)V + col] = from_f32<Tin>(ov);
      }
    }
    // Step 4: S <- Diag(e^gamma_C) S + Kg^T V_new.
    for (int kk = warp; kk < K; kk += kRecWarps) {
      float s = sS[kk * kBV + lane] * __ldg(in.decay + kk);
      for (int i = 0; i < L; ++i) s = fmaf(__ldg(in.kg + (size_t)i * K + kk), sVn[i * kBV + lane], s);
      sS[kk * kBV + lane] = s;
    }
    __syncthreads();
  }
  if (a.final_state != nullptr && cv)
    for (int kk = warp; kk < K; kk += kRecWarps)
      a.final_state[state_base + (a.state_v_first ? (size_t)col * K + kk : (size_t)kk * V + col)] =
          sS[kk * kBV + lane];
}

// Varlen: chunk offsets cs[n] = sum_{m<n} ceil(len_m / C), one block.
__global__ void __launch_bounds__(1024) chunk_table_kernel(const FwdArgs a) {
  const Plan& p = a.plan;
  const int N = p.N;
  int64_t* cs = reinterpret_cast<int64_t*>(a.ws + p.off_chunk_table);
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = min(N, (int)threadIdx.x * per), hi = min(N, lo + per);
  int64_t local = 0;
  bool bad = false;
  for (int m = lo; m < hi; ++m) {
    const int64_t len = a.cu_seqlens[m + 1] - a.cu_seqlens[m];
    bad |= len < 0;
    local += len > 0 ? (len + p.C - 1) / p.C : 0;
  }
  // exclusive block scan of `local`
  __shared__ int64_t warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int64_t t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  int64_t run = (incl - local) + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int m = lo; m < hi; ++m) {
    cs[m] = run;
    const int64_t len = a.cu_seqlens[m + 1] - a.cu_seqlens[m];
    run += len > 0 ? (len + p.C - 1) / p.C : 0;
  }
  if (threadIdx.x == blockDim.x - 1) {
    cs[N] = run;
    if (run != p.nct || a.cu_seqlens[0] != 0 || a.cu_seqlens[N] > p.ntok) bad = true;
  }
  if (bad) flag_status(a.status, KDA_DEV_BAD_SEQLENS);
}

}  // namespace

size_t simt_inter_block_bytes(int C, int K, int V) {
  const size_t f = (size_t)C * (3 * (size_t)K + V + C) + K;
  return (f * sizeof(float) + 255) / 256 * 256;
}

cudaError_t zero_uncovered_rows(const FwdArgs& a, cudaStream_t s) {
  const Plan& p = a.plan;
  if (p.tok_end >= p.ntok) return cudaSuccess;
  const size_t row = (size_t)p.HV * p.V * (a.dtype == KDA_BF16 ? 2 : 4);
  return cudaMemsetAsync(static_cast<char*>(a.o) + (size_t)p.tok_end * row, 0,
                         (size_t)(p.ntok - p.tok_end) * row, s);
}

// The varlen chunk table, and the rows of o past the last sequence set to zero (the
// first stage of every varlen schedule).
cudaError_t launch_chunk_table(const FwdArgs& a, cudaStream_t s) {
  cudaError_t e = zero_uncovered_rows(a, s);
  if (e != cudaSuccess) return e;
  chunk_table_kernel<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_simt_intra(const FwdArgs& a, cudaStream_t s) {
  const Plan& p = a.plan;
  if (p.nct == 0) return cudaSuccess;
  const size_t smem = intra_smem_bytes(p.C, p.K, p.V);
  const dim3 grid((unsigned)p.nct, (unsigned)p.HV);
  cudaError_t e;
  if (a.dtype == KDA_F32) {
    e = cudaFuncSetAttribute(simt_intra_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    simt_intra_kernel<float><<<grid, kIntraThreads, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(simt_intra_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    simt_intra_kernel<__nv_bfloat16><<<grid, kIntraThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_simt_recur(const FwdArgs& a, cudaStream_t s) {
  const Plan& p = a.plan;
  const size_t smem = sizeof(float) * ((size_t)p.K * kBV + (size_t)p.C * kBV);
  // one CTA per (sequence, value head, V tile), V tile fastest so that the tiles of
  // one head run together and share the intermediates through L2
  const dim3 grid((unsigned)((size_t)((p.V + kBV - 1) / kBV) * p.HV * p.N));
  if (a.dtype == KDA_F32)
    simt_recur_kernel<float><<<grid, kRecThreads, smem, s>>>(a);
  else
    simt_recur_kernel<__nv_bfloat16><<<grid, kRecThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kda
