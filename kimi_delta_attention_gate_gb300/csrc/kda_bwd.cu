// GPU kernels and C entry points of the KDA backward pass (include/kda_bwd.h).  The stage
// bodies live in kda_bwd.cuh; here each phase is one thread's share of the work followed
// by a block barrier.

#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "kda_bwd.cuh"
#include "kda_internal.cuh"
#include "tc_common.cuh"

namespace kda {

unsigned int* device_status_word();  // kda_api.cu

namespace bwd {
namespace {

// fp32 pair -> bf16 hi / lo pairs (x = hi + lo to about 2^-16)
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

struct GpuExec {
  static constexpr bool kTensorCores = true;
  // zprod's 64-column tensor-memory accumulator, allocated by the kernel when it starts: a
  // block that allocated in its middle would wait for the other block resident on the SM
  // until that one had allocated and relinquished its allocation permit too
  uint32_t tmem_base = 0;
  template <class F>
  __device__ __forceinline__ void phase(F&& f) {
    f((int)threadIdx.x, (int)blockDim.x);
    __syncthreads();
  }
  __device__ __forceinline__ void atomic_add(float* p, float x) { atomicAdd(p, x); }
  __device__ __forceinline__ void flag(unsigned int* s, unsigned int bits) { atomicOr(s, bits); }
  // 16 bytes global -> shared without a round trip through registers (both 16-byte aligned);
  // complete once copy_wait() has returned and the phase's barrier has passed
  __device__ __forceinline__ void copy16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
  }
  // close this thread's group of copies issued so far (they may stay in flight across phases)
  __device__ __forceinline__ void copy_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
  // wait for every copy this thread has issued
  __device__ __forceinline__ void copy_wait() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  }

  // Z = X V^T + Y (e^Gamma K)^T for chunk 64, K = V = 128 on the tensor cores (every thread of
  // the block; called outside a phase): per 64-column slice of v, then of k, the rows of X
  // (or Y) and of v (or e^Gamma K) become bf16 hi / lo tiles in the 128-byte-swizzled K-major
  // layout (v in bf16 is exact: its high part alone), one thread issues the M = 64, N = 64
  // MMAs (hi hi + lo hi + hi lo) into a tensor-memory accumulator, and the block waits for
  // them before the next slice's tiles; then the accumulator's rows go to sZ.  scratch: at
  // least 33 KB; sTc: 32 bytes (barrier); the accumulator: tmem_base.
  __device__ void zprod(float* sZ, int ldz, float* scratch, float* sTc, const float* X,
                        const float* Y, const void* v_in, size_t v_row0, size_t v_stride,
                        int dtype, const float* EK, int L, unsigned int* status) {
    using namespace tc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t* tiles = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(scratch) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sTc);
    if (tid == 0) {
      mbar_init(bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t t_ah = smem_u32(tiles), t_al = t_ah + 8192u, t_bh = t_ah + 16384u,
                   t_bl = t_ah + 24576u;
    const bool v_exact = dtype == KDA_BF16;
    bool ok = true;
    int open = -1;  // (thread 0) the slice whose MMA group is issued and not yet seen done
    for (int s = 0; s < 4 && ok; ++s) {
      const bool onv = s < 2;
      const int o0 = 64 * (s & 1);
#pragma unroll
      for (int it = 0; it < 2; ++it) {  // rows r, 8-column groups g: 512 items
        const int u = tid + 256 * it, r = u >> 3, g = u & 7;
        const uint32_t off = swz128((uint32_t)r, (uint32_t)(8 * g));
        {
          const float* src = (onv ? X : Y) + (size_t)r * 128 + o0 + 8 * g;
          const float4 x0 = *reinterpret_cast<const float4*>(src);
          const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
          uint4 h, l;
          split_pair(x0.x, x0.y, h.x, l.x);
          split_pair(x0.z, x0.w, h.y, l.y);
          split_pair(x1.x, x1.y, h.z, l.z);
          split_pair(x1.z, x1.w, h.w, l.w);
          *reinterpret_cast<uint4*>(tiles + off) = h;
          *reinterpret_cast<uint4*>(tiles + 8192 + off) = l;
        }
        uint4 h = make_uint4(0u, 0u, 0u, 0u), l = h;
        if (onv && v_exact) {
          if (r < L)
            h = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(v_in) + v_row0 +
                                                     (size_t)r * v_stride + o0 + 8 * g));
        } else {
          float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
          if (!onv) {
            const float* src = EK + (size_t)r * 128 + o0 + 8 * g;
            x0 = *reinterpret_cast<const float4*>(src);
            x1 = *reinterpret_cast<const float4*>(src + 4);
          } else if (r < L) {
            const float* src = static_cast<const float*>(v_in) + v_row0 + (size_t)r * v_stride + o0 + 8 * g;
            x0 = __ldg(reinterpret_cast<const float4*>(src));
            x1 = __ldg(reinterpret_cast<const float4*>(src + 4));
          }
          split_pair(x0.x, x0.y, h.x, l.x);
          split_pair(x0.z, x0.w, h.y, l.y);
          split_pair(x1.x, x1.y, h.z, l.z);
          split_pair(x1.z, x1.w, h.w, l.w);
        }
        *reinterpret_cast<uint4*>(tiles + 16384 + off) = h;
        *reinterpret_cast<uint4*>(tiles + 24576 + off) = l;
      }
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(64, 64);
        const bool b_lo = !(onv && v_exact);
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t o = (uint32_t)ks * 32u;
          const uint64_t Ah = sdesc_sw128(t_ah + o, 16, 1024), Al = sdesc_sw128(t_al + o, 16, 1024);
          const uint64_t Bh = sdesc_sw128(t_bh + o, 16, 1024), Bl = sdesc_sw128(t_bl + o, 16, 1024);
          mma_bf16(tmem, Ah, Bh, id, (s > 0 || ks > 0) ? 1u : 0u);
          mma_bf16(tmem, Al, Bh, id, 1);
          if (b_lo) mma_bf16(tmem, Ah, Bl, id, 1);
        }
        mma_commit(bar);
        open = s;
      }
      if (!mbar_wait(bar, (uint32_t)(s & 1))) ok = false;
      else if (tid == 0) open = -1;
      ok = named_bar_and(1, (int)blockDim.x, ok);  // the tiles are free for the next slice
      tc_fence_after();
    }
    if (ok) {  // rows 16 q + lane (lanes 0-15 of quadrant q = warp % 4); warp / 4: column half
      const int q = warp & 3, half = warp >> 2, i = 16 * q + lane;
      const uint32_t lb = tmem_addr(tmem, 32 * q, 0);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t r[16];
        tmem_ld16(lb + 32 * half + 16 * j, r);
        tmem_wait_ld();
        if (lane < 16) {
#pragma unroll
          for (int x = 0; x < 16; ++x) sZ[(size_t)i * ldz + 32 * half + 16 * j + x] = __uint_as_float(r[x]);
        }
      }
    } else if (tid == 0) {
      atomicOr(status, KDA_DEV_TIMEOUT);
      if (open >= 0) mbar_wait(bar, (uint32_t)(open & 1), 100000000ull);  // in flight: ends first
    }
    tc_fence_before();
    __syncthreads();
  }
};

template <int SC, int SK, int SV>
__global__ void __launch_bounds__(kThreads, 2) prep_kernel(const Args a) {
  extern __shared__ float smem[];
  GpuExec ex;
  prep_body<SC, SK, SV>(ex, a, (int64_t)blockIdx.x, (int)blockIdx.y, smem);
}

__global__ void __launch_bounds__(kThreads) states_kernel(const Args a) {
  extern __shared__ float smem[];
  GpuExec ex;
  states_body(ex, a, (int64_t)blockIdx.x, smem);
}

__global__ void __launch_bounds__(kThreads) dstate_kernel(const Args a) {
  extern __shared__ float smem[];
  GpuExec ex;
  dstate_body(ex, a, (int64_t)blockIdx.x, smem);
}

template <int SC, int SK, int SV>
__global__ void __launch_bounds__(kThreads, 2) grads_kernel(const Args a) {
  extern __shared__ float smem[];
  GpuExec ex;
  constexpr bool kZprod = SC == 64 && SK == 128 && SV == 128;  // the shape zprod serves
  __shared__ uint32_t tmem_slot;
  if (kZprod) {
    if (threadIdx.x < 32) {
      tc::tmem_alloc(&tmem_slot, 64);
      tc::tmem_relinquish();
    }
    __syncthreads();
    tc::tc_fence_after();
    ex.tmem_base = tmem_slot;
  }
  grads_body<SC, SK, SV>(ex, a, (int64_t)blockIdx.x, (int)blockIdx.y, smem);
  if (kZprod) {
    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tc::tmem_dealloc(ex.tmem_base, 64);
  }
}

// Five blocks per SM (48 registers, no spills): the element-wise phases wait on workspace
// rows, and more blocks keep more of those loads in flight (2.82 ms at three blocks per SM,
// 2.43 at four, 2.35 at five on the long workload; six spill)
template <int SC, int SK, int SV>
__global__ void __launch_bounds__(kThreads, 5) gate_kernel(const Args a) {
  extern __shared__ float smem[];
  GpuExec ex;
  gate_body<SC, SK, SV>(ex, a, (int64_t)blockIdx.x, (int)blockIdx.y, smem);
}

// The common shape (chunk 64, K = V = 128) with its dimensions compiled in.
bool common_shape(const Plan& p) { return p.C == 64 && p.K == 128 && p.V == 128; }

thread_local char t_msg[512];

kda_status fail(kda_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof t_msg, fmt, ap);
  va_end(ap);
  set_last_error(t_msg);
  return s;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The forward parameters the backward is checked against: d_o takes the place of o.
kda_fwd_params fwd_view(const kda_bwd_params* p) {
  kda_fwd_params f = p->fwd;
  f.o = const_cast<void*>(p->d_o);
  f.final_state = nullptr;
  f.h_out = nullptr;
  f.workspace = nullptr;
  f.workspace_bytes = 0;
  return f;
}

kda_status check(const kda_bwd_params* p) {
  if (p == nullptr) return fail(KDA_ERR_INVALID_ARG, "params is NULL");
  const kda_fwd_params f = fwd_view(p);
  kda_status s = kda_fwd_check(&f);
  if (s != KDA_OK) return s;  // the forward's message stays
  const bool tokens = (int64_t)f.B * f.T > 0;
  struct { const void* ptr; const char* name; bool required; } ptrs[] = {
      {p->dq, "dq", tokens},         {p->dk, "dk", tokens},
      {p->dv, "dv", tokens},         {p->dg, "dg", tokens},
      {p->dbeta, "dbeta", tokens},   {p->d_final_state, "d_final_state", false},
      {p->dA_log, "dA_log", false},  {p->ddt_bias, "ddt_bias", false},
      {p->dh0, "dh0", false},
  };
  for (auto& e : ptrs) {
    if (e.required && e.ptr == nullptr) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", e.name);
    if (e.ptr != nullptr && !aligned16(e.ptr))
      return fail(KDA_ERR_INVALID_ARG, "%s must be 16-byte aligned", e.name);
  }
  if (p->dA_log != nullptr && (f.A_log == nullptr || f.gate_mode == KDA_GATE_PREGATED))
    return fail(KDA_ERR_INVALID_ARG, "dA_log needs A_log and an in-kernel gate (plain or safe)");
  if (p->ddt_bias != nullptr && (f.dt_bias == nullptr || f.gate_mode == KDA_GATE_PREGATED))
    return fail(KDA_ERR_INVALID_ARG, "ddt_bias needs dt_bias and an in-kernel gate (plain or safe)");
  return KDA_OK;
}

Args make_args(const kda_bwd_params* p, const Plan& pl, unsigned int* status) {
  const kda_fwd_params& f = p->fwd;
  Args a;
  memset(&a, 0, sizeof a);
  a.p = pl;
  a.dtype = f.in_dtype; a.gate_mode = f.gate_mode; a.qk_l2norm = f.qk_l2norm;
  a.beta_sigmoid = f.beta_sigmoid; a.allow_neg_eigval = f.allow_neg_eigval;
  a.state_v_first = f.state_v_first; a.lower_bound = f.lower_bound; a.scale = f.scale;
  a.q = f.q; a.k = f.k; a.v = f.v; a.g = f.g; a.beta = f.beta; a.d_o = p->d_o;
  a.A_log = f.A_log; a.dt_bias = f.dt_bias; a.h0 = f.h0; a.d_final_state = p->d_final_state;
  a.cu_seqlens = f.cu_seqlens;
  a.dq = p->dq; a.dk = p->dk; a.dv = p->dv; a.dg = p->dg; a.dbeta = p->dbeta;
  a.dA_log = p->dA_log; a.ddt_bias = p->ddt_bias; a.dh0 = p->dh0;
  a.ws = static_cast<char*>(p->workspace);
  a.status = status;
  return a;
}

cudaError_t run_zero(const Args& a, cudaStream_t st) {
  float* outs[7] = {a.dq, a.dk, a.dv, a.dg, a.dbeta, a.dA_log, a.ddt_bias};
  ZeroRange z[14];
  const int n = zero_ranges(a.p, z);
  for (int i = 0; i < n; ++i) {
    float* base = outs[z[i].out];
    if (base == nullptr || z[i].count == 0) continue;
    cudaError_t e = cudaMemsetAsync(base + z[i].first, 0, z[i].count * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t run_chunk_table(const Args& a, cudaStream_t st) {
  const Plan& pl = a.p;
  FwdArgs t{};  // the forward's chunk-table kernel, writing into this workspace
  t.plan.N = pl.N; t.plan.C = pl.C; t.plan.nct = pl.nct; t.plan.ntok = pl.ntok;
  t.plan.varlen = true; t.plan.off_chunk_table = pl.off_table;
  t.cu_seqlens = a.cu_seqlens; t.ws = a.ws; t.status = a.status;
  return launch_chunk_table(t, st);
}

template <class Kernel>
cudaError_t launch_smem(Kernel kernel, dim3 grid, size_t smem, const Args& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t run_prep(const Args& a, cudaStream_t st) {
  const dim3 grid((unsigned)a.p.nct, (unsigned)a.p.HV);
  return common_shape(a.p) ? launch_smem(prep_kernel<64, 128, 128>, grid, prep_smem(a.p), a, st)
                           : launch_smem(prep_kernel<0, 0, 0>, grid, prep_smem(a.p), a, st);
}

cudaError_t run_states(const Args& a, cudaStream_t st) {
  return launch_smem(states_kernel, dim3((unsigned)state_blocks(a.p)), states_smem(a.p), a, st);
}

cudaError_t run_dstate(const Args& a, cudaStream_t st) {
  return launch_smem(dstate_kernel, dim3((unsigned)state_blocks(a.p)), dstate_smem(a.p), a, st);
}

cudaError_t run_gate(const Args& a, cudaStream_t st) {
  const dim3 grid((unsigned)a.p.nct, (unsigned)a.p.HV);
  return common_shape(a.p) ? launch_smem(gate_kernel<64, 128, 128>, grid, gate_smem(a.p), a, st)
                           : launch_smem(gate_kernel<0, 0, 0>, grid, gate_smem(a.p), a, st);
}

cudaError_t run_grads(const Args& a, cudaStream_t st) {
  const dim3 grid((unsigned)a.p.nct, (unsigned)a.p.HV);
  return common_shape(a.p) ? launch_smem(grads_kernel<64, 128, 128>, grid, grads_smem(a.p), a, st)
                           : launch_smem(grads_kernel<0, 0, 0>, grid, grads_smem(a.p), a, st);
}

}  // namespace
cudaError_t run_states_tc(const Args& a, cudaStream_t st);   // kda_bwd_tc.cu
cudaError_t run_dstate_tc(const Args& a, cudaStream_t st);   // kda_bwd_tc.cu
cudaError_t run_vprod_tc(const Args& a, cudaStream_t st);    // kda_bwd_tc.cu
namespace {

struct Stage {
  const char* name;
  cudaError_t (*run)(const Args&, cudaStream_t);
};
constexpr int kMaxStages = 9;

// The stages of one backward call, in order: the zeroing of the outputs (cudaMemsetAsync,
// no kernel of this library), then the kernels.
int stages_for(const Plan& pl, Stage* out) {
  int n = 0;
  out[n++] = {"zero_outputs", run_zero};
  if (pl.varlen) out[n++] = {"chunk_table", run_chunk_table};
  if (pl.nct > 0) out[n++] = {"bwd_prep", run_prep};
  if (state_blocks(pl) > 0) {
    out[n++] = {"bwd_states", pl.tc_states ? run_states_tc : run_states};
    out[n++] = {"bwd_dstate", pl.tc_dstate ? run_dstate_tc : run_dstate};
  }
  if (pl.nct > 0 && pl.tc_vprod) out[n++] = {"bwd_vprod", run_vprod_tc};
  if (pl.nct > 0) out[n++] = {"bwd_grads", run_grads};
  if (pl.nct > 0) out[n++] = {"bwd_gate", run_gate};
  return n;
}

// The state stage (chunks in order) and the state-gradient stage (chunks in reverse) read only
// what the recompute stage wrote and write disjoint workspace regions, so kda_bwd runs the
// latter on a library-owned stream beside the former: each occupies one SM per (sequence,
// value head) along its chain.  One stream and its fork / join events per device, created on
// first use; enqueueing holds the context's lock, so concurrent calls cannot swap events.
struct SideCtx {
  std::mutex mu;
  bool ready = false;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideCtx g_side[64];

SideCtx* side_ctx() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideCtx& c = g_side[dev];
  std::lock_guard<std::mutex> lk(c.mu);
  if (!c.ready) {
    if (cudaStreamCreateWithFlags(&c.side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    c.ready = true;
  }
  return &c;
}

// Checks (host), plan, workspace and the device status word; fills the kernel arguments.
kda_status prepare(const kda_bwd_params* p, Args& a) {
  kda_status s = check(p);
  if (s != KDA_OK) return s;
  const kda_fwd_params f = fwd_view(p);
  const Plan pl = make_plan(&f);
  if (p->workspace == nullptr || p->workspace_bytes < pl.total_bytes)
    return fail(KDA_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu%s)", pl.total_bytes,
                p->workspace_bytes, p->workspace ? "" : ", NULL");
  if ((reinterpret_cast<uintptr_t>(p->workspace) & 255u) != 0)
    return fail(KDA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  unsigned int* status = device_status_word();
  if (status == nullptr) return fail(KDA_ERR_CUDA, "no CUDA device / status word unavailable");
  a = make_args(p, pl, status);
  return KDA_OK;
}

}  // namespace
}  // namespace bwd
}  // namespace kda

using kda::set_last_error;
namespace B = kda::bwd;

extern "C" {

kda_status kda_bwd_check(const kda_bwd_params* p) {
  kda_status s = B::check(p);
  if (s == KDA_OK) set_last_error("");
  return s;
}

size_t kda_bwd_workspace_size(const kda_bwd_params* p) {
  if (B::check(p) != KDA_OK) return 0;
  const kda_fwd_params f = B::fwd_view(p);
  return B::make_plan(&f).total_bytes;
}

int32_t kda_bwd_num_launches(const kda_bwd_params* p) {
  if (B::check(p) != KDA_OK) return 0;
  const kda_fwd_params f = B::fwd_view(p);
  B::Stage st[B::kMaxStages];
  return B::stages_for(B::make_plan(&f), st) - 1;  // every stage but the zeroing
}

int32_t kda_bwd_num_stages(const kda_bwd_params* p) {
  if (B::check(p) != KDA_OK) return 0;
  const kda_fwd_params f = B::fwd_view(p);
  B::Stage st[B::kMaxStages];
  return B::stages_for(B::make_plan(&f), st);
}

const char* kda_bwd_stage_name(const kda_bwd_params* p, int32_t stage) {
  if (B::check(p) != KDA_OK) return "";
  const kda_fwd_params f = B::fwd_view(p);
  B::Stage st[B::kMaxStages];
  const int n = B::stages_for(B::make_plan(&f), st);
  return (stage >= 0 && stage < n) ? st[stage].name : "";
}

kda_status kda_bwd_stage(const kda_bwd_params* p, void* stream, int32_t stage) {
  B::Args a;
  kda_status s = B::prepare(p, a);
  if (s != KDA_OK) return s;
  B::Stage st[B::kMaxStages];
  const int n = B::stages_for(a.p, st);
  if (stage < 0 || stage >= n)
    return B::fail(KDA_ERR_INVALID_ARG, "stage %d out of range [0,%d)", stage, n);
  cudaError_t e = st[stage].run(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return B::fail(KDA_ERR_CUDA, "%s failed: %s", st[stage].name, cudaGetErrorString(e));
  set_last_error("");
  return KDA_OK;
}

kda_status kda_bwd(const kda_bwd_params* p, void* stream) {
  B::Args a;
  kda_status s = B::prepare(p, a);
  if (s != KDA_OK) return s;
  B::Stage st[B::kMaxStages];
  const int n = B::stages_for(a.p, st);
  const cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  int i_states = -1, i_dstate = -1;
  for (int i = 0; i < n; ++i) {
    if (strcmp(st[i].name, "bwd_states") == 0) i_states = i;
    if (strcmp(st[i].name, "bwd_dstate") == 0) i_dstate = i;
  }
  B::SideCtx* cx = (i_states >= 0 && i_dstate == i_states + 1) ? B::side_ctx() : nullptr;
  if (i_states >= 0 && cx == nullptr)
    return B::fail(KDA_ERR_CUDA, "could not create the backward's side stream");
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaSuccess;
    if (cx != nullptr && i == i_states) {
      // states on the caller's stream, dstate on the side stream, both after the stages
      // before them; the caller's stream then waits for both
      std::lock_guard<std::mutex> lk(cx->mu);
      if ((e = cudaEventRecord(cx->fork, s0)) == cudaSuccess &&
          (e = cudaStreamWaitEvent(cx->side, cx->fork, 0)) == cudaSuccess &&
          (e = st[i_dstate].run(a, cx->side)) == cudaSuccess &&
          (e = cudaEventRecord(cx->join, cx->side)) == cudaSuccess &&
          (e = st[i_states].run(a, s0)) == cudaSuccess)
        e = cudaStreamWaitEvent(s0, cx->join, 0);
      if (e != cudaSuccess)
        return B::fail(KDA_ERR_CUDA, "bwd_states / bwd_dstate failed: %s", cudaGetErrorString(e));
      ++i;  // dstate was enqueued with states
      continue;
    }
    e = st[i].run(a, s0);
    if (e != cudaSuccess)
      return B::fail(KDA_ERR_CUDA, "%s failed: %s", st[i].name, cudaGetErrorString(e));
  }
  set_last_error("");
  return KDA_OK;
}

}  // extern "C"
