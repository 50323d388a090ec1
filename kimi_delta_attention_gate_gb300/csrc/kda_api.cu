// Host layer of the C ABI: argument checks, workspace plan, kernel launches, status.
//
// Checks follow the parameter rules of "FLA-KDA engineering notes" (section 2.1:
// A_log required for the in-kernel gate without a lower bound, -5 <= lower_bound < 0
// for the safe gate, chunk_size 32 or 64, K <= 256, HV % H == 0, fp32 initial state)
// and the host checks of "FlashKDA gate-bias load path" (section 2 part 2 and
// section 4: fp32 A_log / dt_bias of shapes [HV] and [HV, K], a clear error
// instead of a silent one).

#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "kda_internal.cuh"

namespace kda {

__device__ unsigned int g_device_status;

namespace {

thread_local std::string t_last_error;

kda_status fail(kda_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Pipelined schedule limits: segment only when at most this many (sequence, value head)
// recurrences run (each takes one SM), with about kSegChunks chunks per segment (each
// segment costs a few microseconds of launch and pipeline start-up; 8 segments of 128
// chunks measured best for 1024 chunks).
constexpr int64_t kSegMaxRecurrences = 96;
constexpr int64_t kSegChunks = 128;
constexpr int kMaxSegments = 8;

// Chunk boundary k (0..nseg) of the segments: weights 1, 2, 4, ..., 4, 2, 1 so that the
// first intra-chunk segment (which runs alone) and the last recurrence segment (which
// also runs alone) are short.
int64_t seg_bound(int64_t nct, int nseg, int k) {
  auto weight = [nseg](int j) {
    const int e = j < nseg - 1 - j ? j : nseg - 1 - j;  // distance to the nearer end
    return e == 0 ? 1 : (e == 1 ? 2 : 4);
  };
  int64_t tot = 0, part = 0;
  for (int j = 0; j < nseg; ++j) {
    tot += weight(j);
    if (j < k) part += weight(j);
  }
  return nct * part / tot;
}

// Every check that needs no workspace and no CUDA call.
kda_status check_args(const kda_fwd_params* p) {
  if (p == nullptr) return fail(KDA_ERR_INVALID_ARG, "params is NULL");
  if (p->in_dtype != KDA_BF16 && p->in_dtype != KDA_F32)
    return fail(KDA_ERR_DTYPE, "in_dtype must be KDA_BF16 or KDA_F32 (got %d)", p->in_dtype);
  if (p->B < 1 || p->T < 0 || p->H < 1 || p->HV < 1 || p->K < 1 || p->V < 1)
    return fail(KDA_ERR_SHAPE, "need B>=1, T>=0, H>=1, HV>=1, K>=1, V>=1");
  if (p->K > kMaxK) return fail(KDA_ERR_SHAPE, "K must be <= %d (got %d)", kMaxK, p->K);
  if (p->V > kMaxV) return fail(KDA_ERR_SHAPE, "V must be <= %d (got %d)", kMaxV, p->V);
  if (p->HV % p->H != 0)
    return fail(KDA_ERR_SHAPE, "HV %% H must be 0 for grouped value attention (HV=%d, H=%d)", p->HV,
                p->H);
  if (p->chunk_size != 32 && p->chunk_size != 64)
    return fail(KDA_ERR_SHAPE, "chunk_size must be 32 or 64 (got %d)", p->chunk_size);
  if ((int64_t)p->B * p->T > (int64_t)INT32_MAX)
    return fail(KDA_ERR_SHAPE, "B*T must fit in int32");
  switch (p->gate_mode) {
    case KDA_GATE_PREGATED:
      break;
    case KDA_GATE_PLAIN:
      if (p->A_log == nullptr)
        return fail(KDA_ERR_INVALID_ARG,
                    "the in-kernel gate without lower_bound needs A_log (plain gate "
                    "-exp(A_log)*softplus(g+dt_bias))");
      break;
    case KDA_GATE_SAFE:
      if (!(p->lower_bound >= -5.0f && p->lower_bound < 0.0f))
        return fail(KDA_ERR_INVALID_ARG, "safe gate needs -5 <= lower_bound < 0 (got %g)",
                    (double)p->lower_bound);
      break;
    default:
      return fail(KDA_ERR_INVALID_ARG, "unknown gate_mode %d", p->gate_mode);
  }
  if (!isfinite(p->scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
  if ((p->qk_l2norm != 0 && p->qk_l2norm != 1) || (p->beta_sigmoid != 0 && p->beta_sigmoid != 1) ||
      (p->allow_neg_eigval != 0 && p->allow_neg_eigval != 1) ||
      (p->state_v_first != 0 && p->state_v_first != 1))
    return fail(KDA_ERR_INVALID_ARG,
                "qk_l2norm, beta_sigmoid, allow_neg_eigval and state_v_first must be 0 or 1");
  if (p->allow_neg_eigval && !p->beta_sigmoid)  // reading notes section 2.1
    return fail(KDA_ERR_INVALID_ARG, "allow_neg_eigval needs beta_sigmoid (beta = 2 sigmoid(logit))");
  // sequences
  if (p->cu_seqlens != nullptr) {
    if (p->B != 1) return fail(KDA_ERR_SHAPE, "cu_seqlens requires B == 1 (got B=%d)", p->B);
    if (p->cu_seqlens_host == nullptr)
      return fail(KDA_ERR_INVALID_ARG, "cu_seqlens needs its host copy cu_seqlens_host");
    if (p->N < 1) return fail(KDA_ERR_SHAPE, "N must be >= 1 with cu_seqlens");
    const int64_t* cu = p->cu_seqlens_host;
    if (cu[0] != 0) return fail(KDA_ERR_SHAPE, "cu_seqlens[0] must be 0");
    for (int n = 0; n < p->N; ++n)
      if (cu[n + 1] < cu[n]) return fail(KDA_ERR_SHAPE, "cu_seqlens must be non-decreasing");
    if (cu[p->N] > p->T)
      return fail(KDA_ERR_SHAPE, "cu_seqlens[N]=%lld exceeds T=%d", (long long)cu[p->N], p->T);
    if (!aligned(p->cu_seqlens, 8)) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens misaligned");
  } else {
    if (p->cu_seqlens_host != nullptr)
      return fail(KDA_ERR_INVALID_ARG, "cu_seqlens_host given without cu_seqlens");
    if (p->N != p->B) return fail(KDA_ERR_SHAPE, "N must equal B without cu_seqlens");
  }
  // pointers
  const bool any_tokens = (int64_t)p->B * p->T > 0;
  struct { const void* ptr; const char* name; bool required; } ptrs[] = {
      {p->q, "q", any_tokens},        {p->k, "k", any_tokens},
      {p->v, "v", any_tokens},        {p->g, "g", any_tokens},
      {p->beta, "beta", any_tokens},  {p->o, "o", any_tokens},
      {p->A_log, "A_log", false},     {p->dt_bias, "dt_bias", false},
      {p->h0, "h0", false},           {p->final_state, "final_state", false},
      {p->h_out, "h_out", false},
  };
  for (auto& e : ptrs) {
    if (e.required && e.ptr == nullptr) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", e.name);
    if (e.ptr != nullptr && !aligned(e.ptr, 16))
      return fail(KDA_ERR_INVALID_ARG, "%s must be 16-byte aligned", e.name);
  }
  return KDA_OK;
}

Plan make_plan(const kda_fwd_params* p) {
  Plan pl{};
  pl.B = p->B; pl.T = p->T; pl.H = p->H; pl.HV = p->HV; pl.K = p->K; pl.V = p->V;
  pl.C = p->chunk_size; pl.N = p->N; pl.G = p->HV / p->H;
  pl.ntok = (int64_t)p->B * p->T;
  pl.varlen = p->cu_seqlens != nullptr;
  pl.nc_per_seq = (p->T + pl.C - 1) / pl.C;
  if (pl.varlen) {
    int64_t nct = 0;
    for (int n = 0; n < p->N; ++n) {
      int64_t len = p->cu_seqlens_host[n + 1] - p->cu_seqlens_host[n];
      nct += (len + pl.C - 1) / pl.C;
    }
    pl.nct = nct;
  } else {
    pl.nct = (int64_t)p->B * pl.nc_per_seq;
  }
  size_t off = 256;  // reserved header
  pl.off_chunk_table = off;
  if (pl.varlen) off += round_up(sizeof(int64_t) * (size_t)(p->N + 1), 256);
  pl.off_inter = off;
  pl.tensor_core = tc_eligible(pl, p->in_dtype);
  pl.inter_block_bytes =
      pl.tensor_core ? tc_inter_block_bytes() : simt_inter_block_bytes(pl.C, pl.K, pl.V);
  off += pl.inter_block_bytes * (size_t)pl.nct * (size_t)pl.HV;
  // Pipelined schedule: when few (sequence, head) recurrences leave most SMs idle during
  // the recurrence, the chunk range is cut into segments so that the intra-chunk kernel of
  // segment k+1 runs beside the recurrence of segment k.
  pl.nseg = 1;
  pl.off_state = 0;
  if (pl.tensor_core && (int64_t)pl.N * pl.HV <= kSegMaxRecurrences) {
    int64_t ns = pl.nct / kSegChunks;
    pl.nseg = (int)(ns < 1 ? 1 : (ns > kMaxSegments ? kMaxSegments : ns));
  }
  if (pl.nseg > 1) {
    off = round_up(off, 256);
    pl.off_state = off;
    off += sizeof(float) * (size_t)pl.N * pl.HV * pl.K * pl.V;
  }
  pl.total_bytes = off;
  return pl;
}

// Internal high-priority stream and events of the pipelined schedule, one set per device.
struct PipeCtx {
  std::mutex mu;
  bool ready = false;
  cudaStream_t rs = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaEvent_t seg[kMaxSegments] = {};
};
PipeCtx g_pipe[64];

PipeCtx* pipe_ctx() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  PipeCtx& c = g_pipe[dev];
  std::lock_guard<std::mutex> lk(c.mu);
  if (!c.ready) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithPriority(&c.rs, cudaStreamNonBlocking, greatest) != cudaSuccess)
      return nullptr;
    if (cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    for (int i = 0; i < kMaxSegments; ++i)
      if (cudaEventCreateWithFlags(&c.seg[i], cudaEventDisableTiming) != cudaSuccess) return nullptr;
    c.ready = true;
  }
  return &c;
}

// Segments k = 0..nseg-1: intra(k) on the caller's stream, recur(k) on the internal
// high-priority stream after intra(k) and recur(k-1); the caller's stream then waits for
// the last recurrence.  Stream order alone carries every dependency (no kernel waits on
// another), so the schedule is also valid under stream capture.
cudaError_t launch_pipelined(const FwdArgs& a, cudaStream_t s, const char** what) {
  const Plan& pl = a.plan;
  PipeCtx* cx = pipe_ctx();
  *what = "pipeline setup";
  if (cx == nullptr) return cudaErrorInitializationError;
  std::lock_guard<std::mutex> lk(cx->mu);
  cudaError_t e;
  if (pl.varlen) {
    *what = "chunk_table";
    if ((e = launch_chunk_table(a, s)) != cudaSuccess) return e;
  }
  *what = "pipeline fork";
  if ((e = cudaEventRecord(cx->fork, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(cx->rs, cx->fork, 0)) != cudaSuccess) return e;
  for (int k = 0; k < pl.nseg; ++k) {
    FwdArgs ak = a;
    ak.c_begin = seg_bound(pl.nct, pl.nseg, k);
    ak.c_end = seg_bound(pl.nct, pl.nseg, k + 1);
    *what = "tc_intra";
    if ((e = launch_tc_intra(ak, s)) != cudaSuccess) return e;
    *what = "pipeline event";
    if ((e = cudaEventRecord(cx->seg[k], s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(cx->rs, cx->seg[k], 0)) != cudaSuccess) return e;
    *what = "tc_recur";
    if ((e = launch_tc_recur(ak, cx->rs)) != cudaSuccess) return e;
  }
  *what = "pipeline join";
  if ((e = cudaEventRecord(cx->join, cx->rs)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(s, cx->join, 0);
}

std::mutex g_status_mu;
unsigned int* g_status_ptr[64] = {};

unsigned int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned int*>(ptr);
  }
  return g_status_ptr[dev];
}

struct Stage {
  const char* name;
  cudaError_t (*launch)(const FwdArgs&, cudaStream_t);
};

// The kernels one forward call launches, in order.
int stages_for(const Plan& pl, Stage* out) {
  int n = 0;
  if (pl.varlen) out[n++] = {"chunk_table", launch_chunk_table};
  if (pl.tensor_core) {
    out[n++] = {"tc_intra", launch_tc_intra};
    out[n++] = {"tc_recur", launch_tc_recur};
  } else {
    out[n++] = {"simt_intra", launch_simt_intra};
    out[n++] = {"simt_recur", launch_simt_recur};
  }
  return n;
}

constexpr int kMaxStages = 8;

// Checks (host), workspace, device status word; fills the kernel arguments.
kda_status prepare(const kda_fwd_params* p, FwdArgs& a) {
  kda_status s = check_args(p);
  if (s != KDA_OK) return s;
  Plan pl = make_plan(p);
  if (p->workspace == nullptr || p->workspace_bytes < pl.total_bytes)
    return fail(KDA_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu%s)", pl.total_bytes,
                p->workspace_bytes, p->workspace ? "" : ", NULL");
  if (!aligned(p->workspace, 256)) return fail(KDA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  unsigned int* status = device_status_ptr();
  if (status == nullptr) return fail(KDA_ERR_CUDA, "no CUDA device / status word unavailable");
  a = FwdArgs{};
  a.plan = pl;
  a.dtype = p->in_dtype; a.gate_mode = p->gate_mode;
  a.qk_l2norm = p->qk_l2norm; a.beta_sigmoid = p->beta_sigmoid;
  a.allow_neg_eigval = p->allow_neg_eigval; a.state_v_first = p->state_v_first;
  a.lower_bound = p->lower_bound; a.scale = p->scale;
  a.q = p->q; a.k = p->k; a.v = p->v; a.g = p->g; a.beta = p->beta;
  a.A_log = p->A_log; a.dt_bias = p->dt_bias; a.h0 = p->h0; a.cu_seqlens = p->cu_seqlens;
  a.o = p->o; a.final_state = p->final_state; a.h_out = p->h_out;
  a.ws = static_cast<char*>(p->workspace);
  a.status = status;
  a.c_begin = 0;
  a.c_end = pl.nct;
  return KDA_OK;
}

}  // namespace

void set_last_error(const char* msg) { t_last_error = msg; }

}  // namespace kda

using namespace kda;

extern "C" {

int32_t kda_abi_version(void) { return KDA_ABI_VERSION; }

const char* kda_last_error(void) { return t_last_error.c_str(); }

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_SHAPE: return "invalid shape";
    case KDA_ERR_DTYPE: return "invalid dtype";
    case KDA_ERR_UNSUPPORTED: return "unsupported combination";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_DEVICE_STATUS: return "device status flagged";
    case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
  }
  return "unknown status";
}

kda_status kda_fwd_check(const kda_fwd_params* p) {
  kda_status s = check_args(p);
  if (s == KDA_OK) t_last_error.clear();
  return s;
}

size_t kda_fwd_workspace_size(const kda_fwd_params* p) {
  if (check_args(p) != KDA_OK) return 0;
  return make_plan(p).total_bytes;
}

kda_status kda_fwd(const kda_fwd_params* p, void* stream) {
  FwdArgs a;
  kda_status s = prepare(p, a);
  if (s != KDA_OK) return s;
  if (a.plan.nseg > 1) {
    const char* what = "";
    cudaError_t e = launch_pipelined(a, static_cast<cudaStream_t>(stream), &what);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "%s failed: %s", what, cudaGetErrorString(e));
    t_last_error.clear();
    return KDA_OK;
  }
  Stage st[kMaxStages];
  const int n = stages_for(a.plan, st);
  for (int i = 0; i < n; ++i) {
    cudaError_t e = st[i].launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
      return fail(KDA_ERR_CUDA, "%s launch failed: %s", st[i].name, cudaGetErrorString(e));
  }
  t_last_error.clear();
  return KDA_OK;
}

int32_t kda_fwd_num_launches(const kda_fwd_params* p) {
  if (check_args(p) != KDA_OK) return 0;
  const Plan pl = make_plan(p);
  if (pl.nseg > 1) return (pl.varlen ? 1 : 0) + 2 * pl.nseg;
  Stage st[kMaxStages];
  return stages_for(pl, st);
}

kda_status kda_fused_recurrent_fwd(const kda_fwd_params* p, void* stream) {
  if (p == nullptr) return fail(KDA_ERR_INVALID_ARG, "params is NULL");
  kda_fwd_params c = *p;
  c.chunk_size = 64;  // not used by the token recurrence; every other rule applies
  kda_status s = check_args(&c);
  if (s != KDA_OK) return s;
  if (p->h_out != nullptr)
    return fail(KDA_ERR_INVALID_ARG, "h_out (per-chunk states) is an output of kda_fwd only");
  unsigned int* status = device_status_ptr();
  if (status == nullptr) return fail(KDA_ERR_CUDA, "no CUDA device / status word unavailable");
  FwdArgs a{};
  a.plan = make_plan(&c);
  a.dtype = p->in_dtype; a.gate_mode = p->gate_mode;
  a.qk_l2norm = p->qk_l2norm; a.beta_sigmoid = p->beta_sigmoid;
  a.allow_neg_eigval = p->allow_neg_eigval; a.state_v_first = p->state_v_first;
  a.lower_bound = p->lower_bound; a.scale = p->scale;
  a.q = p->q; a.k = p->k; a.v = p->v; a.g = p->g; a.beta = p->beta;
  a.A_log = p->A_log; a.dt_bias = p->dt_bias; a.h0 = p->h0; a.cu_seqlens = p->cu_seqlens;
  a.o = p->o; a.final_state = p->final_state;
  a.status = status;
  cudaError_t e = launch_recurrent(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "recurrent launch failed: %s", cudaGetErrorString(e));
  t_last_error.clear();
  return KDA_OK;
}

int64_t kda_fwd_num_chunks(const kda_fwd_params* p) {
  if (check_args(p) != KDA_OK) return 0;
  return make_plan(p).nct;
}

int32_t kda_fwd_num_stages(const kda_fwd_params* p) {
  if (check_args(p) != KDA_OK) return 0;
  Stage st[kMaxStages];
  return stages_for(make_plan(p), st);
}

const char* kda_fwd_stage_name(const kda_fwd_params* p, int32_t stage) {
  if (check_args(p) != KDA_OK) return "";
  Stage st[kMaxStages];
  const int n = stages_for(make_plan(p), st);
  return (stage >= 0 && stage < n) ? st[stage].name : "";
}

kda_status kda_fwd_stage(const kda_fwd_params* p, void* stream, int32_t stage) {
  FwdArgs a;
  kda_status s = prepare(p, a);
  if (s != KDA_OK) return s;
  Stage st[kMaxStages];
  const int n = stages_for(a.plan, st);
  if (stage < 0 || stage >= n) return fail(KDA_ERR_INVALID_ARG, "stage %d out of range [0,%d)", stage, n);
  cudaError_t e = st[stage].launch(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(KDA_ERR_CUDA, "%s launch failed: %s", st[stage].name, cudaGetErrorString(e));
  t_last_error.clear();
  return KDA_OK;
}

uint32_t kda_get_device_status(void* stream) {
  unsigned int* status = device_status_ptr();
  if (status == nullptr) return 0xFFFFFFFFu;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return 0xFFFFFFFFu;
  if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return 0xFFFFFFFFu;
  unsigned int zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return 0xFFFFFFFFu;
  return v;
}

}  // extern "C"
