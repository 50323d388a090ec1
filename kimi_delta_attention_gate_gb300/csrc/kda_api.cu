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

#include <algorithm>
#include <mutex>
#include <vector>
#include <string>

#include "kda_internal.cuh"

namespace kda {

__device__ unsigned int g_device_status;

// The intra-chunk kernel launch (kda_tc.cu) with overlap_previous: launched as a
// programmatic dependent of the kernel before it on `s`, so that its CTAs may start while
// that kernel's last CTAs run; only for a kernel that reads nothing the previous one writes
// (the intra-chunk kernels of consecutive chunk ranges).
cudaError_t launch_tc_intra(const FwdArgs& a, cudaStream_t s, bool overlap_previous);

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
// segment costs a few microseconds of launch and recurrence start-up; with the intra-chunk
// segments overlapping one another, 10 segments of ~102 chunks measured best for 1024
// chunks: 1.757 ms against 1.771 for 8 and 1.764 for 12).
constexpr int64_t kSegMaxRecurrences = 96;
constexpr int64_t kSegChunks = 100;
constexpr int kMaxSegments = 10;

// Chunk boundary k (0..nseg) of the segments.  Device inputs: equal segments (measured best
// against schedules with a larger first or smaller last segments).  Host inputs (ramp): weights 1, 2, 4, ..., 4, 2, 1, so that the first
// segment's input copy, after which computing starts, and the last segment's compute and
// output copy, which follow the last input byte, are short: the host link sets the pace.
int64_t seg_bound(int64_t nct, int nseg, int k, bool ramp = false) {
  if (!ramp) return nct * k / nseg;
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
  pl.tok_end = pl.varlen ? p->cu_seqlens_host[p->N] : pl.ntok;
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
  // host-buffer entry: copy-in and copy-out streams and their events
  cudaStream_t cin = nullptr, cout = nullptr;
  cudaEvent_t ein[kMaxSegments] = {}, eout[kMaxSegments] = {};
  cudaEvent_t hfork = nullptr, hdone = nullptr;
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
      if (cudaEventCreateWithFlags(&c.seg[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&c.ein[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&c.eout[i], cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    if (cudaStreamCreateWithFlags(&c.cin, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c.cout, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.hfork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.hdone, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
    c.ready = true;
  }
  return &c;
}

// Work a caller adds around each segment of the pipelined schedule (host-buffer entry:
// wait for the segment's input copies before its intra-chunk kernel, copy its output out
// after its recurrence).  Called with the pipeline context locked.
struct SegHooks {
  virtual cudaError_t before_intra(PipeCtx& cx, int k, int64_t cb, int64_t ce) = 0;
  virtual cudaError_t after_recur(PipeCtx& cx, int k, int64_t cb, int64_t ce) = 0;
  virtual ~SegHooks() = default;
};

// Segments k = 0..nseg-1: intra(k) on the caller's stream, recur(k) on the internal
// high-priority stream after intra(k) and recur(k-1); the caller's stream then waits for
// the last recurrence.  Stream order alone carries every dependency (no kernel waits on
// another), so the schedule is also valid under stream capture.  intra(k), k > 0, is a
// programmatic dependent of intra(k-1): the two share no data, and its CTAs fill the SMs
// while intra(k-1)'s last wave drains instead of after it (1.845 -> 1.771 ms on 1024
// chunks x 32 heads); the event that recur(k-1) waits on still marks the whole of
// intra(k-1).  With hooks (input copies waited for before each intra kernel) every launch
// keeps the full dependency.
cudaError_t launch_pipelined_locked(PipeCtx* cx, const FwdArgs& a, cudaStream_t s,
                                    const char** what, SegHooks* hooks) {
  const Plan& pl = a.plan;
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
    ak.c_begin = seg_bound(pl.nct, pl.nseg, k, hooks != nullptr);
    ak.c_end = seg_bound(pl.nct, pl.nseg, k + 1, hooks != nullptr);
    *what = "input copies";
    if (hooks && (e = hooks->before_intra(*cx, k, ak.c_begin, ak.c_end)) != cudaSuccess) return e;
    *what = "tc_intra";
    if ((e = launch_tc_intra(ak, s, k > 0 && hooks == nullptr)) != cudaSuccess) return e;
    *what = "pipeline event";
    if ((e = cudaEventRecord(cx->seg[k], s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(cx->rs, cx->seg[k], 0)) != cudaSuccess) return e;
    *what = "tc_recur";
    if ((e = launch_tc_recur(ak, cx->rs)) != cudaSuccess) return e;
    *what = "output copies";
    if (hooks && (e = hooks->after_recur(*cx, k, ak.c_begin, ak.c_end)) != cudaSuccess) return e;
  }
  *what = "pipeline join";
  if ((e = cudaEventRecord(cx->join, cx->rs)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(s, cx->join, 0);
}

cudaError_t launch_pipelined(const FwdArgs& a, cudaStream_t s, const char** what) {
  PipeCtx* cx = pipe_ctx();
  *what = "pipeline setup";
  if (cx == nullptr) return cudaErrorInitializationError;
  std::lock_guard<std::mutex> lk(cx->mu);
  return launch_pipelined_locked(cx, a, s, what, nullptr);
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

// ---- host-buffer entry ------------------------------------------------------------------
// Device arena of kda_fwd_host: the device copy of every tensor, then the pass's workspace.
struct HostArena {
  size_t q, k, v, g, beta, o, h0, fs, hout, alog, dt, cu, ws;
};

HostArena host_arena(const kda_fwd_params* p, int64_t nct) {
  HostArena A{};
  const size_t e = p->in_dtype == KDA_BF16 ? 2 : 4;
  const size_t ntok = (size_t)p->B * p->T;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  const size_t st = (size_t)p->N * p->HV * p->K * p->V * sizeof(float);
  A.q = take(ntok * p->H * p->K * e);
  A.k = take(ntok * p->H * p->K * e);
  A.v = take(ntok * p->HV * p->V * e);
  A.g = take(ntok * p->HV * p->K * e);
  A.beta = take(ntok * p->HV * e);
  A.o = take(ntok * p->HV * p->V * e);
  A.h0 = take(p->h0 ? st : 0);
  A.fs = take(p->final_state ? st : 0);
  A.hout = take(p->h_out ? (size_t)nct * p->HV * p->K * p->V * sizeof(float) : 0);
  A.alog = take(p->A_log ? (size_t)p->HV * sizeof(float) : 0);
  A.dt = take(p->dt_bias ? (size_t)p->HV * p->K * sizeof(float) : 0);
  A.cu = take(p->cu_seqlens_host ? (size_t)(p->N + 1) * sizeof(int64_t) : 0);
  A.ws = off;
  return A;
}

// The kda_fwd parameters that run the pass inside the arena at `base`.
kda_fwd_params arena_params(const kda_fwd_params* hp, const HostArena& A, char* base) {
  kda_fwd_params d = *hp;
  d.q = base + A.q; d.k = base + A.k; d.v = base + A.v; d.g = base + A.g;
  d.beta = base + A.beta; d.o = base + A.o;
  d.h0 = hp->h0 ? reinterpret_cast<const float*>(base + A.h0) : nullptr;
  d.final_state = hp->final_state ? reinterpret_cast<float*>(base + A.fs) : nullptr;
  d.h_out = hp->h_out ? reinterpret_cast<float*>(base + A.hout) : nullptr;
  d.A_log = hp->A_log ? reinterpret_cast<const float*>(base + A.alog) : nullptr;
  d.dt_bias = hp->dt_bias ? reinterpret_cast<const float*>(base + A.dt) : nullptr;
  d.cu_seqlens = hp->cu_seqlens_host ? reinterpret_cast<const int64_t*>(base + A.cu) : nullptr;
  d.workspace = base + A.ws;
  d.workspace_bytes = 0;
  return d;
}

// Checks of the host parameters; fills the arena layout and the arena-relative params
// (at a stand-in base when `base` is NULL) and returns the arena size through `bytes`.
kda_status host_plan(const kda_fwd_params* hp, char* base, HostArena& A, kda_fwd_params& dp,
                     size_t& bytes) {
  if (hp == nullptr) return fail(KDA_ERR_INVALID_ARG, "params is NULL");
  const struct { const void* ptr; const char* name; } need[] = {
      {hp->q, "q"}, {hp->k, "k"}, {hp->v, "v"}, {hp->g, "g"}, {hp->beta, "beta"}, {hp->o, "o"}};
  for (auto& e : need)
    if (e.ptr == nullptr) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", e.name);
  kda_fwd_params probe = *hp;  // the device-side rules, checked on a stand-in arena
  char* stand_in = reinterpret_cast<char*>(uintptr_t(1) << 20);
  HostArena A0 = host_arena(hp, 0);
  probe = arena_params(hp, A0, stand_in);
  kda_status s = check_args(&probe);
  if (s != KDA_OK) return s;
  const Plan pl = make_plan(&probe);
  A = host_arena(hp, pl.nct);
  dp = arena_params(hp, A, base ? base : stand_in);
  dp.workspace_bytes = pl.total_bytes;
  bytes = A.ws + pl.total_bytes;
  return KDA_OK;
}

// First token of global chunk c (c == nct: one past the last token of the last sequence).
int64_t chunk_token(const Plan& pl, const kda_fwd_params* hp, const std::vector<int64_t>& cfirst,
                    int64_t c) {
  if (!pl.varlen) {
    const int64_t n = c / pl.nc_per_seq, ci = c - n * pl.nc_per_seq;
    return n * pl.T + ci * pl.C;
  }
  if (c >= pl.nct) return hp->cu_seqlens_host[pl.N];
  int n = (int)(std::upper_bound(cfirst.begin(), cfirst.end(), c) - cfirst.begin()) - 1;
  return hp->cu_seqlens_host[n] + (c - cfirst[n]) * pl.C;
}

// Copies in, per segment, the token rows of q, k, v, g, beta on the copy-in stream; the
// segment's intra-chunk kernel waits for them; its output rows go out on the copy-out
// stream after its recurrence.
struct HostCopies : SegHooks {
  const kda_fwd_params* hp;
  const kda_fwd_params* dp;
  const Plan* pl;
  std::vector<int64_t> cfirst;
  cudaStream_t s;
  size_t e;
  cudaError_t rows_in(cudaStream_t st, int64_t tb, int64_t te) {
    const struct { void* dst; const void* src; size_t row; } t[] = {
        {const_cast<void*>(dp->q), hp->q, (size_t)pl->H * pl->K * e},
        {const_cast<void*>(dp->k), hp->k, (size_t)pl->H * pl->K * e},
        {const_cast<void*>(dp->v), hp->v, (size_t)pl->HV * pl->V * e},
        {const_cast<void*>(dp->g), hp->g, (size_t)pl->HV * pl->K * e},
        {const_cast<void*>(dp->beta), hp->beta, (size_t)pl->HV * e}};
    for (auto& x : t) {
      cudaError_t r = cudaMemcpyAsync(static_cast<char*>(x.dst) + tb * x.row,
                                      static_cast<const char*>(x.src) + tb * x.row,
                                      (te - tb) * x.row, cudaMemcpyHostToDevice, st);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  }
  cudaError_t before_intra(PipeCtx& cx, int k, int64_t, int64_t) override {
    return cudaStreamWaitEvent(s, cx.ein[k], 0);
  }
  cudaError_t after_recur(PipeCtx& cx, int k, int64_t cb, int64_t ce) override {
    cudaError_t r;
    if ((r = cudaEventRecord(cx.eout[k], cx.rs)) != cudaSuccess) return r;
    if ((r = cudaStreamWaitEvent(cx.cout, cx.eout[k], 0)) != cudaSuccess) return r;
    const int64_t tb = chunk_token(*pl, hp, cfirst, cb), te = chunk_token(*pl, hp, cfirst, ce);
    const size_t row = (size_t)pl->HV * pl->V * e;
    return cudaMemcpyAsync(static_cast<char*>(hp->o) + tb * row,
                           static_cast<const char*>(dp->o) + tb * row, (te - tb) * row,
                           cudaMemcpyDeviceToHost, cx.cout);
  }
};

}  // namespace

void set_last_error(const char* msg) { t_last_error = msg; }

// The device status word of the current device (NULL without a device): the backward pass
// (kda_bwd.cu) flags into the same word that kda_get_device_status reads.
unsigned int* device_status_word() { return device_status_ptr(); }

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

size_t kda_fwd_host_arena_size(const kda_fwd_params* p) {
  HostArena A;
  kda_fwd_params dp;
  size_t bytes = 0;
  return host_plan(p, nullptr, A, dp, bytes) == KDA_OK ? bytes : 0;
}

kda_status kda_fwd_host(const kda_fwd_params* p, void* arena, size_t arena_bytes, void* stream) {
  HostArena A;
  kda_fwd_params dp;
  size_t need = 0;
  kda_status st = host_plan(p, static_cast<char*>(arena), A, dp, need);
  if (st != KDA_OK) return st;
  if (arena == nullptr || arena_bytes < need)
    return fail(KDA_ERR_WORKSPACE, "arena needs %zu bytes (got %zu%s)", need, arena_bytes,
                arena ? "" : ", NULL");
  if (!aligned(arena, 256)) return fail(KDA_ERR_WORKSPACE, "arena must be 256-byte aligned");
  FwdArgs a;
  st = prepare(&dp, a);
  if (st != KDA_OK) return st;
  const Plan& pl = a.plan;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t e = p->in_dtype == KDA_BF16 ? 2 : 4;
  const size_t sbytes = (size_t)pl.N * pl.HV * pl.K * pl.V * sizeof(float);
  const char* what = "parameter copies";
  auto h2d = [&](const void* dst, const void* src, size_t n, cudaStream_t on) {
    return n == 0 || src == nullptr
               ? cudaSuccess
               : cudaMemcpyAsync(const_cast<void*>(dst), src, n, cudaMemcpyHostToDevice, on);
  };
  auto d2h = [&](void* dst, const void* src, size_t n, cudaStream_t on) {
    return n == 0 || dst == nullptr ? cudaSuccess
                                    : cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, on);
  };
  cudaError_t r = cudaSuccess;
  auto chk = [&](cudaError_t x) {
    if (r == cudaSuccess) r = x;
    return r == cudaSuccess;
  };
  chk(h2d(dp.A_log, p->A_log, p->A_log ? (size_t)pl.HV * sizeof(float) : 0, s));
  chk(h2d(dp.dt_bias, p->dt_bias, p->dt_bias ? (size_t)pl.HV * pl.K * sizeof(float) : 0, s));
  chk(h2d(dp.h0, p->h0, p->h0 ? sbytes : 0, s));
  chk(h2d(dp.cu_seqlens, p->cu_seqlens_host,
          p->cu_seqlens_host ? (size_t)(pl.N + 1) * sizeof(int64_t) : 0, s));
  const size_t hbytes = (size_t)pl.nct * pl.HV * pl.K * pl.V * sizeof(float);
  if (pl.tok_end < pl.ntok) {  // rows no sequence covers: zero, like the oracle
    const size_t row = (size_t)pl.HV * pl.V * e;
    what = "zeroing uncovered rows";
    chk(cudaMemsetAsync(static_cast<char*>(dp.o) + pl.tok_end * row, 0,
                        (size_t)(pl.ntok - pl.tok_end) * row, s)) &&
        chk(d2h(static_cast<char*>(p->o) + pl.tok_end * row,
                static_cast<const char*>(dp.o) + pl.tok_end * row,
                (size_t)(pl.ntok - pl.tok_end) * row, s));
  }
  if (r == cudaSuccess && pl.nseg > 1) {
    PipeCtx* cx = pipe_ctx();
    if (cx == nullptr) return fail(KDA_ERR_CUDA, "pipeline setup failed");
    std::lock_guard<std::mutex> lk(cx->mu);
    HostCopies hc;
    hc.hp = p; hc.dp = &dp; hc.pl = &pl; hc.s = s; hc.e = e;
    if (pl.varlen) {
      hc.cfirst.resize(pl.N + 1);
      hc.cfirst[0] = 0;
      for (int n = 0; n < pl.N; ++n)
        hc.cfirst[n + 1] = hc.cfirst[n] +
            (p->cu_seqlens_host[n + 1] - p->cu_seqlens_host[n] + pl.C - 1) / pl.C;
    }
    what = "input copies";
    chk(cudaEventRecord(cx->hfork, s)) && chk(cudaStreamWaitEvent(cx->cin, cx->hfork, 0)) &&
        chk(cudaStreamWaitEvent(cx->cout, cx->hfork, 0));
    for (int k = 0; k < pl.nseg && r == cudaSuccess; ++k) {
      const int64_t tb = chunk_token(pl, p, hc.cfirst, seg_bound(pl.nct, pl.nseg, k, true));
      const int64_t te = chunk_token(pl, p, hc.cfirst, seg_bound(pl.nct, pl.nseg, k + 1, true));
      chk(hc.rows_in(cx->cin, tb, te)) && chk(cudaEventRecord(cx->ein[k], cx->cin));
    }
    if (r == cudaSuccess) r = launch_pipelined_locked(cx, a, s, &what, &hc);
    what = "output copies";
    chk(d2h(p->final_state, dp.final_state, p->final_state ? sbytes : 0, cx->cout));
    chk(d2h(p->h_out, dp.h_out, p->h_out ? hbytes : 0, cx->cout));
    chk(cudaEventRecord(cx->hdone, cx->cout)) && chk(cudaStreamWaitEvent(s, cx->hdone, 0));
  } else if (r == cudaSuccess) {
    HostCopies hc;
    hc.hp = p; hc.dp = &dp; hc.pl = &pl; hc.s = s; hc.e = e;
    // rows past the last sequence are neither read nor written
    const int64_t tend = pl.varlen ? p->cu_seqlens_host[pl.N] : pl.ntok;
    what = "input copies";
    if (chk(hc.rows_in(s, 0, tend))) {
      Stage stg[kMaxStages];
      const int n = stages_for(pl, stg);
      for (int i = 0; i < n && r == cudaSuccess; ++i) {
        what = stg[i].name;
        chk(stg[i].launch(a, s));
      }
    }
    what = "output copies";
    chk(d2h(p->o, dp.o, (size_t)tend * pl.HV * pl.V * e, s));
    chk(d2h(p->final_state, dp.final_state, p->final_state ? sbytes : 0, s));
    chk(d2h(p->h_out, dp.h_out, p->h_out ? hbytes : 0, s));
  }
  if (r != cudaSuccess) return fail(KDA_ERR_CUDA, "%s failed: %s", what, cudaGetErrorString(r));
  t_last_error.clear();
  return KDA_OK;
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
  cudaError_t e = zero_uncovered_rows(a, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = launch_recurrent(a, static_cast<cudaStream_t>(stream));
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
