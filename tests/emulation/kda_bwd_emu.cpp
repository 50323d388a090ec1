// Host build of the backward stage bodies (kimi_delta_attention_gate_gb300/csrc/kda_bwd.cuh),
// test infrastructure only.  It runs every block of every stage on the CPU with the GPU's
// block size: each phase runs all 256 threads' shares, in a freshly shuffled thread order,
// before the next phase.  Every buffer is a separate heap allocation of its exact size (so
// that AddressSanitizer sees any access past an end), and the workspace and each block's
// shared memory start as NaN (so that a read before a write shows up in the results).
//
// Usage: kda_bwd_emu DIR.  DIR/spec.txt holds "key value" lines (shapes and options, which
// optional tensors are present, the shuffle seed); the inputs are raw little-endian files
// DIR/<name>.bin (q, k, v, g, beta, d_o in the input dtype -- bf16 as its 16-bit pattern --;
// A_log, dt_bias, h0, d_final_state fp32; cu_seqlens int64).  The gradients are written as
// fp32 files DIR/out_<name>.bin, and DIR/out_status.txt gets the device status bits.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <random>
#include <string>
#include <vector>

#include "kda_bwd.cuh"

namespace {

using kda::bwd::Args;
using kda::bwd::Plan;

struct HostExec {
  static constexpr bool kTensorCores = false;  // the CUDA-core forms of every product
  int nthr = kda::bwd::kThreads;
  std::mt19937* rng = nullptr;
  std::vector<int> order;
  int cur = 0;  // the thread whose share of the phase runs
  // Asynchronous copies issued by each thread and not yet waited for: they land only at that
  // thread's next copy_wait(), so that a read of their destination before it (by any thread)
  // sees the poisoned contents, as it could on the GPU.
  std::vector<std::vector<std::pair<float*, const float*>>> pending;
  template <class F>
  void phase(F&& f) {
    if ((int)order.size() != nthr) {
      order.resize(nthr);
      for (int t = 0; t < nthr; ++t) order[t] = t;
      pending.resize(nthr);
    }
    std::shuffle(order.begin(), order.end(), *rng);
    for (int t : order) {
      cur = t;
      f(t, nthr);
    }
  }
  void atomic_add(float* p, float x) { *p += x; }
  void flag(unsigned int* s, unsigned int bits) { *s |= bits; }
  void copy16(float* dst, const float* src) { pending[cur].emplace_back(dst, src); }
  void copy_commit() {}
  void copy_wait() {
    for (auto& c : pending[cur]) memcpy(c.first, c.second, 16);
    pending[cur].clear();
  }
  // every copy must have been waited for by the end of a stage body
  bool drained() const {
    for (const auto& v : pending)
      if (!v.empty()) return false;
    return true;
  }
};

[[noreturn]] void die(const char* what, const std::string& detail) {
  fprintf(stderr, "kda_bwd_emu: %s %s\n", what, detail.c_str());
  exit(2);
}

std::map<std::string, std::string> read_spec(const std::string& path) {
  std::map<std::string, std::string> m;
  FILE* f = fopen(path.c_str(), "r");
  if (!f) die("cannot open", path);
  char key[128], val[128];
  while (fscanf(f, "%127s %127s", key, val) == 2) m[key] = val;
  fclose(f);
  return m;
}

// A heap buffer of exactly `bytes` bytes read from DIR/name.bin (whose size must match).
void* load(const std::string& dir, const char* name, size_t bytes) {
  const std::string path = dir + "/" + name + ".bin";
  FILE* f = fopen(path.c_str(), "rb");
  if (!f) die("cannot open", path);
  void* buf = malloc(bytes ? bytes : 1);
  if (bytes && fread(buf, 1, bytes, f) != bytes) die("short file", path);
  if (fgetc(f) != EOF) die("file longer than its shape", path);
  fclose(f);
  return buf;
}

void save(const std::string& dir, const char* name, const float* p, size_t n) {
  if (p == nullptr) return;
  const std::string path = dir + "/out_" + name + ".bin";
  FILE* f = fopen(path.c_str(), "wb");
  if (!f) die("cannot write", path);
  if (n) fwrite(p, sizeof(float), n, f);
  fclose(f);
}

float* zeros(size_t n) { return static_cast<float*>(calloc(n ? n : 1, sizeof(float))); }

void poison(void* p, size_t bytes) { memset(p, 0xFF, bytes); }  // every float NaN

}  // namespace

int main(int argc, char** argv) {
  if (argc != 2) die("usage:", "kda_bwd_emu DIR");
  const std::string dir = argv[1];
  auto spec = read_spec(dir + "/spec.txt");
  auto geti = [&](const char* k) {
    if (!spec.count(k)) die("spec misses", k);
    return atoi(spec[k].c_str());
  };
  auto getf = [&](const char* k) {
    if (!spec.count(k)) die("spec misses", k);
    return (float)atof(spec[k].c_str());
  };
  kda_fwd_params f;
  memset(&f, 0, sizeof f);
  f.B = geti("B"); f.T = geti("T"); f.H = geti("H"); f.HV = geti("HV");
  f.K = geti("K"); f.V = geti("V"); f.chunk_size = geti("chunk_size");
  f.in_dtype = geti("in_dtype"); f.gate_mode = geti("gate_mode");
  f.lower_bound = getf("lower_bound"); f.scale = getf("scale");
  f.qk_l2norm = geti("qk_l2norm"); f.beta_sigmoid = geti("beta_sigmoid");
  f.N = geti("N"); f.allow_neg_eigval = geti("allow_neg_eigval");
  f.state_v_first = geti("state_v_first");
  const size_t e = f.in_dtype == KDA_F32 ? 4 : 2;
  const size_t ntok = (size_t)f.B * f.T;
  const size_t qk = ntok * f.H * f.K, vv = ntok * f.HV * f.V, gg = ntok * f.HV * f.K,
               bb = ntok * f.HV, st = (size_t)f.N * f.HV * f.K * f.V;
  f.q = load(dir, "q", qk * e);
  f.k = load(dir, "k", qk * e);
  f.v = load(dir, "v", vv * e);
  f.g = load(dir, "g", gg * e);
  f.beta = load(dir, "beta", bb * e);
  const void* d_o = load(dir, "d_o", vv * e);
  if (geti("has_A_log")) f.A_log = static_cast<float*>(load(dir, "A_log", f.HV * 4));
  if (geti("has_dt_bias")) f.dt_bias = static_cast<float*>(load(dir, "dt_bias", (size_t)f.HV * f.K * 4));
  if (geti("has_h0")) f.h0 = static_cast<float*>(load(dir, "h0", st * 4));
  if (geti("has_cu_seqlens")) {
    const int64_t* cu = static_cast<int64_t*>(load(dir, "cu_seqlens", (size_t)(f.N + 1) * 8));
    f.cu_seqlens = cu;
    f.cu_seqlens_host = cu;
  }
  const float* dfs = geti("has_d_final_state")
                         ? static_cast<float*>(load(dir, "d_final_state", st * 4)) : nullptr;

  const Plan pl = kda::bwd::make_plan(&f);
  char* ws = static_cast<char*>(aligned_alloc(256, pl.total_bytes));
  poison(ws, pl.total_bytes);
  unsigned int status = 0;

  Args a;
  memset(&a, 0, sizeof a);
  a.p = pl;
  a.dtype = f.in_dtype; a.gate_mode = f.gate_mode; a.qk_l2norm = f.qk_l2norm;
  a.beta_sigmoid = f.beta_sigmoid; a.allow_neg_eigval = f.allow_neg_eigval;
  a.state_v_first = f.state_v_first; a.lower_bound = f.lower_bound; a.scale = f.scale;
  a.q = f.q; a.k = f.k; a.v = f.v; a.g = f.g; a.beta = f.beta; a.d_o = d_o;
  a.A_log = f.A_log; a.dt_bias = f.dt_bias; a.h0 = f.h0; a.d_final_state = dfs;
  a.cu_seqlens = f.cu_seqlens;
  a.dq = zeros(qk); a.dk = zeros(qk); a.dv = zeros(vv); a.dg = zeros(gg); a.dbeta = zeros(bb);
  a.dA_log = geti("want_dA_log") ? zeros(f.HV) : nullptr;
  a.ddt_bias = geti("want_ddt_bias") ? zeros((size_t)f.HV * f.K) : nullptr;
  a.dh0 = geti("want_dh0") ? zeros(st) : nullptr;
  {  // the outputs start as NaN except where the zeroing stage clears them: every element the
     // stages must write and do not shows up in the results
    float* outs[7] = {a.dq, a.dk, a.dv, a.dg, a.dbeta, a.dA_log, a.ddt_bias};
    const size_t sizes[7] = {qk, qk, vv, gg, bb, (size_t)f.HV, (size_t)f.HV * f.K};
    for (int o = 0; o < 7; ++o)
      if (outs[o] != nullptr) poison(outs[o], sizes[o] * sizeof(float));
    kda::bwd::ZeroRange z[14];
    const int nz = kda::bwd::zero_ranges(pl, z);
    for (int i = 0; i < nz; ++i)
      if (outs[z[i].out] != nullptr) memset(outs[z[i].out] + z[i].first, 0, z[i].count * sizeof(float));
  }
  a.ws = ws;
  a.status = &status;

  if (pl.varlen) {  // the chunk table the GPU's chunk-table kernel writes
    int64_t* cs = reinterpret_cast<int64_t*>(ws + pl.off_table);
    int64_t run = 0;
    for (int n = 0; n < f.N; ++n) {
      cs[n] = run;
      run += (f.cu_seqlens_host[n + 1] - f.cu_seqlens_host[n] + pl.C - 1) / pl.C;
    }
    cs[f.N] = run;
  }

  std::mt19937 rng((unsigned)geti("seed"));
  HostExec ex;
  ex.rng = &rng;
  auto with_smem = [&](size_t bytes, auto&& run) {
    void* sm = malloc(bytes ? bytes : 1);
    poison(sm, bytes);
    run(static_cast<float*>(sm));
    if (!ex.drained()) die("stage body ended with", "asynchronous copies not waited for");
    free(sm);
  };
  for (int64_t c = 0; c < pl.nct; ++c)
    for (int hv = 0; hv < pl.HV; ++hv)
      with_smem(kda::bwd::prep_smem(pl), [&](float* sm) { kda::bwd::prep_body(ex, a, c, hv, sm); });
  for (int64_t bid = 0; bid < kda::bwd::state_blocks(pl); ++bid)
    with_smem(kda::bwd::states_smem(pl), [&](float* sm) { kda::bwd::states_body(ex, a, bid, sm); });
  for (int64_t bid = 0; bid < kda::bwd::state_blocks(pl); ++bid)
    with_smem(kda::bwd::dstate_smem(pl), [&](float* sm) { kda::bwd::dstate_body(ex, a, bid, sm); });
  if (pl.tc_vprod)  // the products over v (a tensor-core stage on the GPU), plainly
    for (int64_t c = 0; c < pl.nct; ++c)
      for (int hv = 0; hv < pl.HV; ++hv)
        with_smem(16, [&](float* sm) { kda::bwd::vprod_body(ex, a, c, hv, sm); });
  for (int64_t c = 0; c < pl.nct; ++c)
    for (int hv = 0; hv < pl.HV; ++hv)
      with_smem(kda::bwd::grads_smem(pl), [&](float* sm) { kda::bwd::grads_body(ex, a, c, hv, sm); });
  for (int64_t c = 0; c < pl.nct; ++c)
    for (int hv = 0; hv < pl.HV; ++hv)
      with_smem(kda::bwd::gate_smem(pl), [&](float* sm) { kda::bwd::gate_body(ex, a, c, hv, sm); });

  save(dir, "dq", a.dq, qk);
  save(dir, "dk", a.dk, qk);
  save(dir, "dv", a.dv, vv);
  save(dir, "dg", a.dg, gg);
  save(dir, "dbeta", a.dbeta, bb);
  save(dir, "dA_log", a.dA_log, f.HV);
  save(dir, "ddt_bias", a.ddt_bias, (size_t)f.HV * f.K);
  save(dir, "dh0", a.dh0, st);
  FILE* sf = fopen((dir + "/out_status.txt").c_str(), "w");
  if (!sf) die("cannot write", "out_status.txt");
  fprintf(sf, "%u %zu\n", status, pl.total_bytes);
  fclose(sf);
  free(ws);
  return 0;
}
