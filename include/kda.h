/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunk-parallel Kimi Delta Attention forward pass.
 *
 * The operation (one call computes all of it on the GPU):
 *
 *   For every sequence n and value head hv (q/k head h = hv / (HV/H)), with the
 *   activated log-decay gate g'_t in R^K and alpha_t = exp(g'_t):
 *       S_t = Diag(alpha_t) S_{t-1} - beta_t k_t (k_t^T Diag(alpha_t) S_{t-1}) + beta_t k_t v_t^T
 *       o_t = scale * S_t^T q_t
 *   S_0 = initial state (or 0), final_state = S at the end of the sequence.
 *
 *   It is evaluated in the chunk-parallel form of "Reading Notes: Implementation
 *   Notes for KDA in FLA" (forward pass, steps 1-5): chunk-local cumsum of the
 *   gate, intra-chunk Aqk / Akk with (I + Akk)^-1, WY recompute of U and W, the
 *   sequential inter-chunk state recurrence, and the output.
 *
 *   Gate modes ("FLA-KDA engineering notes", section 2, gate input contracts),
 *   x = g + dt_bias (dt_bias optional):
 *       KDA_GATE_PREGATED  g is already the log decay (use_gate_in_kernel=False)
 *       KDA_GATE_PLAIN     g' = -exp(A_log) * softplus(x)
 *       KDA_GATE_SAFE      g' = lower_bound * sigmoid(exp(A_log) * x), in [lower_bound, 0);
 *                          A_log may be NULL, then g' = lower_bound * sigmoid(x)
 *
 * Layouts (row-major, contiguous; same section and section 2.1 of the notes):
 *   q, k      [B, T, H,  K]      in_dtype
 *   v         [B, T, HV, V]      in_dtype
 *   g         [B, T, HV, K]      in_dtype (raw gate input, or log decay if PREGATED)
 *   beta      [B, T, HV]         in_dtype (logits if beta_sigmoid, else the value)
 *   A_log     [HV]               fp32
 *   dt_bias   [HV * K]           fp32 (same memory as [HV, K])
 *   h0        [N, HV, K, V]      fp32 (state stored d_k x d_v, forward step 4 of the reading notes;
 *                                [N, HV, V, K] with state_v_first)
 *   o         [B, T, HV, V]      in_dtype
 *   final_state [N, HV, K, V]    fp32 (layout as h0)
 *   cu_seqlens [N + 1]           int64; with it B must be 1 and sequence n spans tokens
 *                                [cu[n], cu[n+1]) of the flattened batch (varlen, section 2.2)
 *
 * Ownership: the caller owns every buffer.  The library allocates no device
 * memory; the caller provides a workspace of at least kda_fwd_workspace_size()
 * bytes.  Device pointers must be 16-byte aligned, the workspace 256-byte aligned.
 *
 * Errors: argument checks run on the host before any CUDA call and return a
 * status; nothing is thrown across this ABI.  kda_last_error() gives a
 * thread-local message for the last failing call on this thread.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,   /* NULL pointer, misalignment, bad flag or range */
  KDA_ERR_SHAPE = 2,         /* K > 256, HV % H != 0, chunk_size not 32/64, bad cu_seqlens */
  KDA_ERR_DTYPE = 3,         /* unknown in_dtype */
  KDA_ERR_UNSUPPORTED = 4,   /* a combination this build does not implement */
  KDA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
  KDA_ERR_DEVICE_STATUS = 6, /* a kernel flagged an inconsistency (see kda_get_device_status) */
  KDA_ERR_WORKSPACE = 7      /* workspace NULL, too small or misaligned */
} kda_status;

typedef enum { KDA_GATE_PREGATED = 0, KDA_GATE_PLAIN = 1, KDA_GATE_SAFE = 2 } kda_gate_mode;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

/* Device status bits (kda_get_device_status). */
#define KDA_DEV_BAD_SEQLENS 0x1u   /* device cu_seqlens disagree with the host copy */
#define KDA_DEV_TIMEOUT     0x2u   /* a bounded wait in a kernel ran out */

typedef struct kda_fwd_params {
  int32_t B, T, H, HV, K, V;
  int32_t chunk_size;        /* 32 or 64 ("FLA-KDA engineering notes", section 2.1) */
  int32_t in_dtype;          /* kda_dtype of q, k, v, g, beta and o */
  int32_t gate_mode;         /* kda_gate_mode */
  float lower_bound;         /* SAFE only: -5 <= lower_bound < 0 (section 2.1) */
  float scale;               /* multiplies q; the usual choice is K^-0.5 */
  int32_t qk_l2norm;         /* 1: q, k are L2-normalised in-kernel over K (section 2.2) */
  int32_t beta_sigmoid;      /* 1: beta holds logits, the kernel applies sigmoid (section 2.2) */
  int32_t N;                 /* number of sequences: B, or len(cu_seqlens) - 1 */
  int32_t allow_neg_eigval;  /* 1: beta = 2 sigmoid(logit) in [0, 2), so that the transition
                                I - beta k k^T may have a negative eigenvalue; needs
                                beta_sigmoid ("FLA-KDA engineering notes", section 2.1) */
  int32_t state_v_first;     /* 1: h0 and final_state are stored [N, HV, V, K] (the state
                                transposed; "FLA-KDA engineering notes", section 2.2,
                                transpose_state_layout) */
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* beta;
  const float* A_log;        /* required for PLAIN, optional for SAFE, ignored for PREGATED */
  const float* dt_bias;      /* optional (NULL = 0) */
  const float* h0;           /* optional (NULL = zero initial state) */
  const int64_t* cu_seqlens; /* device, optional (varlen) */
  const int64_t* cu_seqlens_host; /* host copy of cu_seqlens, required with it */
  void* o;                   /* output */
  float* final_state;        /* output, optional (NULL = not written) */
  float* h_out;              /* output, optional: the state before every chunk
                                ("return_intermediate_states", "FLA-KDA engineering notes"
                                section 2.2),
                                [nct, HV, K, V] fp32 ([nct, HV, V, K] with state_v_first), chunk c
                                of sequence n at index (chunks of sequences 0..n-1) + c;
                                nct from kda_fwd_num_chunks */
  void* workspace;
  size_t workspace_bytes;
} kda_fwd_params;

/* Bytes of workspace kda_fwd needs for these parameters (0 if they are invalid).
   Host only; makes no CUDA call. */
size_t kda_fwd_workspace_size(const kda_fwd_params* p);

/* Argument checks of kda_fwd without launching anything (host only, no CUDA call).
   Rules: "FLA-KDA engineering notes" section 2.1 (A_log required for the plain
   in-kernel gate; -5 <= lower_bound < 0 for the safe gate; chunk_size 32 or 64;
   K <= 256; HV % H == 0; fp32 initial state) and "FlashKDA gate-bias load path"
   section 4 (fp32 A_log / dt_bias, a clear error rather than a silent one). */
kda_status kda_fwd_check(const kda_fwd_params* p);

/* The forward pass, enqueued on `stream` (a cudaStream_t; NULL = legacy default
   stream).  Asynchronous: returns once the kernels are enqueued.  Writes o and,
   if non-NULL, final_state.  Rows of o that no sequence covers (varlen padding:
   tokens cu_seqlens[N] .. B*T - 1) are set to zero, as the token recurrence
   defines them.  Returns KDA_ERR_CUDA if a launch fails.
   When few (sequence, value head) recurrences would leave most SMs idle (bf16
   tensor-core path, N * HV <= 96, at least 200 chunks), the chunk range is cut into up
   to 10 segments: the intra-chunk kernel of segment k+1 runs on `stream` (a programmatic
   dependent of segment k's, with which it shares no data, so that it starts while that
   one's last CTAs run) while the recurrence of segment k runs on a library-owned stream of
   the highest priority, the fp32 state carried between segments in the workspace.  The
   work is still ordered after everything enqueued on `stream` before the call and before
   everything enqueued after it (event fork / join, valid under stream capture); results
   are bit-identical to the stages run one by one (kda_fwd_num_launches: kernel count). */
kda_status kda_fwd(const kda_fwd_params* p, void* stream);

/* Number of kernel launches one kda_fwd call makes for these parameters (0 if
   they are invalid).  Host only; makes no CUDA call. */
int32_t kda_fwd_num_launches(const kda_fwd_params* p);

/* Bytes of device arena kda_fwd_host needs for these parameters (0 if they are
   invalid): device copies of every tensor plus the pass's workspace.  Host only;
   makes no CUDA call. */
size_t kda_fwd_host_arena_size(const kda_fwd_params* p);

/* kda_fwd on HOST buffers: q, k, v, g, beta, A_log, dt_bias, h0 and
   cu_seqlens_host are read from host memory, o, final_state and h_out written to
   host memory (the device field cu_seqlens and workspace / workspace_bytes are
   ignored; varlen is selected by cu_seqlens_host).  Everything runs in `arena`
   (device memory the caller owns, kda_fwd_host_arena_size bytes, 256-byte
   aligned).  With the pipelined schedule the input rows of segment k+1 are copied
   in while segment k computes and the output rows of each segment are copied out
   as soon as its recurrence finishes, on library-owned copy streams; page-locked
   (pinned) host memory lets these copies run asynchronously.  Ordered on `stream`
   like kda_fwd; the host buffers must stay valid, and o / final_state / h_out may
   be read, only once `stream` has passed this call.  Rows of o that no sequence
   covers are set to zero (copied out from the arena like the others).  The
   source pages have no counterpart to this entry
   point: it is the end-to-end path of a caller whose tensors live in host memory. */
kda_status kda_fwd_host(const kda_fwd_params* p, void* arena, size_t arena_bytes, void* stream);

/* The same forward pass as a token recurrence (decode and short prefill;
   "FLA-KDA engineering notes", section 1, fused_recurrent_kda): per token alpha = exp(g'), S <- Diag(alpha) S,
   S <- S + beta k (v - S^T k)^T, o = scale S^T q, the state read from h0 (or 0)
   and written to final_state.  Same parameters, checks, layouts and outputs as
   kda_fwd, except: chunk_size and the workspace are not used (no workspace is
   needed), and h_out must be NULL.  fp32 arithmetic on every dtype.  Each CTA
   owns one (sequence, value head) and a range of V columns (all 128 of them for
   K = V = 128), processes the tokens in order and keeps the state in registers
   (K <= 128) or shared memory (K > 128).  Asynchronous on `stream`. */
kda_status kda_fused_recurrent_fwd(const kda_fwd_params* p, void* stream);

/* Number of chunks over all sequences, the first dimension of h_out (0 if the
   parameters are invalid).  Host only; makes no CUDA call. */
int64_t kda_fwd_num_chunks(const kda_fwd_params* p);

/* Number of stages of the forward pass for these parameters (0 if they are
   invalid): chunk table (varlen only), intra-chunk kernel, recurrence kernel.
   Host only; makes no CUDA call. */
int32_t kda_fwd_num_stages(const kda_fwd_params* p);

/* Name of stage `stage` (0 <= stage < kda_fwd_num_stages), "" if out of range. */
const char* kda_fwd_stage_name(const kda_fwd_params* p, int32_t stage);

/* Enqueue only stage `stage` of kda_fwd on `stream`, as one launch over the whole
   chunk range.  Calling every stage in order on one stream computes exactly what
   kda_fwd computes (bit-identical); the split exists so that a caller can put
   timing events between the kernels.  Same checks and errors as kda_fwd. */
kda_status kda_fwd_stage(const kda_fwd_params* p, void* stream, int32_t stage);

/* Size of the static device scratch that kda_fwd_noalloc uses: 32 MiB. */
#define KDA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* kda_fwd for callers that cannot allocate device memory.  The source pages
   have no counterpart to this entry point.
   Some callers cannot call cudaMalloc or hand the library a workspace: code that
   runs where an allocator is unavailable or forbidden (inside a framework that
   owns all device memory, a real-time loop that must not allocate, a plugin
   with no allocator handle).  This entry point takes the same parameters as
   kda_fwd, ignores p->workspace / p->workspace_bytes, and puts its scratch in a
   library-owned static device array of KDA_NOALLOC_SCRATCH_BYTES bytes instead.
   Every GPU that loads the library holds that array until the process exits.
   It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
   - Sizes whose kda_fwd_workspace_size exceeds KDA_NOALLOC_SCRATCH_BYTES are
     rejected with KDA_ERR_WORKSPACE and a message giving both sizes.
   - The first call on each device looks up the array's device address
     (cudaGetSymbolAddress) with that device current; make that first call
     before any stream capture.  That lookup is its only set-up: the stages run
     one after another on `stream` (bit-identical to kda_fwd), so this entry
     point creates none of the library's internal streams or events.
   - All calls share the one array and it keeps the last call's contents.
     Nothing in it needs to start at zero: every call writes each scratch
     element it later reads.  Calls whose kernels overlap on the GPU (on
     different streams, or from several host threads) race on the array: order
     them on one stream or synchronise between them. */
kda_status kda_fwd_noalloc(const kda_fwd_params* p, void* stream);

/* Synchronises `stream`, returns the device status bits accumulated by earlier
   calls (KDA_DEV_*) and clears them.  0 means no kernel flagged anything. */
uint32_t kda_get_device_status(void* stream);

/* Static description of a status code. */
const char* kda_status_string(kda_status s);

/* Message of the last failing call on the calling thread ("" if none). */
const char* kda_last_error(void);

/* ABI version of this header (incremented on incompatible changes). */
int32_t kda_abi_version(void);

#define KDA_ABI_VERSION 2

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
