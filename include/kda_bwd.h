/*
 * kda_bwd.h -- C ABI of the backward pass of the GB300 chunk-parallel Kimi Delta Attention
 * forward (kda.h).
 *
 * The operation: for the forward pass that kda_fwd computes from fwd (same inputs, shapes and
 * options), and a loss whose gradients with respect to o and final_state are d_o and
 * d_final_state, write the gradient of that loss with respect to every input: q, k, v, the
 * raw gate input g, beta (the logits when beta_sigmoid), A_log, dt_bias and h0.
 *
 *   It follows the backward-propagation section of "Reading Notes: Implementation Notes for
 *   KDA in FLA" (chunk_kda_bwd): recompute U, W, Qg and the per-chunk states (steps 1-2),
 *   dV_new and dAqk from dO (step 3), the reverse cross-chunk recurrence of the state
 *   gradient (step 4), the WY gradients of v, beta and Akk (step 5), the intra-chunk terms of
 *   Aqk and Akk (step 6), and a reverse cumsum for the gate (step 7), followed by the
 *   backward of the gate activation ("FLA-KDA engineering notes", section 2), of the
 *   in-kernel L2 norm of q and k and of the beta sigmoid.
 *
 * Layouts (row-major, contiguous), with the forward's layouts in kda.h:
 *   d_o            [B, T, HV, V]   fwd.in_dtype, required
 *   d_final_state  [N, HV, K, V]   fp32, optional (NULL = 0); [N, HV, V, K] with state_v_first
 *   dq, dk         [B, T, H, K]    fp32, required
 *   dv             [B, T, HV, V]   fp32, required
 *   dg             [B, T, HV, K]   fp32, required: the gradient with respect to g as passed to
 *                                  the forward (the raw gate input, or the log decay when
 *                                  gate_mode is KDA_GATE_PREGATED)
 *   dbeta          [B, T, HV]      fp32, required
 *   dA_log         [HV]            fp32, optional; needs fwd.A_log and an in-kernel gate
 *   ddt_bias       [HV * K]        fp32, optional; needs fwd.dt_bias and an in-kernel gate
 *   dh0            [N, HV, K, V]   fp32, optional (also without fwd.h0: the gradient at a zero
 *                                  initial state); [N, HV, V, K] with state_v_first
 *   Rows of dq, dk, dv, dg and dbeta that no sequence covers (varlen padding) are set to 0.
 *
 * Arithmetic: fp32 on every dtype (bf16 inputs are widened exactly).  dq and dk sum the
 * contributions of the HV / H value heads that share a q / k head, and dA_log and ddt_bias
 * sum over tokens, with fp32 atomic adds: their rounding order is not fixed.  With HV == H,
 * dq, dk, dv, dg, dbeta and dh0 are the same bits on every run.
 *
 * Ownership: the caller owns every buffer; the library allocates no device memory.  The
 * workspace (kda_bwd_workspace_size bytes, 256-byte aligned) holds the recomputed forward
 * intermediates, the state before and the state gradient after every chunk.  Device
 * pointers must be 16-byte aligned.
 *
 * Errors: checks run on the host before any CUDA call and return a status (kda_status of
 * kda.h, with kda_last_error() giving the message); nothing is thrown across this ABI.  The
 * forward's rules (kda_fwd_check) apply to fwd with d_o in the place of o; fwd.o,
 * fwd.final_state, fwd.h_out, fwd.workspace and fwd.workspace_bytes are not used.
 */
#ifndef KDA_GB300_BWD_H
#define KDA_GB300_BWD_H

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kda_bwd_params {
  kda_fwd_params fwd;         /* the forward pass being differentiated (inputs and options) */
  const void* d_o;            /* gradient of o */
  const float* d_final_state; /* gradient of final_state, optional */
  float* dq;
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  float* dA_log;              /* optional */
  float* ddt_bias;            /* optional */
  float* dh0;                 /* optional */
  void* workspace;
  size_t workspace_bytes;
} kda_bwd_params;

/* Argument checks of kda_bwd without launching anything (host only, no CUDA call). */
kda_status kda_bwd_check(const kda_bwd_params* p);

/* Bytes of workspace kda_bwd needs for these parameters (0 if they are invalid).  Host
   only; makes no CUDA call.  About (11 C K + 4 C V + 2 C^2 + C + K) * 4 bytes per chunk and
   value head for the recomputed intermediates plus 2 K V * 4 bytes per chunk and value head
   for the states. */
size_t kda_bwd_workspace_size(const kda_bwd_params* p);

/* Number of kernel launches one kda_bwd call makes (0 if the parameters are invalid): the
   chunk table (varlen only), prep, states, state gradient, the products over v (bf16 inputs
   with K = V = 128 and chunk 64 only), gradients and gate (the gate, beta and L2-norm
   backward).  The zeroing stage (cudaMemsetAsync of
   what atomics accumulate into, dA_log, ddt_bias and, with HV > H, dq and dk, and of the rows
   no sequence covers; every other output element is written once by the kernels) is not
   counted.  Host only. */
int32_t kda_bwd_num_launches(const kda_bwd_params* p);

/* Number of stages of kda_bwd for these parameters (0 if they are invalid): the zeroing of
   the outputs, then the kernels kda_bwd_num_launches counts.  Host only. */
int32_t kda_bwd_num_stages(const kda_bwd_params* p);

/* Name of stage `stage` ("zero_outputs", "chunk_table", "bwd_prep", "bwd_states",
   "bwd_dstate", "bwd_vprod", "bwd_grads", "bwd_gate"); "" if out of range or the parameters
   are invalid. */
const char* kda_bwd_stage_name(const kda_bwd_params* p, int32_t stage);

/* Enqueue only stage `stage` of kda_bwd on `stream`.  Calling every stage in order on one
   stream computes exactly what kda_bwd computes; the split exists so that a caller can put
   timing events between the kernels.  Same checks and errors as kda_bwd. */
kda_status kda_bwd_stage(const kda_bwd_params* p, void* stream, int32_t stage);

/* The backward pass, enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
   Asynchronous: returns once the work is enqueued.  The state-gradient stage runs on a
   library-owned stream (one per device, created on the first call) beside the state stage:
   it is forked from `stream` after the recompute stage and joined back before the next
   stage with events, so the call stays ordered on `stream` and can be captured into a CUDA
   graph.  Returns KDA_ERR_CUDA if a launch fails or that stream cannot be created;
   kda_get_device_status reports inconsistent device-side cu_seqlens as for kda_fwd. */
kda_status kda_bwd(const kda_bwd_params* p, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_BWD_H */
