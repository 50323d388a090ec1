/*
 * kda_cp.h -- context parallelism for the GB300 KDA forward pass: one long sequence
 * sharded over ranks along time.
 *
 * The state recurrence of "Reading Notes: Implementation Notes for KDA in FLA",
 * forward step 4 (S <- Diag(e^gamma_C) S + Kg^T (U - W S), per chunk), is affine in
 * the state.  So a shard of tokens acts on the state that enters it as
 *
 *     S_out = P S_in + R        P: K x K (the shard's transition), R: K x V,
 *
 * per (sequence, value head), with P and R depending only on the shard's own q, k,
 * v, g, beta.  The ranks form their shards' maps, exchange them, and each rank
 * chains the maps of the shards before its own (an exclusive prefix) to obtain the
 * state entering its shard; then it runs the forward pass on its shard from that
 * state.  The flag table of "FLA-KDA engineering notes" section 2.2 names this
 * option (cp_context); the mechanism is the plain reading of the affine step above.
 * The maps themselves come from kda_fwd (include/kda.h): R is the final state of
 * the shard run from a zero initial state, and P is the final state of the shard
 * run with v = 0 from the identity (K = V), because with v = 0 the recurrence is
 * linear in the state.  This header declares the one extra kernel the exchange
 * needs: applying a batch of maps.
 */
#ifndef KDA_GB300_CP_H
#define KDA_GB300_CP_H

#include <stddef.h>
#include <stdint.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* S_out[i] = P[i] S_in[i] + R[i] for i = 0 .. nmaps-1, fp32, on `stream`
   (asynchronous).
   Layouts (row-major, contiguous, device memory, 4-byte aligned):
     P      [nmaps, K, K]   the transition of each map (acts on the left of a K x V state)
     R      [nmaps, K, V]   ([nmaps, V, K] with state_v_first)
     S_in   [nmaps, K, V]   ([nmaps, V, K] with state_v_first); NULL = zero states
     S_out  [nmaps, K, V]   ([nmaps, V, K] with state_v_first)
   With state_v_first every state and R are stored transposed (the layout of
   kda_fwd_params.state_v_first) and S_out^T = S_in^T P^T + R^T; P keeps its layout.
   Ownership: the caller owns every buffer; nothing is allocated.  S_out must not
   overlap P, R or S_in (KDA_ERR_INVALID_ARG when it starts at the same address as
   one of them; partial overlap is the caller's error and is not detected).
   Errors: K or V outside 1..256, nmaps < 0, a NULL P / R / S_out or a misaligned
   pointer return KDA_ERR_SHAPE / KDA_ERR_INVALID_ARG before any CUDA call; a
   failed launch returns KDA_ERR_CUDA.  nmaps == 0 launches nothing. */
kda_status kda_state_affine_apply(const float* P, const float* R, const float* S_in, float* S_out,
                                  int64_t nmaps, int32_t K, int32_t V, int32_t state_v_first,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_CP_H */
