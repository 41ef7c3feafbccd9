/*
 * tr_synth.h -- device-side generators of the synthetic workload.
 *
 * These calls are NOT part of Token Recycling: they stand in for the target
 * model (its logits, hidden states and attention operands) and for a matrix
 * inherited from earlier requests, so the hot path can be driven and timed on
 * the GPU.  Each value is a pure function of (seed, tag, indices) through the
 * splitmix64 generator (Steele, Lea and Flood, OOPSLA 2014) with keys chained
 * field by field, h <- mix64(h + GAMMA + field); noise is Irwin-Hall of twelve
 * 16-bit uniforms, centred and scaled by 2^-16 (exact in fp32).  The Python
 * module `synth` implements the same definitions; a GPU test compares the two
 * bit for bit.  All pointers are device pointers; calls are asynchronous.
 */
#ifndef TR_SYNTH_H
#define TR_SYNTH_H

#include <stdint.h>

#include "tr.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Logits of the synthetic target for the tree nodes of one step:
 * row b*N + n of out [B*N, ld] is the target's scores after token
 * tree_tok[b, n] at position L[b] + depth(n): Irwin-Hall noise keyed on
 * (seed, 3, b, position, token, v), plus 6.0 on the token's Markov successor
 * and 3.0 on its 7 alternates.  ftype TR_F32 or TR_BF16 (rounded to nearest even). */
int trsyn_logits(uint64_t seed, int B, int64_t V, const struct tr_tree *tree, const int32_t *tree_tok,
                 const int32_t *L, tr_ftype ftype, void *out, int64_t ld, tr_stream_t stream);

/* bf16 noise rows out[((i0*n1 + i1)*n2 + i2), 0..d) keyed on (seed, tag, step, i0, i1, i2);
 * the per-step queries (tag 6) and tree keys/values (tags 7, 8). */
int trsyn_rows_bf16(uint64_t seed, int tag, int64_t step, int n0, int n1, int n2, int d, void *out,
                    tr_stream_t stream);

/* Prefix cache [B, H, cap, d] bf16: positions p < L[b] get the noise row keyed
 * on (seed, tag, b, h, p) (tags 9 for K, 10 for V); the rest is left as is. */
int trsyn_cache_bf16(uint64_t seed, int tag, int B, int H, int cap, int d, const int32_t *L, void *out,
                     tr_stream_t stream);

/* Hidden states of the fused-LM-head workload for the tree nodes of one step
 * (rows b*N + n of out [B*N, D] bf16): grid-rounded noise keyed on
 * (seed, 12, b, position, token) plus the token's class pattern. */
int trsyn_lm_hidden(uint64_t seed, int B, int D, const struct tr_tree *tree, const int32_t *tree_tok,
                    const int32_t *L, void *out, tr_stream_t stream);

/* Output projection Wt [V, D] bf16 of the fused-LM-head workload. */
int trsyn_lm_weight(uint64_t seed, int64_t V, int D, void *out, tr_stream_t stream);

/* Warm-start matrices M [B, V, K]: rows whose key (seed, 5, b, t) is even hold
 * the Markov successor and alternates of t, the others uniform random IDs. */
int trsyn_warm_matrix(uint64_t seed, int B, int64_t V, int K, tr_itype mtype, void *M, tr_stream_t stream);

/* Uniforms for acceptance under sampling, out [B, N, K1] fp32: entry
 * (b, n, j) is the top 24 bits of output j of the stream at key
 * (seed, 17, step, b, n), times 2^-24 (exact in fp32). */
int trsyn_uniforms(uint64_t seed, int64_t step, int B, int N, int K1, float *out, tr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TR_SYNTH_H */
