/*
 * Oracle for the MTP speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded CPU
 * restatement of what the verify step computes, in double precision where the
 * arithmetic is floating point. Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it. The GPU library shares no code,
 * header, table or helper with it.
 *
 * Sources (web pages on MTP speculative decoding):
 *   [TRT]   "MTP in TensorRT-LLM on Blackwell" (makelele.cn): Fig. 1 (verify
 *           example), "MTP Vanilla"/"MTP Eagle" (KV of rejected drafts is
 *           cleared), "attention for MTP" (K+1 queries, causal mask).
 *   [SDMTP] "Speculative decoding and MTP" (mlqm.cn): §2.2-2.3 (parallel
 *           verify, accept / resample at first rejection), §4.3 (KV reuse),
 *           §4.4 (accept with min(1, p/q), temperature 0 = argmax rule).
 *   [K3]    "Multi Token Prediction" note (gitcode/csdn): "overall flow for
 *           K=3 draft tokens", steps 2, 4, 5, 6 (batched attention table,
 *           logits = H x W_o, softmax, compare with draft).
 *   [VLLM]  "MTP principles" (mqxn.cn): §三 stage 3 (greedy and rejection
 *           rules, resample), stage 4 (1..D+1 tokens out), §四 (example).
 *
 * Precision: floating point accumulates in double. Wherever a float decides an
 * integer (accept/reject, race winner) the decision is taken in fp32, the
 * precision the GPU takes it in; near-ties are flagged (tie_flags).
 *
 * Parity pins: every function here is checked by tests against worked
 * examples from the pages, brute force, closed forms and statistics; see the
 * test-suite.
 */
#ifndef MTP_ORACLE_H
#define MTP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type codes for tensors passed to the oracle. */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Return codes. */
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_INDEX = 4 };

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 * Easy as 1, 2, 3", SC'11): ctr[4], key[2] -> out[4]. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Verify attention with KV append ([K3] step 2; [TRT] attention for MTP).
 * R = D+1 rows per request. Row j of request b attends the ctx_lens[b] cached
 * keys plus verify keys 0..j (inclusive), after the verify tokens' K/V have
 * been written into slots ctx_lens[b] .. ctx_lens[b]+D of the paged cache.
 *   q        [B, R, Hq, d_qk]
 *   k_new    [B, R, Hkv, d_qk]            (MLA: latent [B, R, d_qk], Hkv = 1)
 *   v_new    [B, R, Hkv, d_v]             (MLA: NULL; V = first d_v of latent)
 *   k_cache  [num_blocks, block_size, Hkv, d_qk]   updated in place
 *   v_cache  [num_blocks, block_size, Hkv, d_v]    updated in place (MLA NULL)
 *   block_table [B, max_blocks], ctx_lens [B]
 *   out      [B, R, Hq, d_v]  (dtype as q)
 *   parents  [B, R] int32 or NULL (chain): tree drafts ([TRT] future work,
 *            Fig. 9), parents[b][0] = -1 and 0 <= parents[b][k] < k; row j
 *            then sees the context and the verify keys of the nodes on the
 *            path from the root to node j (itself included)
 *   out_exact [B, R, Hq, d_v] double or NULL: the same result before it is
 *            rounded to the output dtype
 * Returns ORACLE_BAD_INDEX if a block id needed is outside [0, num_blocks). */
int oracle_verify_attention(int B, int D, int Hq, int Hkv, int d_qk, int d_v,
                            int block_size, int max_blocks, int num_blocks,
                            int is_mla, float sm_scale, int dtype,
                            const void* q, const void* k_new, const void* v_new,
                            void* k_cache, void* v_cache,
                            const int32_t* block_table, const int32_t* ctx_lens,
                            void* out, const int32_t* parents, double* out_exact);

/* LM head + row statistics + acceptance ([K3] steps 4-6; [VLLM] §三 stages 3-4;
 * [SDMTP] §2.3, §4.4).
 *   hidden [B*R, H], lm_head [V, H] (dtype), tokens [B, R] = [input, d1..dD]
 *   mode [B]: 0 greedy, 1 rejection sampling (a request with mode 1 and
 *   temperature <= 0 is decided greedily: the T -> 0 limit), 2 relaxed
 *   acceptance ([TRT] "MTP optimization: relaxed acceptance", Fig. 6): draft
 *   d of row j is accepted iff d is among the row's relaxed_topk largest
 *   logits (lowest index first on equal logits) and its probability is at
 *   least the top-1 probability minus relaxed_delta (p = softmax of the
 *   logits, T = 1); the first miss is replaced by the row's argmax and the
 *   bonus is the argmax of row D, as for greedy requests
 *   temperature [B] (may be NULL when every request is greedy)
 *   q_draft [B, D, V] fp32 (may be NULL when every request is greedy)
 *   request_index [B]: the request number used as counter word 0 of the
 *   random stream (NULL: 0 .. B-1), so that a subset of a batch draws the
 *   same numbers as the full batch
 *   relaxed_topk, relaxed_delta: the relaxed rule's N (>= 1 when a request
 *   has mode 2) and delta (>= 0)
 * Outputs: out_tokens [B, R] (-1 padded), num_accepted [B] (drafts accepted,
 * 0..D; emitted = num_accepted + 1), tie_flags [B] (bit0: |p - U q| < 1e-5 q
 * at a decision, or for a relaxed decision |p_d - (p_1 - delta)| < 1e-3 or a
 * draft rank that moves across N when its logit moves by 1e-3 (1 + |l_d|);
 * bit1: top-2 race keys within 1e-5 relative), and optional lse_out [B, R],
 * argmax_out [B, R], logits_out [B*R, V] (fp32, / T).
 * parents [B, R] (NULL: chains): tree drafts, greedy requests only (a tree
 * with a sampling or relaxed request is BAD_ARG): node u is accepted when
 * every node on its root path carries the argmax of its parent's row; the
 * deepest accepted node (lowest index among equals) ends the path, and the
 * argmax of its row is the last emitted token. accepted_nodes [B, R]
 * (optional): the path's nodes, root (0) first, then -1. */
int oracle_lmhead_accept(int B, int D, int H, int V, int dtype,
                         const void* hidden, const void* lm_head,
                         const int32_t* tokens, const uint8_t* mode,
                         const float* temperature, const float* q_draft,
                         uint64_t seed, const int32_t* request_index,
                         int32_t* out_tokens, int32_t* num_accepted,
                         uint8_t* tie_flags, float* lse_out,
                         int32_t* argmax_out, float* logits_out,
                         int relaxed_topk, float relaxed_delta,
                         const int32_t* parents, int32_t* accepted_nodes);

/* KV-cache rollback ([TRT] "MTP Vanilla"/"MTP Eagle": KV of discarded drafts
 * is cleared; [K3] "rollback keeps the correct prefix").
 * seq_lens: in = context length before the step, out = ctx + n + 1.
 * Blocks holding slots ctx..ctx+D whose index is >= ceil(seq_len/block_size)
 * are appended to free_list at *free_count (request-major, block ascending)
 * and their table entries set to -1. */
int oracle_kv_rollback(int B, int D, int block_size, int max_blocks,
                       int32_t* block_table, int32_t* seq_lens,
                       const int32_t* num_accepted,
                       int32_t* free_list, int32_t* free_count);

/* KV compaction after a tree verify ([TRT] future work, Fig. 9): for
 * i = 1 .. num_accepted[b], the K/V in slot ctx + accepted_nodes[b][i] is
 * copied to slot ctx + i (in increasing i), so that the kept sequence is
 * contiguous for oracle_kv_rollback. Same cache layout as
 * oracle_verify_attention. */
int oracle_tree_kv_compact(int B, int D, int Hkv, int d_qk, int d_v, int block_size, int max_blocks,
                           int num_blocks, int is_mla, int dtype, void* k_cache, void* v_cache,
                           const int32_t* block_table, const int32_t* ctx_lens,
                           const int32_t* accepted_nodes, const int32_t* num_accepted);

/* Pieces of the acceptance rule exposed for pinning with fixed inputs. */

/* Relaxed acceptance of one row ([TRT] "MTP optimization: relaxed
 * acceptance"): logits [V] of the row (binary32), its log-sum-exp, the draft
 * token d. Returns 1 iff d is among the topk largest logits (lowest index
 * first on equal logits) and expf(l_d - lse) >= expf(l_max - lse) - delta,
 * both decided in binary32; *tie gets bit0 as described above. */
int oracle_relaxed_accept(int V, const float* logits, float lse, int d, int topk, float delta,
                          uint8_t* tie);

/* Rejection-sampling prefix rule ([VLLM] §三 stage 3, [SDMTP] §4.4):
 * accept draft j iff p[j] >= U[j] * q[j]; stop at the first failure.
 * Returns n (0..D); *tie gets bit0 if a decision had |p - U q| < 1e-5 q. */
int oracle_accept_prefix(int D, const float* p, const float* q, const float* U,
                         uint8_t* tie);

/* Exponential race: argmax_v w[v] / E[v] (lowest v on ties); weights that
 * are all zero return -1. *near_tie = 1 when the two best keys are within
 * 1e-5 relative. */
int oracle_race(int V, const float* w, const float* E, uint8_t* near_tie);

/* The uniforms the acceptance step draws: U for the accept test of row j and
 * E_v for the race key of vocab entry v at row j with tag t. */
float oracle_accept_uniform(uint64_t seed, uint32_t b, uint32_t j);
float oracle_race_exponential(uint64_t seed, uint32_t b, uint32_t j, uint32_t v, uint32_t tag);

#ifdef __cplusplus
}
#endif

#endif
