/*
 * mtp_verify.h - C ABI of the GB300 library for the verify step of MTP
 * (multi-token prediction) speculative decoding.
 *
 * One verify step over a batch of B requests, each with R = D+1 verify
 * tokens [input/bonus token, d_1 .. d_D], is three calls on one stream:
 *
 *   1. mtp_verify_attention     multi-query attention of the R rows against
 *                               the request's paged KV cache plus the verify
 *                               tokens' own K/V (causal within the chain),
 *                               after appending those K/V to the cache;
 *   2. mtp_verify_logits_accept LM head over the R hidden states with
 *                               streaming softmax statistics / argmax, then
 *                               greedy or rejection-sampling acceptance;
 *   3. kv_rollback              truncate the cache to the kept prefix and
 *                               release blocks that only held rejected drafts.
 *
 * Sources (web pages on MTP speculative decoding):
 *   "MTP in TensorRT-LLM on Blackwell" (makelele.cn): Fig. 1 verification
 *       example; MTP Vanilla / MTP Eagle (KV of rejected drafts is cleared);
 *       "attention for MTP" (K+1 input tokens, causal mask); Fig. 4 workflow.
 *   "Speculative decoding and MTP" (mlqm.cn): §2.2-2.3 parallel verification,
 *       acceptance and correction; §4.3 KV cache reuse; §4.4 accept with
 *       min(1, p/q), temperature 0 = argmax rule.
 *   "Multi Token Prediction" note (gitcode/csdn): KV cache reuse + batched
 *       forward; overall flow for K=3 draft tokens, steps 2 and 4-6.
 *   "MTP principles" (mqxn.cn): §三 stage 3 (greedy / rejection sampling),
 *       stage 4 (1 .. D+1 tokens per step), §四 worked example.
 *
 * Conventions (all calls):
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise;
 *     the library allocates no device memory of its own apart from one
 *     4-byte device error word per device.
 *   - Scratch space is a caller-provided device buffer ("workspace") of at
 *     least the size the matching *_workspace_size() call reports, 256-byte
 *     aligned. Its contents need not be initialised; it must not be used by
 *     another call that may run concurrently.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Arguments are validated on the host before anything
 *     is launched; device-side range checks (block ids, token ids, lengths)
 *     set the device error word, which mtp_sync_status() reports.
 *   - Return value: one of the mtp_status codes. On failure,
 *     mtp_last_error() returns a message (thread-local, valid until the next
 *     call on the same thread). No C++ exception crosses this boundary.
 *   - Tensors are dense and row-major in the shapes given; bf16 tensors hold
 *     IEEE bfloat16 values.
 *   - The first call on a device allocates the error word and queries kernel
 *     attributes and occupancies (cached per device); make it outside stream
 *     capture. Later calls launch kernels only and can be captured into a
 *     CUDA graph.
 */
#ifndef MTP_VERIFY_H
#define MTP_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MTP_ABI_VERSION 5

typedef enum {
  MTP_OK = 0,
  MTP_INVALID_ARG = 1,   /* null pointer, bad shape, D > MTP_MAX_DRAFTS, block_size != 64, ... */
  MTP_UNSUPPORTED = 2,   /* dtype / shape combination the library does not provide */
  MTP_CUDA_ERROR = 3,    /* a CUDA runtime call or launch failed */
  MTP_DEVICE_ERROR = 4   /* a device-side range check tripped (see mtp_sync_status) */
} mtp_status;

typedef enum { MTP_F32 = 0, MTP_BF16 = 1 } mtp_dtype;

#define MTP_MAX_DRAFTS 15    /* D <= 15, so R = D+1 <= 16 verify rows per request */
#define MTP_BLOCK_SIZE 64    /* tokens per KV-cache block */

/* Device error word bits (reported by mtp_sync_status). */
#define MTP_ERR_BLOCK_ID   0x1u  /* block id outside [0, num_blocks) or table entry < 0 */
#define MTP_ERR_TOKEN_ID   0x2u  /* token id outside [0, V) */
#define MTP_ERR_LENGTH     0x4u  /* context/seq length < 0, or slots beyond max_blocks */
#define MTP_ERR_ACCEPTED   0x8u  /* num_accepted outside [0, D] */
#define MTP_ERR_FREE_LIST  0x10u /* free list capacity exceeded */
#define MTP_ERR_TIMEOUT    0x20u /* a bounded wait inside a kernel gave up */
#define MTP_ERR_MODE       0x40u /* mode > 2, or mode 2 while relaxed_topk is 0 (decided greedily) */
#define MTP_ERR_TREE       0x80u /* malformed parents list (that request is treated as a chain) */

/* ------------------------------------------------------------------------ */
/* 1. Verify attention with KV append.
 *
 * Defined by: "Multi Token Prediction" note, overall flow for K=3 draft
 * tokens, step 2 (batched Q against the reused cache; each verify token's new
 * K/V is added to the cache and seen by the following ones) and
 * "MTP in TensorRT-LLM", attention for MTP (K+1 queries, a causal mask).
 *
 * For request b with cached length ctx = ctx_lens[b]:
 *   append: K/V of verify token j are written into slot ctx+j of the paged
 *           cache (block block_table[b][(ctx+j)/64], offset (ctx+j)%64);
 *   attend: row j, query head h attends slots 0 .. ctx+j (inclusive) of KV
 *           head h / (Hq/Hkv):
 *             out[b,j,h,:] = softmax_t(sm_scale * q[b,j,h,:].k_t) . v_t
 * Absorbed MLA (is_mla = 1): one latent vector of width d_qk per token is
 * both the key and, through its first d_v entries, the value; Hkv = 1,
 * v_new and v_cache are NULL.
 * Tree drafts ("MTP in TensorRT-LLM on Blackwell", future work: tree
 * speculative sampling, Fig. 9), when `parents` is given: verify token j is
 * node j of a tree, node 0 the input token and node k >= 1 a child of
 * parents[b][k] (0 <= parents[b][k] < k, parents[b][0] = -1). Row j then
 * attends slots 0 .. ctx-1 and ctx+k for every node k on the path from the
 * root to node j (itself included). parents = NULL is the chain
 * (parents[b][k] = k-1). A malformed list sets MTP_ERR_TREE and that request
 * is computed as a chain.
 *
 * Layouts (dtype as given; MTP_F32 or MTP_BF16):
 *   q           [B, R, Hq, d_qk]
 *   k_new       [B, R, Hkv, d_qk]        (MLA: [B, R, d_qk])
 *   v_new       [B, R, Hkv, d_v]         (MLA: NULL)
 *   k_cache     [num_blocks, 64, Hkv, d_qk]   written at the verify slots
 *   v_cache     [num_blocks, 64, Hkv, d_v]    (MLA: NULL)
 *   block_table [B, max_blocks] int32;  ctx_lens [B] int32
 *   parents     [B, R] int32 or NULL
 *   out         [B, R, Hq, d_v]
 * Requirements: R = D+1 <= 16; block_size == 64; Hq % Hkv == 0;
 *   GQA/MHA: d_qk == d_v, a multiple of 32, <= 256 (bf16: 64 or 128);
 *   MLA (bf16 only): d_qk == 576, d_v == 512.
 *   Every block of slots 0 .. ctx+D must be present in the table.
 * Inputs other than the cache slots being appended are not modified.
 */
typedef struct {
  const void* q;
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  void* out;
  int32_t B, D, Hq, Hkv, d_qk, d_v;
  int32_t block_size, max_blocks, num_blocks, is_mla;
  float sm_scale;
  int32_t dtype;             /* mtp_dtype */
  const int32_t* parents;    /* [B, R] tree drafts, NULL: chains */
  void* workspace;           /* device, >= mtp_attention_workspace_size() bytes */
  size_t workspace_bytes;
  void* timing_events[2];    /* optional cudaEvent_t pair recorded on `stream` just before and just
                                after the attention kernel proper (append and combine excluded) */
} mtp_attn_args;

size_t mtp_attention_workspace_size(const mtp_attn_args* args);
int mtp_verify_attention(const mtp_attn_args* args, void* stream);

/* ------------------------------------------------------------------------ */
/* 2. LM head, streaming softmax statistics and acceptance.
 *
 * Defined by: "Multi Token Prediction" note, K=3 flow steps 4-6
 * (Logits_i = H_i x W_o for all verify rows in one product, softmax, compare
 * with the drafts); "MTP principles" §三 stage 3 (greedy: accept while the
 * draft equals the target argmax; rejection sampling: accept if
 * P_target/P_draft >= U, otherwise resample) and stage 4 (1 .. D+1 tokens);
 * "Speculative decoding and MTP" §2.3 (stop at the first rejection and draw
 * the replacement from the target's distribution at that position) and §4.4
 * (accept with probability min(1, p/q); temperature 0 = argmax rule).
 *
 * Row m = b*R + j of `hidden` is the target's last hidden state for verify
 * token j of request b; its logits are l[m,v] = sum_k hidden[m,k] W[v,k].
 * Sampling rows use l / T.
 *   greedy request (mode 0, or mode 1 with temperature <= 0):
 *     n = number of leading j < D with argmax(row j) == tokens[b, j+1];
 *     out_tokens[b] = [d_1 .. d_n, argmax(row n)].
 *   relaxed request (mode 2; "MTP in TensorRT-LLM on Blackwell", MTP
 *   optimization: relaxed acceptance, used in a reasoning model's thinking
 *   phase): p_j = softmax(l_j) (no temperature). Draft d_{j+1} is accepted
 *   iff it is among the relaxed_topk largest logits of row j (lowest id first
 *   on equal logits) and p_j(d_{j+1}) >= max_v p_j(v) - relaxed_delta; stop
 *   at the first miss; out_tokens[b] = [d_1 .. d_n, argmax(row n)].
 *   rejection-sampling request (mode 1, temperature > 0):
 *     p_j = softmax(l_j / T). For j = 0 .. D-1: accept d_{j+1} iff
 *     p_j(d_{j+1}) >= U_j * q[b, j, d_{j+1}] (U_j uniform in [0,1)), stop at
 *     the first rejection j* and emit a draw from normalised
 *     max(0, p_j* - q_j*) (from p_j* if that is zero everywhere); if every
 *     draft is accepted emit a draw from p_D.
 *   tree drafts (`parents` given; "MTP in TensorRT-LLM on Blackwell", future
 *   work: tree speculative sampling): row j is node j of a tree as in
 *   mtp_verify_attention, tokens[b][k] the draft token of node k >= 1.
 *   Trees are verified greedily: node u is accepted when every node on the
 *   path from the root to u carries the argmax of its parent's row; the
 *   accepted node of greatest depth (lowest index among equally deep ones)
 *   ends the path u_0 = 0, u_1 .. u_n; out_tokens[b] = [tokens[u_1] ..
 *   tokens[u_n], argmax(row u_n)]. A tree request with mode 1 (temperature
 *   > 0) or mode 2 sets MTP_ERR_MODE and is verified greedily; a malformed
 *   parents list sets MTP_ERR_TREE and that request is verified as a chain.
 * Random numbers: Philox4x32-10 (Salmon et al., SC'11), key = seed (low,
 * high 32 bits), counter = (b, j, v, tag), output word 0:
 *   U_j   = (x >> 8) * 2^-24                                   tag 1, v = 0
 *   draws = argmax_v w_v / E_v,  E_v = -log1p(-x * 2^-32)      tag 2 residual, 3 bonus
 * so tokens are reproducible bit for bit across runs and batch layouts.
 *
 * Layouts:
 *   hidden      [B*R, H]   dtype;   lm_head [V, H] dtype (row v = token v)
 *   tokens      [B, R] int32 = [input/bonus, d_1 .. d_D]
 *   mode        [B] uint8 (0 greedy, 1 rejection sampling, 2 relaxed)
 *   temperature [B] float (NULL allowed when no request samples)
 *   q_draft     [B, D, V] float, the drafter's distributions (NULL allowed
 *               when no request samples, or when D = 0); only rows of
 *               sampling requests are read.
 * Outputs:
 *   out_tokens   [B, R] int32: n+1 emitted tokens then -1
 *   num_accepted [B] int32: n in [0, D] (tokens emitted = n + 1)
 *   tie_flags    [B] uint8: bit0 = an accept decision had |p - U q| < 1e-5 q,
 *                or a relaxed decision had |p_d - (p_1 - delta)| < 1e-3 or a
 *                rank that crosses relaxed_topk when l_d moves by
 *                1e-3 (1 + |l_d|); bit1 = the two best race keys were within
 *                1e-5 relative
 *   lse_out      [B*R] float (optional): log-sum-exp of row (scaled) logits
 *   argmax_out   [B*R] int32 (optional): argmax of row, lowest id on ties
 *   logits_debug [B*R, V] float (optional, validation only): scaled logits
 *   accepted_nodes [B, R] int32 (optional): the accepted path's nodes u_0 = 0,
 *                u_1 .. u_n, then -1 (for a chain: 0 .. n); the input of
 *                mtp_tree_kv_compact
 * dtype MTP_F32 takes H a multiple of 4; MTP_BF16 takes H a multiple of 64.
 */
typedef struct {
  const void* hidden;
  const void* lm_head;
  const int32_t* tokens;
  const uint8_t* mode;
  const float* temperature;
  const float* q_draft;
  uint64_t seed;
  int32_t* out_tokens;
  int32_t* num_accepted;
  uint8_t* tie_flags;
  float* lse_out;
  int32_t* argmax_out;
  float* logits_debug;
  int32_t B, D, H, V;
  int32_t dtype;             /* mtp_dtype */
  int32_t any_sampling;      /* 0: every request is greedy (q_draft/temperature unused) */
  int32_t relaxed_topk;      /* N of the relaxed rule (0: no request uses mode 2), <= V */
  float relaxed_delta;       /* delta of the relaxed rule, >= 0 */
  const int32_t* parents;    /* [B, R] tree drafts, NULL: chains */
  int32_t* accepted_nodes;   /* [B, R] optional output */
  void* workspace;           /* device, >= mtp_lmhead_workspace_size() bytes */
  size_t workspace_bytes;
  void* timing_events[2];    /* optional cudaEvent_t pair recorded on `stream` just before and just
                                after the LM-head GEMM kernel (acceptance kernels excluded) */
  void* q_ready_event;       /* optional cudaEvent_t: after launching the LM-head GEMM the call makes
                                `stream` wait for it (cudaStreamWaitEvent) before the first kernel
                                that reads q_draft, so a caller can still be copying q_draft (e.g.
                                from host memory on another stream) while the GEMM runs; the event
                                must have been recorded (or be recorded in the same graph capture)
                                after that copy. NULL: q_draft is complete when the call is made. */
} mtp_lmhead_args;

size_t mtp_lmhead_workspace_size(const mtp_lmhead_args* args);
int mtp_verify_logits_accept(const mtp_lmhead_args* args, void* stream);

/* 2b. The same call for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that have no way to provide a workspace: for example a plugin inside an
 * inference engine that owns all device memory and gives plugins none, or a
 * latency-critical loop where cudaMalloc's implicit device-wide
 * synchronisation is not acceptable.
 *
 * Arguments, results and errors are those of mtp_verify_logits_accept, except
 * that `workspace` and `workspace_bytes` are ignored. Scratch comes from one
 * array of MTP_NOALLOC_SCRATCH_BYTES (8 MiB) in device memory owned by the
 * library: every GPU that loads the library holds it until the process exits.
 * A batch whose scratch would not fit (mtp_lmhead_workspace_size() larger
 * than the array, e.g. sampling requests with a large M * V) is rejected with
 * MTP_INVALID_ARG and a message. Nothing here allocates: no cudaMalloc,
 * cudaFree or allocating library routine.
 * The first call on a device looks up the array's device address, with that
 * device current; it does so again on the first call after the device's
 * context was replaced (cudaDeviceReset), since the array then sits at a new
 * address. Make that first call before any stream capture begins on the
 * device. Every call on a device shares the one
 * array and leaves its contents behind; each call writes all the scratch it
 * reads before reading it, so nothing needs clearing in between. Calls whose
 * kernels overlap on the GPU (e.g. on two streams) race on the array: issue
 * them in order on one stream. */
#define MTP_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int mtp_verify_logits_accept_noalloc(const mtp_lmhead_args* args, void* stream);
size_t mtp_noalloc_scratch_bytes(void);

/* 2c. Greedy draft step of MTP Eagle: the LM head with a top-1 pick.
 *
 * Defined by: "MTP principles" §一 (the MTP modules share the target's
 * embedding and LM head and predict the D draft tokens one after another);
 * "MTP in TensorRT-LLM on Blackwell", MTP Eagle (one MTP module is run D times,
 * each run taking the draft token the previous run predicted). A draft step
 * gives each of the B requests one token: the argmax of its logits
 * l[b,v] = sum_k hidden[b,k] W[v,k] (lowest id on equal logits) over the
 * shared LM head W. D draft tokens are D calls, each on the hidden states the
 * MTP module produced for the previous token (the module itself is not part
 * of this library).
 *
 * Layouts: hidden [B, H] dtype, lm_head [V, H] dtype; out_tokens [B] int32;
 * lse_out [B] float (optional, log-sum-exp of the row, so that a caller can
 * form the draft probability exp(l[b, d] - lse)). Same dtype and H rules,
 * workspace rules (mtp_draft_workspace_size()), timing events (around the
 * LM-head kernel) and errors as mtp_verify_logits_accept. B = 0 is a no-op. */
typedef struct {
  const void* hidden;
  const void* lm_head;
  int32_t* out_tokens;
  float* lse_out;
  int32_t B, H, V;
  int32_t dtype;             /* mtp_dtype */
  void* workspace;           /* device, >= mtp_draft_workspace_size() bytes, 256-byte aligned */
  size_t workspace_bytes;
  void* timing_events[2];
} mtp_draft_args;

size_t mtp_draft_workspace_size(const mtp_draft_args* args);
int mtp_draft_argmax(const mtp_draft_args* args, void* stream);

/* ------------------------------------------------------------------------ */
/* 2d. KV compaction after a tree verify.
 *
 * Defined by: "MTP in TensorRT-LLM on Blackwell", future work: tree
 * speculative sampling, read with the rollback of the MTP Vanilla / Eagle
 * sections (the K/V of every draft that was not accepted is removed). The
 * verify call appended node k's K/V at slot ctx+k; the kept sequence is the
 * input token and the accepted path, so for i = 1 .. num_accepted[b] the K/V
 * of slot ctx + accepted_nodes[b][i] moves to slot ctx+i (in increasing i,
 * which never overwrites a slot a later move still reads: path nodes
 * increase). kv_rollback then trims the sequence to ctx + n + 1 and frees
 * blocks as for a chain. A chain path (accepted_nodes[b][i] = i) moves
 * nothing. Cache layouts as in mtp_verify_attention; ctx_lens is the
 * context length before the step (kv_rollback's seq_lens on entry).
 * Errors: num_accepted outside [0, D] sets MTP_ERR_ACCEPTED, a path that
 * does not start at 0 or does not increase sets MTP_ERR_TREE, a block id
 * outside [0, num_blocks) sets MTP_ERR_BLOCK_ID; that request is skipped. */
typedef struct {
  void* k_cache;
  void* v_cache;                  /* NULL for MLA */
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* accepted_nodes;  /* [B, D+1] */
  const int32_t* num_accepted;    /* [B] */
  int32_t B, D, Hkv, d_qk, d_v;
  int32_t block_size, max_blocks, num_blocks, is_mla;
  int32_t dtype;                  /* mtp_dtype */
} mtp_kv_compact_args;

int mtp_tree_kv_compact(const mtp_kv_compact_args* args, void* stream);

/* ------------------------------------------------------------------------ */
/* 3. KV-cache rollback.
 *
 * Defined by: "MTP in TensorRT-LLM", MTP Vanilla / MTP Eagle and the Fig. 4
 * workflow (after verification the keys/values of discarded drafts are
 * cleared from the KV cache, outside the engine forward); "Multi Token
 * Prediction" note, rollback mechanism (the verified prefix is kept).
 *
 * For request b: seq_lens[b] holds the context length ctx before the step on
 * entry and ctx + n + 1 on return (the input token and the n accepted drafts
 * keep their K/V). Every block index i with ceil((ctx+n+1)/64) <= i <=
 * (ctx+D)/64 is appended to free_list at position *free_count (request-major,
 * block index ascending) and block_table[b][i] is set to -1; *free_count is
 * advanced. A request is rolled back whole or not at all: when free_list
 * cannot take all of its freed blocks after those of every earlier request
 * (position + count > free_capacity), its table row and seq_lens entry are
 * left as they were (seq_lens[b] still equals ctx, so the caller can find it)
 * and MTP_ERR_FREE_LIST is raised; requests that free no block are still
 * rolled back, and *free_count ends one past the last block appended.
 *   block_table [B, max_blocks] int32 (in/out); seq_lens [B] int32 (in/out)
 *   num_accepted [B] int32; free_list [free_capacity] int32; free_count [1] int32
 */
typedef struct {
  int32_t* block_table;
  int32_t* seq_lens;
  const int32_t* num_accepted;
  int32_t* free_list;
  int32_t* free_count;
  int32_t B, D, block_size, max_blocks, free_capacity;
} mtp_rollback_args;

int kv_rollback(const mtp_rollback_args* args, void* stream);

/* ------------------------------------------------------------------------ */
/* Bounded-wait check (validation only, not on the verify path).
 *
 * The tensor-core kernels wait on shared-memory mbarriers (TMA copies, MMA
 * completion, stage hand-offs); every such wait gives up after a time limit,
 * sets MTP_ERR_TIMEOUT in the device error word, stops issuing work and
 * returns, so the context stays usable. This call runs that same wait on an
 * mbarrier nothing ever arrives on, with a limit of timeout_ns nanoseconds
 * (1 .. 1e9), so that a test can see the path work: afterwards
 * mtp_sync_status() returns MTP_DEVICE_ERROR with the timeout bit set (and
 * clears it). Asynchronous on `stream`; MTP_INVALID_ARG for a limit outside
 * the range. */
int mtp_wait_selftest(uint64_t timeout_ns, void* stream);

/* ------------------------------------------------------------------------ */
/* Random-stream check (validation only, not on the verify path).
 *
 * The generator is Philox4x32-10 of Salmon, Moraes, Dror and Shaw, "Parallel
 * Random Numbers: As Easy as 1, 2, 3" (SC'11); the pages fix no generator.
 * For i in [0, n) with v = v0 + i, writes (device arrays of n entries, any
 * may be NULL):
 *   word0[i]    = output word 0 for key (seed lo, seed hi), counter (b, j, v, tag)
 *   race_e[i]   = the race exponential -log1p(-x * 2^-32) of vocabulary index
 *                 v in row j, x = output word v % 4 of counter (b, j, v / 4, tag)
 *   accept_u[i] = the accept uniform of request b, row v (counter (b, v, 0, 1))
 * Returns MTP_INVALID_ARG if n < 0. */
int mtp_rng_debug(uint64_t seed, uint32_t b, uint32_t j, uint32_t tag, uint32_t v0, int32_t n,
                  uint32_t* word0, float* race_e, float* accept_u, void* stream);

/* ------------------------------------------------------------------------ */
/* Read-bandwidth probe (measurement aid, not on the verify path; the pages
 * have no counterpart).
 *
 * Reads `bytes` of device memory at `buf` once and XORs words of it into
 * *sink (device, 4 bytes; its final value has no meaning beyond keeping the
 * reads live). bulk = 0: 16-byte streaming loads from sm_count * ctas_per_sm
 * CTAs, every word folded in; bulk = 1: bulk copies (the copy engine the
 * verify kernels read through) of 32 KB chunks into a six-deep shared-memory
 * ring, one CTA per SM (ctas_per_sm ignored); a copy that does not complete
 * within 2 s sets MTP_ERR_TIMEOUT in the device error word. Timed with
 * events around it, it gives the read-only bandwidth that bounds the step's
 * read streams (KV cache, LM-head weights). buf and bytes must be multiples
 * of 16 bytes, ctas_per_sm in [1, 4], bulk 0 or 1; MTP_INVALID_ARG
 * otherwise. Asynchronous on `stream`; bytes = 0 is a no-op. */
int mtp_hbm_read_probe(const void* buf, size_t bytes, uint32_t* sink, int32_t ctas_per_sm, int32_t bulk,
                       void* stream);

/* ------------------------------------------------------------------------ */
/* Status and introspection. */

/* Message for the last failing call on this thread ("" if none). */
const char* mtp_last_error(void);

/* Synchronise `stream`, then read and clear the current device's error word.
 * Returns MTP_DEVICE_ERROR (message lists the bits) if any bit was set. */
int mtp_sync_status(void* stream);

/* Number of kernels the last successful call on this thread launched (for
 * launch accounting in benchmarks and tests). */
int mtp_last_launch_count(void);

/* ABI version (MTP_ABI_VERSION) and sizeof of the argument structs
 * (0 = mtp_attn_args, 1 = mtp_lmhead_args, 2 = mtp_rollback_args,
 * 3 = mtp_draft_args, 4 = mtp_kv_compact_args), for
 * bindings to check their struct layouts against. */
int mtp_abi_version(void);
size_t mtp_abi_struct_size(int which);

#ifdef __cplusplus
}
#endif

#endif /* MTP_VERIFY_H */
