/* Oracle: verify attention with KV append (test infrastructure only; see
 * oracle.h).
 *
 * Definition followed ("Multi Token Prediction" note, overall flow for K=3
 * draft tokens, step 2 and its table; "MTP in TensorRT-LLM", attention for
 * MTP): the verify tokens are fed together; each one's K/V goes into the
 * cache after the reused prompt KV; the row of verify token j attends every
 * cached key plus the verify keys 0..j (a causal mask inside the chain),
 * with Attention(Q) = softmax(Q K^T * scale) V, scale = 1/sqrt(d_k) by
 * default (passed in as sm_scale). Grouped-query heads share KV head
 * h / (Hq/Hkv). In the absorbed MLA form one latent of width d_qk is both
 * key and (its first d_v entries) value.
 *
 * Tree drafts ("MTP in TensorRT-LLM on Blackwell", future work: tree
 * speculative sampling, Fig. 9): verify token j is node j of a tree whose
 * node 0 is the input token and whose node k >= 1 hangs under parents[k] < k.
 * Node j's row attends every cached key plus the verify keys of the nodes on
 * the path from the root to j (itself included): the tokens its draft
 * continues. The chain is the tree with parents[k] = k - 1.
 *
 * Scores, softmax and the weighted sum are evaluated in double; the result is
 * rounded once to the output dtype (and, on request, also returned unrounded,
 * so a caller can measure another implementation's error against the exact
 * value rather than against a second rounding of it).
 */
#include <math.h>
#include <stdlib.h>
#include <vector>
#include "oracle.h"
#include "oracle_internal.h"

extern "C" int oracle_verify_attention(int B, int D, int Hq, int Hkv, int d_qk, int d_v,
                                       int block_size, int max_blocks, int num_blocks,
                                       int is_mla, float sm_scale, int dtype,
                                       const void* q, const void* k_new, const void* v_new,
                                       void* k_cache, void* v_cache,
                                       const int32_t* block_table, const int32_t* ctx_lens,
                                       void* out, const int32_t* parents, double* out_exact) {
  if (B < 0 || D < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d_qk <= 0 || d_v <= 0 ||
      block_size <= 0 || max_blocks <= 0 || num_blocks <= 0 || (dtype != 0 && dtype != 1))
    return ORACLE_BAD_ARG;
  if (is_mla && (Hkv != 1 || d_v > d_qk)) return ORACLE_BAD_ARG;
  const int R = D + 1;
  const int group = Hq / Hkv;

  /* Address of element e of key (or value) slot `slot` of request b, head kvh. */
  auto cache_index = [&](int b, int slot, int kvh, int width, int e, int64_t* idx) -> bool {
    int page = slot / block_size;
    if (page >= max_blocks) return false;
    int32_t blk = block_table[(int64_t)b * max_blocks + page];
    if (blk < 0 || blk >= num_blocks) return false;
    int off = slot % block_size;
    *idx = (((int64_t)blk * block_size + off) * Hkv + kvh) * width + e;
    return true;
  };

  for (int b = 0; b < B; ++b) {
    const int ctx = ctx_lens[b];
    if (ctx < 0) return ORACLE_BAD_ARG;
    /* parent of node k (-1 for the root); a tree must list parents before children */
    std::vector<int> parent(R);
    for (int k = 0; k < R; ++k) {
      parent[k] = parents ? parents[(int64_t)b * R + k] : k - 1;
      if (k == 0 ? parent[k] != -1 : (parent[k] < 0 || parent[k] >= k)) return ORACLE_BAD_ARG;
    }

    /* 1. Append: K/V of verify token j lands in slot ctx + j. */
    for (int j = 0; j < R; ++j) {
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        for (int e = 0; e < d_qk; ++e) {
          int64_t dst;
          if (!cache_index(b, ctx + j, kvh, d_qk, e, &dst)) return ORACLE_BAD_INDEX;
          int64_t src = (((int64_t)b * R + j) * Hkv + kvh) * d_qk + e;
          oracle_copy_elem(k_cache, dst, k_new, src, dtype);
        }
        if (!is_mla) {
          for (int e = 0; e < d_v; ++e) {
            int64_t dst;
            if (!cache_index(b, ctx + j, kvh, d_v, e, &dst)) return ORACLE_BAD_INDEX;
            int64_t src = (((int64_t)b * R + j) * Hkv + kvh) * d_v + e;
            oracle_copy_elem(v_cache, dst, v_new, src, dtype);
          }
        }
      }
    }

    /* 2. Attention: row j sees keys 0 .. ctx-1 and ctx + k for every node k
     * on the path from the root to node j. */
    for (int j = 0; j < R; ++j) {
      std::vector<char> on_path(R, 0);
      for (int k = j; k >= 0; k = parent[k]) on_path[k] = 1;
      std::vector<int> keys;
      for (int t = 0; t < ctx; ++t) keys.push_back(t);
      for (int k = 0; k < R; ++k)
        if (on_path[k]) keys.push_back(ctx + k);
      const int L = (int)keys.size();
      for (int h = 0; h < Hq; ++h) {
        const int kvh = h / group;
        const int64_t qbase = (((int64_t)b * R + j) * Hq + h) * d_qk;
        std::vector<double> score(L);
        for (int i = 0; i < L; ++i) {
          const int t = keys[i];
          int64_t k0;
          if (!cache_index(b, t, kvh, d_qk, 0, &k0)) return ORACLE_BAD_INDEX;
          double dot = 0.0;
          for (int e = 0; e < d_qk; ++e)
            dot += oracle_load(q, dtype, qbase + e) * oracle_load(k_cache, dtype, k0 + e);
          score[i] = dot * (double)sm_scale;
        }
        double mx = -INFINITY;
        for (int i = 0; i < L; ++i) mx = score[i] > mx ? score[i] : mx;
        double z = 0.0;
        for (int i = 0; i < L; ++i) {
          score[i] = exp(score[i] - mx);
          z += score[i];
        }
        const int64_t obase = (((int64_t)b * R + j) * Hq + h) * d_v;
        std::vector<double> acc(d_v, 0.0);
        for (int i = 0; i < L; ++i) {
          const int t = keys[i];
          int64_t v0;
          bool ok = is_mla ? cache_index(b, t, 0, d_qk, 0, &v0)
                           : cache_index(b, t, kvh, d_v, 0, &v0);
          if (!ok) return ORACLE_BAD_INDEX;
          const void* vsrc = is_mla ? (const void*)k_cache : (const void*)v_cache;
          for (int e = 0; e < d_v; ++e) acc[e] += score[i] * oracle_load(vsrc, dtype, v0 + e);
        }
        for (int e = 0; e < d_v; ++e) {
          oracle_store(out, dtype, obase + e, acc[e] / z);
          if (out_exact) out_exact[obase + e] = acc[e] / z;
        }
      }
    }
  }
  return ORACLE_OK;
}
