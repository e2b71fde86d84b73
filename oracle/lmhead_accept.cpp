/* Oracle: LM head, row statistics and acceptance (test infrastructure only;
 * see oracle.h).
 *
 * Steps, in the pages' order:
 *  1. Logits_i = H_i x W_o for every verify row ("Multi Token Prediction"
 *     note, K=3 flow, step 4). The sum runs in double and is rounded to
 *     binary32; sampling rows are then multiplied by 1/T in binary32
 *     (p = softmax(logits / T); temperature 0 means the argmax rule,
 *     "Speculative decoding and MTP" §4.4).
 *  2. Softmax statistics per row (same note, step 5): max, log-sum-exp (in
 *     double over the binary32 logits), argmax (lowest index on ties).
 *  3. Acceptance, scanning the drafts in order and stopping at the first
 *     failure ("MTP principles" §三 stage 3; "Speculative decoding and MTP"
 *     §2.3 and §4.4; "MTP in TensorRT-LLM" Fig. 1):
 *       greedy:   accept d_{j+1} iff argmax of row j equals it; the first
 *                 mismatch is replaced by that argmax; if all D match, the
 *                 argmax of row D is the bonus token.
 *       sampling: accept d_{j+1} iff p_j(d) >= U_j * q_j(d) (same as accepting
 *                 with probability min(1, p/q)); at the first rejection draw
 *                 from normalised max(0, p_j - q_j); if all D are accepted
 *                 draw the bonus from p_D.
 *       relaxed:  ("MTP in TensorRT-LLM", MTP optimization: relaxed
 *                 acceptance) the candidates of row j are its top-N tokens
 *                 by logit, minus those whose probability is below the top-1
 *                 probability minus delta; d_{j+1} is accepted iff it is a
 *                 candidate. The first miss is replaced by the argmax and the
 *                 bonus is the argmax of row D, as for greedy requests.
 *       tree:     ("MTP in TensorRT-LLM on Blackwell", future work: tree
 *                 speculative sampling) node k >= 1 carries draft token
 *                 tokens[k] continuing the path that ends at its parent.
 *                 Node u is accepted when every node v on the path from the
 *                 root to u carries the argmax of its parent's row (greedy
 *                 rule per edge). The accepted node of greatest depth (lowest
 *                 index among equally deep ones) ends the accepted path; the
 *                 argmax of its row is the emitted correction/bonus token.
 *                 The chain is the tree with parents[k] = k - 1.
 *     Every step emits n + 1 tokens, 1 .. D+1 ("MTP principles" stage 4).
 *  4. A categorical draw is an exponential race: argmax_v w_v / E_v with
 *     E_v ~ Exp(1) from the counter-based generator (philox.cpp); this picks
 *     v with probability w_v / sum(w). If every residual weight is zero the
 *     draw falls back to p itself.
 * The accept test and the race are evaluated in binary32, the precision the
 * GPU decides in; decisions within 1e-5 of flipping are flagged.
 */
#include <math.h>
#include <stdlib.h>
#include <vector>
#include "oracle.h"
#include "oracle_internal.h"

static const float kTieRel = 1e-5f;
static const float kRelaxedTieAbs = 1e-3f;    /* |p_d - (p_1 - delta)| below this: flagged */
static const float kRelaxedRankEps = 1e-3f;   /* logit band (x (1 + |l_d|)) for an unstable rank */

extern "C" int oracle_relaxed_accept(int V, const float* logits, float lse, int d, int topk, float delta,
                                     uint8_t* tie) {
  const float ld = logits[d];
  /* Rank of d: the tokens ordered before it (larger logit, or equal logit
   * and lower index). Also count the tokens that are surely above it and
   * those that might be, within a band around l_d. */
  const float eps = kRelaxedRankEps * (1.0f + fabsf(ld));
  int before = 0, surely_above = 0, maybe_above = 0;
  int top = 0;
  for (int v = 0; v < V; ++v) {
    if (logits[v] > logits[top]) top = v;
    if (v == d) continue;
    if (logits[v] > ld || (logits[v] == ld && v < d)) ++before;
    if (logits[v] > ld + eps) ++surely_above;
    if (logits[v] >= ld - eps) ++maybe_above;
  }
  const int in_top = before < topk;
  if (surely_above < topk && maybe_above >= topk) *tie |= 1;
  const float pd = expf(ld - lse);
  const float thr = expf(logits[top] - lse) - delta;
  /* (The top-1 token itself meets the probability condition exactly.) */
  if (d != top && fabsf(pd - thr) < kRelaxedTieAbs) *tie |= 1;
  return in_top && pd >= thr;
}

extern "C" int oracle_accept_prefix(int D, const float* p, const float* q, const float* U, uint8_t* tie) {
  int n = 0;
  for (int j = 0; j < D; ++j) {
    float uq = U[j] * q[j];
    if (q[j] > 0.0f && fabsf(p[j] - uq) < kTieRel * q[j]) *tie |= 1;
    if (p[j] >= uq) {
      n = j + 1;
    } else {
      break;
    }
  }
  return n;
}

extern "C" int oracle_race(int V, const float* w, const float* E, uint8_t* near_tie) {
  int best = -1;
  float k1 = -1.0f, k2 = -1.0f;
  for (int v = 0; v < V; ++v) {
    if (!(w[v] > 0.0f)) continue;
    float key = w[v] / E[v]; /* E == 0 gives +inf: that entry wins */
    if (key > k1) {
      k2 = k1;
      k1 = key;
      best = v;
    } else if (key > k2) {
      k2 = key;
    }
  }
  if (best >= 0 && k2 >= 0.0f && (k1 == k2 || k1 - k2 <= kTieRel * k1)) *near_tie = 1;
  return best;
}

extern "C" int oracle_lmhead_accept(int B, int D, int H, int V, int dtype,
                                    const void* hidden, const void* lm_head,
                                    const int32_t* tokens, const uint8_t* mode,
                                    const float* temperature, const float* q_draft,
                                    uint64_t seed, const int32_t* request_index,
                                    int32_t* out_tokens, int32_t* num_accepted,
                                    uint8_t* tie_flags, float* lse_out,
                                    int32_t* argmax_out, float* logits_out,
                                    int relaxed_topk, float relaxed_delta,
                                    const int32_t* parents, int32_t* accepted_nodes) {
  if (B < 0 || D < 0 || H <= 0 || V <= 0 || (dtype != 0 && dtype != 1)) return ORACLE_BAD_ARG;
  if (relaxed_delta < 0.0f) return ORACLE_BAD_ARG;
  const int R = D + 1;
  std::vector<float> logits((size_t)R * V);
  std::vector<float> lse(R);
  std::vector<int> amax(R);
  std::vector<float> w(V), E(V), p(V);

  for (int b = 0; b < B; ++b) {
    for (int j = 0; j < R; ++j) {
      int tok = tokens[(int64_t)b * R + j];
      if (tok < 0 || tok >= V) return ORACLE_BAD_INDEX;
    }
    const uint32_t rid = request_index ? (uint32_t)request_index[b] : (uint32_t)b;
    const bool sampling = mode[b] == 1 && temperature != NULL && temperature[b] > 0.0f;
    const bool relaxed = mode[b] == 2;
    if (sampling && q_draft == NULL) return ORACLE_BAD_ARG;
    if (relaxed && relaxed_topk < 1) return ORACLE_BAD_ARG;
    if (parents && (sampling || relaxed)) return ORACLE_BAD_ARG;   /* trees are verified greedily */
    std::vector<int> parent(R);
    for (int k = 0; k < R; ++k) {
      parent[k] = parents ? parents[(int64_t)b * R + k] : k - 1;
      if (k == 0 ? parent[k] != -1 : (parent[k] < 0 || parent[k] >= k)) return ORACLE_BAD_ARG;
    }
    const float inv_t = sampling ? 1.0f / temperature[b] : 1.0f;

    /* Steps 1-2 for the R rows of request b. */
    for (int j = 0; j < R; ++j) {
      const int64_t m = (int64_t)b * R + j;
      float* row = &logits[(size_t)j * V];
      for (int v = 0; v < V; ++v) {
        double acc = 0.0;
        for (int k = 0; k < H; ++k)
          acc += oracle_load(hidden, dtype, m * H + k) * oracle_load(lm_head, dtype, (int64_t)v * H + k);
        float l = (float)acc;
        row[v] = sampling ? l * inv_t : l;
      }
      double mx = -INFINITY;
      int best = 0;
      for (int v = 0; v < V; ++v) {
        if ((double)row[v] > mx) {
          mx = row[v];
          best = v;
        }
      }
      double s = 0.0;
      for (int v = 0; v < V; ++v) s += exp((double)row[v] - mx);
      lse[j] = (float)(mx + log(s));
      amax[j] = best;
      if (lse_out) lse_out[m] = lse[j];
      if (argmax_out) argmax_out[m] = best;
      if (logits_out)
        for (int v = 0; v < V; ++v) logits_out[m * V + v] = row[v];
    }

    /* Step 3. */
    int32_t* out = &out_tokens[(int64_t)b * R];
    const int32_t* tok = &tokens[(int64_t)b * R];
    for (int j = 0; j < R; ++j) out[j] = -1;
    uint8_t tie = 0;
    int n;
    std::vector<int> path;   /* accepted path, root first */
    if (parents) {
      int best_u = 0, best_depth = 0;
      for (int u = 0; u < R; ++u) {
        std::vector<int> up;   /* u, parent(u), ..., root */
        for (int k = u; k >= 0; k = parent[k]) up.push_back(k);
        bool ok = true;
        for (size_t i = 0; i + 1 < up.size(); ++i) ok = ok && tok[up[i]] == amax[up[i + 1]];
        const int depth = (int)up.size() - 1;
        if (ok && depth > best_depth) {
          best_depth = depth;
          best_u = u;
        }
      }
      for (int k = best_u; k >= 0; k = parent[k]) path.insert(path.begin(), k);
      n = best_depth;
      for (int i = 1; i <= n; ++i) out[i - 1] = tok[path[i]];
      out[n] = amax[best_u];
    } else if (relaxed) {
      n = 0;
      while (n < D && oracle_relaxed_accept(V, &logits[(size_t)n * V], lse[n], tok[n + 1], relaxed_topk,
                                            relaxed_delta, &tie))
        ++n;
      for (int j = 0; j < n; ++j) out[j] = tok[j + 1];
      out[n] = amax[n];
    } else if (!sampling) {
      n = 0;
      while (n < D && amax[n] == tok[n + 1]) ++n;
      for (int j = 0; j < n; ++j) out[j] = tok[j + 1];
      out[n] = amax[n];
    } else {
      std::vector<float> pd(D), qd(D), U(D);
      for (int j = 0; j < D; ++j) {
        int x = tok[j + 1];
        pd[j] = expf(logits[(size_t)j * V + x] - lse[j]);
        qd[j] = q_draft[((int64_t)b * D + j) * V + x];
        U[j] = oracle_accept_uniform(seed, rid, (uint32_t)j);
      }
      n = oracle_accept_prefix(D, pd.data(), qd.data(), U.data(), &tie);
      for (int j = 0; j < n; ++j) out[j] = tok[j + 1];
      /* Step 4: residual draw at row n if a draft was rejected, bonus draw
       * from row D otherwise. */
      const uint32_t tag = n < D ? 2u : 3u;
      const float* row = &logits[(size_t)n * V];
      for (int v = 0; v < V; ++v) {
        p[v] = expf(row[v] - lse[n]);
        float qv = n < D ? q_draft[((int64_t)b * D + n) * V + v] : 0.0f;
        float r = p[v] - qv;
        w[v] = r > 0.0f ? r : 0.0f;
        E[v] = oracle_race_exponential(seed, rid, (uint32_t)n, (uint32_t)v, tag);
      }
      uint8_t race_tie = 0;
      int winner = oracle_race(V, w.data(), E.data(), &race_tie);
      if (winner < 0) {
        race_tie = 0;
        winner = oracle_race(V, p.data(), E.data(), &race_tie);
      }
      if (race_tie) tie |= 2;
      out[n] = winner;
    }
    num_accepted[b] = n;
    tie_flags[b] = tie;
    if (accepted_nodes) {
      if (!parents)
        for (int i = 0; i <= n; ++i) path.push_back(i);
      for (int i = 0; i < R; ++i) accepted_nodes[(int64_t)b * R + i] = i <= n ? path[i] : -1;
    }
  }
  return ORACLE_OK;
}
