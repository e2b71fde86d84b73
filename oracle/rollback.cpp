/* Oracle: KV-cache rollback after verification (test infrastructure only;
 * see oracle.h).
 *
 * "MTP in TensorRT-LLM" (MTP Vanilla / MTP Eagle, and the TensorRT-LLM
 * workflow of Fig. 4): after verification the K/V of the drafts that were not
 * accepted must be removed from the cache. "Multi Token Prediction" note
 * (rollback mechanism): the verified-correct prefix is kept as is.
 *
 * The verify step wrote K/V for the input token and the D drafts into slots
 * ctx .. ctx+D. The input token and the n accepted drafts stay, so the
 * sequence keeps ctx + n + 1 slots; the emitted correction/bonus token has no
 * K/V yet (it is the next step's input). A block that held one of the verify
 * slots and no longer holds any kept slot goes back to the free list.
 */
#include "oracle.h"
#include "oracle_internal.h"

extern "C" int oracle_kv_rollback(int B, int D, int block_size, int max_blocks,
                                  int32_t* block_table, int32_t* seq_lens,
                                  const int32_t* num_accepted,
                                  int32_t* free_list, int32_t* free_count) {
  if (B < 0 || D < 0 || block_size <= 0 || max_blocks <= 0) return ORACLE_BAD_ARG;
  for (int b = 0; b < B; ++b) {
    const int ctx = seq_lens[b];
    const int n = num_accepted[b];
    if (ctx < 0 || n < 0 || n > D) return ORACLE_BAD_ARG;
    const int kept = ctx + n + 1;
    const int first_kept_free = (kept + block_size - 1) / block_size; /* blocks [0, this) stay */
    const int last_written = (ctx + D) / block_size;                  /* block of slot ctx+D */
    if (last_written >= max_blocks) return ORACLE_BAD_INDEX;
    for (int blk = first_kept_free; blk <= last_written; ++blk) {
      int32_t* entry = &block_table[(int64_t)b * max_blocks + blk];
      free_list[(*free_count)++] = *entry;
      *entry = -1;
    }
    seq_lens[b] = kept;
  }
  return ORACLE_OK;
}

/* Tree drafts ("MTP in TensorRT-LLM on Blackwell", future work: tree
 * speculative sampling): the verify step wrote node k's K/V into slot ctx + k.
 * The kept sequence is the input token plus the accepted path, so the K/V of
 * the path's i-th node (accepted_nodes[b][i], i = 1..n) must end in slot
 * ctx + i before the rollback above trims the sequence to ctx + n + 1. Path
 * nodes have increasing indices, so copying in increasing i never overwrites
 * a slot that a later copy still reads. */
extern "C" int oracle_tree_kv_compact(int B, int D, int Hkv, int d_qk, int d_v, int block_size, int max_blocks,
                                      int num_blocks, int is_mla, int dtype, void* k_cache, void* v_cache,
                                      const int32_t* block_table, const int32_t* ctx_lens,
                                      const int32_t* accepted_nodes, const int32_t* num_accepted) {
  if (B < 0 || D < 0 || Hkv <= 0 || d_qk <= 0 || d_v <= 0 || block_size <= 0 || max_blocks <= 0 ||
      num_blocks <= 0 || (dtype != 0 && dtype != 1))
    return ORACLE_BAD_ARG;
  const int R = D + 1;
  auto slot_index = [&](int b, int slot, int kvh, int width, int64_t* idx) -> bool {
    const int page = slot / block_size;
    if (page >= max_blocks) return false;
    const int32_t blk = block_table[(int64_t)b * max_blocks + page];
    if (blk < 0 || blk >= num_blocks) return false;
    *idx = (((int64_t)blk * block_size + slot % block_size) * Hkv + kvh) * width;
    return true;
  };
  for (int b = 0; b < B; ++b) {
    const int ctx = ctx_lens[b];
    const int n = num_accepted[b];
    if (ctx < 0 || n < 0 || n > D) return ORACLE_BAD_ARG;
    const int32_t* path = &accepted_nodes[(int64_t)b * R];
    if (path[0] != 0) return ORACLE_BAD_ARG;
    for (int i = 1; i <= n; ++i) {
      const int src = path[i];
      if (src <= path[i - 1] || src >= R) return ORACLE_BAD_ARG;
      if (src == i) continue;
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        int64_t from, to;
        if (!slot_index(b, ctx + src, kvh, d_qk, &from) || !slot_index(b, ctx + i, kvh, d_qk, &to))
          return ORACLE_BAD_INDEX;
        for (int e = 0; e < d_qk; ++e) oracle_copy_elem(k_cache, to + e, k_cache, from + e, dtype);
        if (!is_mla) {
          if (!slot_index(b, ctx + src, kvh, d_v, &from) || !slot_index(b, ctx + i, kvh, d_v, &to))
            return ORACLE_BAD_INDEX;
          for (int e = 0; e < d_v; ++e) oracle_copy_elem(v_cache, to + e, v_cache, from + e, dtype);
        }
      }
    }
  }
  return ORACLE_OK;
}
