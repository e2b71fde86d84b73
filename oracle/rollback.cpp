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
