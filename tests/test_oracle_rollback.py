"""Pins for the oracle's KV rollback.

  * brute force: a set-based restatement of the block bookkeeping (a block is
    kept iff it holds a kept slot) on random cases;
  * invariants: kept length = ctx + n + 1; table entries plus freed blocks are
    the original blocks, no duplicates; freed order is request-major;
  * the worked examples keep ctx + 4 (four tokens accepted, bonus included)
    and ctx + 3 slots.
"""
import numpy as np
import pytest

from conftest import read_golden

BLOCK = 64


def _tables(rng, B, D, ctx, max_extra=2):
    need = [(c + D + 1 + BLOCK - 1) // BLOCK for c in ctx]
    max_blocks = max(need) + max_extra
    nb = sum(need) + 5
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((B, max_blocks), -1, np.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return table


def _reference(table, ctx, n, D):
    """Set-based: block index i of request b survives iff it holds some slot < ctx+n+1."""
    table = table.copy()
    freed = []
    for b in range(len(ctx)):
        kept = ctx[b] + n[b] + 1
        used = {(s // BLOCK) for s in range(ctx[b] + D + 1)}
        for i in sorted(used):
            holds_kept = any(s // BLOCK == i for s in range(kept))
            if not holds_kept:
                freed.append(int(table[b, i]))
                table[b, i] = -1
    return table, [c + k + 1 for c, k in zip(ctx, n)], freed


@pytest.mark.parametrize("seed", range(6))
def test_rollback_matches_set_based_bookkeeping(orc, seed):
    rng = np.random.default_rng(seed)
    B, D = 12, int(rng.integers(1, 9))
    ctx = [int(x) for x in rng.integers(0, 300, B)]
    ctx[0] = 63 - D // 2          # verify slots straddle a block boundary
    ctx[1] = 64 - D - 1           # last verify slot ends a block exactly
    n = [int(x) for x in rng.integers(0, D + 1, B)]
    table = _tables(rng, B, D, ctx)
    ref_table, ref_len, ref_freed = _reference(table, ctx, n, D)
    t = table.copy()
    seq = np.array(ctx, np.int32)
    free_list = np.full(1000, -9, np.int32)
    free_count = np.array([3], np.int32)
    orc.kv_rollback(t, seq, np.array(n, np.int32), free_list, free_count, D=D, block_size=BLOCK)
    assert seq.tolist() == ref_len
    np.testing.assert_array_equal(t, ref_table)
    assert free_count[0] == 3 + len(ref_freed)
    assert free_list[3:3 + len(ref_freed)].tolist() == ref_freed
    assert (free_list[:3] == -9).all() and (free_list[3 + len(ref_freed):] == -9).all()
    # Conservation: kept entries + freed = original entries, no duplicates.
    before = sorted(table[table >= 0].tolist())
    after = sorted(t[t >= 0].tolist() + ref_freed)
    assert before == after and len(set(after)) == len(after)


@pytest.mark.parametrize("fixture,D", [("trt_fig1_greedy.txt", 5), ("vllm_example_greedy.txt", 3)])
def test_worked_examples_kept_length(orc, fixture, D):
    g = read_golden(fixture)
    n = int(g["num_accepted"][0])
    kept = int(g["kv_kept_after_ctx"][0])
    for ctx in (0, 61, 64, 1000):
        table = _tables(np.random.default_rng(ctx), 1, D, [ctx])
        seq = np.array([ctx], np.int32)
        fl = np.zeros(8, np.int32)
        fc = np.zeros(1, np.int32)
        orc.kv_rollback(table, seq, np.array([n], np.int32), fl, fc, D=D, block_size=BLOCK)
        assert seq[0] == ctx + kept
