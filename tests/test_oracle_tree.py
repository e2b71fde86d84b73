"""Pins for the oracle's tree drafts ("MTP in TensorRT-LLM on Blackwell",
future work: tree speculative sampling, Fig. 9): attention under the tree
mask, greedy tree acceptance and the KV compaction of the accepted path.

  * the chain written as a tree (parents k - 1) gives bit-identical results;
  * brute force: each tree row equals textbook attention over the context and
    the verify keys of its root path, gathered densely; and equals the last
    row of a chain request made of that path's tokens;
  * acceptance: a hand-worked tree, a star, duplicate siblings, and random
    trees against an independent depth-first enumeration of root paths;
  * compaction: slots ctx+1..ctx+n hold the path's K/V afterwards (including
    overlapping moves), every other slot is untouched.
"""
import numpy as np
import pytest

from test_oracle_attention import BLOCK, _case, _dense_sequence, _run, _textbook


def _random_parents(rng, R):
    return np.array([-1] + [int(rng.integers(0, k)) for k in range(1, R)], np.int32)


def _root_path(parents, j):
    path = [j]
    while parents[path[-1]] >= 0:
        path.append(int(parents[path[-1]]))
    return path[::-1]


def _run_tree(orc, c, D, Hq, Hkv, d_qk, d_v, parents, is_mla=False):
    kc = c["k_cache"].copy()
    vc = None if c["v_cache"] is None else c["v_cache"].copy()
    out = orc.verify_attention(c["q"], c["k_new"], c["v_new"], kc, vc, c["block_table"], c["ctx_lens"], D=D,
                               Hq=Hq, Hkv=1 if is_mla else Hkv, d_qk=d_qk, d_v=d_v, block_size=BLOCK,
                               is_mla=is_mla, sm_scale=1 / np.sqrt(d_qk), parents=parents)
    return out, kc, vc


# ------------------------------------------------------------------ attention

@pytest.mark.parametrize("is_mla", [False, True])
def test_chain_as_tree_is_bit_identical(orc, is_mla):
    rng = np.random.default_rng(11)
    B, D, Hq, Hkv = 2, 4, 4, (1 if is_mla else 2)
    d_qk, d_v = (40, 32) if is_mla else (16, 16)
    c = _case(rng, B, D, Hq, Hkv, d_qk, d_v, [70, 3], is_mla=is_mla)
    chain = np.tile(np.arange(-1, D, dtype=np.int32), (B, 1))
    a, ka, va = _run(orc, c, D, Hq, Hkv, d_qk, d_v, is_mla=is_mla)
    t, kt, vt = _run_tree(orc, c, D, Hq, Hkv, d_qk, d_v, chain, is_mla=is_mla)
    assert np.array_equal(a, t) and np.array_equal(ka, kt)


@pytest.mark.parametrize("is_mla", [False, True])
def test_tree_rows_are_textbook_attention_over_the_root_path(orc, is_mla):
    rng = np.random.default_rng(12)
    B, D, Hq, Hkv = 3, 9, 4, (1 if is_mla else 2)
    d_qk, d_v = (40, 32) if is_mla else (16, 16)
    c = _case(rng, B, D, Hq, Hkv, d_qk, d_v, [0, 61, 130], is_mla=is_mla)
    parents = np.stack([_random_parents(rng, D + 1) for _ in range(B)])
    out, _, _ = _run_tree(orc, c, D, Hq, Hkv, d_qk, d_v, parents, is_mla=is_mla)
    group = Hq // Hkv
    for b in range(B):
        ctx = int(c["ctx_lens"][b])
        for kvh in range(Hkv):
            K, V = _dense_sequence(c, b, kvh, D, is_mla, d_v)
            for j in range(D + 1):
                keep = list(range(ctx)) + [ctx + k for k in _root_path(parents[b], j)]
                for h in range(kvh * group, (kvh + 1) * group):
                    want = _textbook(c["q"][b, j, h], K[keep], V[keep], 1 / np.sqrt(d_qk))
                    np.testing.assert_allclose(out[b, j, h], want, rtol=1e-5, atol=1e-6)


def test_tree_row_equals_chain_of_its_path(orc):
    rng = np.random.default_rng(13)
    D, Hq, Hkv, d = 7, 4, 2, 16
    c = _case(rng, 1, D, Hq, Hkv, d, d, [90])
    parents = np.array([[-1, 0, 0, 1, 2, 2, 4, 6]], np.int32)
    out, _, _ = _run_tree(orc, c, D, Hq, Hkv, d, d, parents)
    for j in range(D + 1):
        path = _root_path(parents[0], j)
        Dp = len(path) - 1
        cc = dict(c, q=c["q"][:, path], k_new=c["k_new"][:, path], v_new=c["v_new"][:, path])
        chain_out, _, _ = _run(orc, cc, Dp, Hq, Hkv, d, d)
        np.testing.assert_allclose(out[0, j], chain_out[0, Dp], rtol=1e-6, atol=1e-7)


def test_bad_parents_rejected(orc):
    rng = np.random.default_rng(14)
    c = _case(rng, 1, 3, 2, 2, 16, 16, [10])
    for bad in ([0, 0, 1, 2], [-1, 1, 1, 2], [-1, 0, 3, 1], [-1, -1, 0, 1]):
        with pytest.raises(ValueError):
            _run_tree(orc, c, 3, 2, 2, 16, 16, np.array([bad], np.int32))


# ----------------------------------------------------------------- acceptance

def _onehot_lm(targets, V):
    """hidden rows one-hot at each row's target and W = identity: row j's
    logits are one-hot at targets[j], so its argmax is targets[j]."""
    M = len(targets)
    hidden = np.zeros((M, V), np.float32)
    hidden[np.arange(M), targets] = 1.0
    return hidden, np.eye(V, dtype=np.float32)


def _accept(orc, tokens, targets, parents, V):
    B, R = tokens.shape
    hidden, W = _onehot_lm(np.asarray(targets).reshape(-1), V)
    return orc.lmhead_accept(hidden, W, tokens, np.zeros(B, np.uint8), None, None, 0,
                             parents=None if parents is None else np.asarray(parents, np.int32).reshape(B, R))


def test_hand_worked_tree(orc):
    # Nodes 0..6 with parents [-, 0, 0, 1, 1, 2, 5] and tokens [9, 3, 4, 5, 6, 7, 8].
    # Row targets: 0->4 (node 2 matches, node 1 does not), 1->5, 2->7 (node 5),
    # 3->0, 4->0, 5->8 (node 6), 6->2. Accepted path 0-2-5-6: drafts 4 7 8, then 2.
    tokens = np.array([[9, 3, 4, 5, 6, 7, 8]], np.int32)
    targets = [4, 5, 7, 0, 0, 8, 2]
    r = _accept(orc, tokens, targets, [-1, 0, 0, 1, 1, 2, 5], 10)
    assert r["num_accepted"][0] == 3
    assert list(r["out_tokens"][0]) == [4, 7, 8, 2, -1, -1, -1]
    assert list(r["accepted_nodes"][0]) == [0, 2, 5, 6, -1, -1, -1]


def test_star_tree_accepts_at_most_one(orc):
    rng = np.random.default_rng(15)
    V, R = 12, 6
    for _ in range(50):
        tokens = rng.integers(0, V, (1, R)).astype(np.int32)
        targets = rng.integers(0, V, R)
        r = _accept(orc, tokens, targets, [-1] + [0] * (R - 1), V)
        hits = [k for k in range(1, R) if tokens[0, k] == targets[0]]
        n = int(r["num_accepted"][0])
        assert n == (1 if hits else 0)
        end = hits[0] if hits else 0
        assert r["out_tokens"][0, n] == targets[end]
        assert list(r["accepted_nodes"][0, :n + 1]) == ([0, hits[0]] if hits else [0])


def test_deeper_path_through_a_duplicate_sibling_wins(orc):
    # Nodes 1 and 2 both carry row 0's argmax (7); only node 2 has a matching child (node 3).
    tokens = np.array([[0, 7, 7, 5]], np.int32)
    targets = [7, 1, 5, 4]
    r = _accept(orc, tokens, targets, [-1, 0, 0, 2], 9)
    assert r["num_accepted"][0] == 2
    assert list(r["accepted_nodes"][0]) == [0, 2, 3, -1]
    assert list(r["out_tokens"][0]) == [7, 5, 4, -1]


def _dfs_best(parents, tokens, targets):
    """Independent enumeration: depth-first from the root over child lists,
    extending a path only while each child's token is its parent's target."""
    R = len(parents)
    children = [[] for _ in range(R)]
    for k in range(1, R):
        children[parents[k]].append(k)
    best = [0]

    def visit(path):
        nonlocal best
        u = path[-1]
        if len(path) > len(best) or (len(path) == len(best) and u < best[-1]):
            best = list(path)
        for c in children[u]:
            if tokens[c] == targets[u]:
                visit(path + [c])
    visit([0])
    return best


def test_random_trees_against_depth_first_enumeration(orc):
    rng = np.random.default_rng(16)
    V = 6
    for trial in range(300):
        R = int(rng.integers(1, 17))
        parents = _random_parents(rng, R)
        targets = rng.integers(0, V, R)
        tokens = rng.integers(0, V, R).astype(np.int32)
        for k in range(1, R):          # make about half of the edges match
            if rng.random() < 0.5:
                tokens[k] = targets[parents[k]]
        r = _accept(orc, tokens[None], targets, parents, V)
        best = _dfs_best(parents, tokens, targets)
        n = len(best) - 1
        assert r["num_accepted"][0] == n, trial
        assert list(r["accepted_nodes"][0, :n + 1]) == best and (r["accepted_nodes"][0, n + 1:] == -1).all()
        assert list(r["out_tokens"][0, :n]) == [int(tokens[k]) for k in best[1:]]
        assert r["out_tokens"][0, n] == targets[best[-1]]


def test_chain_as_tree_accepts_like_a_chain(orc):
    rng = np.random.default_rng(17)
    V, R, B = 5, 6, 40
    tokens = rng.integers(0, V, (B, R)).astype(np.int32)
    targets = rng.integers(0, V, (B, R))
    for b in range(B):
        for k in range(1, R):
            if rng.random() < 0.6:
                tokens[b, k] = targets[b, k - 1]
    chain = _accept(orc, tokens, targets, None, V)
    tree = _accept(orc, tokens, targets, np.tile(np.arange(-1, R - 1), (B, 1)), V)
    for k in ("out_tokens", "num_accepted", "accepted_nodes"):
        assert np.array_equal(chain[k], tree[k]), k
    for b in range(B):
        n = chain["num_accepted"][b]
        assert list(chain["accepted_nodes"][b, :n + 1]) == list(range(n + 1))


def test_tree_requests_must_be_greedy(orc):
    tokens = np.array([[1, 2, 3]], np.int32)
    hidden, W = _onehot_lm([2, 3, 0], 5)
    q = np.full((1, 2, 5), 0.2, np.float32)
    with pytest.raises(ValueError):
        orc.lmhead_accept(hidden, W, tokens, np.ones(1, np.uint8), np.ones(1, np.float32), q, 0,
                                 parents=np.array([[-1, 0, 0]], np.int32))
    with pytest.raises(ValueError):
        orc.lmhead_accept(hidden, W, tokens, np.full(1, 2, np.uint8), None, None, 0, relaxed_topk=2,
                                 relaxed_delta=0.1, parents=np.array([[-1, 0, 0]], np.int32))


# ----------------------------------------------------------------- compaction

@pytest.mark.parametrize("is_mla", [False, True])
def test_compaction_moves_the_path_and_nothing_else(orc, is_mla):
    rng = np.random.default_rng(18)
    B, D, Hkv = 3, 7, (1 if is_mla else 2)
    d_qk, d_v = (40, 32) if is_mla else (16, 16)
    c = _case(rng, B, D, 2, Hkv, d_qk, d_v, [62, 0, 100], is_mla=is_mla)
    _, kc, vc = _run(orc, c, D, 2, Hkv, d_qk, d_v, is_mla=is_mla)   # append: node k in slot ctx + k
    R = D + 1
    paths = [[0, 2, 3, 7], [0], [0, 1, 4, 5, 6]]          # overlapping moves: 2->1 then 3->2
    nodes = np.full((B, R), -1, np.int32)
    for b, p in enumerate(paths):
        nodes[b, :len(p)] = p
    n = np.array([len(p) - 1 for p in paths], np.int32)
    k0, v0 = kc.copy(), None if vc is None else vc.copy()
    orc.tree_kv_compact(kc, vc, c["block_table"], c["ctx_lens"], nodes, n, D=D, Hkv=Hkv, d_qk=d_qk,
                               d_v=d_v, block_size=BLOCK, is_mla=is_mla)
    touched = set()
    for b, p in enumerate(paths):
        ctx = int(c["ctx_lens"][b])
        for i, node in enumerate(p):
            s = ctx + i
            blk, off = c["block_table"][b, s // BLOCK], s % BLOCK
            kn = c["k_new"][b, node] if is_mla else c["k_new"][b, node]
            assert np.array_equal(kc[blk, off].reshape(-1), kn.reshape(-1))
            if not is_mla:
                assert np.array_equal(vc[blk, off], c["v_new"][b, node])
            touched.add((int(blk), off))
    for blk in range(kc.shape[0]):
        for off in range(BLOCK):
            if (blk, off) not in touched:
                assert np.array_equal(kc[blk, off], k0[blk, off])
                if vc is not None:
                    assert np.array_equal(vc[blk, off], v0[blk, off])


def test_compaction_rejects_a_path_that_is_not_increasing(orc):
    rng = np.random.default_rng(19)
    c = _case(rng, 1, 3, 2, 2, 16, 16, [5])
    _, kc, vc = _run(orc, c, 3, 2, 2, 16, 16)
    for bad in ([0, 2, 1, -1], [1, 2, 3, -1], [0, 4, -1, -1]):
        with pytest.raises(ValueError):
            orc.tree_kv_compact(kc, vc, c["block_table"], c["ctx_lens"], np.array([bad], np.int32),
                                       np.array([2 if bad[2] >= 0 else 1], np.int32), D=3, Hkv=2, d_qk=16,
                                       d_v=16, block_size=BLOCK, is_mla=False)
