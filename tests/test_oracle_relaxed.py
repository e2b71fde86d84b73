"""Pins of the oracle's relaxed acceptance ("MTP in TensorRT-LLM on Blackwell",
MTP optimization: relaxed acceptance; Fig. 6 is an image lost in the page
text, so the worked example below is built by hand from the rule as stated):
the candidates of a row are its top-N tokens by logit, minus those whose
probability is below the top-1 probability minus delta; a draft is accepted
iff it is a candidate; the first miss is replaced by the row's top-1 token."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _lse(x):
    x = np.asarray(x, np.float64)
    m = x.max()
    return float(m + np.log(np.exp(x - m).sum()))


def test_top1_delta0_is_strict_greedy_rowwise():
    rng = np.random.default_rng(1)
    for _ in range(200):
        V = int(rng.integers(2, 40))
        lg = rng.normal(0, 3, V).astype(np.float32)
        lse = np.float32(_lse(lg))
        for d in range(V):
            acc, tie = oracle.relaxed_accept(lg, lse, d, 1, 0.0)
            if tie:
                continue
            assert acc == int(d == int(np.argmax(lg)))


def test_brute_force_sort_definition():
    """Rank by a stable sort on (-logit, index) instead of counting; the
    probability condition in float64 away from its threshold."""
    rng = np.random.default_rng(2)
    checked = 0
    for _ in range(300):
        V = int(rng.integers(3, 60))
        lg = (rng.normal(0, 1.5, V) * rng.choice([1.0, 4.0])).astype(np.float32)
        if rng.random() < 0.2:   # exact ties in the logits
            lg[rng.integers(0, V)] = lg[rng.integers(0, V)]
        lse = np.float32(_lse(lg))
        order = sorted(range(V), key=lambda v: (-float(lg[v]), v))
        p = np.exp(lg.astype(np.float64) - _lse(lg))
        for _k in range(4):
            d = int(rng.integers(0, V))
            N = int(rng.integers(1, V + 1))
            delta = float(rng.choice([0.0, 0.05, 0.3, 0.6, 1.0]))
            acc, tie = oracle.relaxed_accept(lg, lse, d, N, delta)
            margin = abs(p[d] - (p.max() - delta))
            if tie or margin < 1e-3:
                continue
            want = int(d in order[:N] and p[d] >= p.max() - delta)
            assert acc == want, (V, d, N, delta)
            checked += 1
    assert checked > 800


def test_monotone_in_topk_and_delta():
    rng = np.random.default_rng(3)
    for _ in range(100):
        V = 30
        lg = rng.normal(0, 2, V).astype(np.float32)
        lse = np.float32(_lse(lg))
        d = int(rng.integers(0, V))
        prev = 0
        for N in range(1, V + 1):
            a, _ = oracle.relaxed_accept(lg, lse, d, N, 0.5)
            assert a >= prev
            prev = a
        prev = 0
        for delta in (0.0, 0.01, 0.1, 0.3, 0.6, 0.9, 1.0):
            a, _ = oracle.relaxed_accept(lg, lse, d, 3, delta)
            assert a >= prev
            prev = a


def test_delta_threshold_closed_form():
    """Two tokens hold almost all the mass: p1 = e^a/(e^a+e^b+rest), p2 likewise;
    the runner-up is accepted iff p2 >= p1 - delta."""
    V = 1000
    lg = np.zeros(V, np.float32)
    lg[7], lg[9] = 12.0, 11.0          # p1 ~ 0.727, p2 ~ 0.267 (rest ~ 0.006)
    lse = np.float32(_lse(lg))
    p = np.exp(lg.astype(np.float64) - _lse(lg))
    gap = p[7] - p[9]
    for delta, want in ((gap - 0.01, 0), (gap + 0.01, 1), (0.0, 0), (1.0, 1)):
        acc, tie = oracle.relaxed_accept(lg, lse, 9, 2, delta)
        assert tie == 0 and acc == want, delta
    acc, _ = oracle.relaxed_accept(lg, lse, 9, 1, 1.0)    # rank 1 is outside the top-1
    assert acc == 0
    acc, _ = oracle.relaxed_accept(lg, lse, 7, 1, 0.0)    # the top-1 itself
    assert acc == 1


def _one_hot_lm(rows_logits):
    """hidden = the logits themselves, lm_head = identity: the oracle's logits are
    exactly the given rows (fp32 inputs)."""
    R, V = rows_logits.shape
    return rows_logits.astype(np.float32), np.eye(V, dtype=np.float32)


def test_hand_worked_top3_example():
    """Four drafts against five rows (D = 4). Row j's logits put the draft at
    rank 0, 2, 1, 5; all probabilities are small (flat tail), so with delta 0.6
    only the rank matters: top-3 relaxed acceptance takes drafts 1..3, rejects
    draft 4 and emits row 3's top-1; strict acceptance stops at draft 2."""
    V = 64
    D = 4
    rng = np.random.default_rng(4)
    rows = rng.normal(0, 0.05, (D + 1, V)).astype(np.float32)
    order = [[10, 11, 12, 13, 14, 15], [20, 21, 22, 23, 24, 25], [30, 31, 32, 33, 34, 35],
             [40, 41, 42, 43, 44, 45], [50, 51, 52, 53, 54, 55]]
    for j in range(D + 1):
        for r, v in enumerate(order[j]):
            rows[j, v] = 3.0 - 0.3 * r      # ranks 0..5 at those tokens
    drafts = [order[0][0], order[1][2], order[2][1], order[3][5]]
    tokens = np.array([[5] + drafts], np.int32)
    hidden, W = _one_hot_lm(rows)
    mode = np.array([2], np.uint8)
    res = oracle.lmhead_accept(hidden, W, tokens, mode, None, None, 0, relaxed_topk=3, relaxed_delta=0.6)
    assert res["num_accepted"][0] == 3 and res["tie_flags"][0] == 0
    assert list(res["out_tokens"][0]) == drafts[:3] + [order[3][0], -1]
    strict = oracle.lmhead_accept(hidden, W, tokens, np.array([0], np.uint8), None, None, 0)
    assert strict["num_accepted"][0] == 1
    assert list(strict["out_tokens"][0]) == [drafts[0], order[1][0], -1, -1, -1]
    every = oracle.lmhead_accept(hidden, W, tokens, mode, None, None, 0, relaxed_topk=V, relaxed_delta=1.0)
    assert every["num_accepted"][0] == D and every["out_tokens"][0][D] == order[4][0]


def test_mode2_with_top1_delta0_equals_greedy_end_to_end():
    rng = np.random.default_rng(5)
    B, D, V, H = 6, 3, 97, 16
    W = rng.normal(0, 1, (V, H)).astype(np.float32)
    hidden = rng.normal(0, 1, (B * (D + 1), H)).astype(np.float32)
    tokens = rng.integers(0, V, (B, D + 1)).astype(np.int32)
    # make some drafts the greedy choice so that prefixes of several lengths occur
    logits = hidden @ W.T
    for b in range(B):
        for j in range(D):
            if rng.random() < 0.7:
                tokens[b, j + 1] = int(np.argmax(logits[b * (D + 1) + j]))
    g = oracle.lmhead_accept(hidden, W, tokens, np.zeros(B, np.uint8), None, None, 0)
    r = oracle.lmhead_accept(hidden, W, tokens, np.full(B, 2, np.uint8), None, None, 0, relaxed_topk=1,
                             relaxed_delta=0.0)
    ok = r["tie_flags"] == 0
    assert ok.sum() >= B - 1
    assert (g["num_accepted"][ok] == r["num_accepted"][ok]).all()
    assert (g["out_tokens"][ok] == r["out_tokens"][ok]).all()
    assert len(set(g["num_accepted"].tolist())) > 1


def test_relaxed_needs_topk():
    with pytest.raises(ValueError):
        oracle.lmhead_accept(np.ones((2, 4), np.float32), np.eye(4, dtype=np.float32), np.zeros((1, 2), np.int32),
                             np.array([2], np.uint8), None, None, 0, relaxed_topk=0)


def test_equal_logits_rank_lower_token_id_first():
    """Logits [3, 2, 2, 1] with N = 2 and a delta that admits every token:
    token 1 (lower id of the tied pair) is the second candidate, token 2 is
    third and so outside the top 2. The tie sits on the boundary, so the
    decision is flagged as a near-tie, but the rule itself is fixed."""
    lg = np.array([3.0, 2.0, 2.0, 1.0], np.float32)
    lse = np.float32(_lse(lg))
    acc1, tie1 = oracle.relaxed_accept(lg, lse, 1, 2, 1.0)
    acc2, tie2 = oracle.relaxed_accept(lg, lse, 2, 2, 1.0)
    assert acc1 == 1 and acc2 == 0
    assert tie1 & 1 and tie2 & 1
    # With N = 3 both tied tokens are candidates.
    assert oracle.relaxed_accept(lg, lse, 2, 3, 1.0)[0] == 1
