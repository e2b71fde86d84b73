"""Pins for the oracle's LM head, row statistics and acceptance rules.

What pins what:
  * the worked examples of the pages (tests/golden) fix the greedy rule, the
    counting convention and the rejection rule's prefix behaviour;
  * special cases reduce to the greedy rule (one-hot target) or to "accept
    everything" (q = p);
  * statistics fix the sampling rule: the first emitted token is distributed
    as p_target (lossless), and the acceptance rate equals sum_v min(p, q);
  * logits, log-sum-exp and argmax are checked against numpy / scipy.
"""
import numpy as np
import pytest
from scipy import special, stats

from conftest import read_golden
from philox_py import accept_uniform


def _identity_head(V):
    return np.eye(V, dtype=np.float32)


def _greedy_case(orc, chain, predicted, V):
    """One greedy request whose row-j argmax is predicted[j] (logits = hidden, W = I)."""
    R = len(chain)
    hidden = np.zeros((R, V), np.float32)
    for j, t in enumerate(predicted):
        hidden[j, t] = 5.0
    tokens = np.array([chain], np.int32)
    return orc.lmhead_accept(hidden, _identity_head(V), tokens, np.zeros(1, np.uint8), None, None, 0)


def test_trt_fig1_worked_example(orc):
    g = read_golden("trt_fig1_greedy.txt")
    ids = lambda xs: [ord(c) - ord("A") for c in xs]
    res = _greedy_case(orc, ids(g["chain"]), ids(g["predicted"]), 26)
    n = int(res["num_accepted"][0])
    assert n == int(g["num_accepted"][0])
    emitted = res["out_tokens"][0, :n + 1].tolist()
    assert emitted == ids(g["emitted"])
    assert res["out_tokens"][0, n + 1:].tolist() == [-1] * (len(g["chain"]) - n - 1)


@pytest.mark.parametrize("suffix", ["", "_cx"])
def test_vllm_worked_example(orc, suffix):
    g = read_golden("vllm_example_greedy.txt")
    chain = [int(x) for x in g["chain" + suffix]]
    pred = [int(x) for x in g["predicted" + suffix]]
    res = _greedy_case(orc, chain, pred, 8)
    n = int(res["num_accepted"][0])
    assert n == int(g["num_accepted" + suffix][0])
    assert res["out_tokens"][0, :n + 1].tolist() == [int(x) for x in g["emitted" + suffix]]


def test_sdmtp_prefix_rule_fixed_uniform(orc):
    g = read_golden("sdmtp_probs.txt")
    p = np.array(g["p_target"], np.float32)
    q = np.array(g["q_draft"], np.float32)
    U = np.full(len(p), float(g["uniform"][0]), np.float32)
    n, tie = orc.accept_prefix(p, q, U)
    assert n == int(g["num_accepted"][0]) and tie == 0
    # Stops at the first failure even though later drafts would pass.
    assert orc.accept_prefix(p, q, np.array([0.5, 0.5, 0.5, 0.1, 0.1], np.float32))[0] == 2


def _logits_for_probs(p_draft, draft, V):
    """Row of logits whose softmax gives p_draft at `draft`, the rest spread evenly."""
    row = np.full(V, np.log((1 - p_draft) / (V - 1)), np.float64)
    row[draft] = np.log(p_draft)
    return row.astype(np.float32)


def test_sdmtp_example_through_full_rule(orc):
    """P(draft) = 0.9, 0.8, 0.3, 0.6, 0.7 with q one-hot on the drafts: with
    uniforms in (0.3, 0.8) at rows 0..2 exactly two drafts are accepted and
    the replacement differs from the rejected draft."""
    g = read_golden("sdmtp_probs.txt")
    probs = [float(x) for x in g["p_target"]]
    D, V = len(probs), 8
    drafts = [1, 2, 3, 4, 5]
    seed = next(s for s in range(10000)
                if all(0.35 < accept_uniform(s, 0, j) < 0.75 for j in range(3)))
    hidden = np.zeros((D + 1, V), np.float32)
    for j in range(D):
        hidden[j] = _logits_for_probs(probs[j], drafts[j], V)
    q = np.zeros((1, D, V), np.float32)
    for j in range(D):
        q[0, j, drafts[j]] = 1.0
    tokens = np.array([[0] + drafts], np.int32)
    res = orc.lmhead_accept(hidden, _identity_head(V), tokens, np.ones(1, np.uint8),
                            np.ones(1, np.float32), q, seed)
    assert int(res["num_accepted"][0]) == 2
    out = res["out_tokens"][0]
    assert out[:2].tolist() == drafts[:2]
    assert out[2] != drafts[2] and 0 <= out[2] < V
    assert out[3:].tolist() == [-1] * (D - 2)


def _random_case(rng, B, D, V, H, sampling_frac=0.5, gap=None):
    hidden = rng.standard_normal((B * (D + 1), H)).astype(np.float32)
    W = (rng.standard_normal((V, H)) * 0.5).astype(np.float32)
    tokens = rng.integers(0, V, (B, D + 1)).astype(np.int32)
    mode = (rng.random(B) < sampling_frac).astype(np.uint8)
    temp = rng.uniform(0.5, 1.5, B).astype(np.float32)
    q = rng.random((B, D, V)).astype(np.float32)
    q /= q.sum(-1, keepdims=True)
    return hidden, W, tokens, mode, temp, q


def test_logits_lse_argmax_against_numpy(orc):
    rng = np.random.default_rng(1)
    B, D, V, H = 3, 2, 300, 40
    hidden, W, tokens, mode, temp, q = _random_case(rng, B, D, V, H)
    res = orc.lmhead_accept(hidden, W, tokens, mode, temp, q, 5, want_logits=True)
    ref = (hidden.astype(np.float64) @ W.astype(np.float64).T).astype(np.float32)
    inv_t = (np.float32(1.0) / temp).astype(np.float32)
    for b in range(B):
        if mode[b] == 1:
            ref[b * (D + 1):(b + 1) * (D + 1)] *= inv_t[b]
    np.testing.assert_array_max_ulp(res["logits"], ref, maxulp=1)
    lse_ref = special.logsumexp(res["logits"].astype(np.float64), axis=1)
    np.testing.assert_allclose(res["lse"].reshape(-1), lse_ref, rtol=1e-6)
    assert (res["argmax"].reshape(-1) == np.argmax(res["logits"], axis=1)).all()


def test_argmax_lowest_index_on_ties(orc):
    V = 10
    hidden = np.zeros((2, V), np.float32)
    hidden[0, [3, 7]] = 2.0
    hidden[1, [9, 1]] = 4.0
    res = orc.lmhead_accept(hidden, _identity_head(V), np.array([[0, 3]], np.int32), np.zeros(1, np.uint8),
                            None, None, 0)
    assert res["argmax"][0].tolist() == [3, 1]
    assert int(res["num_accepted"][0]) == 1 and res["out_tokens"][0].tolist() == [3, 1]


def test_bf16_inputs_widen_exactly(orc):
    import torch
    rng = np.random.default_rng(2)
    h = torch.tensor(rng.standard_normal((4, 24)), dtype=torch.bfloat16)
    W = torch.tensor(rng.standard_normal((50, 24)), dtype=torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    res = orc.lmhead_accept(bits(h), bits(W), np.array([[1, 2, 3, 4]], np.int32), np.zeros(1, np.uint8),
                            None, None, 0, want_logits=True)
    ref = (h.double().numpy() @ W.double().numpy().T).astype(np.float32)
    np.testing.assert_array_max_ulp(res["logits"], ref, maxulp=1)


def test_greedy_invariants_random(orc):
    rng = np.random.default_rng(3)
    B, D, V, H = 64, 4, 50, 12
    hidden, W, tokens, mode, temp, q = _random_case(rng, B, D, V, H, sampling_frac=0.0)
    # Plant agreement: some drafts copy the argmax of the previous row.
    ref_argmax = np.argmax(hidden @ W.T, axis=1).reshape(B, D + 1)
    agree = rng.random((B, D)) < 0.7
    tokens[:, 1:] = np.where(agree, ref_argmax[:, :D], tokens[:, 1:])
    res = orc.lmhead_accept(hidden, W, tokens, mode, temp, None, 0)
    amax = res["argmax"]
    for b in range(B):
        n = int(res["num_accepted"][b])
        out = res["out_tokens"][b]
        assert 0 <= n <= D
        assert out[:n].tolist() == tokens[b, 1:n + 1].tolist()
        assert all(amax[b, j] == tokens[b, j + 1] for j in range(n))
        assert n == D or amax[b, n] != tokens[b, n + 1]
        assert out[n] == amax[b, n]
        assert (out[n + 1:] == -1).all()


def test_sampling_invariants_random(orc):
    rng = np.random.default_rng(4)
    B, D, V, H = 64, 5, 40, 10
    hidden, W, tokens, mode, temp, q = _random_case(rng, B, D, V, H, sampling_frac=1.0)
    res = orc.lmhead_accept(hidden, W, tokens, mode, temp, q, 11)
    for b in range(B):
        n = int(res["num_accepted"][b])
        out = res["out_tokens"][b]
        assert 0 <= n <= D
        assert out[:n].tolist() == tokens[b, 1:n + 1].tolist()
        assert 0 <= out[n] < V
        assert (out[n + 1:] == -1).all()


def test_one_hot_target_sampling_equals_greedy(orc):
    """With a one-hot target the rejection rule must reproduce the greedy rule."""
    rng = np.random.default_rng(5)
    B, D, V = 200, 3, 16
    target = rng.integers(0, V, (B, D + 1))
    hidden = np.zeros((B * (D + 1), V), np.float32)
    hidden[np.arange(B * (D + 1)), target.reshape(-1)] = 200.0
    tokens = rng.integers(0, V, (B, D + 1)).astype(np.int32)
    agree = rng.random((B, D)) < 0.6
    tokens[:, 1:] = np.where(agree, target[:, :D], tokens[:, 1:])
    q = rng.random((B, D, V)).astype(np.float32) + 0.01
    q /= q.sum(-1, keepdims=True)
    W = _identity_head(V)
    greedy = orc.lmhead_accept(hidden, W, tokens, np.zeros(B, np.uint8), None, None, 0)
    samp = orc.lmhead_accept(hidden, W, tokens, np.ones(B, np.uint8), np.ones(B, np.float32), q, 77)
    assert (greedy["num_accepted"] == samp["num_accepted"]).all()
    assert (greedy["out_tokens"] == samp["out_tokens"]).all()


def test_q_equal_p_accepts_every_draft(orc):
    rng = np.random.default_rng(6)
    B, D, V = 100, 4, 12
    hidden = rng.standard_normal((B * (D + 1), V)).astype(np.float32)
    p = special.softmax(hidden.astype(np.float64), axis=1).reshape(B, D + 1, V)
    q = (p[:, :D] * (1 - 1e-4)).astype(np.float32)
    tokens = rng.integers(0, V, (B, D + 1)).astype(np.int32)
    res = orc.lmhead_accept(hidden, _identity_head(V), tokens, np.ones(B, np.uint8), np.ones(B, np.float32), q, 3)
    assert (res["num_accepted"] == D).all()


def test_mode1_with_zero_temperature_is_greedy(orc):
    rng = np.random.default_rng(8)
    B, D, V, H = 20, 3, 30, 8
    hidden, W, tokens, mode, temp, q = _random_case(rng, B, D, V, H, sampling_frac=1.0)
    a = orc.lmhead_accept(hidden, W, tokens, np.ones(B, np.uint8), np.zeros(B, np.float32), q, 1)
    b = orc.lmhead_accept(hidden, W, tokens, np.zeros(B, np.uint8), None, None, 1)
    assert (a["out_tokens"] == b["out_tokens"]).all() and (a["num_accepted"] == b["num_accepted"]).all()


def _lossless_run(orc, trials, D, V, seed):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((D + 1, V)).astype(np.float32) * 1.2
    qlog = rng.standard_normal((D, V)) * 1.2
    q = special.softmax(qlog, axis=1).astype(np.float32)
    hidden = np.tile(logits, (trials, 1))
    tokens = np.zeros((trials, D + 1), np.int32)
    for j in range(D):
        tokens[:, j + 1] = rng.choice(V, size=trials, p=q[j] / q[j].sum())
    qd = np.broadcast_to(q, (trials, D, V)).copy()
    res = orc.lmhead_accept(hidden, _identity_head(V), tokens, np.ones(trials, np.uint8),
                            np.ones(trials, np.float32), qd, seed)
    p = special.softmax(logits.astype(np.float64), axis=1)
    return res, p, q


@pytest.mark.parametrize("D", [1, 3])
def test_rejection_sampling_is_lossless_chi2(orc, D):
    """The first emitted token is distributed exactly as p_target of row 0, and
    given that draft 1 was accepted the second is distributed as row 1."""
    trials, V = 300_000, 8
    res, p, q = _lossless_run(orc, trials, D, V, seed=100 + D)
    first = res["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    chi2, pval = stats.chisquare(counts, p[0] * trials)
    assert pval > 1e-3, (counts, p[0] * trials)
    if D >= 2:
        sel = res["num_accepted"] >= 1
        second = res["out_tokens"][sel, 1]
        counts2 = np.bincount(second, minlength=V)
        chi2, pval = stats.chisquare(counts2, p[1] * sel.sum())
        assert pval > 1e-3


def test_acceptance_rate_matches_min_p_q(orc):
    trials, V, D = 300_000, 8, 1
    res, p, q = _lossless_run(orc, trials, D, V, seed=7)
    alpha = np.minimum(p[0], q[0].astype(np.float64)).sum()
    rate = (res["num_accepted"] >= 1).mean()
    sigma = np.sqrt(alpha * (1 - alpha) / trials)
    assert abs(rate - alpha) < 4 * sigma


def test_race_rule_small_cases(orc):
    assert orc.race(np.array([1, 1, 1], np.float32), np.array([3, 1, 2], np.float32)) == (1, 0)
    assert orc.race(np.array([1, 1], np.float32), np.array([1, 1], np.float32)) == (0, 1)
    assert orc.race(np.zeros(4, np.float32), np.ones(4, np.float32))[0] == -1
    assert orc.race(np.array([0.0, 0.2], np.float32), np.array([0.0, 5.0], np.float32))[0] == 1
    assert orc.race(np.array([0.1, 0.2], np.float32), np.array([0.0, 5.0], np.float32))[0] == 0


def test_race_picks_in_proportion_to_weight(orc):
    rng = np.random.default_rng(9)
    w = np.array([0.05, 0.3, 0.0, 0.15, 0.5], np.float32)
    n = 40_000
    wins = np.zeros(len(w), np.int64)
    for _ in range(n):
        E = rng.exponential(size=len(w)).astype(np.float32)
        wins[orc.race(w, E)[0]] += 1
    assert wins[2] == 0
    nz = w > 0
    chi2, pval = stats.chisquare(wins[nz], w[nz] / w.sum() * n)
    assert pval > 1e-3
