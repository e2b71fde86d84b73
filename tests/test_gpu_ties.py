"""GPU tie rules against the oracle, on exactly equal values planted where the
kernels split the work.

"MTP in TensorRT-LLM on Blackwell", Fig. 1: each draft is compared with the
target's own prediction, the argmax of its row. Equal logits are resolved
to the lowest token id; the library splits the vocabulary over 128-row tiles
and CTAs (and the exponential race over vocabulary slices), so the rule has
to hold across those splits:

  * argmax: one W row copied to token ids 5, V/2 + 1 and V - 3 (different
    tiles and CTAs) gives those three exactly equal logits; rows planted on
    that direction must report argmax 5 on the single-CTA and CTA-pair
    tensor-core LM heads and on the fp32 SIMT one, and drafts of V - 3 must be
    rejected with 5 as the correction;
  * relaxed acceptance: tokens tied above the draft count before it and a
    rejection is corrected to the lowest-id argmax; a draft exactly tied
    with others is a near-tie (flagged on both sides), since the library
    takes the draft's own logit from a pre-pass;
  * the race: two vocabulary ids whose race words are equal get equal
    exponentials; with equal weights their keys are equal and the draw must
    be the lower id (and be flagged as a near-tie on both sides).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402
from gpu_util import gpu_lmhead, oracle_lmhead  # noqa: E402
from philox_py import race_words_vec  # noqa: E402

DEV = torch.device("cuda:0")
TAG_BONUS = 3


def _plant_duplicates(lm, ids, scale, rows):
    """W[ids] := one unit vector u (norm 1, far above the other rows' ~0.02*sqrt(H));
    hidden rows `rows` := scale * u, so those rows' largest logits are the
    duplicates', exactly equal on both sides."""
    W = lm["lm_head"]
    H = W.shape[1]
    g = torch.Generator(device="cpu").manual_seed(123)
    u = torch.randn(H, generator=g, dtype=torch.float64)
    u = (u / u.norm()).to(W.dtype).to(W.device)
    for v in ids:
        W[v] = u
    for m in rows:
        lm["hidden"][m] = (scale * u.double()).to(W.dtype)


LM_CASES = {
    "tc_single_cta": dict(dtype="bf16", B=4, D=3, H=128),      # M = 16: single-CTA tensor-core LM head
    "tc_cta_pairs_n64": dict(dtype="bf16", B=10, D=3, H=128),  # M = 40: CTA pairs of N = 64
    "tc_cta_pairs": dict(dtype="bf16", B=50, D=3, H=128),      # M = 200: CTA pairs
    "tc_two_row_groups": dict(dtype="bf16", B=100, D=3, H=64),  # M = 400: two row groups on CTA pairs
    "simt_fp32": dict(dtype="f32", B=4, D=3, H=64),            # fp32 SIMT LM head
}


@pytest.mark.parametrize("name", list(LM_CASES))
def test_argmax_ties_lowest_id_across_tiles_and_ctas(name):
    c = LM_CASES[name]
    V = 5003
    w = synth.CFG0.with_(name="argmax ties " + name, V=V, sampling="none", **c)
    lm = synth.make_lmhead_inputs(w, DEV)
    dup = [5, V // 2 + 1, V - 3]
    planted_rows = [b * w.R + j for b in range(w.B) for j in range(0, w.R, 2)]
    _plant_duplicates(lm, dup, 20.0, planted_rows)
    tok = lm["tokens"]
    for b in range(w.B):
        for j in range(0, w.D, 2):
            tok[b, j + 1] = 5 if b % 2 == 0 else V - 3
    gpu = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    logits = gpu["logits"].cpu().numpy()
    for m in planted_rows:   # the premise: bitwise equal logits at the duplicates
        assert logits[m, dup[0]] == logits[m, dup[1]] == logits[m, dup[2]], m
        assert logits[m, dup[0]] == logits[m].max()
    amax = gpu["argmax"].cpu().numpy().reshape(-1)
    assert (amax[planted_rows] == 5).all()
    ref = oracle_lmhead(w, lm, range(w.B))
    assert (gpu["argmax"].cpu().numpy() == ref["argmax"]).all()
    assert (gpu["out_tokens"].cpu().numpy() == ref["out_tokens"]).all()
    assert (gpu["num_accepted"].cpu().numpy() == ref["num_accepted"]).all()
    n = gpu["num_accepted"].cpu().numpy()
    out = gpu["out_tokens"].cpu().numpy()
    for b in range(1, w.B, 2):   # a draft of V - 3 at row 0 is rejected, corrected to 5
        assert n[b] == 0 and out[b, 0] == 5


@pytest.mark.parametrize("topk", [1, 2, 3])
def test_relaxed_exact_tie_at_the_draft_is_a_near_tie(topk):
    """Draft logit exactly equal to two other tokens' (the lowest-id rule
    decides its rank). The library computes the draft's logit in a pre-pass
    with its own summation order, so where the tied group straddles the top-N
    boundary the decision is a near-tie by construction and both sides flag
    it; the outcome must still be valid, and a rejection is corrected to the
    lowest-id argmax. With N = 3 every tied token is inside: no flag, and the
    GPU equals the oracle."""
    V = 5003
    w = synth.CFG0.with_(name="relaxed ties", V=V, dtype="bf16", B=6, D=1, H=128, sampling="none")
    lm = synth.make_lmhead_inputs(w, DEV)
    dup = [5, V // 2 + 1, V - 3]
    _plant_duplicates(lm, dup, 20.0, [b * w.R for b in range(w.B)])
    for b in range(w.B):
        lm["tokens"][b, 1] = dup[b % 3]
    lm["mode"].fill_(2)
    lm = dict(lm, relaxed_topk=topk, relaxed_delta=1.0)
    gpu = gpu_lmhead(w, lm)
    mv.sync_status()
    ref = oracle_lmhead(w, lm, range(w.B))
    g_tie = gpu["tie_flags"].cpu().numpy()
    n = gpu["num_accepted"].cpu().numpy()
    out = gpu["out_tokens"].cpu().numpy()
    assert (g_tie == ref["tie_flags"]).all()
    if topk < len(dup):   # the tied group straddles the top-N boundary: flagged
        assert (g_tie & 1).all()
        for b in range(w.B):
            assert out[b, 0] == (dup[b % 3] if n[b] == 1 else 5)
    else:                 # every tied token is inside the top N: a sure accept
        assert (g_tie == 0).all() and (n == 1).all() and (n == ref["num_accepted"]).all()
        assert (out == ref["out_tokens"]).all()


@pytest.mark.parametrize("topk,accepted", [(2, 0), (3, 1)])
def test_relaxed_rank_past_tied_top_tokens(topk, accepted):
    """Two tokens tie at the top (ids 5 and V - 3), the draft ranks third with
    a clear margin: accepted for top-3, rejected for top-2 and corrected to
    the lowest-id argmax, 5; no near-tie, so the GPU must equal the oracle."""
    V = 5003
    w = synth.CFG0.with_(name="relaxed, tied top", V=V, dtype="bf16", B=4, D=1, H=128, sampling="none")
    lm = synth.make_lmhead_inputs(w, DEV)
    _plant_duplicates(lm, [5, V - 3], 20.0, [b * w.R for b in range(w.B)])
    c = 100
    lm["lm_head"][c] = (0.95 * lm["lm_head"][5].double()).to(lm["lm_head"].dtype)   # logit ~19: third
    lm["tokens"][:, 1] = c
    lm["mode"].fill_(2)
    lm = dict(lm, relaxed_topk=topk, relaxed_delta=1.0)
    gpu = gpu_lmhead(w, lm)
    mv.sync_status()
    ref = oracle_lmhead(w, lm, range(w.B))
    assert (gpu["tie_flags"].cpu().numpy() == 0).all() and (ref["tie_flags"] == 0).all()
    assert (gpu["num_accepted"].cpu().numpy() == ref["num_accepted"]).all()
    assert (gpu["out_tokens"].cpu().numpy() == ref["out_tokens"]).all()
    assert (gpu["num_accepted"].cpu().numpy() == accepted).all()
    if not accepted:
        assert (gpu["out_tokens"].cpu().numpy()[:, 0] == 5).all()


def _philox_collision(V, b, j, tag, seeds):
    """First (seed, v1, v2) with v1 < v2 whose race words are equal."""
    v = np.arange(V, dtype=np.uint64)
    for seed in seeds:
        x = race_words_vec(seed, b, j, v, tag)
        order = np.argsort(x, kind="stable")
        xs = x[order]
        hit = np.nonzero(xs[1:] == xs[:-1])[0]
        if len(hit):
            v1, v2 = sorted((int(order[hit[0]]), int(order[hit[0] + 1])))
            return seed, v1, v2
    return None


def test_race_equal_keys_draw_the_lower_id():
    """Bonus draw (every draft accepted) over p_D, whose mass sits on two ids
    v1 < v2 with equal logits and equal Philox words: equal race keys."""
    V, D = 65536 + 37, 1
    found = _philox_collision(V, 0, D, TAG_BONUS, range(1, 200))
    assert found is not None
    seed, v1, v2 = found
    w = synth.CFG0.with_(name="race ties", V=V, dtype="bf16", B=2, D=D, H=64, sampling="all")
    lm = synth.make_lmhead_inputs(w, DEV)
    _plant_duplicates(lm, [v1, v2], 50.0, [0, 1])   # request 0: both rows on the tied pair
    lm["tokens"][0, 1] = v1
    q = lm["q_draft"]
    q[0].fill_(1.0 / V)
    q[0, 0, v1] = 1e-6                                # p(v1) ~ 0.5 >= U q: the draft is accepted
    lm = dict(lm, seed=seed)
    gpu = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    lg = gpu["logits"].cpu().numpy()
    assert lg[1, v1] == lg[1, v2] == lg[1].max()
    ref = oracle_lmhead(w, lm, [0])
    assert int(gpu["num_accepted"][0]) == int(ref["num_accepted"][0]) == 1
    assert int(gpu["out_tokens"][0, 1]) == int(ref["out_tokens"][0, 1]) == v1
    assert int(gpu["tie_flags"][0]) & 2 and int(ref["tie_flags"][0]) & 2
