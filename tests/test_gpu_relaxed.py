"""GPU parity of relaxed acceptance (mode 2; "MTP in TensorRT-LLM on
Blackwell", MTP optimization: relaxed acceptance) against the CPU oracle.

The synthetic relaxed rows plant a leader and a runner-up so that every
branch of the rule occurs: drafts accepted as the top-1 token, accepted as a
lower-ranked candidate, rejected by rank and rejected by the probability
threshold. Cases cover the single-CTA and CTA-pair tensor-core LM heads and
the fp32 SIMT LM head, mixed batches
with greedy and sampling requests, N = 1 / delta = 0, long chains and the
full DeepSeek-V3-shaped workload.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402
from gpu_util import (A, TOL_LOGITS, TOL_LSE_REL, check_invariants, compare_accept, gpu_lmhead,  # noqa: E402
                      oracle_lmhead)

DEV = torch.device("cuda:0")

_BASE = synth.CFG3.with_(Hq=8, Hkv=2, ctx=(64, 200))

SMALL = {
    # M = 160 rows: one tensor-core CTA per vocabulary slice; relaxed first half, sampling second half
    "tc_single_mixed": _BASE.with_(name="relaxed TC mixed", B=40, D=3, H=256, V=5003, relaxed="half",
                                   sampling="half", relaxed_topk=4, relaxed_delta=0.3, stream=21),
    # M = 256 rows: CTA-pair tensor-core LM head, every request relaxed
    "tc_pair_all": _BASE.with_(name="relaxed TC pairs", B=64, D=3, H=128, V=7001, relaxed="all",
                               sampling="none", relaxed_topk=8, relaxed_delta=0.6, stream=22),
    # fp32: SIMT LM head
    "simt_f32": synth.CFG0.with_(name="relaxed SIMT fp32", B=12, D=3, H=64, V=3001, relaxed="all",
                                 relaxed_topk=3, relaxed_delta=0.2, stream=23),
    # fp32 SIMT LM head, mixed with sampling requests; ragged vocabulary tail
    "simt_f32_mixed": synth.CFG0.with_(name="relaxed SIMT fp32 mixed", B=10, D=2, H=96, V=1037, relaxed="half",
                                       sampling="half", relaxed_topk=5, relaxed_delta=0.5, stream=24),
    # N = 1, delta = 0: the strict rule
    "top1_delta0": _BASE.with_(name="relaxed N=1 delta=0", B=24, D=3, H=128, V=4099, relaxed="all",
                               sampling="none", relaxed_topk=1, relaxed_delta=0.0, stream=25),
    # long chain, top-N larger than the number of close competitors
    "d7_topk_large": _BASE.with_(name="relaxed D=7", B=16, D=7, H=192, V=6007, relaxed="all", sampling="none",
                                 relaxed_topk=64, relaxed_delta=0.9, stream=26),
}


def _oracle_all(w, lm, reqs):
    W = A(lm["lm_head"])
    res = [oracle_lmhead(w, lm, [b], W, want_logits=True) for b in reqs]
    return {k: np.concatenate([r[k] for r in res]) for k in res[0]}


def _check(w, lm, gpu, reqs):
    """Decisions bit-exact outside near-ties; argmax exact; logits within the
    dtype's tolerance; each row's log-sum-exp within that row's largest logit
    error (log-sum-exp is 1-Lipschitz in the max-norm of the logits: sharp
    rows, whose lse is about their top logit, inherit its accumulation
    error) plus 1e-5 relative."""
    ref = _oracle_all(w, lm, reqs)
    flagged = compare_accept(gpu, ref, reqs)
    idx = torch.tensor(list(reqs), device=DEV)
    assert (gpu["argmax"].index_select(0, idx).cpu().numpy() == ref["argmax"]).all()
    rows = torch.tensor([b * w.R + j for b in reqs for j in range(w.R)], device=DEV)
    dl = np.abs(gpu["logits"].index_select(0, rows).cpu().numpy() - ref["logits"])
    assert float(dl.max()) < TOL_LOGITS[w.dtype], float(dl.max())
    row_err = dl.max(axis=1).reshape(len(reqs), w.R)
    g_lse = gpu["lse"].index_select(0, idx).cpu().numpy()
    bound = row_err + TOL_LSE_REL * np.abs(ref["lse"]) + 1e-6
    assert (np.abs(g_lse - ref["lse"]) <= bound).all(), float(np.abs(g_lse - ref["lse"]).max())
    return flagged, ref


@pytest.mark.parametrize("name", list(SMALL))
def test_relaxed_small_all_requests(name):
    w = SMALL[name]
    lm = synth.make_lmhead_inputs(w, DEV)
    gpu = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    flagged, ref = _check(w, lm, gpu, range(w.B))
    assert flagged <= max(1, w.B // 20)
    check_invariants(w, lm, gpu)
    # The relaxed rows accept beyond the strict rule somewhere (runner-up drafts).
    if w.relaxed_topk > 1:
        mode = lm["mode"].cpu().numpy()
        n = gpu["num_accepted"].cpu().numpy()
        tok = lm["tokens"].cpu().numpy()
        amax = gpu["argmax"].cpu().numpy()
        beyond = sum(1 for b in range(w.B) if mode[b] == 2
                     for j in range(int(n[b])) if amax[b, j] != tok[b, j + 1])
        assert beyond > 0


def test_relaxed_top1_delta0_equals_greedy():
    """With N = 1 and delta = 0 a relaxed request decides exactly like a greedy one."""
    w = SMALL["top1_delta0"]
    lm = synth.make_lmhead_inputs(w, DEV)
    relaxed = gpu_lmhead(w, lm)
    lm_g = dict(lm, mode=torch.zeros_like(lm["mode"]), relaxed_topk=0)
    greedy = gpu_lmhead(w, lm_g)
    mv.sync_status()
    keep = (relaxed["tie_flags"] == 0).cpu()
    assert bool(keep.any())
    for k in ("out_tokens", "num_accepted", "argmax"):
        assert torch.equal(relaxed[k].cpu()[keep], greedy[k].cpu()[keep]), k


def test_relaxed_noalloc_matches_workspace_path():
    w = SMALL["tc_pair_all"]
    lm = synth.make_lmhead_inputs(w, DEV)
    ref = gpu_lmhead(w, lm)
    out = torch.full((w.B, w.R), -9, dtype=torch.int32, device=DEV)
    n = torch.full((w.B,), -9, dtype=torch.int32, device=DEV)
    tie = torch.full((w.B,), 255, dtype=torch.uint8, device=DEV)
    mv.mtp_verify_logits_accept_noalloc(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"], lm["temperature"],
                                        lm["q_draft"], lm["seed"], out, n, tie, relaxed_topk=w.relaxed_topk,
                                        relaxed_delta=w.relaxed_delta)
    mv.sync_status()
    assert torch.equal(out, ref["out_tokens"]) and torch.equal(n, ref["num_accepted"])
    assert torch.equal(tie, ref["tie_flags"])


def test_relaxed_mode_without_topk_is_reported_and_greedy():
    """Mode 2 while relaxed_topk is 0, or a mode above 2: the device error word
    reports "mode" and the request is decided greedily."""
    w = SMALL["tc_single_mixed"]
    lm = synth.make_lmhead_inputs(w, DEV)
    lm0 = dict(lm, relaxed_topk=0)
    got = gpu_lmhead(w, lm0)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert ei.value.code == 4 and "mode" in str(ei.value)
    greedy_mode = torch.where(lm["mode"] == 2, torch.zeros_like(lm["mode"]), lm["mode"])
    ref = gpu_lmhead(w, dict(lm, mode=greedy_mode, relaxed_topk=0))
    mv.sync_status()
    for k in ("out_tokens", "num_accepted"):
        assert torch.equal(got[k], ref[k]), k
    lm3 = dict(lm, mode=torch.where(lm["mode"] == 2, torch.full_like(lm["mode"], 3), lm["mode"]))
    got3 = gpu_lmhead(w, lm3)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert "mode" in str(ei.value)
    assert torch.equal(got3["num_accepted"], ref["num_accepted"])


def test_relaxed_bad_arguments_rejected():
    w = SMALL["simt_f32"]
    lm = synth.make_lmhead_inputs(w, DEV)
    for topk, delta in ((-1, 0.1), (w.V + 1, 0.1), (3, -0.5), (3, float("nan"))):
        with pytest.raises(mv.MtpError) as ei:
            gpu_lmhead(w, dict(lm, relaxed_topk=topk, relaxed_delta=delta))
        assert ei.value.code == 1
    mv.sync_status()


def test_relaxed_full_size_cfg1_sampled_requests():
    """DeepSeek-V3-shaped LM head (B=32, D=3, H=7168, V=129280), every request
    relaxed with N = 10, delta = 0.6; the oracle checks a sample of requests,
    every request is checked for the properties of the rule."""
    w = synth.CFG1.with_(relaxed="all", relaxed_topk=10, relaxed_delta=0.6)
    torch.cuda.empty_cache()
    lm = synth.make_lmhead_inputs(w, DEV)
    gpu = gpu_lmhead(w, lm)                        # the benchmark's launch configuration
    dbg = gpu_lmhead(w, lm, debug_logits=True)     # the same, also writing the logits out
    mv.sync_status()
    for k in ("out_tokens", "num_accepted", "tie_flags", "lse", "argmax"):
        assert torch.equal(gpu[k], dbg[k]), k
    flagged, _ = _check(w, lm, dbg, [0, 17, 31])
    ties = gpu["tie_flags"].cpu().numpy()
    print("relaxed DeepSeek-V3-shaped step: %d of %d requests inside the relaxed near-tie band (excluded from the "
          "bit-exact comparison); sampled requests flagged on either side: %d of 3" %
          (int(((ties & 1) != 0).sum()), w.B, flagged))
    assert flagged <= 1
    check_invariants(w, lm, gpu)
    del lm, gpu, dbg
    torch.cuda.empty_cache()
