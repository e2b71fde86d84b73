"""Whole verify steps at full size against the oracle, on sampled requests.

The sweep on the large-batch shapes (contexts 8192, GQA 32/8 x 128, hidden
4096, vocabulary 151936, every request rejection-sampled at T = 0.7) at
B in {64, 256, 512} x D in {3, 7}, and the large-batch mixed batch with trees
of 15 drafts (M = 4096 rows, the tcgen05 GQA attention on 18 GB of KV), each
in the launch configuration the benchmark times:

  * attention of the sampled requests within the attention bound of the
    oracle's exact result;
  * LM head: tokens, accept counts (bit-exact unless a side flags a near-tie),
    log-sum-exp and argmax of the sampled requests; then the same call with
    the debug logits, whose results must be identical, and the sampled rows'
    logits within 2e-2 of the oracle's;
  * KV compaction (trees) and rollback of every request against the oracle's
    bookkeeping, and the kept K/V of the sampled requests against the
    oracle's cache.

"MTP principles" §三 stage 3 (accept if P_target/P_draft >= U, else resample
from the residual) and stage 4 (1..D+1 tokens per step); "Multi Token
Prediction" note, K=3 flow, steps 2 and 4-6.
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402
from gpu_util import (A, TOL_ATTN, TOL_LOGITS, TOL_LSE_REL, attention_excess, attention_over_plain,  # noqa: E402
                      check_invariants, compare_accept, gpu_attention, gpu_lmhead, gpu_rollback, oracle_attention,
                      oracle_lmhead)

DEV = torch.device("cuda:0")

CASES = {"sweep_B%d_D%d" % (B, D): synth.sweep_point(B, D) for B in (64, 256, 512) for D in (3, 7)}
CASES["tree_cfg3_D15"] = synth.CFG3.with_(name=synth.CFG3.name.replace("D=3", "tree of 15 drafts (3x2x1 fan-out)"),
                                          D=15, tree="full", sampling="none")


def _par(fn, items):
    with cf.ThreadPoolExecutor(max_workers=8) as ex:
        return list(ex.map(fn, items))


def _sample(w, ctx):
    """First, last, the longest context and one in the middle."""
    return sorted({0, w.B // 2 + 1, w.B - 1, int(np.argmax(ctx))})


@pytest.mark.parametrize("name", list(CASES))
def test_whole_step_sampled_requests(name):
    w = CASES[name]
    torch.cuda.empty_cache()
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    parents = lm.get("parents")
    table0, ctx0 = A(att["block_table"]).copy(), A(att["ctx_lens"]).copy()
    reqs = _sample(w, ctx0)

    # Attention (with the append); the oracle gathers its cache pages before
    # the compaction moves any slot.
    out = gpu_attention(w, att, parents)
    mv.sync_status()
    orc = _par(lambda b: oracle_attention(w, att, [b], parents, return_cache=True), reqs)
    exact = np.concatenate([o[0] for o in orc])
    got = out.index_select(0, torch.tensor(reqs, device=DEV)).float().cpu().numpy()
    n_over, frac = attention_over_plain(got, exact, w.dtype)
    print("%s attention: max |err| %.3g, %d element(s) (%.2g) above the plain %g" %
          (name, float(np.abs(got - exact).max()), n_over, frac, TOL_ATTN[w.dtype]))
    assert attention_excess(got, exact, w.dtype) <= 0.0

    # LM head + acceptance as the benchmark runs it, then again with the debug logits.
    gpu = gpu_lmhead(w, lm)
    mv.sync_status()
    dbg = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    for k in ("out_tokens", "num_accepted", "tie_flags", "lse", "argmax", "accepted_nodes"):
        assert torch.equal(gpu[k], dbg[k]), k
    W = A(lm["lm_head"])
    ref = _par(lambda b: oracle_lmhead(w, lm, [b], W, want_logits=True), reqs)
    ref = {k: np.concatenate([r[k] for r in ref]) for k in ref[0]}
    flagged = compare_accept(gpu, ref, reqs)
    idx = torch.tensor(reqs, device=DEV)
    np.testing.assert_allclose(gpu["lse"].index_select(0, idx).cpu().numpy(), ref["lse"], rtol=TOL_LSE_REL,
                               atol=1e-6)
    assert (gpu["argmax"].index_select(0, idx).cpu().numpy() == ref["argmax"]).all()
    rows = torch.tensor([b * w.R + j for b in reqs for j in range(w.R)], device=DEV)
    lg = dbg["logits"].index_select(0, rows).cpu().numpy()
    err = float(np.abs(lg - ref["logits"]).max())
    assert err < TOL_LOGITS[w.dtype], err
    ties = gpu["tie_flags"].cpu().numpy()
    print("%s: logits max |err| %.3g over %d rows; near-ties flagged by the GPU: accept %d, race %d of %d "
          "requests; sampled requests flagged on either side: %d of %d" %
          (name, err, len(rows), int(((ties & 1) != 0).sum()), int(((ties & 2) != 0).sum()), w.B, flagged,
           len(reqs)))
    assert flagged <= 1
    check_invariants(w, lm, gpu)
    del dbg

    # Compaction (trees) and rollback of every request.
    n_gpu = gpu["num_accepted"]
    if parents is not None:
        mv.mtp_tree_kv_compact(att["k_cache"], att["v_cache"], att["block_table"], att["ctx_lens"],
                               gpu["accepted_nodes"], n_gpu)
    table, seq, fl, fc = gpu_rollback(w, att["block_table"], att["ctx_lens"], n_gpu)
    mv.sync_status()
    t_h, s_h = table0.copy(), ctx0.copy()
    fl_h, fc_h = np.full(fl.numel(), -1, np.int32), np.zeros(1, np.int32)
    oracle.kv_rollback(t_h, s_h, n_gpu.cpu().numpy(), fl_h, fc_h, D=w.D, block_size=64)
    assert (seq.cpu().numpy() == s_h).all() and (table.cpu().numpy() == t_h).all()
    assert int(fc.item()) == int(fc_h[0]) and (fl.cpu().numpy() == fl_h).all()
    # The kept verify slots of each sampled request hold the oracle's K/V
    # (after the oracle's own compaction of its cache copy).
    kc_g = att["k_cache"]
    vc_g = att["v_cache"]
    for i, b in enumerate(reqs):
        if ties[b] or ref["tie_flags"][i]:
            continue   # a near-tie may decide differently on the two sides
        _, kc, vc, sub = orc[i]
        n = int(ref["num_accepted"][i])
        if parents is not None:
            oracle.tree_kv_compact(kc, vc, sub, ctx0[b:b + 1], ref["accepted_nodes"][i:i + 1],
                                   ref["num_accepted"][i:i + 1], D=w.D, Hkv=w.Hkv, d_qk=w.d_qk, d_v=w.d_v,
                                   block_size=64, is_mla=w.is_mla)
        for s in range(int(ctx0[b]), int(ctx0[b]) + n + 1):
            blk_g, blk_o, off = int(table0[b, s // 64]), int(sub[0, s // 64]), s % 64
            assert (A(kc_g[blk_g, off]) == kc[blk_o, off]).all(), (b, s)
            if vc is not None:
                assert (A(vc_g[blk_g, off]) == vc[blk_o, off]).all(), (b, s)
    del att, lm, out, gpu
    torch.cuda.empty_cache()
