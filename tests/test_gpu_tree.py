"""GPU parity of tree drafts ("MTP in TensorRT-LLM on Blackwell", future work:
tree speculative sampling, Fig. 9) against the CPU oracle: attention under the
tree mask on every attention kernel (fp32 SIMT, bf16 GQA/MHA, bf16 MLA on
single CTAs and CTA pairs), greedy tree acceptance, and the whole step with
the KV compaction and rollback. Full-size DeepSeek-V3-shaped trees are
checked on sampled requests against the oracle and on every request against
the acceptance the planted targets imply."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402
from gpu_util import (A, attention_excess, compare_accept, gpu_attention, gpu_lmhead, gpu_rollback,  # noqa: E402
                      oracle_attention, oracle_lmhead)

DEV = torch.device("cuda:0")

SMALL = {
    "simt_f32_random": synth.CFG0.with_(name="tree fp32", D=7, ctx=(0, 150), tree="random", B=5, stream=41),
    "gqa_bf16_full": synth.CFG3.with_(name="tree GQA", B=6, D=15, Hq=16, Hkv=2, ctx=(60, 400), H=128, V=3001,
                                      sampling="none", tree="full", stream=42),
    "mha_bf16_d64_random": synth.CFG0.with_(name="tree MHA d64", dtype="bf16", D=9, ctx=(1, 200), B=4, H=64,
                                            V=999, tree="random", stream=43),
    # MLA, 2 row blocks per request (CTA pairs) and 3 (single CTAs)
    "mla_pairs_full": synth.CFG1.with_(name="tree MLA pairs", B=3, D=7, Hq=16, ctx=(60, 700), H=128, V=2000,
                                       tree="full", stream=44),
    "mla_single_random": synth.CFG1.with_(name="tree MLA single", B=2, D=11, Hq=16, ctx=(1, 300), H=64, V=777,
                                          tree="random", stream=45),
}


def _out_np(w, t):
    t = t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
    return t


def _ref_np(ref):
    if ref.dtype in (np.float32, np.float64):
        return ref
    return torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy()


def _planted_expectation(w, lm, parents_row, b):
    """Acceptance implied by the planted targets (argmax of node k's row is
    planted[b, k]): deepest node whose root path matches, lowest index first."""
    tok = lm["tokens"][b].cpu().numpy()
    planted = lm["planted"][b].numpy()
    R = w.R
    acc, depth = [True] + [False] * (R - 1), [0] * R
    best = 0
    for k in range(1, R):
        p = int(parents_row[k])
        acc[k] = acc[p] and tok[k] == planted[p]
        depth[k] = depth[p] + 1
        if acc[k] and depth[k] > depth[best]:
            best = k
    path = [best]
    while path[-1] != 0:
        path.append(int(parents_row[path[-1]]))
    return path[::-1], int(planted[best])


@pytest.mark.parametrize("name", list(SMALL))
def test_tree_small_all_requests(name):
    w = SMALL[name]
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    parents = lm["parents"]
    out = gpu_attention(w, att, parents)
    gpu = gpu_lmhead(w, lm)
    mv.sync_status()
    ref = oracle_attention(w, att, range(w.B), parents)
    assert attention_excess(_out_np(w, out), _ref_np(ref), w.dtype) <= 0.0
    ref_lm = oracle_lmhead(w, lm, range(w.B))
    assert compare_accept(gpu, ref_lm, range(w.B)) == 0
    assert (gpu["argmax"].cpu().numpy() == ref_lm["argmax"]).all()
    # Some request accepts along a branch other than the first child chain.
    nodes = gpu["accepted_nodes"].cpu().numpy()
    n = gpu["num_accepted"].cpu().numpy()
    assert any(list(nodes[b, :n[b] + 1]) != list(range(n[b] + 1)) for b in range(w.B)) or w.B < 3


@pytest.mark.parametrize("name", ["gqa_bf16_full", "mla_pairs_full"])
def test_chain_as_tree_matches_chain(name):
    w = SMALL[name].with_(tree="chain")
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    chain = torch.arange(-1, w.D, dtype=torch.int32, device=DEV).repeat(w.B, 1)
    k0 = att["k_cache"].clone()
    a = gpu_attention(w, att)
    att["k_cache"].copy_(k0)
    t = gpu_attention(w, att, chain)
    g1 = gpu_lmhead(w, lm)
    g2 = gpu_lmhead(w, dict(lm, parents=chain))
    mv.sync_status()
    assert torch.equal(a, t)
    for k in ("out_tokens", "num_accepted", "accepted_nodes"):
        assert torch.equal(g1[k], g2[k]), k


def test_tree_step_with_compaction_and_rollback():
    """Attention (append) -> accept -> compaction -> rollback on the GPU
    against the oracle's same four steps on a host copy of the cache: the
    kept sequence of every request holds the same K/V, the block tables,
    lengths and free lists agree."""
    w = SMALL["gqa_bf16_full"]
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    parents = lm["parents"]
    kc_h, vc_h = A(att["k_cache"]).copy(), A(att["v_cache"]).copy()
    table0 = att["block_table"].clone()
    ctx0 = att["ctx_lens"].clone()
    gpu_attention(w, att, parents)
    gpu = gpu_lmhead(w, lm)
    mv.mtp_tree_kv_compact(att["k_cache"], att["v_cache"], att["block_table"], att["ctx_lens"],
                           gpu["accepted_nodes"], gpu["num_accepted"])
    table, seq, fl, fc = gpu_rollback(w, att["block_table"], att["ctx_lens"], gpu["num_accepted"])
    mv.sync_status()
    # oracle: the same steps on the host
    oracle.verify_attention(A(att["q"]), A(att["k_new"]), A(att["v_new"]), kc_h, vc_h, A(table0), A(ctx0), D=w.D,
                            Hq=w.Hq, Hkv=w.Hkv, d_qk=w.d_qk, d_v=w.d_v, block_size=64, is_mla=False,
                            sm_scale=w.sm_scale, parents=A(parents))
    ref = oracle_lmhead(w, lm, range(w.B))
    oracle.tree_kv_compact(kc_h, vc_h, A(table0), A(ctx0), ref["accepted_nodes"], ref["num_accepted"], D=w.D,
                           Hkv=w.Hkv, d_qk=w.d_qk, d_v=w.d_v, block_size=64, is_mla=False)
    t_h, s_h = A(table0).copy(), A(ctx0).copy()
    fl_h, fc_h = np.full(fl.numel(), -1, np.int32), np.zeros(1, np.int32)
    oracle.kv_rollback(t_h, s_h, ref["num_accepted"], fl_h, fc_h, D=w.D, block_size=64)
    assert (seq.cpu().numpy() == s_h).all() and (table.cpu().numpy() == t_h).all()
    assert int(fc.item()) == int(fc_h[0]) and (fl.cpu().numpy() == fl_h).all()
    kc_g, vc_g = A(att["k_cache"]), A(att["v_cache"])
    tbl0 = A(table0)
    for b in range(w.B):
        for s in range(int(s_h[b])):     # every kept slot: context, input token, accepted path
            blk, off = tbl0[b, s // 64], s % 64
            assert (kc_g[blk, off] == kc_h[blk, off]).all() and (vc_g[blk, off] == vc_h[blk, off]).all(), (b, s)


def test_tree_sampling_request_is_reported_and_greedy():
    w = SMALL["gqa_bf16_full"].with_(sampling="half")
    lm = synth.make_lmhead_inputs(w, DEV)
    got = gpu_lmhead(w, lm)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert "mode" in str(ei.value)
    greedy = dict(lm, mode=torch.zeros_like(lm["mode"]))
    ref = gpu_lmhead(w, greedy)
    mv.sync_status()
    for k in ("out_tokens", "num_accepted", "accepted_nodes"):
        assert torch.equal(got[k], ref[k]), k


def test_malformed_parents_are_reported_and_computed_as_chains():
    w = SMALL["gqa_bf16_full"]
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    bad = lm["parents"].clone()
    bad[1, 5] = 7                                   # parent after its child
    k0 = att["k_cache"].clone()
    out_bad = gpu_attention(w, att, bad)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert "tree" in str(ei.value)
    att["k_cache"].copy_(k0)
    out_chain = gpu_attention(w, att)
    mv.sync_status()
    assert torch.equal(out_bad[1], out_chain[1])     # request 1 computed as a chain
    got = gpu_lmhead(w, dict(lm, parents=bad))
    with pytest.raises(mv.MtpError):
        mv.sync_status()
    chain = gpu_lmhead(w, dict(lm, parents=None))
    mv.sync_status()
    assert torch.equal(got["num_accepted"][1], chain["num_accepted"][1])


def test_tree_full_size_deepseek_v3():
    """DeepSeek-V3-shaped MLA step with full trees of 15 drafts (B=32, R=16,
    H=7168, V=129280): attention of the shortest-context request against the
    oracle, every request's acceptance against the planted targets, and one
    request's LM head and acceptance against the oracle."""
    w = synth.CFG1.with_(D=15, tree="full")
    torch.cuda.empty_cache()
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    parents = lm["parents"]
    out = gpu_attention(w, att, parents)
    gpu = gpu_lmhead(w, lm)
    mv.sync_status()
    b0 = int(torch.argmin(att["ctx_lens"]).item())
    ref = oracle_attention(w, att, [b0], parents)
    assert attention_excess(_out_np(w, out[b0:b0 + 1]), _ref_np(ref), w.dtype) <= 0.0
    par_h = parents.cpu().numpy()
    nodes = gpu["accepted_nodes"].cpu().numpy()
    outs = gpu["out_tokens"].cpu().numpy()
    for b in range(w.B):
        path, last = _planted_expectation(w, lm, par_h[b], b)
        n = len(path) - 1
        assert int(gpu["num_accepted"][b]) == n
        assert list(nodes[b, :n + 1]) == path and (nodes[b, n + 1:] == -1).all()
        assert outs[b, n] == last
    ref_lm = oracle_lmhead(w, lm, [b0])
    assert compare_accept(gpu, ref_lm, [b0]) == 0
    del att, lm, out, gpu
    torch.cuda.empty_cache()


def test_tree_noalloc_matches_workspace_path():
    w = SMALL["gqa_bf16_full"]
    lm = synth.make_lmhead_inputs(w, DEV)
    ref = gpu_lmhead(w, lm)
    out = torch.full((w.B, w.R), -9, dtype=torch.int32, device=DEV)
    n = torch.full((w.B,), -9, dtype=torch.int32, device=DEV)
    tie = torch.full((w.B,), 255, dtype=torch.uint8, device=DEV)
    nodes = torch.full((w.B, w.R), -9, dtype=torch.int32, device=DEV)
    mv.mtp_verify_logits_accept_noalloc(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"], lm["temperature"],
                                        lm["q_draft"], lm["seed"], out, n, tie, parents=lm["parents"],
                                        accepted_nodes=nodes)
    mv.sync_status()
    assert torch.equal(out, ref["out_tokens"]) and torch.equal(n, ref["num_accepted"])
    assert torch.equal(nodes, ref["accepted_nodes"])


def test_tree_single_node_and_chain_shaped_trees():
    """Edge shapes: D = 0 (the root alone) and a tree that is a chain written
    with explicit parents, each against the oracle."""
    for w in (SMALL["gqa_bf16_full"].with_(D=0, tree="random", name="tree D=0"),
              SMALL["mha_bf16_d64_random"].with_(D=15, tree="full", name="full tree D=15 MHA")):
        att = synth.make_attention_inputs(w, DEV)
        lm = synth.make_lmhead_inputs(w, DEV)
        parents = lm["parents"]
        out = gpu_attention(w, att, parents)
        gpu = gpu_lmhead(w, lm)
        mv.sync_status()
        ref = oracle_attention(w, att, range(w.B), parents)
        assert attention_excess(_out_np(w, out), _ref_np(ref), w.dtype) <= 0.0
        assert compare_accept(gpu, oracle_lmhead(w, lm, range(w.B)), range(w.B)) == 0


@pytest.mark.parametrize("name,w", [
    # 16 nodes x 4 heads = 64 rows per KV head: the tcgen05 GQA kernel at head dim 128
    ("wide_two_parts", synth.CFG3.with_(name="tree GQA 64 rows", B=40, D=15, Hq=32, Hkv=8, ctx=(600, 900), H=128,
                                        V=3001, sampling="none", tree="full", stream=46)),
    # the same at head dim 64, on mma.sync: 4 row warps per CTA, the 8-consumer form with 2 key parts
    ("wide_two_parts_d64", synth.CFG3.with_(name="tree GQA 64 rows d64", B=80, D=15, Hq=32, Hkv=8, d_qk=64, d_v=64,
                                            ctx=(600, 900), H=128, V=3001, sampling="none", tree="full",
                                            stream=48)),
    # 2 row warps per CTA (8 nodes x 4 heads): key parts on 7 consumers
    ("two_row_warps", synth.CFG3.with_(name="tree GQA 32 rows", B=80, D=7, Hq=32, Hkv=8, ctx=(800, 1000), H=128,
                                       V=3001, sampling="none", tree="random", stream=47)),
])
def test_tree_gqa_key_parts_all_requests(name, w):
    """Tree attention on grids large enough that spare warps split the tiles
    of each CTA, every request against the oracle (run in threads)."""
    import concurrent.futures as cf
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    parents = lm["parents"]
    out = gpu_attention(w, att, parents)
    mv.sync_status()
    with cf.ThreadPoolExecutor(8) as ex:
        refs = list(ex.map(lambda b: oracle_attention(w, att, [b], parents), range(w.B)))
    ref = np.concatenate(refs)
    assert attention_excess(_out_np(w, out), _ref_np(ref), w.dtype) <= 0.0
