"""The library's calls captured in a CUDA graph and replayed give the same
results as eager calls, bit for bit: a greedy MLA step, a sampling GQA step
with split keys, a relaxed step and a tree step with the KV compaction. (The
benchmark and serving loops replay the step as one graph.)"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402

DEV = torch.device("cuda:0")

CASES = {
    "mla_greedy": synth.CFG1.with_(name="graph MLA", B=4, Hq=32, ctx=(60, 500), H=128, V=3001, stream=51),
    "gqa_sampling_split": synth.CFG2.with_(name="graph GQA sampling", B=3, D=3, Hq=16, Hkv=2, ctx=(900, 1500),
                                           H=128, V=2049, stream=52),
    "relaxed": synth.CFG3.with_(name="graph relaxed", B=8, D=3, Hq=8, Hkv=2, ctx=(64, 300), H=128, V=2500,
                                relaxed="half", sampling="half", relaxed_topk=4, relaxed_delta=0.3, stream=53),
    "tree": synth.CFG3.with_(name="graph tree", B=4, D=7, Hq=8, Hkv=2, ctx=(64, 300), H=128, V=2500,
                             sampling="none", tree="random", stream=54),
}


def _step(w, att, lm, bufs, stream):
    """One verify step: attention (append), LM head + acceptance, tree
    compaction when the drafts form trees, rollback."""
    parents = lm.get("parents")
    with torch.cuda.stream(stream):
        bufs["table"].copy_(att["block_table"])
        bufs["seq"].copy_(att["ctx_lens"])
        bufs["free_count"].zero_()
        mv.mtp_verify_attention(att["q"], att["k_new"], att["v_new"], att["k_cache"], att["v_cache"],
                                att["block_table"], att["ctx_lens"], bufs["out"], sm_scale=w.sm_scale,
                                parents=parents, stream=stream)
        mv.mtp_verify_logits_accept(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"], lm["temperature"],
                                    lm["q_draft"], lm["seed"], bufs["tok"], bufs["n"], bufs["tie"],
                                    relaxed_topk=lm.get("relaxed_topk", 0), relaxed_delta=lm.get("relaxed_delta", 0.0),
                                    parents=parents, accepted_nodes=bufs["nodes"], stream=stream)
        if parents is not None:
            mv.mtp_tree_kv_compact(att["k_cache"], att["v_cache"], att["block_table"], att["ctx_lens"],
                                   bufs["nodes"], bufs["n"], stream=stream)
        mv.kv_rollback(bufs["table"], bufs["seq"], bufs["n"], bufs["free_list"], bufs["free_count"], D=w.D,
                       stream=stream)


def _buffers(w):
    return dict(out=torch.empty((w.B, w.R, w.Hq, w.d_v), dtype=w.torch_dtype, device=DEV),
                tok=torch.empty((w.B, w.R), dtype=torch.int32, device=DEV),
                n=torch.empty(w.B, dtype=torch.int32, device=DEV),
                tie=torch.empty(w.B, dtype=torch.uint8, device=DEV),
                nodes=torch.empty((w.B, w.R), dtype=torch.int32, device=DEV),
                table=torch.empty((w.B, w.max_blocks), dtype=torch.int32, device=DEV),
                seq=torch.empty(w.B, dtype=torch.int32, device=DEV),
                free_list=torch.full((w.B * 2 + 8,), -1, dtype=torch.int32, device=DEV),
                free_count=torch.zeros(1, dtype=torch.int32, device=DEV))


@pytest.mark.parametrize("name", list(CASES))
def test_graph_replay_equals_eager(name):
    w = CASES[name]
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    k0 = att["k_cache"].clone()
    v0 = None if att["v_cache"] is None else att["v_cache"].clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    eager = _buffers(w)
    _step(w, att, lm, eager, stream)            # also the first run of every call on the device
    stream.synchronize()
    mv.sync_status()
    k_eager = att["k_cache"].clone()
    replay = _buffers(w)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _step(w, att, lm, replay, stream)
    for _ in range(2):                          # replays start from the same cache state as the eager run
        att["k_cache"].copy_(k0)
        if v0 is not None:
            att["v_cache"].copy_(v0)
        g.replay()
    torch.cuda.synchronize()
    mv.sync_status()
    for k in ("out", "tok", "n", "tie", "table", "seq", "free_list", "free_count"):
        assert torch.equal(eager[k], replay[k]), k
    if lm.get("parents") is not None:
        assert torch.equal(eager["nodes"], replay["nodes"])
    assert torch.equal(att["k_cache"], k_eager)


@pytest.mark.parametrize("graph", [False, True])
def test_q_copy_overlapping_the_lm_head_matches_resident_q(graph):
    """q_ready_event: the draft distributions still crossing from pinned host
    memory on another stream when the call is made (the library waits for
    them only after launching the LM-head GEMM), eagerly and inside a graph
    capture, give the same tokens, counts and flags as q already resident."""
    w = synth.CFG2.with_(name="q overlap", B=6, D=3, Hq=16, Hkv=2, ctx=(64, 200), H=256, V=5003, stream=55)
    lm = synth.make_lmhead_inputs(w, DEV)

    def outs():
        return dict(tok=torch.full((w.B, w.R), -9, dtype=torch.int32, device=DEV),
                    n=torch.full((w.B,), -9, dtype=torch.int32, device=DEV),
                    tie=torch.full((w.B,), 255, dtype=torch.uint8, device=DEV))

    ref = outs()
    mv.mtp_verify_logits_accept(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"], lm["temperature"],
                                lm["q_draft"], lm["seed"], ref["tok"], ref["n"], ref["tie"])
    torch.cuda.synchronize()
    q_host = lm["q_draft"].cpu().pin_memory()
    q_dev = torch.zeros_like(lm["q_draft"])
    got = outs()
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()

    def step():
        side.wait_stream(main)
        with torch.cuda.stream(side):
            q_dev.copy_(q_host, non_blocking=True)
            ev.record(side)
        mv.mtp_verify_logits_accept(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"], lm["temperature"],
                                    q_dev, lm["seed"], got["tok"], got["n"], got["tie"], stream=main,
                                    q_ready_event=ev)
        main.wait_stream(side)

    if graph:
        g = torch.cuda.CUDAGraph()
        main.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=main):
            step()
        q_dev.zero_()
        torch.cuda.synchronize()
        g.replay()
    else:
        main.wait_stream(torch.cuda.current_stream())
        step()
    torch.cuda.synchronize()
    mv.sync_status()
    assert (lm["mode"] == 1).all()
    for k in ("tok", "n", "tie"):
        assert torch.equal(got[k], ref[k]), k
