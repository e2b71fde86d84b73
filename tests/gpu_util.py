"""Helpers for the GPU parity tests: run the library's three calls on a
workload, and run the CPU oracle on all or a sample of its requests."""
import numpy as np
import torch

import oracle
import mtp_speculative_decoding_verify_gb300 as mv
from mtp_speculative_decoding_verify_gb300 import synth

BLOCK = 64
A = synth.as_oracle_array

# Tolerances (max-abs): logits 1e-4 for fp32 and 2e-2 for bf16, attention
# outputs 1e-2 for bf16 or one bf16 unit in the last place of the exact value,
# whichever is larger (both sides round the output to bf16 once, from fp32 on
# the GPU and from fp64 in the oracle, so they can land on neighbouring bf16
# values; above magnitude 2 that step, 2^-7 |x| at most, exceeds 1e-2); fp32
# attention 1e-4 (fp32 accumulation over at most a few thousand keys stays
# ~1e-6 from the exact result); log-sum-exp 1e-5 relative.
TOL_LOGITS = {"f32": 1e-4, "bf16": 2e-2}
TOL_ATTN = {"f32": 1e-4, "bf16": 1e-2}
ULP_REL_ATTN = {"f32": 0.0, "bf16": 2.0 ** -7}
TOL_LSE_REL = 1e-5


def attention_excess(got, ref, dtype):
    """Largest |got - ref| beyond the attention tolerance (<= 0 when within it)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    allowed = np.maximum(TOL_ATTN[dtype], ULP_REL_ATTN[dtype] * np.abs(ref))
    return float((np.abs(got - ref) - allowed).max())


def gpu_attention(w, att, parents=None):
    out = torch.empty((w.B, w.R, w.Hq, w.d_v), dtype=w.torch_dtype, device=att["q"].device)
    mv.mtp_verify_attention(att["q"], att["k_new"], att["v_new"], att["k_cache"], att["v_cache"],
                            att["block_table"], att["ctx_lens"], out, sm_scale=w.sm_scale, parents=parents)
    return out


def gpu_lmhead(w, lm, debug_logits=False):
    dev = lm["hidden"].device
    res = dict(out_tokens=torch.full((w.B, w.R), -9, dtype=torch.int32, device=dev),
               num_accepted=torch.full((w.B,), -9, dtype=torch.int32, device=dev),
               tie_flags=torch.full((w.B,), 255, dtype=torch.uint8, device=dev),
               lse=torch.empty((w.B, w.R), dtype=torch.float32, device=dev),
               argmax=torch.empty((w.B, w.R), dtype=torch.int32, device=dev),
               accepted_nodes=torch.full((w.B, w.R), -9, dtype=torch.int32, device=dev))
    if debug_logits:
        res["logits"] = torch.empty((w.M, w.V), dtype=torch.float32, device=dev)
    mv.mtp_verify_logits_accept(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"], lm["temperature"],
                                lm["q_draft"], lm["seed"], res["out_tokens"], res["num_accepted"], res["tie_flags"],
                                res["lse"], res["argmax"], res.get("logits"), relaxed_topk=lm.get("relaxed_topk", 0),
                                relaxed_delta=lm.get("relaxed_delta", 0.0), parents=lm.get("parents"),
                                accepted_nodes=res["accepted_nodes"])
    return res


def gpu_rollback(w, block_table, ctx_lens, num_accepted, capacity=None):
    dev = block_table.device
    table = block_table.clone()
    seq = ctx_lens.clone()
    cap = capacity if capacity is not None else w.B * (w.D // BLOCK + 2) + 8
    free_list = torch.full((cap,), -1, dtype=torch.int32, device=dev)
    free_count = torch.zeros(1, dtype=torch.int32, device=dev)
    mv.kv_rollback(table, seq, num_accepted, free_list, free_count, D=w.D)
    return table, seq, free_list, free_count


def request_pages(w, table_h, ctx_h, b):
    n = (int(ctx_h[b]) + w.R + BLOCK - 1) // BLOCK
    return table_h[b, :n]


def oracle_attention(w, att, reqs, parents=None, return_cache=False):
    """Oracle output [len(reqs), R, Hq, d_v] for the given requests. Each
    request's pages are gathered from the (device) cache into a compact
    host cache; the oracle re-does the append into it. return_cache: also
    return that host cache (k, v) and its block table."""
    table_h = A(att["block_table"])
    ctx_h = A(att["ctx_lens"])
    pages = [request_pages(w, table_h, ctx_h, b) for b in reqs]
    all_pages = torch.from_numpy(np.concatenate(pages).astype(np.int64)).to(att["k_cache"].device)
    kc = A(att["k_cache"].index_select(0, all_pages)).copy()
    vc = None if w.is_mla else A(att["v_cache"].index_select(0, all_pages)).copy()
    sub_table = np.full((len(reqs), w.max_blocks), -1, np.int32)
    pos = 0
    for i, p in enumerate(pages):
        sub_table[i, :len(p)] = np.arange(pos, pos + len(p))
        pos += len(p)
    idx = torch.tensor(list(reqs), dtype=torch.int64, device=att["q"].device)
    sel = lambda t: None if t is None else A(t.index_select(0, idx))
    out = oracle.verify_attention(sel(att["q"]), sel(att["k_new"]), sel(att["v_new"]), kc, vc, sub_table,
                                  ctx_h[list(reqs)], D=w.D, Hq=w.Hq, Hkv=1 if w.is_mla else w.Hkv, d_qk=w.d_qk,
                                  d_v=w.d_v, block_size=BLOCK, is_mla=w.is_mla, sm_scale=w.sm_scale,
                                  parents=None if parents is None else A(parents.index_select(0, idx)))
    return (out, kc, vc, sub_table) if return_cache else out


def oracle_lmhead(w, lm, reqs, W_host=None, want_logits=False):
    reqs = list(reqs)
    dev = lm["hidden"].device
    rows = torch.tensor([b * w.R + j for b in reqs for j in range(w.R)], dtype=torch.int64, device=dev)
    idx = torch.tensor(reqs, dtype=torch.int64, device=dev)
    W = W_host if W_host is not None else A(lm["lm_head"])
    q = None if lm["q_draft"] is None else A(lm["q_draft"].index_select(0, idx))
    par = lm.get("parents")
    return oracle.lmhead_accept(A(lm["hidden"].index_select(0, rows)), W, A(lm["tokens"].index_select(0, idx)),
                                A(lm["mode"].index_select(0, idx)), A(lm["temperature"].index_select(0, idx)), q,
                                lm["seed"], want_logits=want_logits, request_index=np.array(reqs, np.int32),
                                relaxed_topk=lm.get("relaxed_topk", 0), relaxed_delta=lm.get("relaxed_delta", 0.0),
                                parents=None if par is None else A(par.index_select(0, idx)))


def compare_accept(gpu, ref, reqs):
    """Bit-exact tokens and accept counts for every request neither side
    flagged as a near-tie; flagged requests only need valid outputs.
    Returns the number of flagged requests."""
    g_tok = gpu["out_tokens"].cpu().numpy()
    g_n = gpu["num_accepted"].cpu().numpy()
    g_tie = gpu["tie_flags"].cpu().numpy()
    flagged = 0
    for i, b in enumerate(reqs):
        if g_tie[b] or ref["tie_flags"][i]:
            flagged += 1
            continue
        assert g_n[b] == ref["num_accepted"][i], (b, g_n[b], ref["num_accepted"][i])
        assert (g_tok[b] == ref["out_tokens"][i]).all(), (b, g_tok[b], ref["out_tokens"][i])
        if "accepted_nodes" in gpu and "accepted_nodes" in ref:
            g_nodes = gpu["accepted_nodes"][b].cpu().numpy()
            assert (g_nodes == ref["accepted_nodes"][i]).all(), (b, g_nodes, ref["accepted_nodes"][i])
    return flagged


def check_invariants(w, lm, gpu):
    """Properties that hold for every request at any size."""
    tok = lm["tokens"].cpu().numpy()
    out = gpu["out_tokens"].cpu().numpy()
    n = gpu["num_accepted"].cpu().numpy()
    amax = gpu["argmax"].cpu().numpy()
    mode = lm["mode"].cpu().numpy()
    temp = lm["temperature"].cpu().numpy()
    assert ((n >= 0) & (n <= w.D)).all()
    for b in range(w.B):
        k = int(n[b])
        assert (out[b, :k] == tok[b, 1:k + 1]).all()
        assert 0 <= out[b, k] < w.V
        assert (out[b, k + 1:] == -1).all()
        if mode[b] == 2:
            assert out[b, k] == amax[b, k]
        elif not (mode[b] == 1 and temp[b] > 0):
            assert all(amax[b, j] == tok[b, j + 1] for j in range(k))
            assert k == w.D or amax[b, k] != tok[b, k + 1]
            assert out[b, k] == amax[b, k]
