"""Helpers for the GPU parity tests: run the library's three calls on a
workload, and run the CPU oracle on all or a sample of its requests."""
import numpy as np
import torch

import oracle
from oracle import requests as oracle_requests
import mtp_speculative_decoding_verify_gb300 as mv
from mtp_speculative_decoding_verify_gb300 import synth

BLOCK = 64
A = synth.as_oracle_array

# Tolerances (max-abs). Logits: 1e-4 for fp32 and 2e-2 for bf16. Attention
# outputs: 1e-2 (bf16) and 1e-4 (fp32) against the oracle's exact (float64,
# unrounded) result, plus half a unit in the last place of the GPU's output
# value: the GPU rounds its fp32 result once to the output dtype, and that
# last rounding alone moves a bf16 value by up to 2^-9..2^-8 of its
# magnitude (0.0078 just below 4, 0.0156 just below 8). fp32 accumulation
# over at most a few thousand keys stays ~1e-6 from the exact result.
# Log-sum-exp: 1e-5 relative.
TOL_LOGITS = {"f32": 1e-4, "bf16": 2e-2}
TOL_ATTN = {"f32": 1e-4, "bf16": 1e-2}
MANT_BITS = {"f32": 24, "bf16": 8}
TOL_LSE_REL = 1e-5


def half_ulp(x, dtype):
    """Half a unit in the last place of |x| in `dtype` (float64 array)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - MANT_BITS[dtype]).astype(np.int64))


def attention_excess(got, exact, dtype):
    """Largest |got - exact| beyond TOL_ATTN + half an ulp of got (<= 0 when within it)."""
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    allowed = TOL_ATTN[dtype] + half_ulp(got, dtype)
    return float((np.abs(got - exact) - allowed).max())


def attention_over_plain(got, exact, dtype):
    """(count, fraction) of elements whose error exceeds the plain TOL_ATTN bound."""
    d = np.abs(np.asarray(got, np.float64) - np.asarray(exact, np.float64))
    n = int((d > TOL_ATTN[dtype]).sum())
    return n, n / max(1, d.size)


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


request_pages = oracle_requests.request_pages


def oracle_attention(w, att, reqs, parents=None, return_cache=False, exact=True):
    """Oracle attention of the given requests: the exact float64 result by
    default, the output rounded to the workload dtype with exact=False."""
    return oracle_requests.attention(w, att, reqs, parents, return_cache=return_cache, exact=exact)


oracle_lmhead = oracle_requests.lmhead


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
    """Properties that hold for every request at any size (chains; for tree
    drafts the emitted prefix is the accepted path's drafts)."""
    tok = lm["tokens"].cpu().numpy()
    out = gpu["out_tokens"].cpu().numpy()
    n = gpu["num_accepted"].cpu().numpy()
    amax = gpu["argmax"].cpu().numpy()
    mode = lm["mode"].cpu().numpy()
    temp = lm["temperature"].cpu().numpy()
    assert ((n >= 0) & (n <= w.D)).all()
    if lm.get("parents") is not None:
        nodes = gpu["accepted_nodes"].cpu().numpy()
        par = lm["parents"].cpu().numpy()
        for b in range(w.B):
            k = int(n[b])
            path = nodes[b, :k + 1]
            assert path[0] == 0 and (nodes[b, k + 1:] == -1).all()
            assert all(par[b, path[i + 1]] == path[i] for i in range(k))
            assert (out[b, :k] == tok[b, path[1:]]).all() and (out[b, k + 1:] == -1).all()
            assert all(amax[b, path[i]] == tok[b, path[i + 1]] for i in range(k))   # greedy per edge
            assert out[b, k] == amax[b, path[k]]
        return
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
