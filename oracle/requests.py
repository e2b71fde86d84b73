"""The oracle applied to whole requests of a synthetic workload (test
infrastructure only: the GPU parity tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline and reference legs use it).

A workload's tensors come from ``synth`` (possibly on a GPU); these helpers
gather the requests asked for, hand them to the oracle as numpy arrays and
return the oracle's results. They only move data: every step of the method is
the oracle's own C code.
"""
import numpy as np
import torch

from mtp_speculative_decoding_verify_gb300 import synth

from . import kv_rollback, lmhead_accept, tree_kv_compact, verify_attention

BLOCK = 64
A = synth.as_oracle_array


def request_pages(w, table_h, ctx_h, b):
    """Cache blocks that hold request b's context and verify slots."""
    n = (int(ctx_h[b]) + w.R + BLOCK - 1) // BLOCK
    return table_h[b, :n]


def attention(w, att, reqs, parents=None, return_cache=False, exact=False):
    """Oracle append + verify attention for the given requests.

    Returns out [len(reqs), R, Hq, d_v] rounded to the workload's dtype, or
    with ``exact`` the float64 result before that rounding. Each request's
    pages are gathered from the cache into a compact host cache; the oracle
    re-does the append into it. ``return_cache``: also return that host cache
    (k, v) and its block table."""
    reqs = list(reqs)
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
    idx = torch.tensor(reqs, dtype=torch.int64, device=att["q"].device)
    sel = lambda t: None if t is None else A(t.index_select(0, idx))  # noqa: E731
    res = verify_attention(sel(att["q"]), sel(att["k_new"]), sel(att["v_new"]), kc, vc, sub_table, ctx_h[reqs],
                           D=w.D, Hq=w.Hq, Hkv=1 if w.is_mla else w.Hkv, d_qk=w.d_qk, d_v=w.d_v,
                           block_size=BLOCK, is_mla=w.is_mla, sm_scale=w.sm_scale,
                           parents=None if parents is None else A(parents.index_select(0, idx)),
                           want_exact=exact)
    out = res[1] if exact else res
    return (out, kc, vc, sub_table) if return_cache else out


def lmhead(w, lm, reqs, W_host=None, want_logits=False):
    """Oracle LM head + row statistics + acceptance for the given requests
    (their Philox counters use their index in the batch)."""
    reqs = list(reqs)
    dev = lm["hidden"].device
    rows = torch.tensor([b * w.R + j for b in reqs for j in range(w.R)], dtype=torch.int64, device=dev)
    idx = torch.tensor(reqs, dtype=torch.int64, device=dev)
    W = W_host if W_host is not None else A(lm["lm_head"])
    q = None if lm["q_draft"] is None else A(lm["q_draft"].index_select(0, idx))
    par = lm.get("parents")
    return lmhead_accept(A(lm["hidden"].index_select(0, rows)), W, A(lm["tokens"].index_select(0, idx)),
                         A(lm["mode"].index_select(0, idx)), A(lm["temperature"].index_select(0, idx)), q,
                         lm["seed"], want_logits=want_logits, request_index=np.array(reqs, np.int32),
                         relaxed_topk=lm.get("relaxed_topk", 0), relaxed_delta=lm.get("relaxed_delta", 0.0),
                         parents=None if par is None else A(par.index_select(0, idx)))


def whole_request(w, att, lm, W, table, ctx, b):
    """The oracle's whole verify step for request b: append + attention, LM
    head + acceptance, KV compaction (tree drafts) and rollback."""
    parents = lm.get("parents")
    _, kc, vc, sub_table = attention(w, att, [b], parents, return_cache=True)
    r = lmhead(w, lm, [b], W)
    if parents is not None:
        tree_kv_compact(kc, vc, sub_table, ctx[b:b + 1], r["accepted_nodes"], r["num_accepted"], D=w.D,
                        Hkv=1 if w.is_mla else w.Hkv, d_qk=w.d_qk, d_v=w.d_v, block_size=BLOCK, is_mla=w.is_mla)
    fl = np.zeros(w.D // BLOCK + 4, np.int32)
    fc = np.zeros(1, np.int32)
    kv_rollback(table[b:b + 1].copy(), ctx[b:b + 1].copy(), r["num_accepted"], fl, fc, D=w.D, block_size=BLOCK)
    return r


def draft_request(w, inp, W, b):
    """The oracle's D greedy draft steps of request b (the argmax of each call's row)."""
    toks = np.zeros((1, 1), np.int32)
    mode = np.zeros(1, np.uint8)
    out = []
    for k in range(w.D):
        h = A(inp["hidden"][k, b:b + 1])
        r = lmhead_accept(h, W, toks, mode, None, None, 0)
        out.append(int(r["argmax"][0, 0]))
    return out
