"""Python access to the CPU oracle (test infrastructure only).

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg use this module. It takes and returns numpy arrays; bf16 tensors
travel as their uint16 bit patterns.
"""
import ctypes

import numpy as np

from . import build as _build

F32, BF16 = 0, 1

_lib = None


def lib():
    """Load (building first if needed) oracle/_build/liboracle.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, u32, u64, f32 = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float
        L.oracle_philox4x32_10.argtypes = [P, P, P]
        L.oracle_philox4x32_10.restype = None
        L.oracle_verify_attention.argtypes = [i32] * 9 + [i32, f32, i32] + [P] * 10
        L.oracle_verify_attention.restype = i32
        L.oracle_lmhead_accept.argtypes = [i32] * 5 + [P] * 6 + [u64] + [P] * 7 + [i32, ctypes.c_float, P, P]
        L.oracle_lmhead_accept.restype = i32
        L.oracle_kv_rollback.argtypes = [i32] * 4 + [P] * 5
        L.oracle_kv_rollback.restype = i32
        L.oracle_tree_kv_compact.argtypes = [i32] * 10 + [P] * 6
        L.oracle_tree_kv_compact.restype = i32
        L.oracle_accept_prefix.argtypes = [i32, P, P, P, P]
        L.oracle_relaxed_accept.argtypes = [i32, P, ctypes.c_float, i32, i32, ctypes.c_float, P]
        L.oracle_relaxed_accept.restype = i32
        L.oracle_accept_prefix.restype = i32
        L.oracle_race.argtypes = [i32, P, P, P]
        L.oracle_race.restype = i32
        L.oracle_accept_uniform.argtypes = [u64, u32, u32]
        L.oracle_accept_uniform.restype = f32
        L.oracle_race_exponential.argtypes = [u64, u32, u32, u32, u32]
        L.oracle_race_exponential.restype = f32
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _storage(a):
    """Contiguous storage for a float32 or bf16 (uint16 bits) tensor, with its dtype code."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError("oracle tensors are float32 or bf16 bit patterns (uint16), got %s" % a.dtype)


def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def accept_uniform(seed, b, j):
    return lib().oracle_accept_uniform(seed, b, j)


def race_exponential(seed, b, j, v, tag):
    return lib().oracle_race_exponential(seed, b, j, v, tag)


def accept_prefix(p, q, U):
    p, q, U = _c(p, np.float32), _c(q, np.float32), _c(U, np.float32)
    tie = np.zeros(1, np.uint8)
    n = lib().oracle_accept_prefix(len(p), _ptr(p), _ptr(q), _ptr(U), _ptr(tie))
    return n, int(tie[0])


def race(w, E):
    w, E = _c(w, np.float32), _c(E, np.float32)
    tie = np.zeros(1, np.uint8)
    v = lib().oracle_race(len(w), _ptr(w), _ptr(E), _ptr(tie))
    return v, int(tie[0])


def verify_attention(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, *, D, Hq, Hkv,
                     d_qk, d_v, block_size, is_mla, sm_scale, parents=None, want_exact=False):
    """Append + verify attention. k_cache / v_cache are updated in place; returns out
    (rounded to the input dtype), or (out, exact) with want_exact, exact being
    the float64 result before that rounding. parents [B, R] int32 (None:
    chains) gives tree drafts."""
    q, dt = _storage(q)
    k_new, _ = _storage(k_new)
    v_new = None if v_new is None else _storage(v_new)[0]
    assert k_cache.flags.c_contiguous and (v_cache is None or v_cache.flags.c_contiguous)
    bt = _c(block_table, np.int32)
    ctx = _c(ctx_lens, np.int32)
    B = ctx.shape[0]
    R = D + 1
    out = np.zeros((B, R, Hq, d_v), dtype=q.dtype)
    exact = np.zeros((B, R, Hq, d_v), dtype=np.float64) if want_exact else None
    num_blocks = k_cache.shape[0]
    rc = lib().oracle_verify_attention(B, D, Hq, Hkv, d_qk, d_v, block_size, bt.shape[1], num_blocks,
                                       int(is_mla), float(sm_scale), dt, _ptr(q), _ptr(k_new), _ptr(v_new),
                                       _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(ctx), _ptr(out),
                                       _ptr(None if parents is None else _c(parents, np.int32)), _ptr(exact))
    if rc != 0:
        raise ValueError("oracle_verify_attention returned %d" % rc)
    return (out, exact) if want_exact else out


def lmhead_accept(hidden, lm_head, tokens, mode, temperature, q_draft, seed, *, want_logits=False,
                  request_index=None, relaxed_topk=0, relaxed_delta=0.0, parents=None):
    """LM head + row statistics + acceptance. Returns a dict of numpy arrays
    (accepted_nodes: the accepted path's nodes, root first, then -1).
    parents [B, R] int32 (None: chains) gives tree drafts (greedy requests)."""
    hidden, dt = _storage(hidden)
    lm_head, dt2 = _storage(lm_head)
    assert dt == dt2
    tokens = _c(tokens, np.int32)
    B, R = tokens.shape
    D = R - 1
    V, H = lm_head.shape
    mode = _c(mode, np.uint8)
    temperature = None if temperature is None else _c(temperature, np.float32)
    q_draft = None if q_draft is None else _c(q_draft, np.float32)
    out_tokens = np.full((B, R), -7, np.int32)
    num_acc = np.full(B, -7, np.int32)
    ties = np.zeros(B, np.uint8)
    lse = np.zeros((B, R), np.float32)
    amax = np.zeros((B, R), np.int32)
    logits = np.zeros((B * R, V), np.float32) if want_logits else None
    rid = None if request_index is None else _c(request_index, np.int32)
    par = None if parents is None else _c(parents, np.int32)
    nodes = np.full((B, R), -7, np.int32)
    rc = lib().oracle_lmhead_accept(B, D, H, V, dt, _ptr(hidden), _ptr(lm_head), _ptr(tokens), _ptr(mode),
                                    _ptr(temperature), _ptr(q_draft), ctypes.c_uint64(seed), _ptr(rid), _ptr(out_tokens),
                                    _ptr(num_acc), _ptr(ties), _ptr(lse), _ptr(amax), _ptr(logits),
                                    int(relaxed_topk), ctypes.c_float(relaxed_delta), _ptr(par), _ptr(nodes))
    if rc != 0:
        raise ValueError("oracle_lmhead_accept returned %d" % rc)
    res = dict(out_tokens=out_tokens, num_accepted=num_acc, tie_flags=ties, lse=lse, argmax=amax,
               accepted_nodes=nodes)
    if want_logits:
        res["logits"] = logits
    return res


def kv_rollback(block_table, seq_lens, num_accepted, free_list, free_count, *, D, block_size):
    """In-place rollback on numpy int32 arrays; free_count is a 1-element int32 array."""
    for a in (block_table, seq_lens, free_list, free_count):
        assert a.dtype == np.int32 and a.flags.c_contiguous
    na = _c(num_accepted, np.int32)
    B, max_blocks = block_table.shape
    rc = lib().oracle_kv_rollback(B, D, block_size, max_blocks, _ptr(block_table), _ptr(seq_lens), _ptr(na),
                                  _ptr(free_list), _ptr(free_count))
    if rc != 0:
        raise ValueError("oracle_kv_rollback returned %d" % rc)


def tree_kv_compact(k_cache, v_cache, block_table, ctx_lens, accepted_nodes, num_accepted, *, D, Hkv, d_qk,
                    d_v, block_size, is_mla):
    """In place: the accepted path's K/V moved to slots ctx + 1 .. ctx + n (numpy caches)."""
    assert k_cache.flags.c_contiguous and (v_cache is None or v_cache.flags.c_contiguous)
    dt = {np.dtype(np.float32): F32, np.dtype(np.uint16): BF16}[k_cache.dtype]
    bt = _c(block_table, np.int32)
    ctx = _c(ctx_lens, np.int32)
    nodes = _c(accepted_nodes, np.int32)
    na = _c(num_accepted, np.int32)
    rc = lib().oracle_tree_kv_compact(ctx.shape[0], D, Hkv, d_qk, d_v, block_size, bt.shape[1], k_cache.shape[0],
                                      int(is_mla), dt, _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(ctx),
                                      _ptr(nodes), _ptr(na))
    if rc != 0:
        raise ValueError("oracle_tree_kv_compact returned %d" % rc)


def relaxed_accept(logits, lse, d, topk, delta):
    """Relaxed acceptance of one row: (accepted 0/1, tie flag byte)."""
    logits = _c(logits, np.float32)
    tie = np.zeros(1, np.uint8)
    r = lib().oracle_relaxed_accept(logits.size, _ptr(logits), ctypes.c_float(lse), int(d), int(topk),
                                    ctypes.c_float(delta), _ptr(tie))
    return int(r), int(tie[0])
