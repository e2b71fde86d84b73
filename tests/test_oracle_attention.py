"""Pins for the oracle's verify attention (with KV append).

  * brute force: every row equals textbook single-query attention over the
    context keys plus verify keys 0..j, computed from a dense copy of the
    sequence (no paging);
  * the causal chain of the K=3 walkthrough table: a later verify token's
    K/V never reaches an earlier row, an earlier one always reaches later rows;
  * the append lands in slots ctx..ctx+D and touches nothing else;
  * special cases: absorbed MLA equals single-KV-head attention whose values
    are the first d_v latent entries; GQA equals MHA with repeated KV heads.
"""
import numpy as np
import pytest
import torch

BLOCK = 64


def _bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _from_bf16(a):
    return torch.tensor(a.view(np.int16)).view(torch.bfloat16).float().numpy()


def _case(rng, B, D, Hq, Hkv, d_qk, d_v, ctx, is_mla=False, spare=3):
    R = D + 1
    need = [(c + R + BLOCK - 1) // BLOCK for c in ctx]
    nb = sum(need) + spare
    perm = rng.permutation(nb).astype(np.int32)
    max_blocks = max(need) + 1
    table = np.full((B, max_blocks), -1, np.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    kv_h = 1 if is_mla else Hkv
    k_cache = rng.standard_normal((nb, BLOCK, kv_h, d_qk)).astype(np.float32)
    v_cache = None if is_mla else rng.standard_normal((nb, BLOCK, kv_h, d_v)).astype(np.float32)
    q = rng.standard_normal((B, R, Hq, d_qk)).astype(np.float32)
    k_new = rng.standard_normal((B, R, kv_h, d_qk)).astype(np.float32)
    v_new = None if is_mla else rng.standard_normal((B, R, kv_h, d_v)).astype(np.float32)
    if is_mla:
        k_new = k_new.reshape(B, R, d_qk)
    return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache, block_table=table,
                ctx_lens=np.array(ctx, np.int32))


def _run(orc, c, D, Hq, Hkv, d_qk, d_v, is_mla=False, scale=None):
    kc = c["k_cache"].copy()
    vc = None if c["v_cache"] is None else c["v_cache"].copy()
    out = orc.verify_attention(c["q"], c["k_new"], c["v_new"], kc, vc, c["block_table"], c["ctx_lens"], D=D,
                               Hq=Hq, Hkv=1 if is_mla else Hkv, d_qk=d_qk, d_v=d_v, block_size=BLOCK,
                               is_mla=is_mla, sm_scale=scale if scale is not None else 1 / np.sqrt(d_qk))
    return out, kc, vc


def _dense_sequence(c, b, kvh, D, is_mla, d_v):
    """Context keys/values gathered through the block table, then the verify tokens'."""
    ctx = int(c["ctx_lens"][b])
    tbl = c["block_table"][b]
    ks, vs = [], []
    for t in range(ctx):
        blk, off = tbl[t // BLOCK], t % BLOCK
        ks.append(c["k_cache"][blk, off, kvh].astype(np.float64))
        vs.append(c["k_cache"][blk, off, 0, :d_v] if is_mla else c["v_cache"][blk, off, kvh])
    for j in range(D + 1):
        kn = c["k_new"][b, j] if is_mla else c["k_new"][b, j, kvh]
        ks.append(kn.astype(np.float64))
        vs.append(kn[:d_v] if is_mla else c["v_new"][b, j, kvh])
    return np.array(ks), np.array(vs, np.float64)


def _textbook(q, K, V, scale):
    s = K @ q.astype(np.float64) * scale
    p = np.exp(s - s.max())
    return (p / p.sum()) @ V


@pytest.mark.parametrize("Hq,Hkv,ctx", [(4, 4, [5, 70, 130]), (8, 2, [0, 63, 64, 200])])
def test_rows_equal_single_query_attention(orc, Hq, Hkv, ctx):
    rng = np.random.default_rng(10 + Hq)
    D, d = 3, 16
    B = len(ctx)
    c = _case(rng, B, D, Hq, Hkv, d, d, ctx)
    out, _, _ = _run(orc, c, D, Hq, Hkv, d, d)
    scale = 1 / np.sqrt(d)
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            K, V = _dense_sequence(c, b, kvh, D, False, d)
            for j in range(D + 1):
                L = ctx[b] + j + 1
                ref = _textbook(c["q"][b, j, h], K[:L], V[:L], scale)
                np.testing.assert_allclose(out[b, j, h], ref, rtol=1e-5, atol=1e-6)


def test_mla_rows_equal_single_query_attention(orc):
    rng = np.random.default_rng(21)
    D, Hq, d_qk, d_v, ctx = 2, 6, 24, 16, [40, 129]
    c = _case(rng, len(ctx), D, Hq, 1, d_qk, d_v, ctx, is_mla=True)
    out, _, _ = _run(orc, c, D, Hq, 1, d_qk, d_v, is_mla=True, scale=0.17)
    for b in range(len(ctx)):
        K, V = _dense_sequence(c, b, 0, D, True, d_v)
        for j in range(D + 1):
            L = ctx[b] + j + 1
            for h in range(Hq):
                np.testing.assert_allclose(out[b, j, h], _textbook(c["q"][b, j, h], K[:L], V[:L], 0.17),
                                           rtol=1e-5, atol=1e-6)


def test_chain_causality_k3_walkthrough(orc):
    """Verify token j's K/V reaches rows j..D and never rows < j (the table of
    the K=3 walkthrough: T12 sees the freshly added K11, T11 does not see K12)."""
    rng = np.random.default_rng(30)
    D, Hq, d = 3, 2, 8
    c = _case(rng, 1, D, Hq, Hq, d, d, [10])
    base, _, _ = _run(orc, c, D, Hq, Hq, d, d)
    for jp in range(D + 1):
        c2 = {k: (None if v is None else v.copy()) for k, v in c.items()}
        c2["k_new"][0, jp] += 3.0
        c2["v_new"][0, jp] += 3.0
        out, _, _ = _run(orc, c2, D, Hq, Hq, d, d)
        for j in range(D + 1):
            changed = not np.allclose(out[0, j], base[0, j])
            assert changed == (j >= jp), (jp, j)


def test_append_writes_only_verify_slots(orc):
    rng = np.random.default_rng(31)
    D, H, d, ctx = 4, 2, 8, [62, 0, 127]
    c = _case(rng, len(ctx), D, H, H, d, d, ctx)
    _, kc, vc = _run(orc, c, D, H, H, d, d)
    touched = np.zeros(kc.shape[:2], bool)
    for b, cl in enumerate(ctx):
        for j in range(D + 1):
            s = cl + j
            blk, off = c["block_table"][b, s // BLOCK], s % BLOCK
            touched[blk, off] = True
            np.testing.assert_array_equal(kc[blk, off], c["k_new"][b, j])
            np.testing.assert_array_equal(vc[blk, off], c["v_new"][b, j])
    np.testing.assert_array_equal(kc[~touched], c["k_cache"][~touched])
    np.testing.assert_array_equal(vc[~touched], c["v_cache"][~touched])


def test_mla_equals_single_head_with_latent_values(orc):
    rng = np.random.default_rng(32)
    D, Hq, d_qk, d_v, ctx = 1, 4, 20, 12, [33, 90]
    c = _case(rng, len(ctx), D, Hq, 1, d_qk, d_v, ctx, is_mla=True)
    out_mla, _, _ = _run(orc, c, D, Hq, 1, d_qk, d_v, is_mla=True)
    g = dict(c)
    g["v_cache"] = np.ascontiguousarray(c["k_cache"][..., :d_v])
    g["k_new"] = c["k_new"].reshape(len(ctx), D + 1, 1, d_qk)
    g["v_new"] = np.ascontiguousarray(g["k_new"][..., :d_v])
    out_gqa, _, _ = _run(orc, g, D, Hq, 1, d_qk, d_v)
    np.testing.assert_array_equal(out_mla, out_gqa)


def test_gqa_equals_mha_with_repeated_heads(orc):
    rng = np.random.default_rng(33)
    D, Hq, Hkv, d, ctx = 2, 6, 2, 8, [20, 70]
    c = _case(rng, len(ctx), D, Hq, Hkv, d, d, ctx)
    out_gqa, _, _ = _run(orc, c, D, Hq, Hkv, d, d)
    g = Hq // Hkv
    m = dict(c)
    m["k_cache"] = np.ascontiguousarray(np.repeat(c["k_cache"], g, axis=2))
    m["v_cache"] = np.ascontiguousarray(np.repeat(c["v_cache"], g, axis=2))
    m["k_new"] = np.ascontiguousarray(np.repeat(c["k_new"], g, axis=2))
    m["v_new"] = np.ascontiguousarray(np.repeat(c["v_new"], g, axis=2))
    out_mha, _, _ = _run(orc, m, D, Hq, Hq, d, d)
    np.testing.assert_array_equal(out_gqa, out_mha)


def test_bf16_output_is_rounded_double_result(orc):
    rng = np.random.default_rng(34)
    D, H, d, ctx = 2, 2, 16, [50]
    c = _case(rng, 1, D, H, H, d, d, ctx)
    cb = {k: (None if v is None or k in ("block_table", "ctx_lens") else _bf16(v)) for k, v in c.items()}
    cb["block_table"], cb["ctx_lens"] = c["block_table"], c["ctx_lens"]
    out, _, _ = _run(orc, cb, D, H, H, d, d)
    cf = {k: (v if k in ("block_table", "ctx_lens") else _from_bf16(v)) for k, v in cb.items()}
    ref, _, _ = _run(orc, cf, D, H, H, d, d)
    np.testing.assert_array_equal(out, _bf16(ref))


def test_bad_block_id_is_reported(orc):
    rng = np.random.default_rng(35)
    c = _case(rng, 1, 1, 2, 2, 8, 8, [10])
    c["block_table"][0, 0] = 10_000
    with pytest.raises(ValueError):
        _run(orc, c, 1, 2, 2, 8, 8)
