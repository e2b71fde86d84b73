"""Brute-force pin of the whole verify step: on a tiny one-layer model, greedy
speculative decoding driven by the oracle's attention, LM-head/accept and
rollback emits exactly the tokens that step-by-step greedy decoding emits.

Toy model (numpy, float64 with the same binary32 roundings the oracle
applies at its outputs): token + position embedding, one attention head, a
residual connection, and an LM head shared with the embedding table.
"""
import numpy as np
import pytest

BLOCK = 64


class Toy:
    def __init__(self, seed, V=32, H=16, d=16, max_pos=256):
        rng = np.random.default_rng(seed)
        self.V, self.H, self.d = V, H, d
        self.E = rng.standard_normal((V, H)).astype(np.float32)
        self.P = rng.standard_normal((max_pos, H)) * 0.5
        self.Wq = rng.standard_normal((H, d)) / np.sqrt(H)
        self.Wk = rng.standard_normal((H, d)) / np.sqrt(H)
        self.Wv = rng.standard_normal((H, d)) / np.sqrt(H)
        self.Wo = rng.standard_normal((d, H)) / np.sqrt(d)

    def embed(self, x, t):
        return self.E[x].astype(np.float64) + self.P[t]

    def qkv(self, x, t):
        e = self.embed(x, t)
        f32 = lambda a: a.astype(np.float32)
        return f32(e @ self.Wq), f32(e @ self.Wk), f32(e @ self.Wv)

    def hidden(self, x, t, attn_out_f32):
        return (self.embed(x, t) + attn_out_f32.astype(np.float64) @ self.Wo).astype(np.float32)


def step_by_step(toy, prompt, steps):
    seq = list(prompt)
    for _ in range(steps):
        t = len(seq) - 1
        K = np.array([toy.qkv(seq[s], s)[1] for s in range(t + 1)], np.float64)
        Vv = np.array([toy.qkv(seq[s], s)[2] for s in range(t + 1)], np.float64)
        q = toy.qkv(seq[t], t)[0].astype(np.float64)
        s = K @ q / np.sqrt(toy.d)
        p = np.exp(s - s.max())
        attn = ((p / p.sum()) @ Vv).astype(np.float32)
        h = toy.hidden(seq[t], t, attn)
        logits = (h.astype(np.float64) @ toy.E.astype(np.float64).T).astype(np.float32)
        seq.append(int(np.argmax(logits)))
    return seq[len(prompt):]


def speculative(orc, toy, prompt, steps, D, agreement, reference, seed):
    rng = np.random.default_rng(seed)
    nb = 16
    max_blocks = 8
    k_cache = np.zeros((nb, BLOCK, 1, toy.d), np.float32)
    v_cache = np.zeros((nb, BLOCK, 1, toy.d), np.float32)
    table = np.full((1, max_blocks), -1, np.int32)
    free = list(range(nb))
    # Prefill: every prompt token but the last goes into the cache.
    ctx = len(prompt) - 1
    for s in range(ctx):
        blk = s // BLOCK
        if table[0, blk] < 0:
            table[0, blk] = free.pop(0)
        _, k, v = toy.qkv(prompt[s], s)
        k_cache[table[0, blk], s % BLOCK, 0] = k
        v_cache[table[0, blk], s % BLOCK, 0] = v
    seq = list(prompt)
    emitted_total = []
    iters = 0
    while len(emitted_total) < steps:
        iters += 1
        pos = len(emitted_total)
        drafts = []
        for j in range(D):
            good = reference[pos + j] if pos + j < len(reference) else 0
            drafts.append(good if rng.random() < agreement else int(rng.integers(0, toy.V)))
        chain = [seq[-1]] + drafts
        for s in range(ctx, ctx + D + 1):           # the engine allocates blocks for the verify slots
            if table[0, s // BLOCK] < 0:
                table[0, s // BLOCK] = free.pop(0)
        qs, ks, vs = zip(*[toy.qkv(x, ctx + j) for j, x in enumerate(chain)])
        R = D + 1
        attn = orc.verify_attention(np.array(qs).reshape(1, R, 1, toy.d), np.array(ks).reshape(1, R, 1, toy.d),
                                    np.array(vs).reshape(1, R, 1, toy.d), k_cache, v_cache, table,
                                    np.array([ctx], np.int32), D=D, Hq=1, Hkv=1, d_qk=toy.d, d_v=toy.d,
                                    block_size=BLOCK, is_mla=False, sm_scale=1 / np.sqrt(toy.d))
        hid = np.array([toy.hidden(x, ctx + j, attn[0, j, 0]) for j, x in enumerate(chain)], np.float32)
        res = orc.lmhead_accept(hid, toy.E, np.array([chain], np.int32), np.zeros(1, np.uint8), None, None, 0)
        n = int(res["num_accepted"][0])
        new = res["out_tokens"][0, :n + 1].tolist()
        seq.extend(new)
        emitted_total.extend(new)
        seq_len = np.array([ctx], np.int32)
        fl = np.zeros(16, np.int32)
        fc = np.zeros(1, np.int32)
        orc.kv_rollback(table, seq_len, np.array([n], np.int32), fl, fc, D=D, block_size=BLOCK)
        free.extend(fl[:fc[0]].tolist())
        assert seq_len[0] == ctx + n + 1 == len(seq) - 1
        ctx = int(seq_len[0])
    return emitted_total[:steps], iters


@pytest.mark.parametrize("D,agreement", [(1, 0.9), (3, 0.7), (5, 0.5), (4, 0.0), (3, 1.0)])
def test_speculative_greedy_equals_step_by_step(orc, D, agreement):
    toy = Toy(seed=42)
    prompt = [3, 1, 4, 1, 5, 9, 2, 6]
    steps = 50
    ref = step_by_step(toy, prompt, steps + D + 1)
    got, iters = speculative(orc, toy, prompt, steps, D, agreement, ref, seed=D)
    assert got == ref[:steps]
    if agreement == 1.0:
        assert iters == -(-steps // (D + 1))     # every draft accepted: D+1 tokens per step
    if agreement == 0.0:
        assert iters >= steps * 0.8              # almost one token per step
