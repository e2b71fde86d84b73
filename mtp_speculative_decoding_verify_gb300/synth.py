"""Seeded synthetic inputs for the verify step.

This module only builds inputs; it holds none of the verify step's own
arithmetic, and both the GPU library's tests/benchmark and the CPU oracle's
checks draw their inputs from it. Everything is drawn from a seeded
``torch.Generator`` on the requested device (the CPU and CUDA generators give
different streams, so a test must hand the same tensors to both sides).

Workload recipe (what the five standard workloads contain):
  * paged KV cache, 64 tokens per block, physical blocks handed out in a
    seeded random order so that block tables are not the identity;
  * Q / K / V ~ N(0, 1);
  * LM-head weights W ~ N(0, 0.02);
  * planted hidden states h = 4 W[t] / ||W[t]|| + N(0, 0.01) so the target
    argmax of each row is its planted token t;
  * greedy drafts copy the planted token of the row before with a given
    agreement probability, else a uniform token;
  * for rejection-sampling requests the draft distribution of row j is
    q_j = softmax(logits_j / T + N(0, 0.5)) (logits = h W^T, a plain float32
    matmul used only to shape the input) and draft d_{j+1} ~ q_j;
  * tree drafts: "full" trees fan out 3 ways at the root, 2 ways below, then
    continue as chains (D = 15: 3 + 6 + 6 nodes, depth 3); "random" trees
    give node k a uniform parent in [0, k). Node k's draft copies the
    planted token of its parent's row with the agreement probability, else a
    uniform token, so several branches of a node can match;
  * relaxed requests (mode 2) get sharper rows with a planted runner-up:
    h = L1 W[t] / ||W[t]||^2 + L2 W[s] / ||W[s]||^2 + N(0, 0.01) with
    L1 ~ U(ln V - 1, ln V + 3) and L2 = L1 - U(0, 3), so that token t leads
    with probability ~0.3-0.95 and s follows it by a random gap; the draft is
    s with probability 0.5, t with 0.25, else a uniform token (which ranks
    far outside any small top-N).
"""
from dataclasses import dataclass, field, replace
import math

import torch

BLOCK = 64


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    D: int
    Hq: int
    Hkv: int
    d_qk: int
    d_v: int
    is_mla: bool
    ctx: tuple            # (lo, hi) inclusive; lo == hi for a fixed context
    dtype: str            # "f32" or "bf16"
    H: int
    V: int
    agreement: float      # greedy draft agreement probability
    sampling: str         # "none" | "all" | "half" (second half of the batch samples)
    temperature: float    # temperature of sampling requests
    seed: int = 0
    stream: int = 0
    spare_blocks: int = 4
    relaxed: str = "none"       # "none" | "all" | "half" (first half of the batch), mode 2 over the sampling mask
    relaxed_topk: int = 0       # N of the relaxed rule
    relaxed_delta: float = 0.0  # delta of the relaxed rule
    tree: str = "chain"         # "chain" | "full" | "random" draft trees (greedy verification)

    @property
    def R(self):
        return self.D + 1

    @property
    def M(self):
        return self.B * (self.D + 1)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def sm_scale(self):
        return 1.0 / math.sqrt(self.d_qk)

    @property
    def max_blocks(self):
        return (self.ctx[1] + self.D + 1 + BLOCK - 1) // BLOCK

    def with_(self, **kw):
        return replace(self, **kw)


# The five standard workloads (names describe them; sizes as stated).
CFG0 = Workload("tiny greedy MHA fp32: B=4 D=3 ctx=128 8x64 H=512 V=8192",
                B=4, D=3, Hq=8, Hkv=8, d_qk=64, d_v=64, is_mla=False, ctx=(128, 128), dtype="f32",
                H=512, V=8192, agreement=0.7, sampling="none", temperature=1.0, seed=0, stream=0)
CFG1 = Workload("DeepSeek-V3-shaped greedy MLA bf16: B=32 D=3 128x576/512 ctx 512-4096 H=7168 V=129280",
                B=32, D=3, Hq=128, Hkv=1, d_qk=576, d_v=512, is_mla=True, ctx=(512, 4096), dtype="bf16",
                H=7168, V=129280, agreement=0.8, sampling="none", temperature=1.0, seed=0, stream=1)
CFG2 = Workload("Llama-70B-shaped rejection sampling GQA bf16: B=64 D=5 64/8x128 ctx=4096 H=8192 V=128256",
                B=64, D=5, Hq=64, Hkv=8, d_qk=128, d_v=128, is_mla=False, ctx=(4096, 4096), dtype="bf16",
                H=8192, V=128256, agreement=0.0, sampling="all", temperature=1.0, seed=0, stream=2)
CFG3 = Workload("large-batch long-context mixed GQA bf16: B=256 D=3 32/8x128 ctx 1k-32k H=4096 V=151936",
                B=256, D=3, Hq=32, Hkv=8, d_qk=128, d_v=128, is_mla=False, ctx=(1024, 32768), dtype="bf16",
                H=4096, V=151936, agreement=0.6, sampling="half", temperature=0.7, seed=0, stream=3)


def sweep_point(B, D):
    """Config-3 shapes at context 8192, every request rejection-sampled (T = 0.7)."""
    return CFG3.with_(name="sweep B=%d D=%d ctx=8192 32/8x128 H=4096 V=151936" % (B, D), B=B, D=D,
                      ctx=(8192, 8192), sampling="all", agreement=0.0, seed=1000 * B + D, stream=4)


def _gen(w, device, salt):
    g = torch.Generator(device=device)
    g.manual_seed(((w.seed * 1_000_003 + w.stream) * 16 + salt) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _sampling_mask(w):
    if w.sampling == "none":
        return torch.zeros(w.B, dtype=torch.bool)
    if w.sampling == "all":
        return torch.ones(w.B, dtype=torch.bool)
    m = torch.zeros(w.B, dtype=torch.bool)
    m[w.B // 2:] = True
    return m


def full_tree_parents(R):
    """Parents of a full tree in breadth-first order: 3 children at the root,
    2 under each of those, then single chains under the leaves, until R nodes."""
    parents = [-1]
    frontier = [0]
    fan = [3, 2]
    level = 0
    while len(parents) < R:
        nxt = []
        for u in frontier:
            for _ in range(fan[level] if level < len(fan) else 1):
                if len(parents) < R:
                    parents.append(u)
                    nxt.append(len(parents) - 1)
        frontier = nxt if nxt else frontier
        level += 1
    return parents


def make_parents(w):
    """[B, R] int32 parents of each request's draft tree (None for chains)."""
    if w.tree == "chain":
        return None
    if w.tree == "full":
        return torch.tensor([full_tree_parents(w.R)] * w.B, dtype=torch.int32)
    g = _gen(w, "cpu", 10)
    par = torch.empty((w.B, w.R), dtype=torch.int32)
    par[:, 0] = -1
    for k in range(1, w.R):
        par[:, k] = torch.randint(0, k, (w.B,), generator=g, dtype=torch.int32)
    return par


def _relaxed_mask(w):
    if w.relaxed == "none":
        return torch.zeros(w.B, dtype=torch.bool)
    if w.relaxed == "all":
        return torch.ones(w.B, dtype=torch.bool)
    m = torch.zeros(w.B, dtype=torch.bool)
    m[:w.B // 2] = True
    return m


def make_attention_inputs(w, device):
    """Paged KV cache, block table, context lengths, Q and the verify tokens' new K/V."""
    g = _gen(w, device, 1)
    R, dt = w.R, w.torch_dtype
    lo, hi = w.ctx
    if lo == hi:
        ctx = torch.full((w.B,), lo, dtype=torch.int32)
    else:
        ctx = torch.randint(lo, hi + 1, (w.B,), generator=_gen(w, "cpu", 2), dtype=torch.int32)
    need = [(int(c) + R + BLOCK - 1) // BLOCK for c in ctx]
    num_blocks = sum(need) + w.spare_blocks
    perm = torch.randperm(num_blocks, generator=_gen(w, "cpu", 3)).to(torch.int32)
    table = torch.full((w.B, w.max_blocks), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    Hkv = 1 if w.is_mla else w.Hkv
    k_cache = torch.randn((num_blocks, BLOCK, Hkv, w.d_qk), generator=g, device=device, dtype=torch.float32).to(dt)
    v_cache = None if w.is_mla else torch.randn((num_blocks, BLOCK, Hkv, w.d_v), generator=g, device=device,
                                                dtype=torch.float32).to(dt)
    q = torch.randn((w.B, R, w.Hq, w.d_qk), generator=g, device=device, dtype=torch.float32).to(dt)
    k_new = torch.randn((w.B, R, Hkv, w.d_qk), generator=g, device=device, dtype=torch.float32).to(dt)
    if w.is_mla:
        k_new = k_new.reshape(w.B, R, w.d_qk)
    v_new = None if w.is_mla else torch.randn((w.B, R, Hkv, w.d_v), generator=g, device=device,
                                              dtype=torch.float32).to(dt)
    return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                block_table=table.to(device), ctx_lens=ctx.to(device), free_spare=perm[pos:].clone())


def make_lmhead_inputs(w, device, chunk=16384):
    """LM-head weights, planted hidden states, verify tokens, modes, temperatures and q."""
    g = _gen(w, device, 4)
    gc = _gen(w, "cpu", 5)
    R, M, dt = w.R, w.M, w.torch_dtype
    W = (torch.randn((w.V, w.H), generator=g, device=device, dtype=torch.float32) * 0.02)
    planted = torch.randint(0, w.V, (w.B, R), generator=gc, dtype=torch.int64)
    Wp = W[planted.reshape(-1).to(device)]
    h = 4.0 * Wp / Wp.norm(dim=1, keepdim=True)
    relx = _relaxed_mask(w)
    runner = None
    if bool(relx.any()):
        gr = _gen(w, "cpu", 6)
        runner = torch.randint(0, w.V, (w.B, R), generator=gr, dtype=torch.int64)
        lv = math.log(w.V)
        L1 = lv - 1.0 + 4.0 * torch.rand((w.B, R), generator=gr)
        L2 = L1 - 3.0 * torch.rand((w.B, R), generator=gr)
        Ws = W[runner.reshape(-1).to(device)]
        sharp = (L1.reshape(-1, 1).to(device) * Wp / (Wp * Wp).sum(dim=1, keepdim=True) +
                 L2.reshape(-1, 1).to(device) * Ws / (Ws * Ws).sum(dim=1, keepdim=True))
        rows = relx.repeat_interleave(R).to(device)
        h = torch.where(rows.reshape(-1, 1), sharp, h)
    h = h + 0.01 * torch.randn((M, w.H), generator=g, device=device, dtype=torch.float32)
    W = W.to(dt)
    h = h.to(dt)
    samp = _sampling_mask(w) & ~relx
    mode = torch.where(relx, torch.tensor(2, dtype=torch.uint8), samp.to(torch.uint8))
    temperature = torch.where(samp, torch.tensor(w.temperature), torch.tensor(1.0)).to(torch.float32)

    # Greedy drafts: d_{j+1} = planted[j] with the agreement probability, else uniform.
    tokens = torch.empty((w.B, R), dtype=torch.int64)
    tokens[:, 0] = torch.randint(0, w.V, (w.B,), generator=gc)
    agree = torch.rand((w.B, w.D), generator=gc) < w.agreement
    rand_tok = torch.randint(0, w.V, (w.B, w.D), generator=gc)
    tokens[:, 1:] = torch.where(agree, planted[:, :w.D], rand_tok)
    parents = make_parents(w)
    if parents is not None:   # node k continues its parent's row: copy that row's planted token
        par = parents[:, 1:].to(torch.int64)
        tokens[:, 1:] = torch.where(agree, torch.gather(planted, 1, par), rand_tok)
    if runner is not None:
        pick = torch.rand((w.B, w.D), generator=_gen(w, "cpu", 7))
        rtok = torch.where(pick < 0.5, runner[:, :w.D], torch.where(pick < 0.75, planted[:, :w.D], rand_tok))
        tokens[:, 1:] = torch.where(relx.reshape(-1, 1), rtok, tokens[:, 1:])

    q_draft = None
    if bool(samp.any()):
        q_draft = torch.zeros((w.B, w.D, w.V), device=device, dtype=torch.float32)
        sb = torch.nonzero(samp).reshape(-1).tolist()
        rows = torch.tensor([b * R + j for b in sb for j in range(w.D)], dtype=torch.int64, device=device)
        hs = h[rows].float()
        logits = torch.empty((rows.numel(), w.V), device=device, dtype=torch.float32)
        for v0 in range(0, w.V, chunk):
            logits[:, v0:v0 + chunk] = hs @ W[v0:v0 + chunk].float().T
        noise = torch.randn(logits.shape, generator=g, device=device, dtype=torch.float32)
        qs = torch.softmax(logits / w.temperature + 0.5 * noise, dim=1)
        del logits, noise
        draws = torch.multinomial(qs, 1, generator=g).reshape(len(sb), w.D).cpu()
        qs = qs.reshape(len(sb), w.D, w.V)
        for i, b in enumerate(sb):
            q_draft[b] = qs[i]
            tokens[b, 1:] = draws[i]
    return dict(hidden=h, lm_head=W, tokens=tokens.to(torch.int32).to(device), mode=mode.to(device),
                temperature=temperature.to(device), q_draft=q_draft, planted=planted.to(torch.int32), seed=w.seed,
                relaxed_topk=w.relaxed_topk, relaxed_delta=w.relaxed_delta,
                parents=None if parents is None else parents.to(device))


def make_draft_inputs(w, device):
    """Inputs of D sequential greedy draft steps over the shared LM head:
    hidden [D, B, H] (draft step k's B rows, planted like the verify rows so
    each row's argmax is its planted token), lm_head W [V, H], planted [D, B]."""
    g = _gen(w, device, 8)
    gc = _gen(w, "cpu", 9)
    W = (torch.randn((w.V, w.H), generator=g, device=device, dtype=torch.float32) * 0.02)
    planted = torch.randint(0, w.V, (w.D, w.B), generator=gc, dtype=torch.int64)
    Wp = W[planted.reshape(-1).to(device)]
    h = 4.0 * Wp / Wp.norm(dim=1, keepdim=True)
    h = h + 0.01 * torch.randn((w.D * w.B, w.H), generator=g, device=device, dtype=torch.float32)
    return dict(hidden=h.to(w.torch_dtype).reshape(w.D, w.B, w.H).contiguous(), lm_head=W.to(w.torch_dtype),
                planted=planted.to(torch.int32))


def as_oracle_array(t):
    """Host numpy view for the oracle: float32 as is, bf16 as uint16 bit patterns."""
    import numpy as np
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
