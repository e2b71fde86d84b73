"""GPU parity: the library's CUDA path against the CPU oracle, element by
element, on the same seeded inputs.

  * reduced workloads (every request compared): several vocab tiles with a
    ragged tail, contexts that straddle block boundaries, both dtypes;
  * the standard workloads at full size, in the benchmark's launch
    configuration: a sample of requests compared with the oracle one by one,
    and properties checked on every request;
  * edge cases: D = 0, D = 15, empty context, tiny vocabularies, a single
    request, device-side range checks.
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
from gpu_util import (A, TOL_ATTN, TOL_LOGITS, attention_excess, attention_over_plain, TOL_LSE_REL,  # noqa: E402
                      check_invariants, compare_accept, gpu_attention, gpu_lmhead, gpu_rollback, oracle_attention,
                      oracle_lmhead)
from philox_py import philox_vec, race_exponential_vec  # noqa: E402

DEV = torch.device("cuda:0")

SMALL = {
    "cfg0": synth.CFG0,
    "cfg1_small_mla": synth.CFG1.with_(name="MLA bf16 small", B=4, Hq=16, ctx=(60, 300), H=512, V=3037),
    "cfg2_small_gqa_sampling": synth.CFG2.with_(name="GQA bf16 sampling small", B=6, Hq=16, Hkv=2, ctx=(300, 300),
                                                H=256, V=5003),
    "cfg3_small_mixed": synth.CFG3.with_(name="GQA bf16 mixed small", B=8, Hq=8, Hkv=2, ctx=(64, 700), H=256,
                                         V=7001),
    "mha_bf16_d64": synth.CFG0.with_(name="MHA bf16 d64", dtype="bf16", ctx=(0, 200), B=5, H=128, V=999),
    # MLA with 4, 3 and 1 row blocks per request: CTA pairs, and single CTAs for odd counts
    "mla_cluster4": synth.CFG1.with_(name="MLA 4 row blocks", B=3, Hq=64, ctx=(60, 700), H=256, V=2000),
    "mla_cluster3": synth.CFG1.with_(name="MLA 3 row blocks", B=2, Hq=48, ctx=(130, 400), H=128, V=777),
    "mla_single_row_block": synth.CFG1.with_(name="MLA 1 row block", B=3, Hq=16, ctx=(100, 900), H=128, V=777),
    # LM head on CTA pairs (M >= 33 rows): ragged row groups (M=40 -> N=64, M=200 -> N=224) and vocabulary tails
    "lm_pair_small_mixed": synth.CFG3.with_(name="LM head pairs, N=64", B=10, D=3, Hq=8, Hkv=2, ctx=(30, 150),
                                            H=192, V=3001),
    "lm_pair_ragged_sampling": synth.CFG2.with_(name="LM head pairs, sampling", B=50, D=3, Hq=8, Hkv=2,
                                                ctx=(40, 90), H=256, V=5003),
    "lm_pair_two_groups_mixed": synth.CFG3.with_(name="LM head pairs, 2 groups", B=100, D=3, Hq=8, Hkv=2,
                                                 ctx=(64, 200), H=128, V=7001),
    # GQA with 16 rows per KV head over a grid of several waves: spare warps split each
    # CTA's tiles (key parts) and merge at the end
    "gqa_key_parts": synth.CFG3.with_(name="GQA key parts", B=80, D=3, Hq=32, Hkv=8, ctx=(1800, 2100), H=128,
                                      V=3001),
    # vocabulary a multiple of 4: the race kernel's 16-byte row scan, ragged last slice
    "sampling_aligned_vocab": synth.CFG2.with_(name="sampling, V % 4 == 0", B=12, D=3, Hq=8, Hkv=2, ctx=(40, 90),
                                               H=128, V=4100),
}


def _par(fn, items, workers=8):
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, items))


def _stack(results):
    keys = results[0].keys()
    return {k: np.concatenate([r[k] for r in results]) for k in keys}


def _oracle_lm_parallel(w, lm, reqs, want_logits=False):
    W = A(lm["lm_head"])
    return _stack(_par(lambda b: oracle_lmhead(w, lm, [b], W, want_logits), list(reqs)))


def _oracle_attn_parallel(w, att, reqs):
    return np.concatenate(_par(lambda b: oracle_attention(w, att, [b]), list(reqs)))


def _check_attention(w, att, out, reqs):
    """Every element within the attention bound of the oracle's exact value;
    the count above the plain bound (the share that only the output's own
    rounding carries over it) is printed."""
    exact = _oracle_attn_parallel(w, att, reqs)
    got = out.index_select(0, torch.tensor(list(reqs), device=DEV)).float().cpu().numpy()
    err = float(np.abs(got - exact).max())
    n_over, frac = attention_over_plain(got, exact, w.dtype)
    print("attention %s: max |err| %.3g, %d element(s) (%.2g) above the plain %g" %
          (w.name, err, n_over, frac, TOL_ATTN[w.dtype]))
    assert attention_excess(got, exact, w.dtype) <= 0.0, err
    return err


def _check_append(w, att, att_before_knew):
    """The verify slots of the cache hold exactly the verify tokens' K (and V)."""
    table = A(att["block_table"])
    ctx = A(att["ctx_lens"])
    for b in range(min(w.B, 8)):
        for j in range(w.R):
            s = int(ctx[b]) + j
            blk = int(table[b, s // 64])
            got = att["k_cache"][blk, s % 64]
            exp = att_before_knew[b, j].reshape(got.shape)
            assert torch.equal(got, exp)


def _full_check_lm(w, lm, gpu, reqs, logits=False):
    ref = _oracle_lm_parallel(w, lm, reqs, want_logits=logits)
    flagged = compare_accept(gpu, ref, reqs)
    idx = torch.tensor(list(reqs), device=DEV)
    lse = gpu["lse"].index_select(0, idx).cpu().numpy()
    np.testing.assert_allclose(lse, ref["lse"], rtol=TOL_LSE_REL, atol=1e-6)
    assert (gpu["argmax"].index_select(0, idx).cpu().numpy() == ref["argmax"]).all()
    if logits:
        rows = torch.tensor([b * w.R + j for b in reqs for j in range(w.R)], device=DEV)
        gl = gpu["logits"].index_select(0, rows).cpu().numpy()
        err = float(np.abs(gl - ref["logits"]).max())
        assert err < TOL_LOGITS[w.dtype], err
    return flagged


def _check_rollback(w, att, gpu_n):
    table, seq, fl, fc = gpu_rollback(w, att["block_table"], att["ctx_lens"], gpu_n)
    t_h = A(att["block_table"]).copy()
    s_h = A(att["ctx_lens"]).copy()
    fl_h = np.full(fl.numel(), -1, np.int32)
    fc_h = np.zeros(1, np.int32)
    oracle.kv_rollback(t_h, s_h, gpu_n.cpu().numpy(), fl_h, fc_h, D=w.D, block_size=64)
    assert (seq.cpu().numpy() == s_h).all()
    assert (table.cpu().numpy() == t_h).all()
    assert int(fc.item()) == int(fc_h[0])
    assert (fl.cpu().numpy() == fl_h).all()


@pytest.mark.parametrize("name", list(SMALL))
def test_small_workload_all_requests(name):
    w = SMALL[name]
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    k_new = att["k_new"].clone()
    out = gpu_attention(w, att)
    gpu = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    _check_append(w, att, k_new)
    _check_attention(w, att, out, range(w.B))
    flagged = _full_check_lm(w, lm, gpu, range(w.B), logits=True)
    assert flagged <= max(1, w.B // 20)
    check_invariants(w, lm, gpu)
    _check_rollback(w, att, gpu["num_accepted"])
    mv.sync_status()


FULL = {
    "cfg1_D3": (synth.CFG1, [0, 31]),
    "cfg1_D1": (synth.CFG1.with_(D=1), [5]),
    "cfg2": (synth.CFG2, [0, 63]),
    "cfg3": (synth.CFG3, [0, 127, 128, 255]),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled_requests(name):
    w, reqs = FULL[name]
    torch.cuda.empty_cache()
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    k_new = att["k_new"].clone()
    out = gpu_attention(w, att)
    gpu = gpu_lmhead(w, lm)
    mv.sync_status()
    _check_append(w, att, k_new)
    _check_attention(w, att, out, reqs)
    flagged = _full_check_lm(w, lm, gpu, reqs)
    assert flagged <= 1
    check_invariants(w, lm, gpu)
    # The same call with the debug logits: identical results, and the sampled
    # rows' logits within the bf16 bound of the oracle's.
    dbg = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    for k in ("out_tokens", "num_accepted", "tie_flags", "lse", "argmax"):
        assert torch.equal(gpu[k], dbg[k]), k
    _full_check_lm(w, lm, dbg, reqs, logits=True)
    ties = gpu["tie_flags"].cpu().numpy()
    print("%s: near-ties flagged by the GPU: accept/relaxed band %d, race %d of %d requests" %
          (name, int(((ties & 1) != 0).sum()), int(((ties & 2) != 0).sum()), w.B))
    del dbg
    if w.sampling == "none" or w.sampling == "half":
        # Planted targets: greedy rows' argmax is the planted token.
        greedy = [b for b in range(w.B) if int(lm["mode"][b]) == 0]
        amax = gpu["argmax"].cpu().numpy()
        assert (amax[greedy] == lm["planted"].numpy()[greedy]).all()
    _check_rollback(w, att, gpu["num_accepted"])
    del att, lm, out, gpu
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,D", [(1, 7), (8, 1)])
def test_sweep_points_sampled(B, D):
    w = synth.sweep_point(B, D)
    lm = synth.make_lmhead_inputs(w, DEV)
    gpu = gpu_lmhead(w, lm)
    mv.sync_status()
    reqs = [0] if B == 1 else [0, B - 1]
    assert _full_check_lm(w, lm, gpu, reqs) <= 1
    check_invariants(w, lm, gpu)


EDGE = {
    "D0": synth.CFG0.with_(name="D=0", D=0, dtype="bf16", H=64, V=300),
    "D0_sampling": synth.CFG0.with_(name="D=0 sampling", D=0, dtype="bf16", H=64, V=300, sampling="all"),
    "D15": synth.CFG0.with_(name="D=15", D=15, dtype="bf16", H=64, V=300, ctx=(50, 130), sampling="half"),
    "ctx0_fp32": synth.CFG0.with_(name="empty context", ctx=(0, 0), V=50, H=16),
    "tiny_vocab_sampling": synth.CFG0.with_(name="V=7 sampling", V=7, H=8, sampling="all", B=16),
    "single_request": synth.CFG1.with_(name="B=1 MLA", B=1, Hq=8, ctx=(63, 63), H=64, V=130),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_cases(name):
    w = EDGE[name]
    att = synth.make_attention_inputs(w, DEV)
    lm = synth.make_lmhead_inputs(w, DEV)
    out = gpu_attention(w, att)
    gpu = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    _check_attention(w, att, out, range(w.B))
    _full_check_lm(w, lm, gpu, range(w.B), logits=True)
    check_invariants(w, lm, gpu)
    _check_rollback(w, att, gpu["num_accepted"])


@pytest.mark.parametrize("V", [7, 3001])
def test_residual_fallback_race(V):
    """q_draft = 1 everywhere (an input the ABI accepts): drafts are rejected
    and every residual weight max(0, p - q) is zero, so the draw falls back to
    p itself; the multi-slice race and the oracle must agree."""
    w = synth.CFG0.with_(name="fallback race V=%d" % V, V=V, H=64, sampling="all", B=12, dtype="bf16")
    lm = synth.make_lmhead_inputs(w, DEV)
    lm["q_draft"].fill_(1.0)
    gpu = gpu_lmhead(w, lm, debug_logits=True)
    mv.sync_status()
    assert (gpu["num_accepted"].cpu().numpy() < w.D).any()
    _full_check_lm(w, lm, gpu, range(w.B), logits=True)
    check_invariants(w, lm, gpu)


def test_rng_streams_bit_exact():
    n = 1 << 20
    for seed, b, j, tag in ((0, 0, 0, 2), (0x1234_5678_9ABC, 77, 5, 3)):
        word0, E, U = mv._binding.rng_debug(seed, b, j, tag, 0, n)
        ref = philox_vec(np.full(n, b), np.full(n, j), np.arange(n), np.full(n, tag), seed & 0xFFFFFFFF, seed >> 32)[0]
        assert (word0 == ref).all()
        refE = race_exponential_vec(seed, b, j, np.arange(n), tag)
        np.testing.assert_array_max_ulp(E, refE, maxulp=2)
        for v in (0, 1, 12345, n - 1):
            assert U[v] == oracle.accept_uniform(seed, b, v)
            assert abs(E[v] - oracle.race_exponential(seed, b, j, v, tag)) <= 2 * np.spacing(E[v])


def test_lossless_sampling_on_gpu_chi2():
    """Through the GPU path: the first emitted token follows p_target exactly."""
    from scipy import special, stats
    rng = np.random.default_rng(5)
    trials, D, V = 200_000, 2, 8
    logits = (rng.standard_normal((D + 1, V)) * 1.2).astype(np.float32)
    q = special.softmax(rng.standard_normal((D, V)) * 1.2, axis=1).astype(np.float32)
    hidden = torch.tensor(np.tile(logits, (trials, 1)), device=DEV)
    W = torch.eye(V, dtype=torch.float32, device=DEV)
    tokens = np.zeros((trials, D + 1), np.int32)
    for j in range(D):
        tokens[:, j + 1] = rng.choice(V, size=trials, p=q[j] / q[j].sum())
    lm = dict(hidden=hidden, lm_head=W, tokens=torch.tensor(tokens, device=DEV),
              mode=torch.ones(trials, dtype=torch.uint8, device=DEV),
              temperature=torch.ones(trials, dtype=torch.float32, device=DEV),
              q_draft=torch.tensor(np.broadcast_to(q, (trials, D, V)).copy(), device=DEV), seed=99)
    w = synth.CFG0.with_(B=trials, D=D, V=V, H=V)
    gpu = gpu_lmhead(w, lm)
    first = gpu["out_tokens"][:, 0].cpu().numpy()
    p = special.softmax(logits.astype(np.float64), axis=1)
    assert stats.chisquare(np.bincount(first, minlength=V), p[0] * trials).pvalue > 1e-3
    # Acceptance rate of draft 1 equals sum_v min(p, q).
    alpha = np.minimum(p[0], q[0]).sum()
    rate = (gpu["num_accepted"].cpu().numpy() >= 1).mean()
    assert abs(rate - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / trials)
    # And the GPU agrees with the oracle request by request on a sample.
    sample = list(range(0, trials, 4001))
    ref = oracle.lmhead_accept(np.tile(logits, (len(sample), 1)), np.eye(V, dtype=np.float32), tokens[sample],
                               np.ones(len(sample), np.uint8), np.ones(len(sample), np.float32),
                               np.broadcast_to(q, (len(sample), D, V)).copy(), 99,
                               request_index=np.array(sample, np.int32))
    assert compare_accept(gpu, ref, sample) <= 1


def test_rollback_many_requests_and_capacity():
    rng = np.random.default_rng(11)
    w = synth.CFG3.with_(B=3000, D=5)
    ctx = rng.integers(0, 500, w.B).astype(np.int32)
    need = (ctx + w.R + 63) // 64
    max_blocks = int(need.max()) + 1
    table = np.full((w.B, max_blocks), -1, np.int32)
    perm = rng.permutation(int(need.sum())).astype(np.int32)
    pos = 0
    for b in range(w.B):
        table[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    n = rng.integers(0, w.D + 1, w.B).astype(np.int32)
    t_d = torch.tensor(table, device=DEV)
    c_d = torch.tensor(ctx, device=DEV)
    n_d = torch.tensor(n, device=DEV)
    cap = 4 * w.B
    g_table, g_seq, g_fl, g_fc = gpu_rollback(w, t_d, c_d, n_d, capacity=cap)
    mv.sync_status()
    fl = np.full(cap, -1, np.int32)
    fc = np.zeros(1, np.int32)
    t_h, s_h = table.copy(), ctx.copy()
    oracle.kv_rollback(t_h, s_h, n, fl, fc, D=w.D, block_size=64)
    assert (g_seq.cpu().numpy() == s_h).all() and (g_table.cpu().numpy() == t_h).all()
    assert int(g_fc.item()) == int(fc[0]) and (g_fl.cpu().numpy() == fl).all()
    # A free list that is too short is reported, not overrun, and no request
    # is left half rolled back: the requests before the first one whose blocks
    # do not fit are rolled back (as the oracle does them), later requests that
    # free nothing get their new length, and the others are left untouched.
    cnt = np.maximum((ctx + w.D) // 64 - (ctx + n + 1 + 63) // 64 + 1, 0)
    total = int(cnt.sum())
    assert total > 12
    for cap in (10, 11, total - 1):
        g_table, g_seq, g_fl, g_fc = gpu_rollback(w, t_d, c_d, n_d, capacity=cap)
        with pytest.raises(mv.MtpError) as ei:
            mv.sync_status()
        assert ei.value.code == 4
        f = int(np.argmax(np.cumsum(cnt) > cap))
        t_h, s_h = table.copy(), ctx.copy()
        fl = np.full(int(cnt[:f].sum()), -1, np.int32)
        fc = np.zeros(1, np.int32)
        t_pre, s_pre = t_h[:f].copy(), s_h[:f].copy()
        oracle.kv_rollback(t_pre, s_pre, n[:f].copy(), fl, fc, D=w.D, block_size=64)
        t_h[:f], s_h[:f] = t_pre, s_pre
        zero = np.arange(w.B) >= f
        zero &= cnt == 0
        s_h[zero] = ctx[zero] + n[zero] + 1
        assert (g_seq.cpu().numpy() == s_h).all() and (g_table.cpu().numpy() == t_h).all()
        assert int(g_fc.item()) == int(fc[0]) <= cap
        assert (g_fl.cpu().numpy()[:int(fc[0])] == fl).all()


def test_device_range_checks_report_and_recover():
    w = SMALL["cfg3_small_mixed"]
    att = synth.make_attention_inputs(w, DEV)
    att["block_table"][1, 0] = 10 ** 6          # block id beyond the cache: skipped and reported
    gpu_attention(w, att)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert ei.value.code == 4 and "block-id" in str(ei.value)
    lm = synth.make_lmhead_inputs(w, DEV)
    lm["tokens"][2, 1] = w.V + 5                # draft id beyond the vocabulary
    gpu_lmhead(w, lm)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert "token-id" in str(ei.value)
    # The context stays usable: a clean call afterwards succeeds.
    w0 = SMALL["cfg0"]
    gpu_lmhead(w0, synth.make_lmhead_inputs(w0, DEV))
    mv.sync_status()


def test_mla_pair_range_checks_report_and_spare_other_requests():
    """The CTA pairs of the MLA kernel are persistent and walk many requests'
    items in turn: one request's first block id lies beyond the cache and
    another's context exceeds its block table. Both are reported (the block
    reads as zeros, the long request is skipped), the pairs go on to their
    next items, and the other requests still match the oracle."""
    # 40 requests x 2 pair groups x 2 key splits: more items than CTA pairs
    w = synth.CFG1.with_(name="MLA pairs, range checks", B=40, Hq=64, ctx=(60, 700), H=256, V=2000)
    att = synth.make_attention_inputs(w, DEV)
    keep = [b for b in range(w.B) if b not in (1, 3)]
    exact = np.concatenate(_par(lambda b: oracle_attention(w, att, [b]), keep))
    att["block_table"][1, 0] = 10 ** 6
    att["ctx_lens"][3] = w.max_blocks * 64
    out = gpu_attention(w, att)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert ei.value.code == 4 and "block-id" in str(ei.value) and "length" in str(ei.value)
    got = out.index_select(0, torch.tensor(keep, device=DEV)).float().cpu().numpy()
    assert attention_excess(got, exact, w.dtype) <= 0.0
    w2 = SMALL["cfg1_small_mla"]
    att2 = synth.make_attention_inputs(w2, DEV)
    out2 = gpu_attention(w2, att2)
    mv.sync_status()
    _check_attention(w2, att2, out2, range(w2.B))


def test_bounded_wait_gives_up_and_context_survives():
    """The kernels' time-limited mbarrier wait, on a barrier nothing arrives on
    (no fault, no trap): it returns after the limit and flags a timeout that
    the host reads; the next calls run normally."""
    import time
    t0 = time.perf_counter()
    mv._binding.wait_selftest(50_000_000)        # 50 ms
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert ei.value.code == 4 and "timeout" in str(ei.value)
    assert time.perf_counter() - t0 >= 0.04
    mv.sync_status()                               # the flag was cleared
    with pytest.raises(mv.MtpError) as ei:
        mv._binding.wait_selftest(0)
    assert ei.value.code == 1
    w = SMALL["cfg1_small_mla"]
    att = synth.make_attention_inputs(w, DEV)
    out = gpu_attention(w, att)
    mv.sync_status()
    _check_attention(w, att, out, range(w.B))
