"""GPU parity of the tcgen05 GQA attention kernel (bf16, head dim 128, 49..64
query rows per KV head) against the CPU oracle, every request of each case:
ragged row counts (50, 52, 60 rows: the Q box is not a whole number of 8-row
swizzle groups, padding rows are zero), 56 and 64 rows, contexts that start
empty or end inside a cache block, KV splits with the combine pass, tree
masks, a batch of several items per CTA with mixed lengths (the longest-first
work order), and one with enough items per persistent CTA that the ring of
published work items wraps. Cache pages are shuffled, so every tile reads two
unrelated blocks."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402
from gpu_util import attention_excess, gpu_attention, oracle_attention  # noqa: E402

DEV = torch.device("cuda:0")

_G = synth.CFG3.with_(sampling="none", H=128, V=1000)

CASES = {
    # 4 heads x 13 verify tokens = 52 rows, contexts from empty
    "rows52_ctx_from_0": _G.with_(name="GQA tc 52 rows", B=5, D=12, Hq=8, Hkv=2, ctx=(0, 300), stream=61),
    # 5 heads x 10 tokens = 50 rows; long contexts: KV splits and the combine
    "rows50_splits": _G.with_(name="GQA tc 50 rows, splits", B=2, D=9, Hq=10, Hkv=2, ctx=(3000, 9000), stream=62),
    # 16 heads x 4 tokens = 64 rows
    "rows64_group16": _G.with_(name="GQA tc 16x4", B=6, D=3, Hq=32, Hkv=2, ctx=(100, 1000), stream=63),
    # 8 heads x 7 tokens = 56 rows: the Llama-70B grouping at D = 6
    "rows56_llama_grouping": _G.with_(name="GQA tc 8x7", B=4, D=6, Hq=64, Hkv=8, ctx=(1, 700), stream=64),
    # 8 heads x 8 tokens = 64 rows, contexts that end inside a block
    "rows64_chain": _G.with_(name="GQA tc 64 rows", B=5, D=7, Hq=16, Hkv=2, ctx=(63, 390), stream=65),
    # 4 heads x 16 tree nodes = 64 rows, random trees
    "rows64_tree_random": _G.with_(name="GQA tc tree 64 rows", B=6, D=15, Hq=8, Hkv=2, ctx=(1, 500),
                                   tree="random", stream=66),
    # 4 heads x 15 nodes = 60 rows, random trees, long requests (splits)
    "rows60_tree_splits": _G.with_(name="GQA tc tree, splits", B=2, D=14, Hq=4, Hkv=1, ctx=(5000, 6000),
                                   tree="random", stream=67),
    # several items per CTA (B * Hkv = 480), mixed lengths: longest-first order
    "rows56_waves_mixed": _G.with_(name="GQA tc waves", B=120, D=13, Hq=16, Hkv=4, ctx=(10, 1500), stream=68),
    # about ten items per persistent CTA: the scheduler's ring of 8 work items wraps
    "rows56_ring_wrap": _G.with_(name="GQA tc ring wrap", B=400, D=13, Hq=16, Hkv=4, ctx=(0, 300), stream=69),
}


def _np(t):
    return t.float().cpu().numpy()


def _ref_float(ref):
    """Oracle output as floats (the exact float64 result, or bf16 bit patterns widened)."""
    if ref.dtype == np.float64:
        return ref
    return torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy()


def _run(w):
    att = synth.make_attention_inputs(w, DEV)
    parents = synth.make_parents(w)
    parents = None if parents is None else parents.to(DEV)
    out = gpu_attention(w, att, parents)
    mv.sync_status()
    with cf.ThreadPoolExecutor(8) as ex:
        refs = list(ex.map(lambda b: oracle_attention(w, att, [b], parents), range(w.B)))
    return _np(out), _ref_float(np.concatenate(refs))


@pytest.mark.parametrize("name", list(CASES))
def test_gqa_tc_all_requests(name):
    w = CASES[name]
    rows = (w.Hq // w.Hkv) * w.R
    assert 48 < rows <= 64 and w.d_qk == 128 and w.dtype == "bf16"
    got, ref = _run(w)
    assert np.isfinite(got).all()
    assert attention_excess(got, ref, w.dtype) <= 0.0


def test_gqa_tc_chain_as_tree_matches_chain():
    """A tree whose parents form the chain gives the chain's output bit for
    bit (same kernel, mask from the path bits instead of the key limit)."""
    w = CASES["rows64_chain"]
    att = synth.make_attention_inputs(w, DEV)
    chain = gpu_attention(w, att)
    att2 = synth.make_attention_inputs(w, DEV)
    parents = torch.arange(-1, w.R - 1, dtype=torch.int32, device=DEV).repeat(w.B, 1).contiguous()
    tree = gpu_attention(w, att2, parents)
    mv.sync_status()
    assert torch.equal(chain, tree)


def test_gqa_tc_range_checks_report_and_spare_other_requests():
    """One request's first block id lies beyond the cache and another's context
    exceeds its block table: both are reported (the block reads as zeros, the
    long request is skipped), the other requests still match the oracle, and
    the next call runs normally."""
    w = CASES["rows64_chain"]
    att = synth.make_attention_inputs(w, DEV)
    keep = [0, 2, 4]
    ref = _ref_float(np.concatenate([oracle_attention(w, att, [b]) for b in keep]))
    att["block_table"][1, 0] = 10 ** 6
    att["ctx_lens"][3] = w.max_blocks * 64
    out = gpu_attention(w, att)
    with pytest.raises(mv.MtpError) as ei:
        mv.sync_status()
    assert ei.value.code == 4 and "block-id" in str(ei.value) and "length" in str(ei.value)
    assert attention_excess(_np(out)[keep], ref, w.dtype) <= 0.0
    got, ref2 = _run(CASES["rows64_tree_random"])
    assert attention_excess(got, ref2, "bf16") <= 0.0
