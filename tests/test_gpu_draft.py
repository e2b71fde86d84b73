"""GPU parity of the greedy draft step of MTP Eagle (mtp_draft_argmax: B rows,
top-1 over the shared LM head) against the CPU oracle, on the tensor-core
LM head (single CTAs and CTA pairs) and the fp32 SIMT one, at full
DeepSeek-V3 / Llama-70B LM-head sizes on sampled rows, and against the verify
call with D = 0 (the same kernels) bit for bit."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402
from gpu_util import A, TOL_LSE_REL  # noqa: E402

DEV = torch.device("cuda:0")

SMALL = {
    "tc_single": synth.CFG0.with_(name="draft bf16", dtype="bf16", B=37, D=2, H=256, V=5003, stream=31),
    "tc_pair": synth.CFG0.with_(name="draft bf16 pairs", dtype="bf16", B=200, D=1, H=128, V=7001, stream=32),
    "simt_f32": synth.CFG0.with_(name="draft fp32", B=9, D=2, H=96, V=1037, stream=33),
    "one_row": synth.CFG0.with_(name="draft B=1", dtype="bf16", B=1, D=1, H=64, V=130, stream=34),
}


def _draft(inp, k):
    B = inp["hidden"].shape[1]
    tok = torch.full((B,), -9, dtype=torch.int32, device=DEV)
    lse = torch.empty(B, dtype=torch.float32, device=DEV)
    mv.mtp_draft_argmax(inp["hidden"][k], inp["lm_head"], tok, lse)
    return tok, lse


def _oracle_rows(inp, k, rows):
    W = A(inp["lm_head"])
    h = A(inp["hidden"][k].index_select(0, torch.tensor(rows, device=DEV)))
    toks = np.zeros((len(rows), 1), np.int32)
    r = oracle.lmhead_accept(h, W, toks, np.zeros(len(rows), np.uint8), None, None, 0)
    return r["argmax"][:, 0], r["lse"][:, 0]


@pytest.mark.parametrize("name", list(SMALL))
def test_draft_small_all_rows(name):
    w = SMALL[name]
    inp = synth.make_draft_inputs(w, DEV)
    for k in range(w.D):
        tok, lse = _draft(inp, k)
        mv.sync_status()
        amax, ref_lse = _oracle_rows(inp, k, list(range(w.B)))
        assert (tok.cpu().numpy() == amax).all()
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=TOL_LSE_REL, atol=1e-6)
        assert (tok.cpu() == inp["planted"][k]).all()


def test_draft_equals_verify_call_with_no_drafts():
    w = SMALL["tc_single"]
    inp = synth.make_draft_inputs(w, DEV)
    tok, lse = _draft(inp, 0)
    out = torch.empty((w.B, 1), dtype=torch.int32, device=DEV)
    n = torch.empty(w.B, dtype=torch.int32, device=DEV)
    tie = torch.empty(w.B, dtype=torch.uint8, device=DEV)
    lse_v = torch.empty((w.B, 1), dtype=torch.float32, device=DEV)
    tokens = inp["planted"][0].reshape(w.B, 1).to(DEV)   # any valid input token
    mv.mtp_verify_logits_accept(inp["hidden"][0], inp["lm_head"], tokens, torch.zeros(w.B, dtype=torch.uint8,
                                                                                          device=DEV),
                                None, None, 0, out, n, tie, lse_v)
    mv.sync_status()
    assert torch.equal(out[:, 0], tok) and torch.equal(lse_v[:, 0], lse)
    assert (n == 0).all()


@pytest.mark.parametrize("base", ["cfg1", "cfg2"])
def test_draft_full_size_sampled_rows(base):
    """DeepSeek-V3 (B=32, H=7168, V=129280) and Llama-70B (B=64, H=8192,
    V=128256) LM heads: every row's top-1 is its planted token, sampled rows
    match the oracle, and repeated calls give identical results."""
    w = (synth.CFG1 if base == "cfg1" else synth.CFG2).with_(D=2)
    torch.cuda.empty_cache()
    inp = synth.make_draft_inputs(w, DEV)
    for k in range(w.D):
        tok, lse = _draft(inp, k)
        tok2, lse2 = _draft(inp, k)
        mv.sync_status()
        assert torch.equal(tok, tok2) and torch.equal(lse, lse2)
        assert (tok.cpu() == inp["planted"][k]).all()
        rows = [0, w.B - 1]
        amax, ref_lse = _oracle_rows(inp, k, rows)
        assert (tok.cpu().numpy()[rows] == amax).all()
        np.testing.assert_allclose(lse.cpu().numpy()[rows], ref_lse, rtol=TOL_LSE_REL, atol=1e-6)
    del inp
    torch.cuda.empty_cache()


def test_draft_bad_arguments():
    w = SMALL["tc_single"]
    inp = synth.make_draft_inputs(w, DEV)
    tok = torch.empty(w.B, dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError):
        mv.mtp_draft_argmax(inp["hidden"][0], inp["lm_head"], tok[:-1])
    bad_h = torch.zeros((w.B, 100), dtype=torch.bfloat16, device=DEV)
    bad_w = torch.zeros((w.V, 100), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mv.MtpError) as ei:
        mv.mtp_draft_argmax(bad_h, bad_w, tok)
    assert "H % 64" in str(ei.value)
    empty = torch.empty((0, w.H), dtype=torch.bfloat16, device=DEV)
    mv.mtp_draft_argmax(empty, inp["lm_head"], torch.empty(0, dtype=torch.int32, device=DEV))
    mv.sync_status()
