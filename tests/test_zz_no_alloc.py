"""mtp_verify_logits_accept_noalloc: the LM-head + acceptance entry point for
callers that cannot allocate device memory (a plugin inside an engine that
owns all device memory, a latency-critical loop that cannot afford
cudaMalloc's device-wide synchronisation). Its scratch is a fixed array owned
by the library instead of a caller workspace.

Checked here through the C ABI: two different calls in a row (the second one
reuses the array the first left behind) give the same results as the regular
entry point, within the parity tolerances, and a batch too large for the
array is refused with a clear error. This file sorts last so that a run
stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import _binding, synth  # noqa: E402
from gpu_util import TOL_LOGITS, TOL_LSE_REL, gpu_lmhead  # noqa: E402

DEV = torch.device("cuda:0")


def _noalloc(w, lm):
    res = dict(out_tokens=torch.full((w.B, w.R), -9, dtype=torch.int32, device=DEV),
               num_accepted=torch.full((w.B,), -9, dtype=torch.int32, device=DEV),
               tie_flags=torch.full((w.B,), 255, dtype=torch.uint8, device=DEV),
               lse=torch.empty((w.B, w.R), dtype=torch.float32, device=DEV),
               argmax=torch.empty((w.B, w.R), dtype=torch.int32, device=DEV),
               logits=torch.empty((w.M, w.V), dtype=torch.float32, device=DEV))
    _binding.mtp_verify_logits_accept_noalloc(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"],
                                              lm["temperature"], lm["q_draft"], lm["seed"], res["out_tokens"],
                                              res["num_accepted"], res["tie_flags"], res["lse"], res["argmax"],
                                              res["logits"])
    return res


def _same(w, a, b):
    assert torch.equal(a["out_tokens"], b["out_tokens"])
    assert torch.equal(a["num_accepted"], b["num_accepted"])
    assert torch.equal(a["tie_flags"], b["tie_flags"])
    assert torch.equal(a["argmax"], b["argmax"])
    np.testing.assert_allclose(a["lse"].cpu().numpy(), b["lse"].cpu().numpy(), rtol=TOL_LSE_REL, atol=1e-6)
    assert float((a["logits"] - b["logits"]).abs().max()) <= TOL_LOGITS[w.dtype]


def test_noalloc_matches_regular_entry_point_two_calls_in_a_row():
    L = _binding.lib()
    assert L.mtp_noalloc_scratch_bytes() == 8 << 20
    first = synth.CFG0                                        # fp32, greedy
    second = synth.CFG2.with_(name="small bf16 sampling", B=6, Hq=16, Hkv=2, ctx=(300, 300), H=256, V=5003)
    for w in (first, second, first):
        lm = synth.make_lmhead_inputs(w, DEV)
        ref = gpu_lmhead(w, lm, debug_logits=True)
        got = _noalloc(w, lm)
        assert L.mtp_last_launch_count() == 2 + (lm["q_draft"] is not None)
        mv.sync_status()
        _same(w, ref, got)


def test_noalloc_refuses_batches_beyond_its_scratch():
    w = synth.CFG0.with_(name="oversized sampling", dtype="bf16", H=64, V=200_000, sampling="all")
    lm = synth.make_lmhead_inputs(w, DEV)                    # 16 rows x 200k logits > 8 MiB
    with pytest.raises(mv.MtpError) as ei:
        _noalloc(w, lm)
    assert ei.value.code == _binding.MTP_INVALID_ARG and "no-alloc" in str(ei.value)
