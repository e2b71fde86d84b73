"""The read-bandwidth probe (a measurement aid of the benchmark, not on the
verify path): both of its paths read every byte they are given. The sink
receives the XOR of the buffer's 32-bit words (loads) or of the first word of
each chunk that a CTA's ring held last (bulk copies), so a buffer of one
repeated word pins the loads path exactly and the bulk path up to parity; the
bulk path must also raise no timeout and leave the context usable."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; the marker keeps them out of -m "not gpu"
    pytest.skip("needs a CUDA device", allow_module_level=True)

import mtp_speculative_decoding_verify_gb300 as mv  # noqa: E402
from mtp_speculative_decoding_verify_gb300 import _binding  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.mark.parametrize("nbytes", [16, 4096, 1 << 20, (37 << 20) + 48])
def test_loads_path_xors_every_word(nbytes):
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 2 ** 32, nbytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(host.view(np.int32).copy()).to(DEV)
    for ctas in (1, 2, 4):
        sink = torch.zeros(1, dtype=torch.int32, device=DEV)
        _binding.hbm_read_probe(buf, sink, ctas, False)
        mv.sync_status()
        want = int(np.bitwise_xor.reduce(host)) if host.size else 0
        assert int(sink.cpu().numpy().view(np.uint32)[0]) == want


@pytest.mark.parametrize("nbytes", [16, 32768, (5 << 20) + 16, 64 << 20])
def test_bulk_path_completes(nbytes):
    word = np.uint32(0x5A5A1234)
    buf = torch.from_numpy(np.full(nbytes // 4, word, np.uint32).view(np.int32)).to(DEV)
    sink = torch.zeros(1, dtype=torch.int32, device=DEV)
    _binding.hbm_read_probe(buf, sink, 1, True)
    mv.sync_status()   # no timeout flagged
    got = int(sink.cpu().numpy().view(np.uint32)[0])
    assert got in (0, int(word))   # an XOR of copies of one word


def test_probe_rejects_bad_arguments():
    buf = torch.zeros(64, dtype=torch.uint8, device=DEV)
    sink = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(mv.MtpError):
        _binding.hbm_read_probe(buf[1:33], sink, 1, False)   # not 16-byte aligned
    with pytest.raises(mv.MtpError):
        _binding.hbm_read_probe(buf, sink, 5, False)         # ctas_per_sm outside [1, 4]
