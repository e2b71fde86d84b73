"""GB300 (sm_103a) library for the verify step of MTP speculative decoding.

The compute path is libmtpverify.so (hand-written CUDA kernels behind a C
ABI, include/mtp_verify.h); this package is its thin ctypes binding plus the
seeded synthetic-workload generators used by the tests and the benchmark.
"""
from ._binding import (  # noqa: F401
    MtpError,
    kv_rollback,
    lib,
    mtp_draft_argmax,
    mtp_tree_kv_compact,
    mtp_verify_attention,
    mtp_verify_logits_accept,
    mtp_verify_logits_accept_noalloc,
    sync_status,
)
