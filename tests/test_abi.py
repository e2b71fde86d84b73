"""The C-ABI library builds, loads, exports every symbol include/*.h declares,
its argument structs match the binding's, and host-side validation rejects
bad arguments before touching a GPU (no compute call is made here)."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="session")
def mtplib():
    from mtp_speculative_decoding_verify_gb300 import build
    build.build()
    from mtp_speculative_decoding_verify_gb300 import _binding
    return _binding


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"typedef struct\s*\{.*?\}\s*\w+\s*;", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\([^;{]*\)\s*;", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_three_calls():
    names = _declared_functions()
    for n in ("mtp_verify_attention", "mtp_verify_logits_accept", "kv_rollback"):
        assert n in names


def test_every_declared_symbol_is_exported(mtplib):
    L = ctypes.CDLL(mtplib.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_struct_layouts_match(mtplib):
    L = mtplib.lib()
    assert L.mtp_abi_version() == mtplib.ABI_VERSION == 5
    for which, st in enumerate((mtplib.AttnArgs, mtplib.LmArgs, mtplib.RollbackArgs, mtplib.DraftArgs,
                                mtplib.KvCompactArgs)):
        assert L.mtp_abi_struct_size(which) == ctypes.sizeof(st)


def _attn_ok(mtplib, **kw):
    a = mtplib.AttnArgs()
    a.q = a.k_new = a.v_new = a.k_cache = a.v_cache = a.block_table = a.ctx_lens = a.out = 16
    a.B, a.D, a.Hq, a.Hkv, a.d_qk, a.d_v = 2, 3, 8, 2, 128, 128
    a.block_size, a.max_blocks, a.num_blocks, a.is_mla = 64, 4, 8, 0
    a.sm_scale, a.dtype = 0.088, 1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(D=16), 1), (dict(D=-1), 1), (dict(block_size=32), 1), (dict(Hkv=3), 1), (dict(q=None), 1),
    (dict(sm_scale=0.0), 1), (dict(dtype=5), 1), (dict(d_qk=96, d_v=96), 2),
    (dict(is_mla=1, Hkv=1, d_qk=576, d_v=512, dtype=0, v_new=None, v_cache=None), 2),
    (dict(is_mla=1, Hkv=1, d_qk=576, d_v=512), 1),     # MLA must not pass v_new / v_cache
])
def test_attention_rejects_bad_args_on_host(mtplib, kw, code):
    L = mtplib.lib()
    rc = L.mtp_verify_attention(ctypes.byref(_attn_ok(mtplib, **kw)), None)
    assert rc == code, L.mtp_last_error()
    assert L.mtp_last_error()


def _lm_ok(mtplib, **kw):
    a = mtplib.LmArgs()
    a.hidden = a.lm_head = a.tokens = a.mode = a.out_tokens = a.num_accepted = a.tie_flags = 16
    a.B, a.D, a.H, a.V, a.dtype, a.any_sampling = 4, 3, 512, 8192, 0, 0
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(D=16), 1), (dict(H=0), 1), (dict(dtype=1, H=100), 2), (dict(any_sampling=1), 1),
    (dict(tokens=None), 1), (dict(dtype=9), 1),
    (dict(relaxed_topk=-1), 1), (dict(relaxed_topk=8193), 1), (dict(relaxed_topk=4, relaxed_delta=-0.1), 1),
    (dict(relaxed_topk=4, relaxed_delta=float("nan")), 1), (dict(relaxed_topk=4, relaxed_delta=float("inf")), 1),
])
def test_lmhead_rejects_bad_args_on_host(mtplib, kw, code):
    L = mtplib.lib()
    assert L.mtp_verify_logits_accept(ctypes.byref(_lm_ok(mtplib, **kw)), None) == code
    assert L.mtp_last_error()


def test_rollback_rejects_bad_args_on_host(mtplib):
    L = mtplib.lib()
    a = mtplib.RollbackArgs(16, 16, 16, 16, 16, 4, 3, 64, 8, 100)
    a.block_size = 128
    assert L.kv_rollback(ctypes.byref(a), None) == 1
    a.block_size = 64
    a.free_list = None
    assert L.kv_rollback(ctypes.byref(a), None) == 1


def test_empty_batch_is_a_no_op(mtplib):
    L = mtplib.lib()
    assert L.mtp_verify_attention(ctypes.byref(_attn_ok(mtplib, B=0)), None) == 0
    assert L.mtp_verify_logits_accept(ctypes.byref(_lm_ok(mtplib, B=0)), None) == 0
    a = mtplib.RollbackArgs(16, 16, 16, 16, 16, 0, 3, 64, 8, 100)
    assert L.kv_rollback(ctypes.byref(a), None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, mtplib):
    monkeypatch.setattr(mtplib, "LIB_PATH", "/nonexistent/libmtpverify.so")
    monkeypatch.setattr(mtplib, "_lib", None)
    with pytest.raises(RuntimeError):
        mtplib.lib()


def _draft_ok(mtplib, **kw):
    a = mtplib.DraftArgs()
    a.hidden = a.lm_head = a.out_tokens = 16
    a.B, a.H, a.V, a.dtype = 4, 512, 8192, 0
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), 1), (dict(H=0), 1), (dict(V=0), 1), (dict(dtype=7), 1), (dict(dtype=1, H=100), 2),
    (dict(dtype=0, H=6), 2), (dict(hidden=None), 1), (dict(out_tokens=None), 1),
])
def test_draft_rejects_bad_args_on_host(mtplib, kw, code):
    L = mtplib.lib()
    assert L.mtp_draft_argmax(ctypes.byref(_draft_ok(mtplib, **kw)), None) == code
    assert L.mtp_last_error()
    assert L.mtp_draft_workspace_size(ctypes.byref(_draft_ok(mtplib, **kw))) == 0


def test_draft_empty_batch_is_a_no_op(mtplib):
    L = mtplib.lib()
    assert L.mtp_draft_argmax(ctypes.byref(_draft_ok(mtplib, B=0)), None) == 0


def _cmp_ok(mtplib, **kw):
    a = mtplib.KvCompactArgs()
    a.k_cache = a.v_cache = a.block_table = a.ctx_lens = a.accepted_nodes = a.num_accepted = 16
    a.B, a.D, a.Hkv, a.d_qk, a.d_v = 2, 7, 2, 128, 128
    a.block_size, a.max_blocks, a.num_blocks, a.is_mla, a.dtype = 64, 4, 8, 0, 1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw", [
    dict(B=-1), dict(D=16), dict(D=-1), dict(block_size=32), dict(Hkv=0), dict(dtype=3), dict(k_cache=None),
    dict(v_cache=None), dict(accepted_nodes=None), dict(num_accepted=None), dict(is_mla=1, Hkv=1),
])
def test_tree_kv_compact_rejects_bad_args_on_host(mtplib, kw):
    L = mtplib.lib()
    assert L.mtp_tree_kv_compact(ctypes.byref(_cmp_ok(mtplib, **kw)), None) == 1
    assert L.mtp_last_error()


def test_tree_kv_compact_empty_batch_is_a_no_op(mtplib):
    L = mtplib.lib()
    assert L.mtp_tree_kv_compact(ctypes.byref(_cmp_ok(mtplib, B=0)), None) == 0
