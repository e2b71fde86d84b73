"""ctypes binding of libmtpverify.so (include/mtp_verify.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their raw pointers go into the C argument structs, and every step
of the verify path runs in the library's CUDA kernels. There is no CPU
fallback: if the library is missing, loading it raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libmtpverify.so")

MTP_OK, MTP_INVALID_ARG, MTP_UNSUPPORTED, MTP_CUDA_ERROR, MTP_DEVICE_ERROR = range(5)
ABI_VERSION = 5   # MTP_ABI_VERSION of the header the structs below mirror
MTP_F32, MTP_BF16 = 0, 1
MAX_DRAFTS = 15
BLOCK_SIZE = 64

_P = ctypes.c_void_p
_I = ctypes.c_int32


class AttnArgs(ctypes.Structure):
    _fields_ = [("q", _P), ("k_new", _P), ("v_new", _P), ("k_cache", _P), ("v_cache", _P),
                ("block_table", _P), ("ctx_lens", _P), ("out", _P),
                ("B", _I), ("D", _I), ("Hq", _I), ("Hkv", _I), ("d_qk", _I), ("d_v", _I),
                ("block_size", _I), ("max_blocks", _I), ("num_blocks", _I), ("is_mla", _I),
                ("sm_scale", ctypes.c_float), ("dtype", _I), ("parents", _P), ("workspace", _P),
                ("workspace_bytes", ctypes.c_size_t), ("timing_events", _P * 2)]


class LmArgs(ctypes.Structure):
    _fields_ = [("hidden", _P), ("lm_head", _P), ("tokens", _P), ("mode", _P), ("temperature", _P),
                ("q_draft", _P), ("seed", ctypes.c_uint64), ("out_tokens", _P), ("num_accepted", _P),
                ("tie_flags", _P), ("lse_out", _P), ("argmax_out", _P), ("logits_debug", _P),
                ("B", _I), ("D", _I), ("H", _I), ("V", _I), ("dtype", _I), ("any_sampling", _I),
                ("relaxed_topk", _I), ("relaxed_delta", ctypes.c_float), ("parents", _P), ("accepted_nodes", _P),
                ("workspace", _P), ("workspace_bytes", ctypes.c_size_t), ("timing_events", _P * 2),
                ("q_ready_event", _P)]


class DraftArgs(ctypes.Structure):
    _fields_ = [("hidden", _P), ("lm_head", _P), ("out_tokens", _P), ("lse_out", _P), ("B", _I), ("H", _I),
                ("V", _I), ("dtype", _I), ("workspace", _P), ("workspace_bytes", ctypes.c_size_t),
                ("timing_events", _P * 2)]


class KvCompactArgs(ctypes.Structure):
    _fields_ = [("k_cache", _P), ("v_cache", _P), ("block_table", _P), ("ctx_lens", _P), ("accepted_nodes", _P),
                ("num_accepted", _P), ("B", _I), ("D", _I), ("Hkv", _I), ("d_qk", _I), ("d_v", _I),
                ("block_size", _I), ("max_blocks", _I), ("num_blocks", _I), ("is_mla", _I), ("dtype", _I)]


class RollbackArgs(ctypes.Structure):
    _fields_ = [("block_table", _P), ("seq_lens", _P), ("num_accepted", _P), ("free_list", _P),
                ("free_count", _P), ("B", _I), ("D", _I), ("block_size", _I), ("max_blocks", _I),
                ("free_capacity", _I)]


class MtpError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("mtp status %d: %s" % (code, msg))
        self.code = code


_lib = None


def lib():
    """Load libmtpverify.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmtpverify.so is not built (run __graft_entry__.build() or "
                               "python -m mtp_speculative_decoding_verify_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        L.mtp_verify_attention.argtypes = [ctypes.POINTER(AttnArgs), _P]
        L.mtp_verify_attention.restype = ctypes.c_int
        L.mtp_attention_workspace_size.argtypes = [ctypes.POINTER(AttnArgs)]
        L.mtp_attention_workspace_size.restype = ctypes.c_size_t
        L.mtp_verify_logits_accept.argtypes = [ctypes.POINTER(LmArgs), _P]
        L.mtp_verify_logits_accept.restype = ctypes.c_int
        L.mtp_lmhead_workspace_size.argtypes = [ctypes.POINTER(LmArgs)]
        L.mtp_lmhead_workspace_size.restype = ctypes.c_size_t
        L.kv_rollback.argtypes = [ctypes.POINTER(RollbackArgs), _P]
        L.kv_rollback.restype = ctypes.c_int
        L.mtp_last_error.argtypes = []
        L.mtp_last_error.restype = ctypes.c_char_p
        L.mtp_sync_status.argtypes = [_P]
        L.mtp_sync_status.restype = ctypes.c_int
        L.mtp_rng_debug.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                    ctypes.c_uint32, ctypes.c_int32, _P, _P, _P, _P]
        L.mtp_rng_debug.restype = ctypes.c_int
        L.mtp_wait_selftest.argtypes = [ctypes.c_uint64, _P]
        L.mtp_wait_selftest.restype = ctypes.c_int
        L.mtp_verify_logits_accept_noalloc.argtypes = [ctypes.POINTER(LmArgs), _P]
        L.mtp_verify_logits_accept_noalloc.restype = ctypes.c_int
        L.mtp_noalloc_scratch_bytes.argtypes = []
        L.mtp_noalloc_scratch_bytes.restype = ctypes.c_size_t
        L.mtp_last_launch_count.argtypes = []
        L.mtp_last_launch_count.restype = ctypes.c_int
        L.mtp_draft_workspace_size.argtypes = [ctypes.POINTER(DraftArgs)]
        L.mtp_draft_workspace_size.restype = ctypes.c_size_t
        L.mtp_draft_argmax.argtypes = [ctypes.POINTER(DraftArgs), _P]
        L.mtp_draft_argmax.restype = ctypes.c_int
        L.mtp_tree_kv_compact.argtypes = [ctypes.POINTER(KvCompactArgs), _P]
        L.mtp_tree_kv_compact.restype = ctypes.c_int
        L.mtp_hbm_read_probe.argtypes = [_P, ctypes.c_size_t, _P, ctypes.c_int32, ctypes.c_int32, _P]
        L.mtp_hbm_read_probe.restype = ctypes.c_int
        L.mtp_abi_version.argtypes = []
        L.mtp_abi_version.restype = ctypes.c_int
        L.mtp_abi_struct_size.argtypes = [ctypes.c_int]
        L.mtp_abi_struct_size.restype = ctypes.c_size_t
        if L.mtp_abi_version() != ABI_VERSION:
            raise RuntimeError("library ABI version %d, binding expects %d" % (L.mtp_abi_version(), ABI_VERSION))
        for which, st in enumerate((AttnArgs, LmArgs, RollbackArgs, DraftArgs, KvCompactArgs)):
            if L.mtp_abi_struct_size(which) != ctypes.sizeof(st):
                raise RuntimeError("ABI mismatch for %s" % st.__name__)
        _lib = L
    return _lib


def _check(rc):
    if rc != MTP_OK:
        raise MtpError(rc, lib().mtp_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _dtype_code(t):
    if t.dtype == torch.float32:
        return MTP_F32
    if t.dtype == torch.bfloat16:
        return MTP_BF16
    raise ValueError("tensors must be float32 or bfloat16, got %s" % t.dtype)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_ws_cache = {}


def _workspace(nbytes, device, key):
    """A cached device buffer of at least nbytes (torch allocator), 256-byte aligned."""
    buf = _ws_cache.get((device, key))
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[(device, key)] = buf
    return buf


def attn_args(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, out, *, sm_scale=None, workspace=None,
              parents=None):
    """Fill AttnArgs from tensors (see mtp_verify_attention for shapes)."""
    is_mla = v_cache is None
    B, R, Hq, d_qk = q.shape
    D = R - 1
    dt = q.dtype
    if is_mla:
        num_blocks, bs, Hkv, dk = k_cache.shape
        d_v = out.shape[-1]
        _dev(k_new, "k_new", dt, (B, R, d_qk))
    else:
        num_blocks, bs, Hkv, dk = k_cache.shape
        d_v = v_cache.shape[-1]
        _dev(k_new, "k_new", dt, (B, R, Hkv, d_qk))
        _dev(v_new, "v_new", dt, (B, R, Hkv, d_v))
        _dev(v_cache, "v_cache", dt, (num_blocks, bs, Hkv, d_v))
    _dev(q, "q", dt)
    _dev(k_cache, "k_cache", dt)
    _dev(out, "out", dt, (B, R, Hq, d_v))
    _dev(block_table, "block_table", torch.int32)
    _dev(ctx_lens, "ctx_lens", torch.int32, (B,))
    _dev(parents, "parents", torch.int32, (B, R))
    if dk != d_qk:
        raise ValueError("k_cache head dim %d != q head dim %d" % (dk, d_qk))
    a = AttnArgs(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                 _ptr(ctx_lens), _ptr(out), B, D, Hq, Hkv, d_qk, d_v, bs, block_table.shape[1], num_blocks,
                 int(is_mla), float(sm_scale if sm_scale is not None else d_qk ** -0.5), _dtype_code(q),
                 _ptr(parents), None, 0)
    n = lib().mtp_attention_workspace_size(ctypes.byref(a))
    if n == 0:
        _check(MTP_INVALID_ARG)
    if workspace is None:
        workspace = _workspace(n, q.device, "attn")
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def mtp_verify_attention(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, out, *, sm_scale=None,
                         workspace=None, stream=None, parents=None):
    """Append the verify tokens' K/V to the paged cache and run verify attention into `out`.

    q [B, R, Hq, d_qk]; GQA/MHA: k_new [B, R, Hkv, d], v_new [B, R, Hkv, d], caches [blocks, 64, Hkv, d];
    absorbed MLA: k_new [B, R, 576], v_new = v_cache = None, k_cache [blocks, 64, 1, 576];
    block_table [B, max_blocks] int32, ctx_lens [B] int32, out [B, R, Hq, d_v];
    parents [B, R] int32 (tree drafts) or None (chains).
    """
    a = attn_args(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, out, sm_scale=sm_scale,
                  workspace=workspace, parents=parents)
    _check(lib().mtp_verify_attention(ctypes.byref(a), _stream_handle(stream)))


def lm_args(hidden, lm_head, tokens, mode, temperature, q_draft, seed, out_tokens, num_accepted, tie_flags,
            lse_out=None, argmax_out=None, logits_debug=None, workspace=None, relaxed_topk=0, relaxed_delta=0.0,
            parents=None, accepted_nodes=None):
    """Fill LmArgs from tensors (see mtp_verify_logits_accept for shapes)."""
    B, R = tokens.shape
    D = R - 1
    V, H = lm_head.shape
    dt = lm_head.dtype
    any_sampling = q_draft is not None
    _dev(hidden, "hidden", dt, (B * R, H))
    _dev(lm_head, "lm_head", dt)
    _dev(tokens, "tokens", torch.int32)
    _dev(mode, "mode", torch.uint8, (B,))
    _dev(temperature, "temperature", torch.float32, (B,))
    _dev(q_draft, "q_draft", torch.float32, (B, D, V))
    _dev(out_tokens, "out_tokens", torch.int32, (B, R))
    _dev(num_accepted, "num_accepted", torch.int32, (B,))
    _dev(tie_flags, "tie_flags", torch.uint8, (B,))
    _dev(lse_out, "lse_out", torch.float32, (B, R))
    _dev(argmax_out, "argmax_out", torch.int32, (B, R))
    _dev(logits_debug, "logits_debug", torch.float32, (B * R, V))
    _dev(parents, "parents", torch.int32, (B, R))
    _dev(accepted_nodes, "accepted_nodes", torch.int32, (B, R))
    a = LmArgs(_ptr(hidden), _ptr(lm_head), _ptr(tokens), _ptr(mode), _ptr(temperature), _ptr(q_draft),
               int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out_tokens), _ptr(num_accepted), _ptr(tie_flags), _ptr(lse_out),
               _ptr(argmax_out), _ptr(logits_debug), B, D, H, V, _dtype_code(lm_head), int(any_sampling),
               int(relaxed_topk), float(relaxed_delta), _ptr(parents), _ptr(accepted_nodes), None, 0)
    n = lib().mtp_lmhead_workspace_size(ctypes.byref(a))
    if n == 0:
        _check(MTP_INVALID_ARG)
    if workspace is None:
        workspace = _workspace(n, hidden.device, "lm")
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def mtp_verify_logits_accept(hidden, lm_head, tokens, mode, temperature, q_draft, seed, out_tokens, num_accepted,
                             tie_flags, lse_out=None, argmax_out=None, logits_debug=None, workspace=None,
                             stream=None, relaxed_topk=0, relaxed_delta=0.0, parents=None, accepted_nodes=None,
                             q_ready_event=None):
    """LM head + streaming softmax statistics + greedy / rejection-sampling / relaxed acceptance.

    hidden [B*R, H], lm_head [V, H] (float32 or bfloat16), tokens [B, R] int32, mode [B] uint8,
    temperature [B] float32 or None, q_draft [B, D, V] float32 or None (None: every request greedy),
    outputs out_tokens [B, R] int32, num_accepted [B] int32, tie_flags [B] uint8, optional lse_out / argmax_out
    [B, R] and logits_debug [B*R, V]. relaxed_topk / relaxed_delta: the relaxed rule of mode-2 requests.
    parents [B, R] int32: tree drafts (greedy); accepted_nodes [B, R] int32: optional output, the accepted path.
    q_ready_event: optional torch.cuda.Event recorded after q_draft's copy; the stream waits for it only
    after the LM-head GEMM has been launched, so the copy may overlap the GEMM.
    """
    a = lm_args(hidden, lm_head, tokens, mode, temperature, q_draft, seed, out_tokens, num_accepted, tie_flags,
                lse_out, argmax_out, logits_debug, workspace, relaxed_topk, relaxed_delta, parents, accepted_nodes)
    a.q_ready_event = None if q_ready_event is None else q_ready_event.cuda_event
    _check(lib().mtp_verify_logits_accept(ctypes.byref(a), _stream_handle(stream)))


def draft_args(hidden, lm_head, out_tokens, lse_out=None, workspace=None):
    """Fill DraftArgs from tensors (see mtp_draft_argmax for shapes)."""
    B, H = hidden.shape
    V = lm_head.shape[0]
    dt = lm_head.dtype
    _dev(hidden, "hidden", dt, (B, H))
    _dev(lm_head, "lm_head", dt, (V, H))
    _dev(out_tokens, "out_tokens", torch.int32, (B,))
    _dev(lse_out, "lse_out", torch.float32, (B,))
    a = DraftArgs(_ptr(hidden), _ptr(lm_head), _ptr(out_tokens), _ptr(lse_out), B, H, V, _dtype_code(lm_head),
                  None, 0)
    n = lib().mtp_draft_workspace_size(ctypes.byref(a))
    if n == 0:
        _check(MTP_INVALID_ARG)
    if workspace is None:
        workspace = _workspace(n, hidden.device, "draft")
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def mtp_draft_argmax(hidden, lm_head, out_tokens, lse_out=None, workspace=None, stream=None):
    """One greedy draft step over the shared LM head: out_tokens[b] = argmax_v hidden[b] . lm_head[v]
    (lowest id on ties); hidden [B, H], lm_head [V, H] (float32 or bfloat16), out_tokens [B] int32,
    optional lse_out [B] float32."""
    a = draft_args(hidden, lm_head, out_tokens, lse_out, workspace)
    _check(lib().mtp_draft_argmax(ctypes.byref(a), _stream_handle(stream)))


def mtp_verify_logits_accept_noalloc(hidden, lm_head, tokens, mode, temperature, q_draft, seed, out_tokens,
                                     num_accepted, tie_flags, lse_out=None, argmax_out=None, logits_debug=None,
                                     stream=None, relaxed_topk=0, relaxed_delta=0.0, parents=None,
                                     accepted_nodes=None):
    """mtp_verify_logits_accept for callers that cannot allocate device memory:
    the scratch lives in a fixed array owned by the library (no workspace is
    allocated or passed). Raises MtpError if the batch needs more scratch
    than that array holds. Calls must not overlap on the GPU."""
    a = LmArgs(_ptr(hidden), _ptr(lm_head), _ptr(tokens), _ptr(mode), _ptr(temperature), _ptr(q_draft),
               int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out_tokens), _ptr(num_accepted), _ptr(tie_flags), _ptr(lse_out),
               _ptr(argmax_out), _ptr(logits_debug), tokens.shape[0], tokens.shape[1] - 1, lm_head.shape[1],
               lm_head.shape[0], _dtype_code(lm_head), int(q_draft is not None), int(relaxed_topk),
               float(relaxed_delta), _ptr(parents), _ptr(accepted_nodes), None, 0)
    for t, n in ((hidden, "hidden"), (lm_head, "lm_head"), (tokens, "tokens"), (mode, "mode"),
                 (temperature, "temperature"), (q_draft, "q_draft"), (out_tokens, "out_tokens"),
                 (num_accepted, "num_accepted"), (tie_flags, "tie_flags"), (lse_out, "lse_out"),
                 (argmax_out, "argmax_out"), (logits_debug, "logits_debug"), (parents, "parents"),
                 (accepted_nodes, "accepted_nodes")):
        _dev(t, n)
    _check(lib().mtp_verify_logits_accept_noalloc(ctypes.byref(a), _stream_handle(stream)))


def compact_args(k_cache, v_cache, block_table, ctx_lens, accepted_nodes, num_accepted):
    """Fill KvCompactArgs from tensors (see mtp_tree_kv_compact)."""
    B, R = accepted_nodes.shape
    is_mla = v_cache is None
    num_blocks, bs, Hkv, d_qk = k_cache.shape
    d_v = d_qk if is_mla else v_cache.shape[-1]
    dt = k_cache.dtype
    _dev(k_cache, "k_cache", dt)
    _dev(v_cache, "v_cache", dt, (num_blocks, bs, Hkv, d_v))
    _dev(block_table, "block_table", torch.int32)
    _dev(ctx_lens, "ctx_lens", torch.int32, (B,))
    _dev(accepted_nodes, "accepted_nodes", torch.int32, (B, R))
    _dev(num_accepted, "num_accepted", torch.int32, (B,))
    return KvCompactArgs(_ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), _ptr(accepted_nodes),
                         _ptr(num_accepted), B, R - 1, Hkv, d_qk, d_v, bs, block_table.shape[1], num_blocks,
                         int(is_mla), _dtype_code(k_cache))


def mtp_tree_kv_compact(k_cache, v_cache, block_table, ctx_lens, accepted_nodes, num_accepted, stream=None):
    """Move each request's accepted tree path K/V (accepted_nodes [B, R], num_accepted [B]) to slots
    ctx+1 .. ctx+n of the paged cache (ctx_lens = context lengths before the step); v_cache None for MLA."""
    a = compact_args(k_cache, v_cache, block_table, ctx_lens, accepted_nodes, num_accepted)
    _check(lib().mtp_tree_kv_compact(ctypes.byref(a), _stream_handle(stream)))


def rollback_args(block_table, seq_lens, num_accepted, free_list, free_count, *, D):
    B, max_blocks = block_table.shape
    _dev(block_table, "block_table", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32, (B,))
    _dev(num_accepted, "num_accepted", torch.int32, (B,))
    _dev(free_list, "free_list", torch.int32)
    _dev(free_count, "free_count", torch.int32, (1,))
    return RollbackArgs(_ptr(block_table), _ptr(seq_lens), _ptr(num_accepted), _ptr(free_list), _ptr(free_count),
                        B, D, BLOCK_SIZE, max_blocks, free_list.numel())


def kv_rollback(block_table, seq_lens, num_accepted, free_list, free_count, *, D, stream=None):
    """Truncate each request to ctx + n + 1 slots and release blocks holding only rejected drafts."""
    a = rollback_args(block_table, seq_lens, num_accepted, free_list, free_count, D=D)
    _check(lib().kv_rollback(ctypes.byref(a), _stream_handle(stream)))


def sync_status(stream=None):
    """Synchronise the stream and raise MtpError if a device-side range check tripped."""
    _check(lib().mtp_sync_status(_stream_handle(stream)))


def rng_debug(seed, b, j, tag, v0, n, device="cuda", stream=None):
    """Philox stream check: (word0 uint32 as int64, race exponential, accept uniform) for v = v0 .. v0+n-1."""
    w = torch.empty(n, dtype=torch.int32, device=device)
    e = torch.empty(n, dtype=torch.float32, device=device)
    u = torch.empty(n, dtype=torch.float32, device=device)
    _check(lib().mtp_rng_debug(int(seed), b, j, tag, v0, n, _ptr(w), _ptr(e), _ptr(u), _stream_handle(stream)))
    return w.cpu().numpy().view("uint32"), e.cpu().numpy(), u.cpu().numpy()


def wait_selftest(timeout_ns, stream=None):
    """Run the kernels' bounded mbarrier wait on a barrier nothing arrives on
    (it must give up after timeout_ns and flag a timeout)."""
    _check(lib().mtp_wait_selftest(int(timeout_ns), _stream_handle(stream)))


def hbm_read_probe(buf, sink, ctas_per_sm=2, bulk=False, stream=None):
    """Stream the bytes of device tensor `buf` once (read-bandwidth probe), by
    16-byte loads or (bulk=True) bulk copies into shared memory; `sink` is a
    1-element int32 device tensor that receives an XOR of the data."""
    _check(lib().mtp_hbm_read_probe(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink), int(ctas_per_sm),
                                    int(bool(bulk)), _stream_handle(stream)))
