#!/usr/bin/env python
"""Benchmark of one MTP verify step on GB300.

A step is the whole verify path for one batch: mtp_verify_attention (KV
append + multi-query verify attention), mtp_verify_logits_accept (LM head
with streaming softmax statistics + acceptance) and kv_rollback, on seeded
synthetic inputs already resident in HBM. The default workload is the
largest one-GPU batch: B=256 requests, D=3 drafts, GQA 32 query / 8 KV heads
x 128, contexts 1k-32k tokens in 64-token pages (17.7 GB of KV cache), hidden
4096, vocabulary 151936, bf16; half the requests greedy, half rejection
sampling at temperature 0.7.

Output: one JSON line on rank 0 with requests/s (value), accepted tokens/s,
the roofline of the dominant kernel (and of the other large one), an
end-to-end number through the C ABI with host buffers, and a CPU baseline
(the oracle on a bounded sample).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own batch
(requests are independent, so the step shards by request with no
collective); value = total requests of all ranks / max-over-ranks time.
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mtp_speculative_decoding_verify_gb300 import synth  # noqa: E402

METRIC = "verify-step requests/s and accepted tokens/s on 1 GB300; % of HBM/TC roofline"
DRAFT_METRIC = "draft-step requests/s (D sequential greedy LM-head calls) on 1 GB300; % of HBM/TC roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HBM_NOMINAL_GBS = 7900.0   # GB300 HBM3e, nominal


def workloads():
    return {
        "cfg1_D3": synth.CFG1,
        "cfg1_D1": synth.CFG1.with_(D=1),
        # Tree drafts (full tree of 15 drafts: 3 at the root, 2 under each, then chains), greedy.
        "tree_cfg0": synth.CFG0.with_(name="tiny fp32 MHA with random draft trees: B=4 D=7 ctx=128 H=512 V=8192",
                                      D=7, tree="random"),
        "tree_cfg1_D15": synth.CFG1.with_(name=synth.CFG1.name.replace("D=3", "tree of 15 drafts (3x2x1 fan-out)"),
                                          D=15, tree="full"),
        "tree_cfg3_D15": synth.CFG3.with_(name=synth.CFG3.name.replace("D=3", "tree of 15 drafts (3x2x1 fan-out)"),
                                          D=15, tree="full", sampling="none"),
        # Relaxed acceptance (top-10, delta 0.6) on the DeepSeek-V3-shaped step.
        "cfg1_D3_relaxed": synth.CFG1.with_(name=synth.CFG1.name + ", relaxed acceptance N=10 delta=0.6",
                                            relaxed="all", relaxed_topk=10, relaxed_delta=0.6),
        "cfg0": synth.CFG0,
        "cfg2": synth.CFG2,
        "cfg3": synth.CFG3,
        **{"sweep_B%d_D%d" % (B, D): synth.sweep_point(B, D) for B in (1, 8, 64, 256, 512) for D in (1, 3, 5, 7)},
        # Reduced cases for profiler captures (inputs still larger than L2).
        "profile_mla_V32k": synth.CFG1.with_(name="profiling case: DeepSeek-V3-shaped MLA B=32 D=3, vocab 32768",
                                             V=32768),
        "profile_gqa_B16": synth.CFG3.with_(name="profiling case: large-batch mixed GQA, B=16", B=16),
        "profile_gqa_B32_keyparts": synth.CFG3.with_(
            name="profiling case: large-batch mixed GQA, B=32 (grid large enough for key parts)", B=32),
        "profile_tree_mla_V32k": synth.CFG1.with_(name="profiling case: DeepSeek-V3-shaped MLA, trees of 15 drafts, "
                                                       "B=32, vocab 32768", D=15, tree="full", V=32768),
        "profile_tree_gqa_B16": synth.CFG3.with_(name="profiling case: large-batch mixed GQA, trees of 15 drafts, "
                                                      "B=16, vocab 32768", B=16, D=15, tree="full", sampling="none",
                                                 V=32768),
        "profile_lm_cfg3_V64k": synth.CFG3.with_(
            name="profiling case: large-batch mixed LM head M=1024 (B=256 D=3), vocab 65536, contexts 64-128",
            V=65536, ctx=(64, 128)),
        "profile_sampling_V32k": synth.CFG2.with_(
            name="profiling case: Llama-70B-shaped rejection sampling B=64 D=5, vocab 32768", V=32768),
        # MTP-Eagle draft steps: D sequential greedy top-1 calls over the shared LM head, B rows each.
        "draft_cfg0": synth.CFG0.with_(name="MTP-Eagle draft steps, tiny fp32 LM head: B=4, 3 sequential greedy "
                                            "top-1 calls, H=512 V=8192"),
        "draft_cfg1_D3": synth.CFG1.with_(name="MTP-Eagle draft steps, DeepSeek-V3-shaped LM head: B=32, 3 "
                                               "sequential greedy top-1 calls, H=7168 V=129280"),
        "draft_cfg2_D5": synth.CFG2.with_(name="MTP-Eagle draft steps, Llama-70B-shaped LM head: B=64, 5 "
                                               "sequential greedy top-1 calls, H=8192 V=128256"),
    }


def is_draft(name):
    return name.startswith("draft_")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return PEAKS_FALLBACK, "fallback"


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# of a workload's large kernels, from one ncu capture of a reduced case of the
# same kernel and shapes, scaled to the full workload by the units it
# processes (the traffic of both kernels grows in proportion to them: every
# W tile and every KV page is read once). Each entry names the kernel's
# source files and their SHA-256 (first 16 hex digits) at capture time; once
# a source changes, the figure no longer describes the kernel and is dropped.
#   workload -> kernel -> (bytes per unit, unit, sources, digest, capture)
KERNEL_SOURCES = {
    "lm_head": ["lmhead_tc.cu", "common.cuh", "sm100.cuh"],
    "attention": ["attention_mma.cu", "common.cuh", "sm100.cuh", "mma_sync.cuh"],
    "attention_mla": ["attention_mla_tc.cu", "common.cuh", "sm100.cuh"],
}

TRAFFIC = {
    "cfg1_D3": {
        # attn_mla_pair_kernel at the same shapes (profile_mla_V32k): 109.45 MB read + 5.29 MB written for
        # 87.35 MB of latent KV (the rest: the queries, 18.9 MB, and the outputs)
        "attention": ((109451776 + 5287168) / 87353856, "KV-cache bytes", KERNEL_SOURCES["attention_mla"],
                      "be101fe337e05d0e", "ncu capture of attn_mla_pair_kernel (profile_mla_V32k)"),
        # lmhead_tc_kernel<4, true> (CTA pairs) at M=128 with vocabulary 32768 (profile_mla_V32k):
        # 471.69 MB read + 2.82 MB written
        "lm_head": ((471687168 + 2816256) / 32768, "vocabulary rows", KERNEL_SOURCES["lm_head"],
                    "1e081f7967bd35e6",
                    "ncu capture of lmhead_tc_kernel at M=128, vocabulary 32768 (profile_mla_V32k)"),
    },
    "cfg2": {
        # attn_gqa_kernel<128> form 0 at the same shapes (profile_sampling_V32k): 1097.26 MB read
        # + 6.97 MB written for 1075.31 MB of KV cache
        "attention": ((1097258240 + 6973696) / 1075314688, "KV-cache bytes", KERNEL_SOURCES["attention"],
                      "6e5b81293843fbdb", "ncu capture of attn_gqa_kernel (profile_sampling_V32k)"),
        # lmhead_tc_kernel<6, true> at M=384 with vocabulary 32768 (profile_sampling_V32k): 543.31 MB read
        # + 21.74 MB written
        "lm_head": ((543312896 + 21744896) / 32768, "vocabulary rows", KERNEL_SOURCES["lm_head"],
                    "1e081f7967bd35e6",
                    "ncu capture of lmhead_tc_kernel at M=384, vocabulary 32768 (profile_sampling_V32k)"),
    },
    "cfg3": {
        # attn_gqa_kernel<128> on the same shapes at B=16 (profile_gqa_B16): 990.31 MB read + 4.53 MB
        # written for 987.60 MB of KV cache
        "attention": ((990305280 + 4533760) / 987598848, "KV-cache bytes", KERNEL_SOURCES["attention"],
                      "6e5b81293843fbdb", "ncu capture of attn_gqa_kernel at B=16 (profile_gqa_B16)"),
        # lmhead_tc_kernel<8, true> at M=1024 with vocabulary 65536 (profile_lm_cfg3_V64k): 616.33 MB read
        # + 102.73 MB written
        "lm_head": ((616330496 + 102726400) / 65536, "vocabulary rows", KERNEL_SOURCES["lm_head"],
                    "1e081f7967bd35e6", "ncu capture of lmhead_tc_kernel at M=1024, vocabulary 65536 "
                                        "(profile_lm_cfg3_V64k)"),
    },
}



def source_digest(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "mtp_speculative_decoding_verify_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(workload, kernel, units):
    """(DRAM bytes of one launch, note) or (None, why not)."""
    e = TRAFFIC.get(workload, {}).get(kernel)
    if e is None:
        return None, "no capture for this workload"
    per_unit, unit, files, digest, capture = e
    if source_digest(files) != digest:
        return None, "kernel source changed since the capture (%s)" % capture
    return per_unit * units, "%s, scaled by %s" % (capture, unit)


COPY_PIECE_BYTES = 1 << 29


def copy_in_pieces(dst, src):
    """dst.copy_(src) on the current stream, as copies of at most 512 MiB
    (one host-to-device copy of 2.2 GB measured at a third of the rate of
    smaller ones)."""
    per = max(1, COPY_PIECE_BYTES // src.element_size())
    if src.numel() <= per or not (dst.is_contiguous() and src.is_contiguous()):
        dst.copy_(src, non_blocking=True)
        return
    d, s = dst.view(-1), src.view(-1)
    for a in range(0, src.numel(), per):
        d[a:a + per].copy_(s[a:a + per], non_blocking=True)


def elem_bytes(w):
    return 4 if w.dtype == "f32" else 2


def path_lengths(w):
    """[B, R] number of verify keys each row sees: j + 1 for chains, the root-path length for trees."""
    par = synth.make_parents(w)
    if par is None:
        return np.tile(np.arange(1, w.R + 1), (w.B, 1))
    par = par.numpy()
    out = np.ones((w.B, w.R), np.int64)
    for k in range(1, w.R):
        out[:, k] = out[np.arange(w.B), par[:, k]] + 1
    return out


def algorithmic(w, ctx, draft=False):
    """Algorithmic bytes and flops of one step: KV read once (ctx + R keys per
    request and KV head), W read once; flops of the LM head and attention.
    A draft-step workload reads W once per call (D calls, B rows each)."""
    eb = elem_bytes(w)
    if draft:
        return dict(kv_bytes=0.0, w_bytes=float(w.V) * w.H * eb * w.D, attn_flops=0.0,
                    lm_flops=2.0 * w.B * w.H * w.V * w.D, calls=w.D)
    R = w.R
    keys = float(np.sum(ctx + R))
    visible = float(np.sum(ctx[:, None] + path_lengths(w)))   # (row, visible key) pairs per head
    if w.is_mla:
        kv_bytes = keys * w.d_qk * eb
        attn_flops = 2.0 * (w.d_qk + w.d_v) * w.Hq * visible
    else:
        kv_bytes = keys * w.Hkv * (w.d_qk + w.d_v) * eb
        attn_flops = 2.0 * (w.d_qk + w.d_v) * w.Hq * visible
    w_bytes = float(w.V) * w.H * eb
    lm_flops = 2.0 * w.M * w.H * w.V
    return dict(kv_bytes=kv_bytes, w_bytes=w_bytes, attn_flops=attn_flops, lm_flops=lm_flops, calls=1)


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class Step:
    """The three C-ABI calls of one verify step, with argument structs built once."""

    def __init__(self, w, dev, seed_offset=0):
        from mtp_speculative_decoding_verify_gb300 import _binding as B
        self.B = B
        self.L = B.lib()
        self.w = w.with_(seed=w.seed + seed_offset)
        w = self.w
        self.att = synth.make_attention_inputs(w, dev)
        self.lm = synth.make_lmhead_inputs(w, dev)
        att, lm = self.att, self.lm
        self.out = torch.empty((w.B, w.R, w.Hq, w.d_v), dtype=w.torch_dtype, device=dev)
        self.out_tokens = torch.empty((w.B, w.R), dtype=torch.int32, device=dev)
        self.num_acc = torch.empty(w.B, dtype=torch.int32, device=dev)
        self.ties = torch.empty(w.B, dtype=torch.uint8, device=dev)
        # The rollback edits the block table, the lengths and the free-list
        # count in place; they live in one buffer so that a single copy from
        # a pristine image restores them before every step.
        nt, nb = att["block_table"].numel(), w.B
        self.book = torch.empty(nt + nb + 1, dtype=torch.int32, device=dev)
        self.book_init = torch.cat([att["block_table"].reshape(-1), att["ctx_lens"].reshape(-1),
                                    torch.zeros(1, dtype=torch.int32, device=dev)])
        self.book.copy_(self.book_init)
        self.table_work = self.book[:nt].view(att["block_table"].shape)
        self.seq = self.book[nt:nt + nb]
        self.free_list = torch.full((w.B * 2 + 8,), -1, dtype=torch.int32, device=dev)
        self.free_count = self.book[nt + nb:]
        self.parents = lm.get("parents")
        self.acc_nodes = torch.empty((w.B, w.R), dtype=torch.int32, device=dev)
        self.a_attn = B.attn_args(att["q"], att["k_new"], att["v_new"], att["k_cache"], att["v_cache"],
                                  att["block_table"], att["ctx_lens"], self.out, sm_scale=w.sm_scale,
                                  parents=self.parents)
        self.a_lm = B.lm_args(lm["hidden"], lm["lm_head"], lm["tokens"], lm["mode"], lm["temperature"],
                              lm["q_draft"], lm["seed"], self.out_tokens, self.num_acc, self.ties,
                              relaxed_topk=w.relaxed_topk, relaxed_delta=w.relaxed_delta, parents=self.parents,
                              accepted_nodes=self.acc_nodes if self.parents is not None else None)
        # Tree drafts: the accepted path's K/V moves to contiguous slots before the rollback.
        self.a_cmp = None if self.parents is None else B.compact_args(
            att["k_cache"], att["v_cache"], att["block_table"], att["ctx_lens"], self.acc_nodes, self.num_acc)
        self.a_rb = B.rollback_args(self.table_work, self.seq, self.num_acc, self.free_list, self.free_count, D=w.D)
        self.launches = 0

    def set_events(self, attn_pair, lm_pair):
        for args, pair in ((self.a_attn, attn_pair), (self.a_lm, lm_pair)):
            args.timing_events[0] = pair[0].cuda_event if pair else None
            args.timing_events[1] = pair[1].cuda_event if pair else None

    def run(self, stream, before_lm=None):
        """The step's calls on `stream`; before_lm(stream), if given, runs
        between the attention call and the LM-head call."""
        h = ctypes.c_void_p(stream.cuda_stream)
        # Reset the rollback's bookkeeping so every step starts from the same state.
        self.book.copy_(self.book_init)
        L, chk = self.L, self.B._check
        chk(L.mtp_verify_attention(ctypes.byref(self.a_attn), h))
        n = L.mtp_last_launch_count()
        if before_lm is not None:
            before_lm(stream)
        chk(L.mtp_verify_logits_accept(ctypes.byref(self.a_lm), h))
        n += L.mtp_last_launch_count()
        if self.a_cmp is not None:
            chk(L.mtp_tree_kv_compact(ctypes.byref(self.a_cmp), h))
            n += L.mtp_last_launch_count()
        chk(L.kv_rollback(ctypes.byref(self.a_rb), h))
        n += L.mtp_last_launch_count()
        self.launches = n

    # Inputs the attention call reads; the others are read from the LM-head call on.
    ATTENTION_INPUTS = ("q", "k_new", "v_new", "ctx_lens", "parents")

    def host_inputs(self):
        """Device tensors that carry a step's inputs (copied from host memory in
        the e2e timing): the verify rows' queries, keys and values, the context
        lengths, the hidden states, tokens, modes and temperatures, the tree
        parents, and the draft distributions q of the rejection-sampling
        requests (the rows of other requests are never read: only those
        requests' slice is copied when they are contiguous)."""
        d = {"q": self.att["q"], "k_new": self.att["k_new"], "ctx_lens": self.att["ctx_lens"],
             "hidden": self.lm["hidden"], "tokens": self.lm["tokens"], "mode": self.lm["mode"],
             "temperature": self.lm["temperature"]}
        if self.att["v_new"] is not None:
            d["v_new"] = self.att["v_new"]
        if self.parents is not None:
            d["parents"] = self.parents
        q = self.lm["q_draft"]
        if q is not None:
            samp = np.nonzero(self.lm["mode"].cpu().numpy() == 1)[0]
            if len(samp) and samp[-1] - samp[0] + 1 == len(samp):
                d["q_draft"] = q[int(samp[0]):int(samp[-1]) + 1]
            elif len(samp):
                d["q_draft"] = q
        return d

    def results(self):
        return [self.out_tokens, self.num_acc]

    def summary(self):
        n_acc = self.num_acc.cpu().numpy()
        ctx = self.att["ctx_lens"].cpu().numpy().astype(np.int64)
        return n_acc, ctx, float(n_acc.sum() + self.w.B)


class DraftStep:
    """D sequential greedy draft steps of MTP Eagle over the shared LM head
    (mtp_draft_argmax, B rows per call); each call's hidden states are their
    own synthetic input (the MTP module between calls is not part of the path)."""

    def __init__(self, w, dev, seed_offset=0):
        from mtp_speculative_decoding_verify_gb300 import _binding as B
        self.B = B
        self.L = B.lib()
        self.w = w.with_(seed=w.seed + seed_offset)
        w = self.w
        self.inp = synth.make_draft_inputs(w, dev)
        self.tokens = torch.empty((w.D, w.B), dtype=torch.int32, device=dev)
        self.args = [B.draft_args(self.inp["hidden"][k], self.inp["lm_head"], self.tokens[k]) for k in range(w.D)]
        self.launches = 0

    def set_events(self, attn_pair, lm_pair):
        self.args[0].timing_events[0] = lm_pair[0].cuda_event if lm_pair else None
        self.args[0].timing_events[1] = lm_pair[1].cuda_event if lm_pair else None

    ATTENTION_INPUTS = ()

    def run(self, stream, before_lm=None):
        h = ctypes.c_void_p(stream.cuda_stream)
        if before_lm is not None:
            before_lm(stream)
        n = 0
        for a in self.args:
            self.B._check(self.L.mtp_draft_argmax(ctypes.byref(a), h))
            n += self.L.mtp_last_launch_count()
        self.launches = n

    def host_inputs(self):
        return {"hidden": self.inp["hidden"]}

    def results(self):
        return [self.tokens]

    def summary(self):
        return np.zeros(self.w.B, np.int64), np.zeros(self.w.B, np.int64), float(self.w.B * self.w.D)


def combine_ranks(ms, e2e_ms, emitted, world, device):
    """Whole-job figures: the slowest rank's times and the total tokens emitted."""
    if world == 1:
        return ms, e2e_ms, emitted
    t = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    e = torch.tensor([emitted], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(e, op=torch.distributed.ReduceOp.SUM)
    return float(t[0]), float(t[1]), float(e[0])


def event_pairs(n):
    """Timing event pairs; each is recorded once so its CUDA event exists before
    its handle goes into an argument struct."""
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in pairs:
        a.record()
        b.record()
    torch.cuda.synchronize()
    return pairs


def run_gpu(args, w, rank, world, dev):
    stream = torch.cuda.current_stream()
    step = (DraftStep if is_draft(args.workload) else Step)(w, dev, seed_offset=rank)
    for _ in range(args.warmup):
        step.run(stream)
    torch.cuda.synchronize()
    step.B.sync_status()

    K = args.steps
    ev_attn, ev_lm = event_pairs(K), event_pairs(K)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    launches = 0
    for k in range(K):
        step.set_events(ev_attn[k], ev_lm[k])
        step.run(stream)
        launches += step.launches
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    step.set_events(None, None)
    step.B.sync_status()
    ms_eager = t0.elapsed_time(t1) / K

    # The same step captured once in a CUDA graph and replayed K times (the
    # library's calls are capture-safe once each has run on the device).
    graph_ms = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step.run(side)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        sampler2 = ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) if rank == 0 else None
        if sampler2:
            sampler2.start()
            time.sleep(0.3)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(K):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        clocks_g = sampler2.stop() if sampler2 else None
        step.B.sync_status()
        graph_ms = g0.elapsed_time(g1) / K
        if clocks_g:
            clocks = clocks_g
    ms = graph_ms if graph_ms is not None else ms_eager
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_attn) if not is_draft(args.workload) else 0.0
    lm_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_lm)
    n_acc, ctx, emitted = step.summary()
    ties = step.ties.cpu().numpy() if hasattr(step, "ties") else np.zeros(0, np.uint8)

    # End to end through the public API with host buffers: each step copies its
    # inputs from pinned host memory, runs the calls and reads the results back.
    dev_t = step.host_inputs()
    host = {k: t.cpu().pin_memory() for k, t in dev_t.items()}
    res_dev = step.results()
    res_host = [torch.empty_like(t, device="cpu").pin_memory() for t in res_dev]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in res_host)
    for _ in range(max(1, args.warmup // 2)):
        step.run(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # A step's inputs cross in three groups: what the attention reads, on the
    # step's stream before the attention call; what the LM head reads (hidden
    # states, tokens, modes, ...), on a second stream during the attention,
    # which the LM-head call waits for; and the draft distributions q, read
    # only by the acceptance kernels, on that stream after them: the library
    # waits for their event (q_ready_event) only once the LM-head GEMM has
    # been launched, so q's copy overlaps the attention and the GEMM.
    first = {k: t for k, t in host.items() if k in step.ATTENTION_INPUTS}
    later = {k: t for k, t in host.items() if k not in step.ATTENTION_INPUTS and k != "q_draft"}
    qcopy = {k: t for k, t in host.items() if k == "q_draft"}
    copy_stream = torch.cuda.Stream()
    ev_lm, ev_q = torch.cuda.Event(), torch.cuda.Event()

    def e2e_step(st):
        for k, t in first.items():
            copy_in_pieces(dev_t[k], t)
        copy_stream.wait_stream(st)
        with torch.cuda.stream(copy_stream):
            for k, t in later.items():
                copy_in_pieces(dev_t[k], t)
            ev_lm.record(copy_stream)
            for k, t in qcopy.items():
                copy_in_pieces(dev_t[k], t)
            ev_q.record(copy_stream)
        if hasattr(step, "a_lm"):
            step.a_lm.q_ready_event = ev_q.cuda_event if qcopy else None
        step.run(st, before_lm=lambda s2: s2.wait_event(ev_lm if hasattr(step, "a_lm") else ev_q))
        st.wait_stream(copy_stream)
        for th, td in zip(res_host, res_dev):
            th.copy_(td, non_blocking=True)

    # With graphs on, the copies from and to pinned host memory and the calls
    # are captured together once and replayed, as a serving loop would.
    g_e2e = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e, stream=side):
                e2e_step(side)
        torch.cuda.synchronize()
        for _ in range(max(1, args.warmup // 2)):
            g_e2e.replay()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e2e_t0 = time.perf_counter()
    for _ in range(K):
        if g_e2e is not None:
            g_e2e.replay()
        else:
            e2e_step(stream)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - e2e_t0) * 1e3 / K
    if hasattr(step, "a_lm"):
        step.a_lm.q_ready_event = None

    ms, e2e_ms, emitted = combine_ranks(ms, e2e_ms, emitted, world, dev)
    ms_eager, _, _ = combine_ranks(ms_eager, 0.0, 0.0, world, dev)
    return dict(ms=ms, ms_eager=ms_eager, graph=graph_ms is not None, e2e_graph=g_e2e is not None, e2e_ms=e2e_ms, attn_ms=attn_ms, lm_ms=lm_ms, emitted=emitted, n_acc=n_acc, ctx=ctx,
                clocks=clocks, launches=launches, h2d=h2d, d2h=d2h, ties=ties)


def decode_baseline(args, w, dev):
    """The same workload with D = 0 (a plain decode step: one query row per
    request, greedy top-1), graph-replayed like the verify step; gives the
    verify/decode cost ratio."""
    wd = w.with_(D=0, relaxed="none", relaxed_topk=0, tree="chain")
    step = Step(wd, dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.run(stream)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step.run(side)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    step.B.sync_status()
    return t0.elapsed_time(t1) / args.steps


def read_ceiling(dev, gib=4, reps=5):
    """Read-only bandwidth of this GPU (GB/s): the library's read probe
    streaming a buffer far larger than L2, by loads and by bulk copies, timed
    with CUDA events; the best over paths, launch shapes and repetitions, and
    the best of each path."""
    from mtp_speculative_decoding_verify_gb300 import _binding as B
    buf = torch.empty(gib << 30, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    best = {}
    for bulk, ctas in ((False, 1), (False, 2), (False, 4), (True, 1)):
        key = "bulk_copies" if bulk else "loads"
        for k in range(3 + reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            B.hbm_read_probe(buf, sink, ctas, bulk, stream)
            b.record(stream)
            b.synchronize()
            if k >= 3:
                best[key] = max(best.get(key, 0.0), buf.numel() / (a.elapsed_time(b) * 1e-3) / 1e9)
    B.sync_status()
    del buf
    return max(best.values()), best


def cpu_model():
    """Host CPU model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def _timed_requests(fn, n_items, seconds, threads):
    """Run fn(i) for i = 0, 1, ... (at most n_items) on `threads` threads until
    `seconds` have passed (each thread finishes the request it is in); returns
    (requests done, elapsed seconds)."""
    import concurrent.futures as cf
    import itertools
    t0 = time.perf_counter()
    stop = t0 + seconds
    counter = itertools.count()

    def worker():
        n = 0
        while time.perf_counter() < stop:
            i = next(counter)
            if i >= n_items:
                break
            fn(i)
            n += 1
        return n
    with cf.ThreadPoolExecutor(threads) as ex:
        done = sum(f.result() for f in [ex.submit(worker) for _ in range(threads)])
    return done, time.perf_counter() - t0


def cpu_baseline(w, seconds, dev=None, draft=False):
    """The oracle, as it stands, on a bounded sample of the same workload:
    whole requests (attention + LM head + acceptance + KV compaction for trees
    + rollback, or the D draft steps), first on one thread, then on every host
    core (one unmodified single-threaded oracle call per request and thread;
    the calls release the interpreter lock)."""
    from oracle import requests as oreq
    gen_dev = dev if dev is not None else torch.device("cpu")
    if draft:
        inp = synth.make_draft_inputs(w, gen_dev)
        W = synth.as_oracle_array(inp["lm_head"])
        fn = lambda i: oreq.draft_request(w, inp, W, i % w.B)  # noqa: E731
        what = "%d greedy draft steps each" % w.D
    else:
        att = synth.make_attention_inputs(w, gen_dev)
        lm = synth.make_lmhead_inputs(w, gen_dev)
        W = synth.as_oracle_array(lm["lm_head"])
        table = synth.as_oracle_array(att["block_table"])
        ctx = synth.as_oracle_array(att["ctx_lens"])
        fn = lambda i: oreq.whole_request(w, att, lm, W, table, ctx, i % w.B)  # noqa: E731
        what = "attention + LM head + acceptance + rollback"
    n1, el1 = _timed_requests(fn, 4 * w.B, seconds, 1)
    cores = os.cpu_count() or 1
    nc, elc = _timed_requests(fn, 4 * w.B, seconds, cores)
    return dict(value=nc / elc, unit="requests/s", cores=cores, cpu_model=cpu_model(), kind="oracle",
                sample="%d request(s) of the %d-request batch (%s), the single-threaded oracle on %d threads, one "
                       "request per thread at a time, %.1f s" % (nc, w.B, what, cores, elc),
                single_thread=dict(value=n1 / el1, unit="requests/s", cores=1,
                                   sample="%d request(s), one thread, %.1f s" % (n1, el1)))


def json_line(**kw):
    print(json.dumps(kw), flush=True)


def run_reference(args, w, rank, world):
    """Reference arm: the CPU oracle on the host cores. Each step is a bounded
    sample of the same workload: one whole request per host core, each on its
    own thread running the unmodified single-threaded oracle."""
    if rank != 0:
        return
    import concurrent.futures as cf
    from oracle import requests as oreq
    gen_dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0"))) if torch.cuda.is_available() else "cpu"
    draft = is_draft(args.workload)
    if draft:
        inp = synth.make_draft_inputs(w, gen_dev)
        Wd = synth.as_oracle_array(inp["lm_head"])
        one = lambda b: oreq.draft_request(w, inp, Wd, b)  # noqa: E731
        what = "%d greedy draft steps" % w.D
    else:
        att = synth.make_attention_inputs(w, gen_dev)
        lm = synth.make_lmhead_inputs(w, gen_dev)
        W = synth.as_oracle_array(lm["lm_head"])
        table = synth.as_oracle_array(att["block_table"])
        ctx = synth.as_oracle_array(att["ctx_lens"])
        one = lambda b: oreq.whole_request(w, att, lm, W, table, ctx, b)  # noqa: E731
        what = "attention + LM head + acceptance + rollback"
    cores = os.cpu_count() or 1
    with cf.ThreadPoolExecutor(cores) as ex:
        def step(k):
            list(ex.map(one, [(k * cores + c) % w.B for c in range(cores)]))
        for k in range(args.warmup):
            step(k)
        t0 = time.perf_counter()
        for k in range(args.steps):
            step(args.warmup + k)
        el = time.perf_counter() - t0
    rps = args.steps * cores / el
    sample = "%d requests per step (one per host core) of the %d-request batch (%s), the single-threaded " \
             "oracle on each of %d threads" % (cores, w.B, what, cores)
    json_line(impl="reference", metric=DRAFT_METRIC if draft else METRIC, value=rps, unit="requests/s",
              n_gpus=world, steps=args.steps, warmup=args.warmup, ms_per_step=el * 1e3 / args.steps,
              higher_is_better=True, scaling="weak", vs_baseline=None, dtype=w.dtype, data="synthetic",
              config=config_of(w, args),
              cpu_baseline=dict(value=rps, unit="requests/s", cores=cores, cpu_model=cpu_model(), kind="oracle",
                                sample=sample),
              e2e=dict(value=rps, unit="requests/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def config_of(w, args):
    return {"workload": w.name, "B": w.B, "D": w.D, "parallelism": "request-sharded replicas",
            "l2": "inputs larger than L2 (LM-head weights %.2f GB streamed every step)" % (w.V * w.H * elem_bytes(w) / 1e9)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="cfg3", choices=sorted(workloads()))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches only (no CUDA-graph replay)")
    ap.add_argument("--no-decode-baseline", action="store_true",
                    help="skip timing the same workload at D = 0 (verify/decode cost ratio)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = workloads()[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)

    draft = is_draft(args.workload)
    r = run_gpu(args, w, rank, world, dev)
    decode_ms = None
    if not draft and w.D > 0 and not args.no_decode_baseline:
        decode_ms = decode_baseline(args, w, dev)
    if rank != 0:
        torch.distributed.destroy_process_group() if world > 1 else None
        return
    peaks, src = load_peaks()
    alg = algorithmic(w, r["ctx"], draft)
    hbm = float(peaks["hbm_gbs"])
    tc_peak = float(peaks["bf16_tflops"])
    ceiling, ceiling_by_path = read_ceiling(dev)
    calls = alg["calls"]   # LM-head launches per step; the events time one of them

    def hbm_roof(kernel, nbytes, ms, units, unit_name):
        a = nbytes / (ms * 1e-3) / 1e9
        t, note = traffic_of(args.workload, kernel, units)
        return dict(kernel=kernel, bound="hbm", achieved=a, peak=hbm, unit="GB/s", frac=a / hbm,
                    peak_source=src + " (hbm_gbs: device-to-device copy)",
                    read_ceiling=ceiling, read_ceiling_by_path=ceiling_by_path, frac_of_read_ceiling=a / ceiling,
                    frac_of_nominal=a / HBM_NOMINAL_GBS, algorithmic_bytes=nbytes,
                    unit_of_work=unit_name, traffic=t, traffic_note=note, avg_launch_ms=ms)

    def tc_roof(kernel, flops, ms, units, unit_name):
        a = flops / (ms * 1e-3) / 1e12
        t, note = traffic_of(args.workload, kernel, units)
        return dict(kernel=kernel, bound="tensor", achieved=a, peak=tc_peak, unit="TFLOP/s", frac=a / tc_peak,
                    peak_source=src + " (bf16_tflops burst)", algorithmic_flops=flops, unit_of_work=unit_name,
                    traffic=t, traffic_note=note, avg_launch_ms=ms)

    # LM head: HBM-bound on W below M ~ 290 rows, tensor-bound above.
    ridge = tc_peak * 1e12 / (hbm * 1e9)
    w_call = alg["w_bytes"] / calls
    if alg["lm_flops"] / alg["w_bytes"] < ridge or w.dtype == "f32":
        lm_roof = hbm_roof("lm_head", w_call, r["lm_ms"], w.V, "vocabulary rows (W bytes V*H*2 per launch)")
    else:
        lm_roof = tc_roof("lm_head", alg["lm_flops"] / calls, r["lm_ms"], w.V,
                          "vocabulary rows (2*M*H flop each)")
    roofs = {"lm_head": lm_roof}
    if not draft:
        if w.is_mla:
            roofs["attention"] = tc_roof("attention", alg["attn_flops"], r["attn_ms"], alg["kv_bytes"],
                                         "(row, visible key) pairs (2*(d_qk+d_v)*Hq flop each)")
        else:
            roofs["attention"] = hbm_roof("attention", alg["kv_bytes"], r["attn_ms"], alg["kv_bytes"],
                                          "KV-cache bytes ((ctx+R)*Hkv*(d_qk+d_v)*2 per request)")
    dominant = max(roofs, key=lambda k: roofs[k]["avg_launch_ms"])
    roof = roofs[dominant]
    step_bound_s = max((alg["kv_bytes"] + alg["w_bytes"]) / (hbm * 1e9),
                       (alg["lm_flops"] + alg["attn_flops"]) / (tc_peak * 1e12))
    per_kernel_s = (alg["kv_bytes"] / (hbm * 1e9) if not w.is_mla else alg["attn_flops"] / (tc_peak * 1e12)) + \
        (lm_roof["algorithmic_bytes"] / (hbm * 1e9) if lm_roof["bound"] == "hbm"
         else lm_roof["algorithmic_flops"] / (tc_peak * 1e12)) * calls
    ties = r["ties"]
    value = world * w.B / (r["ms"] * 1e-3)
    if draft:
        kernels = dict(lm_head_ms_per_call=r["lm_ms"], calls_per_step=calls)
    else:
        kernels = dict(attention_ms=r["attn_ms"], attention_gbs=alg["kv_bytes"] / (r["attn_ms"] * 1e-3) / 1e9,
                       attention_tflops=alg["attn_flops"] / (r["attn_ms"] * 1e-3) / 1e12, lm_head_ms=r["lm_ms"])
    line = dict(metric=DRAFT_METRIC if draft else METRIC, value=value, unit="requests/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
                ms_per_step=r["ms"], ms_per_step_eager=r["ms_eager"], higher_is_better=True, scaling="weak", vs_baseline=None, dtype=w.dtype,
                data="synthetic (seeded; random-init weights of the named shapes)", config=config_of(w, args),
                accepted_tokens_per_s=r["emitted"] / (r["ms"] * 1e-3),
                mean_drafts_accepted=float(np.mean(r["n_acc"])),
                cuda_graph=r["graph"],
                roofline=roof,
                roofline_kernels=roofs,
                step_roofline=dict(bound_ms=step_bound_s * 1e3, frac=step_bound_s * 1e3 / r["ms"],
                                   sum_of_kernel_bounds_ms=per_kernel_s * 1e3,
                                   frac_of_sum_of_kernel_bounds=per_kernel_s * 1e3 / r["ms"],
                                   kv_gb=alg["kv_bytes"] / 1e9, w_gb=alg["w_bytes"] / 1e9,
                                   gflop=(alg["lm_flops"] + alg["attn_flops"]) / 1e9),
                near_ties=dict(requests=int(len(ties)), accept_or_relaxed_band=int(((ties & 1) != 0).sum()),
                               race=int(((ties & 2) != 0).sum()),
                               note="requests whose decision the tie flags mark as within the near-tie band "
                                    "(bit-exact comparison with the oracle excludes them)"),
                kernels=kernels,
                e2e=dict(value=world * w.B / (r["e2e_ms"] * 1e-3), unit="requests/s", h2d_bytes_per_step=r["h2d"],
                         d2h_bytes_per_step=r["d2h"], ms_per_step=r["e2e_ms"],
                         path="pinned host inputs -> device (the attention's inputs first; the LM head's on a "
                              "second stream during the attention, then q of the sampling requests, which the "
                              "library waits for after launching the LM-head GEMM), "
                              "the library calls, results -> pinned host, "
                              + ("captured once as a CUDA graph and replayed" if r["e2e_graph"] else "eager")
                              + ", host wall clock per step including the synchronize"),
                gpu_launches=r["launches"], clocks=r["clocks"])
    if draft:
        for k in ("accepted_tokens_per_s", "mean_drafts_accepted"):
            line.pop(k)
        line["draft_tokens_per_s"] = r["emitted"] / (r["ms"] * 1e-3)
    line["graph_speedup"] = r["ms_eager"] / r["ms"] if r["graph"] else None
    if decode_ms is not None:
        line["decode_baseline"] = dict(workload=w.name + ", D=0", ms_per_step=decode_ms,
                                       verify_over_decode=r["ms"] / decode_ms)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, dev, draft)
    json_line(**line)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
