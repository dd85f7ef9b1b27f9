#!/usr/bin/env python3
"""Benchmark of the paged-KV attention hot path on GB300.

One *step* is one pass of the hot path over one batch of synthetic input held
in HBM.  The headline workload is the batched GQA split-KV decode (batch 64,
32 q heads / 8 KV heads, head_dim 128, page_size 16, cache_seqlens
U[512, 8192], 40k-page pool): a step builds the page-level table from
req_to_token (strided conversion), runs the split-KV paged attention with 4
key chunks per (request, KV head), and combines the chunks with the
log-sum-exp state merge (inside the attention launch).

Metric: decode KV HBM GB/s = algorithmic K+V bytes of the step
(sum_b kv_len_b * H_kv * (D + Dv) * 2 B) / step time.  ``--workload`` selects
one of the other synthetic workloads (sliding-window decode with the
prefill-aware table, varlen causal extend [TFLOP/s], MLA top-k sparse decode).

Arms: ``--impl pkv`` (default) times libpkv; ``--impl reference`` times the
float64 CPU oracle on the host cores on a bounded sample of the same workload
(the pages publish no implementation or numbers to compare with).

Under torchrun each rank runs its own replica of the workload (weak scaling,
no collective on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import paged_kv_cache_203_gb300 as pkv  # noqa: E402
from paged_kv_cache_203_gb300 import workloads  # noqa: E402

HEADLINE = "gqa_split_decode"
L2_BYTES = 129 * 1024 * 1024

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# attention kernel on the full-size workload, from one ncu capture of the
# kernel as it is now; a kernel changed since its capture has no entry (its
# traffic is reported as null).
MEASURED_TRAFFIC = {
    ("gqa_split_decode", "decode_allheads_kernel (page boxes, fixed splits)"): 1_116_558_400,
    ("swa_decode", "decode_allheads_kernel (slot rows)"): 647_964_416,
    ("varlen_extend", "extend_tc_kernel"): 264_708_352,
    ("mla_topk_decode", "mla_topk_kernel"): 335_151_616,
    ("tiny_decode", "decode_short_cluster_kernel"): 594_432,  # its 2 MB of K / V sit in L2
}


# --------------------------------------------------------------------- peaks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks / throttle reasons every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------- workloads

class Step:
    """One pass of the hot path over a device-resident workload.

    ``run()`` launches the step on the current stream; ``attn_events`` (when
    given) brackets the dominant kernel (the attention launch) so its device
    time can be accumulated.  ``algo`` holds the algorithmic bytes / flops of
    one step."""

    def __init__(self, name: str, device, overrides: dict):
        self.name = name
        self.dev = device
        self.g = workloads.make(name, value_device=device, **overrides)
        g = self.g
        self.ws = None
        self.h2d_bytes = 0
        self.d2h_bytes = 0
        d, dv, h_kv = g.q.shape[-1], g.v_cache.shape[-1], g.k_cache.shape[2]
        if g.topk_indices is None:
            kv_tokens = int(g.cache_seqlens.sum())
        else:
            kv_tokens = int((g.topk_indices >= 0).sum())
        self.out = torch.empty(g.q.shape[0], g.q.shape[1], dv, dtype=torch.bfloat16,
                               device=device)
        self.lse = torch.empty(g.q.shape[0], g.q.shape[1], dtype=torch.float32,
                               device=device)
        if (g.kind == "swa"):
            self.pa_max = min(int(g.prefill_lens.max()) + g.window, int(g.seq_lens.max()))
            self.pt = torch.zeros(g.seq_lens.shape[0], self.pa_max, dtype=torch.int32,
                                  device=device)
            self.kv = torch.zeros(g.seq_lens.shape[0], dtype=torch.int32, device=device)
            # algorithmic KV rows: the prefill-aware lengths
            pf = g.prefill_lens[g.req_pool_indices.long()].cpu()
            sl = g.seq_lens.cpu()
            kv_tokens = int(torch.minimum(sl, pf + g.window).sum())
        else:
            self.n_cols = g.page_table.shape[1]
            self.pt = torch.zeros_like(g.page_table)
        self.kv_bytes = kv_tokens * h_kv * (d + dv) * 2 if g.topk_indices is None else \
            kv_tokens * d * 2  # absorbed MLA: one 576-wide row per gathered key
        self.flops = self._flops()
        # where the short decode kernels serve the attention, the library
        # builds the strided table inside the attention launch
        self.one_launch = (g.kind != "swa" and g.topk_indices is None
                           and self.attention_kernel().startswith("decode_short"))
        self.kernels_per_step = 1 if self.one_launch else 2

    def prepare(self):
        """Allocate the library's workspace (library arm only: the reference
        arm never loads the CUDA library)."""
        g = self.g
        self.workspace_bytes = pkv.attn_workspace_size(
            g.q, g.k_cache, g.v_cache, self.pt,
            g.cache_seqlens if not (g.kind == "swa") else self.kv, g.max_seqlen_q,
            g.topk_indices, g.num_splits)
        if self.workspace_bytes:
            self.ws = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=self.dev)
        return self

    def _flops(self):
        g = self.g
        d, dv, h_q = g.q.shape[-1], g.v_cache.shape[-1], g.q.shape[1]
        cs = g.cache_seqlens.cpu().numpy().astype(np.int64)
        cu = g.cu_seqlens_q.cpu().numpy().astype(np.int64)
        if g.topk_indices is not None:
            pairs = int((g.topk_indices >= 0).sum())
        elif (g.kind == "swa"):
            pf = g.prefill_lens[g.req_pool_indices.long()].cpu().numpy()
            pairs = int(np.minimum(g.seq_lens.cpu().numpy(), pf + g.window).sum())
        else:
            pairs = 0
            for b in range(len(cs)):
                ql = cu[b + 1] - cu[b]
                kv = cs[b]
                if g.causal:
                    pairs += ql * (kv - ql) + ql * (ql + 1) // 2
                else:
                    pairs += ql * kv
        return 2 * pairs * h_q * (d + dv)

    def per_request_work(self):
        """Algorithmic work of each request (keys x rows), for sampling."""
        g = self.g
        if g.topk_indices is not None:
            return (g.topk_indices.cpu() >= 0).sum(1).numpy().astype(np.float64)
        cs = g.cache_seqlens.cpu().numpy().astype(np.float64)
        if g.kind == "swa":
            pf = g.prefill_lens[g.req_pool_indices.long()].cpu().numpy()
            return np.minimum(g.seq_lens.cpu().numpy(), pf + g.window).astype(np.float64)
        ql = np.diff(g.cu_seqlens_q.cpu().numpy()).astype(np.float64)
        if g.causal:
            return ql * (cs - ql) + ql * (ql + 1) / 2
        return ql * cs

    def _table_and_attend(self):
        """The table built and the attention run by one library call."""
        g = self.g
        pkv.strided_table_attn_with_kvcache(
            g.req_to_token, g.req_pool_indices, self.pt, g.q, g.k_cache, g.v_cache,
            g.cache_seqlens, g.cu_seqlens_q, g.max_seqlen_q, g.scale, causal=g.causal,
            window_left=g.window_left, num_splits=g.num_splits, out=self.out, lse=self.lse,
            workspace=self.ws)

    def attend(self):
        """The step's attention launch alone (the table built by an earlier
        run); with the table built inside the attention launch, that launch."""
        if self.one_launch:
            self._table_and_attend()
            return
        g = self.g
        pt, cs = (self.pt, self.kv) if g.kind == "swa" else (self.pt, g.cache_seqlens)
        pkv.attn_with_kvcache(g.q, g.k_cache, g.v_cache, pt, cs, g.cu_seqlens_q,
                              g.max_seqlen_q, g.scale, causal=g.causal,
                              window_left=g.window_left, topk_indices=g.topk_indices,
                              num_splits=g.num_splits, out=self.out, lse=self.lse,
                              workspace=self.ws)

    def run(self, ev=None):
        g = self.g
        if self.one_launch:
            if ev is not None:
                ev[0].record()
            self._table_and_attend()
            if ev is not None:
                ev[1].record()
            return
        if (g.kind == "swa"):
            pkv.build_swa_page_table(g.req_to_token, g.req_pool_indices, g.seq_lens,
                                     g.prefill_lens, g.window, self.pt, self.kv)
            pt, cs = self.pt, self.kv
        else:
            pkv.strided_page_table(g.req_to_token, g.req_pool_indices, g.page_size,
                                   self.n_cols, out=self.pt)
            pt, cs = self.pt, g.cache_seqlens
        if ev is not None:
            ev[0].record()
        pkv.attn_with_kvcache(g.q, g.k_cache, g.v_cache, pt, cs, g.cu_seqlens_q,
                              g.max_seqlen_q, g.scale, causal=g.causal,
                              window_left=g.window_left, topk_indices=g.topk_indices,
                              num_splits=g.num_splits, out=self.out, lse=self.lse,
                              workspace=self.ws)
        if ev is not None:
            ev[1].record()

    def attention_kernel(self):
        """Name of the kernel the library picks for this step's attention."""
        g = self.g
        if g.kind == "mla":
            return "mla_topk_kernel"
        if g.kind == "extend":
            return "extend_tc_kernel"
        h_kv, p = g.k_cache.shape[2], g.page_size
        rows = g.max_seqlen_q * (g.q.shape[1] // h_kv)
        if (g.topk_indices is None and g.q.shape[-1] == 128 and rows <= 16
                and g.num_splits <= 1 and self.pt.shape[1] * p <= 256):
            # a 4-CTA cluster per (request, KV head) up to 76 pairs
            if g.cache_seqlens.shape[0] * h_kv <= 76:
                return "decode_short_cluster_kernel"
            return "decode_short_kernel"
        if g.topk_indices is None and g.q.shape[-1] == 128 and h_kv <= 8 and rows <= 16:
            if p < 8:
                return "decode_allheads_kernel (slot rows)"
            if p % 16 == 0 and g.num_splits == 0:
                return "decode_allheads_kernel (page boxes, balanced)"
            if p % 16 == 0:
                return "decode_allheads_kernel (page boxes, fixed splits)"
        return "decode_gqa_kernel"


def _event_ms(fn, reps: int = 20) -> float:
    """Mean device time of ``fn`` (launches on the current stream)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _multi_step_ms(fn, n: int = 20, reps: int = 10) -> float:
    """Device time per call with n calls captured in one CUDA graph: the
    graph launch is paid once per n calls (for steps of a few microseconds
    it is most of a one-call replay)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for _ in range(n):
            fn()
    torch.cuda.synchronize()
    ms = _event_ms(gr.replay, reps) / n
    del gr
    return ms


def _graph_floor_ms(n_ops: int = 1) -> float:
    """Time per replay of a CUDA graph holding ``n_ops`` trivial ops (one-
    element adds), replayed back to back like the steps: the launch-rate
    floor under a step of a few microseconds made of that many kernels."""
    x = torch.zeros(1, device="cuda")

    def ops():
        for _ in range(n_ops):
            x.add_(1.0)
    return _timed(ops, reps=200)[0]


def _timed(fn, reps: int = 20) -> tuple[float, dict]:
    """Device time of ``fn`` as a serving engine runs it: the calls captured
    once into a CUDA graph and replayed (a short call timed eagerly measures
    the host's launch cost, not the GPU); the eager time beside it.  Falls
    back to the eager time, with the reason, if capture fails."""
    eager = _event_ms(fn, reps)
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            fn()
        torch.cuda.synchronize()
    except RuntimeError as e:
        torch.cuda.synchronize()
        return eager, {"eager_ms": eager,
                       "launch": "eager (capture failed: %s)" % str(e).splitlines()[0][:160]}
    ms = _event_ms(gr.replay, reps)
    del gr
    return ms, {"eager_ms": eager, "launch": "CUDA graph replay"}


def local_attention_line(dev, peaks, chunk: int = 2048):
    """Local (chunked) attention on the headline decode batch: the device
    builder of the virtual requests, then one causal call over them.  The
    algorithmic K/V bytes are the keys each request's new tokens can see:
    from the start of the first new token's chunk to the last key."""
    g = workloads.make(HEADLINE, value_device=dev)
    P = g.page_size
    B = g.cache_seqlens.shape[0]
    max_q = g.max_seqlen_q
    cap = pkv.local_virtual_batch_capacity(B, g.q.shape[0], max_q, P)
    bufs = pkv.make_local_attention_virtual_batches(chunk, P, g.cu_seqlens_q, g.cache_seqlens,
                                                    g.page_table, cap)
    max_q_local = min(max_q, max((chunk // P) * P, P))
    out = torch.empty(g.q.shape[0], g.q.shape[1], g.v_cache.shape[-1], dtype=torch.bfloat16,
                      device=dev)
    lse = torch.empty(g.q.shape[0], g.q.shape[1], dtype=torch.float32, device=dev)
    ws_n = pkv.attn_workspace_size(g.q, g.k_cache, g.v_cache, bufs[3], bufs[2], max_q_local)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)

    def build():
        pkv.make_local_attention_virtual_batches(chunk, P, g.cu_seqlens_q, g.cache_seqlens,
                                                 g.page_table, cap, out=bufs)

    def attend():
        pkv.attn_with_kvcache(g.q, g.k_cache, g.v_cache, bufs[3], bufs[2], bufs[1],
                              max_q_local, g.scale, causal=True, out=out, lse=lse,
                              workspace=ws)

    def step():
        build()
        attend()

    kv = g.cache_seqlens.cpu().numpy().astype(np.int64)
    ql = np.diff(g.cu_seqlens_q.cpu().numpy()).astype(np.int64)
    eff = min(chunk, int(kv.max())) // P * P
    eff = max(eff, P)
    keys = int((kv - eff * ((kv - ql) // eff)).sum())
    h_kv, d, dv = g.k_cache.shape[2], g.q.shape[-1], g.v_cache.shape[-1]
    kv_bytes = keys * h_kv * (d + dv) * 2
    (b_ms, b_how), (a_ms, a_how), (s_ms, s_how) = _timed(build), _timed(attend), _timed(step)
    return {"kernel": "local_virtual_batches_kernel + attention", "chunk": chunk,
            "effective_chunk": eff, "virtual_requests_capacity": cap,
            "builder_ms": b_ms, "attn_ms": a_ms, "ms_per_step": s_ms,
            "timing": {"builder": b_how, "attention": a_how, "step": s_how},
            "kv_GBps": kv_bytes / 1e9 / (a_ms / 1e3),
            "kv_frac_hbm": kv_bytes / 1e9 / (a_ms / 1e3) / peaks["hbm_gbs"],
            "tokens_per_s": g.q.shape[0] / (s_ms / 1e3)}


def cascade_line(dev, peaks, prefix_tokens: int = 4096):
    """Cascade attention on the headline decode batch with a shared
    prefix: every request also sees the same prefix_tokens keys (one set of
    pages), then its own keys; prefix call + suffix call + state merge.
    ``kv_GBps_logical`` counts the prefix once per request, ``kv_GBps_unique``
    once per step (the rest is served by L2)."""
    g = workloads.make(HEADLINE, value_device=dev)
    P = g.page_size
    B = g.cache_seqlens.shape[0]
    n_pre = prefix_tokens // P
    pre_pt = torch.arange(n_pre, dtype=torch.int32, device=dev).repeat(B, 1).contiguous()
    pre_len = torch.full((B,), prefix_tokens, dtype=torch.int32, device=dev)
    out = torch.empty(g.q.shape[0], g.q.shape[1], g.v_cache.shape[-1], dtype=torch.bfloat16,
                      device=dev)
    lse = torch.empty(g.q.shape[0], g.q.shape[1], dtype=torch.float32, device=dev)

    def step():
        pkv.cascade_attn_with_kvcache(g.q, g.k_cache, g.v_cache, pre_pt, pre_len,
                                      g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                      g.max_seqlen_q, g.scale, causal=True, out=out, lse=lse)

    s_ms, s_how = _timed(step)
    h_kv, d, dv = g.k_cache.shape[2], g.q.shape[-1], g.v_cache.shape[-1]
    row = h_kv * (d + dv) * 2
    own = int(g.cache_seqlens.sum())
    logical = (own + B * prefix_tokens) * row
    unique = (own + prefix_tokens) * row
    return {"kernel": "2 x attention + merge_state_kernel", "prefix_tokens": prefix_tokens,
            "ms_per_step": s_ms, "timing": s_how,
            "kv_GBps_logical": logical / 1e9 / (s_ms / 1e3),
            "kv_GBps_unique": unique / 1e9 / (s_ms / 1e3),
            "unique_frac_hbm": unique / 1e9 / (s_ms / 1e3) / peaks["hbm_gbs"],
            "tokens_per_s": g.q.shape[0] / (s_ms / 1e3)}


def append_line(dev, peaks):
    """The KV write before attention on the varlen extend workload: every
    new token's K/V rows (8 heads x 128 x 2) stored to its slot, then the
    causal extend attention over the updated pool.  The write moves each new
    row twice (read + write)."""
    g = workloads.make("varlen_extend", value_device=dev)
    P = g.page_size
    cu = g.cu_seqlens_q.cpu().numpy()
    kv = g.cache_seqlens.cpu().numpy()
    pt = g.page_table.cpu().numpy()
    loc = np.concatenate([pt[b, np.arange(kv[b] - (cu[b + 1] - cu[b]), kv[b]) // P] * P +
                          np.arange(kv[b] - (cu[b + 1] - cu[b]), kv[b]) % P
                          for b in range(len(kv))])
    loc = torch.from_numpy(loc.astype(np.int64)).to(dev)
    k_new = g.k_cache.view(-1, *g.k_cache.shape[2:])[loc].clone()
    v_new = g.v_cache.view(-1, *g.v_cache.shape[2:])[loc].clone()
    out = torch.empty(g.q.shape[0], g.q.shape[1], g.v_cache.shape[-1], dtype=torch.bfloat16,
                      device=dev)

    def write():
        pkv.set_kv_buffer(g.k_cache, g.v_cache, loc, k_new, v_new)

    def step():
        pkv.append_attn_with_kvcache(g.q, k_new, v_new, loc, g.k_cache, g.v_cache,
                                     g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                     g.max_seqlen_q, g.scale, causal=True, out=out)

    # the same rows stored into pools of fp8 codes (value / 0.05)
    k8 = torch.zeros(g.k_cache.shape, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    v8 = torch.zeros(g.v_cache.shape, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    scale = torch.tensor([0.05], dtype=torch.float32, device=dev)

    def write_fp8():
        pkv.set_kv_buffer(k8, v8, loc, k_new, v_new, k_scale=scale, v_scale=scale)

    (w_ms, w_how), (s_ms, s_how) = _timed(write), _timed(step)
    w8_ms, w8_how = _timed(write_fp8)
    moved = 2 * (k_new.numel() + v_new.numel()) * 2
    moved8 = (k_new.numel() + v_new.numel()) * 3  # 2 B read + 1 B code written
    return {"kernel": "set_kv_buffer_kernel (+ extend_tc_kernel)", "new_tokens": int(loc.numel()),
            "timing": {"write": w_how, "step": s_how, "write_fp8": w8_how},
            "write_fp8_ms": w8_ms, "write_fp8_GBps": moved8 / 1e9 / (w8_ms / 1e3),
            "write_fp8_frac_hbm": moved8 / 1e9 / (w8_ms / 1e3) / peaks["hbm_gbs"],
            "write_ms": w_ms, "write_GBps": moved / 1e9 / (w_ms / 1e3),
            "write_frac_hbm": moved / 1e9 / (w_ms / 1e3) / peaks["hbm_gbs"],
            "ms_per_step": s_ms, "tokens_per_s": g.q.shape[0] / (s_ms / 1e3)}


def fp8_line(dev, peaks):
    """The headline decode batch over an fp8 (e4m3) cache: the same keys as
    the bf16 cache cast to e4m3 codes, per-(request, KV head) descales, the
    library's split choice.  Algorithmic bytes are the codes read: 1 byte per
    element (2048 B per token at 8 KV heads, head dim 128)."""
    g = workloads.make(HEADLINE, value_device=dev)
    k8 = g.k_cache.to(torch.float8_e4m3fn)
    v8 = g.v_cache.to(torch.float8_e4m3fn)
    del g.k_cache, g.v_cache
    B, h_kv = g.cache_seqlens.shape[0], k8.shape[2]
    kd = torch.full((B, h_kv), 0.75, device=dev)
    vd = torch.full((B, h_kv), 1.25, device=dev)
    out = torch.empty(g.q.shape[0], g.q.shape[1], 128, dtype=torch.bfloat16, device=dev)
    ws_n = pkv.attn_workspace_size(g.q, k8, v8, g.page_table, g.cache_seqlens, g.max_seqlen_q)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)

    def attend():
        pkv.attn_with_kvcache_fp8(g.q, k8, v8, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                  g.max_seqlen_q, g.scale, k_descale=kd, v_descale=vd,
                                  out=out, workspace=ws)

    a_ms, a_how = _timed(attend)
    kv_bytes = int(g.cache_seqlens.sum()) * h_kv * 256
    return {"kernel": "decode_allheads_kernel (page boxes, balanced, fp8)",
            "attn_ms": a_ms, "timing": a_how, "kv_GBps": kv_bytes / 1e9 / (a_ms / 1e3),
            "kv_frac_hbm": kv_bytes / 1e9 / (a_ms / 1e3) / peaks["hbm_gbs"],
            "tokens_per_s": g.q.shape[0] / (a_ms / 1e3)}


def fp8_swa_line(dev, peaks):
    """The sliding-window decode workload over an fp8 cache (page size 1:
    slot rows of codes): the prefill-aware table, then the attention with
    descales 0.75 / 1.25.  Algorithmic bytes are the codes of the kept rows
    (1 byte per element)."""
    st = Step("swa_decode", dev, {})
    g = st.g
    k8 = g.k_cache.to(torch.float8_e4m3fn)
    v8 = g.v_cache.to(torch.float8_e4m3fn)
    del g.k_cache, g.v_cache
    pkv.build_swa_page_table(g.req_to_token, g.req_pool_indices, g.seq_lens, g.prefill_lens,
                             g.window, st.pt, st.kv)
    B, h_kv = st.kv.shape[0], k8.shape[2]
    kd = torch.full((B, h_kv), 0.75, device=dev)
    vd = torch.full((B, h_kv), 1.25, device=dev)
    out = torch.empty(g.q.shape[0], g.q.shape[1], 128, dtype=torch.bfloat16, device=dev)
    ws_n = pkv.attn_workspace_size(g.q, k8, v8, st.pt, st.kv, 1)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)

    def attend():
        pkv.attn_with_kvcache_fp8(g.q, k8, v8, st.pt, st.kv, g.cu_seqlens_q, 1, g.scale,
                                  k_descale=kd, v_descale=vd, out=out, workspace=ws)

    a_ms, a_how = _timed(attend)
    code_bytes = st.kv_bytes // 2
    return {"kernel": "decode_allheads_kernel (slot rows, balanced, fp8)", "attn_ms": a_ms,
            "timing": a_how, "kv_GBps": code_bytes / 1e9 / (a_ms / 1e3),
            "kv_frac_hbm": code_bytes / 1e9 / (a_ms / 1e3) / peaks["hbm_gbs"],
            "tokens_per_s": g.q.shape[0] / (a_ms / 1e3)}


def fp8_mla_line(dev, peaks):
    """The MLA top-k decode workload over an fp8 latent cache (codes of the
    bf16 rows, descales 0.75 / 1.25): algorithmic bytes are the listed rows'
    codes (576 B per key per token), flops as for the bf16 cache."""
    g = workloads.make("mla_topk_decode", value_device=dev)
    st = Step.__new__(Step)
    st.g = g
    flops = Step._flops(st)
    k8 = g.k_cache.to(torch.float8_e4m3fn)
    del g.k_cache, g.v_cache
    B = g.cache_seqlens.shape[0]
    kd = torch.full((B, 1), 0.75, device=dev)
    vd = torch.full((B, 1), 1.25, device=dev)
    out = torch.empty(g.q.shape[0], 128, 512, dtype=torch.bfloat16, device=dev)

    def attend():
        pkv.attn_with_kvcache_fp8(g.q, k8, k8[..., :512], g.page_table, g.cache_seqlens,
                                  g.cu_seqlens_q, g.max_seqlen_q, g.scale,
                                  topk_indices=g.topk_indices, k_descale=kd, v_descale=vd,
                                  out=out)

    a_ms, a_how = _timed(attend)
    code_bytes = int((g.topk_indices >= 0).sum()) * 576
    return {"kernel": "mla_topk_kernel (fp8 cache)", "attn_ms": a_ms, "timing": a_how,
            "kv_GBps": code_bytes / 1e9 / (a_ms / 1e3),
            "kv_frac_hbm": code_bytes / 1e9 / (a_ms / 1e3) / peaks["hbm_gbs"],
            "TFLOPs": flops / 1e12 / (a_ms / 1e3)}


def fp8_extend_line(dev, peaks):
    """The varlen extend workload over an fp8 cache (the bf16 cache cast to
    e4m3 codes, descales 0.75 / 1.25): e4m3 QK^T and f16 PV on the tensor
    cores, flops over the visible (q, k) pairs as for the bf16 cache."""
    g = workloads.make("varlen_extend", value_device=dev)
    st = Step.__new__(Step)
    st.g = g
    flops = Step._flops(st)
    k8 = g.k_cache.to(torch.float8_e4m3fn)
    v8 = g.v_cache.to(torch.float8_e4m3fn)
    del g.k_cache, g.v_cache
    B, h_kv = g.cache_seqlens.shape[0], k8.shape[2]
    kd = torch.full((B, h_kv), 0.75, device=dev)
    vd = torch.full((B, h_kv), 1.25, device=dev)
    out = torch.empty(g.q.shape[0], g.q.shape[1], 128, dtype=torch.bfloat16, device=dev)

    def attend():
        pkv.attn_with_kvcache_fp8(g.q, k8, v8, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                  g.max_seqlen_q, g.scale, causal=True, k_descale=kd,
                                  v_descale=vd, out=out)

    a_ms, a_how = _timed(attend)
    tf = flops / 1e12 / (a_ms / 1e3)
    return {"kernel": "extend_tc_kernel (fp8 cache)", "attn_ms": a_ms, "timing": a_how,
            "TFLOPs": tf, "tflop_frac_bf16": tf / peaks["bf16_tflops"]}


def append_decode_line(dev, peaks):
    """The KV write before decode attention on the GQA decode batch (each
    request's last key is its new token), with the bench's 4 key chunks:
    the unfused pair (set_kv_buffer, then attention) against the fused launch
    (pkv_append_attn_with_kvcache).  Algorithmic bytes: the K/V read plus the
    new rows read and written."""
    g = workloads.make(HEADLINE, value_device=dev)
    P = g.page_size
    kv = g.cache_seqlens.cpu().numpy()
    pt = g.page_table.cpu().numpy()
    loc = torch.tensor([int(pt[b, (kv[b] - 1) // P]) * P + (kv[b] - 1) % P
                        for b in range(len(kv))], dtype=torch.int64, device=dev)
    k_new = g.k_cache.view(-1, *g.k_cache.shape[2:])[loc].clone()
    v_new = g.v_cache.view(-1, *g.v_cache.shape[2:])[loc].clone()
    out = torch.empty(g.q.shape[0], g.q.shape[1], g.v_cache.shape[-1], dtype=torch.bfloat16,
                      device=dev)
    ws_n = pkv.attn_workspace_size(g.q, g.k_cache, g.v_cache, g.page_table, g.cache_seqlens,
                                   g.max_seqlen_q, None, g.num_splits)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)

    def unfused():
        pkv.append_attn_with_kvcache(g.q, k_new, v_new, loc, g.k_cache, g.v_cache,
                                     g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                     g.max_seqlen_q, g.scale, num_splits=g.num_splits,
                                     out=out, workspace=ws)

    def fused():
        pkv.fused_append_attn_with_kvcache(g.q, k_new, v_new, loc, g.k_cache, g.v_cache,
                                           g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                           g.max_seqlen_q, g.scale, num_splits=g.num_splits,
                                           out=out, workspace=ws)

    (u_ms, u_how), (f_ms, f_how) = _timed(unfused), _timed(fused)
    h_kv, d = g.k_cache.shape[2], g.q.shape[-1]
    bytes_ = int(g.cache_seqlens.sum()) * h_kv * 2 * d * 2 + 2 * loc.numel() * h_kv * 2 * d * 2
    return {"kernel": "decode_allheads_kernel (fused append) vs set_kv_buffer_kernel + attention",
            "new_tokens": int(loc.numel()), "unfused_ms": u_ms, "fused_ms": f_ms,
            "timing": {"unfused": u_how, "fused": f_how},
            "fused_GBps": bytes_ / 1e9 / (f_ms / 1e3),
            "fused_frac_hbm": bytes_ / 1e9 / (f_ms / 1e3) / peaks["hbm_gbs"],
            "unfused_GBps": bytes_ / 1e9 / (u_ms / 1e3)}


def topk_line(dev, peaks):
    """The top-k index -> slot transform on its own (the MLA decode batch's
    lists: 128 tokens x 2048 entries, page size 64): reads each entry and its
    page id, writes the slot; 12 B per entry (entry, page id, slot)."""
    g = workloads.make("mla_topk_decode", value_device=dev)
    out = torch.empty_like(g.topk_indices)

    def step():
        pkv.topk_to_slots(g.topk_indices, g.cu_seqlens_q, g.page_table, g.cache_seqlens,
                          g.page_size, out=out)

    s_ms, s_how = _timed(step)
    moved = g.topk_indices.numel() * 12
    return {"kernel": "topk_to_slots_kernel", "entries": int(g.topk_indices.numel()),
            "ms_per_step": s_ms, "timing": s_how, "GBps": moved / 1e9 / (s_ms / 1e3),
            "frac_hbm": moved / 1e9 / (s_ms / 1e3) / peaks["hbm_gbs"]}


def merge_line(dev, peaks, sizes=(("decode_batch", 64), ("prefill", 32768))):
    """The state merge on its own: two bf16 partial states (v [n, 32 heads,
    128], fp32 lse) merged into one; reads 2 x (v + lse), writes v + lse.
    Two sizes: the GQA decode batch's shape (64 tokens, launch-bound) and a
    prefill-sized one (32768 tokens, 805 MB moved, larger than L2)."""
    h, d = 32, 128
    out = {"kernel": "merge_state_kernel"}
    for label, n in sizes:
        gen = torch.Generator(device=dev).manual_seed(1005)
        va = torch.randn(n, h, d, device=dev, generator=gen).to(torch.bfloat16)
        vb = torch.randn(n, h, d, device=dev, generator=gen).to(torch.bfloat16)
        la = torch.randn(n, h, device=dev, generator=gen)
        lb = torch.randn(n, h, device=dev, generator=gen)
        vo, lo = torch.empty_like(va), torch.empty_like(la)

        def step():
            pkv.merge_state(va, la, vb, lb, vo, lo)

        s_ms, s_how = _timed(step)
        moved = 3 * va.numel() * 2 + 3 * la.numel() * 4
        out[label] = {"rows": n * h, "ms_per_step": s_ms, "timing": s_how,
                      "GBps": moved / 1e9 / (s_ms / 1e3),
                      "frac_hbm": moved / 1e9 / (s_ms / 1e3) / peaks["hbm_gbs"]}
        del va, vb, la, lb, vo, lo
    return out


EXTRA_LINES = {"local": local_attention_line, "cascade": cascade_line, "append": append_line,
               "fp8": fp8_line, "topk": topk_line, "merge": merge_line,
               "merge_prefill": lambda dev, peaks: merge_line(dev, peaks, (("prefill", 32768),)),
               "fp8_extend": fp8_extend_line, "fp8_swa": fp8_swa_line,
               "fp8_mla": fp8_mla_line,
               "append_decode": append_decode_line}


def parse_overrides(s: str | None) -> dict:
    out = {}
    if not s:
        return out
    for kv in s.split(","):
        k, v = kv.split("=")
        out[k] = int(v)
    return out


# ------------------------------------------------------------- end to end

def _blob(tensors, device, pin):
    """One byte buffer holding ``tensors`` (256-byte aligned slices) and
    contiguous views of it with their shapes and dtypes."""
    offs, size = [], 0
    for t in tensors:
        offs.append(size)
        size += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(size, 1), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for o, t in zip(offs, tensors)]
    return buf, views


def run_e2e(step: Step, steps: int):
    """Same metric through the public API with the step's inputs in pinned
    host memory: per step, copy q / req_to_token / indices / lengths host ->
    device, run the step, copy out and lse back.  The KV cache stays
    resident in HBM (it is the cache).  As a serving loop would, the inputs
    travel as one packed buffer each way (one copy up, one down per step),
    on their own streams over two sets of buffers: step i+1's inputs go up
    and step i-1's outputs come down while step i computes (each step waits
    for its own inputs; each read-back waits for its step)."""
    g = step.g
    names = ["q", "req_to_token", "req_pool_indices", "cache_seqlens", "cu_seqlens_q"]
    if (g.kind == "swa"):
        names += ["seq_lens", "prefill_lens"]
    if g.topk_indices is not None:
        names += ["topk_indices"]
    first = {n: getattr(g, n) for n in names}
    host_in, host_views = _blob([first[n] for n in names], "cpu", True)
    for hv, n in zip(host_views, names):
        hv.copy_(first[n])
    host_out, (out_h, lse_h) = _blob([step.out, step.lse], "cpu", True)
    h2d, d2h = host_in.numel(), host_out.numel()  # bytes copied (the packed buffers)
    ins = [_blob([first[n] for n in names], step.dev, False) for _ in range(2)]
    outs = [_blob([step.out, step.lse], step.dev, False) for _ in range(2)]
    first_out = (step.out, step.lse)
    comp = torch.cuda.current_stream()
    cp_up, cp_down = torch.cuda.Stream(), torch.cuda.Stream()
    up = [torch.cuda.Event(), torch.cuda.Event()]    # inputs of the set landed
    done = [torch.cuda.Event(), torch.cuda.Event()]  # the step using the set finished
    down = [torch.cuda.Event(), torch.cuda.Event()]  # the set's outputs were read back

    def upload(i):
        k = i % 2
        with torch.cuda.stream(cp_up):
            if i >= 2:
                cp_up.wait_event(done[k])  # step i - 2 no longer reads set k
            ins[k][0].copy_(host_in, non_blocking=True)
            up[k].record(cp_up)

    def use_set(k):
        for n, v in zip(names, ins[k][1]):
            setattr(g, n, v)
        step.out, step.lse = outs[k][1]

    # the step over each buffer set captured once, as the timed loop replays it
    graphs = []
    for k in range(2):
        ins[k][0].copy_(host_in)
        use_set(k)
        try:
            side = torch.cuda.Stream()
            side.wait_stream(comp)
            with torch.cuda.stream(side):
                step.run()
            comp.wait_stream(side)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                step.run()
            graphs.append(gr)
        except RuntimeError:
            torch.cuda.synchronize()
            graphs = []
            break
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    upload(0)
    for i in range(steps):
        k = i % 2
        if i + 1 < steps:
            upload(i + 1)
        comp.wait_event(up[k])
        if i >= 2:
            comp.wait_event(down[k])  # step i - 2's outputs were read back
        if graphs:
            graphs[k].replay()
        else:
            use_set(k)
            step.run()
        done[k].record(comp)
        with torch.cuda.stream(cp_down):
            cp_down.wait_event(done[k])
            host_out.copy_(outs[k][0], non_blocking=True)
            down[k].record(cp_down)
    comp.wait_stream(cp_up)
    comp.wait_stream(cp_down)
    t1.record(comp)
    torch.cuda.synchronize()
    launch = "CUDA graph replay per buffer set" if graphs else "eager"
    del graphs
    for n in names:
        setattr(g, n, first[n])
    step.out, step.lse = first_out
    ms = t0.elapsed_time(t1) / steps
    # the read-back equals a plain step's output (same inputs every step)
    step.run()
    torch.cuda.synchronize()
    same = bool(torch.equal(out_h, step.out.cpu()) and torch.equal(lse_h, step.lse.cpu()))
    return ms, h2d, d2h, same, launch


# ------------------------------------------------------------ cpu baseline

class OracleSample:
    """The oracle as it stands, on the host cores, over a bounded sample of
    the same workload: its own strided / prefill-aware table, then attention
    (and, for split workloads, chunk states combined by its merge) for the
    first ``nreq`` requests.  ``frac`` is the share of the step's algorithmic
    work the sample covers."""

    def __init__(self, step: Step, pass_budget_s: float):
        import oracle

        self.oracle = oracle
        g = step.g
        self.step = step
        self.q = oracle.bf16_bits(g.q)
        self.k = oracle.bf16_bits(g.k_cache)
        self.v = (self.k[..., : g.v_cache.shape[-1]] if g.topk_indices is not None
                  else oracle.bf16_bits(g.v_cache))
        self.rtt = g.req_to_token.cpu().numpy()
        self.rpi = g.req_pool_indices.cpu().numpy()
        self.cu = g.cu_seqlens_q.cpu().numpy()
        self.cs = g.cache_seqlens.cpu().numpy()
        self.topk = None if g.topk_indices is None else g.topk_indices.cpu().numpy()
        self.threads = os.cpu_count() or 1
        batch = len(self.cs)
        t = time.perf_counter()
        self.run(1)
        per_req = max(time.perf_counter() - t, 1e-4)
        self.nreq = batch if per_req * batch <= pass_budget_s else \
            max(1, int(pass_budget_s / per_req))
        work = step.per_request_work()
        self.frac = float(work[: self.nreq].sum() / max(1e-30, work.sum()))
        self.batch = batch

    def run(self, nreq=None):
        o, g, st = self.oracle, self.step.g, self.step
        nreq = self.nreq if nreq is None else nreq
        cu_s = self.cu[: nreq + 1]
        q = self.q[: cu_s[-1]]
        if g.kind == "swa":
            pt, kv, _ = o.swa_page_table(self.rtt, self.rpi[:nreq],
                                         g.seq_lens.cpu().numpy()[:nreq],
                                         g.prefill_lens.cpu().numpy(), g.window, st.pa_max)
            o.attention(q, self.k, self.v, pt, kv, cu_s, g.scale, num_threads=self.threads)
            return
        pt = o.strided_page_table(self.rtt, self.rpi[:nreq], g.page_size, st.n_cols)
        if g.num_splits > 1:
            o.split_attention(q, self.k, self.v, pt, self.cs[:nreq], cu_s, g.scale,
                              g.num_splits, num_threads=self.threads)
        else:
            o.attention(q, self.k, self.v, pt, self.cs[:nreq], cu_s, g.scale,
                        causal=g.causal, window_left=g.window_left,
                        topk=None if self.topk is None else self.topk[: cu_s[-1]],
                        d_v=g.v_cache.shape[-1], num_threads=self.threads)

    def describe(self, passes):
        if self.nreq == self.batch:
            return f"{passes} pass(es) over the full step ({self.batch} requests)"
        return (f"{passes} pass(es) over the first {self.nreq} of {self.batch} "
                f"requests ({self.frac:.1%} of the step's work)")


def oracle_step_time(step: Step, budget_s: float = 10.0):
    """Seconds per full step for the oracle, from whole passes over a sample
    repeated until ``budget_s`` has elapsed."""
    smp = OracleSample(step, budget_s)
    done, t0 = 0, time.perf_counter()
    while True:
        smp.run()
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return el / done / smp.frac, smp.threads, smp.describe(done)


# --------------------------------------------------------------------- main

def roofline_of(step: Step, attn_ms: float, peaks: dict, sized: bool = False) -> dict:
    """Roofline object of a step's attention kernel: algorithmic bytes (decode)
    or flops (extend) per launch over the launch's CUDA-event time, against
    the measured peak; traffic from the ncu table (full-size workloads of
    kernels unchanged since their capture), else null."""
    traffic = None if sized else MEASURED_TRAFFIC.get((step.name, step.attention_kernel()))
    if step.name == "varlen_extend":
        achieved = step.flops / 1e12 / (attn_ms / 1e3)
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": traffic, "kernel": step.attention_kernel(),
                "peak_source": peaks["source"]}
    achieved = step.kv_bytes / 1e9 / (attn_ms / 1e3)
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
            "kernel": step.attention_kernel(), "peak_source": peaks["source"]}


def config_summary(step: Step, attn_ms: float, step_ms: float, peaks: dict) -> dict:
    """Compact per-workload record: the metric, the step time, the attention
    kernel's roofline (and, for the MLA decode, whose bytes and flops meet
    near the ridge, the tensor fraction beside it)."""
    metric, unit, per_step = metric_of(step)
    out = {"metric": metric, "value": per_step / (step_ms / 1e3), "unit": unit,
           "ms_per_step": step_ms, "attn_ms": attn_ms,
           "roofline": roofline_of(step, attn_ms, peaks),
           "tokens_per_s": step.g.q.shape[0] / (step_ms / 1e3)}
    if step.g.kind == "mla":
        tf = step.flops / 1e12 / (attn_ms / 1e3)
        out["tensor"] = {"achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"]}
    return out


def metric_of(step: Step):
    if step.name == "varlen_extend":
        return "extend TFLOP/s", "TFLOP/s", step.flops / 1e12
    return "decode KV HBM GB/s", "GB/s", step.kv_bytes / 1e9


def run_reference(args, rank, world):
    """The oracle on the host cores: W warm-up and K timed passes, each pass a
    bounded sample of the workload sized so the whole run stays within about
    two minutes."""
    if rank != 0:
        return
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    step = Step(args.workload, dev, parse_overrides(args.override))
    metric, unit, per_step = metric_of(step)
    pass_budget = min(args.ref_budget, 120.0 / (args.steps + args.warmup))
    smp = OracleSample(step, pass_budget)
    for _ in range(args.warmup):
        smp.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.run()
    s_per_pass = (time.perf_counter() - t0) / args.steps
    val = per_step * smp.frac / s_per_pass
    line = {
        "impl": "reference", "metric": metric, "value": val, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": s_per_pass * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, **parse_overrides(args.override)},
        "cpu_baseline": {"value": val, "unit": unit, "cores": smp.threads,
                         "kind": "oracle", "sample": smp.describe(args.steps)},
        "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=list(workloads.CONFIGS))
    ap.add_argument("--override", default=None,
                    help="comma list key=int shrinking the workload (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the per-workload summary of the other workloads")
    ap.add_argument("--ref-budget", type=float, default=10.0)
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step with eager launches instead of a CUDA graph replay")
    ap.add_argument("--line", default=None, choices=sorted(EXTRA_LINES),
                    help="run one of the extra lines alone (local attention, cascade, "
                         "KV write) and print its JSON; for profiling")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.line is not None:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        pkv.load_library()
        print(json.dumps({"line": args.line, **EXTRA_LINES[args.line](dev, measured_peaks())}),
              flush=True)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "pkv" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.load_library()
    peaks = measured_peaks()
    step = Step(args.workload, dev, parse_overrides(args.override)).prepare()
    metric, unit, per_step = metric_of(step)

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    pkv.clear_error_flags()

    # A step has no host work or synchronisation inside, so it is captured
    # once into a CUDA graph and replayed (as a serving engine replays its
    # decode step); the attention kernel's own time comes from an eager loop
    # with events around it.
    graph = None
    graph_note = "eager (--no-graph)"
    if not args.no_graph:
        try:
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                step.run()
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step.run()
            graph.replay()
            torch.cuda.synchronize()
        except RuntimeError as e:  # report why, time the step eagerly
            graph = None
            graph_note = "eager (graph capture failed: %s)" % str(e).splitlines()[0][:200]
            print(graph_note, file=sys.stderr, flush=True)
    pkv.clear_error_flags()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step.run()
    t1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(args.steps):  # the attention launch alone, eager
        step.run(evs[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_launch = ("CUDA graph replay of the step (the library's calls captured once)"
                   if graph is not None else graph_note)
    ms = t0.elapsed_time(t1) / args.steps
    attn_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    short_step = {}
    if ms < 0.05:  # a few microseconds: eager launches time the host
        attn_ms = min(attn_ms, _timed(step.attend)[0])
        short_step = {"ms_per_step_20_steps_per_graph": _multi_step_ms(step.run),
                      "ms_per_replay_of_a_one_op_graph": _graph_floor_ms(1),
                      "ms_per_replay_of_a_two_op_graph": _graph_floor_ms(2)}
    flags = pkv.get_error_flags()
    if dist is not None:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # end to end through the public API with host buffers
    e2e_ms, h2d, d2h, e2e_same, e2e_launch = run_e2e(step, max(8, args.steps // 2))
    if dist is not None:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    value = per_step * world / (ms / 1e3)
    e2e_val = per_step * world / (e2e_ms / 1e3)
    # full-size workloads only (a split-count override keeps the sizes)
    sized = bool(set(parse_overrides(args.override)) - {"num_splits"})
    roof = roofline_of(step, attn_ms, peaks, sized)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s_per_step, threads, sample = oracle_step_time(step, 10.0)
        cpu = {"value": per_step / s_per_step, "unit": unit, "cores": threads,
               "kind": "oracle", "sample": sample}

    n_tokens = int(step.g.q.shape[0])
    others = {}
    configs = {}
    if rank == 0 and not args.no_others and args.workload == HEADLINE and not args.override:
        configs[HEADLINE] = config_summary(step, attn_ms, ms, peaks)
        graph = None  # its captured buffers go with the workload
        del step.g
        torch.cuda.empty_cache()
        # the other workloads, and the headline workload with the library's
        # own split choice (balanced schedule) instead of the fixed 4 chunks
        runs = [(n, n, {}) for n in workloads.CONFIGS if n != HEADLINE]
        runs.append((HEADLINE + "@auto_split", HEADLINE, {"num_splits": 0}))
        for label, name, ov in runs:
            try:
                s2 = Step(name, dev, ov).prepare()
                for _ in range(3):
                    s2.run()
                torch.cuda.synchronize()
                e2 = [(torch.cuda.Event(enable_timing=True),
                       torch.cuda.Event(enable_timing=True)) for _ in range(20)]
                for i in range(20):
                    s2.run(e2[i])
                torch.cuda.synchronize()
                kms = sum(x.elapsed_time(y) for x, y in e2) / 20
                sms, how = _timed(s2.run)
                if sms < 0.05:
                    # a step of a few microseconds: eager launches time the
                    # host, so the attention is timed in graph replays too,
                    # and the step also with 20 steps in one graph
                    kms = min(kms, _timed(s2.attend)[0])
                    how = dict(how, ms_per_step_20_steps_per_graph=_multi_step_ms(s2.run),
                               attn_ms_20_per_graph=_multi_step_ms(s2.attend),
                               ms_per_replay_of_a_one_op_graph=_graph_floor_ms(1),
                               ms_per_replay_of_a_two_op_graph=_graph_floor_ms(2))
                if not ov:
                    configs[label] = config_summary(s2, kms, sms, peaks)
                    for key in ("ms_per_step_20_steps_per_graph",
                                "ms_per_replay_of_a_one_op_graph",
                                "ms_per_replay_of_a_two_op_graph"):
                        if key in how:
                            configs[label][key] = how[key]
                others[label] = {
                    "kernel": s2.attention_kernel(),
                    "ms_per_step": sms, "step_timing": how, "attn_ms": kms,
                    "kv_GBps": s2.kv_bytes / 1e9 / (kms / 1e3),
                    "kv_frac_hbm": s2.kv_bytes / 1e9 / (kms / 1e3) / peaks["hbm_gbs"],
                    "TFLOPs": s2.flops / 1e12 / (kms / 1e3),
                    "tflop_frac_bf16": s2.flops / 1e12 / (kms / 1e3) / peaks["bf16_tflops"],
                    "tokens_per_s": s2.g.q.shape[0] / (sms / 1e3)}
                del s2
                torch.cuda.empty_cache()
            except pkv.PkvError as e:
                others[label] = {"unavailable": str(e)}
                if not ov:
                    configs[label] = {"unavailable": str(e)}
        for label, fn in ((HEADLINE + "@local_chunk_2048", local_attention_line),
                          (HEADLINE + "@cascade_shared_prefix_4096", cascade_line),
                          ("varlen_extend@append_then_attend", append_line),
                          (HEADLINE + "@fused_append", append_decode_line),
                          (HEADLINE + "@fp8_kv", fp8_line),
                          ("varlen_extend@fp8_kv", fp8_extend_line),
                          ("swa_decode@fp8_kv", fp8_swa_line),
                          ("mla_topk_decode@fp8_kv", fp8_mla_line)):
            try:
                others[label] = fn(dev, peaks)
            except pkv.PkvError as e:
                others[label] = {"unavailable": str(e)}
            torch.cuda.empty_cache()

    if rank == 0:
        g_cfg = {"workload": args.workload}
        g_cfg.update(workloads.CONFIGS[args.workload])
        g_cfg.pop("kind", None)
        g_cfg.pop("seed", None)
        g_cfg.update(parse_overrides(args.override))
        g_cfg["algorithmic_kv_bytes_per_step"] = step.kv_bytes
        g_cfg["step_launch"] = step_launch
        g_cfg["l2"] = ("inputs larger than L2: %.2f GB of K/V per step vs 129 MB L2"
                       % (step.kv_bytes / 1e9)) if step.kv_bytes > L2_BYTES else \
            "inputs smaller than L2 (no flush)"
        line = {
            "metric": metric, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": g_cfg,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "copies": "one packed copy each way per step, on their own streams, two buffer sets, overlapped with the steps",
                    "step_launch": e2e_launch,
                    "read_back_matches_a_plain_step": e2e_same},
            "gpu_launches": step.kernels_per_step * args.steps,
            "clocks": clk,
            "tokens_per_s": n_tokens * world / (ms / 1e3),
            "error_flags": flags,
        }
        if short_step:  # a step of a few microseconds: device-side times too
            line["short_step"] = short_step
        if configs:  # the five workloads, compact, ahead of the long details
            line["configs"] = configs
        if others:
            line["other_workloads"] = others
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
