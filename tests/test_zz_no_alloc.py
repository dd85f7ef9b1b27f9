"""pkv_attn_with_kvcache_noalloc: attention for callers that cannot allocate.

Some callers of this library get only their input and output buffers and
cannot allocate device memory on this path (a plugin interface without a
workspace hook, a runtime that plans all device memory up front, code that
must not call cudaMalloc / cudaFree because they can synchronise the device
or fail while another allocator holds the memory).  The no-allocation entry
point serves them with the split scratch kept in a fixed array inside the
library.  These checks call it through the C ABI and compare it with the
regular entry point, on two calls in a row with different inputs, so that
anything the first call leaves in the shared array would show up in the
second.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_203_gb300 as pkv
from paged_kv_cache_203_gb300 import workloads

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3
DEV = "cuda"


def _regular(g, num_splits):
    return pkv.attn_with_kvcache(
        g.q, g.k_cache, g.v_cache, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
        g.max_seqlen_q, g.scale, causal=g.causal, window_left=g.window_left,
        num_splits=num_splits, return_softmax_lse=True)


def _noalloc(g, num_splits, out, lse):
    return pkv.attn_with_kvcache_noalloc(
        g.q, g.k_cache, g.v_cache, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
        g.max_seqlen_q, g.scale, out, lse=lse, causal=g.causal,
        window_left=g.window_left, num_splits=num_splits)


def _close(a, b, la, lb):
    err = (a.float() - b.float()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    fin = torch.isfinite(lb)
    assert torch.equal(torch.isfinite(la), fin)
    if fin.any():
        assert (la[fin] - lb[fin]).abs().max().item() <= LSE_ABS


def test_noalloc_matches_regular_entry_point_two_calls_in_a_row():
    pkv.load_library()
    cases = [
        # the batched GQA split-KV decode recipe, reduced: 16 requests, 4 splits
        (workloads.make("gqa_split_decode", batch=16, len_lo=512, len_hi=4096,
                        pool_pages=5000), 4),
        # a different shape and split count on the same scratch
        (workloads.make("tiny_decode", batch=9, h_q=16, h_kv=4, page_size=16,
                        len_lo=1, len_hi=3000, pool_tokens=9 * 3008 + 64), 7),
    ]
    outs = []
    for wl, splits in cases:
        g = wl.to(DEV)
        assert pkv.attn_workspace_size(g.q, g.k_cache, g.v_cache, g.page_table,
                                       g.cache_seqlens, g.max_seqlen_q,
                                       num_splits=splits) > 0  # uses scratch
        out = torch.empty(g.q.shape[0], g.q.shape[1], g.v_cache.shape[-1],
                          dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(g.q.shape[0], g.q.shape[1], dtype=torch.float32, device=DEV)
        torch.cuda.synchronize()
        before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        _noalloc(g, splits, out, lse)
        after = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        assert after == before  # the call allocated nothing through torch
        ref_o, ref_l = _regular(g, splits)
        torch.cuda.synchronize()
        _close(out, ref_o, lse, ref_l)
        outs.append((g, splits, out.clone(), lse.clone()))
    # run the first case again after the second: same answer as before
    g, splits, o0, l0 = outs[0]
    out = torch.empty_like(o0)
    lse = torch.empty_like(l0)
    _noalloc(g, splits, out, lse)
    torch.cuda.synchronize()
    _close(out, o0, lse, l0)


def test_noalloc_rejects_requests_beyond_its_scratch():
    """A call that would need more than the fixed scratch returns
    PKV_ERR_WORKSPACE and launches nothing (the output is left untouched)."""
    wl = workloads.make("tiny_decode", batch=64, h_q=64, h_kv=8, page_size=16,
                        len_lo=100, len_hi=200, pool_tokens=64 * 208 + 64)
    g = wl.to(DEV)
    splits = 64
    need = pkv.attn_workspace_size(g.q, g.k_cache, g.v_cache, g.page_table,
                                   g.cache_seqlens, g.max_seqlen_q, num_splits=splits)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
    out = torch.full((g.q.shape[0], g.q.shape[1], 128), 7.0, dtype=torch.bfloat16,
                     device=DEV)
    with pytest.raises(pkv.PkvError) as e:
        _noalloc(g, splits, out, None)
    assert e.value.code == -4
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_noalloc_serves_an_fp8_cache():
    """The no-allocation entry point with an fp8 (e4m3) cache: descales of 1,
    same answer as the regular entry point, nothing allocated."""
    wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=32, h_kv=8, batch=10,
                        len_lo=1, len_hi=2000, pool_tokens=10 * 2016 + 64, seed=131)
    g = wl.to(DEV)
    k8 = g.k_cache.float().to(torch.float8_e4m3fn)
    v8 = g.v_cache.float().to(torch.float8_e4m3fn)
    out = torch.empty(g.q.shape[0], 32, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(g.q.shape[0], 32, dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    pkv.attn_with_kvcache_noalloc(g.q, k8, v8, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                  g.max_seqlen_q, g.scale, out, lse=lse)
    after = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    assert after == before
    ref_o, ref_l = pkv.attn_with_kvcache_fp8(g.q, k8, v8, g.page_table, g.cache_seqlens,
                                             g.cu_seqlens_q, g.max_seqlen_q, g.scale,
                                             return_softmax_lse=True)
    torch.cuda.synchronize()
    _close(out, ref_o, lse, ref_l)
