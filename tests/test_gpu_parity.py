"""GPU-vs-oracle parity through the C ABI (libpkv) on seeded inputs.

Bars: integer outputs (page tables, kv_lens, slots) bit-exact; bf16 attention
outputs max |err| <= 2e-2 and mean |err| <= 2e-3 against the float64 oracle
(fp32 accumulation on the GPU), lse within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_203_gb300 as pkv
from paged_kv_cache_203_gb300 import workloads

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_flags():
    pkv.clear_error_flags()
    yield


def check_close(out, lse, ref_o, ref_l, what=""):
    o = out.float().cpu().numpy().reshape(ref_o.shape)
    err = np.abs(o - ref_o)
    assert np.isfinite(o).all(), what
    assert err.max() <= MAX_ABS, f"{what}: max|err| {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean|err| {err.mean():.3e}"
    if lse is not None:
        l = lse.cpu().numpy().reshape(ref_l.shape)
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(l), fin), what
        assert np.all(l[~fin] == ref_l[~fin]), what
        if fin.any():
            d = np.abs(l[fin] - ref_l[fin]).max()
            assert d <= LSE_ABS, f"{what}: max|dlse| {d:.3e}"


def oracle_attn(wl, **kw):
    args = dict(causal=wl.causal, window_left=wl.window_left)
    args.update(kw)
    topk = args.pop("topk", wl.topk_indices)
    pt = args.pop("page_table", wl.page_table)
    cs = args.pop("cache_seqlens", wl.cache_seqlens)
    d_v = wl.v_cache.shape[-1]
    return oracle.attention(
        oracle.bf16_bits(wl.q), oracle.bf16_bits(wl.k_cache),
        oracle.bf16_bits(wl.v_cache), np.asarray(pt.cpu()), np.asarray(cs.cpu()),
        wl.cu_seqlens_q.cpu().numpy(), wl.scale,
        topk=None if topk is None else topk.cpu().numpy(), d_v=d_v, **args)


def gpu_attn(g, **kw):
    args = dict(causal=g.causal, window_left=g.window_left, num_splits=g.num_splits,
                topk_indices=g.topk_indices)
    args.update(kw)
    pt = args.pop("page_table", g.page_table)
    cs = args.pop("cache_seqlens", g.cache_seqlens)
    out, lse = pkv.attn_with_kvcache(
        g.q, g.k_cache, g.v_cache, pt, cs, g.cu_seqlens_q, g.max_seqlen_q,
        g.scale, return_softmax_lse=True, **args)
    torch.cuda.synchronize()
    return out, lse


# ------------------------------------------------------------- page tables

@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_strided_page_table_bit_exact(page_size):
    wl = workloads.make("varlen_extend", page_size=page_size,
                        pool_pages=(1 << 17) // page_size, h_q=1, h_kv=1, d=8)
    n_cols = wl.page_table.shape[1]
    ref = oracle.strided_page_table(wl.req_to_token.numpy(),
                                    wl.req_pool_indices.numpy(), page_size, n_cols)
    got = pkv.strided_page_table(wl.req_to_token.to(DEV), wl.req_pool_indices.to(DEV),
                                 page_size, n_cols)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), ref)
    assert np.array_equal(ref, wl.page_table.numpy())
    assert pkv.get_error_flags() == 0


def test_swa_page_table_full_workload_bit_exact():
    """Sliding-window decode workload: batch 32, window 4096, prefill
    U[256, 2048], seq U[pf+1, 32768] -- table and kv_lens bit-exact."""
    wl = workloads.make("swa_decode", value_device="cpu", h_kv=1, d=8, h_q=1)
    w = wl.window
    pa_max = min(int(wl.prefill_lens.max()) + w, int(wl.seq_lens.max()))
    ref, ref_kv, bad = oracle.swa_page_table(
        wl.req_to_token.numpy(), wl.req_pool_indices.numpy(), wl.seq_lens.numpy(),
        wl.prefill_lens.numpy(), w, pa_max, fill=-7)
    assert bad == 0
    for idx_dtype in (torch.int64, torch.int32):
        dst = torch.full((len(wl.seq_lens), pa_max), -7, dtype=torch.int32, device=DEV)
        kv = torch.zeros(len(wl.seq_lens), dtype=torch.int32, device=DEV)
        pkv.build_swa_page_table(wl.req_to_token.to(DEV),
                                 wl.req_pool_indices.to(idx_dtype).to(DEV),
                                 wl.seq_lens.to(DEV), wl.prefill_lens.to(DEV), w, dst, kv)
        torch.cuda.synchronize()
        assert np.array_equal(kv.cpu().numpy(), ref_kv)
        assert np.array_equal(dst.cpu().numpy(), ref)  # tail untouched too
    assert pkv.get_error_flags() == 0


def test_swa_page_table_edge_cases():
    rng = np.random.default_rng(3)
    pool, ctx = 7, 64
    rtt = rng.permutation(pool * ctx).astype(np.int32).reshape(pool, ctx)
    cases = [(3, 10, 4), (5, 7, 4), (0, 10, 4), (8, 9, 1), (10, 4, 3), (4, 20, 0),
             (0, 0, 5), (6, 6, 6), (30, 64, 10)]
    for pf, sl, w in cases:
        pfl = np.zeros(pool, dtype=np.int32)
        pfl[2] = pf
        ref, ref_kv, _ = oracle.swa_page_table(rtt, [2], [sl], pfl, w, 48, fill=-3)
        dst = torch.full((1, 48), -3, dtype=torch.int32, device=DEV)
        kv = torch.zeros(1, dtype=torch.int32, device=DEV)
        pkv.build_swa_page_table(torch.from_numpy(rtt).to(DEV),
                                 torch.tensor([2], device=DEV),
                                 torch.tensor([sl], dtype=torch.int32, device=DEV),
                                 torch.from_numpy(pfl).to(DEV), w, dst, kv)
        torch.cuda.synchronize()
        assert kv.item() == ref_kv[0], (pf, sl, w)
        assert np.array_equal(dst.cpu().numpy(), ref), (pf, sl, w)
    # a row too long for dst: not written, kv_len -1, flag set, no trap
    dst = torch.full((1, 8), -3, dtype=torch.int32, device=DEV)
    kv = torch.zeros(1, dtype=torch.int32, device=DEV)
    pfl = np.zeros(pool, dtype=np.int32)
    pkv.build_swa_page_table(torch.from_numpy(rtt).to(DEV), torch.tensor([0], device=DEV),
                             torch.tensor([40], dtype=torch.int32, device=DEV),
                             torch.from_numpy(pfl).to(DEV), 20, dst, kv)
    torch.cuda.synchronize()
    assert kv.item() == -1 and torch.all(dst == -3)
    assert pkv.get_error_flags() & pkv.EFLAG_ROW_TOO_SHORT


def test_swa_page_table_malformed_rows_and_chunks():
    """Rows the builder must skip whole -- pool index out of range (rows 1,
    4), a source column past req_to_token's width (row 3), kv_len past dst's
    width (row 8) -- next to valid rows spanning up to four 1024-entry chunks,
    one ending exactly on a chunk boundary (row 2): table, kv_lens and flags
    equal the oracle's."""
    rng = np.random.default_rng(98)
    pool, ctx = 6, 5000
    rtt = rng.permutation(pool * ctx).astype(np.int32).reshape(pool, ctx)
    pfl = np.array([3, 0, 1500, 2500, 900, 1024], dtype=np.int32)
    rpi = np.array([0, 9, 1, 2, -1, 3, 4, 5, 3], dtype=np.int64)
    sl = np.array([1027, 5, 2048, 5001, 5, 3000, 4999, 4072, 5600], dtype=np.int32)
    window, W = 3000, 5000
    ref, ref_kv, n = oracle.swa_page_table(rtt, rpi, sl, pfl, window, W, fill=-5)
    assert n == 4 and list(ref_kv[[1, 3, 4, 8]]) == [-1] * 4
    assert list(ref_kv[[0, 2, 5, 6, 7]]) == [1027, 2048, 3000, 3900, 4024]
    dst = torch.full((len(rpi), W), -5, dtype=torch.int32, device=DEV)
    kv = torch.zeros(len(rpi), dtype=torch.int32, device=DEV)
    pkv.build_swa_page_table(torch.from_numpy(rtt).to(DEV), torch.from_numpy(rpi).to(DEV),
                             torch.from_numpy(sl).to(DEV), torch.from_numpy(pfl).to(DEV),
                             window, dst, kv)
    torch.cuda.synchronize()
    assert np.array_equal(kv.cpu().numpy(), ref_kv)
    assert np.array_equal(dst.cpu().numpy(), ref)
    assert pkv.get_error_flags() == pkv.EFLAG_SRC_OOB | pkv.EFLAG_ROW_TOO_SHORT


def test_topk_to_slots_bit_exact():
    wl = workloads.make("mla_topk_decode", batch=16, d_qk=64, d_v=32, h_q=1,
                        pool_pages=16 * 128 + 10)
    topk = wl.topk_indices.clone()
    topk[:, -5:] = -1
    topk[3, 7] = 8192       # == kv_len: out of range
    topk[5, 9] = -2         # below -1: out of range
    row_req = np.arange(16)
    ref, bad = oracle.topk_to_slots(topk.numpy(), row_req, wl.page_table.numpy(),
                                    wl.page_size, wl.cache_seqlens.numpy())
    assert bad == 2
    got = pkv.topk_to_slots(topk.to(DEV), wl.cu_seqlens_q.to(DEV), wl.page_table.to(DEV),
                            wl.cache_seqlens.to(DEV), wl.page_size)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), ref)
    assert pkv.get_error_flags() & pkv.EFLAG_TOPK_OOB


# ------------------------------------------------------------------ merge

@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.float32, torch.float32),
                                                (torch.bfloat16, torch.bfloat16),
                                                (torch.float32, torch.bfloat16)])
def test_merge_state(in_dtype, out_dtype):
    g = torch.Generator().manual_seed(5)
    n, h, d = 257, 8, 128
    va = torch.randn(n, h, d, generator=g).to(in_dtype)
    vb = torch.randn(n, h, d, generator=g).to(in_dtype)
    la = torch.randn(n, h, generator=g) * 4
    lb = torch.randn(n, h, generator=g) * 4
    la[0, :] = -float("inf")
    la[1, :] = -float("inf")
    lb[1, :] = -float("inf")
    lb[2, :3] = la[2, :3]
    ref_o, ref_l = oracle.merge_state(va.double().numpy(), la.double().numpy(),
                                      vb.double().numpy(), lb.double().numpy())
    vo = torch.empty(n, h, d, dtype=out_dtype, device=DEV)
    o, l = pkv.merge_state(va.to(DEV), la.to(DEV), vb.to(DEV), lb.to(DEV), v_out=vo)
    torch.cuda.synchronize()
    tol = 1e-5 if out_dtype == torch.float32 else 2e-2
    np.testing.assert_allclose(o.float().cpu().numpy(), ref_o, atol=tol, rtol=tol)
    lg = l.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(lg[fin], ref_l[fin], atol=1e-5)
    # in place into v_a
    va_d = va.to(DEV)
    pkv.merge_state(va_d, la.to(DEV), vb.to(DEV), lb.to(DEV), v_out=va_d)
    torch.cuda.synchronize()
    np.testing.assert_allclose(va_d.float().cpu().numpy(), ref_o, atol=2e-2, rtol=2e-2)


# -------------------------------------------------------------- attention

@pytest.mark.parametrize("num_splits", [1, 2, 0])
def test_tiny_decode_full_workload(num_splits):
    """Tiny paged decode: batch 4, 8/2 heads, D 128, page 1, seqlens U[1,256]."""
    wl = workloads.make("tiny_decode")
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=num_splits)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"splits={num_splits}")
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("num_splits", [4, 1, 0, 7])
def test_gqa_split_decode_reduced(num_splits):
    """GQA split-KV decode recipe (32/8 heads, D 128, page 16) at a size the
    oracle finishes quickly: 12 requests, lengths U[1, 3000]."""
    wl = workloads.make("gqa_split_decode", batch=12, len_lo=1, len_hi=3000,
                        pool_pages=4000)
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=num_splits)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"splits={num_splits}")


@pytest.mark.parametrize("batch,len_lo,len_hi", [(40, 300, 300), (40, 0, 900), (200, 1, 400)])
def test_split_decode_request_order(batch, len_lo, len_hi):
    """The fixed-split kernel serves the longest requests first (each CTA
    ranks the batch's key counts): equal lengths (ties by index), empty
    requests among long ones, and a batch above the ranking's limit (launch
    order kept) all match the oracle, and every request's in-kernel merge
    fires once."""
    wl = workloads.make("gqa_split_decode", batch=batch, len_lo=len_lo, len_hi=len_hi,
                        pool_pages=batch * (len_hi // 16 + 2) + 64, h_q=8, h_kv=2)
    if len_lo == 0:
        wl.cache_seqlens[::7] = 0
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=3)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"batch={batch}")
    assert pkv.get_error_flags() == 0


def test_split_states_merged_by_merge_state_equal_single_call():
    """Four explicit chunk calls (each chunk a request of its own page-table
    slice) combined with pkv_merge_state equal one unsplit call and the
    oracle: the split-KV route of the gqa split decode workload."""
    wl = workloads.make("gqa_split_decode", batch=6, len_lo=100, len_hi=2000,
                        pool_pages=2000)
    g = wl.to(DEV)
    P = wl.page_size
    acc_o = acc_l = None
    cs = wl.cache_seqlens.numpy()
    for c in range(4):
        pt_c = torch.zeros_like(wl.page_table)
        len_c = torch.zeros_like(wl.cache_seqlens)
        for b in range(len(cs)):
            lo, hi = oracle.split_bounds(int(cs[b]), 4, P)[c]
            p0 = lo // P
            pt_c[b, : pt_c.shape[1] - p0] = wl.page_table[b, p0:]
            len_c[b] = hi - lo
        o_c, l_c = gpu_attn(g, page_table=pt_c.to(DEV), cache_seqlens=len_c.to(DEV),
                            num_splits=1)
        if acc_o is None:
            acc_o, acc_l = o_c.float(), l_c
        else:
            acc_o, acc_l = pkv.merge_state(acc_o, acc_l, o_c.float(), l_c)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(acc_o, acc_l, ref_o, ref_l, "chunked + merge_state")


def test_swa_decode_reduced_prefill_aware():
    """Sliding-window decode recipe (64/8 heads, page 1, window 4096) with the
    table built on the GPU by the prefill-aware rule, then attended with no
    window; compared with the oracle's table + attention."""
    wl = workloads.make("swa_decode", batch=6, sl_hi=9000)
    g = wl.to(DEV)
    w = wl.window
    pa_max = min(int(wl.prefill_lens.max()) + w, int(wl.seq_lens.max()))
    dst = torch.zeros(6, pa_max, dtype=torch.int32, device=DEV)
    kv = torch.zeros(6, dtype=torch.int32, device=DEV)
    pkv.build_swa_page_table(g.req_to_token, g.req_pool_indices, g.seq_lens,
                             g.prefill_lens, w, dst, kv)
    ref_pt, ref_kv, _ = oracle.swa_page_table(
        wl.req_to_token.numpy(), wl.req_pool_indices.numpy(), wl.seq_lens.numpy(),
        wl.prefill_lens.numpy(), w, pa_max)
    out, lse = gpu_attn(g, page_table=dst, cache_seqlens=kv, num_splits=0)
    assert np.array_equal(kv.cpu().numpy(), ref_kv)
    ref_o, ref_l, _ = oracle_attn(wl, page_table=torch.from_numpy(ref_pt),
                                  cache_seqlens=torch.from_numpy(ref_kv))
    check_close(out, lse, ref_o, ref_l, "pa-swa")


def test_prefill_aware_with_no_prompt_equals_dense_window():
    """With prefill_len 0 the prefill-aware table keeps the last `window`
    tokens, i.e. dense attention with window_left = window - 1."""
    wl = workloads.make("swa_decode", batch=4, sl_hi=6000, pf_lo=0, pf_hi=0,
                        window=1000, h_q=16, h_kv=4)
    g = wl.to(DEV)
    dst = torch.zeros(4, 1000, dtype=torch.int32, device=DEV)
    kv = torch.zeros(4, dtype=torch.int32, device=DEV)
    pkv.build_swa_page_table(g.req_to_token, g.req_pool_indices, g.seq_lens,
                             g.prefill_lens, 1000, dst, kv)
    o1, l1 = gpu_attn(g, page_table=dst, cache_seqlens=kv)
    pt = g.req_to_token[g.req_pool_indices.long()].contiguous()
    o2, l2 = gpu_attn(g, page_table=pt, cache_seqlens=g.seq_lens, window_left=999)
    assert torch.allclose(o1.float(), o2.float(), atol=1e-2)
    assert torch.allclose(l1, l2, atol=1e-3)


@pytest.mark.parametrize("d,page_size,h_q,h_kv,q_len,window,causal", [
    (64, 16, 8, 8, 1, -1, False),      # MHA, D 64
    (128, 3, 6, 2, 1, -1, False),      # page size not a power of two
    (128, 64, 32, 2, 1, 100, False),   # group 16, window
    (128, 16, 64, 2, 1, -1, False),    # group 32: two row tiles per token
    (128, 16, 16, 4, 5, -1, True),     # short causal runs (MTP-style)
    (128, 1, 8, 1, 3, 40, True),       # causal + window, group 8
    (64, 8, 4, 2, 17, 7, True),        # rows across tiles, tiny window
])
def test_attention_variants(d, page_size, h_q, h_kv, q_len, window, causal):
    wl = workloads.make("tiny_decode", d=d, page_size=page_size, h_q=h_q, h_kv=h_kv,
                        q_len=q_len, window_left=window, causal=causal,
                        len_lo=q_len, len_hi=700, pool_tokens=8 * 700 * 2 + 64,
                        batch=5)
    g = wl.to(DEV)
    for splits in (1, 3):
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"splits={splits}")


def test_gqa_topk_sparse_decode():
    """Top-k lists (with -1 padding and duplicates) on a GQA cache."""
    wl = workloads.make("tiny_decode", batch=6, h_q=16, h_kv=4, page_size=16,
                        len_lo=300, len_hi=900, pool_tokens=6 * 912 + 64)
    cs = wl.cache_seqlens.numpy()
    g_ = torch.Generator().manual_seed(9)
    topk = torch.full((6, 256), -1, dtype=torch.int32)
    for b in range(6):
        n = 200 + b * 8
        topk[b, :n] = torch.randperm(int(cs[b]), generator=g_)[:n].to(torch.int32)
    topk[0, 250] = topk[0, 3]  # a duplicate counts twice
    wl.topk_indices = topk
    g = wl.to(DEV)
    for splits in (1, 2, 0):
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"topk splits={splits}")
    assert pkv.get_error_flags() == 0


def test_empty_rows_and_requests():
    """kv_len 0 -> out 0, lse -inf; a request with no new tokens is skipped."""
    wl = workloads.make("tiny_decode", batch=4, len_lo=5, len_hi=60)
    wl.cache_seqlens[1] = 0
    g = wl.to(DEV)
    for splits in (1, 4):
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"empty splits={splits}")
        assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    # request 2 has no new token: cu = [0,1,2,2,3] over 3 tokens
    wl3 = workloads.make("tiny_decode", batch=4, len_lo=5, len_hi=60)
    wl3.cu_seqlens_q = torch.tensor([0, 1, 2, 2, 3], dtype=torch.int32)
    wl3.q = wl3.q[:3].contiguous()
    g3 = wl3.to(DEV)
    out, lse = gpu_attn(g3, num_splits=2)
    ref_o, ref_l, _ = oracle_attn(wl3)
    check_close(out, lse, ref_o, ref_l, "zero-length request")


def test_bad_page_ids_are_skipped_and_flagged():
    """Out-of-pool page ids never trap: those keys are skipped (as the oracle
    skips them) and PKV_EFLAG_PAGE_OOB is raised."""
    wl = workloads.make("gqa_split_decode", batch=4, len_lo=100, len_hi=400,
                        pool_pages=200, h_q=8, h_kv=2)
    wl.page_table[1, 2] = 10_000_000
    wl.page_table[2, 0] = -5
    g = wl.to(DEV)
    for splits in (2, 0):
        pkv.clear_error_flags()
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, skipped = oracle_attn(wl)
        assert skipped > 0
        check_close(out, lse, ref_o, ref_l, f"bad pages splits={splits}")
        assert pkv.get_error_flags() & pkv.EFLAG_PAGE_OOB


@pytest.mark.parametrize("page_size,h_q,h_kv,q_len,window", [
    (1, 8, 2, 1, -1),    # the tiny decode shape
    (3, 16, 4, 1, 50),   # odd page size, window
    (16, 32, 8, 2, -1),  # two new tokens per request (causal)
    (1, 64, 8, 1, -1),   # 8 rows per KV head
    (8, 16, 1, 1, 100),  # one KV head, 16 rows
    (2, 32, 8, 4, 7)])   # 4 new tokens x group 4 = 16 rows, window
@pytest.mark.parametrize("batch", [9, 80])
def test_short_decode(page_size, h_q, h_kv, q_len, window, batch):
    """Page tables of at most 256 keys, no split: the short-decode kernels --
    a 4-CTA cluster per (request, KV head) for batches of at most 76 pairs
    (batch 9), one CTA per pair above that (batch 80).  NaN in every slot
    outside the valid rows, an empty request, an out-of-pool page id (skipped
    and flagged, as the oracle skips it), lengths up to the table's last key;
    no workspace; against the oracle and against the all-heads kernel with
    two splits."""
    len_hi = 256 - 256 % page_size
    wl = workloads.make("tiny_decode", d=128, page_size=page_size, h_q=h_q, h_kv=h_kv,
                        q_len=q_len, causal=q_len > 1, window_left=window, len_lo=q_len,
                        len_hi=len_hi, batch=batch,
                        pool_tokens=batch * (len_hi + page_size) + 64, seed=17 + page_size)
    assert wl.page_table.shape[1] * page_size <= 256
    wl.cache_seqlens[2] = 0
    wl.cache_seqlens[5] = wl.page_table.shape[1] * page_size  # the table's last key
    wl.cache_seqlens[5] = max(int(wl.cache_seqlens[5]), q_len)
    valid = torch.zeros(wl.k_cache.shape[0] * page_size, dtype=torch.bool)
    for b in range(batch):
        n = int(wl.cache_seqlens[b])
        j = torch.arange(n)
        slots = wl.page_table[b, j // page_size].long() * page_size + j % page_size
        valid[slots] = True
    valid = valid.view(-1, page_size)
    wl.k_cache[~valid] = float("nan")
    wl.v_cache[~valid] = float("nan")
    # out of the pool: the page of request 7's last key (inside any window)
    wl.page_table[7, (int(wl.cache_seqlens[7]) - 1) // page_size] = 10_000_000
    g = wl.to(DEV)
    assert pkv.attn_workspace_size(g.q, g.k_cache, g.v_cache, g.page_table, g.cache_seqlens,
                                   g.max_seqlen_q, num_splits=1) == 0
    ref_o, ref_l, skipped = oracle_attn(wl)
    assert skipped > 0
    for splits in (1, 0):
        pkv.clear_error_flags()
        out, lse = gpu_attn(g, num_splits=splits)
        check_close(out, lse, ref_o, ref_l, f"short decode splits={splits}")
        assert pkv.get_error_flags() == pkv.EFLAG_PAGE_OOB
        assert torch.all(out[2 * q_len:3 * q_len] == 0)
        assert torch.all(torch.isneginf(lse[2 * q_len:3 * q_len]))
    out2, lse2 = gpu_attn(g, num_splits=2)  # the all-heads kernel
    assert (out.float() - out2.float()).abs().max().item() <= MAX_ABS


@pytest.mark.parametrize("batch", [9, 80])
def test_short_decode_lengths_past_the_table(batch):
    """Short page tables (at most 256 keys) whose requests claim more keys
    than the table holds (up to 300 against 256): those keys are skipped, as
    the oracle skips them, and the row-too-short bit is set, on the cluster
    kernel (batch 9) and the one-CTA kernel (batch 80)."""
    wl = workloads.make("tiny_decode", batch=batch, len_lo=200, len_hi=256,
                        pool_tokens=batch * 256 + 64, seed=23)
    assert wl.page_table.shape[1] * wl.page_size <= 256
    wl.cache_seqlens[1] = 300
    wl.cache_seqlens[batch - 1] = 257
    g = wl.to(DEV)
    ref_o, ref_l, skipped = oracle_attn(wl)
    assert skipped > 0
    pkv.clear_error_flags()
    out, lse = gpu_attn(g, num_splits=1)
    check_close(out, lse, ref_o, ref_l, f"batch {batch}")
    assert pkv.get_error_flags() == pkv.EFLAG_ROW_TOO_SHORT


@pytest.mark.parametrize("one_launch", [False, True])
def test_table_then_attention_in_order_across_replays(one_launch):
    """The strided table builder and the short decode kernel are launched with
    programmatic serialization: the attention may start before the builder
    ends and must still read the table the builder wrote in the same step
    (with `one_launch`, the table is built inside the attention launch,
    which may start before the previous step's launch ends).
    The requests' pool rows and lengths are permuted before every replay of
    a captured step (and before every eager step), so a table read ahead of
    its write would show as another request's keys."""
    wl = workloads.make("tiny_decode")
    g = wl.to(DEV)
    batch, n_cols, P = wl.page_table.shape[0], wl.page_table.shape[1], wl.page_size
    rpi = g.req_pool_indices.clone()
    cs = g.cache_seqlens.clone()
    pt = torch.empty(batch, n_cols, dtype=torch.int32, device=DEV)
    out = torch.empty(g.q.shape[0], g.q.shape[1], wl.v_cache.shape[-1], dtype=torch.bfloat16,
                      device=DEV)
    lse = torch.empty(g.q.shape[0], g.q.shape[1], dtype=torch.float32, device=DEV)

    def step():
        if one_launch:
            pkv.strided_table_attn_with_kvcache(g.req_to_token, rpi, pt, g.q, g.k_cache,
                                                g.v_cache, cs, g.cu_seqlens_q, g.max_seqlen_q,
                                                g.scale, num_splits=1, out=out, lse=lse)
            return
        pkv.strided_page_table(g.req_to_token, rpi, P, n_cols, out=pt)
        pkv.attn_with_kvcache(g.q, g.k_cache, g.v_cache, pt, cs, g.cu_seqlens_q, g.max_seqlen_q,
                              g.scale, num_splits=1, out=out, lse=lse)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    perms = [np.roll(np.arange(batch), k) for k in range(1, batch)] + \
            [rng.permutation(batch) for _ in range(3)]
    for mode in ("graph", "eager"):
        for perm in perms:
            idx = torch.as_tensor(perm, device=DEV)
            rpi.copy_(g.req_pool_indices[idx])
            cs.copy_(g.cache_seqlens[idx])
            if mode == "graph":
                graph.replay()
            else:
                step()
            torch.cuda.synchronize()
            ref_pt = oracle.strided_page_table(wl.req_to_token.numpy(),
                                               wl.req_pool_indices.numpy()[perm], P, n_cols)
            assert np.array_equal(pt.cpu().numpy(), ref_pt), mode
            ref_o, ref_l, _ = oracle_attn(wl, page_table=torch.from_numpy(ref_pt),
                                          cache_seqlens=wl.cache_seqlens[torch.as_tensor(perm)])
            check_close(out, lse, ref_o, ref_l, f"{mode} perm={perm.tolist()}")
    assert pkv.get_error_flags() == 0


def _two_call_step(g, rtt, rpi, pt, cu, q, n_cols, num_splits):
    """The builder followed by the attention: (table, out, lse, error bits)."""
    pkv.clear_error_flags()
    table = pkv.strided_page_table(rtt, rpi, g.page_size, n_cols, out=pt.clone())
    out, lse = pkv.attn_with_kvcache(q, g.k_cache, g.v_cache, table, g.cache_seqlens, cu,
                                     g.max_seqlen_q, g.scale, causal=g.causal,
                                     window_left=g.window_left, num_splits=num_splits,
                                     return_softmax_lse=True)
    torch.cuda.synchronize()
    return table, out, lse, pkv.get_error_flags()


def _one_call_step(g, rtt, rpi, pt, cu, q, num_splits):
    pkv.clear_error_flags()
    table = pt.clone()
    out, lse = pkv.strided_table_attn_with_kvcache(
        rtt, rpi, table, q, g.k_cache, g.v_cache, g.cache_seqlens, cu, g.max_seqlen_q, g.scale,
        causal=g.causal, window_left=g.window_left, num_splits=num_splits,
        return_softmax_lse=True)
    torch.cuda.synchronize()
    return table, out, lse, pkv.get_error_flags()


@pytest.mark.parametrize("batch,page_size,idx64,narrow,q_len,window", [
    (4, 1, True, False, 1, -1),    # the tiny decode shape: cluster kernel
    (9, 3, False, True, 1, -1),    # cluster kernel, odd page size, narrow token pool
    (9, 2, True, False, 2, 40),    # two new tokens (causal) per request, a window
    (80, 1, True, True, 1, -1),    # one CTA per (request, KV head)
    (80, 16, False, False, 2, 7)])
def test_strided_table_attention_one_launch(batch, page_size, idx64, narrow, q_len, window):
    """pkv_strided_table_attn_with_kvcache served by the short kernels (the
    table built inside the attention launch): the table it writes is
    bit-exact against the oracle's strided table, the attention matches the
    oracle over that table, and table, out, lse and error bits are identical
    to the builder followed by pkv_attn_with_kvcache.  In the same launch: a
    request whose pool row lies outside req_to_token (its row all -1,
    SRC_OOB, its keys skipped with PAGE_OOB), a request with no new tokens
    (its table row still written, no output rows), and with `narrow` a token
    pool narrower than the table's last column (that column -1, SRC_OOB)."""
    len_hi = 256 - 256 % page_size
    wl = workloads.make("tiny_decode", page_size=page_size, batch=batch, len_lo=q_len,
                        len_hi=len_hi, pool_tokens=batch * (len_hi + page_size) + 64,
                        q_len=q_len, causal=q_len > 1, window_left=window,
                        h_q=16 if q_len > 1 else 8, h_kv=4 if q_len > 1 else 2,
                        seed=31 + page_size + q_len)
    P, n_cols = page_size, wl.page_table.shape[1]
    assert n_cols * P <= 256
    rtt = wl.req_to_token
    if narrow:
        rtt = rtt[:, :(n_cols - 1) * P]  # a view: rows keep their stride
    rpi = wl.req_pool_indices.clone().to(torch.int64 if idx64 else torch.int32)
    rpi[1] = rtt.shape[0] + 3
    # request 2 has no new tokens: its query rows are dropped
    cu = wl.cu_seqlens_q.clone()
    cu[3:] -= q_len
    q = torch.cat([wl.q[:2 * q_len], wl.q[3 * q_len:]])
    # expected table: the oracle's strided table where the source lies in
    # the token pool, -1 (the documented value) where it does not
    full = np.full((batch, n_cols), -1, dtype=np.int32)
    rows = rpi.numpy().astype(np.int64)
    ok = (rows >= 0) & (rows < rtt.shape[0])
    n_in = -(-rtt.shape[1] // P)  # columns c with c * P inside the pool's width
    assert n_in == (n_cols - 1 if narrow else n_cols)
    full[ok, :n_in] = oracle.strided_page_table(
        np.ascontiguousarray(rtt.numpy()), rows[ok], P, n_in)
    ref_o, ref_l, skipped = oracle.attention(
        oracle.bf16_bits(q), oracle.bf16_bits(wl.k_cache), oracle.bf16_bits(wl.v_cache),
        full, wl.cache_seqlens.numpy(), cu.numpy(), wl.scale, causal=wl.causal,
        window_left=wl.window_left, d_v=wl.v_cache.shape[-1])
    assert skipped > 0
    g = wl.to(DEV)
    args = (g, rtt.to(DEV), rpi.to(DEV), torch.full((batch, n_cols), -5, dtype=torch.int32,
                                                    device=DEV), cu.to(DEV), q.to(DEV))
    with pytest.raises(pkv.PkvError) as e:  # every descriptor arrives in its place
        pkv.strided_table_attn_with_kvcache(
            args[1], args[2], args[3], args[5], g.k_cache, g.v_cache, g.cache_seqlens, args[4],
            g.max_seqlen_q, g.scale, num_splits=1, lse=torch.empty(1, 1, device=DEV))
    assert e.value.code == -1
    t1, o1, l1, f1 = _one_call_step(*args, num_splits=1)
    assert np.array_equal(t1.cpu().numpy(), full)
    check_close(o1, l1, ref_o, ref_l, f"one launch batch={batch} P={P}")
    want = pkv.EFLAG_SRC_OOB | pkv.EFLAG_PAGE_OOB
    assert (f1 & want) == want and (f1 & ~(want | pkv.EFLAG_ROW_TOO_SHORT)) == 0
    t2, o2, l2, f2 = _two_call_step(*args, n_cols=n_cols, num_splits=1)
    assert torch.equal(t1, t2) and torch.equal(o1, o2) and torch.equal(l1, l2)
    assert f1 == f2


def test_strided_table_attention_two_launches():
    """Calls the short kernels do not serve (a split asked for; a table of
    more than 256 keys) run the builder, then the attention: the same table,
    and the attention of the two separate calls."""
    for kw, splits in ((dict(batch=6), 2), (dict(batch=6, len_lo=300, len_hi=900), 1)):
        wl = workloads.make("tiny_decode", pool_tokens=8192, seed=41, **kw)
        n_cols = wl.page_table.shape[1]
        g = wl.to(DEV)
        args = (g, g.req_to_token, g.req_pool_indices,
                torch.full((wl.page_table.shape[0], n_cols), -5, dtype=torch.int32, device=DEV),
                g.cu_seqlens_q, g.q)
        t1, o1, l1, f1 = _one_call_step(*args, num_splits=splits)
        assert np.array_equal(t1.cpu().numpy(), wl.page_table.numpy())
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(o1, l1, ref_o, ref_l, f"two launches {kw} splits={splits}")
        t2, o2, l2, f2 = _two_call_step(*args, n_cols=n_cols, num_splits=splits)
        assert torch.equal(t1, t2) and f1 == f2 == 0
        assert (o1.float() - o2.float()).abs().max().item() <= MAX_ABS


# ------------------------------------- full-size workloads, every output row

@pytest.mark.parametrize("num_splits", [4, 0])
def test_gqa_split_decode_full_size(num_splits):
    """Full batched GQA split-KV decode workload (batch 64, 32/8 heads,
    seqlens U[512, 8192], 40k-page pool) in the bench's launch configuration
    (4 key chunks) and with the library's balanced schedule (requests cut at
    CTA boundaries, partial last tiles): every (token, head) row of out and
    lse against the oracle."""
    g = workloads.make("gqa_split_decode", value_device=DEV)
    out, lse = gpu_attn(g, num_splits=num_splits)
    ref_o, ref_l, _ = oracle.attention(
        oracle.bf16_bits(g.q), oracle.bf16_bits(g.k_cache), oracle.bf16_bits(g.v_cache),
        g.page_table.cpu().numpy(), g.cache_seqlens.cpu().numpy(),
        g.cu_seqlens_q.cpu().numpy(), g.scale)
    check_close(out, lse, ref_o, ref_l, f"full size, splits {num_splits}")
    assert pkv.get_error_flags() == 0


def test_swa_decode_full_size():
    """Full sliding-window decode workload (batch 32, 64/8 heads, window
    4096, seq up to 32768) as the bench runs it: GPU-built table, then the
    attention with the library's split choice; every row."""
    g = workloads.make("swa_decode", value_device=DEV)
    w = g.window
    pa_max = min(int(g.prefill_lens.max()) + w, int(g.seq_lens.max()))
    dst = torch.zeros(32, pa_max, dtype=torch.int32, device=DEV)
    kv = torch.zeros(32, dtype=torch.int32, device=DEV)
    pkv.build_swa_page_table(g.req_to_token, g.req_pool_indices, g.seq_lens,
                             g.prefill_lens, w, dst, kv)
    out, lse = gpu_attn(g, page_table=dst, cache_seqlens=kv, num_splits=0)
    ref_o, ref_l, _ = oracle.attention(
        oracle.bf16_bits(g.q), oracle.bf16_bits(g.k_cache), oracle.bf16_bits(g.v_cache),
        dst.cpu().numpy(), kv.cpu().numpy(), g.cu_seqlens_q.cpu().numpy(), g.scale)
    ref_pt, ref_kv, _ = oracle.swa_page_table(
        g.req_to_token.cpu().numpy(), g.req_pool_indices.cpu().numpy(),
        g.seq_lens.cpu().numpy(), g.prefill_lens.cpu().numpy(), w, pa_max)
    assert np.array_equal(kv.cpu().numpy(), ref_kv)
    kvn = ref_kv
    d = dst.cpu().numpy()
    for b in range(32):
        assert np.array_equal(d[b, :kvn[b]], ref_pt[b, :kvn[b]])
    check_close(out, lse, ref_o, ref_l, "swa full size")


# ------------------------------------------- loader coverage (TMA / cp.async)

@pytest.mark.parametrize("page_size,q_len,window,causal", [
    (8, 1, -1, False), (32, 1, 300, False), (64, 4, -1, True), (128, 1, -1, False),
    (128, 3, 200, True), (16, 2, 0, True),
])
def test_page_box_sizes(page_size, q_len, window, causal):
    """Page sizes served by whole-page tensor-map boxes (multiples of 8, and
    pages longer than a 64-key stage), with windows and causal runs."""
    wl = workloads.make("tiny_decode", d=128, page_size=page_size, h_q=16, h_kv=4,
                        q_len=q_len, window_left=window, causal=causal,
                        len_lo=q_len, len_hi=1500, batch=6,
                        pool_tokens=6 * (1500 + page_size) * 2)
    g = wl.to(DEV)
    for splits in (1, 3, 0):  # 0: balanced all-heads schedule (page boxes when P % 16 == 0)
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"P={page_size} splits={splits}")
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("page_size", [16, 3, 64])
def test_garbage_outside_valid_rows_never_leaks(page_size):
    """Every cache row that is not one of a request's first kv_len keys is
    NaN (e.g. the unused tail of the last page): outputs must equal the
    oracle's, which reads only valid rows."""
    wl = workloads.make("tiny_decode", page_size=page_size, h_q=8, h_kv=2, batch=5,
                        len_lo=1, len_hi=900, pool_tokens=5 * (900 + 64) * 2)
    valid = torch.zeros(wl.k_cache.shape[0] * page_size, dtype=torch.bool)
    for b in range(5):
        n = int(wl.cache_seqlens[b])
        j = torch.arange(n)
        slots = wl.page_table[b, j // page_size].long() * page_size + j % page_size
        valid[slots] = True
    valid = valid.view(-1, page_size)
    wl.k_cache[~valid] = float("nan")
    wl.v_cache[~valid] = float("nan")
    g = wl.to(DEV)
    for splits in (1, 4, 0):
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"nan P={page_size} splits={splits}")


@pytest.mark.parametrize("page_size,h_q,h_kv,q_len,window,causal", [
    (1, 64, 8, 1, -1, False),     # sliding-window decode shape: 8 KV heads, group 8
    (2, 16, 8, 2, -1, True),      # 16 rows per KV head: a causal pair of tokens
    (5, 8, 4, 4, 30, True),       # window + causal, group 2
    (7, 4, 1, 4, -1, True),       # one KV head, group 4
    (3, 2, 2, 16, 50, True),      # group 1, 16 query tokens per request
    (1, 6, 2, 1, 0, False),       # window 0: the diagonal key only
])
def test_small_page_all_heads_decode(page_size, h_q, h_kv, q_len, window, causal):
    """Small pages (< 8 slots) with at most 16 query rows per KV head run the
    kernel that covers every KV head of a request in one CTA; unused slots hold
    NaN, one page id is out of the pool (that key is skipped and flagged)."""
    wl = workloads.make("tiny_decode", d=128, page_size=page_size, h_q=h_q, h_kv=h_kv,
                        q_len=q_len, window_left=window, causal=causal,
                        len_lo=q_len, len_hi=1300, batch=6,
                        pool_tokens=6 * (1300 + page_size) * 2)
    valid = torch.zeros(wl.k_cache.shape[0] * page_size, dtype=torch.bool)
    for b in range(6):
        n = int(wl.cache_seqlens[b])
        j = torch.arange(n)
        slots = wl.page_table[b, j // page_size].long() * page_size + j % page_size
        valid[slots] = True
    valid = valid.view(-1, page_size)
    wl.k_cache[~valid] = float("nan")
    wl.v_cache[~valid] = float("nan")
    wl.cache_seqlens[4] = 0
    if int(wl.cache_seqlens[2]) > 2 * page_size:
        wl.page_table[2, 1] = 50_000_000
    g = wl.to(DEV)
    for splits in (1, 3, 0):
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"P={page_size} splits={splits}")
    assert (pkv.get_error_flags() & ~pkv.EFLAG_PAGE_OOB) == 0


def test_small_page_balanced_schedule_mixed_batch():
    """The balanced schedule (num_splits 0) lays the batch's 16-key tiles end
    to end over one CTA per SM: requests of very different lengths, requests
    with no cached key and requests with no new token all land where the
    oracle puts them."""
    batch = 60
    wl = workloads.make("tiny_decode", d=128, page_size=1, h_q=16, h_kv=4, batch=batch,
                        len_lo=1, len_hi=3000, pool_tokens=batch * 3000 + 64, seed=77)
    cs = wl.cache_seqlens
    cs[3] = 0
    cs[17] = 0
    cs[40] = wl.page_table.shape[1]  # the longest request the table holds
    no_tok = {5, 6, 31, 59}
    cu = [0]
    for b in range(batch):
        cu.append(cu[-1] + (0 if b in no_tok else 1))
    keep = [b for b in range(batch) if b not in no_tok]
    wl.cu_seqlens_q = torch.tensor(cu, dtype=torch.int32)
    wl.q = wl.q[keep].contiguous()
    g = wl.to(DEV)
    for splits in (0, 1, 2):
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"mixed batch splits={splits}")
    assert pkv.get_error_flags() == 0


def test_small_page_batch_beyond_the_balanced_limit():
    """More requests than the balanced schedule handles (2048): the library's
    split choice falls back to fixed splits of the all-heads kernel; every
    row against the oracle."""
    batch = 2100  # tables of 300 keys: wider than the short-decode kernel serves
    wl = workloads.make("tiny_decode", d=128, page_size=1, h_q=16, h_kv=8, batch=batch,
                        len_lo=1, len_hi=300, pool_tokens=batch * 300 + 64, seed=91)
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=0)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, "batch 2100")
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("page_size,q_len,window", [(16, 8, 100), (32, 4, -1), (64, 2, 0)])
def test_page_box_balanced_sixteen_rows_per_kv_head(page_size, q_len, window):
    """Page boxes under the balanced schedule with up to 16 query rows per KV
    head (causal runs of new tokens, windows), NaN in every unused slot."""
    h_kv = 8
    h_q = h_kv * (16 // q_len)  # q_len * group = 16 rows per KV head
    wl = workloads.make("tiny_decode", d=128, page_size=page_size, h_q=h_q, h_kv=h_kv,
                        q_len=q_len, window_left=window, causal=True, len_lo=q_len,
                        len_hi=1500, batch=7, pool_tokens=7 * (1500 + page_size) * 2, seed=31)
    valid = torch.zeros(wl.k_cache.shape[0] * page_size, dtype=torch.bool)
    for b in range(7):
        n = int(wl.cache_seqlens[b])
        j = torch.arange(n)
        slots = wl.page_table[b, j // page_size].long() * page_size + j % page_size
        valid[slots] = True
    valid = valid.view(-1, page_size)
    wl.k_cache[~valid] = float("nan")
    wl.v_cache[~valid] = float("nan")
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=0)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"P={page_size} q_len={q_len}")
    assert pkv.get_error_flags() == 0


def test_cascade_shared_prefix_attention():
    """Cascade attention through the library: every request shares the same
    prefix pages (a common system prompt) and owns its suffix pages; prefix
    call + suffix call + state merge equals the oracle's single call over
    the concatenated table (causal runs of new tokens at the suffix end)."""
    P, batch, q_len = 16, 5, 3
    pre_pages = 6
    wl = workloads.make("tiny_decode", d=128, page_size=P, h_q=16, h_kv=4, q_len=q_len,
                        causal=True, len_lo=q_len + 1, len_hi=500, batch=batch,
                        pool_tokens=(batch * 520 + pre_pages * P) * 2, seed=55)
    n_own = [-(-int(wl.cache_seqlens[b]) // P) for b in range(batch)]
    used = set()
    for b in range(batch):
        used.update(wl.page_table[b, :n_own[b]].tolist())
    free = [p for p in range(wl.k_cache.shape[0]) if p not in used]
    shared = torch.tensor(free[1::2][:pre_pages], dtype=torch.int32)  # pool pages no request owns
    assert shared.numel() == pre_pages
    full_pt = torch.zeros(batch, pre_pages + wl.page_table.shape[1], dtype=torch.int32)
    suf_pt = torch.zeros(batch, wl.page_table.shape[1], dtype=torch.int32)
    for b in range(batch):
        own = wl.page_table[b, :n_own[b]]
        full_pt[b, :pre_pages] = shared
        full_pt[b, pre_pages:pre_pages + n_own[b]] = own
        suf_pt[b, :n_own[b]] = own
    suf_len = wl.cache_seqlens.clone()
    pre_len = torch.full((batch,), pre_pages * P, dtype=torch.int32)
    full_len = pre_len + suf_len
    wl.page_table, wl.cache_seqlens = full_pt, full_len
    g = wl.to(DEV)
    # the prefix call reads the shared pages (the first columns of the full
    # table); the suffix call reads each request's own pages
    out, lse = pkv.cascade_attn_with_kvcache(
        g.q, g.k_cache, g.v_cache, full_pt.to(DEV), pre_len.to(DEV), suf_pt.to(DEV),
        suf_len.to(DEV), g.cu_seqlens_q, q_len, g.scale, causal=True, return_softmax_lse=True)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, "cascade")
    assert pkv.get_error_flags() == 0


def test_head_major_cache_layout():
    """A cache laid out [pages, H_kv, P, D] (head outside position) is read
    through its strides; results equal the oracle's."""
    wl = workloads.make("tiny_decode", page_size=16, h_q=8, h_kv=2, batch=4,
                        len_lo=10, len_hi=700, pool_tokens=4 * 720 * 2)
    k_hm = wl.k_cache.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    v_hm = wl.v_cache.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert k_hm.stride(1) == 128 and k_hm.stride(2) == 16 * 128
    g = wl.to(DEV)
    g.k_cache = k_hm.to(DEV).permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    g.v_cache = v_hm.to(DEV).permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    for splits in (2, 0):
        out, lse = gpu_attn(g, num_splits=splits)
        ref_o, ref_l, _ = oracle_attn(wl)
        check_close(out, lse, ref_o, ref_l, f"head-major splits={splits}")


# ------------------------------------------------ varlen extend (tcgen05 path)

@pytest.mark.parametrize("page_size,window,causal", [
    (64, -1, True), (16, -1, True), (128, -1, True), (64, 300, True), (64, -1, False),
])
def test_varlen_extend_reduced(page_size, window, causal):
    """Varlen causal extend recipe (32/8 heads, D 128) at oracle-friendly
    size: 4 requests, new U[64, 700] on a prefix U[0, 900] (ragged q tiles,
    prefix 0 allowed)."""
    wl = workloads.make("varlen_extend", batch=4, new_lo=64, new_hi=700, prefix_lo=0,
                        prefix_hi=900, page_size=page_size,
                        pool_pages=4 * (1600 // page_size + 2) + 8, window_left=window)
    wl.causal = causal
    g = wl.to(DEV)
    out, lse = gpu_attn(g)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"extend P={page_size} w={window} c={causal}")
    assert pkv.get_error_flags() == 0


def test_varlen_extend_garbage_and_bad_pages():
    """Extend with NaN everywhere outside the requests' valid rows, plus an
    out-of-pool page id: the bad page's keys are skipped and flagged,
    nothing else changes."""
    P = 64
    wl = workloads.make("varlen_extend", batch=3, new_lo=100, new_hi=400, prefix_lo=50,
                        prefix_hi=600, page_size=P, pool_pages=3 * 17 + 10)
    valid = torch.zeros(wl.k_cache.shape[0] * P, dtype=torch.bool)
    for b in range(3):
        j = torch.arange(int(wl.cache_seqlens[b]))
        valid[wl.page_table[b, j // P].long() * P + j % P] = True
    valid = valid.view(-1, P)
    wl.k_cache[~valid] = float("nan")
    wl.v_cache[~valid] = float("nan")
    wl.page_table[1, 1] = 1 << 30
    g = wl.to(DEV)
    out, lse = gpu_attn(g)
    ref_o, ref_l, skipped = oracle_attn(wl)
    assert skipped > 0
    check_close(out, lse, ref_o, ref_l, "extend garbage/bad page")
    assert pkv.get_error_flags() & pkv.EFLAG_PAGE_OOB


def test_varlen_extend_full_size():
    """Full varlen extend workload (batch 8, new U[128, 2048], prefix
    U[0, 4096], page 64) as the bench runs it; every row."""
    g = workloads.make("varlen_extend", value_device=DEV)
    out, lse = gpu_attn(g)
    ref_o, ref_l, _ = oracle.attention(
        oracle.bf16_bits(g.q), oracle.bf16_bits(g.k_cache), oracle.bf16_bits(g.v_cache),
        g.page_table.cpu().numpy(), g.cache_seqlens.cpu().numpy(),
        g.cu_seqlens_q.cpu().numpy(), g.scale, causal=True)
    check_close(out, lse, ref_o, ref_l, "extend full size")
    assert pkv.get_error_flags() == 0


def test_extend_shapes_with_negative_scale_use_the_decode_path():
    """A non-positive softmax scale is served (by the decode kernel) with the
    same results as the oracle."""
    wl = workloads.make("varlen_extend", batch=2, new_lo=64, new_hi=200, prefix_hi=300,
                        pool_pages=40)
    wl.scale = -0.05
    g = wl.to(DEV)
    out, lse = gpu_attn(g)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, "negative scale")


# --------------------------------------------- MLA top-k sparse decode (tcgen05)

def _mla_reduced(batch=6, kv_len=1500, topk=600, seed=None):
    return workloads.make("mla_topk_decode", batch=batch, kv_len=kv_len, topk=topk,
                          pool_pages=batch * (kv_len // 64 + 1) + 4, seed=seed)


@pytest.mark.parametrize("num_splits", [1, 2, 0, 5])
def test_mla_topk_decode_reduced(num_splits):
    """Absorbed MLA (128 heads, 576/512, one latent head, page 64) over
    top-k lists with -1 padding and a duplicate, against the oracle."""
    wl = _mla_reduced()
    wl.topk_indices[:, -37:] = -1
    wl.topk_indices[2, 5] = wl.topk_indices[2, 6]  # a duplicate counts twice
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=num_splits)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"mla splits={num_splits}")
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_mla_topk_fp8(num_splits):
    """Absorbed MLA over an fp8 latent cache: the codes gathered and widened
    to f16 inside the kernel, q rounded to e4m3, per-request k / v descales;
    top-k lists with -1 padding, a duplicate and an out-of-range entry
    (skipped and flagged); against the fp8 oracle."""
    wl = _mla_reduced()
    wl.topk_indices[:, -37:] = -1
    wl.topk_indices[2, 5] = wl.topk_indices[2, 6]
    wl.topk_indices[4, 9] = int(wl.cache_seqlens[0]) + 5  # past kv_len
    B = wl.cache_seqlens.shape[0]
    k8 = wl.k_cache.float().to(torch.float8_e4m3fn)
    gen = torch.Generator().manual_seed(31 + num_splits)
    kd = torch.rand(B, 1, generator=gen) * 1.5 + 0.5
    vd = torch.rand(B, 1, generator=gen) * 1.5 + 0.5
    g = wl.to(DEV)
    k8d = k8.to(DEV)
    out, lse = pkv.attn_with_kvcache_fp8(
        g.q, k8d, k8d[..., :512], g.page_table, g.cache_seqlens, g.cu_seqlens_q,
        g.max_seqlen_q, g.scale, topk_indices=g.topk_indices, k_descale=kd.to(DEV),
        v_descale=vd.to(DEV), num_splits=num_splits, return_softmax_lse=True)
    torch.cuda.synchronize()
    codes = k8.view(torch.uint8).numpy()
    ref_o, ref_l, skipped = oracle.attention_fp8(
        oracle.bf16_bits(wl.q), codes, codes[..., :512], wl.page_table.numpy(),
        wl.cache_seqlens.numpy(), wl.cu_seqlens_q.numpy(), wl.scale, k_descale=kd.numpy(),
        v_descale=vd.numpy(), topk=wl.topk_indices.numpy())
    assert skipped > 0
    check_close(out, lse, ref_o, ref_l, f"mla fp8 splits={num_splits}")
    assert pkv.get_error_flags() == pkv.EFLAG_TOPK_OOB


@pytest.mark.parametrize("num_splits", [1, 3])
def test_mla_topk_reference_max_rises(num_splits):
    """Scores that grow along the list (rope parts of later tiles' keys scaled up) make
    the softmax raise its reference max mid-list, so the accumulated output
    rows are rescaled before the next product; against the oracle."""
    wl = _mla_reduced(batch=3, kv_len=1200, topk=640, seed=77)
    P = wl.page_size
    k = wl.k_cache.view(-1, wl.k_cache.shape[-1])
    for t in range(wl.q.shape[0]):
        lst = wl.topk_indices[t]
        for j, idx in enumerate(lst.tolist()):
            if idx < 0:
                continue
            slot = int(wl.page_table[t, idx // P]) * P + idx % P
            # the rope columns only: the value row (the first 512) is unchanged
            k[slot, 512:] = (k[slot, 512:].float() * (1.0 + 3.0 * (j // 64))).to(torch.bfloat16)
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=num_splits)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"mla rising scores splits={num_splits}")
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("batch,topk,seed", [(100, 256, 5), (90, 200, 6), (77, 64, 7)])
def test_mla_topk_more_tokens_than_sm_pairs(batch, topk, seed):
    """More tokens than SM pairs (clusters in a second wave) with the
    library's split choice; ragged last tiles, -1 padding, a duplicate, an
    out-of-range entry (skipped, flagged) and a row of only -1; every row
    against the oracle."""
    wl = _mla_reduced(batch=batch, kv_len=700, topk=topk, seed=seed)
    wl.topk_indices[:, -9:] = -1
    wl.topk_indices[2, 5] = wl.topk_indices[2, 6]
    wl.topk_indices[7, 1] = 700                # == kv_len
    wl.topk_indices[batch - 1, :] = -1         # nothing to attend
    g = wl.to(DEV)
    pkv.clear_error_flags()
    out, lse = gpu_attn(g, num_splits=0)
    ref_o, ref_l, skipped = oracle_attn(wl)
    assert skipped == 1
    check_close(out, lse, ref_o, ref_l, f"mla batch={batch} topk={topk}")
    assert pkv.get_error_flags() == pkv.EFLAG_TOPK_OOB
    assert torch.all(out[batch - 1] == 0) and torch.all(torch.isneginf(lse[batch - 1]))


def test_mla_topk_fp8_more_tokens_than_sm_pairs():
    """More tokens than SM pairs over an fp8 latent cache (codes widened to
    f16, q rounded to e4m3, per-request descales); against the fp8 oracle."""
    wl = _mla_reduced(batch=80, kv_len=700, topk=192, seed=8)
    wl.topk_indices[:, -5:] = -1
    B = wl.cache_seqlens.shape[0]
    k8 = wl.k_cache.float().to(torch.float8_e4m3fn)
    gen = torch.Generator().manual_seed(41)
    kd = torch.rand(B, 1, generator=gen) * 1.5 + 0.5
    vd = torch.rand(B, 1, generator=gen) * 1.5 + 0.5
    g = wl.to(DEV)
    k8d = k8.to(DEV)
    pkv.clear_error_flags()
    out, lse = pkv.attn_with_kvcache_fp8(
        g.q, k8d, k8d[..., :512], g.page_table, g.cache_seqlens, g.cu_seqlens_q,
        g.max_seqlen_q, g.scale, topk_indices=g.topk_indices, k_descale=kd.to(DEV),
        v_descale=vd.to(DEV), num_splits=0, return_softmax_lse=True)
    torch.cuda.synchronize()
    codes = k8.view(torch.uint8).numpy()
    ref_o, ref_l, _ = oracle.attention_fp8(
        oracle.bf16_bits(wl.q), codes, codes[..., :512], wl.page_table.numpy(),
        wl.cache_seqlens.numpy(), wl.cu_seqlens_q.numpy(), wl.scale, k_descale=kd.numpy(),
        v_descale=vd.numpy(), topk=wl.topk_indices.numpy())
    check_close(out, lse, ref_o, ref_l, "mla fp8, more tokens than SM pairs")
    assert pkv.get_error_flags() == 0


def test_mla_topk_bad_indices_and_empty_rows():
    """Out-of-range top-k entries are skipped and flagged; a row of only -1
    gives out 0 / lse -inf."""
    wl = _mla_reduced(batch=4, kv_len=700, topk=256)
    wl.topk_indices[1, 3] = 700          # == kv_len
    wl.topk_indices[1, 9] = -4           # below -1
    wl.topk_indices[3, :] = -1           # nothing to attend
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=2)
    ref_o, ref_l, skipped = oracle_attn(wl)
    assert skipped == 2
    check_close(out, lse, ref_o, ref_l, "mla bad indices")
    assert torch.all(out[3] == 0) and torch.all(torch.isneginf(lse[3]))
    assert pkv.get_error_flags() & pkv.EFLAG_TOPK_OOB


def test_mla_topk_full_size():
    """Full MLA top-k workload (batch 128, kv_len 8192, top-k 2048) in the
    bench's launch configuration; every (token, head) row."""
    g = workloads.make("mla_topk_decode", value_device=DEV)
    out, lse = gpu_attn(g)
    kb = oracle.bf16_bits(g.k_cache)
    ref_o, ref_l, _ = oracle.attention(
        oracle.bf16_bits(g.q), kb, kb, g.page_table.cpu().numpy(),
        g.cache_seqlens.cpu().numpy(), g.cu_seqlens_q.cpu().numpy(), g.scale,
        topk=g.topk_indices.cpu().numpy(), d_v=512)
    check_close(out, lse, ref_o, ref_l, "mla full size")
    assert pkv.get_error_flags() == 0


# ------------------------------------------- local (chunked) attention batches

def _lvb_run(chunk, P, cu, kv, pt, cap, bt_cols=None):
    """GPU build and oracle build of the virtual requests; every output
    array and the info words must agree bit for bit."""
    cols = bt_cols if bt_cols is not None else max(chunk // P, 1)
    cu_t = torch.as_tensor(np.asarray(cu), dtype=torch.int32).to(DEV)
    kv_t = torch.as_tensor(np.asarray(kv), dtype=torch.int32).to(DEV)
    pt_t = torch.as_tensor(np.asarray(pt), dtype=torch.int32).to(DEV)
    # outputs pre-filled with garbage: every entry must be written
    out = (torch.full((cap,), -7, dtype=torch.int32, device=DEV),
           torch.full((cap + 1,), -7, dtype=torch.int32, device=DEV),
           torch.full((cap,), -7, dtype=torch.int32, device=DEV),
           torch.full((cap, cols), -7, dtype=torch.int32, device=DEV),
           torch.full((4,), -7, dtype=torch.int32, device=DEV))
    pkv.make_local_attention_virtual_batches(chunk, P, cu_t, kv_t, pt_t, cap, out=out)
    torch.cuda.synchronize()
    sq, cuq, sk, bt, info = (t.cpu().numpy() for t in out)
    ref = oracle.local_virtual_batches(chunk, P, cu, kv, pt, capacity=cap, bt_cols=cols)
    assert np.array_equal(sq, ref["seqlens_q_local"])
    assert np.array_equal(cuq, ref["cu_seqlens_q_local"])
    assert np.array_equal(sk, ref["seqlens_k_local"])
    assert np.array_equal(bt, ref["block_table_local"])
    assert list(info) == [ref["num_virtual"], ref["chunk"], ref["max_q_local"],
                          ref["max_k_local"]]
    return ref


def _lvb_batch(rng, B, q_hi, kv_extra_hi, P, decode_share=0.0):
    q = rng.integers(1, q_hi + 1, B)
    q[rng.random(B) < decode_share] = 1
    kv = q + rng.integers(0, kv_extra_hi + 1, B)
    cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
    width = int(-(-kv.max() // P))
    pt = rng.integers(0, 1 << 20, (B, width)).astype(np.int32)
    return cu, kv.astype(np.int32), pt


@pytest.mark.parametrize("P", [1, 2, 4])
def test_local_virtual_batches_printed_example_on_gpu(P):
    """The printed example (chunk 4, q_seqlens [4, 10, 5], kv [6, 17, 9]) at
    its exact row count and with padding rows."""
    cu, kv = [0, 4, 14, 19], [6, 17, 9]
    pt = np.arange(3 * 17, dtype=np.int32).reshape(3, 17)[:, :-(-17 // P)] * 3 + 1
    for cap in (8, 13):
        ref = _lvb_run(4, P, cu, kv, pt, cap)
        assert list(ref["seqlens_q_local"][:8]) == [2, 2, 1, 4, 4, 1, 4, 1]
        assert list(ref["seqlens_k_local"][:8]) == [4, 2, 4, 4, 4, 1, 4, 1]
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("B,P,chunk,q_hi,kv_hi,decode_share", [
    (1, 1, 4, 10, 30, 0.0),
    (37, 16, 256, 700, 5000, 0.3),        # extend and decode mixed
    (512, 64, 8192, 1, 100000, 1.0),      # decode, long contexts
    (3000, 16, 1024, 40, 20000, 0.5),     # several scan tiles
    (16384, 16, 2048, 1, 9000, 1.0),      # largest batch
    (200, 16, 100, 300, 3000, 0.0),       # chunk not a page multiple -> 96
    (50, 64, 8192, 100, 2000, 0.0),       # chunk beyond the longest sequence
    (9, 4, 3, 30, 50, 0.0),               # chunk below a page -> one page
])
def test_local_virtual_batches_bit_exact(B, P, chunk, q_hi, kv_hi, decode_share):
    rng = np.random.default_rng(B * 7 + P + chunk)
    cu, kv, pt = _lvb_batch(rng, B, q_hi, kv_hi, P, decode_share)
    cap = pkv.local_virtual_batch_capacity(B, int(cu[-1]), int(np.diff(cu).max()), P)
    ref = _lvb_run(chunk, P, cu, kv, pt, cap)
    assert ref["num_virtual"] <= cap
    assert pkv.get_error_flags() == 0


def test_local_virtual_batches_edge_cases():
    """Empty batch; idle requests; a wider table than needed; a request
    with more new tokens than keys (flagged, key-less rows); a capacity
    below the count (flagged, rows up to the capacity)."""
    pt1 = np.zeros((0, 1), dtype=np.int32)
    _lvb_run(16, 4, [5], np.zeros(0, np.int32), pt1, 3)
    assert pkv.get_error_flags() == 0
    cu = np.array([0, 0, 9, 9, 20], dtype=np.int32)
    kv = np.array([4, 40, 0, 11], dtype=np.int32)
    pt = (np.arange(4 * 10, dtype=np.int32).reshape(4, 10) * 5) + 2
    _lvb_run(8, 4, cu, kv, pt, 12, bt_cols=5)
    assert pkv.get_error_flags() == 0
    kv_bad = kv.copy()
    kv_bad[3] = 6                                   # 11 new tokens, 6 keys
    ref = _lvb_run(8, 4, cu, kv_bad, pt, 12)
    assert ref["bad"] == 1
    assert pkv.get_error_flags() == pkv.EFLAG_BAD_LENGTHS
    pkv.clear_error_flags()
    ref = _lvb_run(4, 4, cu, kv, pt, 3)
    assert ref["num_virtual"] > 3
    assert pkv.get_error_flags() == pkv.EFLAG_CAPACITY


def _local_check(wl, chunk, num_splits=0):
    g = wl.to(DEV)
    out, lse = pkv.local_attn_with_kvcache(
        g.q, g.k_cache, g.v_cache, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
        g.max_seqlen_q, chunk, g.scale, num_splits=num_splits, return_softmax_lse=True)
    torch.cuda.synchronize()
    P = wl.k_cache.shape[1]
    eff = oracle.local_virtual_batches(chunk, P, wl.cu_seqlens_q.numpy(),
                                       wl.cache_seqlens.numpy(), wl.page_table.numpy())["chunk"]
    ref_o, ref_l, _ = oracle_attn(wl, causal=True, window_left=-1, attn_chunk=eff)
    check_close(out, lse, ref_o, ref_l, f"local chunk={chunk} (effective {eff})")
    assert pkv.get_error_flags() == 0
    return eff


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_local_attention_decode(num_splits):
    """Local attention on a GQA decode batch (32/8 heads, D 128, P 16):
    each token sees only its own 512-key chunk."""
    wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=32, h_kv=8, batch=48,
                        len_lo=1, len_hi=3000, pool_tokens=48 * 3008 + 64, seed=61)
    assert _local_check(wl, 512, num_splits) == 512


@pytest.mark.parametrize("page_size,chunk", [(64, 256), (16, 192), (64, 8192)])
def test_local_attention_extend(page_size, chunk):
    """Local attention on the varlen extend recipe, reduced (4 requests, new
    U[64, 700] on a prefix U[0, 900]): requests cut into several virtual
    requests of up to one chunk; a chunk beyond the longest sequence takes
    the longest sequence's whole pages."""
    wl = workloads.make("varlen_extend", batch=4, new_lo=64, new_hi=700, prefix_lo=0,
                        prefix_hi=900, page_size=page_size,
                        pool_pages=4 * (1600 // page_size + 2) + 8, seed=62)
    eff = _local_check(wl, chunk)
    if chunk < 1000:
        assert eff == chunk


# ------------------------------------------------------------ KV write (append)

def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("P,H,D,T,loc64,head_major", [
    (16, 8, 128, 37, False, False),
    (1, 8, 128, 4096, True, False),
    (64, 2, 64, 1, False, False),
    (16, 4, 128, 3000, True, True),
])
def test_set_kv_buffer_bit_exact(P, H, D, T, loc64, head_major):
    """New rows scattered to distinct random slots: both pools equal the
    oracle's scatter bit for bit (every other slot untouched)."""
    g = torch.Generator().manual_seed(P * 1000 + T)
    pages = T // P + 40
    shape = (pages, H, P, D) if head_major else (pages, P, H, D)
    kc = torch.randn(shape, generator=g).to(torch.bfloat16)
    vc = torch.randn(shape, generator=g).to(torch.bfloat16)
    if head_major:
        kc, vc = kc.permute(0, 2, 1, 3), vc.permute(0, 2, 1, 3)
    k = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    loc = torch.randperm(pages * P, generator=g)[:T].to(torch.int64 if loc64 else torch.int32)
    ref_k = _bits(kc.permute(0, 2, 1, 3)).transpose(0, 2, 1, 3).copy() if head_major \
        else _bits(kc).copy()
    ref_v = _bits(vc.permute(0, 2, 1, 3)).transpose(0, 2, 1, 3).copy() if head_major \
        else _bits(vc).copy()
    assert oracle.set_kv_buffer(ref_k, _bits(k), loc.numpy()) == 0
    assert oracle.set_kv_buffer(ref_v, _bits(v), loc.numpy()) == 0
    if head_major:
        kd = kc.permute(0, 2, 1, 3).contiguous().to(DEV).permute(0, 2, 1, 3)
        vd = vc.permute(0, 2, 1, 3).contiguous().to(DEV).permute(0, 2, 1, 3)
    else:
        kd, vd = kc.to(DEV), vc.to(DEV)
    pkv.set_kv_buffer(kd, vd, loc.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    got_k = _bits(kd.permute(0, 2, 1, 3)).transpose(0, 2, 1, 3) if head_major else _bits(kd)
    got_v = _bits(vd.permute(0, 2, 1, 3)).transpose(0, 2, 1, 3) if head_major else _bits(vd)
    assert np.array_equal(got_k, ref_k) and np.array_equal(got_v, ref_v)
    assert pkv.get_error_flags() == 0


def test_set_kv_buffer_out_of_pool_and_k_only():
    """Slots outside the pool are skipped and flagged; a K-only write leaves
    V alone."""
    P, H, D, pages = 16, 2, 128, 6
    kc = torch.zeros(pages, P, H, D, dtype=torch.bfloat16, device=DEV)
    k = torch.ones(4, H, D, dtype=torch.bfloat16, device=DEV)
    loc = torch.tensor([3, pages * P, -5, 95], dtype=torch.int32, device=DEV)
    pkv.set_kv_buffer(kc, None, loc, k)
    torch.cuda.synchronize()
    assert pkv.get_error_flags() == pkv.EFLAG_PAGE_OOB
    flat = kc.view(pages * P, H, D)
    assert torch.all(flat[3] == 1) and torch.all(flat[95] == 1)
    assert flat.abs().sum().item() == 2 * H * D


def test_set_mla_kv_buffer_bit_exact():
    """MLA latent rows: nope into columns 0..511, rope into 512..575 of the
    576-wide pool."""
    g = torch.Generator().manual_seed(81)
    P, pages, T = 64, 40, 300
    pool = torch.randn(pages, P, 1, 576, generator=g).to(torch.bfloat16)
    nope = torch.randn(T, 1, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(T, 1, 64, generator=g).to(torch.bfloat16)
    loc = torch.randperm(pages * P, generator=g)[:T]
    ref = _bits(pool).copy()
    assert oracle.set_kv_buffer(ref[..., :512], _bits(nope), loc.numpy()) == 0
    assert oracle.set_kv_buffer(ref[..., 512:], _bits(rope), loc.numpy()) == 0
    pd = pool.to(DEV)
    pkv.set_mla_kv_buffer(pd, loc.to(DEV), nope.to(DEV), rope.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(pd), ref)
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("kind", ["decode", "extend"])
def test_append_then_attend(kind):
    """The backend's order: the new tokens' rows are written to their slots
    (given as out_cache_loc), then attention reads them.  The pool starts
    with NaN in those slots; afterwards it equals the workload's pool bit for
    bit and the output equals the oracle's."""
    if kind == "decode":
        wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=32, h_kv=8, batch=24,
                            len_lo=1, len_hi=2000, pool_tokens=24 * 2008 + 64, seed=83)
    else:
        wl = workloads.make("varlen_extend", batch=3, new_lo=64, new_hi=500, prefix_lo=0,
                            prefix_hi=700, page_size=64, pool_pages=3 * 22 + 8, seed=84)
    P = wl.k_cache.shape[1]
    cu = wl.cu_seqlens_q.numpy()
    kv = wl.cache_seqlens.numpy()
    pt = wl.page_table.numpy()
    loc = []
    for b in range(len(kv)):
        for j in range(kv[b] - (cu[b + 1] - cu[b]), kv[b]):
            loc.append(int(pt[b, j // P]) * P + j % P)
    loc = torch.tensor(loc, dtype=torch.int64)
    kf = wl.k_cache.view(-1, *wl.k_cache.shape[2:])
    vf = wl.v_cache.view(-1, *wl.v_cache.shape[2:])
    k_new, v_new = kf[loc].clone(), vf[loc].clone()
    g = wl.to(DEV)
    kd, vd = g.k_cache.clone(), g.v_cache.clone()
    kd.view(-1, *kd.shape[2:])[loc.to(DEV)] = float("nan")
    vd.view(-1, *vd.shape[2:])[loc.to(DEV)] = float("nan")
    out, lse = pkv.append_attn_with_kvcache(
        g.q, k_new.to(DEV), v_new.to(DEV), loc.to(DEV), kd, vd, g.page_table,
        g.cache_seqlens, g.cu_seqlens_q, g.max_seqlen_q, g.scale, causal=g.causal,
        return_softmax_lse=True)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kd), _bits(wl.k_cache))
    assert np.array_equal(_bits(vd), _bits(wl.v_cache))
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, f"append+attend {kind}")
    assert pkv.get_error_flags() == 0


def _new_rows(wl):
    """Slots of every request's new positions (the last q_len of its keys)
    and those rows' K / V, taken from the workload's pool."""
    P = wl.k_cache.shape[1]
    cu, kv, pt = wl.cu_seqlens_q.numpy(), wl.cache_seqlens.numpy(), wl.page_table.numpy()
    loc = [int(pt[b, j // P]) * P + j % P
           for b in range(len(kv)) for j in range(kv[b] - (cu[b + 1] - cu[b]), kv[b])]
    loc = torch.tensor(loc, dtype=torch.int64)
    kf = wl.k_cache.view(-1, *wl.k_cache.shape[2:])
    vf = wl.v_cache.view(-1, *wl.v_cache.shape[2:])
    return loc, kf[loc].clone(), vf[loc].clone()


@pytest.mark.parametrize("page_size,q_len,num_splits,window",
                         [(16, 1, 0, -1), (16, 1, 4, -1), (16, 4, 0, -1), (16, 3, 2, 300),
                          (1, 1, 0, -1), (1, 1, 3, -1), (1, 4, 0, 200), (64, 2, 5, -1)])
def test_fused_append_attend(page_size, q_len, num_splits, window):
    """The KV write and the attention in one launch (slot rows and page
    boxes, the balanced schedule and fixed splits, runs of new tokens that
    straddle key tiles, windows): the pool starts with NaN in the new slots;
    afterwards it equals the workload's pool bit for bit, the output equals
    the oracle's, and it is bit-identical to the unfused write-then-attend
    pair in the same launch configuration."""
    h_q, h_kv = 8 * (4 // q_len if q_len <= 4 else 1), 8
    wl = workloads.make("tiny_decode", d=128, page_size=page_size, h_q=h_q, h_kv=h_kv, batch=19,
                        q_len=q_len, causal=True, window_left=window, len_lo=q_len,
                        len_hi=1500, pool_tokens=19 * (1500 + page_size) + 64,
                        seed=90 + page_size + q_len)
    loc, k_new, v_new = _new_rows(wl)
    g = wl.to(DEV)
    outs = []
    for fused in (True, False):
        kd, vd = g.k_cache.clone(), g.v_cache.clone()
        kd.view(-1, *kd.shape[2:])[loc.to(DEV)] = float("nan")
        vd.view(-1, *vd.shape[2:])[loc.to(DEV)] = float("nan")
        fn = pkv.fused_append_attn_with_kvcache if fused else pkv.append_attn_with_kvcache
        out, lse = fn(g.q, k_new.to(DEV), v_new.to(DEV), loc.to(DEV), kd, vd, g.page_table,
                      g.cache_seqlens, g.cu_seqlens_q, g.max_seqlen_q, g.scale, causal=True,
                      window_left=window, num_splits=num_splits, return_softmax_lse=True)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(kd), _bits(wl.k_cache))
        assert np.array_equal(_bits(vd), _bits(wl.v_cache))
        outs.append((out, lse))
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(outs[0][0], outs[0][1], ref_o, ref_l, "fused append+attend")
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    assert pkv.get_error_flags() == 0


def test_fused_append_attend_bad_slot_and_unsupported():
    """A slot outside the pool is skipped and flagged (the attention still
    uses the new row); fp8 caches and shapes off the all-heads kernel are
    refused without a launch."""
    wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=32, h_kv=8, batch=5,
                        len_lo=20, len_hi=300, pool_tokens=5 * 320 + 64, seed=97)
    loc, k_new, v_new = _new_rows(wl)
    bad = loc.clone()
    bad[2] = wl.k_cache.shape[0] * 16 + 5
    g = wl.to(DEV)
    kd, vd = g.k_cache.clone(), g.v_cache.clone()
    out, lse = pkv.fused_append_attn_with_kvcache(
        g.q, k_new.to(DEV), v_new.to(DEV), bad.to(DEV), kd, vd, g.page_table, g.cache_seqlens,
        g.cu_seqlens_q, g.max_seqlen_q, g.scale, return_softmax_lse=True)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, "fused append, bad slot")
    assert pkv.get_error_flags() & pkv.EFLAG_PAGE_OOB
    pkv.clear_error_flags()
    k8, v8 = g.k_cache.to(torch.float8_e4m3fn), g.v_cache.to(torch.float8_e4m3fn)
    with pytest.raises(pkv.PkvError, match="UNSUPPORTED"):
        pkv.fused_append_attn_with_kvcache(
            g.q, k_new.to(DEV), v_new.to(DEV), loc.to(DEV), k8, v8, g.page_table,
            g.cache_seqlens, g.cu_seqlens_q, g.max_seqlen_q, g.scale)
    wl64 = workloads.make("tiny_decode", d=64, page_size=16, h_q=8, h_kv=2, batch=3,
                          len_lo=20, len_hi=100, pool_tokens=3 * 120 + 64, seed=98)
    loc64, kn64, vn64 = _new_rows(wl64)
    g64 = wl64.to(DEV)
    with pytest.raises(pkv.PkvError, match="UNSUPPORTED"):
        pkv.fused_append_attn_with_kvcache(
            g64.q, kn64.to(DEV), vn64.to(DEV), loc64.to(DEV), g64.k_cache, g64.v_cache,
            g64.page_table, g64.cache_seqlens, g64.cu_seqlens_q, g64.max_seqlen_q, g64.scale)


def test_fused_append_attend_full_size():
    """The GQA decode batch (64 requests, 32/8 heads, kv U[512, 8192], page
    16) with each request's last key as its new token, in the bench's launch
    configuration (4 key chunks): pool bit for bit, every output row against
    the oracle."""
    wl = workloads.make("gqa_split_decode", value_device=DEV)
    loc, k_new, v_new = _new_rows_device(wl)
    kd, vd = wl.k_cache.clone(), wl.v_cache.clone()
    kd.view(-1, *kd.shape[2:])[loc] = float("nan")
    vd.view(-1, *vd.shape[2:])[loc] = float("nan")
    out, lse = pkv.fused_append_attn_with_kvcache(
        wl.q, k_new, v_new, loc, kd, vd, wl.page_table, wl.cache_seqlens, wl.cu_seqlens_q,
        wl.max_seqlen_q, wl.scale, num_splits=4, return_softmax_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(kd.view(torch.int16), wl.k_cache.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), wl.v_cache.view(torch.int16))
    ref_o, ref_l, _ = oracle.attention(
        oracle.bf16_bits(wl.q), oracle.bf16_bits(wl.k_cache), oracle.bf16_bits(wl.v_cache),
        wl.page_table.cpu().numpy(), wl.cache_seqlens.cpu().numpy(),
        wl.cu_seqlens_q.cpu().numpy(), wl.scale)
    check_close(out, lse, ref_o, ref_l, "fused append full size")
    assert pkv.get_error_flags() == 0


def _new_rows_device(wl):
    P = wl.k_cache.shape[1]
    cu, kv = wl.cu_seqlens_q.cpu().numpy(), wl.cache_seqlens.cpu().numpy()
    pt = wl.page_table.cpu().numpy()
    loc = [int(pt[b, j // P]) * P + j % P
           for b in range(len(kv)) for j in range(kv[b] - (cu[b + 1] - cu[b]), kv[b])]
    loc = torch.tensor(loc, dtype=torch.int64, device=wl.k_cache.device)
    kf = wl.k_cache.view(-1, *wl.k_cache.shape[2:])
    vf = wl.v_cache.view(-1, *wl.v_cache.shape[2:])
    return loc, kf[loc].clone(), vf[loc].clone()


# ------------------------------------------------------------------ FP8 KV

def _to_fp8(t):
    return t.float().to(torch.float8_e4m3fn)


def _fp8_run(wl, descale=True, seed=0, entry="fp8", scale=None):
    """GPU fp8 attention and the oracle's, on the workload's cache cast to
    e4m3 codes; per-(request, KV head) descales drawn in [0.5, 2)."""
    scale = wl.scale if scale is None else scale
    B, h_kv = wl.cache_seqlens.shape[0], wl.k_cache.shape[2]
    k8, v8 = _to_fp8(wl.k_cache), _to_fp8(wl.v_cache)
    gen = torch.Generator().manual_seed(seed)
    kd = (torch.rand(B, h_kv, generator=gen) * 1.5 + 0.5) if descale else None
    vd = (torch.rand(B, h_kv, generator=gen) * 1.5 + 0.5) if descale else None
    g = wl.to(DEV)
    if entry == "fp8":
        out, lse = pkv.attn_with_kvcache_fp8(
            g.q, k8.to(DEV), v8.to(DEV), g.page_table, g.cache_seqlens, g.cu_seqlens_q,
            g.max_seqlen_q, scale, causal=g.causal, window_left=g.window_left,
            k_descale=None if kd is None else kd.to(DEV),
            v_descale=None if vd is None else vd.to(DEV), return_softmax_lse=True)
    else:  # the bf16 entry point with an fp8 cache: descales of 1
        out, lse = pkv.attn_with_kvcache(
            g.q, k8.to(DEV), v8.to(DEV), g.page_table, g.cache_seqlens, g.cu_seqlens_q,
            g.max_seqlen_q, scale, causal=g.causal, window_left=g.window_left,
            return_softmax_lse=True)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle.attention_fp8(
        oracle.bf16_bits(wl.q), k8.view(torch.uint8).numpy(), v8.view(torch.uint8).numpy(),
        wl.page_table.numpy(), wl.cache_seqlens.numpy(), wl.cu_seqlens_q.numpy(), scale,
        causal=wl.causal, window_left=wl.window_left,
        k_descale=None if kd is None else kd.numpy(),
        v_descale=None if vd is None else vd.numpy())
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("page_size,h_q,q_len", [(16, 32, 1), (64, 32, 2), (16, 64, 2),
                                                 (1, 32, 1), (2, 16, 2)])
def test_fp8_decode(page_size, h_q, q_len):
    """FP8 cache (e4m3 codes), per-(request, KV head) descales, q cast to
    e4m3 in the kernel: GQA decode shapes, 8 KV heads, head dim 128, up to 16
    query rows per KV head, ragged lengths (the balanced schedule splits the
    long requests over CTAs); page boxes and slot rows (page sizes 1, 2)."""
    wl = workloads.make("tiny_decode", d=128, page_size=page_size, h_q=h_q, h_kv=8,
                        q_len=q_len, causal=q_len > 1, batch=24, len_lo=q_len,
                        len_hi=3000, pool_tokens=24 * 3072 + 256, seed=101 + page_size)
    out, lse, ref_o, ref_l = _fp8_run(wl, seed=page_size)
    check_close(out, lse, ref_o, ref_l, f"fp8 P={page_size} h_q={h_q} q_len={q_len}")
    assert pkv.get_error_flags() == 0


@pytest.mark.parametrize("page_size,window,causal,entry", [
    (64, -1, True, "fp8"), (16, -1, True, "fp8"), (128, 300, True, "fp8"),
    (64, -1, False, "fp8"), (32, -1, True, "bf16")])
def test_fp8_extend(page_size, window, causal, entry):
    """Varlen extend over an fp8 cache on the tcgen05 kernel: q rounded to
    e4m3, QK^T on e4m3 tensor-core MMAs, V widened to f16 for PV, descales
    per (request, KV head) (or 1 through the bf16 entry point); NaN in every
    unused slot of the pool."""
    wl = workloads.make("varlen_extend", batch=4, new_lo=64, new_hi=700, prefix_lo=0,
                        prefix_hi=900, page_size=page_size,
                        pool_pages=4 * (1600 // page_size + 2) + 8, window_left=window,
                        seed=1203 + page_size)
    wl.causal = causal
    valid = torch.zeros(wl.k_cache.shape[0] * page_size, dtype=torch.bool)
    for b in range(4):
        j = torch.arange(int(wl.cache_seqlens[b]))
        valid[wl.page_table[b, j // page_size].long() * page_size + j % page_size] = True
    valid = valid.view(-1, page_size)
    wl.k_cache[~valid] = float("nan")
    wl.v_cache[~valid] = float("nan")
    out, lse, ref_o, ref_l = _fp8_run(wl, descale=entry == "fp8", seed=page_size, entry=entry)
    check_close(out, lse, ref_o, ref_l, f"fp8 extend P={page_size} w={window} c={causal}")
    assert pkv.get_error_flags() == 0


def test_fp8_extend_negative_scale_and_bad_page():
    """The fp8 extend kernel with a negative softmax scale (its row maxima
    are taken on sign-flipped scores) and an out-of-pool page id (those keys
    skipped and flagged, as the oracle skips them)."""
    wl = workloads.make("varlen_extend", batch=3, new_lo=100, new_hi=400, prefix_lo=50,
                        prefix_hi=600, page_size=64, pool_pages=3 * 17 + 10, seed=1301)
    wl.page_table[1, 2] = 10_000_000
    wl.cache_seqlens[1] = max(int(wl.cache_seqlens[1]), 3 * 64 + 1)
    wl.cache_seqlens[1] = min(int(wl.cache_seqlens[1]), wl.page_table.shape[1] * 64)
    out, lse, ref_o, ref_l = _fp8_run(wl, seed=9, scale=-0.08)
    check_close(out, lse, ref_o, ref_l, "fp8 extend negative scale")
    assert pkv.get_error_flags() == pkv.EFLAG_PAGE_OOB


def test_fp8_unit_descale_entry_and_edges():
    """The bf16 entry point with an fp8 cache (descales of 1); a request with
    no keys (0 / -inf); a page id outside the pool (its keys skipped, V rows
    zeroed, the flag set)."""
    wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=16, h_kv=4, batch=12,
                        len_lo=0, len_hi=900, pool_tokens=12 * 912 + 64, seed=111)
    wl.cache_seqlens[3] = 0
    out, lse, ref_o, ref_l = _fp8_run(wl, descale=False, entry="bf16")
    check_close(out, lse, ref_o, ref_l, "fp8 unit descales")
    assert pkv.get_error_flags() == 0
    n_pages = wl.k_cache.shape[0]
    wl.page_table[5, 1] = n_pages + 7  # the second page of request 5 is bad
    wl.cache_seqlens[5] = max(int(wl.cache_seqlens[5]), 40)
    out, lse, ref_o, ref_l = _fp8_run(wl, seed=3)
    check_close(out, lse, ref_o, ref_l, "fp8 bad page")
    assert pkv.get_error_flags() & pkv.EFLAG_PAGE_OOB


def test_fp8_unsupported_shapes_are_refused():
    """Decode shapes outside the fp8 path return PKV_ERR_UNSUPPORTED: page
    size 8, fixed splits (runs of >= 64 new tokens go to the extend kernel,
    test_fp8_extend)."""
    wl = workloads.make("tiny_decode", d=128, page_size=8, h_q=8, h_kv=2, batch=2,
                        len_lo=10, len_hi=50, pool_tokens=256, seed=112)
    g = wl.to(DEV)
    k8, v8 = _to_fp8(g.k_cache), _to_fp8(g.v_cache)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_with_kvcache_fp8(g.q, k8, v8, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                  g.max_seqlen_q, g.scale)
    assert e.value.code == -2
    wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=8, h_kv=2, batch=2,
                        len_lo=10, len_hi=50, pool_tokens=512, seed=113)
    g = wl.to(DEV)
    k8, v8 = _to_fp8(g.k_cache), _to_fp8(g.v_cache)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_with_kvcache(g.q, k8, v8, g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                              g.max_seqlen_q, g.scale, num_splits=2)
    assert e.value.code == -2


# ------------------------------------------------------- CUDA graph capture

def test_paths_replay_from_cuda_graphs_with_new_lengths():
    """Decode and local attention (device-built virtual requests) need no
    host work inside a call: both are captured once into a CUDA graph, the
    request lengths are changed in place, and the replay's results equal the
    oracle's for the new lengths."""
    wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=32, h_kv=8, batch=8,
                        len_lo=64, len_hi=1500, pool_tokens=8 * 1536 + 64, seed=121)
    g = wl.to(DEV)
    P = 16
    cap = pkv.local_virtual_batch_capacity(8, g.q.shape[0], 1, P)
    out_d = torch.empty(g.q.shape[0], 32, 128, dtype=torch.bfloat16, device=DEV)
    lse_d = torch.empty(g.q.shape[0], 32, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(1, pkv.attn_workspace_size(g.q, g.k_cache, g.v_cache, g.page_table,
                                                    g.cache_seqlens, 1)),
                     dtype=torch.uint8, device=DEV)
    out_l = torch.empty_like(out_d)
    lse_l = torch.empty_like(lse_d)
    bufs = (torch.empty(cap, dtype=torch.int32, device=DEV),
            torch.empty(cap + 1, dtype=torch.int32, device=DEV),
            torch.empty(cap, dtype=torch.int32, device=DEV),
            torch.empty(cap, 512 // P, dtype=torch.int32, device=DEV),
            torch.empty(4, dtype=torch.int32, device=DEV))
    ws_l = torch.empty(max(1, pkv.attn_workspace_size(g.q, g.k_cache, g.v_cache, bufs[3],
                                                      bufs[2], 1)),
                       dtype=torch.uint8, device=DEV)

    def run():
        pkv.attn_with_kvcache(g.q, g.k_cache, g.v_cache, g.page_table, g.cache_seqlens,
                              g.cu_seqlens_q, 1, g.scale, out=out_d, lse=lse_d, workspace=ws)
        pkv.make_local_attention_virtual_batches(512, P, g.cu_seqlens_q, g.cache_seqlens,
                                                 g.page_table, cap, out=bufs)
        pkv.attn_with_kvcache(g.q, g.k_cache, g.v_cache, bufs[3], bufs[2], bufs[1], 1, g.scale,
                              causal=True, out=out_l, lse=lse_l, workspace=ws_l)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    own = wl.cache_seqlens.clone()  # lengths stay within each request's pages
    for trial in range(2):
        frac = torch.rand(8, generator=torch.Generator().manual_seed(trial))
        new_len = (1 + (frac * own.float()).long()).clamp(max=own.long())
        wl.cache_seqlens.copy_(new_len.to(torch.int32))
        g.cache_seqlens.copy_(wl.cache_seqlens.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        ref_o, ref_l, _ = oracle_attn(wl, causal=False)
        check_close(out_d, lse_d, ref_o, ref_l, f"graph decode {trial}")
        eff = oracle.local_virtual_batches(512, P, wl.cu_seqlens_q.numpy(),
                                           wl.cache_seqlens.numpy(),
                                           wl.page_table.numpy())["chunk"]
        ref_o, ref_l, _ = oracle_attn(wl, causal=True, attn_chunk=eff)
        check_close(out_l, lse_l, ref_o, ref_l, f"graph local {trial}")
    assert pkv.get_error_flags() == 0


# ------------------------------------ full-size checks of the composed rows

def test_fp8_full_size():
    """The bench's fp8 line: the GQA decode batch (64 requests, 32/8 heads,
    kv U[512, 8192]) with its cache cast to e4m3 and descales 0.75 / 1.25,
    the library's split choice; every request (all rows) against the
    oracle."""
    g = workloads.make("gqa_split_decode", value_device=DEV)
    k8, v8 = g.k_cache.to(torch.float8_e4m3fn), g.v_cache.to(torch.float8_e4m3fn)
    B, h_kv = g.cache_seqlens.shape[0], k8.shape[2]
    kd = torch.full((B, h_kv), 0.75, device=DEV)
    vd = torch.full((B, h_kv), 1.25, device=DEV)
    out, lse = pkv.attn_with_kvcache_fp8(g.q, k8, v8, g.page_table, g.cache_seqlens,
                                         g.cu_seqlens_q, g.max_seqlen_q, g.scale,
                                         k_descale=kd, v_descale=vd, return_softmax_lse=True)
    torch.cuda.synchronize()
    pick = np.arange(B)                                  # decode: token b is request b
    pt = g.page_table.cpu().numpy()[pick]
    ks = g.cache_seqlens.cpu().numpy()[pick]
    ref_o, ref_l, _ = oracle.attention_fp8(
        oracle.bf16_bits(g.q[torch.from_numpy(pick).to(DEV)]), k8.view(torch.uint8).cpu().numpy(),
        v8.view(torch.uint8).cpu().numpy(), pt, ks, np.arange(len(pick) + 1, dtype=np.int32),
        g.scale, k_descale=kd.cpu().numpy()[pick], v_descale=vd.cpu().numpy()[pick])
    idx = torch.from_numpy(pick).long()
    check_close(out.cpu()[idx], lse.cpu()[idx], ref_o, ref_l, "fp8 full-size")
    assert pkv.get_error_flags() == 0


def test_local_attention_full_size():
    """The bench's local-attention line: the GQA decode batch with 2048-key
    chunks (device-built virtual requests, one attention call); every row
    against the oracle's chunk-masked attention."""
    g = workloads.make("gqa_split_decode", value_device=DEV)
    out, lse = pkv.local_attn_with_kvcache(g.q, g.k_cache, g.v_cache, g.page_table,
                                           g.cache_seqlens, g.cu_seqlens_q, g.max_seqlen_q,
                                           2048, g.scale, return_softmax_lse=True)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle.attention(
        oracle.bf16_bits(g.q), oracle.bf16_bits(g.k_cache), oracle.bf16_bits(g.v_cache),
        g.page_table.cpu().numpy(), g.cache_seqlens.cpu().numpy(),
        g.cu_seqlens_q.cpu().numpy(), g.scale, causal=True, attn_chunk=2048)
    check_close(out, lse, ref_o, ref_l, "local full size")
    assert pkv.get_error_flags() == 0


def test_cascade_full_size():
    """The bench's cascade line: every request of the GQA decode batch also
    sees a shared 4096-token prefix (pages 0-255 of the pool); every row
    against one oracle call over the prefix pages followed by the request's
    own pages."""
    g = workloads.make("gqa_split_decode", value_device=DEV)
    B = g.cache_seqlens.shape[0]
    pre_pt = torch.arange(256, dtype=torch.int32, device=DEV).repeat(B, 1).contiguous()
    pre_len = torch.full((B,), 4096, dtype=torch.int32, device=DEV)
    out, lse = pkv.cascade_attn_with_kvcache(g.q, g.k_cache, g.v_cache, pre_pt, pre_len,
                                             g.page_table, g.cache_seqlens, g.cu_seqlens_q,
                                             g.max_seqlen_q, g.scale, causal=True,
                                             return_softmax_lse=True)
    torch.cuda.synchronize()
    full_pt = torch.cat([pre_pt.cpu(), g.page_table.cpu()], dim=1).numpy()
    full_len = (g.cache_seqlens.cpu() + 4096).numpy()
    ref_o, ref_l, _ = oracle.attention(
        oracle.bf16_bits(g.q), oracle.bf16_bits(g.k_cache), oracle.bf16_bits(g.v_cache),
        full_pt, full_len, g.cu_seqlens_q.cpu().numpy(), g.scale, causal=True)
    check_close(out, lse, ref_o, ref_l, "cascade full size")
    assert pkv.get_error_flags() == 0


def test_set_kv_buffer_full_size_bit_exact():
    """The bench's KV-write line: the varlen extend workload's new rows
    (10k tokens, 8 heads x 128) stored to their slots; both pools equal the
    oracle's scatter bit for bit."""
    g = workloads.make("varlen_extend", value_device=DEV)
    P = g.page_size
    cu = g.cu_seqlens_q.cpu().numpy()
    kv = g.cache_seqlens.cpu().numpy()
    pt = g.page_table.cpu().numpy()
    loc = np.concatenate([pt[b, np.arange(kv[b] - (cu[b + 1] - cu[b]), kv[b]) // P] * P +
                          np.arange(kv[b] - (cu[b + 1] - cu[b]), kv[b]) % P
                          for b in range(len(kv))]).astype(np.int64)
    gen = torch.Generator(device=DEV).manual_seed(5)
    k_new = torch.randn(len(loc), 8, 128, device=DEV, generator=gen).to(torch.bfloat16)
    v_new = torch.randn(len(loc), 8, 128, device=DEV, generator=gen).to(torch.bfloat16)
    ref_k = _bits(g.k_cache).copy()
    ref_v = _bits(g.v_cache).copy()
    assert oracle.set_kv_buffer(ref_k, _bits(k_new), loc) == 0
    assert oracle.set_kv_buffer(ref_v, _bits(v_new), loc) == 0
    pkv.set_kv_buffer(g.k_cache, g.v_cache, torch.from_numpy(loc).to(DEV), k_new, v_new)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(g.k_cache), ref_k)
    assert np.array_equal(_bits(g.v_cache), ref_v)
    assert pkv.get_error_flags() == 0


# ----------------------------------------------- KV write into an fp8 pool

def _scale_t(s):
    return None if s is None else torch.tensor([s], dtype=torch.float32, device=DEV)


@pytest.mark.parametrize("P,H,D,T,scales", [
    (16, 8, 128, 300, (0.02, 0.7)),
    (64, 2, 64, 37, (None, 0.05)),
    (1, 8, 128, 2000, (0.3, None)),
])
def test_set_kv_buffer_fp8_bit_exact(P, H, D, T, scales):
    """Quantising write into pools of e4m3 codes: every stored code equals
    the oracle's (binary32 quotient value / scale, nearest code, ties to
    even) and every other byte keeps its prior contents; an out-of-pool slot
    is skipped and flagged.  Quotients stay inside the format's range."""
    g = torch.Generator().manual_seed(P * 7 + T)
    pages = T // P + 40
    prior_k = torch.randint(0, 0x7e, (pages, P, H, D), generator=g, dtype=torch.uint8)
    prior_v = torch.randint(0, 0x7e, (pages, P, H, D), generator=g, dtype=torch.uint8)
    k = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    loc = torch.randperm(pages * P, generator=g)[:T].to(torch.int64)
    loc[T // 2] = pages * P                          # outside the pool
    ks, vs = scales
    ref_k, ref_v = prior_k.numpy().copy(), prior_v.numpy().copy()
    assert oracle.set_kv_buffer_fp8(ref_k, _bits(k), loc.numpy(), 1.0 if ks is None else ks) == 1
    assert oracle.set_kv_buffer_fp8(ref_v, _bits(v), loc.numpy(), 1.0 if vs is None else vs) == 1
    k8 = prior_k.to(DEV).view(torch.float8_e4m3fn)
    v8 = prior_v.to(DEV).view(torch.float8_e4m3fn)
    pkv.set_kv_buffer(k8, v8, loc.to(DEV), k.to(DEV), v.to(DEV),
                      k_scale=_scale_t(ks), v_scale=_scale_t(vs))
    torch.cuda.synchronize()
    assert np.array_equal(k8.view(torch.uint8).cpu().numpy(), ref_k)
    assert np.array_equal(v8.view(torch.uint8).cpu().numpy(), ref_v)
    assert pkv.get_error_flags() == pkv.EFLAG_PAGE_OOB


def test_fp8_write_then_attend():
    """A decode step over an fp8 pool as the backend runs it: the new
    token's K/V stored as codes of value / scale, then attention with the
    scales as per-(request, KV head) descales; against the oracle's write
    followed by the oracle's fp8 attention."""
    wl = workloads.make("tiny_decode", d=128, page_size=16, h_q=32, h_kv=8, batch=12,
                        len_lo=20, len_hi=900, pool_tokens=12 * 928 * 2, seed=78)
    ks, vs = 0.03, 0.05
    k_scale, v_scale = _scale_t(ks), _scale_t(vs)
    # the cached keys as codes, then each request's newest token rewritten
    k_codes = (wl.k_cache.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
    v_codes = (wl.v_cache.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
    P = wl.page_size
    kv = wl.cache_seqlens.numpy()
    loc = np.array([wl.page_table[b, (kv[b] - 1) // P].item() * P + (kv[b] - 1) % P
                    for b in range(len(kv))], dtype=np.int64)
    gen = torch.Generator().manual_seed(5)
    k_new = torch.randn(len(kv), 8, 128, generator=gen).to(torch.bfloat16)
    v_new = torch.randn(len(kv), 8, 128, generator=gen).to(torch.bfloat16)
    ref_k, ref_v = k_codes.numpy().copy(), v_codes.numpy().copy()
    assert oracle.set_kv_buffer_fp8(ref_k, _bits(k_new), loc, ks) == 0
    assert oracle.set_kv_buffer_fp8(ref_v, _bits(v_new), loc, vs) == 0
    g = wl.to(DEV)
    k8 = k_codes.to(DEV).view(torch.float8_e4m3fn)
    v8 = v_codes.to(DEV).view(torch.float8_e4m3fn)
    out, lse = pkv.append_attn_with_kvcache(
        g.q, k_new.to(DEV), v_new.to(DEV), torch.from_numpy(loc).to(DEV), k8, v8,
        g.page_table, g.cache_seqlens, g.cu_seqlens_q, g.max_seqlen_q, g.scale,
        k_scale=k_scale, v_scale=v_scale, return_softmax_lse=True)
    torch.cuda.synchronize()
    assert np.array_equal(k8.view(torch.uint8).cpu().numpy(), ref_k)
    assert np.array_equal(v8.view(torch.uint8).cpu().numpy(), ref_v)
    B, h_kv = len(kv), 8
    ref_o, ref_l, _ = oracle.attention_fp8(
        oracle.bf16_bits(wl.q), ref_k, ref_v, wl.page_table.numpy(), kv,
        wl.cu_seqlens_q.numpy(), wl.scale,
        k_descale=np.full((B, h_kv), ks, np.float32), v_descale=np.full((B, h_kv), vs, np.float32))
    check_close(out, lse, ref_o, ref_l, "fp8 write then attend")
    assert pkv.get_error_flags() == 0


# ------------------------------------------------ bounded in-kernel waits

def test_bounded_wait_expires_and_the_context_stays_usable():
    """The expiry path of the library's bounded waits, exercised without a
    fault: a CTA waits on a barrier that nothing arrives on, both wait
    flavours give up after their bound (about a second), PKV_EFLAG_TIMEOUT
    is set, the kernel ends, and the next attention call on the same
    context is correct and raises no flag."""
    import time
    pkv.clear_error_flags()
    t0 = time.perf_counter()
    pkv.check_bounded_wait()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert pkv.get_error_flags() == pkv.EFLAG_TIMEOUT
    assert 0.2 < waited < 30.0, waited
    pkv.clear_error_flags()
    wl = workloads.make("tiny_decode", batch=3, len_lo=5, len_hi=120)
    g = wl.to(DEV)
    out, lse = gpu_attn(g, num_splits=1)
    ref_o, ref_l, _ = oracle_attn(wl)
    check_close(out, lse, ref_o, ref_l, "after an expired wait")
    assert pkv.get_error_flags() == 0
