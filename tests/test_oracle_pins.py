"""Pins for the float64 oracle: checks against facts that the pages and the
mathematics fix, independent of the oracle's own code.

Each test names what it pins.  A plausible slip anywhere in the oracle (a
dropped term, a wrong sign or index, a transposed operand, an off-by-one mask
or window, a wrong page/slot map, a wrong merge weight) fails at least one.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from conftest import read_golden
from paged_kv_cache_203_gb300 import workloads


def bf16(a):
    """float array -> (bf16 bit patterns, exact float64 values)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return oracle.bf16_bits(t), t.to(torch.float64).numpy()


def paged_from_logical(rng, kv_logical, page_size, extra_pages=3):
    """Scatter per-request logical rows [L_b, H_kv, D] into a shuffled page
    pool.  Returns (cache [pages, P, H_kv, D] float, page_table int32)."""
    h_kv, d = kv_logical[0].shape[1:]
    n_pages_req = [max(1, -(-len(x) // page_size)) for x in kv_logical]
    num_pages = sum(n_pages_req) + extra_pages
    perm = rng.permutation(num_pages)
    cache = rng.standard_normal((num_pages, page_size, h_kv, d))  # junk fill
    pt = np.full((len(kv_logical), max(n_pages_req)), 0, dtype=np.int32)
    off = 0
    for b, x in enumerate(kv_logical):
        for c in range(n_pages_req[b]):
            page = perm[off]
            off += 1
            pt[b, c] = page
            rows = x[c * page_size:(c + 1) * page_size]
            cache[page, : len(rows)] = rows
    return cache, pt


def dense_reference_row(q, K, V, scale):
    """Attention of one query over explicit key/value rows via scipy's
    softmax / logsumexp (a library routine)."""
    s = scale * (K @ q)
    return scipy.special.softmax(s) @ V, scipy.special.logsumexp(s)


# ----------------------------------------------------------------- page tables

def test_strided_page_table_recovers_allocated_pages():
    """a1 closed form: when request b owns pages pt[b, c] and req_to_token
    holds slot pt[b, j//P]*P + j%P, the strided table is pt itself."""
    for p in (1, 16, 64):
        wl = workloads.make("varlen_extend", batch=5, new_lo=3, new_hi=70,
                            prefix_hi=200, page_size=p, pool_pages=4096 // p + 64,
                            h_q=2, h_kv=1, d=8)
        n_cols = wl.page_table.shape[1]
        got = oracle.strided_page_table(wl.req_to_token.numpy(),
                                        wl.req_pool_indices.numpy(), p, n_cols)
        assert np.array_equal(got, wl.page_table.numpy())


def test_strided_page_table_hand_example():
    """a1 on a hand-built row: slots 40..47 then 8..15 with P=8 are pages 5, 1;
    floor division of the first slot of each page."""
    rtt = np.array([[40, 41, 42, 43, 44, 45, 46, 47, 8, 9, 10, 11, 12, 13, 14, 15]],
                   dtype=np.int32)
    got = oracle.strided_page_table(rtt, np.array([0]), 8, 2)
    assert got.tolist() == [[5, 1]]


@pytest.mark.parametrize("row", read_golden("swa_rows.txt"))
def test_swa_rows_hand_worked(row):
    """a2: hand-worked rows of the prefill-aware SWA rule (golden fixture)."""
    (pf, sl, w), (kv_len,), kept = row
    rtt = (np.arange(64, dtype=np.int32) * 7 + 3)[None, :]  # distinct slots
    dst, kv, bad = oracle.swa_page_table(rtt, np.array([0]), np.array([sl]),
                                         np.array([pf]), w, 32, fill=-5)
    assert bad == 0
    assert kv.tolist() == [kv_len]
    assert dst[0, :kv_len].tolist() == [int(rtt[0, i]) for i in kept]
    assert np.all(dst[0, kv_len:] == -5)  # the tail is left untouched


def test_swa_rows_match_set_membership():
    """a2 against the set definition: position i of the sequence is kept iff
    it is part of the prompt (i < pf) or among the last `window` tokens
    (i >= sl - window); kept positions stay in order."""
    rng = np.random.default_rng(7)
    pool = 9
    rtt = rng.permutation(pool * 300).astype(np.int32).reshape(pool, 300)
    for _ in range(40):
        b = 6
        rpi = rng.permutation(pool)[:b]
        pf_pool = rng.integers(0, 120, pool).astype(np.int32)
        sl = rng.integers(1, 300, b).astype(np.int32)
        w = int(rng.integers(0, 150))
        dst, kv, bad = oracle.swa_page_table(rtt, rpi, sl, pf_pool, w, 300)
        assert bad == 0
        for r in range(b):
            pf = pf_pool[rpi[r]]
            kept = [i for i in range(sl[r]) if i < pf or i >= sl[r] - w]
            assert kv[r] == len(kept)
            assert dst[r, : kv[r]].tolist() == [int(rtt[rpi[r], i]) for i in kept]


def test_swa_row_too_long_is_reported():
    rtt = np.arange(40, dtype=np.int32)[None, :]
    dst, kv, bad = oracle.swa_page_table(rtt, np.array([0]), np.array([30]),
                                         np.array([10]), 8, 12)
    assert bad == 1 and kv.tolist() == [-1]


def test_topk_to_slots_matches_token_level_table():
    """a3: the page-level map pt[b, idx//P]*P + idx%P equals the token-level
    lookup req_to_token[req_b, idx] (the page_size-1 table of the NSA path),
    -1 stays -1, out-of-range entries become -1 and are counted."""
    for p in (1, 16, 64):
        wl = workloads.make("varlen_extend", batch=4, new_lo=1, new_hi=40,
                            prefix_hi=300, page_size=p,
                            pool_pages=2048 // p + 40, h_q=1, h_kv=1, d=8)
        rng = np.random.default_rng(p)
        kv = wl.cache_seqlens.numpy()
        rows, row_req = [], []
        for b in range(4):
            for _ in range(3):
                idx = rng.integers(0, kv[b], 10)
                idx[rng.random(10) < 0.2] = -1
                rows.append(idx)
                row_req.append(b)
        topk = np.array(rows, dtype=np.int32)
        topk[0, 0] = kv[0]          # one past the end -> counted, -1
        topk[1, 1] = -7             # below -1 -> counted, -1
        slots, bad = oracle.topk_to_slots(topk, row_req, wl.page_table.numpy(),
                                          p, kv)
        assert bad == 2
        rtt = wl.req_to_token.numpy()
        rpi = wl.req_pool_indices.numpy()
        for r, b in enumerate(row_req):
            for k, idx in enumerate(topk[r]):
                want = -1 if (idx < 0 or idx >= kv[b]) else rtt[rpi[b], idx]
                assert slots[r, k] == want


# -------------------------------------------------------------------- attention

def _tiny_case(rng, batch, q_lens, kv_lens, h_q, h_kv, d, page_size, d_v=None):
    d_v = d if d_v is None else d_v
    kl = [rng.standard_normal((n, h_kv, d)) for n in kv_lens]
    vl = [rng.standard_normal((n, h_kv, d_v)) for n in kv_lens]
    kc, pt = paged_from_logical(np.random.default_rng(11), kl, page_size)
    vc, pt2 = paged_from_logical(np.random.default_rng(11), vl, page_size)
    assert np.array_equal(pt, pt2)
    total_q = sum(q_lens)
    q = rng.standard_normal((total_q, h_q, d))
    qb, qf = bf16(q)
    kb, kf = bf16(kc)
    vb, vf = bf16(vc)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    # exact (bf16-rounded) logical rows, for the reference computations
    klog = [np.stack([kf[pt[b, j // page_size], j % page_size] for j in range(n)])
            if n else np.zeros((0, h_kv, d)) for b, n in enumerate(kv_lens)]
    vlog = [np.stack([vf[pt[b, j // page_size], j % page_size] for j in range(n)])
            if n else np.zeros((0, h_kv, d_v)) for b, n in enumerate(kv_lens)]
    return dict(qb=qb, qf=qf, kb=kb, vb=vb, pt=pt, cu=cu,
                kv=np.array(kv_lens, dtype=np.int32), klog=klog, vlog=vlog)


@pytest.mark.parametrize("page_size", [1, 3, 16])
def test_attention_matches_scipy_softmax(page_size):
    """Dense paged attention equals softmax(scale K q) V computed by scipy on
    the logical (unpaged) rows, GQA head map h -> h // (H_q/H_kv), causal
    bottom-right alignment and windows included."""
    rng = np.random.default_rng(page_size)
    h_q, h_kv, d = 6, 2, 16
    q_lens, kv_lens = [1, 4, 3], [9, 13, 3]
    c = _tiny_case(rng, 3, q_lens, kv_lens, h_q, h_kv, d, page_size)
    scale = 0.37
    for causal, wl in [(False, -1), (True, -1), (True, 2), (False, 5)]:
        out, lse, sk = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                        c["cu"], scale, causal, wl)
        assert sk == 0
        for b in range(3):
            for u in range(q_lens[b]):
                t = c["cu"][b] + u
                i = kv_lens[b] - q_lens[b] + u
                js = [j for j in range(kv_lens[b])
                      if (not causal or j <= i) and (wl < 0 or i - wl <= j <= i)]
                for h in range(h_q):
                    kvh = h // (h_q // h_kv)
                    K = c["klog"][b][js, kvh]
                    V = c["vlog"][b][js, kvh]
                    o_ref, l_ref = dense_reference_row(c["qf"][t, h], K, V, scale)
                    np.testing.assert_allclose(out[t, h], o_ref, rtol=0, atol=1e-12)
                    assert abs(lse[t, h] - l_ref) < 1e-12


@pytest.mark.parametrize("row", read_golden("causal_counts.txt"))
def test_visible_key_counts(row):
    """Bottom-right causal alignment and the (W, 0) window (golden fixture):
    with q = 0 every visible key gets weight 1/n, so with V = identity rows
    the output is 1/n on exactly the visible keys and lse = log n."""
    (kv_len, q_len, wl), counts = row
    d = kv_len
    kc = np.zeros((kv_len, 1, 1, d))
    vc = np.eye(kv_len).reshape(kv_len, 1, 1, d)
    qb, _ = bf16(np.zeros((q_len, 1, d)))
    kb, _ = bf16(kc)
    vb, _ = bf16(vc)
    pt = np.arange(kv_len, dtype=np.int32)[None, :]
    out, lse, _ = oracle.attention(qb, kb, vb, pt, [kv_len], [0, q_len], 1.0,
                                   causal=True, window_left=wl)
    for u in range(q_len):
        n = counts[u]
        i = kv_len - q_len + u
        expect = np.zeros(kv_len)
        expect[i - n + 1: i + 1] = 1.0 / n  # the n keys ending at position i
        np.testing.assert_allclose(out[u, 0], expect, atol=1e-15)
        assert abs(lse[u, 0] - math.log(n)) < 1e-14


def test_single_key_returns_its_value_row():
    """One visible key: weight 1, o = V_0 exactly, lse = s_0."""
    rng = np.random.default_rng(3)
    c = _tiny_case(rng, 1, [1], [1], 2, 1, 8, 4)
    out, lse, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                   c["cu"], 0.5)
    for h in range(2):
        assert np.array_equal(out[0, h], c["vlog"][0][0, 0])
        s0 = 0.5 * float(np.dot(c["qf"][0, h], c["klog"][0][0, 0]))
        assert abs(lse[0, h] - s0) < 1e-13


def test_constant_value_rows_return_the_constant():
    """Softmax weights sum to 1: V_j = v for all j gives o = v."""
    rng = np.random.default_rng(4)
    c = _tiny_case(rng, 2, [1, 1], [37, 5], 4, 2, 8, 4)
    vc = np.broadcast_to(np.array([1.5, -2.0, 0.25, 3.0, 0.0, 1.0, -0.5, 8.0]),
                         (c["vb"].shape)).copy()
    vb, _ = bf16(vc)
    out, _, _ = oracle.attention(c["qb"], c["kb"], vb, c["pt"], c["kv"], c["cu"], 0.9)
    np.testing.assert_allclose(out, np.broadcast_to(vc[0, 0, 0], out.shape),
                               rtol=0, atol=1e-13)


def test_two_keys_closed_form():
    """Two keys: o = sigma(s0 - s1) V0 + sigma(s1 - s0) V1,
    lse = s0 + log(1 + exp(s1 - s0))."""
    kc = np.array([[[[1.0, 0.0]]], [[[0.0, 1.0]]]])  # keys e0, e1
    vc = np.array([[[[2.0, -1.0]]], [[[0.5, 4.0]]]])
    qb, _ = bf16(np.array([[[3.0, 1.0]]]))
    kb, _ = bf16(kc)
    vb, _ = bf16(vc)
    out, lse, _ = oracle.attention(qb, kb, vb, np.array([[0, 1]]), [2], [0, 1], 0.5)
    s0, s1 = 1.5, 0.5
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    np.testing.assert_allclose(out[0, 0], w0 * vc[0, 0, 0] + (1 - w0) * vc[1, 0, 0],
                               atol=1e-15)
    assert abs(lse[0, 0] - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-15


def test_large_scale_selects_argmax_row():
    """scale -> infinity: softmax -> one-hot on the largest score."""
    rng = np.random.default_rng(5)
    c = _tiny_case(rng, 1, [1], [50], 1, 1, 16, 1)
    out, _, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                 c["cu"], 1e4)
    s = c["klog"][0][:, 0] @ c["qf"][0, 0]
    np.testing.assert_allclose(out[0, 0], c["vlog"][0][int(np.argmax(s)), 0], atol=1e-9)


def test_empty_kv_gives_zero_and_minus_inf():
    """cache_seqlens == 0 -> out = 0, lse = -inf
    (dual_chunk_flashattention_backend.py, exp-sums decode)."""
    rng = np.random.default_rng(6)
    c = _tiny_case(rng, 2, [1, 1], [0, 4], 2, 1, 8, 2)
    out, lse, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                   c["cu"], 1.0)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_page_permutation_invariance():
    """Relabelling physical pages (moving their contents and remapping the
    table) leaves every output bit unchanged."""
    rng = np.random.default_rng(8)
    c = _tiny_case(rng, 3, [1, 2, 1], [30, 17, 45], 4, 2, 8, 4)
    out0, lse0, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                     c["cu"], 0.4, causal=True)
    perm = rng.permutation(c["kb"].shape[0])  # new page id of old page p
    kb2 = np.empty_like(c["kb"])
    vb2 = np.empty_like(c["vb"])
    kb2[perm] = c["kb"]
    vb2[perm] = c["vb"]
    pt2 = perm[c["pt"]].astype(np.int32)
    out1, lse1, _ = oracle.attention(c["qb"], kb2, vb2, pt2, c["kv"], c["cu"], 0.4,
                                     causal=True)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_page_size_does_not_change_result():
    """The same logical KV laid out with P=1 and P=16 gives the same output."""
    rng = np.random.default_rng(9)
    kl = [rng.standard_normal((n, 1, 8)) for n in (21, 40)]
    vl = [rng.standard_normal((n, 1, 8)) for n in (21, 40)]
    qb, _ = bf16(rng.standard_normal((2, 2, 8)))
    outs = []
    for p in (1, 16):
        kc, pt = paged_from_logical(np.random.default_rng(1), kl, p)
        vc, _ = paged_from_logical(np.random.default_rng(1), vl, p)
        kb, _ = bf16(kc)
        vb, _ = bf16(vc)
        outs.append(oracle.attention(qb, kb, vb, pt, [21, 40], [0, 1, 2], 0.3)[:2])
    np.testing.assert_allclose(outs[0][0], outs[1][0], atol=1e-14)
    np.testing.assert_allclose(outs[0][1], outs[1][1], atol=1e-14)


def test_wide_window_equals_no_window_and_decode_equals_extend():
    rng = np.random.default_rng(10)
    c = _tiny_case(rng, 2, [1, 1], [25, 9], 2, 1, 8, 4)
    a = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"], c["cu"], 0.3)
    b = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"], c["cu"], 0.3,
                         causal=True, window_left=25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_mla_zero_rope_equals_mqa_over_latent():
    """Absorbed MLA (q = q_nope || q_rope, K row = c_kv || k_rope, V = c_kv):
    with k_rope = 0 the score is q_nope . c_kv, i.e. plain MQA over the latent
    dims with the value rows equal to the key rows."""
    rng = np.random.default_rng(12)
    d_l, d_r = 16, 4
    rows = rng.standard_normal((20, 1, 1, d_l + d_r))
    rows[..., d_l:] = 0.0
    kb, _ = bf16(rows)
    qb, _ = bf16(rng.standard_normal((1, 3, d_l + d_r)))
    pt = np.arange(20, dtype=np.int32)[None, :]
    mla = oracle.attention(qb, kb, kb, pt, [20], [0, 1], 0.2, d_v=d_l)
    lat = np.ascontiguousarray(kb[..., :d_l])
    mqa = oracle.attention(np.ascontiguousarray(qb[..., :d_l]), lat, lat, pt, [20],
                           [0, 1], 0.2)
    np.testing.assert_allclose(mla[0], mqa[0], atol=1e-14)
    np.testing.assert_allclose(mla[1], mqa[1], atol=1e-14)


def test_topk_full_list_equals_dense_and_duplicates_count():
    rng = np.random.default_rng(13)
    c = _tiny_case(rng, 2, [1, 1], [19, 33], 2, 1, 8, 4)
    dense = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"], c["cu"], 0.3)
    topk = np.full((2, 40), -1, dtype=np.int32)
    topk[0, :19] = rng.permutation(19)
    topk[1, :33] = rng.permutation(33)
    sparse = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"], c["cu"],
                              0.3, topk=topk)
    np.testing.assert_allclose(dense[0], sparse[0], atol=1e-14)
    np.testing.assert_allclose(dense[1], sparse[1], atol=1e-14)
    # an index listed twice counts twice: weight 2 e^{s_a} against e^{s_b}
    two = np.array([[3, 3, 7, -1], [0, -1, -1, -1]], dtype=np.int32)
    out, lse, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                   c["cu"], 0.3, topk=two)
    s = 0.3 * (c["klog"][0][[3, 7], 0] @ c["qf"][0, 0])
    wa = 2 * math.exp(s[0]) / (2 * math.exp(s[0]) + math.exp(s[1]))
    want = wa * c["vlog"][0][3, 0] + (1 - wa) * c["vlog"][0][7, 0]
    np.testing.assert_allclose(out[0, 0], want, atol=1e-13)
    # all -1: empty
    empty = np.full((2, 4), -1, dtype=np.int32)
    out, lse, sk = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                    c["cu"], 0.3, topk=empty)
    assert sk == 0 and np.all(out == 0) and np.all(np.isneginf(lse))
    # out of range entries are skipped and counted
    bad = np.array([[3, 19, -3, -1], [0, 1, 2, 3]], dtype=np.int32)
    _, _, sk = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                c["cu"], 0.3, topk=bad)
    assert sk == 2


def test_row_subset_matches_full():
    rng = np.random.default_rng(14)
    c = _tiny_case(rng, 2, [3, 2], [10, 20], 4, 2, 8, 4)
    full, lfull, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                      c["cu"], 0.3, causal=True)
    rows = np.array([[0, 3], [4, 1], [2, 0]], dtype=np.int32)
    sub, lsub, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                    c["cu"], 0.3, causal=True, rows=rows)
    for n, (t, h) in enumerate(rows):
        assert np.array_equal(sub[n], full[t, h]) and lsub[n] == lfull[t, h]


# ------------------------------------------------------------------------ merge

def test_merge_of_two_halves_equals_full_attention():
    """Merging the states of any two disjoint key halves equals attention
    over the whole key set (every split point, empty halves included)."""
    rng = np.random.default_rng(15)
    n = 23
    c = _tiny_case(rng, 1, [1], [n], 2, 1, 8, 1)
    full_o, full_l, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                         c["cu"], 0.6)
    for cut in range(0, n + 1):
        pa = c["pt"][:, :max(cut, 1)]
        pb = np.ascontiguousarray(c["pt"][:, cut:]) if cut < n else c["pt"][:, :1]
        oa, la, _ = oracle.attention(c["qb"], c["kb"], c["vb"], pa, [cut], c["cu"], 0.6)
        ob, lb, _ = oracle.attention(c["qb"], c["kb"], c["vb"], pb, [n - cut], c["cu"], 0.6)
        om, lm = oracle.merge_state(oa, la, ob, lb)
        np.testing.assert_allclose(om, full_o, atol=1e-13)
        np.testing.assert_allclose(lm, full_l, atol=1e-13)


def test_cascade_prefix_and_suffix_merge_to_single_call():
    """Cascade attention (flashattention_backend.py, `use_cascade_attn`): a
    call over the prefix pages without causal mask, a call over the suffix
    pages with the suffix's own lengths (causal, bottom-right), merged by
    log-sum-exp, equals one causal call over the whole table; prefixes of
    zero, one and several pages."""
    rng = np.random.default_rng(41)
    P = 4
    q_lens, kv_lens = [1, 3, 2], [13, 22, 9]
    c = _tiny_case(rng, 3, q_lens, kv_lens, 4, 2, 8, P)
    full_o, full_l, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"],
                                         c["cu"], 0.4, causal=True)
    for pre_pages in ([0, 0, 0], [1, 2, 1], [3, 4, 1]):
        pre_len = np.array([n * P for n in pre_pages], dtype=np.int32)
        suf_len = (c["kv"] - pre_len).astype(np.int32)
        assert np.all(suf_len >= np.array(q_lens))  # queries sit in the suffix
        width = c["pt"].shape[1]
        suf_pt = np.zeros_like(c["pt"])
        for b, n in enumerate(pre_pages):
            suf_pt[b, :width - n] = c["pt"][b, n:]
        oa, la, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], pre_len, c["cu"], 0.4,
                                     causal=False)
        ob, lb, _ = oracle.attention(c["qb"], c["kb"], c["vb"], suf_pt, suf_len, c["cu"], 0.4,
                                     causal=True)
        om, lm = oracle.merge_state(oa, la, ob, lb)
        np.testing.assert_allclose(om, full_o, atol=1e-13)
        np.testing.assert_allclose(lm, full_l, atol=1e-13)


def test_merge_closed_forms_and_algebra():
    rng = np.random.default_rng(16)
    va, vb, vc = (rng.standard_normal((5, 3, 4)) for _ in range(3))
    la, lb, lc = (rng.standard_normal((5, 3)) * 3 for _ in range(3))
    # equal lse: plain average, lse + log 2
    o, l = oracle.merge_state(va, la, vb, la)
    np.testing.assert_allclose(o, (va + vb) / 2, atol=1e-15)
    np.testing.assert_allclose(l, la + math.log(2), atol=1e-15)
    # commutative and associative
    o1, l1 = oracle.merge_state(va, la, vb, lb)
    o2, l2 = oracle.merge_state(vb, lb, va, la)
    np.testing.assert_allclose(o1, o2, atol=1e-15)
    np.testing.assert_allclose(l1, l2, atol=1e-15)
    x, lx = oracle.merge_state(*oracle.merge_state(va, la, vb, lb), vc, lc)
    y, ly = oracle.merge_state(va, la, *oracle.merge_state(vb, lb, vc, lc))
    np.testing.assert_allclose(x, y, atol=1e-14)
    np.testing.assert_allclose(lx, ly, atol=1e-14)
    # the n-way form on the pages (weights softmax(lse_i), merged lse of two
    # states = max + log1p(exp(-|lse_0 - lse_1|)))
    w = scipy.special.softmax(np.stack([la, lb, lc]), axis=0)
    np.testing.assert_allclose(x, w[0][..., None] * va + w[1][..., None] * vb
                               + w[2][..., None] * vc, atol=1e-14)
    np.testing.assert_allclose(l1, np.maximum(la, lb) + np.log1p(np.exp(-np.abs(la - lb))),
                               atol=1e-14)
    # an empty state is the identity; two empty states give (0, -inf)
    ninf = np.full_like(la, -np.inf)
    o, l = oracle.merge_state(va, la, np.zeros_like(vb), ninf)
    np.testing.assert_allclose(o, va, atol=0)
    np.testing.assert_allclose(l, la, atol=0)
    o, l = oracle.merge_state(va, ninf, vb, ninf)
    assert np.all(o == 0) and np.all(np.isneginf(l))


@pytest.mark.parametrize("num_splits", [1, 2, 4, 7])
def test_split_attention_equals_full(num_splits):
    """Split-KV partial states merged left to right equal single-pass
    attention, whatever the chunk boundaries."""
    wl = workloads.make("gqa_split_decode", batch=5, len_lo=1, len_hi=150,
                        pool_pages=200, h_q=4, h_kv=2, d=16)
    args = (oracle.bf16_bits(wl.q), oracle.bf16_bits(wl.k_cache),
            oracle.bf16_bits(wl.v_cache), wl.page_table.numpy(),
            wl.cache_seqlens.numpy(), wl.cu_seqlens_q.numpy(), wl.scale)
    full_o, full_l, _ = oracle.attention(*args)
    so, sl = oracle.split_attention(*args, num_splits=num_splits)
    np.testing.assert_allclose(so, full_o, atol=1e-13)
    np.testing.assert_allclose(sl, full_l, atol=1e-13)


def test_split_bounds_are_page_aligned_and_cover():
    for kv in (0, 1, 15, 16, 17, 1000, 8191):
        for p in (1, 16, 64):
            for s in (1, 2, 4, 5):
                b = oracle.split_bounds(kv, s, p)
                assert b[0][0] == 0 and b[-1][1] == kv
                for (lo, hi), (lo2, _) in zip(b, b[1:]):
                    assert hi == lo2 and (lo % p == 0 or lo == kv)


# ------------------------------------------- local (chunked) attention batches

def _vb_requests(cu, kv, out):
    """Request index of every virtual batch, from where its query tokens lie."""
    cu = np.asarray(cu)
    reqs = []
    for v in range(out["num_virtual"]):
        lo = out["cu_seqlens_q_local"][v]
        b = int(np.searchsorted(cu, lo, side="right") - 1)
        while cu[b + 1] - cu[b] == 0:  # requests with no new tokens own none
            b += 1
        reqs.append(b)
    return reqs


def _check_chunk_picture(cu, kv, pt, P, out):
    """Every virtual batch is the part of one request's queries that falls in
    one chunk: its queries are consecutive absolute positions of one chunk,
    the last of them is the last key the batch holds (bottom-right), its
    keys are the chunk's keys up to there, and its table row maps local key
    l to the page of absolute key chunk_start + l."""
    C = out["chunk"]
    cu = np.asarray(cu)
    reqs = _vb_requests(cu, kv, out)
    covered = np.zeros(cu[-1], dtype=int)
    for v, b in enumerate(reqs):
        lo, hi = out["cu_seqlens_q_local"][v], out["cu_seqlens_q_local"][v + 1]
        assert hi - lo == out["seqlens_q_local"][v] >= 1
        covered[lo:hi] += 1
        q_len = cu[b + 1] - cu[b]
        pos = [kv[b] - q_len + (t - cu[b]) for t in range(lo, hi)]
        assert len({p // C for p in pos}) == 1
        start = (pos[0] // C) * C
        k_local = out["seqlens_k_local"][v]
        assert start + k_local - 1 == pos[-1]
        assert k_local == min(C, kv[b] - start)
        for l in range(k_local):
            assert out["block_table_local"][v, l // P] == pt[b, (start + l) // P]
    # every query token is in exactly one virtual batch
    assert np.all(covered[cu[0]:] == 1)


@pytest.mark.parametrize("row", read_golden("local_virtual_batches.txt"))
def test_local_virtual_batches_printed_example(row):
    """The worked example printed with `make_local_attention_virtual_batches`
    (golden fixture): q_seqlens_local, seqlens_k_local, first-block tokens and
    local_blocks as printed; cu_seqlens_q_local is the running sum of the
    query lengths, and the printed cu line is the running sum of the key
    lengths."""
    (chunk, P), cu, kv, first, blocks, q_local, k_local, printed_cu = row
    width = -(-max(kv) // P)
    pt = np.array([[1000 * b + j for j in range(width)] for b in range(len(kv))])
    out = oracle.local_virtual_batches(chunk, P, cu, kv, pt)
    assert out["bad"] == 0 and out["chunk"] == chunk
    assert out["num_virtual"] == sum(blocks) == len(q_local)
    assert list(out["seqlens_q_local"]) == q_local
    assert list(out["seqlens_k_local"]) == k_local
    assert list(out["cu_seqlens_q_local"]) == [0] + list(np.cumsum(q_local))
    assert printed_cu == [0] + list(np.cumsum(k_local))
    starts = np.concatenate([[0], np.cumsum(blocks)[:-1]])
    assert [q_local[s] for s in starts] == first
    for b, (s, n) in enumerate(zip(starts, blocks)):
        assert sum(q_local[s:s + n]) == cu[b + 1] - cu[b]
    assert out["max_q_local"] == max(q_local) and out["max_k_local"] == max(k_local)
    _check_chunk_picture(cu, kv, pt, P, out)


def test_local_mask_printed_example():
    """The regular and the local (chunk 4) masks printed for batch index 0 of
    the example (q_seqlens 4, kv_seqlens 6), read off the oracle's attention:
    with q = 0 every visible key gets the same weight and one-hot value rows
    show which keys those are."""
    rows = read_golden("local_mask.txt")
    kv_len, q_len = 6, 4
    qb = np.zeros((q_len, 1, kv_len), dtype=np.uint16)
    eye = bf16(np.eye(kv_len)[:, None, :])[0]  # value row j = e_j
    kb = eye[None]  # one page of 6 slots, 1 head, D = 6
    vb = eye[None]
    pt = np.array([[0]], dtype=np.int32)
    for chunk in (0, 4):
        out, _, _ = oracle.attention(qb, kb, vb, pt, [kv_len], [0, q_len], 1.0,
                                     causal=True, attn_chunk=chunk)
        for (c, t), vis in rows:
            if c != chunk:
                continue
            got = (out[t, 0] > 0).astype(int)
            assert list(got) == vis
            np.testing.assert_allclose(out[t, 0][got == 1], 1.0 / sum(vis), atol=1e-15)


def _local_case(rng, q_lens, kv_lens, P, h_q=4, h_kv=2, d=8):
    c = _tiny_case(rng, len(q_lens), q_lens, kv_lens, h_q, h_kv, d, P)
    return c


@pytest.mark.parametrize("chunk,P,q_lens,kv_lens", [
    (4, 1, [4, 10, 5], [6, 17, 9]),          # the printed example
    (8, 4, [1, 1, 1, 1], [1, 8, 9, 30]),     # decode: one virtual batch each
    (8, 4, [13, 3, 8, 1], [13, 20, 16, 40]),  # extend spanning chunks
    (12, 4, [7, 20, 2], [30, 45, 2]),        # chunk of three pages
    (32, 4, [5, 17], [9, 17]),               # chunk > longest: cut to 16
    (6, 4, [9, 4], [25, 11]),                # chunk not a page multiple: 4
    (3, 4, [2, 5], [7, 12]),                 # chunk below a page: one page
])
def test_local_virtual_batches_equal_local_mask_attention(chunk, P, q_lens, kv_lens):
    """Brute force: causal attention over the virtual batches (their query
    offsets, key lengths and local tables) equals causal attention with the
    local chunk mask over the original table, element by element; and every
    virtual batch matches the chunk picture."""
    rng = np.random.default_rng(sum(kv_lens) + chunk)
    c = _local_case(rng, q_lens, kv_lens, P)
    out = oracle.local_virtual_batches(chunk, P, c["cu"], c["kv"], c["pt"])
    assert out["bad"] == 0
    _check_chunk_picture(c["cu"], c["kv"], c["pt"], P, out)
    ref_o, ref_l, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"], c["cu"],
                                       0.35, causal=True, attn_chunk=out["chunk"])
    got_o, got_l, _ = oracle.attention(c["qb"], c["kb"], c["vb"], out["block_table_local"],
                                       out["seqlens_k_local"], out["cu_seqlens_q_local"],
                                       0.35, causal=True)
    np.testing.assert_allclose(got_o, ref_o, atol=1e-13)
    np.testing.assert_allclose(got_l, ref_l, atol=1e-13)


def test_local_chunk_mask_changes_the_result():
    """The chunk mask is not a no-op: a query in the second chunk differs
    from plain causal attention, one in the first chunk does not."""
    rng = np.random.default_rng(3)
    c = _local_case(rng, [6], [6], 1)
    a, _, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"], c["cu"], 0.5,
                               causal=True, attn_chunk=4)
    b, _, _ = oracle.attention(c["qb"], c["kb"], c["vb"], c["pt"], c["kv"], c["cu"], 0.5,
                               causal=True)
    np.testing.assert_allclose(a[:4], b[:4], atol=1e-15)
    assert np.abs(a[4:] - b[4:]).max() > 1e-3
    # the token at position 4 sees only itself: its output is its value row
    np.testing.assert_allclose(a[4], c["vlog"][0][4][np.arange(4) // 2], atol=1e-15)


def test_local_effective_chunk_rule():
    """The chunk actually used: the given one, no longer than the longest
    sequence, cut down to whole pages, and never below one page."""
    def chunk_of(chunk, P, kv):
        cu = np.arange(len(kv) + 1)
        pt = np.zeros((len(kv), max(1, -(-max(kv) // P))), dtype=np.int32)
        return oracle.local_virtual_batches(chunk, P, cu, kv, pt)["chunk"]
    assert chunk_of(8192, 16, [100, 3000, 9000]) == 8192
    assert chunk_of(8192, 16, [100, 3000]) == 2992      # longest, whole pages
    assert chunk_of(32, 4, [17, 2]) == 16
    assert chunk_of(6, 4, [40]) == 4                     # whole pages
    assert chunk_of(3, 4, [40]) == 4                     # at least a page
    assert chunk_of(8, 4, [2]) == 4


def test_local_single_chunk_reproduces_the_input():
    """When the chunk covers every sequence, each request is one virtual
    batch with its own lengths and its own table row."""
    q_lens, kv = [3, 1, 16], [5, 9, 16]
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    pt = np.arange(3 * 4, dtype=np.int32).reshape(3, 4) + 50
    out = oracle.local_virtual_batches(64, 4, cu, kv, pt)
    assert out["chunk"] == 16 and out["num_virtual"] == 3
    assert list(out["seqlens_q_local"]) == q_lens
    assert list(out["seqlens_k_local"]) == kv
    assert list(out["cu_seqlens_q_local"]) == list(cu)
    assert np.array_equal(out["block_table_local"], pt)


def test_local_padding_idle_and_malformed_requests():
    """Rows past the count up to the capacity are padding (lengths 0, the
    running sum repeated, table row 0); a request with no new tokens makes
    no virtual batch; one with fewer keys than new tokens is counted and its
    tokens get key-less virtual batches of at most a chunk each, so later
    batches still address their own query rows; a table narrower than
    needed is rejected."""
    cu = np.array([0, 2, 2, 7, 13, 15])   # request 1 idle
    kv = np.array([5, 4, 12, 1, 3])       # request 3 malformed (kv < q)
    pt = np.arange(5 * 3, dtype=np.int32).reshape(5, 3) + 7
    out = oracle.local_virtual_batches(4, 2, cu, kv, pt, capacity=10, bt_cols=3)
    assert out["bad"] == 1 and out["chunk"] == 4
    n = out["num_virtual"]
    # request 0: positions 3, 4 (chunks 0, 1); request 2: positions 7..11
    # (chunks 1, 2); request 3: 6 tokens, no keys, chunks of 4 and 2;
    # request 4: positions 1, 2 (chunk 0)
    assert n == 2 + 2 + 2 + 1
    assert list(out["seqlens_q_local"][:n]) == [1, 1, 1, 4, 4, 2, 2]
    assert list(out["seqlens_k_local"][:n]) == [4, 1, 4, 4, 0, 0, 3]
    assert list(out["cu_seqlens_q_local"][:n + 1]) == [0, 1, 2, 3, 7, 11, 13, 15]
    assert np.all(out["block_table_local"][4:6] == 0)
    assert out["max_q_local"] == 4 and out["max_k_local"] == 4
    assert np.all(out["seqlens_q_local"][n:] == 0) and np.all(out["seqlens_k_local"][n:] == 0)
    assert np.all(out["cu_seqlens_q_local"][n:] == out["cu_seqlens_q_local"][n])
    assert np.all(out["block_table_local"][n:] == 0)
    assert np.all(out["block_table_local"][:n, 2] == 0)   # columns past C / P
    assert list(out["block_table_local"][0, :2]) == [pt[0, 0], pt[0, 1]]
    # request 0's second chunk is keys [4, 8): pages 2 and 3 of a 3-column
    # row -> the column past the row repeats its last entry
    assert list(out["block_table_local"][1, :2]) == [pt[0, 2], pt[0, 2]]
    with pytest.raises(ValueError):
        oracle.local_virtual_batches(8, 2, cu, kv, pt, capacity=8, bt_cols=3)


# ------------------------------------------------------------ KV write (append)

@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_set_kv_buffer_builds_the_paged_cache(page_size):
    """Writing every logical row of every request to slot
    page_table[b][j / P] * P + j % P reproduces the paged cache built
    page by page (the layout attention reads); the junk in unused slots is
    untouched."""
    rng = np.random.default_rng(71 + page_size)
    kv_lens = [5, 17, 1, 33]
    logical = [rng.standard_normal((n, 2, 8)) for n in kv_lens]
    want, pt = paged_from_logical(np.random.default_rng(9), logical, page_size)
    want_b, _ = bf16(want)
    # start from the same junk, with every slot some request owns cleared
    got = want_b.copy()
    for b, n in enumerate(kv_lens):
        for j in range(n):
            got[pt[b, j // page_size], j % page_size] = 0
    rows = np.concatenate([bf16(x)[0] for x in logical])
    loc = np.concatenate([[pt[b, j // page_size] * page_size + j % page_size
                           for j in range(n)] for b, n in enumerate(kv_lens)])
    assert oracle.set_kv_buffer(got, rows, loc) == 0
    assert np.array_equal(got, want_b)


def test_set_kv_buffer_then_attention_equals_dense_rows():
    """Append then attend: a pool holding each request's old keys, the new
    tokens' K/V written to their slots, then causal attention equals scipy
    softmax over the request's full logical rows."""
    rng = np.random.default_rng(72)
    P, q_lens, kv_lens = 4, [1, 3, 6], [9, 14, 6]
    c = _tiny_case(rng, 3, q_lens, kv_lens, 4, 2, 8, P)
    kb = c["kb"].copy()
    vb = c["vb"].copy()
    new_k, new_v, loc = [], [], []
    for b, (ql, n) in enumerate(zip(q_lens, kv_lens)):
        for j in range(n - ql, n):
            slot = c["pt"][b, j // P] * P + j % P
            loc.append(slot)
            new_k.append(kb[slot // P, slot % P].copy())
            new_v.append(vb[slot // P, slot % P].copy())
            kb[slot // P, slot % P] = 0x7fc0  # NaN until written
            vb[slot // P, slot % P] = 0x7fc0
    assert oracle.set_kv_buffer(kb, np.stack(new_k), loc) == 0
    assert oracle.set_kv_buffer(vb, np.stack(new_v), loc) == 0
    out, lse, _ = oracle.attention(c["qb"], kb, vb, c["pt"], c["kv"], c["cu"], 0.3,
                                   causal=True)
    for b, (ql, n) in enumerate(zip(q_lens, kv_lens)):
        for u in range(ql):
            t = c["cu"][b] + u
            i = n - ql + u
            for h in range(4):
                o, l = dense_reference_row(c["qf"][t, h], c["klog"][b][:i + 1, h // 2],
                                           c["vlog"][b][:i + 1, h // 2], 0.3)
                np.testing.assert_allclose(out[t, h], o, atol=1e-12)
                assert abs(lse[t, h] - l) < 1e-12


def test_set_kv_buffer_strides_and_out_of_pool_slots():
    """A head-major pool (strided view) is written through its strides; slots
    outside the pool are skipped and counted, nothing else changes; a
    repeated slot keeps the later row."""
    rng = np.random.default_rng(73)
    pool = bf16(rng.standard_normal((5, 2, 4, 8)))[0]      # [pages, H, P, D]
    view = pool.transpose(0, 2, 1, 3)                       # [pages, P, H, D]
    before = pool.copy()
    rows = bf16(rng.standard_normal((4, 2, 8)))[0]
    loc = [3, 19, -1, 20]                                   # 20 = 5 * 4 is past the pool
    assert oracle.set_kv_buffer(view, rows, loc) == 2
    assert np.array_equal(view[0, 3], rows[0]) and np.array_equal(view[4, 3], rows[1])
    mask = np.ones(pool.shape, bool)
    mask[0, :, 3] = False
    mask[4, :, 3] = False
    assert np.array_equal(pool[mask], before[mask])
    assert oracle.set_kv_buffer(view, rows[:2], [7, 7]) == 0
    assert np.array_equal(view[1, 3], rows[1])


# ------------------------------------------------------------------ FP8 KV

def test_e4m3_values_match_torch():
    """All 256 e4m3 codes widen to torch's float8_e4m3fn values (a library
    conversion), NaN codes included."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    assert oracle.e4m3_value(0x7e) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_rounding_matches_torch():
    """Round to nearest, ties to the even code, NaN past the largest value,
    subnormals: the oracle's encoder gives torch's codes for random values
    over the whole range, every tie point and the overflow edge."""
    rng = np.random.default_rng(91)
    vals = list(rng.standard_normal(2000) * np.exp2(rng.integers(-12, 9, 2000)))
    codes = np.arange(127)
    mags = np.array([oracle.e4m3_value(c) for c in codes])
    vals += list((mags[:-1] + mags[1:]) / 2)          # every midpoint (ties)
    vals += [448.0, 450.0, 463.9, 464.0, 464.1, 470.0, 479.0, 480.0, 1e4, 2.0 ** -10,
             3 * 2.0 ** -11, 2.0 ** -11, 0.0]
    vals += [-v for v in vals[:500]]
    vals += [-0.0, -1e-30, -(2.0 ** -11), -(3 * 2.0 ** -11)]   # zero keeps its sign
    vals += [float("inf"), float("-inf"), -464.0, -464.1, 1e30, -1e30]  # past the range
    x = torch.tensor(vals, dtype=torch.float64)
    ref = x.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_round(v) for v in x.to(torch.float32).double().tolist()])
    assert np.array_equal(got, ref)


def _fp8_case(rng, q_lens, kv_lens, P, h_q=4, h_kv=2, d=16):
    c = _tiny_case(rng, len(q_lens), q_lens, kv_lens, h_q, h_kv, d, P)
    codes = rng.integers(0, 256, size=c["kb"].shape, dtype=np.uint8)
    codes[(codes & 0x7f) == 0x7f] = 0x38           # no NaN codes in the cache
    vcodes = rng.integers(0, 256, size=c["vb"].shape, dtype=np.uint8)
    vcodes[(vcodes & 0x7f) == 0x7f] = 0x30
    return c, codes, vcodes


def _codes_to_bf16_bits(codes):
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float()
    return oracle.bf16_bits(vals.to(torch.bfloat16))


def test_fp8_attention_equals_bf16_attention_on_the_widened_values():
    """With unit descales, fp8 attention equals the bf16-path attention over
    caches holding the widened codes and q replaced by its e4m3 rounding
    (all exactly representable in bf16)."""
    rng = np.random.default_rng(92)
    c, kc, vc = _fp8_case(rng, [1, 3, 2], [9, 20, 5], 4)
    q32 = torch.from_numpy(c["qf"].astype(np.float32))
    q8 = q32.to(torch.float8_e4m3fn).float().to(torch.bfloat16)
    out, lse, _ = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.3,
                                       causal=True)
    ref_o, ref_l, _ = oracle.attention(oracle.bf16_bits(q8), _codes_to_bf16_bits(kc),
                                       _codes_to_bf16_bits(vc), c["pt"], c["kv"], c["cu"], 0.3,
                                       causal=True)
    np.testing.assert_allclose(out, ref_o, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, atol=1e-12)


def test_fp8_descale_closed_forms():
    """k_descale multiplies every score (same as a larger softmax scale);
    v_descale multiplies the output and leaves the lse alone."""
    rng = np.random.default_rng(93)
    c, kc, vc = _fp8_case(rng, [2, 1], [7, 12], 4)
    ones = np.ones((2, 2), np.float32)
    base_o, base_l, _ = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.6,
                                             k_descale=ones, v_descale=ones)
    o2, l2, _ = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.3,
                                     k_descale=2 * ones, v_descale=ones)
    np.testing.assert_allclose(o2, base_o, atol=1e-12)
    np.testing.assert_allclose(l2, base_l, atol=1e-12)
    o3, l3, _ = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.6,
                                     k_descale=ones, v_descale=3 * ones)
    np.testing.assert_allclose(o3, 3 * base_o, atol=1e-12)
    np.testing.assert_allclose(l3, base_l, atol=1e-12)


def test_fp8_per_request_descales_against_scipy():
    """Descales differ per (request, KV head): each row equals scipy's
    softmax over that request's rows dequantized with its own factors."""
    rng = np.random.default_rng(94)
    q_lens, kv_lens, P = [1, 2], [6, 11], 4
    c, kc, vc = _fp8_case(rng, q_lens, kv_lens, P, h_q=4, h_kv=2, d=8)
    kd = rng.uniform(0.5, 2.0, (2, 2)).astype(np.float32)
    vd = rng.uniform(0.5, 2.0, (2, 2)).astype(np.float32)
    out, lse, _ = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.45,
                                       causal=True, k_descale=kd, v_descale=vd)
    kval = torch.from_numpy(kc.copy()).view(torch.float8_e4m3fn).double().numpy()
    vval = torch.from_numpy(vc.copy()).view(torch.float8_e4m3fn).double().numpy()
    q8 = torch.from_numpy(c["qf"].astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    for b, (ql, n) in enumerate(zip(q_lens, kv_lens)):
        rows = [c["pt"][b, j // P] * P + j % P for j in range(n)]
        for u in range(ql):
            t = c["cu"][b] + u
            i = n - ql + u
            for h in range(4):
                kvh = h // 2
                K = np.stack([kval[s // P, s % P, kvh] for s in rows[:i + 1]]) * kd[b, kvh]
                V = np.stack([vval[s // P, s % P, kvh] for s in rows[:i + 1]]) * vd[b, kvh]
                o, l = dense_reference_row(q8[t, h], K, V, 0.45)
                np.testing.assert_allclose(out[t, h], o, atol=1e-12)
                assert abs(lse[t, h] - l) < 1e-12


def _topk_lists(rng, cu, kv_lens, width):
    """Per token: a random subset of its request's positions in random order,
    one repeated position, one position past kv_len, -1 padding."""
    total_q = int(cu[-1])
    tk = np.full((total_q, width), -1, np.int32)
    for b, n in enumerate(kv_lens):
        for t in range(int(cu[b]), int(cu[b + 1])):
            k = int(rng.integers(1, n + 1))
            sel = list(rng.permutation(n)[:k])
            sel = sel + [sel[0], n + 3]
            tk[t, :len(sel)] = np.array(sel[:width], np.int32)
    return tk


def test_fp8_topk_full_list_equals_dense_fp8():
    """A top-k list that names every position once (in any order, -1
    padded) gives the dense fp8 attention."""
    rng = np.random.default_rng(95)
    q_lens, kv_lens = [1, 2], [7, 12]
    c, kc, vc = _fp8_case(rng, q_lens, kv_lens, 4)
    tk = np.full((3, 16), -1, np.int32)
    for b, n in enumerate(kv_lens):
        for t in range(int(c["cu"][b]), int(c["cu"][b + 1])):
            tk[t, :n] = rng.permutation(n)
    kd = rng.uniform(0.5, 2.0, (2, 2)).astype(np.float32)
    vd = rng.uniform(0.5, 2.0, (2, 2)).astype(np.float32)
    o1, l1, _ = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.4,
                                     k_descale=kd, v_descale=vd, topk=tk)
    o2, l2, _ = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.4,
                                     k_descale=kd, v_descale=vd)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_fp8_topk_equals_bf16_topk_on_the_widened_values():
    """With unit descales, fp8 attention over top-k lists (repeats, -1,
    positions past kv_len, causal) equals the bf16-path attention over the
    same lists on the widened codes and q rounded to e4m3, with V the first
    columns of the K rows as for absorbed MLA; the skipped entries agree."""
    rng = np.random.default_rng(96)
    q_lens, kv_lens, P = [1, 3, 2], [9, 20, 5], 4
    c, kc, _ = _fp8_case(rng, q_lens, kv_lens, P, h_q=4, h_kv=1, d=24)
    vc = kc[..., :16]
    tk = _topk_lists(rng, c["cu"], kv_lens, 24)
    q8 = torch.from_numpy(c["qf"].astype(np.float32)).to(torch.float8_e4m3fn).float()
    kb = _codes_to_bf16_bits(kc)
    out, lse, sk = oracle.attention_fp8(c["qb"], kc, vc, c["pt"], c["kv"], c["cu"], 0.3,
                                        causal=True, topk=tk)
    ref_o, ref_l, ref_sk = oracle.attention(oracle.bf16_bits(q8.to(torch.bfloat16)), kb,
                                            kb[..., :16], c["pt"], c["kv"], c["cu"], 0.3,
                                            causal=True, topk=tk, d_v=16)
    np.testing.assert_allclose(out, ref_o, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, atol=1e-12)
    assert sk > 0 and sk == ref_sk * 4  # (per row here, per token's head 0 there)


# ------------------------------------------------- KV write into an fp8 pool

@pytest.mark.parametrize("scale", [1.0, 0.05, 0.3, 7.0])
def test_fp8_kv_write_equals_torch_division_and_cast(scale):
    """The quantising write stores, at each slot, torch's e4m3 cast of the
    binary32 quotient row / scale (a library routine the oracle does not
    call): random rows over a wide range, rows whose quotients fall exactly
    on midpoints between codes (ties), quotients past the format's range,
    a strided pool and out-of-pool slots (skipped, counted, pool untouched)."""
    rng = np.random.default_rng(95)
    T, H, D, P, NP = 9, 2, 32, 4, 8
    vals = rng.standard_normal((T, H, D)) * np.exp2(rng.integers(-6, 5, (T, H, D)))
    mags = np.array([oracle.e4m3_value(c) for c in range(127)])
    mids = (mags[:-1] + mags[1:]) / 2
    vals[0, 0, :] = mids[rng.integers(40, 120, D)] * scale     # ties after division
    vals[1, 1, :4] = [460.0 * scale, 470.0 * scale, -500.0 * scale, 448.0 * scale]
    rows = torch.from_numpy(vals).to(torch.bfloat16)
    bits = oracle.bf16_bits(rows)
    big = np.zeros((NP, P, H + 1, D + 16), np.uint8)            # strided view
    pool = big[:, :, 1:, 8:8 + D]
    loc = np.array([5, 0, 31, -1, 17, 32, 2, 9, 30])
    n = oracle.set_kv_buffer_fp8(pool, bits, loc, scale)
    assert n == 2
    ref = (rows.float() / torch.tensor(scale, dtype=torch.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    want = np.zeros_like(pool)
    for t, s in enumerate(loc):
        if 0 <= s < NP * P:
            want[s // P, s % P] = ref[t]
    assert np.array_equal(pool, want)
    assert not big[:, :, 0].any() and not big[:, :, :, :8].any() and not big[:, :, :, 8 + D:].any()


def test_fp8_kv_write_reads_back_within_e4m3_precision():
    """Reading a stored code back as value(code) * scale recovers the row
    to e4m3 precision: relative error at most 2^-4 for normal codes, at most
    half the subnormal step times the scale below them."""
    rng = np.random.default_rng(96)
    rows = torch.from_numpy(rng.standard_normal((16, 2, 64))).to(torch.bfloat16)
    scale = 0.02
    pool = np.zeros((4, 4, 2, 64), np.uint8)
    assert oracle.set_kv_buffer_fp8(pool, oracle.bf16_bits(rows), np.arange(16), scale) == 0
    back = np.vectorize(oracle.e4m3_value)(pool.reshape(16, 2, 64)) * scale
    x = rows.double().numpy()
    normal = np.abs(x) / scale >= 2.0 ** -6
    assert np.all(np.abs(back - x)[normal] <= np.abs(x)[normal] * 2.0 ** -4 + 1e-12)
    assert np.all(np.abs(back - x)[~normal] <= 2.0 ** -10 * scale + 1e-12)


def test_fp8_kv_write_rejects_bad_scales():
    pool = np.zeros((1, 1, 1, 16), np.uint8)
    rows = np.zeros((1, 1, 16), np.uint16)
    for s in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(ValueError):
            oracle.set_kv_buffer_fp8(pool, rows, np.zeros(1), s)


def test_swa_page_table_skips_malformed_rows_whole():
    """A row with a pool index out of range, a kv_len past dst's width or a
    source column past req_to_token's width is not written at all and gets
    kv_len -1; the valid rows of the same batch follow the rule (brute-force
    membership: position p kept iff p < pf or p >= sl - window)."""
    rng = np.random.default_rng(97)
    pool, ctx = 5, 40
    rtt = rng.permutation(pool * ctx).astype(np.int32).reshape(pool, ctx)
    pfl = np.array([3, 0, 6, 2, 9], dtype=np.int32)
    rpi = [0, 7, 1, 2, -1, 3, 4]
    sl = [12, 5, 30, 41, 5, 20, 35]        # row 3 needs column 40 of a 40-wide row
    window, W = 8, 16                       # row 6: kv_len 17 > 16
    dst, kv, n = oracle.swa_page_table(rtt, rpi, sl, pfl, window, W, fill=-9)
    assert n == 4
    for b, (r, s) in enumerate(zip(rpi, sl)):
        if b in (1, 3, 4, 6):
            assert kv[b] == -1 and np.all(dst[b] == -9), b
            continue
        keep = [p for p in range(s) if p < pfl[r] or p >= s - window]
        assert kv[b] == len(keep)
        assert list(dst[b, :len(keep)]) == [rtt[r, p] for p in keep]
        assert np.all(dst[b, len(keep):] == -9)
