"""Seeded synthetic workloads for paged-KV attention.

This module only draws inputs: lengths, page permutations, top-k lists and
N(0, 1) values rounded to bf16.  It holds none of the attention arithmetic and
is shared, unchanged, by the CUDA-path tests, the bench and the oracle checks,
so both sides always see bit-identical inputs.

Layout produced (the paged KV layout of the SGLang FlashAttention backend,
flashattention_backend.py ``forward_extend``: K/V buffers viewed
``[num_pages, page_size, H_kv, D]``):

* ``req_to_token``  int32 ``[pool_rows, max_ctx]`` token -> KV slot, row
  ``req_pool_indices[b]`` belongs to request b;
* ``page_table``    int32 ``[B, max_pages]`` page ids, request b's token j in
  slot ``page_table[b, j // P] * P + j % P`` (the allocator hands each request
  whole pages drawn from one seeded permutation of the pool);
* ``k_cache`` / ``v_cache`` bf16 ``[num_pages, P, H_kv, D]``; for absorbed MLA
  ``v_cache`` is the view ``k_cache[..., :512]`` of the 576-wide latent rows.

Integer structure is always drawn on the CPU (seed ``1000 + config``), so it is
the same whichever device the values are drawn on.  Values are drawn on
``value_device`` with a generator of that device: on the CPU for the small
cases, on the GPU for the full-size ones (CPU drawing of several GB takes
minutes).  The oracle always consumes the bits that were actually drawn.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

BF16 = torch.bfloat16

# The five synthetic workloads (names, then their parameters).
CONFIGS = {
    # batch 4, 1 query token each, 8 q heads / 2 kv heads, head_dim 128,
    # page_size 1, cache_seqlens ~ U[1, 256], pool of 2048 slots
    "tiny_decode": dict(kind="decode", batch=4, h_q=8, h_kv=2, d=128,
                        page_size=1, len_lo=1, len_hi=256, pool_tokens=2048,
                        num_splits=1, seed=1000),
    # batch 64, 32/8 heads, head_dim 128, page_size 16, U[512, 8192],
    # 40k-page pool, KV split into 4 chunks combined by the state merge
    "gqa_split_decode": dict(kind="decode", batch=64, h_q=32, h_kv=8, d=128,
                             page_size=16, len_lo=512, len_hi=8192,
                             pool_pages=40000, num_splits=4, seed=1001),
    # batch 32, 64/8 heads, head_dim 128, page_size 1, window 4096,
    # prefill_len ~ U[256, 2048], seq_len ~ U[prefill_len+1, 32768]
    "swa_decode": dict(kind="swa", batch=32, h_q=64, h_kv=8, d=128,
                       page_size=1, window=4096, pf_lo=256, pf_hi=2048,
                       sl_hi=32768, num_splits=0, seed=1002),
    # batch 8, new ~ U[128, 2048] on a prefix ~ U[0, 4096], 32/8 heads,
    # head_dim 128, page_size 64, 1024-page pool, causal
    "varlen_extend": dict(kind="extend", batch=8, h_q=32, h_kv=8, d=128,
                          page_size=64, new_lo=128, new_hi=2048, prefix_lo=0,
                          prefix_hi=4096, pool_pages=1024, seed=1003),
    # batch 128, 128 q heads / 1 latent head, K 576 (512 + 64), V 512,
    # kv_len 8192, page_size 64, top-k 2048 drawn without replacement
    "mla_topk_decode": dict(kind="mla", batch=128, h_q=128, h_kv=1, d_qk=576,
                            d_v=512, page_size=64, kv_len=8192, topk=2048,
                            pool_pages=16384, seed=1004),
}


@dataclass
class PagedBatch:
    """One batch of paged-attention inputs (see module docstring)."""

    name: str
    kind: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    req_to_token: torch.Tensor
    req_pool_indices: torch.Tensor
    page_table: torch.Tensor
    cache_seqlens: torch.Tensor
    cu_seqlens_q: torch.Tensor
    max_seqlen_q: int
    scale: float
    causal: bool = False
    window_left: int = -1
    num_splits: int = 1
    topk_indices: Optional[torch.Tensor] = None
    # prefill-aware sliding window inputs (pool-sized prefill_lens)
    prefill_lens: Optional[torch.Tensor] = None
    seq_lens: Optional[torch.Tensor] = None
    window: int = -1
    extra: dict = field(default_factory=dict)

    @property
    def page_size(self) -> int:
        return int(self.k_cache.shape[1])

    def to(self, device) -> "PagedBatch":
        def mv(t):
            return None if t is None else t.to(device)

        out = PagedBatch(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("q", "req_to_token", "req_pool_indices", "page_table",
                  "cache_seqlens", "cu_seqlens_q", "topk_indices",
                  "prefill_lens", "seq_lens"):
            setattr(out, k, mv(getattr(self, k)))
        out.k_cache = self.k_cache.to(device)
        if self.v_cache.data_ptr() == self.k_cache.data_ptr():
            out.v_cache = out.k_cache[..., : self.v_cache.shape[-1]]
        else:
            out.v_cache = self.v_cache.to(device)
        return out


def _randint(g, lo, hi, n):
    """n integers uniform on the closed interval [lo, hi]."""
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)


def _normal_bf16(shape, value_device, seed):
    g = torch.Generator(device=value_device).manual_seed(seed)
    out = torch.empty(shape, dtype=BF16, device=value_device)
    flat = out.view(-1)
    step = 1 << 26
    for s in range(0, flat.numel(), step):
        e = min(s + step, flat.numel())
        flat[s:e] = torch.randn(e - s, generator=g, device=value_device).to(BF16)
    return out


def _assign_pages(g, kv_lens, page_size, num_pages, pool_rows):
    """Each request gets whole pages: disjoint consecutive segments of one
    seeded permutation of the page pool.  Returns (page_table, req_to_token,
    req_pool_indices)."""
    batch = len(kv_lens)
    pages_needed = [max(1, -(-int(n) // page_size)) for n in kv_lens]
    if sum(pages_needed) > num_pages:
        raise ValueError("page pool too small for the drawn lengths")
    perm = torch.randperm(num_pages, generator=g, dtype=torch.int64)
    max_pages = max(pages_needed)
    page_table = torch.zeros(batch, max_pages, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_needed):
        page_table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    # request b lives in a seeded row of a slightly larger req_to_token pool
    req_pool_indices = torch.randperm(pool_rows, generator=g)[:batch].to(torch.int64)
    max_ctx = max_pages * page_size
    req_to_token = torch.zeros(pool_rows, max_ctx, dtype=torch.int32)
    within = torch.arange(max_ctx, dtype=torch.int32) % page_size
    for b in range(batch):
        pages = page_table[b].repeat_interleave(page_size)
        req_to_token[req_pool_indices[b]] = pages * page_size + within
    return page_table, req_to_token, req_pool_indices


def make(name: str, value_device="cpu", seed: Optional[int] = None,
         **overrides) -> PagedBatch:
    """Draw the workload ``name`` (a key of CONFIGS).  ``overrides`` shrink a
    workload for tests (e.g. ``batch=2, len_hi=300``); the structure recipe is
    unchanged.  All tensors are returned on ``value_device``."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    seed = cfg["seed"] if seed is None else seed
    g = torch.Generator().manual_seed(seed)
    kind = cfg["kind"]
    if kind == "decode":
        b = cfg["batch"]
        p = cfg["page_size"]
        kv = _randint(g, cfg["len_lo"], cfg["len_hi"], b)
        num_pages = cfg.get("pool_pages") or cfg["pool_tokens"] // p
        pt, rtt, rpi = _assign_pages(g, kv.tolist(), p, num_pages, b + 3)
        q_len = cfg.get("q_len", 1)
        cu = torch.arange(0, b * q_len + 1, q_len, dtype=torch.int32)
        kc = _normal_bf16((num_pages, p, cfg["h_kv"], cfg["d"]), value_device, seed + 1)
        vc = _normal_bf16((num_pages, p, cfg["h_kv"], cfg["d"]), value_device, seed + 2)
        q = _normal_bf16((b * q_len, cfg["h_q"], cfg["d"]), value_device, seed + 3)
        batch = PagedBatch(
            name=name, kind=kind, q=q, k_cache=kc, v_cache=vc, req_to_token=rtt,
            req_pool_indices=rpi, page_table=pt, cache_seqlens=kv.to(torch.int32),
            cu_seqlens_q=cu, max_seqlen_q=q_len, scale=1.0 / math.sqrt(cfg["d"]),
            causal=bool(cfg.get("causal", q_len > 1)),
            window_left=cfg.get("window_left", -1), num_splits=cfg["num_splits"])
    elif kind == "swa":
        b = cfg["batch"]
        pf = _randint(g, cfg["pf_lo"], cfg["pf_hi"], b)
        sl = torch.stack([_randint(g, int(x) + 1, cfg["sl_hi"], 1)[0] for x in pf])
        # one slot permutation of a pool of sum(seq_len) slots; request b owns
        # a disjoint consecutive segment of it (page_size 1: a page is a slot)
        num_slots = int(sl.sum())
        pt, rtt, rpi = _assign_pages(g, sl.tolist(), 1, num_slots, b + 3)
        prefill_lens = torch.zeros(b + 3, dtype=torch.int32)
        prefill_lens[rpi] = pf.to(torch.int32)
        kc = _normal_bf16((num_slots, 1, cfg["h_kv"], cfg["d"]), value_device, seed + 1)
        vc = _normal_bf16((num_slots, 1, cfg["h_kv"], cfg["d"]), value_device, seed + 2)
        q = _normal_bf16((b, cfg["h_q"], cfg["d"]), value_device, seed + 3)
        batch = PagedBatch(
            name=name, kind=kind, q=q, k_cache=kc, v_cache=vc, req_to_token=rtt,
            req_pool_indices=rpi, page_table=pt, cache_seqlens=sl.to(torch.int32),
            cu_seqlens_q=torch.arange(b + 1, dtype=torch.int32), max_seqlen_q=1,
            scale=1.0 / math.sqrt(cfg["d"]), causal=False, window_left=-1,
            num_splits=cfg["num_splits"], prefill_lens=prefill_lens,
            seq_lens=sl.to(torch.int32), window=cfg["window"])
    elif kind == "extend":
        b = cfg["batch"]
        p = cfg["page_size"]
        new = _randint(g, cfg["new_lo"], cfg["new_hi"], b)
        prefix = _randint(g, cfg["prefix_lo"], cfg["prefix_hi"], b)
        kv = new + prefix
        pt, rtt, rpi = _assign_pages(g, kv.tolist(), p, cfg["pool_pages"], b + 3)
        cu = torch.zeros(b + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(new, 0).to(torch.int32)
        kc = _normal_bf16((cfg["pool_pages"], p, cfg["h_kv"], cfg["d"]), value_device, seed + 1)
        vc = _normal_bf16((cfg["pool_pages"], p, cfg["h_kv"], cfg["d"]), value_device, seed + 2)
        q = _normal_bf16((int(new.sum()), cfg["h_q"], cfg["d"]), value_device, seed + 3)
        batch = PagedBatch(
            name=name, kind=kind, q=q, k_cache=kc, v_cache=vc, req_to_token=rtt,
            req_pool_indices=rpi, page_table=pt, cache_seqlens=kv.to(torch.int32),
            cu_seqlens_q=cu, max_seqlen_q=int(new.max()),
            scale=1.0 / math.sqrt(cfg["d"]), causal=True,
            window_left=cfg.get("window_left", -1), num_splits=1)
        batch.extra["prefix_lens"] = prefix.to(torch.int32)
    elif kind == "mla":
        b = cfg["batch"]
        p = cfg["page_size"]
        kv_len = cfg["kv_len"]
        kv = torch.full((b,), kv_len, dtype=torch.int64)
        pt, rtt, rpi = _assign_pages(g, kv.tolist(), p, cfg["pool_pages"], b + 3)
        topk = torch.stack([torch.randperm(kv_len, generator=g)[:cfg["topk"]]
                            for _ in range(b)]).to(torch.int32)
        kc = _normal_bf16((cfg["pool_pages"], p, 1, cfg["d_qk"]), value_device, seed + 1)
        q = _normal_bf16((b, cfg["h_q"], cfg["d_qk"]), value_device, seed + 3)
        batch = PagedBatch(
            name=name, kind=kind, q=q, k_cache=kc, v_cache=kc[..., : cfg["d_v"]],
            req_to_token=rtt, req_pool_indices=rpi, page_table=pt,
            cache_seqlens=kv.to(torch.int32),
            cu_seqlens_q=torch.arange(b + 1, dtype=torch.int32), max_seqlen_q=1,
            scale=1.0 / math.sqrt(192.0), causal=False, window_left=-1,
            num_splits=cfg.get("num_splits", 0), topk_indices=topk)
    else:
        raise ValueError(kind)
    return batch.to(value_device) if str(value_device) != "cpu" else batch
