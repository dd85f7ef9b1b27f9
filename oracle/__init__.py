"""float64 CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls it, and it shares no code with the CUDA library: the arithmetic lives in
``pkv_oracle.c`` (plain C, float64), this module only marshals numpy arrays.

Every function restates a definition from the SGLang attention-backend pages:

* ``strided_page_table`` -- flashattention_backend.py, ``init_forward_metadata``
  ("Convert the page table to a strided format").
* ``swa_page_table`` -- flashattention_backend.py, ``_build_pa_page_table_kernel``.
* ``topk_to_slots`` -- nsa_backend.py, ``TopkTransformMethod.PAGED``.
* ``set_kv_buffer`` -- flashattention_backend.py ``forward_extend`` /
  ``forward_decode``: the new tokens' K/V written to their slots
  (``set_kv_buffer`` / ``set_mla_kv_buffer``) before attention.
* ``e4m3_value`` / ``e4m3_round`` / ``attention_fp8`` -- flashattention_backend.py
  fp8 KV cache: q cast to the cache dtype, ``k_descale`` / ``v_descale`` per
  (request, KV head).
* ``local_virtual_batches`` -- flashattention_backend.py,
  ``make_local_attention_virtual_batches`` (local chunked attention as
  virtual batches) and the mask drawn in its worked example
  (``attention(..., attn_chunk=C)``).
* ``attention`` -- flashattention_backend.py ``forward_decode`` /
  ``forward_extend`` (``flash_attn_with_kvcache``), absorbed MLA call,
  nsa_backend.py ``forward_decode`` (top-k), bottom-right causal alignment
  (nsa_backend.py ``seqlens_expanded``), empty-KV convention
  (dual_chunk_flashattention_backend.py,
  ``_dual_chunk_flash_attn_decoding_with_exp_sums``).
* ``merge_state`` -- dual_chunk_flashattention_backend.py,
  ``_merge_attn_outputs``; ``merge_state_v2`` call in flashattention_backend.py.
* ``split_bounds`` / ``split_attention`` -- split-KV partials combined by the
  state merge (flashattention_backend.py ``num_splits``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from ._build import build_oracle, oracle_lib_path

__all__ = [
    "strided_page_table",
    "swa_page_table",
    "topk_to_slots",
    "local_virtual_batches",
    "set_kv_buffer",
    "e4m3_value",
    "e4m3_round",
    "attention_fp8",
    "attention",
    "merge_state",
    "split_bounds",
    "split_attention",
    "bf16_bits",
]

_LIB = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64
_int = ctypes.c_int


def _lib():
    global _LIB
    if _LIB is None:
        path = oracle_lib_path()
        if not os.path.exists(path) or os.path.getmtime(path) < _src_mtime():
            build_oracle()
        lib = ctypes.CDLL(path)
        lib.orc_strided_page_table.argtypes = [
            _i32p, _i64, _i64, _i64p, _int, _int, _int, _i32p, _i64]
        lib.orc_swa_page_table.argtypes = [
            _i32p, _i64, _i64, _i64, _i64p, _i32p, _i32p, _int, _int, _i32p, _i64,
            _int, _i32p]
        lib.orc_topk_to_slots.argtypes = [
            _i32p, _i64, _int, _int, _i32p, _i32p, _i64, _int, _int, _i32p,
            _i32p, _i64]
        lib.orc_attention.argtypes = [
            _u16p, _i64, _i64, _int, _int, _int,
            _u16p, _i64, _i64, _i64,
            _u16p, _i64, _i64, _i64, _int,
            _int, _int, _i64,
            _i32p, _i64, _int,
            _i32p, _i32p, _int, ctypes.c_double, _int, _int, _int,
            _i32p, _i64, _int,
            _i32p, _int, _f64p, _f64p, _int]
        _u8p = ctypes.POINTER(ctypes.c_uint8)
        _f32p = ctypes.POINTER(ctypes.c_float)
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_e4m3_round.argtypes = [ctypes.c_double]
        lib.orc_e4m3_round.restype = ctypes.c_uint8
        lib.orc_attention_fp8.argtypes = [
            _u16p, _i64, _i64, _int, _int, _int,
            _u8p, _i64, _i64, _i64,
            _u8p, _i64, _i64, _i64, _int,
            _int, _int, _i64,
            _i32p, _i64, _int,
            _i32p, _i32p, _int, ctypes.c_double, _int, _int,
            _f32p, _f32p, _i32p, _i64, _int, _f64p, _f64p, _int]
        lib.orc_attention_fp8.restype = ctypes.c_int
        lib.orc_set_kv_buffer.argtypes = [
            _u16p, _i64, _i64, _int, _int, _int, _i64p, _u16p, _i64, _i64, _i64,
            _i64, _int]
        lib.orc_set_kv_buffer_fp8.argtypes = [
            _u16p, _i64, _i64, _int, _int, _int, _i64p, ctypes.c_float, _u8p, _i64, _i64,
            _i64, _i64, _int]
        lib.orc_set_kv_buffer_fp8.restype = ctypes.c_int
        lib.orc_local_virtual_batches.argtypes = [
            _int, _int, _i32p, _i32p, _int, _i32p, _i64, _int, _int,
            _i32p, _i32p, _i32p, _i32p, _i64, _int, _i32p]
        lib.orc_merge_state.argtypes = [
            _f64p, _f64p, _f64p, _f64p, _i64, _int, _f64p, _f64p]
        for fn in ("orc_strided_page_table", "orc_swa_page_table",
                   "orc_topk_to_slots", "orc_attention", "orc_merge_state",
                   "orc_local_virtual_batches", "orc_set_kv_buffer"):
            getattr(lib, fn).restype = ctypes.c_int
        _LIB = lib
    return _LIB


def _src_mtime() -> float:
    here = os.path.dirname(os.path.abspath(__file__))
    return max(os.path.getmtime(os.path.join(here, f))
               for f in ("pkv_oracle.c", "pkv_oracle.h"))


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def bf16_bits(t) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU torch bf16 tensor, as a uint16 array."""
    import torch

    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _elem_strides(a: np.ndarray) -> tuple[int, ...]:
    return tuple(s // a.itemsize for s in a.strides)


def strided_page_table(req_to_token, req_pool_indices, page_size: int,
                       n_cols: int) -> np.ndarray:
    rtt = np.ascontiguousarray(req_to_token, dtype=np.int32)
    rpi = np.ascontiguousarray(req_pool_indices, dtype=np.int64)
    out = np.zeros((len(rpi), n_cols), dtype=np.int32)
    rc = _lib().orc_strided_page_table(
        _ptr(rtt, ctypes.c_int32), rtt.shape[1], rtt.shape[1],
        _ptr(rpi, ctypes.c_int64), len(rpi), page_size, n_cols,
        _ptr(out, ctypes.c_int32), n_cols)
    if rc != 0:
        raise ValueError(f"orc_strided_page_table rejected its arguments ({rc})")
    return out


def swa_page_table(req_to_token, req_pool_indices, seq_lens, prefill_lens,
                   window: int, dst_cols: int, fill: int = 0):
    """Returns (dst [B, dst_cols] int32, kv_lens [B] int32, n_rows_skipped).

    Columns at or past kv_len keep ``fill``; a malformed row (pool index out
    of range, kv_len past dst_cols, a source column past the table's width)
    is left as ``fill`` with kv_len -1 and counted."""
    rtt = np.ascontiguousarray(req_to_token, dtype=np.int32)
    rpi = np.ascontiguousarray(req_pool_indices, dtype=np.int64)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    pf = np.ascontiguousarray(prefill_lens, dtype=np.int32)
    dst = np.full((len(rpi), dst_cols), fill, dtype=np.int32)
    kv = np.zeros(len(rpi), dtype=np.int32)
    rc = _lib().orc_swa_page_table(
        _ptr(rtt, ctypes.c_int32), rtt.shape[1], rtt.shape[1], rtt.shape[0],
        _ptr(rpi, ctypes.c_int64), _ptr(sl, ctypes.c_int32),
        _ptr(pf, ctypes.c_int32), len(rpi), window, _ptr(dst, ctypes.c_int32),
        dst_cols, dst_cols, _ptr(kv, ctypes.c_int32))
    if rc < 0:
        raise ValueError(f"orc_swa_page_table rejected its arguments ({rc})")
    return dst, kv, rc


def topk_to_slots(topk, row_req, page_table, page_size: int,
                  cache_seqlens=None):
    """Returns (slots [rows, topk] int32, n_out_of_range)."""
    tk = np.ascontiguousarray(topk, dtype=np.int32)
    rr = np.ascontiguousarray(row_req, dtype=np.int32)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cs = None if cache_seqlens is None else np.ascontiguousarray(
        cache_seqlens, dtype=np.int32)
    out = np.zeros_like(tk)
    rc = _lib().orc_topk_to_slots(
        _ptr(tk, ctypes.c_int32), tk.shape[1], tk.shape[0], tk.shape[1],
        _ptr(rr, ctypes.c_int32), _ptr(pt, ctypes.c_int32), pt.shape[1],
        pt.shape[1], page_size, _ptr(cs, ctypes.c_int32),
        _ptr(out, ctypes.c_int32), tk.shape[1])
    if rc < 0:
        raise ValueError(f"orc_topk_to_slots rejected its arguments ({rc})")
    return out, rc


def e4m3_value(code: int) -> float:
    """Value of one e4m3 code (NaN for 0x7f / 0xff)."""
    return _lib().orc_e4m3_value(int(code))


def e4m3_round(x: float) -> int:
    """Nearest e4m3 code to x (ties to the even code; NaN code past 464)."""
    return int(_lib().orc_e4m3_round(float(x)))


def attention_fp8(q_bits, k_codes, v_codes, page_table, cache_seqlens, cu_seqlens_q,
                  scale: float, causal: bool = False, window_left: int = -1,
                  k_descale=None, v_descale=None, num_threads: int = 0, topk=None):
    """Attention over an fp8 (e4m3) paged cache in float64: q rounded to
    e4m3, K/V codes widened and multiplied by their (request, KV head)
    descales.  q_bits: uint16 [total_q, H_q, D]; k_codes / v_codes: uint8
    [num_pages, P, H_kv, D] (D contiguous; V may be a column slice of K, as
    for absorbed MLA); descales: float32 [B, H_kv] or None; topk: optional
    int32 [total_q, L] position lists (as in attention).  Returns (out
    [total_q, H_q, Dv], lse [total_q, H_q], n_skipped)."""
    q = np.asarray(q_bits)
    k = np.asarray(k_codes)
    v = np.asarray(v_codes)
    assert q.dtype == np.uint16 and k.dtype == np.uint8 and v.dtype == np.uint8
    assert q.strides[2] == 2 and k.strides[3] == 1 and v.strides[3] == 1
    total_q, h_q, d = q.shape
    num_pages, page_size, h_kv, _ = k.shape
    d_v = v.shape[3]
    qs, ks, vs = _elem_strides(q), _elem_strides(k), _elem_strides(v)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cs = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    kd = None if k_descale is None else np.ascontiguousarray(k_descale, dtype=np.float32)
    vd = None if v_descale is None else np.ascontiguousarray(v_descale, dtype=np.float32)
    tk = None if topk is None else np.ascontiguousarray(topk, dtype=np.int32)
    out = np.zeros((total_q * h_q, d_v), dtype=np.float64)
    lse = np.zeros(total_q * h_q, dtype=np.float64)
    rc = _lib().orc_attention_fp8(
        _ptr(q, ctypes.c_uint16), qs[0], qs[1], total_q, h_q, d,
        k.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), ks[0], ks[1], ks[2],
        v.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), vs[0], vs[1], vs[2], d_v,
        h_kv, page_size, num_pages, _ptr(pt, ctypes.c_int32), pt.shape[1], pt.shape[1],
        _ptr(cs, ctypes.c_int32), _ptr(cu, ctypes.c_int32), len(cs), float(scale),
        int(bool(causal)), int(window_left), _ptr(kd, ctypes.c_float), _ptr(vd, ctypes.c_float),
        _ptr(tk, ctypes.c_int32), 0 if tk is None else tk.shape[1],
        0 if tk is None else tk.shape[1],
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), int(num_threads))
    if rc < 0:
        raise ValueError(f"orc_attention_fp8 rejected its arguments ({rc})")
    return out.reshape(total_q, h_q, d_v), lse.reshape(total_q, h_q), rc


def set_kv_buffer(cache_bits, rows_bits, loc):
    """Writes new rows into a paged pool in place and returns the number of
    skipped (out-of-pool) slots.  cache_bits: uint16 [num_pages, P, H, D]
    (any element strides, D contiguous, writable); rows_bits: uint16
    [T, H, D] (D contiguous); loc: T slot ids."""
    c = cache_bits
    r = np.asarray(rows_bits)
    assert c.dtype == np.uint16 and r.dtype == np.uint16
    assert c.strides[3] == 2 and r.strides[2] == 2 and c.flags.writeable
    lc = np.ascontiguousarray(loc, dtype=np.int64)
    cs = _elem_strides(c)
    rs = _elem_strides(r)
    n = _lib().orc_set_kv_buffer(
        _ptr(r, ctypes.c_uint16), rs[0], rs[1], r.shape[0], r.shape[1], r.shape[2],
        _ptr(lc, ctypes.c_int64), c.ctypes.data_as(_u16p), cs[0], cs[1], cs[2],
        c.shape[0], c.shape[1])
    if n < 0:
        raise ValueError(f"orc_set_kv_buffer rejected its arguments ({n})")
    return n


def set_kv_buffer_fp8(cache_codes, rows_bits, loc, scale: float):
    """The KV write into a pool of e4m3 codes, in place: code of value /
    scale (binary32 quotient, nearest code, ties to even; see
    orc_set_kv_buffer_fp8).  cache_codes: uint8 [num_pages, P, H, D] (D
    contiguous, writable); rows_bits: uint16 bf16 bits [T, H, D]; loc: T slot
    ids.  Returns the number of skipped (out-of-pool) slots."""
    c = cache_codes
    r = np.asarray(rows_bits)
    assert c.dtype == np.uint8 and r.dtype == np.uint16
    assert c.strides[3] == 1 and r.strides[2] == 2 and c.flags.writeable
    lc = np.ascontiguousarray(loc, dtype=np.int64)
    cs = _elem_strides(c)
    rs = _elem_strides(r)
    n = _lib().orc_set_kv_buffer_fp8(
        _ptr(r, ctypes.c_uint16), rs[0], rs[1], r.shape[0], r.shape[1], r.shape[2],
        _ptr(lc, ctypes.c_int64), float(scale),
        c.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), cs[0], cs[1], cs[2],
        c.shape[0], c.shape[1])
    if n < 0:
        raise ValueError(f"orc_set_kv_buffer_fp8 rejected its arguments ({n})")
    return n


def local_virtual_batches(attn_chunk_size: int, page_size: int, cu_seqlens_q,
                          seq_lens, page_table, capacity: int | None = None,
                          bt_cols: int | None = None):
    """Local (chunked) attention split into virtual batches.

    Returns a dict with ``seqlens_q_local`` [cap], ``cu_seqlens_q_local``
    [cap + 1], ``seqlens_k_local`` [cap], ``block_table_local`` [cap,
    bt_cols] (int32), ``num_virtual``, ``chunk`` (the effective chunk),
    ``max_q_local``, ``max_k_local`` and ``bad`` (malformed requests).
    ``capacity`` defaults to the exact number of virtual batches and
    ``bt_cols`` to chunk / page_size."""
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    assert pt.ndim == 2 and pt.shape[0] == len(sl) and len(cu) == len(sl) + 1

    def run(cap, cols):
        outs = (np.zeros(cap, np.int32), np.zeros(cap + 1, np.int32),
                np.zeros(cap, np.int32), np.zeros((cap, cols), np.int32))
        info = np.zeros(4, np.int32)
        rc = _lib().orc_local_virtual_batches(
            int(attn_chunk_size), int(page_size), _ptr(cu, ctypes.c_int32),
            _ptr(sl, ctypes.c_int32), len(sl), _ptr(pt, ctypes.c_int32),
            pt.shape[1], pt.shape[1], cap, _ptr(outs[0], ctypes.c_int32),
            _ptr(outs[1], ctypes.c_int32), _ptr(outs[2], ctypes.c_int32),
            _ptr(outs[3], ctypes.c_int32), cols, cols, _ptr(info, ctypes.c_int32))
        if rc < 0:
            raise ValueError(f"orc_local_virtual_batches rejected its arguments ({rc})")
        return outs, info, rc

    if capacity is None or bt_cols is None:
        # a sizing pass: no rows, table width large enough for any chunk
        _, info, _ = run(0, max(attn_chunk_size // page_size, 1))
        if capacity is None:
            capacity = int(info[0])
        if bt_cols is None:
            bt_cols = int(info[1]) // page_size
    (sq, cuq, sk, bt), info, rc = run(int(capacity), int(bt_cols))
    return {"seqlens_q_local": sq, "cu_seqlens_q_local": cuq,
            "seqlens_k_local": sk, "block_table_local": bt,
            "num_virtual": int(info[0]), "chunk": int(info[1]),
            "max_q_local": int(info[2]), "max_k_local": int(info[3]),
            "bad": rc}


def attention(q_bits, k_bits, v_bits, page_table, cache_seqlens, cu_seqlens_q,
              scale: float, causal: bool = False, window_left: int = -1,
              topk=None, rows=None, d_v: int | None = None,
              num_threads: int = 0, attn_chunk: int = 0):
    """Paged attention in float64.

    ``attn_chunk`` > 0 restricts each query to the keys of its own
    attn_chunk-sized chunk (local chunked attention).

    q_bits: uint16 [total_q, H_q, D_qk]; k_bits / v_bits: uint16
    [num_pages, P, H_kv, D] views (any element strides; D contiguous).
    ``d_v`` defaults to v_bits.shape[3] (pass 512 with v_bits = k_bits for
    absorbed MLA).  ``rows``: optional int array [n, 2] of (token, head).
    Returns (out [n, d_v] float64, lse [n] float64, n_skipped); without
    ``rows`` out is [total_q, H_q, d_v] and lse [total_q, H_q].
    """
    q = np.asarray(q_bits)
    k = np.asarray(k_bits)
    v = np.asarray(v_bits)
    assert q.dtype == np.uint16 and k.dtype == np.uint16 and v.dtype == np.uint16
    assert q.strides[2] == 2 and k.strides[3] == 2 and v.strides[3] == 2
    total_q, h_q, d_qk = q.shape
    num_pages, page_size, h_kv, dk = k.shape
    assert dk >= d_qk
    if d_v is None:
        d_v = v.shape[3]
    qs = _elem_strides(q)
    ks = _elem_strides(k)
    vs = _elem_strides(v)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cs = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    tk = None if topk is None else np.ascontiguousarray(topk, dtype=np.int32)
    rw = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = total_q * h_q if rw is None else rw.shape[0]
    out = np.zeros((n, d_v), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = _lib().orc_attention(
        _ptr(q, ctypes.c_uint16), qs[0], qs[1], total_q, h_q, d_qk,
        _ptr(k, ctypes.c_uint16), ks[0], ks[1], ks[2],
        _ptr(v, ctypes.c_uint16), vs[0], vs[1], vs[2], d_v,
        h_kv, page_size, num_pages,
        _ptr(pt, ctypes.c_int32), pt.shape[1] if pt.ndim == 2 else 0,
        pt.shape[1] if pt.ndim == 2 else 0,
        _ptr(cs, ctypes.c_int32), _ptr(cu, ctypes.c_int32), len(cs),
        float(scale), int(bool(causal)), int(window_left), int(attn_chunk),
        _ptr(tk, ctypes.c_int32), 0 if tk is None else tk.shape[1],
        0 if tk is None else tk.shape[1],
        _ptr(rw, ctypes.c_int32), 0 if rw is None else rw.shape[0],
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
        int(num_threads))
    if rc < 0:
        raise ValueError(f"orc_attention rejected its arguments ({rc})")
    if rw is None:
        out = out.reshape(total_q, h_q, d_v)
        lse = lse.reshape(total_q, h_q)
    return out, lse, rc


def merge_state(v_a, lse_a, v_b, lse_b):
    """Two-state log-sum-exp merge in float64: v [..., D], lse [...]."""
    va = np.ascontiguousarray(v_a, dtype=np.float64)
    vb = np.ascontiguousarray(v_b, dtype=np.float64)
    la = np.ascontiguousarray(lse_a, dtype=np.float64)
    lb = np.ascontiguousarray(lse_b, dtype=np.float64)
    assert va.shape == vb.shape and la.shape == lb.shape == va.shape[:-1]
    d = va.shape[-1]
    n = la.size
    vo = np.zeros_like(va)
    lo = np.zeros_like(la)
    rc = _lib().orc_merge_state(
        _ptr(va, ctypes.c_double), _ptr(la, ctypes.c_double),
        _ptr(vb, ctypes.c_double), _ptr(lb, ctypes.c_double), n, d,
        _ptr(vo, ctypes.c_double), _ptr(lo, ctypes.c_double))
    if rc != 0:
        raise ValueError("orc_merge_state rejected its arguments")
    return vo, lo


def split_bounds(kv_len: int, num_splits: int, page_size: int):
    """Split-KV chunk boundaries used by the oracle: contiguous, page-aligned,
    near-equal chunks.  Chunk c covers [c*S, min((c+1)*S, kv_len)) with
    S = ceil(ceil(kv_len / num_splits) / page_size) * page_size; trailing
    chunks may be empty.  The pages leave the boundaries open; the merged
    result does not depend on them."""
    per = -(-kv_len // num_splits)
    size = -(-per // page_size) * page_size
    return [(min(c * size, kv_len), min((c + 1) * size, kv_len))
            for c in range(num_splits)]


def split_attention(q_bits, k_bits, v_bits, page_table, cache_seqlens,
                    cu_seqlens_q, scale: float, num_splits: int,
                    num_threads: int = 0):
    """Decode attention computed as ``num_splits`` partial states over
    disjoint key chunks, combined by repeated two-state merges (left to
    right).  Decode only (one query token per request, every key visible).
    Each chunk is an ordinary paged-attention call whose page table holds
    the chunk's pages and whose key window selects the chunk."""
    k = np.asarray(k_bits)
    page_size = k.shape[1]
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cs = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    assert np.all(np.diff(cu) == 1), "split_attention is decode-only"
    b_count = len(cs)
    acc_o = acc_l = None
    for c in range(num_splits):
        # Chunk c of request b: keys [lo_b, hi_b).  Present it as a request
        # whose page table starts at page lo_b / P and whose length is
        # hi_b - lo_b, so the chunk's keys are exactly its visible keys.
        cols = pt.shape[1]
        pt_c = np.zeros_like(pt)
        len_c = np.zeros(b_count, dtype=np.int32)
        for b in range(b_count):
            lo, hi = split_bounds(int(cs[b]), num_splits, page_size)[c]
            p0 = lo // page_size
            n_pages = cols - p0
            pt_c[b, :n_pages] = pt[b, p0:]
            len_c[b] = hi - lo
        o_c, l_c, _ = attention(q_bits, k_bits, v_bits, pt_c, len_c, cu, scale,
                                num_threads=num_threads)
        if acc_o is None:
            acc_o, acc_l = o_c, l_c
        else:
            acc_o, acc_l = merge_state(acc_o, acc_l, o_c, l_c)
    return acc_o, acc_l
