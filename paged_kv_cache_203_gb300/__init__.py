"""paged_kv_cache_203_gb300 -- paged-KV attention on GB300 (sm_103a).

Thin Python binding over the C ABI of ``libpkv.so`` (declared in
``include/pkv.h``).  The functions here only marshal torch tensors into
``pkv_tensor`` descriptors, allocate outputs / workspace with torch and pass
torch's current stream; every step of the computation runs in the library's
CUDA kernels.  There is no CPU or eager fallback: if the library is missing
the first call raises.

Entry points (names as in the C ABI, without the ``pkv_`` prefix):

* ``attn_with_kvcache_fp8`` -- the same over an fp8 (e4m3) cache with
  per-(request, KV head) descales (fp8 ``kv_cache_dtype``).
* ``attn_with_kvcache`` -- paged attention of new query tokens
  (flashattention_backend.py ``flash_attn_with_kvcache`` calls; nsa_backend.py
  top-k sparse decode), with split-KV combined by the state merge.
* ``merge_state`` -- log-sum-exp merge of two attention states
  (``merge_state_v2`` / ``_merge_attn_outputs``).
* ``build_swa_page_table`` -- prefill-aware sliding-window page table
  (``_build_pa_page_table``).
* ``strided_page_table`` -- token-level to page-level table.
* ``topk_to_slots`` -- top-k logical positions to KV slots
  (``TopkTransformMethod.PAGED``).
* ``make_local_attention_virtual_batches`` -- local (chunked) attention cut
  into virtual requests (``make_local_attention_virtual_batches``), built on
  the device; ``local_attn_with_kvcache`` runs it and the attention.
* ``cascade_attn_with_kvcache`` -- shared-prefix attention as two calls and
  a state merge (``use_cascade_attn``).
* ``set_kv_buffer`` / ``set_mla_kv_buffer`` -- the new tokens' K/V stored
  into their pool slots (``set_kv_buffer`` / ``set_mla_kv_buffer`` before
  attention); ``append_attn_with_kvcache`` stores them and attends.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import build_library, lib_path

__all__ = [
    "check_bounded_wait",
    "cascade_attn_with_kvcache",
    "attn_with_kvcache",
    "attn_workspace_size",
    "attn_with_kvcache_noalloc",
    "attn_with_kvcache_fp8",
    "NOALLOC_SCRATCH_BYTES",
    "merge_state",
    "build_swa_page_table",
    "strided_page_table",
    "strided_table_attn_with_kvcache",
    "topk_to_slots",
    "make_local_attention_virtual_batches",
    "local_virtual_batch_capacity",
    "set_kv_buffer",
    "set_mla_kv_buffer",
    "append_attn_with_kvcache",
    "fused_append_attn_with_kvcache",
    "local_attn_with_kvcache",
    "get_error_flags",
    "clear_error_flags",
    "load_library",
    "build_library",
    "PkvError",
    "EXPORTED_SYMBOLS",
    "EFLAG_PAGE_OOB",
    "EFLAG_TOPK_OOB",
    "EFLAG_ROW_TOO_SHORT",
    "EFLAG_SRC_OOB",
    "EFLAG_TIMEOUT",
    "EFLAG_LAYOUT",
    "EFLAG_BAD_LENGTHS",
    "EFLAG_CAPACITY",
]

# dtype codes and status codes of include/pkv.h
_BF16, _F32, _I32, _I64 = 1, 2, 3, 4
_STATUS = {0: "PKV_OK", -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_UNSUPPORTED",
           -3: "PKV_ERR_CUDA", -4: "PKV_ERR_WORKSPACE"}
EFLAG_PAGE_OOB, EFLAG_TOPK_OOB, EFLAG_ROW_TOO_SHORT, EFLAG_SRC_OOB = 1, 2, 4, 8
EFLAG_TIMEOUT = 16
EFLAG_LAYOUT = 32
EFLAG_BAD_LENGTHS = 64
EFLAG_CAPACITY = 128

EXPORTED_SYMBOLS = (
    "pkv_attn_with_kvcache",
    "pkv_attn_workspace_size",
    "pkv_merge_state",
    "pkv_build_swa_page_table",
    "pkv_strided_page_table",
    "pkv_topk_to_slots",
    "pkv_get_error_flags",
    "pkv_clear_error_flags",
    "pkv_version",
    "pkv_attn_with_kvcache_noalloc",
    "pkv_make_local_attention_virtual_batches",
    "pkv_set_kv_buffer",
    "pkv_attn_with_kvcache_fp8",
    "pkv_set_kv_buffer_fp8",
    "pkv_append_attn_with_kvcache",
    "pkv_check_bounded_wait",
    "pkv_strided_table_attn_with_kvcache",
)

_FP8 = 5
_DTYPES = {torch.bfloat16: _BF16, torch.float32: _F32, torch.int32: _I32,
           torch.int64: _I64, torch.float8_e4m3fn: _FP8}


class PkvError(RuntimeError):
    """A libpkv entry point returned a negative status."""

    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {_STATUS.get(code, code)}")
        self.code = code


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * 4),
                ("stride", ctypes.c_int64 * 4)]


_ABSENT = _Tensor()
_LIB = None


def load_library(path: str | None = None):
    """Load libpkv.so (built by ``build_library()`` / ``__graft_entry__.build``).
    Raises if it is missing: there is no fallback path."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"libpkv.so not found at {path}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    T = _Tensor
    c_int, c_float, c_void_p, c_size_t = (ctypes.c_int, ctypes.c_float,
                                          ctypes.c_void_p, ctypes.c_size_t)
    lib.pkv_attn_with_kvcache.argtypes = [T, T, T, T, T, T, c_int, c_float, c_int,
                                          c_int, T, c_int, T, T, c_void_p, c_size_t,
                                          c_void_p]
    lib.pkv_attn_workspace_size.argtypes = [T, T, T, T, T, c_int, T, c_int,
                                            ctypes.POINTER(c_size_t)]
    lib.pkv_attn_with_kvcache_noalloc.argtypes = [T, T, T, T, T, T, c_int, c_float,
                                                  c_int, c_int, T, c_int, T, T,
                                                  c_void_p]
    lib.pkv_merge_state.argtypes = [T, T, T, T, T, T, c_void_p]
    lib.pkv_build_swa_page_table.argtypes = [T, T, T, T, c_int, T, T, c_void_p]
    lib.pkv_strided_page_table.argtypes = [T, T, c_int, T, c_void_p]
    lib.pkv_topk_to_slots.argtypes = [T, T, T, T, c_int, T, c_void_p]
    lib.pkv_set_kv_buffer.argtypes = [T, T, T, T, T, c_void_p]
    lib.pkv_set_kv_buffer_fp8.argtypes = [T, T, T, T, T, c_void_p, c_void_p, c_void_p]
    lib.pkv_attn_with_kvcache_fp8.argtypes = [T, T, T, T, T, T, c_int, c_float, c_int, c_int,
                                              T, c_void_p, c_void_p, c_int, T, T, c_void_p,
                                              c_size_t, c_void_p]
    TP = ctypes.POINTER(T)
    lib.pkv_append_attn_with_kvcache.argtypes = [T, T, T, T, T, T, c_int, c_float, c_int,
                                                 c_int, TP, TP, TP, c_int, T, T, c_void_p,
                                                 c_size_t, c_void_p]
    lib.pkv_strided_table_attn_with_kvcache.argtypes = [T, T, T, T, T, T, c_int, c_float,
                                                        c_int, c_int, T, c_int, T, T, TP, TP,
                                                        c_void_p, c_size_t, c_void_p]
    lib.pkv_make_local_attention_virtual_batches.argtypes = [
        c_int, c_int, T, T, T, T, T, T, T, T, c_void_p]
    lib.pkv_get_error_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.pkv_clear_error_flags.argtypes = []
    lib.pkv_version.argtypes = []
    lib.pkv_check_bounded_wait.argtypes = [c_void_p]
    for name in EXPORTED_SYMBOLS:
        getattr(lib, name).restype = ctypes.c_int
    _LIB = lib
    return lib


def _desc(t: torch.Tensor | None) -> _Tensor:
    if t is None:
        return _ABSENT
    if t.dim() > 4:
        raise ValueError("pkv tensors have at most 4 dimensions")
    d = _Tensor()
    d.data = t.data_ptr() if t.numel() > 0 else (t.data_ptr() or 16)
    d.dtype = _DTYPES.get(t.dtype, 0)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _check(fn: str, rc: int):
    if rc != 0:
        raise PkvError(fn, rc)


def attn_workspace_size(q, k_cache, v_cache, page_table, cache_seqlens,
                        max_seqlen_q: int, topk_indices=None,
                        num_splits: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_attn_workspace_size", load_library().pkv_attn_workspace_size(
        _desc(q), _desc(k_cache), _desc(v_cache), _desc(page_table),
        _desc(cache_seqlens), int(max_seqlen_q), _desc(topk_indices),
        int(num_splits), ctypes.byref(n)))
    return n.value


def attn_with_kvcache(q, k_cache, v_cache, page_table, cache_seqlens,
                      cu_seqlens_q, max_seqlen_q: int, softmax_scale: float,
                      causal: bool = False, window_left: int = -1,
                      topk_indices=None, num_splits: int = 0, out=None,
                      lse=None, return_softmax_lse: bool = False,
                      workspace=None):
    """Paged attention (see include/pkv.h, pkv_attn_with_kvcache).

    Returns ``out`` or ``(out, lse)`` when ``return_softmax_lse``; ``lse`` is
    [total_q, H_q] fp32 (natural log)."""
    lib = load_library()
    if out is None:
        out = torch.empty(q.shape[0], q.shape[1], v_cache.shape[-1],
                          dtype=torch.bfloat16, device=q.device)
    if return_softmax_lse and lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32,
                          device=q.device)
    # each descriptor is built once and serves both calls (marshalling is most
    # of the binding's host time)
    dq, dk, dv, dpt, dcs, dtk = (_desc(q), _desc(k_cache), _desc(v_cache), _desc(page_table),
                                 _desc(cache_seqlens), _desc(topk_indices))
    n = ctypes.c_size_t(0)
    _check("pkv_attn_workspace_size", lib.pkv_attn_workspace_size(
        dq, dk, dv, dpt, dcs, int(max_seqlen_q), dtk, int(num_splits), ctypes.byref(n)))
    ws_bytes = n.value
    if ws_bytes > 0 and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if ws_bytes > 0 else None
    _check("pkv_attn_with_kvcache", lib.pkv_attn_with_kvcache(
        dq, dk, dv, dpt, dcs, _desc(cu_seqlens_q), int(max_seqlen_q),
        float(softmax_scale), int(bool(causal)), int(window_left),
        dtk, int(num_splits), _desc(out), _desc(lse), ws_ptr,
        ws_bytes, _stream(q)))
    return (out, lse) if return_softmax_lse else out


def _descale_ptr(t, cache_seqlens, k_cache):
    """Device pointer of a [B, H_kv] fp32 descale tensor (None -> NULL)."""
    if t is None:
        return None
    want = (cache_seqlens.shape[0], k_cache.shape[2])
    if (t.dtype != torch.float32 or tuple(t.shape) != want or not t.is_contiguous()
            or t.device != k_cache.device):
        raise ValueError(f"descale must be a contiguous float32 tensor of shape {want} "
                         "on the cache's device")
    return t.data_ptr()


def attn_with_kvcache_fp8(q, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                          max_seqlen_q: int, softmax_scale: float, causal: bool = False,
                          window_left: int = -1, k_descale=None, v_descale=None,
                          out=None, lse=None, return_softmax_lse: bool = False,
                          workspace=None, topk_indices=None, num_splits: int = 0):
    """Paged attention over an fp8 (e4m3) cache (include/pkv.h,
    pkv_attn_with_kvcache_fp8): ``k_cache`` / ``v_cache`` are
    torch.float8_e4m3fn tensors, ``k_descale`` / ``v_descale`` optional fp32
    [B, H_kv]; q (bf16) is rounded to e4m3 inside the kernel.  Absorbed MLA
    (576 / 512 dims, one latent head, ``v_cache`` the first 512 columns of
    ``k_cache``) takes ``topk_indices`` as pkv_attn_with_kvcache does."""
    lib = load_library()
    if out is None:
        out = torch.empty(q.shape[0], q.shape[1], v_cache.shape[-1], dtype=torch.bfloat16,
                          device=q.device)
    if return_softmax_lse and lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    dq, dk, dv, dpt, dcs, dtk = (_desc(q), _desc(k_cache), _desc(v_cache), _desc(page_table),
                                 _desc(cache_seqlens), _desc(topk_indices))
    n = ctypes.c_size_t(0)
    _check("pkv_attn_workspace_size", lib.pkv_attn_workspace_size(
        dq, dk, dv, dpt, dcs, int(max_seqlen_q), dtk, int(num_splits), ctypes.byref(n)))
    ws_bytes = n.value
    if ws_bytes > 0 and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if ws_bytes > 0 else None
    _check("pkv_attn_with_kvcache_fp8", lib.pkv_attn_with_kvcache_fp8(
        dq, dk, dv, dpt, dcs,
        _desc(cu_seqlens_q), int(max_seqlen_q), float(softmax_scale), int(bool(causal)),
        int(window_left), dtk,
        _descale_ptr(k_descale, cache_seqlens, k_cache),
        _descale_ptr(v_descale, cache_seqlens, k_cache), int(num_splits), _desc(out),
        _desc(lse), ws_ptr, ws_bytes, _stream(q)))
    return (out, lse) if return_softmax_lse else out


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # PKV_NOALLOC_SCRATCH_BYTES


def attn_with_kvcache_noalloc(q, k_cache, v_cache, page_table, cache_seqlens,
                              cu_seqlens_q, max_seqlen_q: int,
                              softmax_scale: float, out, lse=None,
                              causal: bool = False, window_left: int = -1,
                              topk_indices=None, num_splits: int = 0):
    """pkv_attn_with_kvcache_noalloc: the same attention for callers that
    cannot allocate device memory.  The caller passes every buffer,
    including ``out`` (and ``lse`` if wanted); the split scratch is the
    library's own fixed per-device array, so this call allocates nothing.
    Calls that would need more than NOALLOC_SCRATCH_BYTES of scratch raise
    PkvError (PKV_ERR_WORKSPACE); calls that overlap on the GPU race on the
    shared array."""
    _check("pkv_attn_with_kvcache_noalloc", load_library().pkv_attn_with_kvcache_noalloc(
        _desc(q), _desc(k_cache), _desc(v_cache), _desc(page_table),
        _desc(cache_seqlens), _desc(cu_seqlens_q), int(max_seqlen_q),
        float(softmax_scale), int(bool(causal)), int(window_left),
        _desc(topk_indices), int(num_splits), _desc(out), _desc(lse), _stream(q)))
    return out


def merge_state(v_a, lse_a, v_b, lse_b, v_out=None, lse_out=None):
    """Log-sum-exp merge of two states; returns (v_out, lse_out)."""
    lib = load_library()
    if v_out is None:
        v_out = torch.empty_like(v_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    _check("pkv_merge_state", lib.pkv_merge_state(
        _desc(v_a), _desc(lse_a), _desc(v_b), _desc(lse_b), _desc(v_out),
        _desc(lse_out), _stream(v_a)))
    return v_out, lse_out


def cascade_attn_with_kvcache(q, k_cache, v_cache, prefix_page_table, prefix_seqlens,
                              suffix_page_table, suffix_seqlens, cu_seqlens_q,
                              max_seqlen_q: int, softmax_scale: float, causal: bool = False,
                              num_splits: int = 0, out=None, lse=None,
                              return_softmax_lse: bool = False):
    """Cascade attention over a key range held in two parts, as the
    FlashAttention backend runs it (flashattention_backend.py, `forward_decode`
    with `use_cascade_attn`): attention over the committed prefix with no
    causal mask, attention over the suffix with its own page table and
    lengths (causal within it when asked), and the log-sum-exp merge of the
    two states (`merge_state_v2`).  Every step is a call into libpkv; the
    partial outputs are bf16, as on that path.

    prefix_page_table / prefix_seqlens: the part every query sees in full
    (keys [0, prefix_len) of each request); suffix_page_table /
    suffix_seqlens: the remaining keys, positioned after the prefix (the
    queries sit at the end of the suffix, bottom-right).  No window."""
    o1, l1 = attn_with_kvcache(q, k_cache, v_cache, prefix_page_table, prefix_seqlens,
                               cu_seqlens_q, max_seqlen_q, softmax_scale, causal=False,
                               num_splits=num_splits, return_softmax_lse=True)
    o2, l2 = attn_with_kvcache(q, k_cache, v_cache, suffix_page_table, suffix_seqlens,
                               cu_seqlens_q, max_seqlen_q, softmax_scale, causal=causal,
                               num_splits=num_splits, return_softmax_lse=True)
    out, lse = merge_state(o1, l1, o2, l2, out, lse)
    return (out, lse) if return_softmax_lse else out


def build_swa_page_table(req_to_token, req_pool_indices, seq_lens,
                         prefill_lens, window: int, dst_page_table,
                         dst_kv_lens):
    """Prefill-aware SWA page table, written in place; returns the two
    destination tensors."""
    _check("pkv_build_swa_page_table", load_library().pkv_build_swa_page_table(
        _desc(req_to_token), _desc(req_pool_indices), _desc(seq_lens),
        _desc(prefill_lens), int(window), _desc(dst_page_table),
        _desc(dst_kv_lens), _stream(req_to_token)))
    return dst_page_table, dst_kv_lens


def strided_page_table(req_to_token, req_pool_indices, page_size: int,
                       n_cols: int, out=None):
    if out is None:
        out = torch.empty(req_pool_indices.shape[0], n_cols, dtype=torch.int32,
                          device=req_to_token.device)
    _check("pkv_strided_page_table", load_library().pkv_strided_page_table(
        _desc(req_to_token), _desc(req_pool_indices), int(page_size),
        _desc(out), _stream(req_to_token)))
    return out


def strided_table_attn_with_kvcache(req_to_token, req_pool_indices, page_table, q, k_cache,
                                    v_cache, cache_seqlens, cu_seqlens_q, max_seqlen_q: int,
                                    softmax_scale: float, causal: bool = False,
                                    window_left: int = -1, topk_indices=None,
                                    num_splits: int = 0, out=None, lse=None,
                                    return_softmax_lse: bool = False, workspace=None):
    """The strided page table written into ``page_table`` ([B, n_cols] int32)
    and the attention over it, in one launch where the short decode kernels
    serve the call (see include/pkv.h, pkv_strided_table_attn_with_kvcache).

    Returns ``out`` or ``(out, lse)`` when ``return_softmax_lse``."""
    lib = load_library()
    if out is None:
        out = torch.empty(q.shape[0], q.shape[1], v_cache.shape[-1],
                          dtype=torch.bfloat16, device=q.device)
    if return_softmax_lse and lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32,
                          device=q.device)
    dq, dk, dv, dpt, dcs, dtk = (_desc(q), _desc(k_cache), _desc(v_cache), _desc(page_table),
                                 _desc(cache_seqlens), _desc(topk_indices))
    n = ctypes.c_size_t(0)
    _check("pkv_attn_workspace_size", lib.pkv_attn_workspace_size(
        dq, dk, dv, dpt, dcs, int(max_seqlen_q), dtk, int(num_splits), ctypes.byref(n)))
    ws_bytes = n.value
    if ws_bytes > 0 and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if ws_bytes > 0 else None
    _check("pkv_strided_table_attn_with_kvcache", lib.pkv_strided_table_attn_with_kvcache(
        dq, dk, dv, dpt, dcs, _desc(cu_seqlens_q), int(max_seqlen_q), float(softmax_scale),
        int(bool(causal)), int(window_left), dtk, int(num_splits), _desc(out), _desc(lse),
        ctypes.byref(_desc(req_to_token)), ctypes.byref(_desc(req_pool_indices)), ws_ptr,
        ws_bytes, _stream(q)))
    return (out, lse) if return_softmax_lse else out


def topk_to_slots(topk, cu_seqlens_q, page_table, cache_seqlens,
                  page_size: int, out=None):
    if out is None:
        out = torch.empty_like(topk)
    _check("pkv_topk_to_slots", load_library().pkv_topk_to_slots(
        _desc(topk), _desc(cu_seqlens_q), _desc(page_table),
        _desc(cache_seqlens), int(page_size), _desc(out), _stream(topk)))
    return out


def _scale_ptr(t, k_cache):
    """Device pointer of a one-element fp32 scale tensor (None -> NULL)."""
    if t is None:
        return None
    if t.dtype != torch.float32 or t.numel() != 1 or t.device != k_cache.device:
        raise ValueError("a scale must be a one-element float32 tensor on the cache's device")
    return t.data_ptr()


def set_kv_buffer(k_cache, v_cache, loc, k, v=None, k_scale=None, v_scale=None):
    """Stores new K (and V) rows into their pool slots (include/pkv.h,
    pkv_set_kv_buffer): k_cache[loc // P, loc % P] = k, same for v.  For
    pools of fp8 codes (torch.float8_e4m3fn) each value is stored as the
    e4m3 code of value / scale (pkv_set_kv_buffer_fp8); ``k_scale`` /
    ``v_scale`` are one-element float32 device tensors (None: 1)."""
    lib = load_library()
    vc = None if v is None else v_cache
    if k_cache.dtype == torch.float8_e4m3fn:
        _check("pkv_set_kv_buffer_fp8", lib.pkv_set_kv_buffer_fp8(
            _desc(loc), _desc(k), _desc(v), _desc(k_cache), _desc(vc),
            _scale_ptr(k_scale, k_cache), _scale_ptr(v_scale, k_cache), _stream(k)))
    else:
        if k_scale is not None or v_scale is not None:
            raise ValueError("scales apply to pools of fp8 codes only")
        _check("pkv_set_kv_buffer", lib.pkv_set_kv_buffer(
            _desc(loc), _desc(k), _desc(v), _desc(k_cache), _desc(vc), _stream(k)))
    return k_cache, v_cache


def set_mla_kv_buffer(kv_cache, loc, k_nope, k_rope):
    """MLA latent rows: columns [0, Dn) of the [pages, P, 1, Dn + Dr] pool get
    k_nope [T, 1, Dn], columns [Dn, Dn + Dr) get k_rope [T, 1, Dr]."""
    dn = k_nope.shape[-1]
    set_kv_buffer(kv_cache[..., :dn], kv_cache[..., dn:], loc, k_nope, k_rope)
    return kv_cache


def append_attn_with_kvcache(q, k, v, cache_loc, k_cache, v_cache, page_table,
                             cache_seqlens, cu_seqlens_q, max_seqlen_q: int,
                             softmax_scale: float, k_scale=None, v_scale=None,
                             **attn_kwargs):
    """The backend's forward order (flashattention_backend.py
    `forward_extend` / `forward_decode`): the new tokens' K/V go to their
    slots ``cache_loc`` first, then paged attention reads the cache that now
    holds them.  Both launches are on the current stream, so attention sees
    the stored rows; ``attn_kwargs`` are those of ``attn_with_kvcache``.
    With pools of fp8 codes the rows are stored as codes of value / scale and
    the attention reads them back with the scales as per-(request, KV head)
    descales (the backend's ``k_scale.expand(batch, num_kv_heads)``)."""
    set_kv_buffer(k_cache, v_cache, cache_loc, k, v, k_scale=k_scale, v_scale=v_scale)
    if k_cache.dtype != torch.float8_e4m3fn:
        return attn_with_kvcache(q, k_cache, v_cache, page_table, cache_seqlens,
                                 cu_seqlens_q, max_seqlen_q, softmax_scale, **attn_kwargs)
    shape = (cache_seqlens.shape[0], k_cache.shape[2])
    kd = None if k_scale is None else k_scale.reshape(1, 1).expand(shape).contiguous()
    vd = None if v_scale is None else v_scale.reshape(1, 1).expand(shape).contiguous()
    return attn_with_kvcache_fp8(q, k_cache, v_cache, page_table, cache_seqlens, cu_seqlens_q,
                                 max_seqlen_q, softmax_scale, k_descale=kd, v_descale=vd,
                                 **attn_kwargs)


def fused_append_attn_with_kvcache(q, k, v, cache_loc, k_cache, v_cache, page_table,
                                   cache_seqlens, cu_seqlens_q, max_seqlen_q: int,
                                   softmax_scale: float, causal: bool = False,
                                   window_left: int = -1, num_splits: int = 0, out=None,
                                   lse=None, return_softmax_lse: bool = False,
                                   workspace=None):
    """The KV write and the attention in one launch (include/pkv.h,
    pkv_append_attn_with_kvcache): the same result as
    ``append_attn_with_kvcache`` (bf16 caches, the all-heads decode shapes);
    ``k`` / ``v`` [total_q, H_kv, D] are the new tokens' rows and
    ``cache_loc`` their slots."""
    lib = load_library()
    if out is None:
        out = torch.empty(q.shape[0], q.shape[1], v_cache.shape[-1], dtype=torch.bfloat16,
                          device=q.device)
    if return_softmax_lse and lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    ws_bytes = attn_workspace_size(q, k_cache, v_cache, page_table, cache_seqlens,
                                   max_seqlen_q, None, num_splits)
    if ws_bytes > 0 and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if ws_bytes > 0 else None
    _check("pkv_append_attn_with_kvcache", lib.pkv_append_attn_with_kvcache(
        _desc(q), _desc(k_cache), _desc(v_cache), _desc(page_table), _desc(cache_seqlens),
        _desc(cu_seqlens_q), int(max_seqlen_q), float(softmax_scale), int(bool(causal)),
        int(window_left), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)),
        ctypes.byref(_desc(cache_loc)), int(num_splits),
        _desc(out), _desc(lse), ws_ptr, ws_bytes, _stream(q)))
    return (out, lse) if return_softmax_lse else out


def local_virtual_batch_capacity(batch: int, total_q: int, max_seqlen_q: int,
                                 page_size: int) -> int:
    """Rows that always hold the virtual requests of a batch: each request
    makes at most one per new token, and at most 1 + ceil((q - 1) / C) with
    the effective chunk C >= page_size."""
    per_request = 1 + max(0, -(-(int(max_seqlen_q) - 1) // int(page_size)))
    return max(0, min(int(total_q), int(batch) * per_request))


def make_local_attention_virtual_batches(attn_chunk_size: int, page_size: int,
                                         cu_seqlens_q, seq_lens, page_table,
                                         capacity: int, out=None):
    """Local (chunked) attention as virtual requests, built on the device
    (include/pkv.h, pkv_make_local_attention_virtual_batches).

    Returns ``(seqlens_q_local [V], cu_seqlens_q_local [V + 1],
    seqlens_k_local [V], block_table_local [V, Wl], info [4])`` int32 device
    tensors, V = ``capacity``, Wl = max(attn_chunk_size // page_size, 1);
    ``info`` = (virtual requests, effective chunk, max local q, max local k).
    ``out`` may pass those five tensors to be written in place."""
    dev = cu_seqlens_q.device
    cap = int(capacity)
    if out is None:
        wl = max(int(attn_chunk_size) // int(page_size), 1)
        out = (torch.empty(cap, dtype=torch.int32, device=dev),
               torch.empty(cap + 1, dtype=torch.int32, device=dev),
               torch.empty(cap, dtype=torch.int32, device=dev),
               torch.empty(cap, wl, dtype=torch.int32, device=dev),
               torch.empty(4, dtype=torch.int32, device=dev))
    sq, cuq, sk, bt, info = out
    _check("pkv_make_local_attention_virtual_batches",
           load_library().pkv_make_local_attention_virtual_batches(
               int(attn_chunk_size), int(page_size), _desc(cu_seqlens_q), _desc(seq_lens),
               _desc(page_table), _desc(sq), _desc(cuq), _desc(sk), _desc(bt), _desc(info),
               _stream(cu_seqlens_q)))
    return out


def local_attn_with_kvcache(q, k_cache, v_cache, page_table, cache_seqlens,
                            cu_seqlens_q, max_seqlen_q: int, attn_chunk_size: int,
                            softmax_scale: float, num_splits: int = 0, out=None,
                            lse=None, return_softmax_lse: bool = False):
    """Local (chunked) causal attention, as the FlashAttention backend runs
    it (flashattention_backend.py, `use_local_attn`): the batch is cut into
    virtual requests on the device, then one causal attention call runs over
    them (their query offsets, key lengths and local page table).  The
    virtual requests keep the query rows in order, so ``out`` / ``lse`` are
    indexed like ``q``.  No host synchronisation."""
    page_size = k_cache.shape[1]
    cap = local_virtual_batch_capacity(cache_seqlens.shape[0], q.shape[0], max_seqlen_q,
                                       page_size)
    _, cu_local, k_local, bt_local, _ = make_local_attention_virtual_batches(
        attn_chunk_size, page_size, cu_seqlens_q, cache_seqlens, page_table, cap)
    # a virtual request holds at most one effective chunk of new tokens, and
    # the effective chunk is at most max(whole pages of attn_chunk_size, 1 page)
    chunk_bound = max((int(attn_chunk_size) // page_size) * page_size, page_size)
    max_q_local = min(int(max_seqlen_q), chunk_bound)
    return attn_with_kvcache(q, k_cache, v_cache, bt_local, k_local, cu_local, max_q_local,
                             softmax_scale, causal=True, num_splits=num_splits, out=out,
                             lse=lse, return_softmax_lse=return_softmax_lse)


def get_error_flags() -> int:
    v = ctypes.c_uint32(0)
    _check("pkv_get_error_flags", load_library().pkv_get_error_flags(ctypes.byref(v)))
    return v.value


def clear_error_flags() -> None:
    _check("pkv_clear_error_flags", load_library().pkv_clear_error_flags())


def check_bounded_wait(stream=None) -> None:
    """pkv_check_bounded_wait: one CTA waits on a barrier that nothing
    arrives on through the library's bounded waits; they expire after about
    a second and set EFLAG_TIMEOUT (asynchronous; synchronise, then read
    get_error_flags)."""
    lib = load_library()
    s = torch.cuda.current_stream() if stream is None else stream
    _check("pkv_check_bounded_wait", lib.pkv_check_bounded_wait(ctypes.c_void_p(s.cuda_stream)))
