"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/pkv.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t)\s+(pkv_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    import paged_kv_cache_203_gb300 as pkv
    from paged_kv_cache_203_gb300 import _build

    if _build.sources_newer_than_library():
        _build.build_library()
    return pkv.load_library()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("pkv_attn_with_kvcache", "pkv_merge_state", "pkv_build_swa_page_table"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    import paged_kv_cache_203_gb300 as pkv

    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)
    assert set(declared_symbols()) == set(pkv.EXPORTED_SYMBOLS)


def test_version_without_gpu(lib):
    assert lib.pkv_version() == 1


def test_binding_rejects_bad_arguments_on_host(lib):
    """Argument validation runs on the host: malformed descriptors are
    refused with a status code before anything touches a device."""
    import torch

    import paged_kv_cache_203_gb300 as pkv

    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16)
    k = torch.zeros(8, 16, 2, 128, dtype=torch.bfloat16)
    pt = torch.zeros(2, 4, dtype=torch.int32)
    cs = torch.zeros(2, dtype=torch.int32)
    # H_q not a multiple of H_kv
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_workspace_size(q[:, :3], k, k, pt, cs, 1)
    assert e.value.code == -1
    # unsupported head dim
    q96 = torch.zeros(2, 4, 96, dtype=torch.bfloat16)
    k96 = torch.zeros(8, 16, 2, 96, dtype=torch.bfloat16)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_workspace_size(q96, k96, k96, pt, cs, 1)
    assert e.value.code == -2
    # wrong dtype of the page table
    with pytest.raises(pkv.PkvError):
        pkv.attn_workspace_size(q, k, k, pt.long(), cs, 1)
    # the fp8 KV write wants pools of e4m3 codes; a bf16 pool is refused
    # (and a bf16 write refuses scales) before any device work
    loc = torch.zeros(2, dtype=torch.int32)
    rows = torch.zeros(2, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(pkv.PkvError) as e:
        pkv.load_library().pkv_set_kv_buffer_fp8  # exported
        pkv._check("pkv_set_kv_buffer_fp8", pkv.load_library().pkv_set_kv_buffer_fp8(
            pkv._desc(loc), pkv._desc(rows), pkv._desc(None), pkv._desc(k), pkv._desc(None),
            None, None, None))
    assert e.value.code == -1
    with pytest.raises(ValueError):
        pkv.set_kv_buffer(k, None, loc, rows, k_scale=torch.ones(1))
    # the table-building attention call: its descriptors arrive in order (an
    # lse of the wrong shape, a missing or malformed token pool and a pool
    # index list of the wrong length are refused)
    rtt = torch.zeros(3, 64, dtype=torch.int32)
    rpi = torch.zeros(2, dtype=torch.int64)
    cu = torch.zeros(3, dtype=torch.int32)
    out = torch.zeros(2, 4, 128, dtype=torch.bfloat16)
    fused = pkv.load_library().pkv_strided_table_attn_with_kvcache

    def call(lse, r=rtt, ri=rpi, byref=True):
        d = pkv._desc
        return fused(d(q), d(k), d(k), d(pt), d(cs), d(cu), 1, 0.1, 0, -1, d(None), 0, d(out),
                     d(lse), ctypes.byref(d(r)) if byref else None,
                     ctypes.byref(d(ri)) if byref else None, None, 0, None)

    assert call(torch.zeros(3, 4)) == -1
    assert call(torch.zeros(2, 4), byref=False) == -1
    assert call(torch.zeros(2, 4), r=rtt.t()) == -1
    assert call(torch.zeros(2, 4), ri=rpi[:1]) == -1
    if not torch.cuda.is_available():  # (host tensors must not reach a device)
        assert call(torch.zeros(2, 4)) == -3  # well formed: stops at the missing device
    # workspace planning: no split -> no workspace; 4 splits -> partials
    assert pkv.attn_workspace_size(q, k, k, pt, cs, 1, num_splits=1) == 0
    ws = pkv.attn_workspace_size(q, k, k, pt, cs, 1, num_splits=4)
    assert ws >= 4 * 2 * 4 * 128 * 4 + 4 * 2 * 4 * 4
