"""The C-ABI library loads, exports every symbol include/mla.h declares, and
rejects bad arguments on the host (no GPU needed)."""
import ctypes
import os
import re

import pytest

from mla_family_attention_gb300 import _lib
from mla_family_attention_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("mla_prefill", "mla_decode", "dsa_index_topk", "dsa_sparse_decode"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"
    assert set(_lib.SIGNATURES) == set(names)


def test_workspace_sizes(lib):
    ws = lib.mla_workspace_size
    assert ws(_lib.OP_PREFILL, 1, 96, 128, 0) == 0
    d = ws(_lib.OP_DECODE, 32, 96, 8192, 0)
    assert d > 0 and d % 256 == 0
    # 8 chunks of 1024 positions per (b,h): acc[128] + (max, sum) floats each
    assert d >= 32 * 96 * 8 * 130 * 4
    assert ws(_lib.OP_DECODE, 0, 96, 8192, 0) == 0
    assert ws(_lib.OP_SPARSE_DECODE, 8, 96, 0, 4096) == 0
    assert ws(_lib.OP_SPARSE_DECODE, 8, 96, 0, 2048) > 0
    assert ws(99, 1, 1, 1, 1) == 0


def _err(lib):
    return lib.mla_last_error().decode()


def test_host_validation_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    good = P(1 << 20)
    st = lib.mla_decode(None, good, good, good, 1, 1, 8, None, good, 0.1, None, 0, None)
    assert st == _lib.MLA_ERR_INVALID_ARG and "null" in _err(lib)
    st = lib.mla_decode(P((1 << 20) + 2), good, good, good, 1, 1, 8, None, good, 0.1, None, 0,
                        None)
    assert st == _lib.MLA_ERR_INVALID_ARG and "aligned" in _err(lib)
    st = lib.mla_decode(good, good, good, good, 0, 1, 8, None, good, 0.1, None, 0, None)
    assert st == _lib.MLA_ERR_INVALID_ARG
    st = lib.mla_decode(good, good, good, good, 2, 4, 100, None, good, 0.1, None, 0, None)
    assert st == _lib.MLA_ERR_WORKSPACE
    need = lib.mla_workspace_size(_lib.OP_DECODE, 2, 4, 100, 0)
    st = lib.mla_decode(good, good, good, good, 2, 4, 100, None, good, 0.1, good, need - 256, None)
    assert st == _lib.MLA_ERR_WORKSPACE and "too small" in _err(lib)
    st = lib.mla_decode(good, good, good, good, 2, 4, 100, None, good, -1.0, good, need, None)
    assert st == _lib.MLA_ERR_INVALID_ARG
    st = lib.dsa_sparse_decode(good, good, good, good, good, 4096, 1, 1, None, good, 0.1, good,
                               1 << 30, None)
    assert st == _lib.MLA_ERR_UNSUPPORTED


def test_debug_knobs(lib):
    assert lib.mla_debug_set(12345, 0) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_debug_set(_lib.DEBUG_WAIT_LIMIT_NS, 0) == _lib.MLA_OK
    assert lib.mla_debug_set(_lib.DEBUG_STALL_STAGE, -1) == _lib.MLA_OK
    for v in (1, 2, 0):
        assert lib.mla_debug_set(_lib.DEBUG_PREFILL_CTAS, v) == _lib.MLA_OK
    assert lib.mla_debug_set(_lib.DEBUG_PREFILL_CTAS, 3) == _lib.MLA_ERR_INVALID_ARG


def test_binding_raises_when_library_missing(tmp_path):
    with pytest.raises(RuntimeError):
        _lib.load(str(tmp_path / "nope.so"))


def test_host_validation_of_the_other_entry_points(lib):
    """Each entry point rejects malformed calls on the host, before any CUDA
    call, with the documented status and a message naming the problem."""
    P = ctypes.c_void_p
    g = P(1 << 20)                       # a 16-byte aligned stand-in pointer
    bad = P((1 << 20) + 2)               # misaligned
    E = _lib

    # prefill: Tq > Tk, null pointer, misaligned pointer, bad scale
    assert lib.mla_prefill(g, g, g, None, g, 1, 1, 8, 4, 0.1, None, 0, None) == E.MLA_ERR_INVALID_ARG
    assert lib.mla_prefill(None, g, g, None, g, 1, 1, 8, 8, 0.1, None, 0, None) == E.MLA_ERR_INVALID_ARG
    assert "null" in _err(lib)
    assert lib.mla_prefill(bad, g, g, None, g, 1, 1, 8, 8, 0.1, None, 0, None) == E.MLA_ERR_INVALID_ARG
    assert "aligned" in _err(lib)
    assert lib.mla_prefill(g, g, g, None, g, 1, 1, 8, 8, 0.0, None, 0, None) == E.MLA_ERR_INVALID_ARG
    assert "scale" in _err(lib)

    # cache append: the uniform start must leave room for the new rows
    assert lib.mla_cache_append(g, g, g, g, None, 10, 1, 1, 8, 16, None) == E.MLA_ERR_INVALID_ARG
    assert "kv_capacity" in _err(lib)
    # chunked prefill: P + Tq past the capacity
    assert lib.mla_prefill_chunk(g, g, g, g, g, None, g, 1, 1, 8, 10, 16, 0.1, None, 0,
                                 None) == E.MLA_ERR_INVALID_ARG

    # DSA indexer: 32 index heads only, topk at most 2048, B >= 1
    assert lib.dsa_index_topk(g, g, g, g, 1, 16, 100, 100, 64, g, None, g, 1 << 20,
                              None) == E.MLA_ERR_UNSUPPORTED
    assert lib.dsa_index_topk(g, g, g, g, 1, 32, 100, 100, 4096, g, None, g, 1 << 20,
                              None) == E.MLA_ERR_UNSUPPORTED
    assert lib.dsa_index_topk(g, g, g, g, 0, 32, 100, 100, 64, g, None, g, 1 << 20,
                              None) == E.MLA_ERR_INVALID_ARG
    assert lib.dsa_index_topk_fp8(g, g, g, g, g, 1, 16, 100, 100, 64, g, None, g, 1 << 20,
                                  None) == E.MLA_ERR_UNSUPPORTED
    assert lib.dsa_prefill_index_topk(g, g, g, 8, 4, 32, 64, g, None, g, 1 << 20,
                                      None) == E.MLA_ERR_INVALID_ARG

    # latent decode: head counts that are multiples of 16 up to 96
    assert lib.mla_decode_latent(g, g, g, 100, 1, 40, 100, g, g, None, g, 0.1, g, 1 << 20,
                                 None) == E.MLA_ERR_UNSUPPORTED
    assert lib.mla_decode_latent(g, g, g, 100, 1, 96, 100, g, None, None, g, 0.1, g, 1 << 20,
                                 None) == E.MLA_ERR_INVALID_ARG
    assert lib.mla_sparse_prefill_latent(g, g, g, 8, 4, 64, 96, g, g, None, g, 0.1, g, 1 << 20,
                                         None) == E.MLA_ERR_INVALID_ARG

    # quantisers: negative counts
    assert lib.dsa_quantize_index_keys(g, g, g, -1, None) == E.MLA_ERR_INVALID_ARG
    assert lib.mla_quantize_latent_cache(g, g, -1, None) == E.MLA_ERR_INVALID_ARG
