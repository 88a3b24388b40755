"""mla_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).

Each of two calls in a row with different shapes (the second runs on scratch
that still holds the first call's contents) is checked against the fp64
oracle at the parity tolerance, and bit for bit against mla_decode, which
runs the same kernels on a caller workspace: leftover scratch reaching the
output would show as a difference even where it is below the tolerance.
It must also reject a problem whose scratch need exceeds the built-in array.
Kept in a file that pytest collects last.
"""
import ctypes

import pytest
import torch

import mla_inputs as mi
import oracle
import mla_family_attention_gb300 as mla
from mla_family_attention_gb300 import _lib
from parity import assert_close

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def noalloc_decode(dec, max_seqlen):
    lib = _lib.load()
    B, H = dec.q.shape[0], dec.q.shape[1]
    out = torch.empty((B, H * 128), dtype=torch.bfloat16, device=dec.q.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.mla_decode_noalloc(_p(dec.q), _p(dec.k), _p(dec.v), _p(dec.cu_seqlens), B, H,
                                int(max_seqlen), _p(dec.gate), _p(out), float(dec.scale), stream)
    _lib.check(st, lib)
    return out


def test_noalloc_matches_oracle_and_workspace_decode_on_two_calls_in_a_row():
    cases = [([3000, 1500, 8192, 64], 8, 8192, 41),   # several chunks per (b,h)
             ([700, 129, 1], 3, 1024, 42)]             # smaller problem on reused scratch
    for lengths, H, max_len, cfg in cases:
        dec = mi.make_decode(lengths, H, True, device="cuda", config=cfg)
        got = noalloc_decode(dec, max_len)
        mla.check_device_status()
        ref = oracle.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, dec.gate, dec.scale)
        assert_close(got, ref, what=f"noalloc vs oracle {lengths}")
        ws_out = mla.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, max_len, gate=dec.gate,
                                scale=dec.scale)
        mla.check_device_status()
        assert torch.equal(got, ws_out), f"noalloc vs workspace decode {lengths}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    need = lib.mla_workspace_size(_lib.OP_DECODE, 64, 96, 65536, 0)
    assert need > _lib.NOALLOC_SCRATCH_BYTES
    x = torch.empty(1024, dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(65, dtype=torch.int64, device="cuda")
    st = lib.mla_decode_noalloc(_p(x), _p(x), _p(x), _p(cu), 64, 96, 65536, None, _p(x), 0.07,
                                None)
    assert st == _lib.MLA_ERR_WORKSPACE
    assert b"built-in scratch" in lib.mla_last_error()
