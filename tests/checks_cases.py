"""Small parity cases run against whichever build of the library
MLA_GB300_LIB names (the bounds-checked debug build, in test_gpu_checks.py).

Every entry point's small case from the smoke run (each followed by a device
status check, which raises on MLA_ERR_CHECK, and a comparison with the fp64
oracle), then the paths the smoke run leaves at their defaults: the top-k
in its separate cluster kernel, the two-SM prefill shape and the decode on
the library's built-in scratch.
"""
import ctypes
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))


def main():
    import numpy as np
    import torch

    import __graft_entry__ as ge
    import mla_inputs as mi
    import mla_family_attention_gb300 as mla
    import oracle
    from mla_family_attention_gb300 import _lib
    from parity import assert_close

    lib = _lib.load()
    assert os.path.samefile(lib._name, os.environ["MLA_GB300_LIB"]), lib._name
    ge.smoke()
    dev = "cuda:0"
    # indexer top-k over several ragged sequences
    lengths = [5000, 700, 2300]
    d = mi.make_dsa(lengths, H=4, device=dev, config=61)
    cu = mi.cu_from_lengths(lengths)
    ref = oracle.dsa_topk(oracle.dsa_index_scores(d.index_q, d.index_k, d.w, cu), cu, 512)
    idx = mla.dsa_index_topk(d.index_q, d.index_k, d.w, cu.to(dev), max(lengths), 512)
    mla.check_device_status()
    got = idx.cpu().numpy()
    assert np.array_equal(got[1], ref[1])
    for b in (0, 2):
        assert len(set(got[b]) & set(ref[b])) >= 505, f"top-k b{b}"
    # the two-SM prefill shape over ragged tiles
    pf = mi.make_prefill(1, 2, 300, 300, True, device=dev, config=62)
    mla.debug_set(_lib.DEBUG_PREFILL_CTAS, 2)
    out = mla.mla_prefill(pf.q, pf.k, pf.v, pf.gate, scale=pf.scale)
    mla.check_device_status()
    mla.debug_set(_lib.DEBUG_PREFILL_CTAS, 0)
    assert_close(out, oracle.mla_prefill(pf.q, pf.k, pf.v, pf.gate, pf.scale), what="pair prefill")
    # the decode on the library's built-in scratch
    dec = mi.make_decode([3000, 64, 1500], 4, True, device=dev, config=63)
    outd = torch.empty((3, 4 * 128), dtype=torch.bfloat16, device=dev)
    P = ctypes.c_void_p
    st = lib.mla_decode_noalloc(P(dec.q.data_ptr()), P(dec.k.data_ptr()), P(dec.v.data_ptr()),
                                P(dec.cu_seqlens.data_ptr()), 3, 4, 3000, P(dec.gate.data_ptr()),
                                P(outd.data_ptr()), float(dec.scale),
                                P(torch.cuda.current_stream().cuda_stream))
    _lib.check(st, lib)
    mla.check_device_status()
    assert_close(outd, oracle.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, dec.gate, dec.scale),
                 what="decode on built-in scratch")
    print("checked cases ok")


if __name__ == "__main__":
    main()
