"""GPU parity of mla_prefill (tcgen05 causal gated MLA prefill) against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle
import mla_family_attention_gb300 as mla
from mla_family_attention_gb300 import _lib
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(pf):
    out = mla.mla_prefill(pf.q, pf.k, pf.v, pf.gate, scale=pf.scale)
    mla.check_device_status()
    return out


@pytest.fixture(params=[1, 2], ids=["one_cta", "cta_pair"])
def ctas(request):
    """Both kernel shapes: one CTA per 128-row query tile (M = 128 MMAs) and
    a pair of CTAs on two SMs sharing each M = 256 MMA."""
    mla.debug_set(_lib.DEBUG_PREFILL_CTAS, request.param)
    yield request.param
    mla.debug_set(_lib.DEBUG_PREFILL_CTAS, 0)


@pytest.mark.parametrize("B,H,Tq,Tk,gated", [
    (1, 1, 1, 1, True),
    (1, 2, 128, 128, True),        # one tile
    (1, 2, 200, 200, True),        # ragged query and key tiles
    (2, 3, 64, 64, False),
    (1, 2, 100, 300, True),        # non-empty cache: bottom-right causal
    (1, 2, 1, 257, True),          # one new token over a ragged cache
    (1, 4, 257, 257, True),
    (2, 2, 130, 390, False),
    (1, 1, 640, 640, True),        # five query tiles, seven 96-key tiles
    (1, 2, 96, 96, True),          # exactly one key tile
    (1, 3, 288, 289, False),       # three key tiles (every score buffer) and one key more
    (1, 2, 1000, 1000, True),      # the score-buffer ring wraps several times
    (1, 2, 60, 1100, True),        # short chunk over a long cache, mask on the last tiles only
])
def test_prefill_small_matches_oracle(B, H, Tq, Tk, gated, ctas):
    pf = mi.make_prefill(B, H, Tq, Tk, gated, device=DEV, config=61)
    out = run(pf)
    ref = oracle.mla_prefill(pf.q, pf.k, pf.v, pf.gate, pf.scale)
    assert_close(out, ref, what=f"prefill B{B} H{H} Tq{Tq} Tk{Tk}")


def test_prefill_b1_h96_t128_full():
    """The 128-token gated prefill, B=1, H=96, compared in full."""
    w = mi.WORKLOADS["prefill_b1_h96_t128"]
    pf = mi.make_prefill(w["B"], w["H"], w["T"], w["T"], True, device=DEV, config=w["config"])
    out = run(pf)
    ref = oracle.mla_prefill(pf.q, pf.k, pf.v, pf.gate, pf.scale)
    assert_close(out, ref)


def test_prefill_is_deterministic():
    pf = mi.make_prefill(1, 3, 300, 300, True, device=DEV, config=62)
    assert torch.equal(run(pf), run(pf))


def test_prefill_scale_argument_is_used():
    pf = mi.make_prefill(1, 2, 130, 130, True, device=DEV, config=63)
    out = mla.mla_prefill(pf.q, pf.k, pf.v, pf.gate, scale=0.2)
    mla.check_device_status()
    ref = oracle.mla_prefill(pf.q, pf.k, pf.v, pf.gate, 0.2)
    assert_close(out, ref)


def test_prefill_rejects_tq_above_tk():
    pf = mi.make_prefill(1, 1, 8, 8, True, device=DEV, config=64)
    with pytest.raises(ValueError):
        mla.mla_prefill(pf.q, pf.k[:, :, :4].contiguous(), pf.v[:, :, :4].contiguous(), pf.gate)
    lib = _lib.load()
    import ctypes
    P = ctypes.c_void_p
    st = lib.mla_prefill(P(pf.q.data_ptr()), P(pf.k.data_ptr()), P(pf.v.data_ptr()), None,
                         P(pf.q.data_ptr()), 1, 1, 8, 4, 0.1, None, 0, None)
    assert st == _lib.MLA_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["prefill_b1_h96_t16384", "prefill_b1_h64_t16384_nogate"])
def test_prefill_long_full_size_sampled(name):
    """B=1, T=16384 (H=96 gated / H=64 ungated) in the launch configuration the
    benchmark times; sampled rows checked against the oracle one by one."""
    w = mi.WORKLOADS[name]
    T, H = w["T"], w["H"]
    pf = mi.make_prefill(1, H, T, T, w["gated"], device=DEV, config=w["config"])
    out = run(pf)
    rng = np.random.default_rng(3)
    rows = [0, 1, 127, 128, 8191, T - 1] + [int(x) for x in rng.integers(0, T, 4)]
    heads = [0, H - 1, int(rng.integers(0, H))]
    for h in heads:
        for i in rows:
            g = pf.gate[:, i:i + 1, h * 128:(h + 1) * 128] if pf.gate is not None else None
            ref = oracle.mla_prefill(pf.q[:, h:h + 1, i:i + 1], pf.k[:, h:h + 1, :i + 1],
                                     pf.v[:, h:h + 1, :i + 1], g, pf.scale)
            assert_close(out[:, i:i + 1, h * 128:(h + 1) * 128], ref, what=f"h{h} row{i}")
    del pf, out
    torch.cuda.empty_cache()
