"""GPU parity of mla_decode_latent (absorbed 576-feature latent cache,
tcgen05 attention with the heads as M) against the fp64 oracle, which
expands the cache by W^K, W^V (eq. (8)) and runs the plain decode."""
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


def run(d, max_len=None, out=None):
    o = mla.mla_decode_latent(d.q, d.ckv, d.cu_seqlens, max_len or max(d.lengths), d.w_kc,
                              d.w_vc, gate=d.gate, out=out, scale=d.scale)
    mla.check_device_status()
    return o


def ref(d, heads=None):
    if heads is None:
        return oracle.mla_decode_latent(d.q, d.ckv, d.cu_seqlens, d.w_kc, d.w_vc, d.gate, d.scale)
    cols = np.concatenate([np.arange(h * 128, (h + 1) * 128) for h in heads])
    g = d.gate[:, cols] if d.gate is not None else None
    return oracle.mla_decode_latent(d.q[:, heads], d.ckv, d.cu_seqlens, d.w_kc[heads],
                                    d.w_vc[heads], g, d.scale), cols


@pytest.mark.parametrize("lengths,H,gated", [
    ([1], 96, True),
    ([63, 64, 65, 1, 200], 96, True),       # ragged tiles, one-position sequence
    ([130, 7], 16, False),
    ([300, 1000], 48, True),
    ([513, 90, 4], 64, False),
])
def test_latent_small_matches_oracle(lengths, H, gated):
    d = mi.make_latent_decode(lengths, H, gated, device=DEV, config=81)
    assert_close(run(d), ref(d), what=f"latent {lengths} H{H}")


def test_latent_many_sequences_ragged():
    """B=40 (several absorb and merge blocks), lengths 1..3000: many CTA
    ranges start or end inside a sequence."""
    lengths = mi.ragged_lengths(40, 1, 3000, 82)
    d = mi.make_latent_decode(lengths, 96, True, device=DEV, config=82)
    out = run(d)
    heads = [0, 37, 95]
    r, cols = ref(d, heads)
    assert_close(out[:, cols], r, what="latent ragged B=40")


def test_latent_one_long_sequence_spans_every_cta():
    d = mi.make_latent_decode([20000], 96, True, device=DEV, config=83)
    out = run(d)
    r, cols = ref(d, [1, 50, 94])
    assert_close(out[:, cols], r, what="latent T=20000")


def test_latent_is_deterministic():
    d = mi.make_latent_decode([5000, 17, 900], 96, True, device=DEV, config=84)
    assert torch.equal(run(d), run(d))


def test_latent_matches_expanded_gpu_decode():
    """The same cache expanded (keys and values rounded to bf16) and run
    through mla_decode agrees within the parity tolerance."""
    d = mi.make_latent_decode([700, 2048], 96, True, device=DEV, config=85)
    out = run(d)
    lat = d.ckv[:, :512].float()
    k = torch.einsum("hdj,nj->hnd", d.w_kc.float(), lat)
    v = torch.einsum("hdj,nj->hnd", d.w_vc.float(), lat)
    ks, vs = [], []
    for b in range(2):
        a, e = int(d.cu_seqlens[b]), int(d.cu_seqlens[b + 1])
        kb = torch.cat([k[:, a:e], d.ckv[a:e, 512:].float()[None].expand(96, -1, -1)], 2)
        ks.append(kb.to(torch.bfloat16).reshape(-1))
        vs.append(v[:, a:e].to(torch.bfloat16).reshape(-1))
    exp = mla.mla_decode(d.q, torch.cat(ks), torch.cat(vs), d.cu_seqlens, 2048, gate=d.gate,
                         scale=d.scale)
    mla.check_device_status()
    err = (out.float() - exp.float()).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3


def test_latent_invalid_length_is_reported_and_skipped():
    d = mi.make_latent_decode([100, 300], 32, True, device=DEV, config=86)
    out = torch.zeros((2, 32 * 128), dtype=torch.bfloat16, device=DEV)
    mla.mla_decode_latent(d.q, d.ckv, d.cu_seqlens, 200, d.w_kc, d.w_vc, gate=d.gate, out=out,
                          scale=d.scale)
    with pytest.raises(mla.MlaError) as e:
        mla.check_device_status()
    assert e.value.status == _lib.MLA_ERR_INVALID_ARG
    r = oracle.mla_decode_latent(d.q[:1], d.ckv[:100], d.cu_seqlens[:2], d.w_kc, d.w_vc,
                                 d.gate[:1], d.scale)
    assert_close(out[:1], r)
    assert not out[1].any()


def test_latent_rejects_unsupported_heads():
    d = mi.make_latent_decode([10], 96, True, device=DEV, config=87)
    lib = _lib.load()
    import ctypes
    P = ctypes.c_void_p
    st = lib.mla_decode_latent(P(d.q.data_ptr()), P(d.ckv.data_ptr()), P(d.cu_seqlens.data_ptr()),
                               10, 1, 40, 10, P(d.w_kc.data_ptr()), P(d.w_vc.data_ptr()), None,
                               P(d.q.data_ptr()), 0.1, None, 0, None)
    assert st == _lib.MLA_ERR_UNSUPPORTED


def test_latent_full_size_sampled():
    """B=32, H=96, T=8192 in the configuration the benchmark times; two
    sequences and three heads checked against the oracle."""
    w = mi.WORKLOADS["latent_decode_b32_h96_t8192"]
    d = mi.make_latent_decode([w["T"]] * w["B"], w["H"], True, device=DEV, config=w["config"])
    out = run(d)
    for b in (0, w["B"] - 1):
        sub = mi.LatentDecode(d.q[b:b + 1], d.ckv[b * w["T"]:(b + 1) * w["T"]],
                              torch.tensor([0, w["T"]], device=DEV), [w["T"]], d.w_kc, d.w_vc,
                              d.gate[b:b + 1], d.scale, d.H)
        r, cols = ref(sub, [0, 48, 95])
        assert_close(out[b:b + 1, cols], r, what=f"latent full b{b}")
