"""Pins of the oracle's cache update, chunked prefill and fixed-capacity
decode against things other than themselves:

* a prompt fed in chunks gives the same rows as one prefill over the whole
  prompt, and as the NumPy brute force (a wrong offset P, a top-left instead
  of bottom-right causal alignment, or reading past P+Tq fails this);
* appends compose: Tn single-token appends equal one append of Tn tokens, and
  an append never touches positions outside its span (NaN-filled capacity
  stays NaN, the prefix stays bit-identical);
* a decode step over a capacity cache (with and without appending the
  current token) equals the last row of the brute-force prefill over the same
  keys, per sequence of a ragged batch.
"""
import numpy as np
import pytest

import oracle
from test_oracle_pins import SCALE, bf16_like, brute_prefill

RNG = np.random.default_rng(77)


def nan_cache(B, H, cap, D):
    return np.full((B, H, cap, D), np.nan)


@pytest.mark.parametrize("chunks,gated", [([4, 4, 3], True), ([1, 10], False), ([11], True),
                                          ([3, 1, 1, 6], True)])
def test_chunked_prefill_equals_whole_prompt(chunks, gated):
    B, H, T, cap = 2, 2, sum(chunks), 16
    q, k = bf16_like((B, H, T, 192), RNG), bf16_like((B, H, T, 192), RNG)
    v = bf16_like((B, H, T, 128), RNG)
    g = bf16_like((B, T, H * 128), RNG) if gated else None
    whole = oracle.mla_prefill(q, k, v, g, SCALE)
    np.testing.assert_allclose(whole, brute_prefill(q, k, v, g, SCALE), rtol=0, atol=1e-12)
    kc, vc = nan_cache(B, H, cap, 192), nan_cache(B, H, cap, 128)
    P = 0
    for n in chunks:
        sl = slice(P, P + n)
        gc = g[:, sl] if gated else None
        out = oracle.mla_prefill_chunk(q[:, :, sl], kc, vc, k[:, :, sl], v[:, :, sl], P, gc,
                                       SCALE)
        np.testing.assert_array_equal(out, whole[:, sl])
        np.testing.assert_allclose(
            out, brute_prefill(q[:, :, sl], k[:, :, :P + n], v[:, :, :P + n], gc, SCALE),
            rtol=0, atol=1e-12)
        kc, vc = oracle.cache_append(kc, vc, k[:, :, sl], v[:, :, sl], P)
        P += n
    np.testing.assert_array_equal(kc[:, :, :T], k)
    assert np.isnan(kc[:, :, T:]).all() and np.isnan(vc[:, :, T:]).all()


def test_single_token_appends_equal_one_append():
    B, H, cap, Tn = 3, 2, 12, 5
    kc, vc = bf16_like((B, H, cap, 192), RNG), bf16_like((B, H, cap, 128), RNG)
    kn, vn = bf16_like((B, H, Tn, 192), RNG), bf16_like((B, H, Tn, 128), RNG)
    start = [0, 4, 7]
    k1, v1 = oracle.cache_append(kc, vc, kn, vn, start)
    k2, v2 = kc, vc
    for t in range(Tn):
        k2, v2 = oracle.cache_append(k2, v2, kn[:, :, t:t + 1], vn[:, :, t:t + 1],
                                     [s + t for s in start])
    np.testing.assert_array_equal(k1, k2)
    np.testing.assert_array_equal(v1, v2)
    for b, s in enumerate(start):
        np.testing.assert_array_equal(k1[b, :, :s], kc[b, :, :s])
        np.testing.assert_array_equal(k1[b, :, s:s + Tn], kn[b])
        np.testing.assert_array_equal(k1[b, :, s + Tn:], kc[b, :, s + Tn:])


def test_append_past_capacity_is_rejected():
    kc, vc = nan_cache(1, 1, 4, 192), nan_cache(1, 1, 4, 128)
    kn, vn = bf16_like((1, 1, 2, 192), RNG), bf16_like((1, 1, 2, 128), RNG)
    with pytest.raises(ValueError):
        oracle.cache_append(kc, vc, kn, vn, 3)


@pytest.mark.parametrize("append", [False, True])
def test_decode_cached_is_last_prefill_row(append):
    B, H, cap, lens = 3, 2, 10, [1, 6, 9]
    kc, vc = nan_cache(B, H, cap, 192), nan_cache(B, H, cap, 128)
    keys = [bf16_like((H, L + 1, 192), RNG) for L in lens]
    vals = [bf16_like((H, L + 1, 128), RNG) for L in lens]
    for b, L in enumerate(lens):
        kc[b, :, :L], vc[b, :, :L] = keys[b][:, :L], vals[b][:, :L]
        if not append:
            kc[b, :, L], vc[b, :, L] = keys[b][:, L], vals[b][:, L]
    q, g = bf16_like((B, H, 192), RNG), bf16_like((B, H * 128), RNG)
    kn = np.stack([keys[b][:, L:L + 1] for b, L in enumerate(lens)]) if append else None
    vn = np.stack([vals[b][:, L:L + 1] for b, L in enumerate(lens)]) if append else None
    cached = np.array(lens) + (0 if append else 1)
    got = oracle.mla_decode_cached(q, kc, vc, cached, kn, vn, g, SCALE)
    for b, L in enumerate(lens):
        ref = brute_prefill(q[b][None, :, None], keys[b][None], vals[b][None],
                            g[b][None, None], SCALE)
        np.testing.assert_allclose(got[b], ref.reshape(-1), rtol=0, atol=1e-12)
