"""Pins of the oracle's absorbed-latent decode (expansion of a 576-feature
latent cache by W^K, W^V, then the decode definition):

* the absorbed evaluation written out here in NumPy (W^K folded into the
  query, attention over the latent, W^V applied to the latent output) gives
  the same rows to 1e-12 -- a transposed weight, a wrong 512/64 split of the
  latent or a rope part routed through W^K fails it;
* brute force over keys and values built position by position with explicit
  matrix-vector products;
* identity weights reduce it to the plain decode over k = [c[:128]; r],
  v = c[:128].
"""
import numpy as np
from scipy.special import expit, softmax

import oracle
from test_oracle_pins import SCALE, bf16_like

RNG = np.random.default_rng(91)


def make(lengths, H):
    N = sum(lengths)
    ckv = bf16_like((N, 576), RNG)
    wk = bf16_like((H, 128, 512), RNG) / 16
    wv = bf16_like((H, 128, 512), RNG) / 16
    q = bf16_like((len(lengths), H, 192), RNG)
    g = bf16_like((len(lengths), H * 128), RNG)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return ckv, wk, wv, q, g, cu


def absorbed(q, ckv, cu, wk, wv, g, scale):
    B, H = q.shape[:2]
    out = np.empty((B, H * 128))
    for b in range(B):
        c = ckv[cu[b]:cu[b + 1]]
        for h in range(H):
            qt = wk[h].T @ q[b, h, :128]                     # [512]
            s = (c[:, :512] @ qt + c[:, 512:] @ q[b, h, 128:]) * scale
            zt = softmax(s) @ c[:, :512]                     # [512]
            out[b, h * 128:(h + 1) * 128] = (wv[h] @ zt) * expit(g[b, h * 128:(h + 1) * 128])
    return out


def test_absorbed_order_matches_expanded_oracle():
    ckv, wk, wv, q, g, cu = make([1, 7, 20], 3)
    got = oracle.mla_decode_latent(q, ckv, cu, wk, wv, g, SCALE)
    np.testing.assert_allclose(got, absorbed(q, ckv, cu, wk, wv, g, SCALE), rtol=0, atol=1e-12)


def test_brute_force_per_position():
    ckv, wk, wv, q, g, cu = make([5, 3], 2)
    got = oracle.mla_decode_latent(q, ckv, cu, wk, wv, None, SCALE)
    for b in range(2):
        rows = ckv[cu[b]:cu[b + 1]]
        for h in range(2):
            k = np.array([np.concatenate([wk[h] @ r[:512], r[512:]]) for r in rows])
            v = np.array([wv[h] @ r[:512] for r in rows])
            p = softmax(np.array([q[b, h] @ kk for kk in k]) * SCALE)
            np.testing.assert_allclose(got[b, h * 128:(h + 1) * 128], p @ v, rtol=0, atol=1e-12)


def test_identity_weights_reduce_to_plain_decode():
    ckv, _, _, q, g, cu = make([4, 9], 2)
    eye = np.zeros((2, 128, 512))
    eye[:, :, :128] = np.eye(128)
    got = oracle.mla_decode_latent(q, ckv, cu, eye, eye, g, SCALE)
    k = [np.broadcast_to(np.concatenate([ckv[cu[b]:cu[b + 1], :128],
                                         ckv[cu[b]:cu[b + 1], 512:]], 1), (2, cu[b + 1] - cu[b], 192))
         for b in range(2)]
    v = [np.broadcast_to(ckv[cu[b]:cu[b + 1], :128], (2, cu[b + 1] - cu[b], 128)) for b in range(2)]
    ref = oracle.mla_decode(q, np.concatenate([x.reshape(-1) for x in k]),
                            np.concatenate([x.reshape(-1) for x in v]), cu, g, SCALE)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
