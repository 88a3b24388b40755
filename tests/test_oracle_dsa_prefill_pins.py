"""Pins of the oracle's DSA prefill (per-token index scores, per-token top-k,
gated MLA over each token's own selection of the latent cache):

* index scores against an explicit triple loop (ReLU per head, then the
  weighted head sum; positions after the token are never visible);
* every row's selection is the full-sort top-k of its visible scores, short
  rows keep every visible position;
* with a top-k at least as large as the context the sparse prefill equals
  the dense causal prefill over the expanded cache, row for row;
* the output does not depend on cache rows no token selected.
"""
import numpy as np

import oracle
from test_oracle_pins import SCALE, bf16_like

RNG = np.random.default_rng(2024)


def make(Tq, Tk, H=2):
    iq = bf16_like((Tq, 32, 128), RNG)
    ik = bf16_like((Tk, 128), RNG)
    w = bf16_like((Tq, 32), RNG) / 64
    q = bf16_like((Tq, H, 192), RNG)
    ckv = bf16_like((Tk, 576), RNG)
    wk = bf16_like((H, 128, 512), RNG) / 16
    wv = bf16_like((H, 128, 512), RNG) / 16
    g = bf16_like((Tq, H * 128), RNG)
    return iq, ik, w, q, ckv, wk, wv, g


def test_index_scores_triple_loop():
    iq, ik, w, *_ = make(5, 9)
    got = oracle.dsa_prefill_index_scores(iq, ik, w)
    P = 4
    for i in range(5):
        for s in range(9):
            if s > P + i:
                assert got[i, s] == -np.inf
                continue
            ref = sum(w[i, h] * max(0.0, float(np.dot(iq[i, h], ik[s]))) for h in range(32))
            assert abs(got[i, s] - ref) <= 1e-9 * (1 + abs(ref))


def test_topk_rows_are_full_sort_of_visible_scores():
    iq, ik, w, *_ = make(12, 40)
    s = oracle.dsa_prefill_index_scores(iq, ik, w)
    idx = oracle.dsa_prefill_topk(s, 8)
    P = 28
    for i in range(12):
        n = P + i + 1
        order = sorted(range(n), key=lambda j: (-s[i, j], j))[:8]
        assert list(idx[i]) == sorted(order)
    short = oracle.dsa_prefill_topk(s[:, :], 64)
    for i in range(12):
        n = P + i + 1
        assert list(short[i, :n]) == list(range(n)) and (short[i, n:] == -1).all()


def test_full_selection_equals_dense_causal_prefill():
    Tq, Tk, H = 6, 10, 2
    iq, ik, w, q, ckv, wk, wv, g = make(Tq, Tk, H)
    idx = oracle.dsa_prefill_topk(oracle.dsa_prefill_index_scores(iq, ik, w), 16)
    got = oracle.dsa_prefill_latent(q, ckv, wk, wv, idx, g, SCALE)
    k, v = oracle.expand_latent(ckv, wk, wv)
    dense = oracle.mla_prefill(q.transpose(1, 0, 2)[None], k[None], v[None], g[None], SCALE)[0]
    np.testing.assert_allclose(got, dense, rtol=0, atol=1e-12)


def test_unselected_rows_do_not_matter():
    Tq, Tk, H = 4, 30, 2
    iq, ik, w, q, ckv, wk, wv, g = make(Tq, Tk, H)
    idx = oracle.dsa_prefill_topk(oracle.dsa_prefill_index_scores(iq, ik, w), 5)
    a = oracle.dsa_prefill_latent(q, ckv, wk, wv, idx, g, SCALE)
    used = np.zeros(Tk, bool)
    used[idx[idx >= 0]] = True
    ckv2 = ckv.copy()
    ckv2[~used] = bf16_like((int((~used).sum()), 576), RNG)
    b = oracle.dsa_prefill_latent(q, ckv2, wk, wv, idx, g, SCALE)
    np.testing.assert_array_equal(a, b)
