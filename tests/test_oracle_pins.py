"""Pins of the fp64 oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle (a dropped scale,
a wrong mask index, a transposed output layout, sigmoid(-g) for sigmoid(g), a
missing ReLU, a reversed tie-break) fails at least one of them:

* brute force: a NumPy float64 restatement in matrix form (full score matrix,
  -inf mask, SciPy's softmax) on tiny shapes;
* invariants: probabilities sum to one; future keys do not change past rows;
  a constant added to every score changes nothing;
* closed forms: one key, zero query, equal keys, zero gate logits, a gate of
  ln 3 (sigmoid = 3/4), a dominant key, hand-solvable two-key rows;
* DSA: NumPy scores, full lexicographic sort for top-k, short context keeps
  every position, positive rescaling of w keeps the set, one-hot w ranks by a
  single head, sparse decode over every position equals dense decode.
"""
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle

RNG = np.random.default_rng(1234)
SCALE = 192 ** -0.5


def bf16_like(shape, rng=RNG):
    """Random values exactly representable in bf16 (8 significant bits)."""
    x = rng.standard_normal(shape)
    m, e = np.frexp(x)
    return np.ldexp(np.round(m * 256) / 256, e)


def brute_prefill(q, k, v, g, scale):
    B, H, Tq, _ = q.shape
    Tk, Dv = k.shape[2], v.shape[3]
    s = np.einsum("bhid,bhjd->bhij", q, k) * scale
    i = np.arange(Tq)[:, None]
    j = np.arange(Tk)[None, :]
    s = np.where(j <= (Tk - Tq) + i, s, -np.inf)
    p = softmax(s, axis=-1)
    z = np.einsum("bhij,bhjd->bhid", p, v)
    out = z.transpose(0, 2, 1, 3).reshape(B, Tq, H * Dv)
    return out * expit(g) if g is not None else out


def pack(kseqs):
    """List of per-sequence [H,T,D] arrays -> flat packed array."""
    return np.concatenate([x.reshape(-1) for x in kseqs])


# ---------------------------------------------------------------------------
# P1: brute force
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,H,Tq,Tk,gated", [(1, 1, 1, 1, True), (2, 3, 5, 5, True),
                                             (1, 2, 3, 9, True), (2, 2, 7, 7, False),
                                             (1, 3, 9, 9, True)])
def test_prefill_brute_force(B, H, Tq, Tk, gated):
    q, k = bf16_like((B, H, Tq, 192)), bf16_like((B, H, Tk, 192))
    v = bf16_like((B, H, Tk, 128))
    g = bf16_like((B, Tq, H * 128)) if gated else None
    got = oracle.mla_prefill(q, k, v, g, SCALE)
    np.testing.assert_allclose(got, brute_prefill(q, k, v, g, SCALE), rtol=0, atol=1e-12)


def test_decode_brute_force_ragged():
    H, lens = 3, [1, 4, 9]
    ks = [bf16_like((H, T, 192)) for T in lens]
    vs = [bf16_like((H, T, 128)) for T in lens]
    q = bf16_like((len(lens), H, 192))
    g = bf16_like((len(lens), H * 128))
    cu = np.concatenate([[0], np.cumsum(lens)])
    got = oracle.mla_decode(q, pack(ks), pack(vs), cu, g, SCALE)
    for b, T in enumerate(lens):
        # decode = the last row of a prefill whose query sees all T keys
        ref = brute_prefill(q[b][None, :, None, :], ks[b][None], vs[b][None],
                            g[b][None, None, :], SCALE)[0, 0]
        np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-12)


def test_output_channel_layout_is_head_major():
    """Channel h*128+d holds head h, feature d: give each head a constant value row."""
    B, H, T = 1, 3, 4
    q, k = bf16_like((B, H, T, 192)), bf16_like((B, H, T, 192))
    v = np.zeros((B, H, T, 128))
    for h in range(H):
        v[0, h] = np.arange(128) + 1000 * h
    out = oracle.mla_prefill(q, k, v, None, SCALE)
    for h in range(H):
        np.testing.assert_allclose(out[0, :, h * 128:(h + 1) * 128],
                                   np.broadcast_to(np.arange(128) + 1000 * h, (T, 128)),
                                   rtol=1e-13)


# ---------------------------------------------------------------------------
# P2: invariants
# ---------------------------------------------------------------------------
def test_probabilities_sum_to_one():
    for n in (1, 2, 17, 300):
        q, k, v = bf16_like(192) * 3, bf16_like((n, 192)) * 3, bf16_like((n, 128))
        z, p = oracle.attention_probs(q, k, v, SCALE)
        assert np.all(p >= 0)
        assert abs(p.sum() - 1.0) < 1e-12
        np.testing.assert_allclose(z, p @ v, atol=1e-12)


def test_probabilities_are_softmax_of_scaled_scores():
    n = 11
    q, k, v = bf16_like(192), bf16_like((n, 192)), bf16_like((n, 128))
    _, p = oracle.attention_probs(q, k, v, SCALE)
    s = k @ q * SCALE
    np.testing.assert_allclose(np.log(p) - np.log(p[0]), s - s[0], atol=1e-12)


def test_future_keys_do_not_change_past_rows():
    B, H, T = 1, 2, 8
    q, k = bf16_like((B, H, T, 192)), bf16_like((B, H, T, 192))
    v, g = bf16_like((B, H, T, 128)), bf16_like((B, T, H * 128))
    base = oracle.mla_prefill(q, k, v, g, SCALE)
    for cut in range(1, T):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, cut:] += 5.0
        v2[:, :, cut:] -= 7.0
        out = oracle.mla_prefill(q, k2, v2, g, SCALE)
        assert np.array_equal(out[:, :cut], base[:, :cut])     # bit for bit
        assert not np.allclose(out[:, cut:], base[:, cut:])


def test_constant_shared_key_part_changes_nothing():
    """q_rot . k_rot equal for every position adds one constant to all scores."""
    B, H, T = 1, 2, 6
    q, k = bf16_like((B, H, T, 192)), bf16_like((B, H, T, 192))
    v = bf16_like((B, H, T, 128))
    k1, k2 = k.copy(), k.copy()
    k1[..., 128:] = 0.0
    k2[..., 128:] = bf16_like(64)          # one shared vector, same at every position
    a = oracle.mla_prefill(q, k1, v, None, SCALE)
    b = oracle.mla_prefill(q, k2, v, None, SCALE)
    np.testing.assert_allclose(a, b, atol=1e-12)


# ---------------------------------------------------------------------------
# P3: closed forms
# ---------------------------------------------------------------------------
def test_single_key_gives_its_value_times_gate():
    q, k, v = bf16_like((1, 2, 1, 192)), bf16_like((1, 2, 1, 192)), bf16_like((1, 2, 1, 128))
    g = bf16_like((1, 1, 256))
    out = oracle.mla_prefill(q, k, v, g, SCALE)
    np.testing.assert_allclose(out[0, 0], v[0, :, 0].reshape(-1) / (1 + np.exp(-g[0, 0])),
                               atol=1e-15)


def test_zero_query_averages_visible_values():
    B, H, T = 1, 1, 5
    q = np.zeros((B, H, T, 192))
    k, v = bf16_like((B, H, T, 192)), bf16_like((B, H, T, 128))
    out = oracle.mla_prefill(q, k, v, None, SCALE)
    for i in range(T):
        np.testing.assert_allclose(out[0, i], v[0, 0, :i + 1].mean(0), atol=1e-14)


def test_equal_keys_average_values_and_zero_gate_halves():
    T = 7
    q = bf16_like((1, 192))
    k = np.broadcast_to(bf16_like(192), (T, 192)).copy()
    v = bf16_like((1, T, 128))
    cu = np.array([0, T])
    out = oracle.mla_decode(q[None], k, v, cu, np.zeros((1, 128)), SCALE)
    np.testing.assert_allclose(out[0], v[0].mean(0) / 2, atol=1e-14)


def test_gate_of_ln3_is_three_quarters():
    q, k, v = np.zeros((1, 1, 192)), np.zeros((1, 192)), np.ones((1, 128))
    g = np.full((1, 128), math.log(3.0))
    out = oracle.mla_decode(q, k, v, np.array([0, 1]), g, SCALE)
    np.testing.assert_allclose(out, 0.75, atol=1e-15)


def test_hand_solved_two_key_row():
    """Scores differ by ln 3 -> p = (1/4, 3/4) (hand-derived, see golden file)."""
    import json
    import os
    case = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                       "hand_cases.json")))["two_keys"]
    q = np.zeros(192)
    q[0] = case["q0"]
    k = np.zeros((2, 192))
    k[1, 0] = case["k1_0"]
    v = np.zeros((2, 128))
    v[0, 0], v[1, 0] = case["v0_0"], case["v1_0"]
    z, p = oracle.attention_probs(q, k, v, case["scale"])
    np.testing.assert_allclose(p, case["p"], atol=1e-15)
    assert abs(z[0] - case["z0"]) < 1e-14


def test_dominant_key_selects_its_value():
    T = 6
    q = np.zeros((1, 1, 192))
    q[0, 0, 0] = 40.0
    k = np.zeros((T, 192))
    k[3, 0] = 40.0                      # score 1600/sqrt(192) ~ 115 above the rest
    v = bf16_like((1, T, 128))
    out = oracle.mla_decode(q, k, v, np.array([0, T]), None, SCALE)
    np.testing.assert_allclose(out[0], v[0, 3], atol=1e-12)


def test_scale_is_applied():
    """Doubling the scale is the same as doubling q."""
    q, k, v = bf16_like((1, 1, 4, 192)), bf16_like((1, 1, 4, 192)), bf16_like((1, 1, 4, 128))
    a = oracle.mla_prefill(q, k, v, None, 2 * SCALE)
    b = oracle.mla_prefill(2 * q, k, v, None, SCALE)
    np.testing.assert_allclose(a, b, atol=1e-13)
    c = oracle.mla_prefill(q, k, v, None, SCALE)
    assert not np.allclose(a, c)


# ---------------------------------------------------------------------------
# P4: DSA indexer, top-k and sparse decode
# ---------------------------------------------------------------------------
def brute_scores(iq, ik, w, cu):
    out = []
    for b in range(len(cu) - 1):
        z = ik[cu[b]:cu[b + 1]] @ iq[b].T          # [T, NH]
        out.append(((z + np.abs(z)) / 2) @ w[b])   # ReLU(z) = (z + |z|)/2
    return np.concatenate(out)


def brute_topk(scores, cu, topk):
    B = len(cu) - 1
    idx = np.full((B, topk), -1, dtype=np.int32)
    for b in range(B):
        s = scores[cu[b]:cu[b + 1]]
        order = np.lexsort((np.arange(s.size), -s))      # score desc, position asc
        sel = np.sort(order[:min(topk, s.size)])
        idx[b, :sel.size] = sel
    return idx


def test_index_scores_brute_force():
    lens = [1, 5, 40]
    cu = np.concatenate([[0], np.cumsum(lens)])
    iq, ik = bf16_like((3, 32, 128)), bf16_like((cu[-1], 128))
    w = RNG.standard_normal((3, 32))
    np.testing.assert_allclose(oracle.dsa_index_scores(iq, ik, w, cu),
                               brute_scores(iq, ik, w, cu), atol=1e-10)


def test_index_score_relu_matters():
    """Negative head dot products contribute nothing (w > 0, all dots < 0 -> 0)."""
    iq = -np.abs(bf16_like((1, 32, 128)))
    ik = np.abs(bf16_like((3, 128)))
    w = np.abs(RNG.standard_normal((1, 32)))
    assert np.all(oracle.dsa_index_scores(iq, ik, w, np.array([0, 3])) == 0.0)


@pytest.mark.parametrize("lens,topk", [([50, 7, 33], 8), ([3], 8), ([64, 64], 64), ([100], 1)])
def test_topk_matches_full_sort(lens, topk):
    cu = np.concatenate([[0], np.cumsum(lens)])
    iq, ik = bf16_like((len(lens), 32, 128)), bf16_like((cu[-1], 128))
    w = RNG.standard_normal((len(lens), 32))
    s = oracle.dsa_index_scores(iq, ik, w, cu)
    got = oracle.dsa_topk(s, cu, topk)
    np.testing.assert_array_equal(got, brute_topk(s, cu, topk))


def test_topk_ties_prefer_lower_positions():
    s = np.array([1.0, 5.0, 5.0, 2.0, 5.0, 5.0, 0.0])
    got = oracle.dsa_topk(s, np.array([0, 7]), 3)
    np.testing.assert_array_equal(got, [[1, 2, 4]])


def test_short_context_keeps_every_position():
    s = RNG.standard_normal(5)
    np.testing.assert_array_equal(oracle.dsa_topk(s, np.array([0, 5]), 8),
                                  [[0, 1, 2, 3, 4, -1, -1, -1]])


def test_topk_set_invariant_to_positive_weight_scale_and_one_hot():
    T, topk = 200, 16
    cu = np.array([0, T])
    iq, ik = bf16_like((1, 32, 128)), bf16_like((T, 128))
    w = RNG.standard_normal((1, 32))
    a = oracle.dsa_topk(oracle.dsa_index_scores(iq, ik, w, cu), cu, topk)
    b = oracle.dsa_topk(oracle.dsa_index_scores(iq, ik, w * 3.5, cu), cu, topk)
    np.testing.assert_array_equal(a, b)
    h = 5
    onehot = np.zeros((1, 32))
    onehot[0, h] = 1.0
    got = oracle.dsa_topk(oracle.dsa_index_scores(iq, ik, onehot, cu), cu, topk)
    z = np.maximum(ik @ iq[0, h], 0)
    np.testing.assert_array_equal(got[0], np.sort(np.lexsort((np.arange(T), -z))[:topk]))


def test_sparse_over_every_position_equals_dense():
    H, lens = 2, [5, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    ks = [bf16_like((H, T, 192)) for T in lens]
    vs = [bf16_like((H, T, 128)) for T in lens]
    q, g = bf16_like((2, H, 192)), bf16_like((2, H * 128))
    idx = np.full((2, 16), -1, dtype=np.int32)
    for b, T in enumerate(lens):
        idx[b, :T] = np.arange(T)
    dense = oracle.mla_decode(q, pack(ks), pack(vs), cu, g, SCALE)
    sparse = oracle.dsa_sparse_decode(q, pack(ks), pack(vs), cu, idx, g, SCALE)
    assert np.array_equal(dense, sparse)


def test_sparse_uses_only_selected_positions():
    H, T = 1, 10
    k, v = bf16_like((H, T, 192)), bf16_like((H, T, 128))
    q = bf16_like((1, H, 192))
    sel = np.array([[7, 2, 4, -1]], dtype=np.int32)
    got = oracle.dsa_sparse_decode(q, k, v, np.array([0, T]), sel, None, SCALE)
    ref = brute_prefill(q[:, :, None, :], k[None, :, [2, 4, 7]], v[None, :, [2, 4, 7]], None,
                        SCALE)[0, 0]
    np.testing.assert_allclose(got[0], ref, atol=1e-12)
    # order of the selected list does not matter
    got2 = oracle.dsa_sparse_decode(q, k, v, np.array([0, T]),
                                    np.array([[4, -1, 2, 7]], dtype=np.int32), None, SCALE)
    np.testing.assert_allclose(got, got2, atol=1e-13)


def test_sparse_rejects_out_of_range_index():
    k, v, q = bf16_like((1, 4, 192)), bf16_like((1, 4, 128)), bf16_like((1, 1, 192))
    with pytest.raises(ValueError):
        oracle.dsa_sparse_decode(q, k, v, np.array([0, 4]), np.array([[4]], dtype=np.int32),
                                 None, SCALE)


def test_large_score_gaps_stay_finite():
    """Scores about 1000 apart: the max-subtracted softmax stays exact."""
    q = np.zeros((1, 1, 192))
    q[0, 0, 0] = 120.0
    k = np.zeros((3, 192))
    k[0, 0], k[1, 0], k[2, 0] = -120.0, 0.0, 120.0
    v = bf16_like((1, 3, 128))
    out = oracle.mla_decode(q, k, v, np.array([0, 3]), None, SCALE)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0], v[0, 2], atol=1e-12)
