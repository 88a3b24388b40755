"""GPU parity of dsa_index_topk (indexer score + top-k) and of the whole DSA
decode path against the fp64 oracle, through the C ABI.

Top-k sets are compared the way the scores allow: every position whose
oracle score is outside the band of 1e-5 (relative) around the oracle's k-th
score must be classified identically; inside the band the GPU may pick any
positions, as long as it picks the right number of them.
"""
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
BAND = 1e-5


def check_selection(got_idx, got_scores, scores64, lengths, topk):
    """got_idx [B,topk] from the GPU; scores64 packed oracle scores."""
    got_idx = got_idx.cpu().numpy()
    off = 0
    for b, T in enumerate(lengths):
        row = got_idx[b]
        K = min(T, topk)
        sel = row[:K]
        assert np.all(row[K:] == -1), f"b{b}: padding"
        assert np.all(np.diff(sel) > 0), f"b{b}: not strictly ascending"
        assert sel.min() >= 0 and sel.max() < T
        if T <= topk:
            assert np.array_equal(sel, np.arange(T))
            off += T
            continue
        s = scores64[off:off + T]
        order = np.lexsort((np.arange(T), -s))
        kth = s[order[K - 1]]
        tol = BAND * abs(kth)
        must = set(np.nonzero(s > kth + tol)[0].tolist())
        band = set(np.nonzero(np.abs(s - kth) <= tol)[0].tolist())
        chosen = set(sel.tolist())
        assert must <= chosen, f"b{b}: {len(must - chosen)} clear winners missing"
        assert chosen <= must | band, f"b{b}: {len(chosen - must - band)} clear losers chosen"
        if got_scores is not None:
            gs = got_scores[b, :K].cpu().double().numpy()
            np.testing.assert_allclose(gs, s[sel], rtol=0, atol=1e-5 * np.abs(s).max() + 1e-6)
        off += T


def run_index(d, lengths, topk, max_seqlen=None):
    B = len(lengths)
    idx = torch.empty((B, topk), dtype=torch.int32, device=DEV)
    sc = torch.empty((B, topk), dtype=torch.float32, device=DEV)
    mla.dsa_index_topk(d.index_q, d.index_k, d.w, mi.cu_from_lengths(lengths).to(DEV),
                       max_seqlen or max(lengths), topk, topk_idx=idx, topk_scores=sc)
    mla.check_device_status()
    return idx, sc


@pytest.mark.parametrize("lengths,topk", [
    ([1, 100, 2048, 2049, 5000, 20000], 2048),   # short contexts, one-past, ragged tails
    ([3000, 129, 777], 64),
    ([400], 1),
    ([131072], 2048),
    ([2100 + 37 * i for i in range(40)], 2048),   # many sequences per CTA, ragged tails
    ([70000, 1, 2049, 130000, 5, 9000, 2048, 33000], 1000),
    ([131073, 5000], 2048),                       # one past the register-resident bound
    ([2100 + 13 * i for i in range(300)], 2048),  # more sequences than scoring CTAs: most
                                                  # are claimed by CTAs homed elsewhere
])
def test_index_topk_matches_oracle(lengths, topk):
    d = mi.make_dsa(lengths, device=DEV, config=51, with_main=False)
    idx, sc = run_index(d, lengths, topk)
    cu = mi.cu_from_lengths(lengths)
    s64 = oracle.dsa_index_scores(d.index_q, d.index_k, d.w, cu)
    check_selection(idx, sc, s64, lengths, topk)


@pytest.mark.parametrize("T,rows", [
    (6000, 200),       # 37 keys tie with the k-th: ranked one against another
    (60000, 2000),     # 42 tie, eight full ranges
    (6000, 100),       # 62 tie
    (6000, 40),        # 134 tie: the third radix level, then ties by position
    (6000, 10),        # 604 tie
    (300000, 2000),    # 162 tie, over ranges re-read in steps: ranked
    (300000, 300),     # 1025 tie: the third level
])
def test_index_topk_exact_ties_prefer_lower_positions(T, rows):
    """Keys drawn from a few distinct rows: scores tie exactly in fp32 and
    fp64, so the selection must equal the oracle's bit for bit."""
    g = torch.Generator(device="cpu").manual_seed(9)
    topk = 2048
    base = torch.randn((rows, 128), generator=g).to(torch.bfloat16)
    pick = torch.randint(0, rows, (T,), generator=g)
    ik = base[pick].contiguous()
    iq = torch.randn((1, 32, 128), generator=g).to(torch.bfloat16)
    w = torch.randn((1, 32), generator=g)
    cu = torch.tensor([0, T])
    idx = mla.dsa_index_topk(iq.to(DEV), ik.to(DEV), w.to(DEV), cu.to(DEV), T, topk)
    mla.check_device_status()
    ref = oracle.dsa_topk(oracle.dsa_index_scores(iq, ik, w, cu), cu, topk)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)


def test_index_topk_all_equal_scores():
    T, topk = 5000, 2048
    ik = torch.ones((T, 128), dtype=torch.bfloat16)
    iq = torch.ones((1, 32, 128), dtype=torch.bfloat16)
    w = torch.ones((1, 32))
    cu = torch.tensor([0, T])
    idx = mla.dsa_index_topk(iq.to(DEV), ik.to(DEV), w.to(DEV), cu.to(DEV), T, topk)
    mla.check_device_status()
    np.testing.assert_array_equal(idx.cpu().numpy()[0], np.arange(topk))


def test_index_topk_negative_weights_and_zero_scores():
    """Negative head weights make scores negative; all-negative dots give 0."""
    g = torch.Generator(device="cpu").manual_seed(10)
    T, topk = 3000, 512
    ik = torch.randn((T, 128), generator=g).to(torch.bfloat16)
    iq = torch.randn((1, 32, 128), generator=g).to(torch.bfloat16)
    w = -torch.rand((1, 32), generator=g)
    cu = torch.tensor([0, T])
    idx = mla.dsa_index_topk(iq.to(DEV), ik.to(DEV), w.to(DEV), cu.to(DEV), T, topk)
    mla.check_device_status()
    s64 = oracle.dsa_index_scores(iq, ik, w, cu)
    check_selection(idx, None, s64, [T], topk)


def test_index_topk_short_sequences_under_a_long_bound():
    """A bound above 8 x 16,384 positions selects the general top-k kernel even
    for sequences that would fit the register-resident one."""
    lengths = [5000, 20000, 2100]
    d = mi.make_dsa(lengths, device=DEV, config=53, with_main=False)
    idx, sc = run_index(d, lengths, 2048, max_seqlen=200000)
    s64 = oracle.dsa_index_scores(d.index_q, d.index_k, d.w, mi.cu_from_lengths(lengths))
    check_selection(idx, sc, s64, lengths, 2048)


def test_index_topk_is_deterministic():
    lengths = [70000, 9000]
    d = mi.make_dsa(lengths, device=DEV, config=52, with_main=False)
    a, _ = run_index(d, lengths, 2048)
    b, _ = run_index(d, lengths, 2048)
    assert torch.equal(a, b)


def test_index_topk_length_outside_bound_is_reported():
    lengths = [3000, 5000]
    d = mi.make_dsa(lengths, device=DEV, config=53, with_main=False)
    idx = torch.zeros((2, 256), dtype=torch.int32, device=DEV)
    mla.dsa_index_topk(d.index_q, d.index_k, d.w, mi.cu_from_lengths(lengths).to(DEV), 4000, 256,
                       topk_idx=idx)
    with pytest.raises(mla.MlaError) as ei:
        mla.check_device_status()
    assert ei.value.status == _lib.MLA_ERR_INVALID_ARG
    assert torch.all(idx[1] == -1)
    s64 = oracle.dsa_index_scores(d.index_q[:1], d.index_k[:3000], d.w[:1], torch.tensor([0, 3000]))
    check_selection(idx[:1], None, s64, [3000], 256)


def test_dsa_decode_path_small():
    """Indexer -> top-k -> sparse gated decode against the oracle's own selection."""
    lengths = [9000, 2500, 700]
    topk = 1024
    d = mi.make_dsa(lengths, H=8, device=DEV, config=54)
    m = d.main
    idx, _ = run_index(d, lengths, topk)
    out = mla.dsa_sparse_decode(m.q, m.k, m.v, m.cu_seqlens, idx, gate=m.gate, scale=m.scale)
    mla.check_device_status()
    cu = mi.cu_from_lengths(lengths)
    sel = oracle.dsa_topk(oracle.dsa_index_scores(d.index_q, d.index_k, d.w, cu), cu, topk)
    ref = oracle.dsa_sparse_decode(m.q, m.k, m.v, m.cu_seqlens, sel, m.gate, m.scale)
    assert_close(out, ref)


def test_dsa_decode_full_size_sampled():
    """B=8, T=131072, 32 index heads, top-2048, 96-head gated MLA (64 GB cache),
    in the launch configuration the benchmark times."""
    name = "dsa_decode_b8_t131072"
    w = mi.WORKLOADS[name]
    lengths = mi.workload_lengths(name)
    d = mi.make_dsa(lengths, H=w["H"], device=DEV, config=w["config"])
    m = d.main
    idx, sc = run_index(d, lengths, w["topk"])
    out = mla.dsa_sparse_decode(m.q, m.k, m.v, m.cu_seqlens, idx, gate=m.gate, scale=m.scale)
    mla.check_device_status()
    cu = mi.cu_from_lengths(lengths)
    s64 = oracle.dsa_index_scores(d.index_q, d.index_k, d.w, cu)
    check_selection(idx, sc, s64, lengths, w["topk"])
    sel = oracle.dsa_topk(s64, cu, w["topk"])
    for b in (0, 5):
        T = lengths[b]
        H = w["H"]
        for h in (0, 77):
            o = int(cu[b]) * H + h * T
            kb = m.k[o * 192:(o + T) * 192].view(T, 192)
            vb = m.v[o * 128:(o + T) * 128].view(T, 128)
            ref = oracle.dsa_sparse_decode(m.q[b:b + 1, h:h + 1], kb, vb, torch.tensor([0, T]),
                                           sel[b:b + 1], m.gate[b:b + 1, h * 128:(h + 1) * 128],
                                           m.scale)
            assert_close(out[b:b + 1, h * 128:(h + 1) * 128], ref, what=f"b{b} h{h}")
    del d, m
    torch.cuda.empty_cache()


def test_gather_probe_reads_exactly_the_selected_rows():
    """The measurement aid reads each selected (key, value) row pair once: the
    XOR of all its per-CTA words equals the XOR of every 32-bit word of the
    rows the selection names (entries -1 and past T_b skipped)."""
    lengths = [3000, 700, 1]
    H, topk = 4, 256
    d = mi.make_dsa(lengths, H=H, device=DEV, config=57)
    m = d.main
    g = torch.Generator(device="cpu").manual_seed(12)
    idx = torch.full((3, topk), -1, dtype=torch.int32)
    idx[0] = torch.randperm(3000, generator=g)[:topk].to(torch.int32)
    idx[1, :200] = torch.randperm(700, generator=g)[:200].to(torch.int32)
    idx[2, :1] = 0
    idx[1, 250] = 700                              # past the sequence: skipped
    sink = mla.gather_probe(m.k, m.v, m.cu_seqlens, idx.to(DEV), H)
    torch.cuda.synchronize()
    got = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
    k32 = m.k.view(torch.int32).cpu().numpy().view(np.uint32)
    v32 = m.v.view(torch.int32).cpu().numpy().view(np.uint32)
    want = np.uint32(0)
    cu = [0, 3000, 3700, 3701]
    for b, T in enumerate(lengths):
        for h in range(H):
            for s in idx[b].tolist():
                if 0 <= s < T:
                    row = cu[b] * H + h * T + s
                    want ^= np.bitwise_xor.reduce(k32[row * 96:(row + 1) * 96])
                    want ^= np.bitwise_xor.reduce(v32[row * 64:(row + 1) * 64])
    assert got == want


@pytest.mark.parametrize("lengths", [[300000, 2049], [1048576]])
def test_index_topk_long_contexts(lengths):
    """Sequences whose share of the 8-CTA top-k exceeds one 16,384-score
    shared-memory step (every pass then re-stages its scores from L2), up to
    the million-position context the DSA post's complexity section takes."""
    d = mi.make_dsa(lengths, device=DEV, config=58, with_main=False)
    idx, sc = run_index(d, lengths, 2048)
    cu = mi.cu_from_lengths(lengths)
    s64 = oracle.dsa_index_scores(d.index_q, d.index_k, d.w, cu)
    check_selection(idx, sc, s64, lengths, 2048)
    del d
    torch.cuda.empty_cache()
