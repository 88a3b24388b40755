"""GPU parity of the DSA prefill path through the C ABI: per-token index
scores and top-k (dsa_prefill_index_topk) against the fp64 oracle, with the
same tie-band rule as the decode indexer (every position whose oracle score
is outside 1e-5 relative of the row's k-th score is classified identically)."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle
import mla_family_attention_gb300 as mla
from mla_family_attention_gb300 import _lib
from test_gpu_dsa import check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_index(d, topk):
    Tq = d.index_q.shape[0]
    idx = torch.empty((Tq, topk), dtype=torch.int32, device=DEV)
    sc = torch.empty((Tq, topk), dtype=torch.float32, device=DEV)
    mla.dsa_prefill_index_topk(d.index_q, d.index_k, d.w, topk, topk_idx=idx, topk_scores=sc)
    mla.check_device_status()
    return idx, sc


def oracle_row(d, i, topk):
    """Token i's index scores over its visible prefix and its top-k, both from
    the oracle on a one-token slice: with Tq = 1 and Tk = n = P+i+1 the token
    sits at position n-1 and sees every position of the slice, so the full
    [Tq, Tk] score matrix is never built."""
    Tq, Tk = d.index_q.shape[0], d.index_k.shape[0]
    n = Tk - Tq + i + 1
    s = oracle.dsa_prefill_index_scores(d.index_q[i:i + 1], d.index_k[:n], d.w[i:i + 1])
    return s[0], oracle.dsa_prefill_topk(s, topk)[0], n


def check_rows(d, idx, sc, topk, rows=None):
    """Every row equals the oracle's selection, or differs from it only by
    positions whose oracle score lies in the 1e-5 band around the k-th score
    (check_selection proves that for the rows that differ).  Returns the
    number of rows that differ."""
    Tq = d.index_q.shape[0]
    rows = range(Tq) if rows is None else rows
    got = idx.cpu().numpy()
    differ = 0
    for i in rows:
        s, ref, n = oracle_row(d, i, topk)
        check_selection(idx[i:i + 1], sc[i:i + 1], s, [n], topk)
        if not np.array_equal(got[i], ref):
            differ += 1
    return differ


@pytest.mark.parametrize("Tq,Tk,topk", [
    (1, 1, 2048),
    (7, 7, 4),            # short rows keep everything, later rows select
    (130, 130, 64),       # two query tiles of keys, ragged token block
    (300, 300, 2048),     # every row shorter than topk
    (100, 400, 128),      # cached prefix: token i sees 300+i+1 positions
    (64, 3000, 2048),     # rows longer than topk, several key tiles
])
def test_prefill_index_topk_matches_oracle(Tq, Tk, topk):
    d = mi.make_dsa_prefill(Tq, Tk, 8, device=DEV, config=91)
    idx, sc = run_index(d, topk)
    check_rows(d, idx, sc, topk)
    if Tq <= 130 and Tk <= 400:
        # the whole-prompt oracle call agrees with the per-token slices
        ref = oracle.dsa_prefill_topk(oracle.dsa_prefill_index_scores(d.index_q, d.index_k, d.w),
                                      topk)
        for i in range(Tq):
            assert np.array_equal(ref[i], oracle_row(d, i, topk)[1])


def test_prefill_index_topk_is_deterministic():
    d = mi.make_dsa_prefill(200, 2600, 8, device=DEV, config=92)
    a, _ = run_index(d, 256)
    b, _ = run_index(d, 256)
    assert torch.equal(a, b)


def test_prefill_index_rejects_bad_shapes():
    d = mi.make_dsa_prefill(8, 8, 8, device=DEV, config=93)
    lib = _lib.load()
    import ctypes
    P = ctypes.c_void_p
    st = lib.dsa_prefill_index_topk(P(d.index_q.data_ptr()), P(d.index_k.data_ptr()),
                                    P(d.w.data_ptr()), 8, 4, 32, 16, P(d.w.data_ptr()), None,
                                    None, 0, None)
    assert st == _lib.MLA_ERR_INVALID_ARG           # Tk < Tq
    st = lib.dsa_prefill_index_topk(P(d.index_q.data_ptr()), P(d.index_k.data_ptr()),
                                    P(d.w.data_ptr()), 8, 8, 32, 4096, P(d.w.data_ptr()), None,
                                    None, 0, None)
    assert st == _lib.MLA_ERR_UNSUPPORTED           # topk > 2048


def test_prefill_index_topk_full_size_sampled():
    """The 16384-token prompt of the DSA prefill workload; sampled rows
    (short, around the top-k boundary, long) against the oracle."""
    w = mi.WORKLOADS["dsa_prefill_t16384"]
    d = mi.make_dsa_prefill(w["T"], w["T"], 8, device=DEV, config=w["config"])
    idx, sc = run_index(d, w["topk"])
    rng = np.random.default_rng(11)
    rows = [0, 2046, 2047, 2048, 8191, w["T"] - 1] + [int(x) for x in rng.integers(2048, w["T"], 3)]
    check_rows(d, idx, sc, w["topk"], rows)
    del d, idx, sc
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Sparse prefill over the latent cache.  The selections given to the kernel
# come from the oracle (scores and top-k in fp64), so both sides attend over
# the same positions.
# ---------------------------------------------------------------------------
def oracle_selection(d, topk):
    return oracle.dsa_prefill_topk(oracle.dsa_prefill_index_scores(d.index_q, d.index_k, d.w),
                                   topk)


def run_sparse(d, idx):
    out = mla.mla_sparse_prefill_latent(d.q, d.ckv, idx, d.w_kc, d.w_vc, gate=d.gate,
                                        scale=d.scale)
    mla.check_device_status()
    return out


@pytest.mark.parametrize("Tq,Tk,H,topk", [
    (1, 1, 16, 2048),
    (150, 150, 96, 64),     # rows of 1..64 selected positions, several 64-key tiles
    (40, 700, 48, 256),     # cached prefix, four tiles per token
    (300, 300, 32, 2048),   # every token keeps its whole history (ragged tails)
])
def test_sparse_prefill_latent_matches_oracle(Tq, Tk, H, topk):
    from parity import assert_close
    d = mi.make_dsa_prefill(Tq, Tk, H, device=DEV, config=94)
    idx = oracle_selection(d, topk)
    out = run_sparse(d, torch.from_numpy(idx).to(DEV))
    ref = oracle.dsa_prefill_latent(d.q, d.ckv, d.w_kc, d.w_vc, idx, d.gate, d.scale)
    assert_close(out, ref, what=f"sparse prefill Tq{Tq} Tk{Tk} H{H} k{topk}")


def test_sparse_prefill_full_selection_is_dense_causal_prefill():
    from parity import assert_close
    Tq, H = 200, 16
    d = mi.make_dsa_prefill(Tq, Tq, H, device=DEV, config=95)
    idx = np.full((Tq, 256), -1, np.int32)
    for i in range(Tq):
        idx[i, :i + 1] = np.arange(i + 1)
    out = run_sparse(d, torch.from_numpy(idx).to(DEV))
    k, v = oracle.expand_latent(d.ckv, d.w_kc, d.w_vc)
    dense = oracle.mla_prefill(d.q.transpose(0, 1)[None], k[None], v[None], d.gate[None],
                               d.scale)[0]
    assert_close(out, dense, what="full selection")


def test_sparse_prefill_bad_index_is_reported():
    d = mi.make_dsa_prefill(4, 4, 16, device=DEV, config=96)
    idx = torch.tensor([[0, -1], [1, 0], [2, 3], [3, 0]], dtype=torch.int32, device=DEV)
    mla.mla_sparse_prefill_latent(d.q, d.ckv, idx, d.w_kc, d.w_vc, gate=d.gate, scale=d.scale)
    with pytest.raises(mla.MlaError) as e:          # token 2 may not see position 3
        mla.check_device_status()
    assert e.value.status == _lib.MLA_ERR_BAD_INDEX


def test_dsa_prefill_path_small():
    """Indexer + top-k + sparse prefill on the GPU against the oracle running
    the same three steps.  Every row whose GPU selection differs from the
    oracle's must differ only inside the tie band; those rows are then
    attended over the oracle's selection, so every row's output is compared."""
    from parity import assert_close
    Tq, Tk, H, topk = 96, 500, 32, 128
    d = mi.make_dsa_prefill(Tq, Tk, H, device=DEV, config=97)
    gidx, gsc = run_index(d, topk)
    check_rows(d, gidx, gsc, topk)
    idx = oracle_selection(d, topk)
    differ = ~(gidx.cpu().numpy() == idx).all(axis=1)
    used = gidx.clone()
    used[torch.from_numpy(differ).to(DEV)] = torch.from_numpy(idx[differ]).to(DEV)
    out = run_sparse(d, used)
    ref = oracle.dsa_prefill_latent(d.q, d.ckv, d.w_kc, d.w_vc, idx, d.gate, d.scale)
    assert_close(out, ref, what="DSA prefill path")


def test_sparse_prefill_full_size_sampled():
    """The 16384-token prompt: GPU indexer and sparse prefill; sampled rows
    use the oracle's selection (written into those rows of the index tensor),
    so the sampled outputs are compared like for like."""
    from parity import assert_close
    w = mi.WORKLOADS["dsa_prefill_t16384"]
    T, H, K = w["T"], w["H"], w["topk"]
    d = mi.make_dsa_prefill(T, T, H, device=DEV, config=w["config"])
    gidx, gsc = run_index(d, K)
    rows = [0, 5, 2047, 2048, 9000, T - 1]
    check_rows(d, gidx, gsc, K, rows)
    sel = np.stack([oracle_row(d, i, K)[1] for i in rows])
    gidx[rows] = torch.from_numpy(sel).to(DEV)
    out = run_sparse(d, gidx)
    ref = oracle.dsa_prefill_latent(d.q[rows], d.ckv, d.w_kc, d.w_vc,
                                    np.stack([sel[r] for r in range(len(rows))]), d.gate[rows],
                                    d.scale)
    assert_close(out[rows], ref, what="sparse prefill full size")
    del d, gidx, out
    torch.cuda.empty_cache()
