"""GPU parity of the FP8 index-key path through the C ABI: e4m3 row
quantisation (bit-exact codes and scales against the oracle) and the FP8
indexer (top-k sets against the oracle's scores on the dequantised keys and
queries, with the same tie band as the bf16 indexer)."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle
import mla_family_attention_gb300 as mla
from test_gpu_dsa import check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_quantize_index_keys_is_bit_exact():
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    x = torch.randn((1000, 128), generator=g) * torch.exp(torch.randn((1000, 1), generator=g) * 3)
    x[7] = 0.0
    x[8, :] = 1e-30                  # flushes below bf16's normal range are fine too
    x[9, 0] = 448.0
    x = x.to(torch.bfloat16).to(DEV)
    k8, ks = mla.dsa_quantize_index_keys(x)
    mla.check_device_status()
    codes, scale = oracle.quantize_e4m3_rows(x)
    assert np.array_equal(k8.cpu().numpy(), codes)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), scale.view(np.uint32))


def run_fp8(d, lengths, topk, k8, ks):
    B = len(lengths)
    idx = torch.empty((B, topk), dtype=torch.int32, device=DEV)
    sc = torch.empty((B, topk), dtype=torch.float32, device=DEV)
    mla.dsa_index_topk_fp8(d.index_q, k8, ks, d.w, mi.cu_from_lengths(lengths).to(DEV),
                           max(lengths), topk, topk_idx=idx, topk_scores=sc)
    mla.check_device_status()
    return idx, sc


@pytest.mark.parametrize("lengths,topk", [([300, 5000, 129], 64), ([100], 2048),
                                          ([4096, 4097, 1], 2048), ([20000], 512)])
def test_fp8_index_topk_matches_oracle(lengths, topk):
    d = mi.make_dsa(lengths, H=8, device=DEV, config=101, with_main=False)
    k8, ks = mla.dsa_quantize_index_keys(d.index_k)
    idx, sc = run_fp8(d, lengths, topk, k8, ks)
    cu = mi.cu_from_lengths(lengths)
    s64 = oracle.dsa_index_scores_fp8(d.index_q, k8, ks, d.w, cu)
    check_selection(idx, sc, s64, lengths, topk)


def test_fp8_selection_overlaps_bf16_selection():
    """Not a parity claim: e4m3 keys change scores by a few percent, so the
    FP8 top-k keeps most, not all, of the bf16 top-k."""
    lengths = [30000, 30000]
    d = mi.make_dsa(lengths, H=8, device=DEV, config=102, with_main=False)
    k8, ks = mla.dsa_quantize_index_keys(d.index_k)
    idx8, _ = run_fp8(d, lengths, 2048, k8, ks)
    idx16 = mla.dsa_index_topk(d.index_q, d.index_k, d.w, mi.cu_from_lengths(lengths).to(DEV),
                               30000, 2048)
    mla.check_device_status()
    for b in range(2):
        a, c = set(idx8[b].tolist()), set(idx16[b].tolist())
        assert len(a & c) >= 0.8 * 2048


def test_fp8_index_full_size_sampled():
    """B=8, T=131072 as the DSA decode workload; two sequences checked."""
    w = mi.WORKLOADS["dsa_index_fp8_b8_t131072"]
    lengths = [w["T"]] * w["B"]
    d = mi.make_dsa(lengths, H=8, device=DEV, config=w["config"], with_main=False)
    k8, ks = mla.dsa_quantize_index_keys(d.index_k)
    idx, sc = run_fp8(d, lengths, w["topk"], k8, ks)
    T = w["T"]
    for b in (0, w["B"] - 1):
        s64 = oracle.dsa_index_scores_fp8(d.index_q[b:b + 1], k8[b * T:(b + 1) * T],
                                          ks[b * T:(b + 1) * T], d.w[b:b + 1],
                                          torch.tensor([0, T]))
        check_selection(idx[b:b + 1], sc[b:b + 1], s64, [T], w["topk"])
    del d, k8, ks
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# FP8 latent cache records (656 bytes per position)
# ---------------------------------------------------------------------------
def test_quantize_latent_cache_is_bit_exact():
    d = mi.make_latent_decode([300, 77], 16, True, device=DEV, config=103)
    ckv = d.ckv.clone()
    ckv[5, 128:256] = 0                                  # a zero group
    rec = mla.mla_quantize_latent_cache(ckv)
    mla.check_device_status()
    assert np.array_equal(rec.cpu().numpy(), oracle.quantize_latent_records(ckv))


@pytest.mark.parametrize("lengths,H", [([1, 63, 64, 65, 700], 96), ([2000], 16),
                                       (mi.ragged_lengths(40, 1, 3000, 104), 96)])
def test_fp8_latent_decode_matches_oracle(lengths, H):
    from parity import assert_close
    d = mi.make_latent_decode(lengths, H, True, device=DEV, config=104)
    rec = mla.mla_quantize_latent_cache(d.ckv)
    out = mla.mla_decode_latent_fp8(d.q, rec, d.cu_seqlens, max(lengths), d.w_kc, d.w_vc,
                                    gate=d.gate, scale=d.scale)
    mla.check_device_status()
    heads = list(range(H)) if len(lengths) < 10 else [0, 41, 95]
    cols = np.concatenate([np.arange(h * 128, (h + 1) * 128) for h in heads])
    ref = oracle.mla_decode_latent_fp8(d.q[:, heads], rec, d.cu_seqlens, d.w_kc[heads],
                                       d.w_vc[heads], d.gate[:, cols], d.scale)
    assert_close(out[:, cols], ref, what=f"fp8 latent decode {len(lengths)} seqs H{H}")


def test_fp8_sparse_prefill_matches_oracle():
    from parity import assert_close
    Tq, Tk, H, topk = 120, 600, 32, 128
    d = mi.make_dsa_prefill(Tq, Tk, H, device=DEV, config=105)
    idx = oracle.dsa_prefill_topk(oracle.dsa_prefill_index_scores(d.index_q, d.index_k, d.w),
                                  topk)
    rec = mla.mla_quantize_latent_cache(d.ckv)
    out = mla.mla_sparse_prefill_latent_fp8(d.q, rec, torch.from_numpy(idx).to(DEV), d.w_kc,
                                            d.w_vc, gate=d.gate, scale=d.scale)
    mla.check_device_status()
    ref = oracle.dsa_prefill_latent(d.q, oracle.dequantize_latent_records(rec), d.w_kc, d.w_vc,
                                    idx, d.gate, d.scale)
    assert_close(out, ref, what="fp8 sparse prefill")


def test_fp8_latent_decode_full_size_sampled():
    from parity import assert_close
    w = mi.WORKLOADS["latent_decode_fp8_b32_h96_t8192"]
    T, B = w["T"], w["B"]
    d = mi.make_latent_decode([T] * B, w["H"], True, device=DEV, config=w["config"])
    rec = mla.mla_quantize_latent_cache(d.ckv)
    out = mla.mla_decode_latent_fp8(d.q, rec, d.cu_seqlens, T, d.w_kc, d.w_vc, gate=d.gate,
                                    scale=d.scale)
    mla.check_device_status()
    heads = [0, 48, 95]
    cols = np.concatenate([np.arange(h * 128, (h + 1) * 128) for h in heads])
    for b in (0, B - 1):
        ref = oracle.mla_decode_latent_fp8(d.q[b:b + 1, heads], rec[b * T:(b + 1) * T],
                                           torch.tensor([0, T]), d.w_kc[heads], d.w_vc[heads],
                                           d.gate[b:b + 1, cols], d.scale)
        assert_close(out[b:b + 1, cols], ref, what=f"fp8 latent full b{b}")
    del d, rec, out
    torch.cuda.empty_cache()
