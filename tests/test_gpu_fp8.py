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
