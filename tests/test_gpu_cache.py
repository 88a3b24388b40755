"""GPU parity of the cache-update path through the C ABI: in-place append
(bit-exact), chunked prefill over a fixed-capacity cache, and the decode step
over fixed-capacity caches, against the fp64 oracle.  Unused cache capacity
is filled with NaN throughout, so a kernel that reads past the live
positions shows up as NaN in the output."""
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


def bits(t):
    return t.detach().cpu().view(torch.int16).numpy()


def rand_bits(shape, seed):
    """bf16 tensor of arbitrary bit patterns (NaNs and infinities included)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randint(-32768, 32768, shape, generator=g, dtype=torch.int32).to(torch.int16)
    return x.view(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("B,H,Tn,cap,start", [
    (1, 1, 1, 1, 0),
    (2, 3, 5, 16, 11),             # fills the capacity exactly
    (1, 96, 1, 40, 7),             # one decode token, many heads
    (2, 4, 300, 1024, 129),        # a chunk at an odd offset
])
def test_append_uniform_start_is_bit_exact(B, H, Tn, cap, start):
    kc, vc = rand_bits((B, H, cap, 192), 1), rand_bits((B, H, cap, 128), 2)
    kn, vn = rand_bits((B, H, Tn, 192), 3), rand_bits((B, H, Tn, 128), 4)
    ek, ev = oracle.cache_append(kc, vc, kn, vn, start)
    mla.mla_cache_append(kn, vn, kc, vc, start)
    mla.check_device_status()
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)


def test_append_per_sequence_start_is_bit_exact():
    B, H, Tn, cap = 5, 3, 2, 64
    kc, vc = rand_bits((B, H, cap, 192), 5), rand_bits((B, H, cap, 128), 6)
    kn, vn = rand_bits((B, H, Tn, 192), 7), rand_bits((B, H, Tn, 128), 8)
    start = [0, 62, 17, 1, 33]
    ek, ev = oracle.cache_append(kc, vc, kn, vn, start)
    mla.mla_cache_append(kn, vn, kc, vc, torch.tensor(start, dtype=torch.int64, device=DEV))
    mla.check_device_status()
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)


def test_append_out_of_range_device_start_is_reported_and_skipped():
    B, H, Tn, cap = 2, 2, 3, 8
    kc, vc = rand_bits((B, H, cap, 192), 9), rand_bits((B, H, cap, 128), 10)
    kn, vn = rand_bits((B, H, Tn, 192), 11), rand_bits((B, H, Tn, 128), 12)
    before_k = bits(kc)
    ek, _ = oracle.cache_append(kc, vc, kn, vn, [1, 0])
    mla.mla_cache_append(kn, vn, kc, vc, torch.tensor([1, 6], dtype=torch.int64, device=DEV))
    with pytest.raises(mla.MlaError) as e:
        mla.check_device_status()
    assert e.value.status == _lib.MLA_ERR_INVALID_ARG
    got = bits(kc)
    assert np.array_equal(got[0], ek[0])          # the valid sequence was appended
    assert np.array_equal(got[1], before_k[1])    # the other one left alone


def test_append_host_checks():
    kc = torch.zeros((1, 1, 4, 192), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros((1, 1, 4, 128), dtype=torch.bfloat16, device=DEV)
    kn = torch.zeros((1, 1, 2, 192), dtype=torch.bfloat16, device=DEV)
    vn = torch.zeros((1, 1, 2, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_cache_append(kn, vn, kc, vc, 3)
    assert e.value.status == _lib.MLA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        mla.mla_cache_append(kn, vn[:, :, :1].contiguous(), kc, vc, 0)


def run_chunks(pf, chunks, cap):
    """Feed the prompt of `pf` through mla_prefill_chunk; returns the outputs
    of every chunk concatenated, the caches, and the oracle's rows."""
    B, H, T = pf.q.shape[0], pf.q.shape[1], pf.q.shape[2]
    kc, vc = mi.nan_filled((B, H, cap, 192), DEV), mi.nan_filled((B, H, cap, 128), DEV)
    outs, P = [], 0
    for n in chunks:
        sl = slice(P, P + n)
        g = pf.gate[:, sl].contiguous() if pf.gate is not None else None
        outs.append(mla.mla_prefill_chunk(pf.q[:, :, sl].contiguous(), pf.k[:, :, sl].contiguous(),
                                          pf.v[:, :, sl].contiguous(), kc, vc, P, gate=g,
                                          scale=pf.scale))
        P += n
    mla.check_device_status()
    return torch.cat(outs, dim=1), kc, vc


@pytest.mark.parametrize("B,H,chunks,cap,gated", [
    (1, 2, [300, 256, 144], 1024, True),     # ragged chunks, ragged tiles
    (2, 3, [1, 1, 130], 200, False),         # one-token chunks (decode-like)
    (1, 2, [128, 128, 128], 384, True),      # tile-aligned, capacity exactly full
    (1, 1, [77, 640], 1000, True),
])
def test_chunked_prefill_matches_oracle(B, H, chunks, cap, gated):
    T = sum(chunks)
    pf = mi.make_prefill(B, H, T, T, gated, device=DEV, config=71)
    out, kc, vc = run_chunks(pf, chunks, cap)
    assert torch.isfinite(out.float()).all()
    ref = oracle.mla_prefill(pf.q, pf.k, pf.v, pf.gate, pf.scale)
    assert_close(out, ref, what=f"chunks {chunks}")
    assert torch.equal(kc[:, :, :T], pf.k) and torch.equal(vc[:, :, :T], pf.v)
    assert torch.isnan(kc[:, :, T:].float()).all()


def test_tile_aligned_chunks_equal_one_prefill_bitwise():
    """With chunk boundaries on 128-row tiles every query tile meets the same
    key tiles in the same order as in one prefill over the whole prompt."""
    pf = mi.make_prefill(1, 4, 512, 512, True, device=DEV, config=72)
    out, _, _ = run_chunks(pf, [256, 128, 128], 640)
    whole = mla.mla_prefill(pf.q, pf.k, pf.v, pf.gate, scale=pf.scale)
    mla.check_device_status()
    assert torch.equal(out, whole)


def test_prefill_chunk_host_checks():
    pf = mi.make_prefill(1, 1, 8, 8, True, device=DEV, config=73)
    kc, vc = mi.nan_filled((1, 1, 10, 192), DEV), mi.nan_filled((1, 1, 10, 128), DEV)
    with pytest.raises(mla.MlaError) as e:      # P + Tq > capacity
        mla.mla_prefill_chunk(pf.q, pf.k, pf.v, kc, vc, 3, gate=pf.gate)
    assert e.value.status == _lib.MLA_ERR_INVALID_ARG


def test_chunked_prefill_full_size_sampled():
    """The 16384-token H=96 gated prompt in four 4096-token chunks, in the
    launch configuration the benchmark times; sampled rows against the oracle."""
    w = mi.WORKLOADS["chunked_prefill_b1_h96_t16384_c4096"]
    T, H, c = w["T"], w["H"], w["chunk"]
    pf = mi.make_prefill(1, H, T, T, True, device=DEV, config=w["config"])
    out, kc, vc = run_chunks(pf, [c] * (T // c), T)
    assert torch.equal(kc, pf.k) and torch.equal(vc, pf.v)
    rng = np.random.default_rng(5)
    rows = [0, c - 1, c, 2 * c + 1, T - 1] + [int(x) for x in rng.integers(0, T, 3)]
    for h in [0, H - 1, int(rng.integers(0, H))]:
        for i in rows:
            g = pf.gate[:, i:i + 1, h * 128:(h + 1) * 128]
            ref = oracle.mla_prefill(pf.q[:, h:h + 1, i:i + 1], pf.k[:, h:h + 1, :i + 1],
                                     pf.v[:, h:h + 1, :i + 1], g, pf.scale)
            assert_close(out[:, i:i + 1, h * 128:(h + 1) * 128], ref, what=f"h{h} row{i}")
    del pf, out, kc, vc
    torch.cuda.empty_cache()


@pytest.mark.parametrize("append", [True, False])
@pytest.mark.parametrize("lengths,H,cap", [([1, 700, 64, 129], 3, 800), ([5], 96, 8),
                                           ([1000, 3000], 2, 4096)])
def test_decode_cached_matches_oracle_and_packed_decode(lengths, H, cap, append):
    extra = 1 if append else 0
    cd = mi.make_capacity_decode(lengths, H, cap, True, device=DEV, config=74, append=append)
    cached = lengths
    seqlens = torch.tensor(cached, dtype=torch.int64, device=DEV)
    max_len = max(cached) + extra
    out = mla.mla_decode_cached(cd.q, cd.k_cache, cd.v_cache, seqlens, max_len,
                                k_new=cd.k_new, v_new=cd.v_new, gate=cd.gate, scale=cd.scale)
    mla.check_device_status()
    assert torch.isfinite(out.float()).all()
    ref = oracle.mla_decode_cached(cd.q, cd.k_cache, cd.v_cache, cached, cd.k_new, cd.v_new,
                                   cd.gate, cd.scale)
    assert_close(out, ref, what=f"cached decode {lengths} append={append}")
    # the same keys packed back to back give bitwise the same result
    dd = mi.make_decode([L + extra for L in cached], H, True, device=DEV, config=74)
    packed = mla.mla_decode(dd.q, dd.k, dd.v, dd.cu_seqlens, max_len, gate=dd.gate,
                            scale=dd.scale)
    mla.check_device_status()
    assert torch.equal(out, packed)
    if append:           # the current token landed at position lengths[b]
        for b, L in enumerate(cached):
            assert torch.equal(cd.k_cache[b, :, L], cd.k_new[b, :, 0])


def test_decode_cached_length_outside_capacity_is_reported():
    cd = mi.make_capacity_decode([4, 8], 2, 8, True, device=DEV, config=75, append=True)
    seqlens = torch.tensor([4, 8], dtype=torch.int64, device=DEV)   # second one is full
    out = torch.zeros((2, 2 * 128), dtype=torch.bfloat16, device=DEV)
    mla.mla_decode_cached(cd.q, cd.k_cache, cd.v_cache, seqlens, 8, k_new=cd.k_new,
                          v_new=cd.v_new, gate=cd.gate, out=out, scale=cd.scale)
    with pytest.raises(mla.MlaError) as e:
        mla.check_device_status()
    assert e.value.status == _lib.MLA_ERR_INVALID_ARG
    ref = oracle.mla_decode_cached(cd.q[:1], cd.k_cache[:1], cd.v_cache[:1], [4],
                                   cd.k_new[:1], cd.v_new[:1], cd.gate[:1], cd.scale)
    assert_close(out[:1], ref)
    assert not out[1].any()                        # skipped: left untouched


def test_decode_cached_full_size():
    """B=32, H=96: 8191 cached positions plus the appended current token, in
    the configuration the benchmark times; sampled heads against the oracle."""
    w = mi.WORKLOADS["decode_cached_b32_h96_t8192"]
    B, H, T = w["B"], w["H"], w["T"]
    cd = mi.make_capacity_decode([T - 1] * B, H, T, True, device=DEV, config=w["config"])
    seqlens = torch.full((B,), T - 1, dtype=torch.int64, device=DEV)
    out = mla.mla_decode_cached(cd.q, cd.k_cache, cd.v_cache, seqlens, T, k_new=cd.k_new,
                                v_new=cd.v_new, gate=cd.gate, scale=cd.scale)
    mla.check_device_status()
    for b in [0, B - 1]:
        for h in [0, 47, H - 1]:
            kb = torch.cat([cd.k_cache[b:b + 1, h:h + 1, :T - 1], cd.k_new[b:b + 1, h:h + 1]], 2)
            vb = torch.cat([cd.v_cache[b:b + 1, h:h + 1, :T - 1], cd.v_new[b:b + 1, h:h + 1]], 2)
            ref = oracle.mla_prefill(cd.q[b:b + 1, h:h + 1, None], kb, vb,
                                     cd.gate[b:b + 1, None, h * 128:(h + 1) * 128], cd.scale)
            assert_close(out[b:b + 1, h * 128:(h + 1) * 128], ref.reshape(1, 128),
                         what=f"b{b} h{h}")
    del cd, out
    torch.cuda.empty_cache()
