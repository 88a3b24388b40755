"""GPU parity of mla_decode and dsa_sparse_decode against the fp64 oracle,
called through the C ABI (via the package's ctypes binding)."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle
from mla_family_attention_gb300 import _lib
import mla_family_attention_gb300 as mla
from parity import assert_close, decode_slice

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_decode(dec, max_seqlen=None):
    out = mla.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, max_seqlen or max(dec.lengths),
                         gate=dec.gate, scale=dec.scale)
    mla.check_device_status()
    return out


@pytest.mark.parametrize("lengths,H,gated", [
    ([1], 1, True),
    ([64], 2, True),
    ([65, 63, 1, 130], 3, True),           # ragged tails around one stage
    ([1000, 3000, 77], 4, False),           # several chunks, no gate
    ([5000, 4097], 2, True),                # chunk boundaries (chunk shrinks with few items)
])
def test_decode_small_matches_oracle(lengths, H, gated):
    dec = mi.make_decode(lengths, H, gated, device=DEV, config=11)
    out = run_decode(dec)
    ref = oracle.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, dec.gate, dec.scale)
    assert_close(out, ref, what=f"decode {lengths}")


def test_decode_max_seqlen_larger_than_needed():
    dec = mi.make_decode([100, 200], 2, True, device=DEV, config=12)
    out = run_decode(dec, max_seqlen=50000)
    ref = oracle.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, dec.gate, dec.scale)
    assert_close(out, ref)


def test_decode_is_deterministic():
    dec = mi.make_decode([3000, 1234, 999], 4, True, device=DEV, config=13)
    a = run_decode(dec)
    b = run_decode(dec)
    assert torch.equal(a, b)


def test_decode_length_outside_bound_is_reported_not_faulted():
    dec = mi.make_decode([100, 200], 2, True, device=DEV, config=14)
    out = torch.full((2, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    mla.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, 150, gate=dec.gate, out=out)
    with pytest.raises(mla.MlaError) as ei:
        mla.check_device_status()
    assert ei.value.status == _lib.MLA_ERR_INVALID_ARG
    ref = oracle.mla_decode(dec.q[:1], dec.k[:100 * 2 * 192], dec.v[:100 * 2 * 128],
                            torch.tensor([0, 100]), dec.gate[:1], dec.scale)
    assert_close(out[:1], ref)                         # the valid sequence is still right
    assert torch.all(out[1] == 7.0)                    # the invalid one is left untouched
    mla.check_device_status()                          # status was cleared


def test_decode_wait_timeout_is_reported_and_context_survives():
    dec = mi.make_decode([4096, 4096], 2, True, device=DEV, config=15)
    try:
        mla.debug_set(_lib.DEBUG_WAIT_LIMIT_NS, 20_000_000)   # 20 ms
        mla.debug_set(_lib.DEBUG_STALL_STAGE, 1)
        mla.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, 4096, gate=dec.gate)
        with pytest.raises(mla.MlaError) as ei:
            mla.check_device_status()
        assert ei.value.status == _lib.MLA_ERR_TIMEOUT
    finally:
        mla.debug_set(_lib.DEBUG_STALL_STAGE, -1)
        mla.debug_set(_lib.DEBUG_WAIT_LIMIT_NS, 0)
    out = run_decode(dec)
    ref = oracle.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, dec.gate, dec.scale)
    assert_close(out, ref)


def test_decode_full_size_uniform_sampled():
    """B=32, H=96, T=8192 in the launch configuration the benchmark times;
    sampled (b,h) rows checked against the oracle one by one."""
    name = "decode_b32_h96_t8192"
    w = mi.WORKLOADS[name]
    dec = mi.make_decode(mi.workload_lengths(name), w["H"], True, device=DEV, config=w["config"])
    out = run_decode(dec)
    rng = np.random.default_rng(7)
    for b, h in [(0, 0), (31, 95)] + [tuple(x) for x in rng.integers([0, 0], [32, 96], (6, 2))]:
        k, v = decode_slice(dec, b, h)
        ref = oracle.mla_decode(dec.q[b:b + 1, h:h + 1], k, v, torch.tensor([0, k.shape[0]]),
                                dec.gate[b:b + 1, h * 128:(h + 1) * 128], dec.scale)
        assert_close(out[b:b + 1, h * 128:(h + 1) * 128], ref, what=f"b{b} h{h}")
    del dec
    torch.cuda.empty_cache()


def test_decode_full_size_ragged_sampled():
    """B=64 ragged lengths U{1024..65536}, H=96 (about 131 GB of cache)."""
    name = "ragged_decode_b64_h96_t1024_65536"
    w = mi.WORKLOADS[name]
    lengths = mi.workload_lengths(name)
    dec = mi.make_decode(lengths, w["H"], True, device=DEV, config=w["config"])
    out = run_decode(dec, max_seqlen=w["hi"])
    longest = int(np.argmax(lengths))
    shortest = int(np.argmin(lengths))
    for b, h in [(longest, 0), (shortest, 95), (0, 17), (63, 50)]:
        k, v = decode_slice(dec, b, h)
        ref = oracle.mla_decode(dec.q[b:b + 1, h:h + 1], k, v, torch.tensor([0, k.shape[0]]),
                                dec.gate[b:b + 1, h * 128:(h + 1) * 128], dec.scale)
        assert_close(out[b:b + 1, h * 128:(h + 1) * 128], ref, what=f"b{b} h{h} T{lengths[b]}")
    del dec
    torch.cuda.empty_cache()


# ------------------------------ sparse decode ------------------------------
def random_selection(lengths, topk, seed, pad_frac=0.0):
    rng = np.random.default_rng(seed)
    idx = np.full((len(lengths), topk), -1, dtype=np.int32)
    for b, T in enumerate(lengths):
        n = min(T, topk)
        sel = rng.choice(T, size=n, replace=False).astype(np.int32)
        if pad_frac:
            sel[rng.random(n) < pad_frac] = -1
        idx[b, :n] = sel                               # unsorted on purpose
    return torch.from_numpy(idx)


@pytest.mark.parametrize("lengths,H,topk", [([10], 2, 16), ([300, 5000, 64], 3, 256),
                                            ([4096, 4096], 4, 2048), ([3000], 96, 2048)])
def test_sparse_decode_matches_oracle(lengths, H, topk):
    dec = mi.make_decode(lengths, H, True, device=DEV, config=21)
    idx = random_selection(lengths, topk, 5, pad_frac=0.1)
    out = mla.dsa_sparse_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, idx.to(DEV), gate=dec.gate)
    mla.check_device_status()
    ref = oracle.dsa_sparse_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, idx, dec.gate, dec.scale)
    assert_close(out, ref, what=f"sparse {lengths}")


def test_sparse_over_every_position_equals_decode():
    lengths = [700, 1500]
    dec = mi.make_decode(lengths, 4, True, device=DEV, config=22)
    idx = torch.full((2, 2048), -1, dtype=torch.int32)
    for b, T in enumerate(lengths):
        idx[b, :T] = torch.arange(T)
    sp = mla.dsa_sparse_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, idx.to(DEV), gate=dec.gate)
    de = run_decode(dec)
    ref = oracle.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, dec.gate, dec.scale)
    assert_close(sp, ref)
    assert_close(de, ref)


def test_sparse_bad_index_is_reported_and_skipped():
    lengths = [100]
    dec = mi.make_decode(lengths, 2, True, device=DEV, config=23)
    idx = torch.tensor([[5, 100, 7, -3, 9, -1]], dtype=torch.int32)
    out = mla.dsa_sparse_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, idx.to(DEV), gate=dec.gate)
    with pytest.raises(mla.MlaError) as ei:
        mla.check_device_status()
    assert ei.value.status == _lib.MLA_ERR_BAD_INDEX
    good = torch.tensor([[5, 7, 9]], dtype=torch.int32)
    ref = oracle.dsa_sparse_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, good, dec.gate, dec.scale)
    assert_close(out, ref)


def test_sparse_all_skipped_gives_zero():
    dec = mi.make_decode([50], 2, True, device=DEV, config=24)
    idx = torch.full((1, 64), -1, dtype=torch.int32, device=DEV)
    out = mla.dsa_sparse_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, idx, gate=dec.gate)
    mla.check_device_status()
    assert torch.all(out == 0)


def test_decode_one_million_positions():
    """One sequence of 1,048,576 cached positions (2 heads): 1,024 split-KV
    chunks per head merged by log-sum-exp."""
    from parity import assert_close
    T = 1 << 20
    dec = mi.make_decode([T, 300], 2, True, device="cuda", config=47)
    out = mla.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, T, gate=dec.gate, scale=dec.scale)
    mla.check_device_status()
    ref = oracle.mla_decode(dec.q, dec.k, dec.v, dec.cu_seqlens, dec.gate, dec.scale)
    assert_close(out, ref, what="decode over 1M positions")
    del dec
    torch.cuda.empty_cache()
