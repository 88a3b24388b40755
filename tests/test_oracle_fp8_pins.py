"""Pins of the oracle's FP8 (e4m3) quantisation and FP8 index scores:

* the rounding step reproduces e4m3 codes worked out by hand from the format
  (sign, 4 exponent bits with bias 7, 3 mantissa bits; largest finite 448);
* a quantised row has its largest element at exactly +-448 codes, every
  dequantised value within half an e4m3 step (relative 2^-4) of the input,
  and an all-zero row has scale 0;
* when every query and key feature is already an e4m3 value and the row
  maxima are 448, the FP8 scores equal the bf16-path scores exactly; when
  such rows are further multiplied by per-row powers of two, the scales are
  exactly those powers and the FP8 scores still equal the exact scores (so
  a dropped or misapplied key or query scale fails).
"""
import numpy as np

import oracle
from test_oracle_pins import bf16_like

RNG = np.random.default_rng(808)


def test_hand_computed_e4m3_codes():
    # value -> code: 448 = 1.75*2^8 -> 0 1111 110; 1 = 2^0 -> 0 0111 000;
    # -2 -> 1 1000 000; 2^-6 (smallest normal) -> 0 0001 000;
    # 2^-9 (smallest subnormal) -> 0 0000 001; 0.3125 = 1.25*2^-2 -> 0 0101 010
    vals = np.array([[448.0, 1.0, -2.0, 2.0 ** -6, 2.0 ** -9, 0.3125, 0.0, -448.0]])
    codes, scale = oracle.quantize_e4m3_rows(vals)
    assert scale[0] == np.float32(1.0)
    assert list(codes[0]) == [0x7E, 0x38, 0xC0, 0x08, 0x01, 0x2A, 0x00, 0xFE]
    np.testing.assert_array_equal(oracle.e4m3_values(codes), vals)


def test_rounding_to_nearest_even_between_codes():
    # 1.0625 lies halfway between 1.0 (mantissa 000) and 1.125 (001): even -> 1.0;
    # 1.1875 halfway between 1.125 (001) and 1.25 (010): even -> 1.25
    vals = np.array([[448.0, 1.0625, 1.1875, 0.0]])
    codes, _ = oracle.quantize_e4m3_rows(vals)
    np.testing.assert_array_equal(oracle.e4m3_values(codes)[0, 1:3], [1.0, 1.25])


def test_quantised_rows_bounds():
    x = bf16_like((64, 128), RNG) * np.exp(RNG.normal(size=(64, 1)))
    x[5] = 0.0
    codes, scale = oracle.quantize_e4m3_rows(x)
    deq = oracle.e4m3_values(codes) * scale.astype(np.float64)[:, None]
    assert scale[5] == 0 and not codes[5].any()
    for r in range(64):
        if r == 5:
            continue
        j = np.argmax(np.abs(x[r]))
        assert abs(oracle.e4m3_values(codes[r:r + 1, j:j + 1])[0, 0]) == 448.0
        big = np.abs(x[r]) >= 2.0 ** -6 * scale[r]
        rel = np.abs(deq[r][big] - x[r][big]) / np.abs(x[r][big])
        assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)


def test_fp8_scores_equal_bf16_scores_on_representable_inputs():
    grid = oracle.e4m3_values(np.arange(0, 0x7E, dtype=np.uint8).reshape(1, -1))[0]
    grid = np.concatenate([grid, -grid])
    B, T = 3, 40
    q = RNG.choice(grid, size=(B, 32, 128))
    q[..., 0] = 448.0
    k = RNG.choice(grid, size=(B * T, 128))
    k[:, 0] = 448.0
    w = RNG.normal(size=(B, 32))
    cu = np.arange(0, B * T + 1, T, dtype=np.int64)
    k8, ks = oracle.quantize_e4m3_rows(k)
    assert (ks == 1.0).all()
    got = oracle.dsa_index_scores_fp8(q, k8, ks, w, cu)
    ref = oracle.dsa_index_scores(q, k, w, cu)
    np.testing.assert_array_equal(got, ref)


def test_fp8_scores_apply_each_scale_exactly():
    grid = oracle.e4m3_values(np.arange(0, 0x7E, dtype=np.uint8).reshape(1, -1))[0]
    grid = np.concatenate([grid, -grid])
    B, T = 2, 30
    q = RNG.choice(grid, size=(B, 32, 128))
    q[..., 0] = 448.0
    q *= 2.0 ** RNG.integers(-3, 4, size=(B, 32, 1))
    k = RNG.choice(grid, size=(B * T, 128))
    k[:, 0] = 448.0
    kpow = 2.0 ** RNG.integers(-4, 5, size=(B * T, 1))
    k *= kpow
    w = RNG.normal(size=(B, 32))
    cu = np.arange(0, B * T + 1, T, dtype=np.int64)
    k8, ks = oracle.quantize_e4m3_rows(k)
    np.testing.assert_array_equal(ks, kpow[:, 0].astype(np.float32))
    assert len(np.unique(ks)) > 1
    got = oracle.dsa_index_scores_fp8(q, k8, ks, w, cu)
    ref = oracle.dsa_index_scores(q, k, w, cu)
    np.testing.assert_array_equal(got, ref)


def test_latent_record_layout():
    """Byte layout of the 656-byte record: codes of features 0..511 first,
    then the four group scales (little-endian fp32), then the 64 bf16
    shared-key features, bit for bit."""
    import torch
    x = bf16_like((3, 576), RNG)
    x[1, 128:256] = 0.0                            # a zero group: scale 0, codes 0
    rec = oracle.quantize_latent_records(x)
    assert rec.shape == (3, 656)
    codes, scale = oracle.quantize_e4m3_rows(x[:, :512].reshape(12, 128))
    np.testing.assert_array_equal(rec[:, :512], codes.reshape(3, 512))
    np.testing.assert_array_equal(rec[:, 512:528].copy().view("<f4").reshape(12), scale)
    assert scale[5] == 0 and not rec[1, 128:256].any()
    rope = torch.from_numpy(x[:, 512:].astype(np.float32)).to(torch.bfloat16)
    np.testing.assert_array_equal(rec[:, 528:], rope.view(torch.uint8).numpy())
    deq = oracle.dequantize_latent_records(rec)
    np.testing.assert_array_equal(deq[:, 512:], x[:, 512:])
    rel = np.abs(deq[:, :512] - x[:, :512]) / np.maximum(np.abs(x[:, :512]), 1e-30)
    big = np.abs(x[:, :512]) >= 2.0 ** -6 * np.repeat(scale.reshape(3, 4), 128, axis=1)
    assert rel[big].max() <= 2.0 ** -4 * (1 + 1e-6)


def test_fp8_latent_decode_equals_bf16_on_representable_cache():
    grid = oracle.e4m3_values(np.arange(0, 0x7E, dtype=np.uint8).reshape(1, -1))[0]
    grid = np.concatenate([grid, -grid])
    lengths, H = [5, 9], 2
    N = sum(lengths)
    ckv = bf16_like((N, 576), RNG)
    ckv[:, :512] = RNG.choice(grid, size=(N, 512))
    ckv[:, :512:128] = 448.0                       # every group's maximum is 448: scale 1
    wk = bf16_like((H, 128, 512), RNG) / 64
    wv = bf16_like((H, 128, 512), RNG) / 64
    q = bf16_like((2, H, 192), RNG)
    g = bf16_like((2, H * 128), RNG)
    cu = np.array([0, 5, 14], dtype=np.int64)
    rec = oracle.quantize_latent_records(ckv)
    np.testing.assert_array_equal(oracle.dequantize_latent_records(rec), ckv)
    got = oracle.mla_decode_latent_fp8(q, rec, cu, wk, wv, g, 192 ** -0.5)
    ref = oracle.mla_decode_latent(q, ckv, cu, wk, wv, g, 192 ** -0.5)
    np.testing.assert_array_equal(got, ref)
