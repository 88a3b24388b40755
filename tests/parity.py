"""Comparison helpers for GPU-vs-oracle parity (tolerances are the north-star
bar: bf16 I/O with fp32 accumulation against the fp64 oracle)."""
import numpy as np

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def to_f64(t):
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    got = to_f64(got) if hasattr(got, "detach") else np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= max_abs, f"{what}: max-abs {err.max():.3g} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean-abs {err.mean():.3g} > {mean_abs}"
    return float(err.max()), float(err.mean())


def decode_slice(dec, b, h):
    """K/V rows of one (sequence, head) of a packed decode cache (device tensors)."""
    import torch
    T = dec.lengths[b]
    o = int(dec.cu_seqlens[b].item()) * dec.H + h * T
    k = dec.k[o * 192:(o + T) * 192].view(T, 192)
    v = dec.v[o * 128:(o + T) * 128].view(T, 128)
    return k, v
