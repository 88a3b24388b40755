"""fp64 CPU oracle for Gated MLA / Gated DSA attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library's GPU path neither imports
it nor shares code with it.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64, OpenMP over
independent rows); this module builds it with gcc, converts inputs to
contiguous float64 arrays and calls it through ctypes. Each wrapper names the
passage it follows in the C file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_I32 = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False, extra_flags=(), out: str | None = None,
          src: str | None = None) -> str:
    """Compile the oracle with gcc (no -ffast-math, no FMA contraction)."""
    out = out or _LIB
    src = src or _SRC
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            # MLA_ORACLE_LIB lets the mutation test point the pins at a planted-bug build
            _lib = _bind(ctypes.CDLL(os.environ.get("MLA_ORACLE_LIB") or build()))
    return _lib


def _bind(lib):
    lib.orc_set_threads.argtypes = [ctypes.c_int]
    lib.orc_set_threads.restype = ctypes.c_int
    lib.orc_mla_prefill.argtypes = [_D, _D, _D, _D, _D] + [ctypes.c_int] * 6 + [ctypes.c_double]
    lib.orc_mla_decode.argtypes = [_D, _D, _D, _I64] + [ctypes.c_int] * 4 + [_D, _D, ctypes.c_double]
    lib.orc_attention_probs.argtypes = [_D, _D, _D, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_double, _D, _D]
    lib.orc_dsa_index_scores.argtypes = [_D, _D, _D, _I64, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, _D]
    lib.orc_dsa_topk.argtypes = [_D, _I64, ctypes.c_int, ctypes.c_int, _I32]
    lib.orc_dsa_sparse_decode.argtypes = [_D, _D, _D, _I64, _I32] + [ctypes.c_int] * 5 + \
        [_D, _D, ctypes.c_double]
    for f in ("orc_mla_prefill", "orc_mla_decode", "orc_attention_probs",
              "orc_dsa_index_scores", "orc_dsa_topk", "orc_dsa_sparse_decode"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _f64(x) -> np.ndarray:
    """Exact widening of bf16/fp32 (torch or numpy) to a contiguous float64 array."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int64)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a, t=_D):
    return None if a is None else a.ctypes.data_as(t)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def set_threads(n: int = 0, lib=None) -> int:
    """Set the OpenMP thread count (0 keeps the default); returns the count in use."""
    return (lib or load()).orc_set_threads(int(n))


def mla_prefill(q, k, v, gate, scale: float, lib=None) -> np.ndarray:
    """Causal gated MLA prefill; returns out [B,Tq,H*Dv] in float64."""
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gate)
    B, H, Tq, Dqk = q.shape
    Tk, Dv = k.shape[2], v.shape[3]
    if k.shape != (B, H, Tk, Dqk) or v.shape != (B, H, Tk, Dv):
        raise ValueError("prefill shape mismatch")
    if g is not None and g.shape != (B, Tq, H * Dv):
        raise ValueError("gate shape mismatch")
    out = np.empty((B, Tq, H * Dv))
    _check((lib or load()).orc_mla_prefill(_p(q), _p(k), _p(v), _p(g), _p(out), B, H, Tq, Tk,
                                           Dqk, Dv, float(scale)), "prefill")
    return out


def mla_decode(q, k, v, cu_seqlens, gate, scale: float, lib=None) -> np.ndarray:
    """Decode over the packed cache; returns out [B,H*Dv] in float64."""
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gate)
    cu = _i64(cu_seqlens)
    B, H, Dqk = q.shape
    Dv = v.size // (int(cu[-1]) * H)
    if k.size != int(cu[-1]) * H * Dqk:
        raise ValueError("decode cache size mismatch")
    out = np.empty((B, H * Dv))
    _check((lib or load()).orc_mla_decode(_p(q), _p(k), _p(v), _p(cu, _I64), B, H, Dqk, Dv,
                                          _p(g), _p(out), float(scale)), "decode")
    return out


def attention_probs(q, k, v, scale: float, lib=None):
    """One attention row over all n keys: returns (z [Dv], p [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, Dqk = k.shape
    Dv = v.shape[1]
    z, p = np.empty(Dv), np.empty(n)
    _check((lib or load()).orc_attention_probs(_p(q), _p(k), _p(v), n, Dqk, Dv, float(scale),
                                               _p(z), _p(p)), "probs")
    return z, p


def dsa_index_scores(index_q, index_k, w, cu_seqlens, lib=None) -> np.ndarray:
    """Packed index scores [cu[B]] in float64."""
    iq, ik, ww = _f64(index_q), _f64(index_k), _f64(w)
    cu = _i64(cu_seqlens)
    B, NH, Di = iq.shape
    out = np.empty(int(cu[-1]))
    _check((lib or load()).orc_dsa_index_scores(_p(iq), _p(ik), _p(ww), _p(cu, _I64), B, NH, Di,
                                                _p(out)), "index scores")
    return out


def dsa_topk(scores, cu_seqlens, topk: int, lib=None) -> np.ndarray:
    """Top-k positions per sequence, ascending, -1 padded: int32 [B,topk]."""
    s = _f64(scores)
    cu = _i64(cu_seqlens)
    B = cu.size - 1
    idx = np.empty((B, topk), dtype=np.int32)
    _check((lib or load()).orc_dsa_topk(_p(s), _p(cu, _I64), B, int(topk), _p(idx, _I32)), "topk")
    return idx


def dsa_sparse_decode(q, k, v, cu_seqlens, idx, gate, scale: float, lib=None) -> np.ndarray:
    """Gated MLA over the selected positions only; returns out [B,H*Dv]."""
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(gate)
    cu = _i64(cu_seqlens)
    ix = _i32(idx)
    B, H, Dqk = q.shape
    topk = ix.shape[1]
    Dv = v.size // (int(cu[-1]) * H)
    out = np.empty((B, H * Dv))
    _check((lib or load()).orc_dsa_sparse_decode(_p(q), _p(k), _p(v), _p(cu, _I64), _p(ix, _I32),
                                                 topk, B, H, Dqk, Dv, _p(g), _p(out),
                                                 float(scale)), "sparse decode")
    return out


# ---------------------------------------------------------------------------
# KV-cache update and the attention calls that follow it.  The pages' cache
# grows by concatenation on the sequence axis (Kimi K2 "KV cache" page, the
# update step: the new keys and values are appended after the cached ones and
# the full cache is returned for attention).  The library keeps a cache of
# fixed capacity instead; these functions state what such a cache holds after
# an append, then run the attention definitions above on the concatenated keys.
# ---------------------------------------------------------------------------
def _host(x) -> np.ndarray:
    """Any torch tensor (bf16 as raw 16-bit patterns) or array -> numpy array."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu")
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.numpy()
    return np.asarray(x)


def cache_append(k_cache, v_cache, k_new, v_new, start):
    """Caches [B,H,cap,D] after writing the Tn new rows of every (b, h) at
    positions start_b .. start_b+Tn-1: for each b, the prefix before start_b,
    then the new rows, then whatever followed them before.  Works on the raw
    element patterns, so the result is exact for any dtype.  `start` is an int
    or a length-B sequence."""
    kc, vc, kn, vn = (_host(x) for x in (k_cache, v_cache, k_new, v_new))
    B, Tn = kc.shape[0], kn.shape[2]
    starts = [int(start)] * B if np.ndim(_host(start)) == 0 else [int(s) for s in _host(start)]
    k_out, v_out = [], []
    for b in range(B):
        s = starts[b]
        if s < 0 or s + Tn > kc.shape[2]:
            raise ValueError("append past the cache capacity")
        k_out.append(np.concatenate([kc[b, :, :s], kn[b], kc[b, :, s + Tn:]], axis=1))
        v_out.append(np.concatenate([vc[b, :, :s], vn[b], vc[b, :, s + Tn:]], axis=1))
    return np.stack(k_out), np.stack(v_out)


def mla_prefill_chunk(q, k_cache, v_cache, k_new, v_new, P: int, gate, scale: float,
                      lib=None) -> np.ndarray:
    """Chunked prefill: Tq new tokens after P cached ones.  The key set is the
    first P cached positions followed by the new keys (the concatenation), and
    the queries attend causally with bottom-right alignment (query i sits at
    absolute position P+i).  Returns out [B,Tq,H*Dv] in float64."""
    kc, vc = _f64(k_cache), _f64(v_cache)
    k = np.concatenate([kc[:, :, :P], _f64(k_new)], axis=2)
    v = np.concatenate([vc[:, :, :P], _f64(v_new)], axis=2)
    return mla_prefill(q, k, v, gate, scale, lib=lib)


def mla_decode_cached(q, k_cache, v_cache, lengths, k_new, v_new, gate, scale: float,
                      lib=None) -> np.ndarray:
    """Decode over fixed-capacity caches: sequence b's keys are its first
    lengths[b] cached positions, followed by the current token's key when
    k_new is given.  Packs them back to back and runs the decode definition."""
    kc, vc = _f64(k_cache), _f64(v_cache)
    kn, vn = _f64(k_new), _f64(v_new)
    lens = [int(x) for x in _i64(lengths)]
    ks, vs, cu = [], [], [0]
    for b, L in enumerate(lens):
        kb, vb = kc[b, :, :L], vc[b, :, :L]
        if kn is not None:
            kb = np.concatenate([kb, kn[b]], axis=1)
            vb = np.concatenate([vb, vn[b]], axis=1)
        ks.append(kb.reshape(-1))
        vs.append(vb.reshape(-1))
        cu.append(cu[-1] + kb.shape[1])
    return mla_decode(q, np.concatenate(ks), np.concatenate(vs), np.array(cu, dtype=np.int64),
                      gate, scale, lib=lib)


# ---------------------------------------------------------------------------
# Absorbed-latent MLA (DSA post, eqs. (7)-(8) and the remark after eq. (10)
# that inference may absorb W^K into the query and apply W^V after attention).
# The cache holds, per position, the normalised 512-feature latent c_s and the
# 64-feature shared key r_s (576 values).  Head h's key and value are
#   k_{s,h} = [W^K_h c_s ; r_s] in R^192,   v_{s,h} = W^V_h c_s in R^128,
# with W^K_h, W^V_h in R^{128 x 512}.  The oracle expands the cache this way
# in float64 and runs the plain decode definition on the expanded keys; the
# absorbed evaluation order is the GPU path's business.
# ---------------------------------------------------------------------------
def expand_latent(ckv, w_kc, w_vc):
    """ckv [N,576], w_kc / w_vc [H,128,512] -> k [H,N,192], v [H,N,128] (float64)."""
    c, wk, wv = _f64(ckv), _f64(w_kc), _f64(w_vc)
    lat, rope = c[:, :512], c[:, 512:]
    H, N = wk.shape[0], c.shape[0]
    k = np.empty((H, N, 192))
    k[:, :, :128] = np.einsum("hdj,nj->hnd", wk, lat)
    k[:, :, 128:] = rope[None]
    v = np.einsum("hdj,nj->hnd", wv, lat)
    return k, v


def mla_decode_latent(q, ckv, cu_seqlens, w_kc, w_vc, gate, scale: float,
                      lib=None) -> np.ndarray:
    """Gated MLA decode over a packed latent cache (sequence b = rows
    cu[b]..cu[b+1]-1 of ckv [N,576]); q [B,H,192] is the expanded-form query.
    Returns out [B,H*128] in float64."""
    cu = _i64(cu_seqlens)
    c = _f64(ckv)
    ks, vs = [], []
    for b in range(cu.size - 1):
        kb, vb = expand_latent(c[cu[b]:cu[b + 1]], w_kc, w_vc)
        ks.append(kb.reshape(-1))
        vs.append(vb.reshape(-1))
    return mla_decode(q, np.concatenate(ks), np.concatenate(vs), cu, gate, scale, lib=lib)


# ---------------------------------------------------------------------------
# DSA prefill (DSA post, eqs. (5), (6), (9), (10) for every new token, and the
# complexity section: each token of a prompt scores its whole visible history
# and keeps its own top-k).  A prompt of Tq tokens follows P = Tk - Tq cached
# positions; token i sits at position P + i and sees positions 0..P+i.
# ---------------------------------------------------------------------------
def dsa_prefill_index_scores(index_q, index_k, w) -> np.ndarray:
    """scores [Tq, Tk] in float64: sum_h w[i,h] * max(0, q^I[i,h] . k^I[s]) for
    s <= P+i (eq. (5), the constant folded into w), -inf where s > P+i."""
    iq, ik, ww = _f64(index_q), _f64(index_k), _f64(w)
    Tq, Tk = iq.shape[0], ik.shape[0]
    dots = np.einsum("ihd,sd->ihs", iq, ik)
    scores = np.einsum("ih,ihs->is", ww, np.maximum(dots, 0.0))
    P = Tk - Tq
    mask = np.arange(Tk)[None, :] > (P + np.arange(Tq))[:, None]
    scores[mask] = -np.inf
    return scores


def dsa_prefill_topk(scores, topk: int, lib=None) -> np.ndarray:
    """Per token i, the top min(topk, P+i+1) visible positions (eq. (6)) by the
    same ranking as dsa_topk: int32 [Tq, topk], ascending, -1 padded."""
    s = _f64(scores)
    Tq, Tk = s.shape
    P = Tk - Tq
    out = np.empty((Tq, topk), dtype=np.int32)
    for i in range(Tq):
        n = P + i + 1
        out[i] = dsa_topk(s[i, :n], np.array([0, n], dtype=np.int64), topk, lib=lib)[0]
    return out


def dsa_prefill_latent(q, ckv, w_kc, w_vc, idx, gate, scale: float, lib=None) -> np.ndarray:
    """Gated MLA of every prompt token over its own selection (eq. (9) on S_i,
    then eq. (10)), with the keys and values expanded from the latent cache
    (eq. (8)).  q [Tq,H,192], ckv [Tk,576], idx [Tq,topk] (-1 entries skipped).
    Returns out [Tq,H*128] in float64."""
    qq = _f64(q)
    c = _f64(ckv)
    ix = _i32(idx)
    g = _f64(gate)
    Tq, H = qq.shape[0], qq.shape[1]
    out = np.empty((Tq, H * 128))
    for i in range(Tq):
        sel = ix[i][ix[i] >= 0]
        k, v = expand_latent(c[sel], w_kc, w_vc)
        cu = np.array([0, sel.size], dtype=np.int64)
        out[i] = mla_decode(qq[i:i + 1], k.reshape(-1), v.reshape(-1), cu,
                            None if g is None else g[i:i + 1], scale, lib=lib)[0]
    return out


# ---------------------------------------------------------------------------
# FP8 caches (DSA post, cache section): the index key of a position is 128
# one-byte FP8 features plus one fp32 scale (132 B); the main cache record is
# 512 FP8 latent features, four fp32 scales (one per 128 features) and the 64
# bf16 shared-key features (656 B).  The pages fix the byte counts, not the
# encoding; the reading taken: e4m3 (the "fn" variant, largest finite 448),
# scale = amax/448 per group in fp32, code = e4m3(x * (448/amax)) computed in
# fp32 and rounded to nearest even; an all-zero group has scale 0 and zero
# codes.  torch's float8_e4m3fn conversion is the rounding step.
# ---------------------------------------------------------------------------
def quantize_e4m3_rows(x):
    """Rows of x -> (codes uint8 [rows, cols], scale float32 [rows])."""
    import torch
    xf = _f64(x).astype(np.float32)
    xf = xf.reshape(-1, xf.shape[-1])
    amax = np.abs(xf).max(axis=1).astype(np.float32)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, np.float32(448.0) / amax, np.float32(0.0)).astype(np.float32)
    y = (xf * inv[:, None]).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    codes[amax == 0] = 0
    return codes, scale


def e4m3_values(codes) -> np.ndarray:
    """The real values of e4m3 codes (float64, exact)."""
    import torch
    c = np.ascontiguousarray(_host(codes), dtype=np.uint8)
    return torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dsa_index_scores_fp8(index_q, k8, kscale, w, cu_seqlens, lib=None) -> np.ndarray:
    """Index scores (eq. (5)) over FP8 index keys: the keys are the codes times
    their scale, the queries are quantised per (sequence, head) the same way
    and dequantised; the score is then computed in float64."""
    iq = _f64(index_q)
    B, NH, D = iq.shape
    qc, qs = quantize_e4m3_rows(iq.reshape(B * NH, D))
    q_deq = (e4m3_values(qc) * qs.astype(np.float64)[:, None]).reshape(B, NH, D)
    k_deq = e4m3_values(k8) * _f64(kscale)[:, None]
    return dsa_index_scores(q_deq, k_deq, w, cu_seqlens, lib=lib)


LATENT_RECORD_BYTES = 656   # 512 e4m3 codes + 4 fp32 scales + 64 bf16 shared-key features


def quantize_latent_records(ckv) -> np.ndarray:
    """Latent cache rows [N,576] (bf16) -> FP8 records uint8 [N,656] in the
    order the DSA post lists them: the 512 latent features as e4m3 codes in
    four groups of 128 (quantised like quantize_e4m3_rows), the four fp32
    group scales, then the 64 shared-key features unchanged (bf16)."""
    import torch
    c = _f64(ckv)
    N = c.shape[0]
    codes, scale = quantize_e4m3_rows(c[:, :512].reshape(N * 4, 128))
    rec = np.zeros((N, LATENT_RECORD_BYTES), dtype=np.uint8)
    rec[:, :512] = codes.reshape(N, 512)
    rec[:, 512:528] = scale.astype("<f4").reshape(N, 4).view(np.uint8)
    rope = torch.from_numpy(c[:, 512:].astype(np.float32)).to(torch.bfloat16)
    rec[:, 528:] = rope.view(torch.uint8).numpy().reshape(N, 128)
    return rec


def dequantize_latent_records(rec) -> np.ndarray:
    """FP8 records [N,656] -> the latent rows they stand for, [N,576] float64."""
    import torch
    r = np.ascontiguousarray(_host(rec), dtype=np.uint8)
    N = r.shape[0]
    codes = e4m3_values(r[:, :512]).reshape(N, 4, 128)
    scale = r[:, 512:528].copy().view("<f4").astype(np.float64).reshape(N, 4, 1)
    out = np.empty((N, 576))
    out[:, :512] = (codes * scale).reshape(N, 512)
    rope = torch.from_numpy(r[:, 528:].copy()).view(torch.bfloat16).to(torch.float64)
    out[:, 512:] = rope.numpy().reshape(N, 64)
    return out


def mla_decode_latent_fp8(q, rec, cu_seqlens, w_kc, w_vc, gate, scale: float,
                          lib=None) -> np.ndarray:
    """Latent decode over FP8 records: the records' latent rows, then the
    latent decode definition."""
    return mla_decode_latent(q, dequantize_latent_records(rec), cu_seqlens, w_kc, w_vc, gate,
                             scale, lib=lib)
