"""GB300 (sm_103a) Gated MLA / Gated DSA attention.

Thin PyTorch-facing binding of the C ABI in ``include/mla.h``: the functions
below check shapes, dtypes, devices and contiguity (raising ``ValueError``
on a mismatch, as the Kimi K2 modeling code does for a wrong attention-weight
shape), allocate outputs and workspace with torch when the caller does not
pass them, and call the library on the current CUDA stream. Every step of the
computation runs in the library's CUDA kernels; nothing here computes.

Entry points (names as in the C ABI):

* ``mla_prefill(q, k, v, gate)``            causal gated MLA prefill
* ``mla_decode(q, k, v, cu_seqlens, ...)``  split-KV gated MLA decode
* ``dsa_index_topk(index_q, index_k, w, cu_seqlens, ...)``  DSA indexer + top-k
* ``dsa_sparse_decode(q, k, v, cu_seqlens, topk_idx, ...)`` gated MLA over a selection
* ``mla_cache_append(k_new, v_new, k_cache, v_cache, start)``  in-place cache append
* ``mla_prefill_chunk(q, k_new, v_new, k_cache, v_cache, P)``  append + causal prefill
* ``mla_decode_cached(q, k_cache, v_cache, cache_seqlens, ...)`` decode step over
  fixed-capacity caches (optionally appending the current token first)
* ``mla_decode_latent(q, ckv, cu_seqlens, w_kc, w_vc, ...)`` decode over the absorbed
  576-feature latent cache
* ``dsa_prefill_index_topk(index_q, index_k, w, ...)``  per-token DSA index + top-k
* ``mla_sparse_prefill_latent(q, ckv, topk_idx, w_kc, w_vc, ...)`` every prompt token
  over its own selection of the latent cache
* ``dsa_quantize_index_keys(index_k)`` / ``dsa_index_topk_fp8(...)``  FP8 index keys
* ``mla_quantize_latent_cache(ckv)`` / ``mla_decode_latent_fp8(...)`` /
  ``mla_sparse_prefill_latent_fp8(...)``  656-byte FP8 latent cache records
"""
from __future__ import annotations

from . import _lib
from ._lib import MlaError  # noqa: F401

DQK, DV, INDEX_HEADS, INDEX_DIM, MAX_TOPK = 192, 128, 32, 128, 2048


def _torch():
    import torch
    return torch


def _need(t, name, dtype, shape=None, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} should be of size {tuple(shape)}, but is {tuple(t.shape)}")


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes_ptr(s.cuda_stream)


def ctypes_ptr(x):
    import ctypes
    return ctypes.c_void_p(int(x))


def _ptr(t):
    return None if t is None else ctypes_ptr(t.data_ptr())


def workspace_size(op: int, B: int = 1, H: int = 1, max_seqlen: int = 1, topk: int = 1) -> int:
    return int(_lib.load().mla_workspace_size(op, B, H, max_seqlen, topk))


def _workspace(ws, nbytes, device):
    torch = _torch()
    if nbytes == 0:
        return None, 0
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    return ws, ws.numel() * ws.element_size()


def default_scale() -> float:
    return DQK ** -0.5


def mla_prefill(q, k, v, gate=None, out=None, scale=None, ws=None, stream=None):
    """Causal gated MLA prefill.  q [B,H,Tq,192], k [B,H,Tk,192], v [B,H,Tk,128],
    gate [B,Tq,H*128] or None -> out [B,Tq,H*128] (bf16)."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4 or q.shape[3] != DQK:
        raise ValueError("q must be [B,H,Tq,192]")
    B, H, Tq, _ = q.shape
    Tk = k.shape[2] if k.dim() == 4 else -1
    if Tk < Tq:
        raise ValueError(f"the cache must hold the {Tq} new tokens (Tk={Tk} < Tq={Tq})")
    _need(k, "k", torch.bfloat16, (B, H, Tk, DQK), q.device)
    _need(v, "v", torch.bfloat16, (B, H, Tk, DV), q.device)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (B, Tq, H * DV), q.device)
    if out is None:
        out = torch.empty((B, Tq, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, Tq, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_PREFILL, B, H, Tk, 0)
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.mla_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out), B, H, Tq, Tk,
                               float(default_scale() if scale is None else scale), _ptr(ws), wsb,
                               _stream(stream)), lib)
    return out


def _check_cache(q, k, v, cu_seqlens, H, total):
    torch = _torch()
    _need(k, "k", torch.bfloat16, None, q.device)
    _need(v, "v", torch.bfloat16, None, q.device)
    _need(cu_seqlens, "cu_seqlens", torch.int64, (q.shape[0] + 1,), q.device)
    if total is not None:
        if k.numel() != total * H * DQK or v.numel() != total * H * DV:
            raise ValueError("packed cache size does not match cu_seqlens[-1]")


def mla_decode(q, k, v, cu_seqlens, max_seqlen: int, gate=None, out=None, scale=None,
               ws=None, stream=None, total_positions: int | None = None):
    """Split-KV gated MLA decode over a packed cache.  q [B,H,192]; k/v packed with
    sequence b = [H,T_b,D] from element cu[b]*H*D; gate [B,H*128] or None."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [B,H,192]")
    B, H, _ = q.shape
    _check_cache(q, k, v, cu_seqlens, H, total_positions)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (B, H * DV), q.device)
    if out is None:
        out = torch.empty((B, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_DECODE, B, H, int(max_seqlen), 0)
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.mla_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B, H, int(max_seqlen),
                              _ptr(gate), _ptr(out),
                              float(default_scale() if scale is None else scale), _ptr(ws), wsb,
                              _stream(stream)), lib)
    return out


def dsa_index_topk(index_q, index_k, w, cu_seqlens, max_seqlen: int, topk: int = MAX_TOPK,
                   topk_idx=None, topk_scores=None, ws=None, stream=None):
    """DSA indexer score + top-k.  index_q [B,32,128] bf16, index_k [cu[B],128] bf16,
    w [B,32] fp32 -> topk_idx [B,topk] int32 (ascending, -1 padded)."""
    torch = _torch()
    _need(index_q, "index_q", torch.bfloat16)
    if index_q.dim() != 3 or index_q.shape[2] != INDEX_DIM:
        raise ValueError("index_q must be [B,NH,128]")
    B, NH, _ = index_q.shape
    _need(index_k, "index_k", torch.bfloat16, None, index_q.device)
    if index_k.dim() != 2 or index_k.shape[1] != INDEX_DIM:
        raise ValueError("index_k must be [total,128]")
    _need(w, "w", torch.float32, (B, NH), index_q.device)
    _need(cu_seqlens, "cu_seqlens", torch.int64, (B + 1,), index_q.device)
    if topk_idx is None:
        topk_idx = torch.empty((B, topk), dtype=torch.int32, device=index_q.device)
    _need(topk_idx, "topk_idx", torch.int32, (B, topk), index_q.device)
    if topk_scores is not None:
        _need(topk_scores, "topk_scores", torch.float32, (B, topk), index_q.device)
    nbytes = workspace_size(_lib.OP_INDEX_TOPK, B, NH, int(max_seqlen), topk)
    ws, wsb = _workspace(ws, nbytes, index_q.device)
    lib = _lib.load()
    _lib.check(lib.dsa_index_topk(_ptr(index_q), _ptr(index_k), _ptr(w), _ptr(cu_seqlens), B, NH,
                                  int(index_k.shape[0]), int(max_seqlen), int(topk),
                                  _ptr(topk_idx), _ptr(topk_scores), _ptr(ws), wsb,
                                  _stream(stream)), lib)
    return topk_idx


def dsa_sparse_decode(q, k, v, cu_seqlens, topk_idx, gate=None, out=None, scale=None,
                      ws=None, stream=None):
    """Gated MLA over the selected positions only (all heads share a selection)."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [B,H,192]")
    B, H, _ = q.shape
    _check_cache(q, k, v, cu_seqlens, H, None)
    _need(topk_idx, "topk_idx", torch.int32, None, q.device)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != B:
        raise ValueError("topk_idx must be [B,topk]")
    topk = topk_idx.shape[1]
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (B, H * DV), q.device)
    if out is None:
        out = torch.empty((B, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_SPARSE_DECODE, B, H, 0, topk)
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.dsa_sparse_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(topk_idx),
                                     topk, B, H, _ptr(gate), _ptr(out),
                                     float(default_scale() if scale is None else scale),
                                     _ptr(ws), wsb, _stream(stream)), lib)
    return out


def _check_capacity_cache(k_cache, v_cache, device):
    torch = _torch()
    _need(k_cache, "k_cache", torch.bfloat16, None, device)
    if k_cache.dim() != 4 or k_cache.shape[3] != DQK:
        raise ValueError("k_cache must be [B,H,capacity,192]")
    B, H, cap, _ = k_cache.shape
    _need(v_cache, "v_cache", torch.bfloat16, (B, H, cap, DV), device)
    return B, H, cap


def mla_cache_append(k_new, v_new, k_cache, v_cache, start, stream=None):
    """Copy k_new [B,H,Tn,192] / v_new [B,H,Tn,128] into positions start_b..start_b+Tn-1
    of the caches [B,H,capacity,D].  `start` is an int (every sequence) or a device
    int64 tensor [B] (per sequence)."""
    torch = _torch()
    B, H, cap = _check_capacity_cache(k_cache, v_cache, k_cache.device)
    _need(k_new, "k_new", torch.bfloat16, None, k_cache.device)
    if k_new.dim() != 4 or tuple(k_new.shape[:2]) != (B, H) or k_new.shape[3] != DQK:
        raise ValueError(f"k_new must be [{B},{H},Tn,192]")
    Tn = k_new.shape[2]
    _need(v_new, "v_new", torch.bfloat16, (B, H, Tn, DV), k_cache.device)
    if isinstance(start, torch.Tensor):
        _need(start, "start", torch.int64, (B,), k_cache.device)
        sp, s_all = _ptr(start), 0
    else:
        sp, s_all = None, int(start)
    lib = _lib.load()
    _lib.check(lib.mla_cache_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), sp,
                                    s_all, B, H, Tn, cap, _stream(stream)), lib)


def mla_prefill_chunk(q, k_new, v_new, k_cache, v_cache, P: int, gate=None, out=None,
                      scale=None, stream=None):
    """Chunked prefill: append the Tq new keys/values at positions P.. of the caches,
    then causal gated attention of q [B,H,Tq,192] over cache positions 0..P+Tq-1."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4 or q.shape[3] != DQK:
        raise ValueError("q must be [B,H,Tq,192]")
    B, H, Tq, _ = q.shape
    if _check_capacity_cache(k_cache, v_cache, q.device)[:2] != (B, H):
        raise ValueError("k_cache and q disagree on B or H")
    cap = k_cache.shape[2]
    _need(k_new, "k_new", torch.bfloat16, (B, H, Tq, DQK), q.device)
    _need(v_new, "v_new", torch.bfloat16, (B, H, Tq, DV), q.device)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (B, Tq, H * DV), q.device)
    if out is None:
        out = torch.empty((B, Tq, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, Tq, H * DV), q.device)
    lib = _lib.load()
    _lib.check(lib.mla_prefill_chunk(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(gate), _ptr(out), B, H, Tq, int(P), cap,
                                     float(default_scale() if scale is None else scale), None, 0,
                                     _stream(stream)), lib)
    return out


def mla_decode_cached(q, k_cache, v_cache, cache_seqlens, max_seqlen: int, k_new=None,
                      v_new=None, gate=None, out=None, scale=None, ws=None, stream=None):
    """Decode step over fixed-capacity caches [B,H,capacity,D]: sequence b holds
    cache_seqlens[b] positions (device int64 [B]).  With k_new/v_new ([B,H,1,D]) the
    current token is appended at position cache_seqlens[b] first and attended to."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [B,H,192]")
    B, H, _ = q.shape
    if _check_capacity_cache(k_cache, v_cache, q.device)[:2] != (B, H):
        raise ValueError("k_cache and q disagree on B or H")
    cap = k_cache.shape[2]
    _need(cache_seqlens, "cache_seqlens", torch.int64, (B,), q.device)
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new or neither")
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16, (B, H, 1, DQK), q.device)
        _need(v_new, "v_new", torch.bfloat16, (B, H, 1, DV), q.device)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (B, H * DV), q.device)
    if out is None:
        out = torch.empty((B, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_DECODE, B, H, int(max_seqlen), 0)
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.mla_decode_cached(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                     _ptr(v_cache), _ptr(cache_seqlens), B, H, cap,
                                     int(max_seqlen), _ptr(gate), _ptr(out),
                                     float(default_scale() if scale is None else scale),
                                     _ptr(ws), wsb, _stream(stream)), lib)
    return out


def mla_decode_latent(q, ckv, cu_seqlens, max_seqlen: int, w_kc, w_vc, gate=None, out=None,
                      scale=None, ws=None, stream=None):
    """Gated MLA decode over a packed latent cache ckv [total,576] (latent c_s ++ shared
    key r_s per position); q [B,H,192] expanded-form queries; w_kc / w_vc [H,128,512]."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [B,H,192]")
    B, H, _ = q.shape
    _need(ckv, "ckv", torch.bfloat16, None, q.device)
    if ckv.dim() != 2 or ckv.shape[1] != 576:
        raise ValueError("ckv must be [total,576]")
    _need(cu_seqlens, "cu_seqlens", torch.int64, (B + 1,), q.device)
    _need(w_kc, "w_kc", torch.bfloat16, (H, 128, 512), q.device)
    _need(w_vc, "w_vc", torch.bfloat16, (H, DV, 512), q.device)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (B, H * DV), q.device)
    if out is None:
        out = torch.empty((B, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_LATENT_DECODE, B, H, int(max_seqlen), 0)
    if nbytes == 0:
        raise ValueError(f"unsupported latent decode shape B={B} H={H}")
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.mla_decode_latent(_ptr(q), _ptr(ckv), _ptr(cu_seqlens), int(ckv.shape[0]), B,
                                     H, int(max_seqlen), _ptr(w_kc), _ptr(w_vc), _ptr(gate),
                                     _ptr(out), float(default_scale() if scale is None else scale),
                                     _ptr(ws), wsb, _stream(stream)), lib)
    return out


def dsa_prefill_index_topk(index_q, index_k, w, topk: int = MAX_TOPK, topk_idx=None,
                           topk_scores=None, ws=None, stream=None):
    """Per-token DSA index score + top-k for a prompt: index_q [Tq,32,128], index_k
    [Tk,128] (token i sees positions 0..Tk-Tq+i), w [Tq,32] fp32 -> [Tq,topk] int32."""
    torch = _torch()
    _need(index_q, "index_q", torch.bfloat16)
    if index_q.dim() != 3 or index_q.shape[2] != INDEX_DIM:
        raise ValueError("index_q must be [Tq,NH,128]")
    Tq, NH, _ = index_q.shape
    _need(index_k, "index_k", torch.bfloat16, None, index_q.device)
    if index_k.dim() != 2 or index_k.shape[1] != INDEX_DIM:
        raise ValueError("index_k must be [Tk,128]")
    Tk = index_k.shape[0]
    _need(w, "w", torch.float32, (Tq, NH), index_q.device)
    if topk_idx is None:
        topk_idx = torch.empty((Tq, topk), dtype=torch.int32, device=index_q.device)
    _need(topk_idx, "topk_idx", torch.int32, (Tq, topk), index_q.device)
    if topk_scores is not None:
        _need(topk_scores, "topk_scores", torch.float32, (Tq, topk), index_q.device)
    nbytes = workspace_size(_lib.OP_PREFILL_INDEX_TOPK, Tq, 0, Tk, topk)
    ws, wsb = _workspace(ws, nbytes, index_q.device)
    lib = _lib.load()
    _lib.check(lib.dsa_prefill_index_topk(_ptr(index_q), _ptr(index_k), _ptr(w), Tq, Tk, NH,
                                          int(topk), _ptr(topk_idx), _ptr(topk_scores), _ptr(ws),
                                          wsb, _stream(stream)), lib)
    return topk_idx


def mla_sparse_prefill_latent(q, ckv, topk_idx, w_kc, w_vc, gate=None, out=None, scale=None,
                              ws=None, stream=None):
    """DSA sparse prefill over the latent cache: q [Tq,H,192], ckv [Tk,576], topk_idx
    [Tq,topk] int32 (token i at position Tk-Tq+i), w_kc / w_vc [H,128,512]."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [Tq,H,192]")
    Tq, H, _ = q.shape
    _need(ckv, "ckv", torch.bfloat16, None, q.device)
    if ckv.dim() != 2 or ckv.shape[1] != 576:
        raise ValueError("ckv must be [Tk,576]")
    Tk = ckv.shape[0]
    _need(topk_idx, "topk_idx", torch.int32, None, q.device)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != Tq:
        raise ValueError("topk_idx must be [Tq,topk]")
    topk = topk_idx.shape[1]
    _need(w_kc, "w_kc", torch.bfloat16, (H, 128, 512), q.device)
    _need(w_vc, "w_vc", torch.bfloat16, (H, DV, 512), q.device)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (Tq, H * DV), q.device)
    if out is None:
        out = torch.empty((Tq, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (Tq, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_SPARSE_PREFILL_LATENT, Tq, H, Tk, topk)
    if nbytes == 0:
        raise ValueError(f"unsupported sparse prefill shape Tq={Tq} H={H}")
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.mla_sparse_prefill_latent(_ptr(q), _ptr(ckv), _ptr(topk_idx), Tq, Tk, topk, H,
                                             _ptr(w_kc), _ptr(w_vc), _ptr(gate), _ptr(out),
                                             float(default_scale() if scale is None else scale),
                                             _ptr(ws), wsb, _stream(stream)), lib)
    return out


def dsa_quantize_index_keys(index_k, k8=None, kscale=None, stream=None):
    """bf16 index keys [N,128] -> (e4m3 codes uint8 [N,128], fp32 scales [N])."""
    torch = _torch()
    _need(index_k, "index_k", torch.bfloat16)
    if index_k.dim() != 2 or index_k.shape[1] != INDEX_DIM:
        raise ValueError("index_k must be [N,128]")
    N = index_k.shape[0]
    if k8 is None:
        k8 = torch.empty((N, INDEX_DIM), dtype=torch.uint8, device=index_k.device)
    if kscale is None:
        kscale = torch.empty((N,), dtype=torch.float32, device=index_k.device)
    _need(k8, "k8", torch.uint8, (N, INDEX_DIM), index_k.device)
    _need(kscale, "kscale", torch.float32, (N,), index_k.device)
    lib = _lib.load()
    _lib.check(lib.dsa_quantize_index_keys(_ptr(index_k), _ptr(k8), _ptr(kscale), N,
                                           _stream(stream)), lib)
    return k8, kscale


def dsa_index_topk_fp8(index_q, k8, kscale, w, cu_seqlens, max_seqlen: int, topk: int = MAX_TOPK,
                       topk_idx=None, topk_scores=None, ws=None, stream=None):
    """dsa_index_topk over FP8 index keys (k8 [total,128] uint8, kscale [total] fp32)."""
    torch = _torch()
    _need(index_q, "index_q", torch.bfloat16)
    if index_q.dim() != 3 or index_q.shape[2] != INDEX_DIM:
        raise ValueError("index_q must be [B,NH,128]")
    B, NH, _ = index_q.shape
    _need(k8, "k8", torch.uint8, None, index_q.device)
    if k8.dim() != 2 or k8.shape[1] != INDEX_DIM:
        raise ValueError("k8 must be [total,128]")
    _need(kscale, "kscale", torch.float32, (k8.shape[0],), index_q.device)
    _need(w, "w", torch.float32, (B, NH), index_q.device)
    _need(cu_seqlens, "cu_seqlens", torch.int64, (B + 1,), index_q.device)
    if topk_idx is None:
        topk_idx = torch.empty((B, topk), dtype=torch.int32, device=index_q.device)
    _need(topk_idx, "topk_idx", torch.int32, (B, topk), index_q.device)
    if topk_scores is not None:
        _need(topk_scores, "topk_scores", torch.float32, (B, topk), index_q.device)
    nbytes = workspace_size(_lib.OP_INDEX_TOPK_FP8, B, NH, int(max_seqlen), topk)
    ws, wsb = _workspace(ws, nbytes, index_q.device)
    lib = _lib.load()
    _lib.check(lib.dsa_index_topk_fp8(_ptr(index_q), _ptr(k8), _ptr(kscale), _ptr(w),
                                      _ptr(cu_seqlens), B, NH, int(k8.shape[0]), int(max_seqlen),
                                      int(topk), _ptr(topk_idx), _ptr(topk_scores), _ptr(ws), wsb,
                                      _stream(stream)), lib)
    return topk_idx


RECORD_BYTES = 656


def mla_quantize_latent_cache(ckv, rec=None, stream=None):
    """Latent rows [N,576] bf16 -> FP8 records [N,656] uint8."""
    torch = _torch()
    _need(ckv, "ckv", torch.bfloat16)
    if ckv.dim() != 2 or ckv.shape[1] != 576:
        raise ValueError("ckv must be [N,576]")
    N = ckv.shape[0]
    if rec is None:
        rec = torch.empty((N, RECORD_BYTES), dtype=torch.uint8, device=ckv.device)
    _need(rec, "rec", torch.uint8, (N, RECORD_BYTES), ckv.device)
    lib = _lib.load()
    _lib.check(lib.mla_quantize_latent_cache(_ptr(ckv), _ptr(rec), N, _stream(stream)), lib)
    return rec


def mla_decode_latent_fp8(q, rec, cu_seqlens, max_seqlen: int, w_kc, w_vc, gate=None, out=None,
                          scale=None, ws=None, stream=None):
    """mla_decode_latent over FP8 records rec [total,656] uint8."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [B,H,192]")
    B, H, _ = q.shape
    _need(rec, "rec", torch.uint8, None, q.device)
    if rec.dim() != 2 or rec.shape[1] != RECORD_BYTES:
        raise ValueError("rec must be [total,656]")
    _need(cu_seqlens, "cu_seqlens", torch.int64, (B + 1,), q.device)
    _need(w_kc, "w_kc", torch.bfloat16, (H, 128, 512), q.device)
    _need(w_vc, "w_vc", torch.bfloat16, (H, DV, 512), q.device)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (B, H * DV), q.device)
    if out is None:
        out = torch.empty((B, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (B, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_LATENT_DECODE, B, H, int(max_seqlen), 0)
    if nbytes == 0:
        raise ValueError(f"unsupported latent decode shape B={B} H={H}")
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.mla_decode_latent_fp8(_ptr(q), _ptr(rec), _ptr(cu_seqlens), int(rec.shape[0]),
                                         B, H, int(max_seqlen), _ptr(w_kc), _ptr(w_vc),
                                         _ptr(gate), _ptr(out),
                                         float(default_scale() if scale is None else scale),
                                         _ptr(ws), wsb, _stream(stream)), lib)
    return out


def mla_sparse_prefill_latent_fp8(q, rec, topk_idx, w_kc, w_vc, gate=None, out=None, scale=None,
                                  ws=None, stream=None):
    """mla_sparse_prefill_latent over FP8 records rec [Tk,656] uint8."""
    torch = _torch()
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != DQK:
        raise ValueError("q must be [Tq,H,192]")
    Tq, H, _ = q.shape
    _need(rec, "rec", torch.uint8, None, q.device)
    if rec.dim() != 2 or rec.shape[1] != RECORD_BYTES:
        raise ValueError("rec must be [Tk,656]")
    Tk = rec.shape[0]
    _need(topk_idx, "topk_idx", torch.int32, None, q.device)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != Tq:
        raise ValueError("topk_idx must be [Tq,topk]")
    topk = topk_idx.shape[1]
    _need(w_kc, "w_kc", torch.bfloat16, (H, 128, 512), q.device)
    _need(w_vc, "w_vc", torch.bfloat16, (H, DV, 512), q.device)
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, (Tq, H * DV), q.device)
    if out is None:
        out = torch.empty((Tq, H * DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, (Tq, H * DV), q.device)
    nbytes = workspace_size(_lib.OP_SPARSE_PREFILL_LATENT, Tq, H, Tk, topk)
    if nbytes == 0:
        raise ValueError(f"unsupported sparse prefill shape Tq={Tq} H={H}")
    ws, wsb = _workspace(ws, nbytes, q.device)
    lib = _lib.load()
    _lib.check(lib.mla_sparse_prefill_latent_fp8(_ptr(q), _ptr(rec), _ptr(topk_idx), Tq, Tk, topk,
                                                 H, _ptr(w_kc), _ptr(w_vc), _ptr(gate), _ptr(out),
                                                 float(default_scale() if scale is None else scale),
                                                 _ptr(ws), wsb, _stream(stream)), lib)
    return out


def check_device_status(stream=None) -> None:
    """Synchronise and raise MlaError if a kernel recorded a device-side fault."""
    lib = _lib.load()
    _lib.check(lib.mla_check_device_status(_stream(stream)), lib)


def debug_set(knob: int, value: int) -> None:
    lib = _lib.load()
    _lib.check(lib.mla_debug_set(int(knob), int(value)), lib)


def gather_probe(k, v, cu_seqlens, topk_idx, H, sink=None, stream=None):
    """Measurement aid: gather the rows dsa_sparse_decode(k, v, cu_seqlens,
    topk_idx, ...) reads, with plain loads and no arithmetic (the achievable
    gather rate for that kernel).  Returns the per-CTA XOR words (uint32 as
    int32)."""
    torch = _torch()
    lib = _lib.load()
    _need(topk_idx, "topk_idx", torch.int32)
    B, topk = topk_idx.shape
    dev = topk_idx.device
    _need(k, "k", torch.bfloat16, device=dev)
    _need(v, "v", torch.bfloat16, device=dev)
    _need(cu_seqlens, "cu_seqlens", torch.int64, (B + 1,), device=dev)
    if sink is None:
        sink = torch.empty(lib.mla_gather_probe_blocks(), dtype=torch.int32, device=dev)
    _lib.check(lib.mla_gather_probe(_ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(topk_idx), topk, B,
                                    H, _ptr(sink), _stream(stream)), lib)
    return sink


def timing_enable(on: bool = True) -> None:
    """Record CUDA events around each call's dominant kernel (instrumentation)."""
    lib = _lib.load()
    _lib.check(lib.mla_timing_enable(1 if on else 0), lib)


def timing_read(op: int):
    """(total kernel ms, launches) of operation `op` since the last read."""
    import ctypes
    lib = _lib.load()
    ms, n = ctypes.c_double(0), ctypes.c_longlong(0)
    _lib.check(lib.mla_timing_read(int(op), ctypes.byref(ms), ctypes.byref(n)), lib)
    return ms.value, n.value
