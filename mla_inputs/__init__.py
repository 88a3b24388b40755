"""Seeded synthetic inputs for the Gated MLA / Gated DSA attention path.

This module is shared by the CPU oracle's tests and the GPU path. It holds
none of the method's arithmetic: it only draws N(0,1) tensors from seeded
generators and lays them out in the shapes the library takes. Nothing here
scores, masks, normalises or gates anything.

Shapes follow the Kimi K3 "Gated MLA > KV cache" page (cache
``k [B,96,T,192]``, ``v [B,96,T,128]``) and the Kimi K2 "Latent attention >
KV cache" page (64 heads). The last 64 key features are one vector per
(batch, position) broadcast to every head, unrotated, as the "Take the shared
key part" page describes. DSA inputs follow the K3.1 Gated DSA blog post,
eqs. (2)-(4): 32 index heads of 128 features, one 128-feature index key per
cached position, and 32 fp32 head weights per query.

Recipe (every tensor is ~N(0,1), drawn in fp32 and rounded once to bf16):

* seed of a tensor = ``SEED + 1_000_003*config + 10_007*tensor + index``,
  where ``index`` is the batch row for per-sequence tensors and 0 otherwise;
* torch ``Generator`` on the device the tensor is made on (CPU tensors and
  CUDA tensors therefore differ; tests always hand the oracle a copy of the
  tensors the GPU path receives);
* ragged cache lengths come from numpy's PCG64 ``integers(lo, hi+1)`` so they
  are the same on every machine.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

SEED = 0x4D4C41

DQK = 192          # 128 content + 64 shared (K3) / rotary (K2) key features
D_NOPE = 128
D_SHARED = 64
DV = 128
INDEX_HEADS = 32   # K3.1 indexer heads
INDEX_DIM = 128    # K3.1 index key / query features

# tensor ids used in the seed formula
T_Q, T_K, T_SHARED, T_V, T_GATE, T_IQ, T_IK, T_W, T_CKV, T_WK, T_WV = range(11)
D_LATENT = 512     # normalised KV latent c_s (DSA post, eq. (7))
D_CKV = D_LATENT + D_SHARED   # cached per position: c_s and the shared key r_s


def seed_of(config: int, tensor: int, index: int = 0) -> int:
    return SEED + 1_000_003 * config + 10_007 * tensor + index


def _randn(shape, seed: int, device, dtype=torch.bfloat16) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def ragged_lengths(B: int, lo: int, hi: int, seed: int) -> list[int]:
    """Per-sequence cache lengths, uniform on the integers lo..hi."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=B)]


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for t in lengths:
        cu.append(cu[-1] + int(t))
    return torch.tensor(cu, dtype=torch.int64)


@dataclass
class Prefill:
    q: torch.Tensor        # [B,H,Tq,192]
    k: torch.Tensor        # [B,H,Tk,192]
    v: torch.Tensor        # [B,H,Tk,128]
    gate: torch.Tensor | None  # [B,Tq,H*128] logits
    scale: float


@dataclass
class Decode:
    q: torch.Tensor        # [B,H,192]
    k: torch.Tensor        # packed: seq b = [H,T_b,192] from element cu[b]*H*192
    v: torch.Tensor        # packed: seq b = [H,T_b,128] from element cu[b]*H*128
    cu_seqlens: torch.Tensor  # [B+1] int64 (on the tensors' device)
    lengths: list[int]
    gate: torch.Tensor | None  # [B,H*128]
    scale: float
    H: int = 96


@dataclass
class Dsa:
    index_q: torch.Tensor  # [B,32,128]
    index_k: torch.Tensor  # packed [cu[B],128]
    w: torch.Tensor        # [B,32] fp32
    main: Decode = field(default=None)


def default_scale() -> float:
    """1/sqrt(q_head_dim) with q_head_dim = 128 + 64."""
    return DQK ** -0.5


def make_prefill(B: int, H: int, Tq: int, Tk: int, gated: bool, device="cpu",
                 config: int = 0, scale: float | None = None) -> Prefill:
    q = _randn((B, H, Tq, DQK), seed_of(config, T_Q), device)
    k = _randn((B, H, Tk, DQK), seed_of(config, T_K), device)
    shared = _randn((B, 1, Tk, D_SHARED), seed_of(config, T_SHARED), device)
    k[..., D_NOPE:] = shared          # one shared key part per (b, position), every head
    v = _randn((B, H, Tk, DV), seed_of(config, T_V), device)
    gate = _randn((B, Tq, H * DV), seed_of(config, T_GATE), device) if gated else None
    return Prefill(q, k, v, gate, default_scale() if scale is None else scale)


def _seq_kv(H: int, T: int, device, config: int, b: int):
    kb = _randn((H, T, DQK), seed_of(config, T_K, b), device)
    sb = _randn((T, D_SHARED), seed_of(config, T_SHARED, b), device)
    kb[:, :, D_NOPE:] = sb             # broadcast over heads
    vb = _randn((H, T, DV), seed_of(config, T_V, b), device)
    return kb, vb


def make_decode(lengths, H: int, gated: bool, device="cpu", config: int = 1,
                scale: float | None = None) -> Decode:
    """Packed per-sequence cache: seq b holds [H, T_b, D] contiguous."""
    lengths = [int(t) for t in lengths]
    B = len(lengths)
    total = sum(lengths)
    cu = cu_from_lengths(lengths)
    k = torch.empty(total * H * DQK, dtype=torch.bfloat16, device=device)
    v = torch.empty(total * H * DV, dtype=torch.bfloat16, device=device)
    for b, T in enumerate(lengths):
        kb, vb = _seq_kv(H, T, device, config, b)
        o = int(cu[b]) * H
        k[o * DQK:(o + H * T) * DQK] = kb.reshape(-1)
        v[o * DV:(o + H * T) * DV] = vb.reshape(-1)
        del kb, vb
    q = _randn((B, H, DQK), seed_of(config, T_Q), device)
    gate = _randn((B, H * DV), seed_of(config, T_GATE), device) if gated else None
    return Decode(q, k, v, cu.to(device), lengths, gate,
                  default_scale() if scale is None else scale, H)


@dataclass
class LatentDecode:
    q: torch.Tensor        # [B,H,192] expanded-form queries (128 content ++ 64 shared)
    ckv: torch.Tensor      # packed [cu[B],576]: latent c_s (512) ++ shared key r_s (64)
    cu_seqlens: torch.Tensor
    lengths: list[int]
    w_kc: torch.Tensor     # [H,128,512] W^K (key up-projection of the latent)
    w_vc: torch.Tensor     # [H,128,512] W^V (value up-projection)
    gate: torch.Tensor | None
    scale: float
    H: int


def make_latent_decode(lengths, H: int, gated: bool = True, device="cpu", config: int = 5,
                       scale: float | None = None) -> LatentDecode:
    """Latent cache rows ~N(0,1) (c_s is RMS-normalised on the pages, so unit
    scale per feature); W^K, W^V entries ~N(0, 1/512), so the expanded keys and
    values are ~N(0,1) like the expanded-cache workloads."""
    lengths = [int(t) for t in lengths]
    B = len(lengths)
    cu = cu_from_lengths(lengths)
    ckv = torch.empty((int(cu[-1]), D_CKV), dtype=torch.bfloat16, device=device)
    for b, T in enumerate(lengths):
        ckv[int(cu[b]):int(cu[b]) + T] = _randn((T, D_CKV), seed_of(config, T_CKV, b), device)
    std = D_LATENT ** -0.5
    w_kc = (_randn((H, D_NOPE, D_LATENT), seed_of(config, T_WK), device, torch.float32)
            * std).to(torch.bfloat16)
    w_vc = (_randn((H, DV, D_LATENT), seed_of(config, T_WV), device, torch.float32)
            * std).to(torch.bfloat16)
    q = _randn((B, H, DQK), seed_of(config, T_Q), device)
    gate = _randn((B, H * DV), seed_of(config, T_GATE), device) if gated else None
    return LatentDecode(q, ckv, cu.to(device), lengths, w_kc, w_vc, gate,
                        default_scale() if scale is None else scale, H)


@dataclass
class DsaPrefill:
    index_q: torch.Tensor  # [Tq,32,128]
    index_k: torch.Tensor  # [Tk,128]
    w: torch.Tensor        # [Tq,32] fp32
    q: torch.Tensor        # [Tq,H,192] expanded-form queries
    ckv: torch.Tensor      # [Tk,576] latent cache
    w_kc: torch.Tensor     # [H,128,512]
    w_vc: torch.Tensor     # [H,128,512]
    gate: torch.Tensor | None  # [Tq,H*128]
    scale: float
    H: int


def make_dsa_prefill(Tq: int, Tk: int, H: int = 96, gated: bool = True, device="cpu",
                     config: int = 6) -> DsaPrefill:
    """One prompt of Tq tokens after Tk - Tq cached positions: index queries,
    keys and head weights as in make_dsa, the main cache as in
    make_latent_decode (one sequence)."""
    iq = _randn((Tq, INDEX_HEADS, INDEX_DIM), seed_of(config, T_IQ), device)
    ik = _randn((Tk, INDEX_DIM), seed_of(config, T_IK), device)
    w = _randn((Tq, INDEX_HEADS), seed_of(config, T_W), device, dtype=torch.float32)
    lat = make_latent_decode([Tk], H, False, device, config)
    q = _randn((Tq, H, DQK), seed_of(config, T_Q), device)
    gate = _randn((Tq, H * DV), seed_of(config, T_GATE), device) if gated else None
    return DsaPrefill(iq, ik, w, q, lat.ckv, lat.w_kc, lat.w_vc, gate, default_scale(), H)


NAN_BF16 = 0x7FC0   # a quiet-NaN bit pattern, used to fill unused cache capacity


def nan_filled(shape, device) -> torch.Tensor:
    """bf16 tensor whose every element is NaN (stands for uninitialised memory)."""
    return torch.full(shape, NAN_BF16, dtype=torch.int16, device=device).view(torch.bfloat16)


@dataclass
class CapacityDecode:
    q: torch.Tensor            # [B,H,192]
    k_cache: torch.Tensor      # [B,H,cap,192]; positions past lengths[b] hold NaN
    v_cache: torch.Tensor      # [B,H,cap,128]
    lengths: list[int]         # positions cached per sequence
    k_new: torch.Tensor | None     # [B,H,1,192]: position lengths[b] of each sequence
    v_new: torch.Tensor | None
    gate: torch.Tensor | None
    scale: float
    H: int


def make_capacity_decode(lengths, H: int, cap: int, gated: bool, device="cpu", config: int = 1,
                         append: bool = True) -> CapacityDecode:
    """Fixed-capacity caches holding the same keys and values as
    make_decode(lengths + [1 if append]) for the same config: sequence b's
    first lengths[b] positions in the cache, its next position (the current
    token) in k_new / v_new when `append`, NaN everywhere else."""
    lengths = [int(t) for t in lengths]
    B = len(lengths)
    kc, vc = nan_filled((B, H, cap, DQK), device), nan_filled((B, H, cap, DV), device)
    extra = 1 if append else 0
    kn = torch.empty((B, H, 1, DQK), dtype=torch.bfloat16, device=device) if append else None
    vn = torch.empty((B, H, 1, DV), dtype=torch.bfloat16, device=device) if append else None
    for b, L in enumerate(lengths):
        kb, vb = _seq_kv(H, L + extra, device, config, b)
        kc[b, :, :L], vc[b, :, :L] = kb[:, :L], vb[:, :L]
        if append:
            kn[b], vn[b] = kb[:, L:], vb[:, L:]
        del kb, vb
    q = _randn((B, H, DQK), seed_of(config, T_Q), device)
    gate = _randn((B, H * DV), seed_of(config, T_GATE), device) if gated else None
    return CapacityDecode(q, kc, vc, lengths, kn, vn, gate, default_scale(), H)


def make_dsa(lengths, H: int = 96, device="cpu", config: int = 4, with_main=True) -> Dsa:
    lengths = [int(t) for t in lengths]
    B = len(lengths)
    cu = cu_from_lengths(lengths)
    total = int(cu[-1])
    iq = _randn((B, INDEX_HEADS, INDEX_DIM), seed_of(config, T_IQ), device)
    ik = torch.empty((total, INDEX_DIM), dtype=torch.bfloat16, device=device)
    for b, T in enumerate(lengths):
        ik[int(cu[b]):int(cu[b]) + T] = _randn((T, INDEX_DIM), seed_of(config, T_IK, b), device)
    w = _randn((B, INDEX_HEADS), seed_of(config, T_W), device, dtype=torch.float32)
    main = make_decode(lengths, H, True, device, config) if with_main else None
    return Dsa(iq, ik, w, main)


# ---------------------------------------------------------------------------
# The five workloads (sizes and seeds). Config ids 0..4 enter the seeds.
# ---------------------------------------------------------------------------
WORKLOADS = {
    "prefill_b1_h96_t128": dict(kind="prefill", config=0, B=1, H=96, T=128, gated=True),
    # Workloads whose inputs are small come first: the benchmark times them in
    # this order, and a short kernel timed right after another workload's
    # multi-GB input generation read up to 25 % slow (the 268 MB indexer:
    # 0.079 ms there, 0.061 ms here, every other line unchanged).
    # the indexer part of the DSA workload alone (same index keys, queries, weights)
    "dsa_index_b8_t131072": dict(kind="index", config=4, B=8, H=96, T=131072, topk=2048),
    # the indexer of the DSA decode workload over FP8 index keys (132 B/position)
    "dsa_index_fp8_b8_t131072": dict(kind="index_fp8", config=4, B=8, H=96, T=131072, topk=2048),
    "decode_b32_h96_t8192": dict(kind="decode", config=1, B=32, H=96, T=8192, gated=True),
    "ragged_decode_b64_h96_t1024_65536": dict(kind="decode", config=2, B=64, H=96,
                                              lo=1024, hi=65536, gated=True),
    "prefill_b1_h96_t16384": dict(kind="prefill", config=3, B=1, H=96, T=16384, gated=True),
    "prefill_b1_h64_t16384_nogate": dict(kind="prefill", config=3, B=1, H=64, T=16384,
                                         gated=False),
    "dsa_decode_b8_t131072": dict(kind="dsa", config=4, B=8, H=96, T=131072, topk=2048),
    # the cache-update path: a 16384-token prompt fed in four 4096-token chunks
    # into a 16384-position cache; a decode step that appends the current token
    # to 8191 cached positions of 32 sequences
    "chunked_prefill_b1_h96_t16384_c4096": dict(kind="chunked_prefill", config=3, B=1, H=96,
                                                T=16384, chunk=4096, gated=True),
    "decode_cached_b32_h96_t8192": dict(kind="decode_cached", config=1, B=32, H=96, T=8192,
                                        gated=True),
    # decode over the absorbed 576-feature latent cache (1,152 bytes per position
    # instead of 61,440): the decode workload's batch and length
    "latent_decode_b32_h96_t8192": dict(kind="latent_decode", config=5, B=32, H=96, T=8192,
                                        gated=True),
    # the latent decode over 656-byte FP8 records (the same cache, quantised)
    "latent_decode_fp8_b32_h96_t8192": dict(kind="latent_decode_fp8", config=5, B=32, H=96,
                                            T=8192, gated=True),
    # DSA prefill: a 16384-token prompt, every token scoring its whole visible
    # history and attending over its own top-2048 of the latent cache
    "dsa_prefill_t16384": dict(kind="dsa_prefill", config=6, B=1, H=96, T=16384, topk=2048,
                               gated=True),
    # a reference rate, not a step of the method: the rows the DSA decode's
    # sparse attention reads, gathered with plain loads and no arithmetic
    "dsa_gather_probe_b8_t131072": dict(kind="gather_probe", config=4, B=8, H=96, T=131072,
                                        topk=2048),
    # smaller cases of the same kernels, a few GB on the device, for ncu captures
    "dsa_decode_b2_t16384": dict(kind="dsa", config=4, B=2, H=96, T=16384, topk=2048,
                                 profile_only=True),
    "dsa_gather_probe_b2_t16384": dict(kind="gather_probe", config=4, B=2, H=96, T=16384,
                                       topk=2048, profile_only=True),
    "prefill_b1_h8_t16384": dict(kind="prefill", config=3, B=1, H=8, T=16384, gated=True,
                                 profile_only=True),
    "dsa_prefill_t4096": dict(kind="dsa_prefill", config=6, B=1, H=96, T=4096, topk=2048,
                              gated=True, profile_only=True),
}


def workload_lengths(name: str) -> list[int]:
    w = WORKLOADS[name]
    if w["kind"] == "prefill":
        return [w["T"]] * w["B"]
    if "lo" in w:
        return ragged_lengths(w["B"], w["lo"], w["hi"], seed_of(w["config"], 99))
    return [w["T"]] * w["B"]


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)

