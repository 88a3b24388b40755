"""Byte and flop accounting for the Gated MLA / Gated DSA hot path.

These are the denominators of the roofline figures. They count the work the
method defines, not what a kernel happens to move:

* a cached position of one layer holds H*(192+128) bf16 values
  (Kimi K3 "Gated MLA > KV cache": 96*(192+128) = 30,720 values;
  Kimi K2 "Latent attention > KV cache": 64 heads -> 20,480 values);
  decode reads all of them, the 64 shared key features of every head
  included, because the cache layout stores them per head;
* causal prefill does 2*(192+128) flops per visible (query, key, head);
* the DSA indexer reads one 128-feature bf16 index key per position and does
  2*32*128 flops per position (K3.1 Gated DSA post, complexity section);
* sparse decode reads min(topk, T) cached positions per sequence.
"""
from __future__ import annotations

DQK, DV, INDEX_HEADS, INDEX_DIM = 192, 128, 32, 128
BF16 = 2


def kv_values_per_position(H: int) -> int:
    return H * (DQK + DV)


def kv_bytes_per_position(H: int) -> int:
    return kv_values_per_position(H) * BF16


def decode_kv_bytes(lengths, H: int) -> int:
    return kv_bytes_per_position(H) * sum(int(t) for t in lengths)


def causal_pairs(Tq: int, Tk: int) -> int:
    """Visible (query, key) pairs with bottom-right alignment, diagonal included."""
    P = Tk - Tq
    return Tq * P + Tq * (Tq + 1) // 2


def prefill_flops(B: int, H: int, Tq: int, Tk: int) -> int:
    return B * H * causal_pairs(Tq, Tk) * 2 * (DQK + DV)


def latent_kv_bytes(lengths) -> int:
    """Bytes of the absorbed latent cache read by a decode step: 576 bf16 values
    (latent c_s and shared key r_s) per position, shared by every head."""
    return sum(int(t) for t in lengths) * (512 + 64) * BF16


def dsa_prefill_index_flops(Tq: int, Tk: int) -> int:
    """Index scoring of a prompt: 2*32*128 flops per visible (token, position) pair."""
    return 2 * INDEX_HEADS * INDEX_DIM * causal_pairs(Tq, Tk)


def sparse_latent_core_flops(Tq: int, Tk: int, H: int, topk: int) -> int:
    """The attention kernel's own part of the sparse latent prefill: every
    prompt token over its min(topk, visible) selected positions, 2*(576 + 512)
    flops per selected (token, position, head) (Q.K^T over 576 features,
    P.V over 512)."""
    P = Tk - Tq
    sel = sum(min(topk, P + i + 1) for i in range(Tq))
    return sel * H * 2 * (576 + 512)


def sparse_latent_attention_flops(Tq: int, Tk: int, H: int, topk: int) -> int:
    """The whole sparse latent prefill: the attention (above) plus the W^K
    absorption and the W^V projection, 2*128*512 flops each per (token,
    head), which run in kernels of their own."""
    return sparse_latent_core_flops(Tq, Tk, H, topk) + Tq * H * 2 * 2 * 128 * 512


def latent_kv_bytes_fp8(lengths) -> int:
    """Bytes of the FP8 latent cache read by a decode step: one 656-byte record
    (512 e4m3 codes, 4 fp32 scales, 64 bf16 shared-key features) per position."""
    return sum(int(t) for t in lengths) * 656


def append_bytes(B: int, H: int, Tn: int) -> int:
    """HBM bytes of appending Tn positions to every (b, h): read once, written once."""
    return 2 * B * Tn * kv_bytes_per_position(H)


def index_key_bytes(lengths) -> int:
    return sum(int(t) for t in lengths) * INDEX_DIM * BF16


def index_key_bytes_fp8(lengths) -> int:
    """FP8 index keys: 128 one-byte features and one fp32 scale per position."""
    return sum(int(t) for t in lengths) * (INDEX_DIM + 4)


def index_flops(lengths) -> int:
    return sum(int(t) for t in lengths) * 2 * INDEX_HEADS * INDEX_DIM


def sparse_kv_bytes(lengths, H: int, topk: int) -> int:
    return sum(min(int(t), topk) for t in lengths) * kv_bytes_per_position(H)


def kda_state_values(heads: int = 96, head_dim: int = 128, conv: int = 4) -> int:
    """Values one KDA layer keeps whatever the length.

    Reading of the K3 "Gated MLA > KV cache" page, which prints only the total
    (1,720,320): the recurrent state heads*dk*dv plus a short-convolution state
    of heads*dim*kernel for each of q, k and v (kernel 4)."""
    return heads * head_dim * head_dim + 3 * heads * head_dim * conv


def latent_cache_gib(layers: int, values_per_token: int, tokens: int, bytes_per_value: int = 2):
    return layers * values_per_token * bytes_per_value * tokens / 2 ** 30
