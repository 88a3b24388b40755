"""The byte/flop accounting reproduces the fixed counts printed on the pages."""
import json
import os

from mla_family_attention_gb300 import accounting as acc

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_counts.json")))


def test_values_per_position():
    assert acc.kv_values_per_position(96) == G["k3_values_per_position"]["value"]
    assert acc.kv_values_per_position(64) == G["k2_values_per_position"]["value"]
    assert acc.kv_bytes_per_position(96) == 61440


def test_kda_crossover():
    kda = acc.kda_state_values()
    assert kda == G["kda_state_values"]["value"]
    first = next(t for t in range(1, 1000) if t * acc.kv_values_per_position(96) > kda)
    assert first == G["kda_state_values"]["crossover_position"]


def test_cache_sizes():
    for key in ("k3_latent_cache_gib", "k31_cache_with_index_gib"):
        c = G[key]
        assert acc.latent_cache_gib(c["layers"], c["values_per_token"], c["tokens"]) == c["value"]
    f = G["fp8_record_bytes"]
    gib = acc.latent_cache_gib(f["layers"], f["main"] + f["index"], f["tokens"], 1)
    assert abs(gib - f["total_gib"]) < 0.005


def test_indexer_and_sparse_counts():
    assert acc.index_flops([1]) == G["indexer_flops_per_position"]["value"]
    s = G["sparse_fraction_at_1m"]
    assert s["topk"] / s["t"] == s["fraction"]
    assert acc.sparse_kv_bytes([s["t"]], 96, s["topk"]) == s["topk"] * 61440


def test_workload_denominators():
    assert acc.decode_kv_bytes([8192] * 32, 96) == 16_106_127_360
    assert acc.prefill_flops(1, 96, 128, 128) == 507_248_640
    assert acc.prefill_flops(1, 96, 16384, 16384) == 96 * 16384 * 16385 // 2 * 640
    assert acc.index_key_bytes([131072] * 8) == 268_435_456
    assert acc.sparse_kv_bytes([131072] * 8, 96, 2048) == 1_006_632_960
