"""Pins of the oracle's counting functions against the numbers the pages print."""
import math

from oracle import shapes


def test_qkv_params_8b(printed):
    p = printed["qkv_params_8b"]
    assert shapes.qkv_params(4096, 32, 8) == p["value"]
    assert 32 * shapes.qkv_params(4096, 32, 8) == p["per_32_blocks"]
    assert 4096 * 4096 == p["parts"]["q"] and 4096 * 8 * 128 == p["parts"]["k"]


def test_d_ff_rule_8b(printed):
    p = printed["d_ff_8b"]
    assert int(2 * 4 * p["d_model"] / 3) == p["two_thirds_4d"]
    assert int(p["two_thirds_4d"] * p["ffn_dim_multiplier"]) == p["scaled_approx"]
    assert shapes.ffn_hidden_dim(p["d_model"], p["ffn_dim_multiplier"], p["multiple_of"]) == p["value"]
    # without the multiplier the rule lands on the next multiple of 1024 above 10922
    assert shapes.ffn_hidden_dim(4096, None, 1024) == 11264


def test_block_params_8b(printed):
    p = printed["block_params_8b"]
    assert shapes.block_params(4096, 14336, 32, 8) == p["block"]
    assert round(100 * shapes.ffn_share(4096, 14336, 32, 8), 1) == p["ffn_share_pct"]
    total, non_emb = shapes.model_params(4096, 14336, 32, 32, 8, 128256)
    assert round(total / 1e9, 2) == p["total_billions"]
    assert round(non_emb / 1e9, 2) == p["non_embedding_billions"]


def test_block_params_qwen(printed):
    p = printed["block_params_qwen25_7b"]
    c = p["config"]
    d, ff, L = c["hidden_size"], c["intermediate_size"], c["num_hidden_layers"]
    h, kv, V = c["num_attention_heads"], c["num_key_value_heads"], c["vocab_size"]
    assert shapes.block_params(d, ff, h, kv, qkv_bias=True) == p["block"]
    assert round(100 * shapes.ffn_share(d, ff, h, kv, qkv_bias=True), 1) == p["ffn_share_pct"]
    total, non_emb = shapes.model_params(d, ff, L, h, kv, V, qkv_bias=True)
    assert total == p["total_exact"]
    assert round(total / 1e9, 2) == p["total_billions"]
    assert round(non_emb / 1e9, 2) == p["non_embedding_billions"]


def test_head_and_embedding(printed):
    assert shapes.lm_head_params(4096, 128256) == printed["lm_head_params_8b"]["value"]
    e = printed["embedding_params_70b"]
    assert round(shapes.embedding_params(e["d_model"], e["vocab"]) / 1e9, 2) == e["billions"]


def test_kaplan_and_per_block_d2(printed):
    k = printed["kaplan_8b"]
    assert round(shapes.kaplan_params(4096, 32) / 1e9, 2) == k["twelve_L_d2_billions"]
    d = 4096
    attn = 2 * d * d + 2 * d * 1024
    ffn = 3 * d * 14336
    assert attn / d ** 2 == k["per_block_d2"]["attention"]
    assert ffn / d ** 2 == k["per_block_d2"]["ffn"]
    assert (attn + ffn) / d ** 2 == k["per_block_d2"]["total"]


def test_flop_figures(printed):
    f = printed["flops_8b"]
    _, n = shapes.model_params(4096, 14336, 32, 32, 8, 128256)
    total, _ = shapes.model_params(4096, 14336, 32, 32, 8, 128256)
    assert round(shapes.kaplan_context_flops(32, 131072, 4096) / 1e9, 1) == f["context_gflops_at_128k"]
    assert shapes.kaplan_context_flops(32, 131072, 4096) > 2 * n       # attention overtakes 2N
    share = shapes.kaplan_context_flops(32, 8192, 4096) / (2 * n)
    assert round(100 * share) == f["context_share_of_2N_at_8k_pct"]
    assert round(6 * n / 1e9) == f["six_n_gflops_without_embeddings"]
    assert round(6 * total / 1e9) == f["six_n_gflops_with_embeddings"]


def test_block_work_counts():
    # the algorithmic FLOP count: 2 per weight MAC + 4*Hq*dh per unmasked pair
    macs = shapes.block_weight_macs(4096, 14336, 32, 8, 128)
    assert macs == shapes.block_params(4096, 14336, 32, 8) - 2 * 4096
    assert shapes.attention_pairs_causal(4) == 1 + 2 + 3 + 4
    assert shapes.attention_pairs_causal(1, start=1000) == 1001
    fl = shapes.block_flops(4096, 14336, 32, 8, 128, 1, 512)
    assert math.isclose(fl / 1e12, 0.2255, rel_tol=2e-3)
    # decode bytes at B=1, pos=1000: weights (436 MB) + KV (4.1 MB) + small terms
    by = shapes.decode_block_bytes(4096, 14336, 32, 8, 128, 1, 1000)
    assert math.isclose(by / 1e6, 440.3, rel_tol=1e-3)
