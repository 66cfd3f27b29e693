"""The byte / flop accounting (the bench's roofline numerator) reproduces the
figures the pages print (tests/golden/page_figures.json)."""
import json
import os

import pytest

from gqa_decode_attention_02_gb300 import analytic as A

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def g(name):
    return GOLD[name]["value"], GOLD[name]["inputs"]


def test_kv_bytes_per_token_formula():
    v, i = g("kv_bytes_per_token_24L_2kv_h64_fp16")
    assert A.kv_bytes_per_token(i["layers"], i["kv_heads"], i["head_dim"], i["elem_bytes"]) == v


def test_allocator_bytes_for_295_tokens():
    v, i = g("allocator_bytes_295_tokens")
    assert i["tokens"] * A.kv_bytes_per_token(i["layers"], i["kv_heads"], i["head_dim"],
                                              i["elem_bytes"]) == v
    # the paged reservation: 19 blocks of 16 = 304 slots, 9 slots of fragmentation
    assert A.paged_kv_bytes(295, 24, 2, 64, 2) == 304 * 12288 == 3735552


def test_cache_depends_only_on_total_tokens():
    v, i = g("cache_bytes_65536_tokens_MB")
    per = A.kv_bytes_per_token(i["layers"], i["kv_heads"], i["head_dim"], i["elem_bytes"])
    for users, tokens in ((32, 2048), (64, 1024), (128, 512)):
        assert users * tokens * per == v * 2**20


def test_mha_and_7b_figures():
    v, i = g("mha_bytes_per_token_14_heads")
    assert A.kv_bytes_per_token(i["layers"], i["kv_heads"], i["head_dim"], i["elem_bytes"]) == v
    assert v // 12288 == 7  # exactly the 14 / 2 head ratio
    v, i = g("kv_bytes_per_token_7b_KB")
    assert A.kv_bytes_per_token(i["layers"], i["kv_heads"], i["head_dim"],
                                i["elem_bytes"]) == v * 1024


def test_score_buffer_sizes():
    v, i = g("score_bytes_4096_recompute_MB")
    assert round(A.score_matrix_bytes(i["n"], cached=False) / 1e6) == v
    v, i = g("score_bytes_4096_cached_KB")
    assert A.score_matrix_bytes(i["n"], cached=True) == v * 1024


def test_accelerator_intensities():
    for name in ("h100_intensity", "rtx4080_intensity"):
        v, i = g(name)
        assert round(A.accelerator_intensity(i["flops"], i["bytes"])) == v
    assert A.decode_attention_intensity(1024) < 1.0
    assert A.decode_attention_intensity(1024, T=1024) == 512


def test_llama2_13b_tables():
    v, i = g("llama2_13b_num_params")
    assert A.transformer_params(i["V"], i["D"], i["F"], i["L"], i["N"], i["K"], i["H"]) == v
    v, i = g("llama2_13b_kv_per_seq_1024")
    assert i["S"] * i["K"] * i["H"] * i["L"] * 2 * 2 == v
    t = GOLD["llama2_13b_table"]
    c = t["inputs"]
    for row in t["rows"]:
        mem, lat, tput = A.decode_step_model(row["B"], c["S"], c["V"], c["D"], c["F"], c["L"],
                                             c["N"], row["K"], c["H"], c["bandwidth"])
        assert A.round_half_up(mem / 1e9, 1) == pytest.approx(row["memory_GB"])
        assert A.round_half_up(lat * 1e3, 1) == pytest.approx(row["latency_ms"])
        assert A.round_half_up(tput) == row["tokens_per_s"]


@pytest.mark.parametrize("name", ["spec_tokens_alpha_0p3_gamma_4", "spec_speedup_alpha_0p9_gamma_8",
                                  "spec_speedup_alpha_0p3_gamma_8",
                                  "spec_speedup_alpha_0p3_gamma_4_c_fifth"])
def test_speculative_calculator(name):
    v, i = g(name)
    d = GOLD[name]["digits"]
    if "c" in i:
        got = A.spec_speedup(i["alpha"], i["gamma"], i["c"])
    else:
        got = A.spec_expected_tokens(i["alpha"], i["gamma"])
    assert A.round_half_up(got, d) == pytest.approx(v)


def test_algorithmic_bytes_config_1():
    # one sequence of 295 tokens, N=14/K=2/H=64 fp16: 75,520 bytes of keys and
    # as many of values, plus q in / out back, 19 block ids and one length
    b = A.attention_algorithmic_bytes([295], T=1, N=14, K=2, H=64, elem_bytes=2)
    assert 295 * 2 * 64 * 2 == 75520
    assert b == 2 * 75520 + 2 * 14 * 64 * 2 + 4 * 19 + 4


def test_accept_sampled_bytes_by_hand():
    # T=5 (4 drafts), V=1000.  a=0: one test, a residual draw over q and p;
    # a=4: four tests, a draw over q alone.
    T, V = 5, 1000
    per_seq_fixed = 8 * 5 + 4 * 4 + 16
    assert A.accept_sampled_bytes([0], T, V) == per_seq_fixed + 8 * 1 + 2 * 4000
    assert A.accept_sampled_bytes([4], T, V) == per_seq_fixed + 8 * 4 + 1 * 4000
    assert A.accept_sampled_bytes([0, 4], T, V) == (A.accept_sampled_bytes([0], T, V)
                                                    + A.accept_sampled_bytes([4], T, V))
    # T=1: no drafts, one uniform, a draw over q
    assert A.accept_sampled_bytes([0], 1, V) == 8 + 16 + 4000


def test_windowed_bytes_by_hand():
    # ctx 100, T=1, W=20: positions 80..99 (20 tokens) in blocks 5 and 6;
    # ctx 10: all 10 tokens in block 0.  K=2, H=64, fp16.
    b = A.attention_algorithmic_bytes([100, 10], T=1, N=4, K=2, H=64, elem_bytes=2, window=20)
    assert b == (20 + 10) * 2 * 2 * 64 * 2 + 2 * 2 * 1 * 4 * 64 * 2 + 4 * (2 + 1) + 4 * 2
    # a window wider than every context is full attention
    assert (A.attention_algorithmic_bytes([100, 10], 3, 4, 2, 64, 2, window=500)
            == A.attention_algorithmic_bytes([100, 10], 3, 4, 2, 64, 2))
    # T=3, W=20, ctx 100: positions 78..99 (22 tokens) from block 4
    b3 = A.attention_algorithmic_bytes([100], T=3, N=4, K=2, H=64, elem_bytes=2, window=20)
    assert b3 == 22 * 2 * 2 * 64 * 2 + 2 * 3 * 4 * 64 * 2 + 4 * (7 - 4) + 4


def test_one_byte_cache_bytes_by_hand():
    # ctx 100, T=1, K=2, H=128: 100 tokens x 2 (K, V) x 2 heads x (128 + 4) bytes,
    # q and out in bf16, 7 block ids, one length
    b = A.attention_algorithmic_bytes([100], T=1, N=8, K=2, H=128, elem_bytes=2,
                                      kv_elem_bytes=1, row_scale_bytes=4)
    assert b == 100 * 2 * 2 * 132 + 2 * 1 * 8 * 128 * 2 + 4 * 7 + 4
    assert A.kv_append_quant_bytes(3, 1, 2, 128, 2) == 2 * 3 * 2 * (256 + 128 + 4) + 12 + 12


def test_tree_acceptance_and_compaction_bytes_by_hand():
    # B=2 sequences of a 26-node tree over V=1000: logits, 25 drafts and 26
    # parent entries each; accepted / next token / length read and written and
    # a 25-entry branch out
    assert A.accept_tree_bytes(2, 26, 1000) == (2 * 26 * 1000 * 4 + 2 * 25 * 4 + 2 * 26 * 4
                                                + 2 * 4 * (25 + 4))
    # compaction of 3 + 0 kept nodes, K=8, H=128: each row of K and V read and
    # written once (bf16), plus the branch and two ints per sequence
    assert A.kv_compact_bytes([3, 0], 8, 128, 2, 26) == (3 * 2 * 2 * 8 * 128 * 2
                                                         + 2 * 4 * (25 + 2))
    # one-byte rows carry their fp32 scale
    assert A.kv_compact_bytes([1], 2, 128, 1, 4, scale_bytes=4) == 2 * 2 * 2 * 132 + 4 * 5
