"""The byte/FLOP model behind the roofline numbers, pinned to the per-token
accounting of "Dynamic Speculative Decoding" (Attention Analysis)."""

import os

from speculative_decoding_tree_sv_gb300 import cost

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLDEN, "roofline_blog_accounting.txt")) as f:
        for line in f:
            t = line.split()
            if t and t[0] == "case":
                yield [int(x) for x in t[1:]]


def test_blog_per_token_accounting():
    for batch, heads, dim, ctx, n, f_tok, b_tok, ai in _cases():
        # multi-head attention: as many KV heads as query heads
        flops, bytes_ = cost.per_context_token(heads, heads, dim, n)
        assert flops * batch == f_tok
        assert bytes_ * batch == b_tok
        assert flops // bytes_ == ai
        # the whole-launch model agrees on the context part
        tot_f = cost.attention_flops([ctx], [[0] + [1] * (n - 1)], heads, dim)
        tree_f = 4 * heads * dim * (1 + 2 * (n - 1))
        assert tot_f - tree_f == f_tok * ctx


def test_gqa_multiplies_intensity_by_group():
    f1, b1 = cost.per_context_token(32, 32, 128, 60)
    f4, b4 = cost.per_context_token(32, 8, 128, 60)
    assert f1 == f4 and b1 == 4 * b4
    assert f4 / b4 == 60 * 4


def test_llama_eagle_bytes_per_layer():
    # 4096 context tokens, 60 nodes, 8 KV heads of 128: ~18 MB per layer
    b = cost.attention_bytes([4096], [60], 32, 8, 128)
    assert 17.9e6 < b < 18.1e6


def test_partial_context_keys():
    assert cost.context_keys(37, 16, [0, 2]) == 16 + 5
    assert cost.context_keys(60000, 16) == 60000
