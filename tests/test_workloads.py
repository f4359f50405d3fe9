"""The seeded workloads: sizes pinned to the numbers the pages print (CPU only)."""
import json
import os

import numpy as np

from paged_kv_cache_05_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "pages_facts.json")))


def test_opt13b_kv_bytes_per_token_is_800_kib():
    sh = FACTS["opt13b_shape"]
    per_token = 2 * sh["layers"] * sh["heads"] * sh["head_dim"] * 2   # K+V, fp16
    assert per_token == FACTS["opt13b_kv_per_token_kib"]["value"] * 1024
    assert per_token == W.OPT13B_KV_BYTES_PER_TOKEN


def test_opt13b_capacity_reading_is_gib():
    cap = FACTS["opt13b_capacity"]
    slots = cap["kv_gb"] * W.GIB / W.OPT13B_KV_BYTES_PER_TOKEN
    assert round(slots / 1000, 1) == cap["max_slots_k"]      # 15,728.6 -> 15.7K
    spec = W.SPECS["opt13b"]
    ctx = W.context_lens(spec)
    blocks = W.pool_blocks(spec, ctx)
    assert (cap["kv_gb"] * W.GIB // spec.layers) // (2 * 40 * 16 * 128 * 2) == 983
    assert blocks >= 983 and blocks >= W.blocks_needed(ctx, 16)


def test_default_block_size_is_16():
    assert W.SPECS["opt13b"].block_size == FACTS["default_block_size"]["value"]


def test_context_lengths_seeded_and_in_range():
    for name, (lo, hi) in {"opt13b": (1, 2048), "short": (20, 300),
                           "long": (8192, 32768)}.items():
        spec = W.SPECS[name]
        a, b = W.context_lens(spec), W.context_lens(spec)
        assert np.array_equal(a, b) and a.shape == (spec.num_seqs,)
        assert a.min() >= lo and a.max() <= hi
    ctx = W.context_lens(W.SPECS["opt13b"])
    assert 200 < np.median(ctx) < 450          # lognormal, median ~300
    assert list(W.context_lens(W.SPECS["tiny"])) == [1, 15, 16, 37]


def test_shared_prefix_lengths():
    spec = W.SPECS["shared_prefix"]
    p, s = W.prompt_and_suffix_lens(spec)
    assert p.shape == (32,) and s.shape == (192,)
    assert p.min() >= 128 and p.max() <= 1024 and s.min() >= 1 and s.max() <= 512
    ctx = W.context_lens(spec)
    assert np.array_equal(ctx, np.repeat(p, 6) + s)


def test_long_pool_is_80_gb():
    spec = W.SPECS["long"]
    nb = W.pool_blocks(spec, W.context_lens(spec))
    per_block = 2 * 32 * 16 * 128 * 2
    assert nb * per_block <= 80e9 < (nb + 1) * per_block


def test_normal_words_are_16_bit_and_seeded():
    a = W.normal_words((3, 4), "f16", 1, 0)
    b = W.normal_words((3, 4), "bf16", 1, 0)
    assert a.dtype == np.uint16 and b.dtype == np.uint16
    assert np.array_equal(a, W.normal_words((3, 4), "f16", 1, 0))
