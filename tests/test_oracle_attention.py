"""Pins for the oracle's attention (CPU only).

Each test checks the oracle against something other than itself: numpy's and
torch's own 16-bit decoders, torch's fp64 scaled-dot-product attention on the
gathered sequence, closed forms, the block-indexed formula of the paper's
section 4.1 (zhaifeiyue.github.io detail page), and the invariances the pages
claim (non-contiguous placement is transparent; shared blocks give shared
results).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.block_manager import BlockManagerModel

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "pages_facts.json")))


def rand_words(shape, dtype, rs):
    x = rs.standard_normal(size=shape).astype(np.float32)
    if dtype == oracle.F16:
        return x.astype(np.float16).view(np.uint16)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def widen(words, dtype):
    """Library decode of 16-bit words (numpy float16 / torch bfloat16)."""
    if dtype == oracle.F16:
        return words.view(np.float16).astype(np.float64)
    return torch.from_numpy(words.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def make_batch(rs, S, H, D, B, ctx, dtype=oracle.F16, spare=3):
    """Random pool and a random (non-contiguous) placement of each sequence's blocks."""
    nblk = [-(-c // B) for c in ctx]
    num_blocks = sum(nblk) + spare
    max_blocks = max(max(nblk), 1)
    perm = rs.permutation(num_blocks)
    bt = np.full((S, max_blocks), -1, dtype=np.int32)
    k = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[k:k + nblk[s]]
        k += nblk[s]
    kc = rand_words((num_blocks, H, B, D), dtype, rs)
    vc = rand_words((num_blocks, H, B, D), dtype, rs)
    q = rand_words((S, H, D), dtype, rs)
    return q, kc, vc, bt, np.array(ctx, dtype=np.int32)


def gathered(kc, bt_row, n, h, B):
    """Contiguous [n][D] rows of one sequence/head by library fancy indexing."""
    pos = np.arange(n)
    return kc[bt_row[pos // B], h, pos % B, :]


# --- decoders ---------------------------------------------------------------

def test_f16_decode_matches_numpy_all_patterns():
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(w)
    ref = w.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_matches_torch_all_patterns():
    w = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(w)
    ref = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


# --- library special case ----------------------------------------------------

@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_matches_torch_sdpa_fp64(dtype, B):
    rs = np.random.default_rng(7 + B + dtype)
    S, H, D = 5, 3, 64
    ctx = [1, B - 1, B, 2 * B + 3, 70]
    q, kc, vc, bt, cl = make_batch(rs, S, H, D, B, ctx, dtype)
    scale = float(np.float32(1 / math.sqrt(D)))
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, scale, dtype)
    qd, kd, vd = widen(q, dtype), widen(kc, dtype), widen(vc, dtype)
    for s in range(S):
        for h in range(H):
            K = torch.from_numpy(gathered(kd, bt[s], ctx[s], h, B))
            V = torch.from_numpy(gathered(vd, bt[s], ctx[s], h, B))
            Q = torch.from_numpy(qd[s, h])
            ref = torch.nn.functional.scaled_dot_product_attention(
                Q.view(1, 1, 1, D), K.view(1, 1, -1, D), V.view(1, 1, -1, D), scale=scale)
            np.testing.assert_allclose(out[s, h], ref.view(D).numpy(), rtol=1e-12, atol=1e-13)


# --- the block-indexed formula (section 4.1) ----------------------------------

@pytest.mark.parametrize("B", [4, 8, 16, 64])
def test_blockwise_formula_equals_contiguous(B):
    rs = np.random.default_rng(100 + B)
    ctx = [1, 2, B, B + 1, 3 * B - 1, 97]
    q, kc, vc, bt, cl = make_batch(rs, len(ctx), 2, 32, B, ctx)
    a = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.17)
    b = oracle.paged_attention_decode_blockwise(q, kc, vc, bt, cl, 0.17)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


# --- closed forms --------------------------------------------------------------

def test_context_one_returns_v_exactly():
    rs = np.random.default_rng(3)
    q, kc, vc, bt, cl = make_batch(rs, 3, 4, 64, 16, [1, 1, 1])
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.125)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(out[s, h], widen(vc, oracle.F16)[bt[s, 0], h, 0])


def test_two_tokens_closed_form():
    rs = np.random.default_rng(4)
    B, D = 16, 64
    q, kc, vc, bt, cl = make_batch(rs, 1, 1, D, B, [2])
    scale = 0.3
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, scale)[0, 0]
    qd = widen(q, oracle.F16)[0, 0]
    k0, k1 = widen(kc, oracle.F16)[bt[0, 0], 0, :2]
    v0, v1 = widen(vc, oracle.F16)[bt[0, 0], 0, :2]
    z0, z1 = scale * float(qd @ k0), scale * float(qd @ k1)
    w1 = 1.0 / (1.0 + math.exp(z0 - z1))  # logistic weight of the second token
    np.testing.assert_allclose(out, v0 + w1 * (v1 - v0), rtol=1e-12, atol=1e-14)


def test_zero_scale_gives_mean_of_values():
    rs = np.random.default_rng(5)
    ctx = [5, 16, 33]
    q, kc, vc, bt, cl = make_batch(rs, 3, 2, 32, 16, ctx)
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.0)
    vd = widen(vc, oracle.F16)
    for s, n in enumerate(ctx):
        for h in range(2):
            np.testing.assert_allclose(out[s, h], gathered(vd, bt[s], n, h, 16).mean(axis=0),
                                       rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value():
    # q parallel to one key and a large scale: softmax mass concentrates there
    B, D, n = 16, 64, 20
    rs = np.random.default_rng(6)
    q, kc, vc, bt, cl = make_batch(rs, 1, 1, D, B, [n])
    vd = widen(vc, oracle.F16)
    kc[:] = np.float16(0).view(np.uint16)
    target = 13
    blk, off = bt[0, target // B], target % B
    kc[blk, 0, off, :] = np.float16(1.0).view(np.uint16)
    q[0, 0, :] = np.float16(1.0).view(np.uint16)
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 1.0)[0, 0]
    # scores: 64 for the target, 0 elsewhere -> weight of the rest = 19 e^-64
    np.testing.assert_allclose(out, vd[blk, 0, off], rtol=0, atol=1e-25)


def test_zero_context_gives_zero_row():
    rs = np.random.default_rng(8)
    q, kc, vc, bt, cl = make_batch(rs, 2, 2, 64, 16, [0, 5])
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.125)
    assert np.all(out[0] == 0) and np.any(out[1] != 0)


# --- invariances the pages claim ----------------------------------------------

def test_physical_placement_is_transparent():
    """Any permutation of physical block ids (pool rows moved with it): identical output."""
    rs = np.random.default_rng(9)
    ctx = [3, 17, 40, 64, 65]
    q, kc, vc, bt, cl = make_batch(rs, 5, 4, 64, 16, ctx, spare=20)
    a = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.125)
    perm = rs.permutation(kc.shape[0])          # new id of old block i is perm[i]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    b = oracle.paged_attention_decode(q, kc2, vc2, bt2, cl, 0.125)
    assert np.array_equal(a, b)


def test_output_independent_of_block_size():
    """Same per-token values written with block sizes 8..64: bit-identical output."""
    rs = np.random.default_rng(10)
    S, H, D = 4, 2, 64
    ctx = [1, 20, 63, 130]
    q = rand_words((S, H, D), oracle.BF16, rs)
    toks = [(rand_words((n, H, D), oracle.BF16, rs), rand_words((n, H, D), oracle.BF16, rs))
            for n in ctx]
    outs = []
    for B in (8, 16, 32, 64):
        bm = BlockManagerModel(64, B, seed=11)
        nb = 64
        kc = np.zeros((nb, H, B, D), np.uint16)
        vc = np.zeros((nb, H, B, D), np.uint16)
        maxb = max(-(-n // B) for n in ctx)
        bt = np.full((S, maxb), -1, np.int32)
        for s, n in enumerate(ctx):
            slots = bm.add_sequence(s, n)
            oracle.reshape_and_cache(toks[s][0], toks[s][1], kc, vc, np.array(slots))
            t = bm.block_table(s)
            bt[s, :len(t)] = t
        outs.append(oracle.paged_attention_decode(q, kc, vc, bt, np.array(ctx), 0.125,
                                                  oracle.BF16))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def test_sharing_diagram_shared_blocks_give_shared_results():
    """Garden section 5.1: tables [7,3,12] and [7,3,9]; equal queries over the
    shared part give equal outputs, and diverge once the unique block is read."""
    f = FACTS["sharing_diagram"]
    rs = np.random.default_rng(12)
    B, H, D = 16, 2, 64
    kc = rand_words((16, H, B, D), oracle.F16, rs)
    vc = rand_words((16, H, B, D), oracle.F16, rs)
    q1 = rand_words((1, H, D), oracle.F16, rs)
    q = np.concatenate([q1, q1])
    bt = np.array([f["table_a"], f["table_b"]], dtype=np.int32)
    same = oracle.paged_attention_decode(q, kc, vc, bt, np.array([32, 32]), 0.125)
    assert np.array_equal(same[0], same[1])
    diff = oracle.paged_attention_decode(q, kc, vc, bt, np.array([40, 40]), 0.125)
    assert not np.array_equal(diff[0], diff[1])


def test_bad_table_rejected():
    rs = np.random.default_rng(13)
    q, kc, vc, bt, cl = make_batch(rs, 1, 1, 32, 16, [20])
    bt[0, 1] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.1)
