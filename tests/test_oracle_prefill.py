"""Pins for the oracle's prompt-phase attention (CPU only): torch's fp64 causal
scaled-dot-product attention on the gathered prompt (library special case),
a query of one token equals the decode definition, the first token of a
prompt returns its own V exactly, and a prompt split in chunks gives the same
rows as the whole prompt."""
import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_attention import gathered, make_batch, widen


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
@pytest.mark.parametrize("B", [8, 16, 64])
def test_full_prompt_matches_torch_causal_sdpa(dtype, B):
    rs = np.random.default_rng(40 + B + dtype)
    ctx = [1, 5, 33, 70]
    H, D = 2, 32
    _, kc, vc, bt, cl = make_batch(rs, len(ctx), H, D, B, ctx, dtype)
    qs = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    from test_oracle_attention import rand_words
    q = rand_words((int(qs[-1]), H, D), dtype, rs)
    scale = float(np.float32(1 / math.sqrt(D)))
    out = oracle.paged_attention_prefill(q, kc, vc, bt, cl, qs, scale, dtype)
    qd, kd, vd = widen(q, dtype), widen(kc, dtype), widen(vc, dtype)
    for s, n in enumerate(ctx):
        for h in range(H):
            K = torch.from_numpy(gathered(kd, bt[s], n, h, B)).view(1, 1, n, D)
            V = torch.from_numpy(gathered(vd, bt[s], n, h, B)).view(1, 1, n, D)
            Q = torch.from_numpy(qd[qs[s]:qs[s + 1], h]).view(1, 1, n, D)
            ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale,
                                                                   is_causal=True)
            np.testing.assert_allclose(out[qs[s]:qs[s + 1], h], ref.view(n, D).numpy(),
                                       rtol=1e-12, atol=1e-13)


def test_one_query_token_is_the_decode_definition():
    rs = np.random.default_rng(50)
    ctx = [3, 17, 40]
    q, kc, vc, bt, cl = make_batch(rs, 3, 4, 64, 16, ctx)
    qs = np.arange(4, dtype=np.int32)
    a = oracle.paged_attention_prefill(q, kc, vc, bt, cl, qs, 0.125)
    b = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.125)
    assert np.array_equal(a, b)


def test_first_prompt_token_returns_its_value_and_chunks_agree():
    rs = np.random.default_rng(51)
    n, H, D, B = 45, 2, 64, 16
    _, kc, vc, bt, cl = make_batch(rs, 1, H, D, B, [n])
    from test_oracle_attention import rand_words
    q = rand_words((n, H, D), oracle.F16, rs)
    whole = oracle.paged_attention_prefill(q, kc, vc, bt, cl, np.array([0, n]), 0.1)
    first = whole[0]
    assert np.array_equal(first, widen(vc, oracle.F16)[bt[0, 0], :, 0, :])
    # the same prompt processed as a 20-token chunk after a 25-token prefix
    tail = oracle.paged_attention_prefill(q[25:], kc, vc, bt, cl, np.array([0, 20]), 0.1)
    assert np.array_equal(tail, whole[25:])


def test_query_longer_than_context_is_rejected():
    rs = np.random.default_rng(52)
    q, kc, vc, bt, cl = make_batch(rs, 1, 1, 32, 16, [4])
    with pytest.raises(ValueError):
        oracle.paged_attention_prefill(np.zeros((5, 1, 32), np.uint16), kc, vc, bt, cl,
                                       np.array([0, 5]), 0.1)
