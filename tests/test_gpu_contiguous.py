"""GPU parity of the contiguous-layout decode kernel (the baseline layout that
paging is measured against: each sequence's K/V in one region reserved for the
maximum length, no block table).

The oracle takes a paged pool, so the same K/V are also laid out as a pool
whose block tables are the identity (sequence s holds blocks s*n .. s*n+n-1);
placement does not change attention, which the oracle's own pins fix."""
import math

import numpy as np
import pytest

import oracle
from helpers import ORC_DTYPE, attn_check, host_threads, to_dev, words
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def as_identity_pool(kv: np.ndarray, B: int):
    """[S][H][T][D] words -> a pool [S*n][H][B][D] holding the same tokens, with
    the identity tables [S][n] (n = ceil(T / B); padding tokens are zero)."""
    S, H, T, D = kv.shape
    n = -(-T // B)
    pad = np.zeros((S, H, n * B, D), kv.dtype)
    pad[:, :, :T] = kv
    pool = pad.reshape(S, H, n, B, D).transpose(0, 2, 1, 3, 4).reshape(S * n, H, B, D)
    tables = np.arange(S * n, dtype=np.int32).reshape(S, n)
    return np.ascontiguousarray(pool), tables


def oracle_rows(q, k, v, ctx, scale, dtype):
    kp, tables = as_identity_pool(k, 16)
    vp, _ = as_identity_pool(v, 16)
    return oracle.paged_attention_decode_threaded(q, kp, vp, tables, np.asarray(ctx, np.int32),
                                                  scale, ORC_DTYPE[dtype],
                                                  threads=host_threads())


def run(pkv, q, k, v, ctx, scale, partition):
    import torch
    out = torch.full_like(q, float("nan"))
    pkv.contiguous_attention_decode(out, q, k, v, torch.from_numpy(np.asarray(ctx, np.int32))
                                    .cuda(), scale, partition_size=partition)
    assert pkv.get_device_error() == 0
    return out


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_contiguous_parity_ragged(pkv, dtype, D):
    rs = np.random.default_rng(2100 + D + (dtype == "bf16"))
    T = 1037                                     # not a multiple of the step
    ctx = [1, 2, 15, 16, 17, 0, 31, 32, 33, 300, 1000, T]
    S, H = len(ctx), 3
    q_h = words((S, H, D), dtype, rs)
    k_h = words((S, H, T, D), dtype, rs)
    v_h = words((S, H, T, D), dtype, rs)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle_rows(q_h, k_h, v_h, ctx, scale, dtype)
    q, k, v = to_dev(q_h, dtype), to_dev(k_h, dtype), to_dev(v_h, dtype)
    sub = 2048 // D
    for part in (0, sub, 512):
        out = run(pkv, q, k, v, ctx, scale, part)
        attn_check(out, ref, "contiguous %s D=%d partition=%d" % (dtype, D, part))
    zero = [s for s in range(S) if ctx[s] == 0]
    assert (out[zero] == 0).all()


def test_contiguous_equals_paged_with_identity_tables_bit_for_bit(pkv):
    """With a fixed split the two kernels stream the same steps in the same
    order and differ only in how a step's address is found: the outputs are
    the same bits."""
    import torch
    rs = np.random.default_rng(2200)
    S, H, D, T = 40, 8, 128, 700
    ctx = [int(c) for c in rs.integers(0, T + 1, size=S)]
    q_h = words((S, H, D), "f16", rs)
    k_h = words((S, H, T, D), "f16", rs)
    v_h = words((S, H, T, D), "f16", rs)
    q, k, v = to_dev(q_h, "f16"), to_dev(k_h, "f16"), to_dev(v_h, "f16")
    kp, tables = as_identity_pool(k_h, 16)
    vp, _ = as_identity_pool(v_h, 16)
    scale = 0.0883883
    cl = torch.from_numpy(np.asarray(ctx, np.int32)).cuda()
    for part in (16, 512):
        a = run(pkv, q, k, v, ctx, scale, part)
        b = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(b, q, to_dev(kp, "f16"), to_dev(vp, "f16"),
                                   torch.from_numpy(tables).cuda(), cl, scale,
                                   partition_size=part)
        assert pkv.get_device_error() == 0
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), part


def test_contiguous_opt13b_shape_every_row(pkv):
    """The OPT-13B-shaped batch (64 x 40 heads x 128, fp16, lognormal lengths up
    to 2048) in the contiguous layout, every row against the oracle, balanced
    and 512-token splits."""
    import torch
    spec = W.SPECS["opt13b"]
    ctx = W.context_lens(spec)
    S, H, D = spec.num_seqs, spec.num_heads, spec.head_dim
    T = int(ctx.max())
    q = W.device_normal((S, H, D), "f16", 9101)
    k = W.device_normal((S, H, T, D), "f16", 9102)
    v = W.device_normal((S, H, T, D), "f16", 9103)
    ref = oracle_rows(W.torch_to_words(q), W.torch_to_words(k), W.torch_to_words(v), ctx,
                      spec.scale, "f16")
    for part in (0, 512):
        attn_check(run(pkv, q, k, v, ctx, spec.scale, part), ref,
                   "contiguous opt13b partition=%d" % part)
    del k, v
    torch.cuda.empty_cache()


def test_contiguous_context_beyond_the_layout_is_flagged(pkv):
    """A context length above max_context_len is clamped (never read past the
    row) and reported."""
    import torch
    from paged_kv_cache_05_gb300 import pagedkv as P
    rs = np.random.default_rng(2300)
    S, H, D, T = 4, 2, 64, 100
    q_h = words((S, H, D), "f16", rs)
    k_h = words((S, H, T, D), "f16", rs)
    v_h = words((S, H, T, D), "f16", rs)
    q, k, v = to_dev(q_h, "f16"), to_dev(k_h, "f16"), to_dev(v_h, "f16")
    out = torch.full_like(q, float("nan"))
    pkv.contiguous_attention_decode(out, q, k, v,
                                    torch.tensor([5, T + 50, 7, T], dtype=torch.int32,
                                                 device="cuda"), 0.125)
    assert pkv.get_device_error() == P.DEVERR_BAD_CONTEXT
    ref = oracle_rows(q_h, k_h, v_h, [5, T, 7, T], 0.125, "f16")
    attn_check(out, ref, "clamped context")
