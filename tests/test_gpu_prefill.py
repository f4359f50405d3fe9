"""GPU parity of the prompt-phase attention (tensor cores) against the fp64
oracle: whole prompts, prompts continued after a cached prefix, one-token
queries and empty queries, ragged in every dimension."""
import math

import numpy as np
import pytest

import oracle
from helpers import (ORC_DTYPE, attn_check, prefill_oracle_threaded, random_case, to_dev,
                     words)
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def run_case(pkv, rs, ctx, qlen, H, D, B, dtype, scale=None):
    import torch
    case = random_case(rs, len(ctx), H, D, B, ctx, dtype)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qs[-1])
    q = words((max(T, 1), H, D), dtype, rs)[:T]
    if scale is None:
        scale = float(np.float32(1 / math.sqrt(D)))
    ref = prefill_oracle_threaded(q, case["kc"], case["vc"], case["bt"], case["ctx"], qs, scale,
                                  dtype)
    dq = to_dev(q, dtype) if T else torch.empty((0, H, D), dtype=torch.float16, device="cuda")
    out = torch.full_like(dq, float("nan"))
    pkv.paged_attention_prefill(out, dq, to_dev(case["kc"], dtype), to_dev(case["vc"], dtype),
                                torch.from_numpy(case["bt"]).cuda(),
                                torch.from_numpy(case["ctx"]).cuda(),
                                torch.from_numpy(qs).cuda(), scale, max(qlen) if qlen else 0)
    assert pkv.get_device_error() == 0
    if T:
        attn_check(out, ref, "prefill dtype=%s D=%d B=%d" % (dtype, D, B))
    return out


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_prefill_parity(pkv, dtype, D, B):
    rs = np.random.default_rng(600 + D + B + (dtype == "bf16"))
    # (context, new tokens): whole prompts, continued prompts, one-token rows
    pairs = [(1, 1), (17, 17), (64, 64), (65, 65), (130, 130), (300, 37), (129, 1), (77, 0),
             (200, 150)]
    ctx = [c for c, _ in pairs]
    qlen = [n for _, n in pairs]
    run_case(pkv, rs, ctx, qlen, 3, D, B, dtype)


@pytest.mark.parametrize("scale", [-0.125, 0.0])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_negative_and_zero_scale(pkv, scale, dtype):
    """A negative scale turns the row max into the min of the raw scores, on
    full tiles and on tiles that cross the diagonal alike; a zero scale gives
    every visible key the same weight (the mean of V over positions 0..p)."""
    rs = np.random.default_rng(650 + int(scale < 0) + 2 * (dtype == "bf16"))
    pairs = [(1, 1), (130, 130), (300, 37), (500, 500), (129, 1)]
    run_case(pkv, rs, [c for c, _ in pairs], [n for _, n in pairs], 3, 128, 16, dtype,
             scale=scale)


def test_prefill_long_prompt(pkv):
    rs = np.random.default_rng(700)
    run_case(pkv, rs, [1024, 700], [1024, 300], 4, 128, 16, "f16")


def test_one_token_queries_match_decode(pkv):
    """qlen == 1 rows are decode rows: both kernels agree within the tolerance."""
    import torch
    rs = np.random.default_rng(701)
    ctx = [5, 40, 333, 1000]
    case = random_case(rs, 4, 8, 128, 16, ctx, "f16")
    q = to_dev(case["q"], "f16")
    kc, vc = to_dev(case["kc"], "f16"), to_dev(case["vc"], "f16")
    bt, cl = torch.from_numpy(case["bt"]).cuda(), torch.from_numpy(case["ctx"]).cuda()
    a, b = torch.empty_like(q), torch.empty_like(q)
    pkv.paged_attention_decode(a, q, kc, vc, bt, cl, 0.088)
    pkv.paged_attention_prefill(b, q, kc, vc, bt, cl,
                                torch.arange(5, dtype=torch.int32, device="cuda"), 0.088, 1)
    ref = oracle.paged_attention_decode(case["q"], case["kc"], case["vc"], case["bt"],
                                        case["ctx"], 0.088)
    attn_check(a, ref, "decode")
    attn_check(b, ref, "prefill qlen=1")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("B", [8, 32])
def test_prefill_unwritten_slots_never_matter(pkv, dtype, B):
    """Slots past each context in its last block, and every block no sequence
    uses, hold NaN / Inf bit patterns: the result equals the one with finite
    contents there, bit for bit (keys past the context get weight 0 and their
    values must never be multiplied in)."""
    import torch
    rs = np.random.default_rng(900 + B + (dtype == "bf16"))
    ctx = [5, 130, 255, 256, 300, 1]
    qlen = [5, 130, 100, 256, 1, 1]
    H, D = 2, 128
    case = random_case(rs, len(ctx), H, D, B, ctx, dtype, spare=9)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qs[-1])
    q = words((T, H, D), dtype, rs)
    nan = 0x7E00 if dtype == "f16" else 0x7FC0
    inf = 0x7C00 if dtype == "f16" else 0x7F80

    def run(kc, vc):
        out = torch.full((T, H, D), float("nan"), dtype=W.torch_dtype(dtype), device="cuda")
        pkv.paged_attention_prefill(out, to_dev(q, dtype), to_dev(kc, dtype), to_dev(vc, dtype),
                                    torch.from_numpy(case["bt"]).cuda(),
                                    torch.from_numpy(case["ctx"]).cuda(),
                                    torch.from_numpy(qs).cuda(), 0.088, max(qlen))
        assert pkv.get_device_error() == 0
        return out

    a = run(case["kc"], case["vc"])
    kc, vc = case["kc"].copy(), case["vc"].copy()
    used = set()
    for s, n in enumerate(ctx):
        nb = -(-n // B)
        used.update(int(x) for x in case["bt"][s, :nb])
        last = case["bt"][s, nb - 1]
        kc[last, :, n - (nb - 1) * B:, :] = nan
        vc[last, :, n - (nb - 1) * B:, :] = inf
    for blk in range(case["nb"]):
        if blk not in used:
            kc[blk] = nan
            vc[blk] = nan
    b = run(kc, vc)
    assert torch.isfinite(b.float()).all()
    assert torch.equal(a, b)
    ref = oracle.paged_attention_prefill(q, case["kc"], case["vc"], case["bt"], case["ctx"], qs,
                                         0.088, ORC_DTYPE[dtype])
    attn_check(a, ref, "prefill dtype=%s B=%d" % (dtype, B))



@pytest.mark.parametrize("dtype,D", [("f16", 128), ("bf16", 128), ("f16", 64)])
def test_prefill_many_items_per_cta(pkv, dtype, D):
    """About 480 (sequence, head, 256-row) work items for 152 persistent CTAs,
    so each CTA takes several in turn and the loads and products that run ahead
    across item boundaries are exercised: prompts of two items, items with both
    128-row tiles, many short continued prompts (one tile, partly filled), and
    empty queries, in random order."""
    rs = np.random.default_rng(950 + D + (dtype == "bf16"))
    pairs = []
    for _ in range(4):                       # whole prompts past 256 rows
        c = int(rs.integers(260, 331))
        pairs.append((c, c))
    for _ in range(8):                       # both tiles of one item
        c = int(rs.integers(140, 301))
        pairs.append((c, int(rs.integers(129, min(c, 256) + 1))))
    for i in range(44):                      # short continuations
        c = int(rs.integers(1, 201))
        pairs.append((c, 0 if i % 15 == 7 else int(rs.integers(1, min(c, 40) + 1))))
    rs.shuffle(pairs)
    ctx = [c for c, _ in pairs]
    qlen = [n for _, n in pairs]
    H = 8
    assert sum(-(-n // 256) for n in qlen) * H > 2 * 152
    run_case(pkv, rs, ctx, qlen, H, D, 16, dtype)


def test_prefill_workload_full_size_sampled(pkv):
    """The prompt-phase workload at its full size (16 prompts of 543..1729
    tokens, 40 heads x 128, fp16, B 16), set up as the benchmark does (block
    manager slots, every prompt token written by reshape_and_cache), checked on
    sampled query rows of every prompt: the rows on each side of the 128-row
    tile and 256-row item edges, the last row and random rows.  Causal row p of
    a prompt is the same attention as a one-token query at context p + 1, so
    each sampled row goes to the oracle as its own one-row sequence."""
    import torch
    spec = W.SPECS["prefill"]
    ctx = W.context_lens(spec)
    S, H, D, B = spec.num_seqs, spec.num_heads, spec.head_dim, spec.block_size
    nb = W.pool_blocks(spec, ctx)
    bm = pkv.BlockManager(nb, B, spec.seed)
    slots = np.concatenate([bm.add_sequence(s, int(ctx[s])) for s in range(S)])
    maxb = max(-(-int(c) // B) for c in ctx)
    tables, _ = bm.export(list(range(S)), maxb)
    T = int(ctx.sum())
    kc = torch.zeros((nb, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    k = W.device_normal((T, H, D), "f16", spec.seed + 1)
    v = W.device_normal((T, H, D), "f16", spec.seed + 2)
    q = W.device_normal((T, H, D), "f16", spec.seed + 3)
    qs = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    pkv.reshape_and_cache(k, v, kc, vc, torch.from_numpy(slots).cuda())
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_prefill(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                                torch.from_numpy(ctx).cuda(), torch.from_numpy(qs).cuda(),
                                spec.scale, int(ctx.max()))
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    rs = np.random.default_rng(951)
    seq, rows = [], []
    for s in range(S):
        n = int(ctx[s])
        pick = {0, 1, n - 1} | {e + d for e in range(128, n, 128) for d in (-1, 0)}
        pick |= {int(x) for x in rs.integers(0, n, size=3)}
        for p in sorted(x for x in pick if 0 <= x < n):
            seq.append(s)
            rows.append(p)
    seq, rows = np.array(seq), np.array(rows)
    grow = qs[seq] + rows                            # row index into q / out
    qh = W.torch_to_words(q[torch.from_numpy(grow).cuda()])
    kh, vh = W.torch_to_words(kc), W.torch_to_words(vc)
    n = len(rows)
    ref = prefill_oracle_threaded(qh, kh, vh, tables[seq], (rows + 1).astype(np.int32),
                                  np.arange(n + 1, dtype=np.int32), spec.scale, "f16")
    attn_check(out[torch.from_numpy(grow).cuda()], ref,
               "prefill workload, %d sampled rows x %d heads" % (n, H))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_output_16_byte_aligned(pkv, dtype):
    """An output that is 16- but not 32-byte aligned takes the 16-byte stores:
    the same bits as a 32-byte aligned output."""
    import torch
    rs = np.random.default_rng(960 + (dtype == "bf16"))
    ctx, qlen, H, D, B = [300, 129, 64], [300, 60, 64], 4, 128, 16
    case = random_case(rs, len(ctx), H, D, B, ctx, dtype)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qs[-1])
    q = to_dev(words((T, H, D), dtype, rs), dtype)
    args = (q, to_dev(case["kc"], dtype), to_dev(case["vc"], dtype),
            torch.from_numpy(case["bt"]).cuda(), torch.from_numpy(case["ctx"]).cuda(),
            torch.from_numpy(qs).cuda(), 0.088, max(qlen))
    a32 = torch.full_like(q, float("nan"))
    pkv.paged_attention_prefill(a32, *args)
    buf = torch.full((T * H * D + 8,), float("nan"), dtype=q.dtype, device="cuda")
    a16 = buf[8:].view(T, H, D)                      # 16 bytes past a 256-byte boundary
    assert a16.data_ptr() % 32 == 16
    pkv.paged_attention_prefill(a16, *args)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(a32.view(torch.int16), a16.view(torch.int16))
    assert not torch.isnan(a32).any()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("jumps", [((128, 8.0),), ((48, 8.0),), ((40, 4.0), (200, 16.0))],
                         ids=["tile-start", "mid-tile", "two-rises"])
def test_prefill_running_max_rises(pkv, dtype, jumps):
    """Keys from a position on are several times larger, so a row's running
    max jumps by far more than the lazy-rescale margin: at the start of the
    second key tile, inside the first (a quarter of 32 keys after others of the
    same tile), or twice (inside the first tile and inside the second).  The
    output rescale, the row-sum rescale and any rescale of weights already
    written for the tile are exercised, on whole and continued prompts."""
    import torch
    rs = np.random.default_rng(970 + (dtype == "bf16") + 7 * len(jumps) + jumps[0][0])
    ctx, qlen, H, D, B = [600, 420], [600, 200], 2, 64, 16
    case = random_case(rs, len(ctx), H, D, B, ctx, dtype)
    kc = case["kc"].copy()
    fl = (lambda w: w.view(np.float16).astype(np.float32)) if dtype == "f16" else \
        (lambda w: (w.astype(np.uint32) << 16).view(np.float32))
    to_w = (lambda f: f.astype(np.float16).view(np.uint16)) if dtype == "f16" else \
        (lambda f: (f.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    for start, factor in jumps:
        for s, n in enumerate(ctx):
            for t in range(start, n):
                b = case["bt"][s, t // B]
                kc[b, :, t % B, :] = to_w(fl(kc[b, :, t % B, :]) * factor)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qs[-1])
    q = words((T, H, D), dtype, rs)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = prefill_oracle_threaded(q, kc, case["vc"], case["bt"], case["ctx"], qs, scale, dtype)
    out = torch.full((T, H, D), float("nan"), dtype=W.torch_dtype(dtype), device="cuda")
    pkv.paged_attention_prefill(out, to_dev(q, dtype), to_dev(kc, dtype), to_dev(case["vc"], dtype),
                                torch.from_numpy(case["bt"]).cuda(),
                                torch.from_numpy(case["ctx"]).cuda(), torch.from_numpy(qs).cuda(),
                                scale, max(qlen))
    assert pkv.get_device_error() == 0
    attn_check(out, ref, "prefill rising max %s dtype=%s" % (jumps, dtype))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_long_context_continued(pkv, dtype):
    """300 new tokens after a 5,700-token cached prefix (about 47 key tiles per
    item), next to a short whole prompt: the long key loop, its running max and
    rescales, and the last partial block."""
    rs = np.random.default_rng(980 + (dtype == "bf16"))
    run_case(pkv, rs, [6000, 90], [300, 90], 2, 128, 16, dtype)


def test_prefill_bad_lengths_flagged_and_skipped(pkv):
    """A sequence with more new tokens than context is flagged and skipped (its
    rows stay unwritten); a sequence with more new tokens than max_query_len
    is flagged, its rows past the last 256-row item the call plans stay
    unwritten and the others are computed; the sequences beside them are
    computed.  Three heads: the second CTA of a pair has no head in the last
    head pair."""
    import torch
    from paged_kv_cache_05_gb300 import pagedkv as P
    rs = np.random.default_rng(960)
    H, D, B, dt = 3, 128, 16, "f16"
    ctx = [300, 90, 500, 600, 40]
    qlen = [300, 120, 200, 600, 1]                  # sequence 1: 120 new tokens, context 90
    case = random_case(rs, len(ctx), H, D, B, [max(c, n) for c, n in zip(ctx, qlen)], dt)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qs[-1])
    q = words((T, H, D), dt, rs)
    out = torch.full((T, H, D), float("nan"), dtype=torch.float16, device="cuda")
    max_query_len = 300                              # two items: sequence 3 keeps rows 0..511
    pkv.paged_attention_prefill(out, to_dev(q, dt), to_dev(case["kc"], dt),
                                to_dev(case["vc"], dt), torch.from_numpy(case["bt"]).cuda(),
                                torch.from_numpy(np.array(ctx, np.int32)).cuda(),
                                torch.from_numpy(qs).cuda(), 0.088, max_query_len)
    assert pkv.get_device_error() == P.DEVERR_BAD_CONTEXT
    got = out.cpu()
    assert torch.isnan(got[qs[1]:qs[2]]).all()
    assert torch.isnan(got[qs[3] + 512:qs[4]]).all()
    for s, rows in [(0, qlen[0]), (2, qlen[2]), (3, 512), (4, qlen[4])]:
        # rows 0 .. rows-1 of sequence s, as a sequence of its own cut at
        # context ctx - qlen + rows (causal rows attend up to their own)
        cut = ctx[s] - qlen[s] + rows
        ref = oracle.paged_attention_prefill(q[qs[s]:qs[s] + rows], case["kc"], case["vc"],
                                             case["bt"][s:s + 1], np.array([cut], np.int32),
                                             np.array([0, rows], np.int32), 0.088, ORC_DTYPE[dt])
        attn_check(got[qs[s]:qs[s] + rows], ref, "sequence %d" % s)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_single_head(pkv, dtype):
    """One head: the units pair heads 0 and 1, so the second CTA of every pair
    has no head and the first computes every item; whole and continued prompts
    of one to five 256-row items."""
    rs = np.random.default_rng(961 + (dtype == "bf16"))
    run_case(pkv, rs, [1200, 700, 300, 90], [1200, 513, 300, 17], 1, 128, 16, dtype)
