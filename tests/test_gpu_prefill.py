"""GPU parity of the prompt-phase attention (tensor cores) against the fp64
oracle: whole prompts, prompts continued after a cached prefix, one-token
queries and empty queries, ragged in every dimension."""
import math

import numpy as np
import pytest

import oracle
from helpers import ORC_DTYPE, attn_check, random_case, to_dev, words
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def run_case(pkv, rs, ctx, qlen, H, D, B, dtype):
    import torch
    case = random_case(rs, len(ctx), H, D, B, ctx, dtype)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(qs[-1])
    q = words((max(T, 1), H, D), dtype, rs)[:T]
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.paged_attention_prefill(q, case["kc"], case["vc"], case["bt"], case["ctx"], qs,
                                         scale, ORC_DTYPE[dtype])
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
@pytest.mark.parametrize("B", [8, 16, 64])
def test_prefill_parity(pkv, dtype, D, B):
    rs = np.random.default_rng(600 + D + B + (dtype == "bf16"))
    # (context, new tokens): whole prompts, continued prompts, one-token rows
    pairs = [(1, 1), (17, 17), (64, 64), (65, 65), (130, 130), (300, 37), (129, 1), (77, 0),
             (200, 150)]
    ctx = [c for c, _ in pairs]
    qlen = [n for _, n in pairs]
    run_case(pkv, rs, ctx, qlen, 3, D, B, dtype)


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
