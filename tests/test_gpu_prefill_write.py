"""GPU parity of the prompt phase with the cache write in the same kernel
(whole prompts): the cache it leaves is the one the new-token write
(reshape_and_cache, and the oracle's) leaves, every byte of the pool, and
its attention equals the two-step path's bit for bit and the fp64 oracle
within the tolerance."""
import math

import numpy as np
import pytest

import oracle
from helpers import attn_check, prefill_oracle_threaded, to_dev, words
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def whole_prompts(rs, ctx, H, D, B, dtype, spare=7):
    """Tables and slots from the oracle's block-manager model (seeded, scattered
    placement), the pool's prior contents, and the prompts' q, k, v."""
    need = sum(-(-c // B) for c in ctx)
    m = BlockManagerModel(need + spare, B, int(rs.integers(1 << 30)))
    slots = []
    for s, c in enumerate(ctx):
        slots.extend(m.add_sequence(s, c))
    mb = max(1, max(-(-c // B) for c in ctx))
    bt = np.full((len(ctx), mb), -1, np.int32)
    for s in range(len(ctx)):
        t = m.block_table(s)
        bt[s, :len(t)] = t
    T = sum(ctx)
    return dict(bt=bt, ctx=np.array(ctx, np.int32), slots=np.array(slots, np.int64),
                qs=np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32),
                kc=words((m.num_blocks, H, B, D), dtype, rs),
                vc=words((m.num_blocks, H, B, D), dtype, rs),
                q=words((T, H, D), dtype, rs), k=words((T, H, D), dtype, rs),
                v=words((T, H, D), dtype, rs), T=T, H=H, D=D, B=B, dtype=dtype)


def both_paths(pkv, c, scale):
    """(two-step out, caches) and (fused out, caches), all device tensors."""
    import torch
    dt = c["dtype"]
    q, k, v = to_dev(c["q"], dt), to_dev(c["k"], dt), to_dev(c["v"], dt)
    bt = torch.from_numpy(c["bt"]).cuda()
    cl = torch.from_numpy(c["ctx"]).cuda()
    qs = torch.from_numpy(c["qs"]).cuda()
    maxq = int(c["ctx"].max())
    ka, va = to_dev(c["kc"], dt), to_dev(c["vc"], dt)
    pkv.reshape_and_cache(k, v, ka, va, torch.from_numpy(c["slots"]).cuda())
    oa = torch.full_like(q, float("nan"))
    pkv.paged_attention_prefill(oa, q, ka, va, bt, cl, qs, scale, maxq)
    kb, vb = to_dev(c["kc"], dt), to_dev(c["vc"], dt)
    ob = torch.full_like(q, float("nan"))
    pkv.paged_attention_prefill_write(ob, q, k, v, kb, vb, bt, cl, qs, scale, maxq)
    assert pkv.get_device_error() == 0
    return (oa, ka, va), (ob, kb, vb)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_prefill_write_parity(pkv, dtype, D, B):
    import torch
    rs = np.random.default_rng(5100 + 3 * D + B + (dtype == "bf16"))
    # tile (128) and item (256) boundaries, partial and whole last blocks
    ctx = [1, 17, 64, 65, 127, 128, 129, 255, 256, 257, 300, 600]
    c = whole_prompts(rs, ctx, 3, D, B, dtype)
    scale = float(np.float32(1 / math.sqrt(D)))
    (oa, ka, va), (ob, kb, vb) = both_paths(pkv, c, scale)
    # the cache: every byte as the two-step path and the oracle's write leave it
    kh, vh = c["kc"].copy(), c["vc"].copy()
    oracle.reshape_and_cache(c["k"], c["v"], kh, vh, c["slots"])
    assert np.array_equal(W.torch_to_words(kb), kh)
    assert np.array_equal(W.torch_to_words(vb), vh)
    assert torch.equal(kb, ka) and torch.equal(vb, va)
    # the attention: the same bits as the two-step path, the oracle within tolerance
    assert torch.equal(ob.view(torch.int16), oa.view(torch.int16))
    ref = prefill_oracle_threaded(c["q"], kh, vh, c["bt"], c["ctx"], c["qs"], scale, dtype)
    attn_check(ob, ref, "prefill_write %s D=%d B=%d" % (dtype, D, B))


def test_prefill_write_skips_continued_prompts(pkv):
    """A sequence whose new tokens do not start at position 0 is not a whole
    prompt: it is skipped (rows unwritten, cache untouched) and flagged; the
    whole prompts beside it are computed and written."""
    import torch
    from paged_kv_cache_05_gb300 import pagedkv as P
    rs = np.random.default_rng(5200)
    c = whole_prompts(rs, [40, 300, 90], 2, 128, 16, "f16")
    dt = "f16"
    q, k, v = to_dev(c["q"], dt), to_dev(c["k"], dt), to_dev(c["v"], dt)
    bt = torch.from_numpy(c["bt"]).cuda()
    ctx = c["ctx"].copy()
    ctx[1] += 50                     # sequence 1: 300 new tokens after 50 cached ones
    cl = torch.from_numpy(ctx).cuda()
    bt2 = torch.full((3, bt.shape[1] + 4), -1, dtype=torch.int32, device="cuda")
    bt2[:, :bt.shape[1]] = bt
    kb, vb = to_dev(c["kc"], dt), to_dev(c["vc"], dt)
    out = torch.full_like(q, float("nan"))
    qs = torch.from_numpy(c["qs"]).cuda()
    pkv.paged_attention_prefill_write(out, q, k, v, kb, vb, bt2, cl, qs, 0.088, 300)
    assert pkv.get_device_error() == P.DEVERR_BAD_CONTEXT
    rows1 = slice(int(c["qs"][1]), int(c["qs"][2]))
    assert torch.isnan(out[rows1]).all()
    s1_blocks = [int(x) for x in c["bt"][1] if x >= 0]
    kh = c["kc"].copy()
    vh = c["vc"].copy()
    keep = [i for i in range(len(c["slots"])) if not (rows1.start <= i < rows1.stop)]
    oracle.reshape_and_cache(c["k"][keep], c["v"][keep], kh, vh, c["slots"][keep])
    assert np.array_equal(W.torch_to_words(kb), kh)
    assert np.array_equal(W.torch_to_words(vb), vh)
    assert s1_blocks
    others = [r for r in range(len(c["slots"])) if r not in range(rows1.start, rows1.stop)]
    assert not torch.isnan(out[others]).any()


def test_prefill_write_workload_full_size(pkv):
    """The prompt-phase workload (16 prompts of 543..1729 tokens, 40 heads x
    128, fp16, B 16): the fused call leaves the same pool and the same output
    bits as the two-step path."""
    import torch
    spec = W.SPECS["prefill"]
    ctx = [int(x) for x in W.context_lens(spec)]
    H, D, B = spec.num_heads, spec.head_dim, spec.block_size
    m = BlockManagerModel(sum(-(-c // B) for c in ctx) + 9, B, spec.seed)
    slots = []
    for s_, c in enumerate(ctx):
        slots.extend(m.add_sequence(s_, c))
    mb = max(-(-c // B) for c in ctx)
    bt = np.full((len(ctx), mb), -1, np.int32)
    for s_ in range(len(ctx)):
        t = m.block_table(s_)
        bt[s_, :len(t)] = t
    T = sum(ctx)
    q = W.device_normal((T, H, D), "f16", 5301)
    k = W.device_normal((T, H, D), "f16", 5302)
    v = W.device_normal((T, H, D), "f16", 5303)
    ka = W.device_normal((m.num_blocks, H, B, D), "f16", 5304)
    va = W.device_normal((m.num_blocks, H, B, D), "f16", 5305)
    kb, vb = ka.clone(), va.clone()
    tb, cl = torch.from_numpy(bt).cuda(), torch.tensor(ctx, dtype=torch.int32, device="cuda")
    qs = torch.from_numpy(np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)).cuda()
    pkv.reshape_and_cache(k, v, ka, va, torch.tensor(slots, dtype=torch.int64, device="cuda"))
    oa = torch.full_like(q, float("nan"))
    pkv.paged_attention_prefill(oa, q, ka, va, tb, cl, qs, spec.scale, max(ctx))
    ob = torch.full_like(q, float("nan"))
    pkv.paged_attention_prefill_write(ob, q, k, v, kb, vb, tb, cl, qs, spec.scale, max(ctx))
    assert pkv.get_device_error() == 0
    assert torch.equal(kb, ka) and torch.equal(vb, va)
    assert torch.equal(ob.view(torch.int16), oa.view(torch.int16))
