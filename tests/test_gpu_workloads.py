"""GPU parity at the workloads' full sizes.

Cache kernels: whole pools compared bit for bit with the oracle's own
copy-on-write and new-token writes applied to host copies of the same seeded
inputs.  Attention: every element of every row (all sequences, all heads)
against the fp64 oracle computed from the oracle's pools, in each split mode the
workload runs (the balanced split's dynamically claimed chunks only exist at
these sizes).  Block tables: the C++ manager's, checked equal to the oracle's
model first.
"""
import numpy as np
import pytest

import oracle
from helpers import attn_check, device_blocks_to_host, host_threads, sampled_oracle
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def managers(pkv, nb, B, seed):
    return pkv.BlockManager(nb, B, seed), BlockManagerModel(nb, B, seed)


def same_tables(bm, model, ids, max_blocks):
    tables, ctx = bm.export(ids, max_blocks)
    for i, s in enumerate(ids):
        t = model.block_table(s)
        assert tables[i, :len(t)].tolist() == t
        assert ctx[i] == model.context_len(s)
    return tables, ctx


def test_opt13b_decode_step(pkv):
    """64 sequences x 40 heads x 128, fp16, B 16, lognormal lengths; one layer."""
    import torch
    spec = W.SPECS["opt13b"]
    ctx = W.context_lens(spec)
    S, H, D, B = spec.num_seqs, spec.num_heads, spec.head_dim, spec.block_size
    nb = W.pool_blocks(spec, ctx)
    bm, model = managers(pkv, nb, B, spec.seed)
    ids = list(range(S))
    for s in ids:
        bm.add_sequence(s, int(ctx[s]) - 1)
        model.add_sequence(s, int(ctx[s]) - 1)
    slots, pairs = bm.append_slots(ids)
    ref = [model.append_slot(s) for s in ids]
    assert slots.tolist() == [r[0] for r in ref] and len(pairs) == 0
    maxb = max(-(-int(c) // B) for c in ctx)
    tables, _ = same_tables(bm, model, ids, maxb)

    kc = W.device_normal((nb, H, B, D), "f16", 5001)
    vc = W.device_normal((nb, H, B, D), "f16", 5002)
    q = W.device_normal((S, H, D), "f16", 5003)
    kn = W.device_normal((S, H, D), "f16", 5004)
    vn = W.device_normal((S, H, D), "f16", 5005)
    kc_h, vc_h = W.torch_to_words(kc), W.torch_to_words(vc)
    q_h, kn_h, vn_h = W.torch_to_words(q), W.torch_to_words(kn), W.torch_to_words(vn)

    pkv.reshape_and_cache(kn, vn, kc, vc, torch.from_numpy(slots).cuda())
    oracle.reshape_and_cache(kn_h, vn_h, kc_h, vc_h, np.array([r[0] for r in ref]))
    assert np.array_equal(W.torch_to_words(kc), kc_h)
    assert np.array_equal(W.torch_to_words(vc), vc_h)

    expect = sampled_oracle(q_h, kc_h, vc_h, tables, ctx, ids, spec.scale, "f16")
    bt, cl = torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda()
    for part in (0, 512):
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, spec.scale, partition_size=part)
        assert pkv.get_device_error() == 0
        attn_check(out, expect, "opt13b partition=%d" % part)


def test_short_batch_block_size_sweep(pkv):
    """256 sequences, lengths U[20,300], bf16, B in {8,16,32,64}: the same
    per-token K/V written through each block size's tables."""
    import torch
    spec = W.SPECS["short"]
    ctx = W.context_lens(spec)
    S, H, D = spec.num_seqs, spec.num_heads, spec.head_dim
    T = int(ctx.sum())
    kt = W.device_normal((T, H, D), "bf16", 6001)        # per-token values, sequence-major
    vt = W.device_normal((T, H, D), "bf16", 6002)
    q = W.device_normal((S, H, D), "bf16", 6003)
    kt_h, vt_h, q_h = W.torch_to_words(kt), W.torch_to_words(vt), W.torch_to_words(q)
    seqs = list(range(S))
    expects = []
    for B in spec.extra["block_sizes"]:
        nb = W.pool_blocks(spec, ctx, B)
        bm, model = managers(pkv, nb, B, spec.seed)
        slots, mslots = [], []
        for s in range(S):
            slots.append(bm.add_sequence(s, int(ctx[s])))
            mslots.extend(model.add_sequence(s, int(ctx[s])))
        slots = np.concatenate(slots)
        assert slots.tolist() == mslots
        maxb = max(-(-int(c) // B) for c in ctx)
        tables, _ = same_tables(bm, model, list(range(S)), maxb)
        kc = torch.zeros((nb, H, B, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        pkv.reshape_and_cache(kt, vt, kc, vc, torch.from_numpy(slots).cuda())
        kc_h = np.zeros((nb, H, B, D), np.uint16)
        vc_h = np.zeros_like(kc_h)
        oracle.reshape_and_cache(kt_h, vt_h, kc_h, vc_h, np.array(mslots))
        assert np.array_equal(W.torch_to_words(kc), kc_h)
        assert np.array_equal(W.torch_to_words(vc), vc_h)
        expect = sampled_oracle(q_h, kc_h, vc_h, tables, ctx, seqs, spec.scale, "bf16")
        expects.append(expect)
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                                   torch.from_numpy(ctx).cuda(), spec.scale)
        assert pkv.get_device_error() == 0
        attn_check(out, expect, "short B=%d" % B)
        del kc, vc
    for e in expects[1:]:                    # the oracle does not depend on the block size
        assert np.array_equal(e, expects[0])


def test_shared_prefix_copy_on_write(pkv):
    """32 prompts x 6 samples, prompt U[128,1024] shared (refcount 6), suffix
    U[1,512] per sample; the partial last prompt block is copied (copy_blocks)
    before the suffix tokens are written (reshape_and_cache)."""
    import torch
    spec = W.SPECS["shared_prefix"]
    p_len, s_len = W.prompt_and_suffix_lens(spec)
    ctx = W.context_lens(spec)
    g = spec.extra["per_group"]
    S, H, D, B = spec.num_seqs, spec.num_heads, spec.head_dim, spec.block_size
    nb = W.pool_blocks(spec, ctx)
    bm, model = managers(pkv, nb, B, spec.seed)
    for gi in range(len(p_len)):
        for m in (bm, model):
            m.add_sequence(gi * g, int(p_len[gi]))
            for c in range(1, g):
                m.fork(gi * g, gi * g + c)
    for gi in range(len(p_len)):
        t = model.block_table(gi * g)
        assert all(model.refcount(b) == g for b in t)
    slots, pairs, tok_seq = [], [], []
    for t in range(int(s_len.max())):
        act = [s for s in range(S) if t < s_len[s]]
        sl, pr = bm.append_slots(act)
        ref = [model.append_slot(s) for s in act]
        assert sl.tolist() == [r[0] for r in ref]
        assert pr.tolist() == [[r[1], r[2]] for r in ref if r[1] >= 0]
        slots.append(sl)
        pairs.append(pr)
        tok_seq.extend(act)
    slots = np.concatenate(slots)
    pairs = np.concatenate(pairs).astype(np.int32).reshape(-1, 2)
    partial = sum(1 for p in p_len if p % B)
    assert len(pairs) == (g - 1) * partial          # the last sharer writes in place
    maxb = max(-(-int(c) // B) for c in ctx)
    tables, _ = same_tables(bm, model, list(range(S)), maxb)

    kc = W.device_normal((nb, H, B, D), "f16", 7001)
    vc = W.device_normal((nb, H, B, D), "f16", 7002)
    T = len(slots)
    kt = W.device_normal((T, H, D), "f16", 7003)
    vt = W.device_normal((T, H, D), "f16", 7004)
    q = W.device_normal((S, H, D), "f16", 7005)
    kc_h, vc_h = W.torch_to_words(kc), W.torch_to_words(vc)
    kt_h, vt_h, q_h = W.torch_to_words(kt), W.torch_to_words(vt), W.torch_to_words(q)

    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    pkv.reshape_and_cache(kt, vt, kc, vc, torch.from_numpy(slots).cuda())
    oracle.copy_blocks(kc_h, vc_h, pairs)
    oracle.reshape_and_cache(kt_h, vt_h, kc_h, vc_h, slots)
    assert np.array_equal(W.torch_to_words(kc), kc_h)
    assert np.array_equal(W.torch_to_words(vc), vc_h)

    expect = sampled_oracle(q_h, kc_h, vc_h, tables, ctx, list(range(S)), spec.scale, "f16")
    bt, cl = torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda()
    for part in (0, 512):
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, spec.scale, partition_size=part)
        assert pkv.get_device_error() == 0
        attn_check(out, expect, "shared prefix partition=%d" % part)
    # the shared-prefix entry point: each group's prompt blocks read once
    for part in (0, 512):
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode_shared(out, q, kc, vc, bt, cl, spec.scale,
                                          partition_size=part)
        assert pkv.get_device_error() == 0
        attn_check(out, expect, "shared prefix, groups read once, partition=%d" % part)


def test_long_context_split_k(pkv):
    """8 sequences, lengths U[8192,32768], 32 heads, fp16, an 80 GB pool left
    uninitialised except the blocks in use; split length 512 and balanced."""
    import torch
    spec = W.SPECS["long"]
    ctx = W.context_lens(spec)
    S, H, D, B = spec.num_seqs, spec.num_heads, spec.head_dim, spec.block_size
    nb = W.pool_blocks(spec, ctx)
    bm, model = managers(pkv, nb, B, spec.seed)
    for s in range(S):
        bm.add_sequence(s, int(ctx[s]))
        model.add_sequence(s, int(ctx[s]))
    maxb = max(-(-int(c) // B) for c in ctx)
    tables, _ = same_tables(bm, model, list(range(S)), maxb)
    kc = torch.empty((nb, H, B, D), dtype=torch.float16, device="cuda")
    vc = torch.empty_like(kc)
    used = np.unique(np.concatenate([tables[s, :-(-int(ctx[s]) // B)] for s in range(S)]))
    ui = torch.from_numpy(used).long().cuda()
    kc.index_copy_(0, ui, W.device_normal((len(used), H, B, D), "f16", 8001))
    vc.index_copy_(0, ui, W.device_normal((len(used), H, B, D), "f16", 8002))
    q = W.device_normal((S, H, D), "f16", 8003)
    seqs = list(range(S))
    uniq = sorted({int(b) for s in seqs for b in tables[s, :-(-int(ctx[s]) // B)]})
    kb, vb = device_blocks_to_host(kc, vc, uniq)
    remap = {b: i for i, b in enumerate(uniq)}
    bt = np.full((len(seqs), maxb), -1, np.int32)
    for i, s in enumerate(seqs):
        n = -(-int(ctx[s]) // B)
        bt[i, :n] = [remap[int(b)] for b in tables[s, :n]]
    expect = oracle.paged_attention_decode_threaded(
        W.torch_to_words(q)[seqs], kb, vb, bt, ctx[seqs], float(np.float32(spec.scale)),
        oracle.F16, threads=host_threads())
    for part in (512, 0):
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, torch.from_numpy(tables).cuda(),
                                   torch.from_numpy(ctx).cuda(), spec.scale, partition_size=part)
        assert pkv.get_device_error() == 0
        attn_check(out, expect, "long partition=%d" % part)
