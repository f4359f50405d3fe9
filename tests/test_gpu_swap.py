"""GPU parity of the block swap (wywy.jp notes, "Swapping"): a forked group of
sequences is swapped out to a pinned CPU pool and back into fresh GPU blocks
with pkv_swap_blocks; pools are compared bit for bit with the oracle's copies
and the decode output is unchanged, bit for bit."""
import numpy as np
import pytest

import oracle
from helpers import attn_check, sampled_oracle
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


@pytest.mark.parametrize("B", [8, 16, 64])
def test_swap_out_and_in_round_trip(pkv, B):
    import torch
    H, D, nb, ncpu = 8, 128, 200, 120
    bm, model = pkv.BlockManager(nb, B, 21), BlockManagerModel(nb, B, 21)
    for m in (bm, model):
        m.add_cpu_pool(ncpu, 22)
        m.add_sequence(0, 150)
        m.fork(0, 1)
        m.fork(0, 2)
        m.add_sequence(3, 77)
    slots, cow = bm.append_slots([0, 1, 2, 3])
    ref = [model.append_slot(s) for s in (0, 1, 2, 3)]
    assert slots.tolist() == [r[0] for r in ref]
    ids = [0, 1, 2, 3]
    maxb = max(len(bm.block_table(s)) for s in ids)
    kc = W.device_normal((nb, H, B, D), "f16", 9001)
    vc = W.device_normal((nb, H, B, D), "f16", 9002)
    q = W.device_normal((4, H, D), "f16", 9003)
    pkv.copy_blocks(kc, vc, torch.from_numpy(cow).cuda())
    tables, ctx = bm.export(ids, maxb)
    out_before = torch.empty_like(q)
    pkv.paged_attention_decode(out_before, q, kc, vc, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(ctx).cuda(), 0.088)
    kc_h, vc_h = W.torch_to_words(kc), W.torch_to_words(vc)

    # swap the forked group out to pinned host memory
    pairs = bm.swap_out([0, 1, 2])
    assert pairs.tolist() == [list(p) for p in model.swap_out([0, 1, 2])]
    ck = torch.zeros((ncpu, H, B, D), dtype=torch.float16).pin_memory()
    cv = torch.zeros_like(ck).pin_memory()
    pkv.swap_blocks(ck, cv, kc, vc, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ck_h, cv_h = np.zeros((ncpu, H, B, D), np.uint16), np.zeros((ncpu, H, B, D), np.uint16)
    oracle.swap_blocks(ck_h, cv_h, kc_h, vc_h, pairs)
    assert np.array_equal(W.torch_to_words(ck), ck_h)
    assert np.array_equal(W.torch_to_words(cv), cv_h)

    # the freed GPU blocks get reused: scribble over all of them
    freed = torch.from_numpy(pairs[:, 0].astype(np.int64)).cuda()
    kc.index_fill_(0, freed, float("nan"))
    vc.index_fill_(0, freed, float("nan"))
    kc_h, vc_h = W.torch_to_words(kc), W.torch_to_words(vc)

    # and back into fresh GPU blocks
    back = bm.swap_in([0, 1, 2])
    assert back.tolist() == [list(p) for p in model.swap_in([0, 1, 2])]
    pkv.swap_blocks(kc, vc, ck, cv, torch.from_numpy(back).cuda())
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    oracle.swap_blocks(kc_h, vc_h, ck_h, cv_h, back)
    assert np.array_equal(W.torch_to_words(kc), kc_h)
    assert np.array_equal(W.torch_to_words(vc), vc_h)

    tables2, ctx2 = bm.export(ids, maxb)
    assert np.array_equal(ctx2, ctx)
    out_after = torch.empty_like(q)
    pkv.paged_attention_decode(out_after, q, kc, vc, torch.from_numpy(tables2).cuda(),
                               torch.from_numpy(ctx2).cuda(), 0.088)
    assert torch.equal(out_before, out_after)          # placement changed, no bit did
    expect = sampled_oracle(W.torch_to_words(q), kc_h, vc_h, tables2, ctx2, ids, 0.088, "f16")
    attn_check(out_after, expect, "after swap-in B=%d" % B)
