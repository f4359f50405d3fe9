"""The decode entry point that allocates nothing (GPU).

For callers that cannot allocate device memory -- a serving loop whose memory
is planned once at start-up, or a plugin whose enqueue callback must not
allocate -- pkv_paged_attention_decode_noalloc keeps its scratch in the
library's static per-device array instead of a caller workspace.  Its output
must match the workspace entry point's, call after call, since the array keeps
whatever the previous call left in it: the claim word of the dynamic chunks
included, which a large balanced call uses and the next call must not count.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import math

import numpy as np
import pytest

from helpers import ORC_DTYPE, attn_check, host_threads, random_case, to_dev
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def device_case(case):
    import torch
    dt = case["dtype"]
    return dict(q=to_dev(case["q"], dt), kc=to_dev(case["kc"], dt), vc=to_dev(case["vc"], dt),
                bt=torch.from_numpy(case["bt"]).cuda(), cl=torch.from_numpy(case["ctx"]).cuda())


def oracle_rows(case, scale):
    return oracle.paged_attention_decode_threaded(
        case["q"], case["kc"], case["vc"], case["bt"], case["ctx"], scale,
        ORC_DTYPE[case["dtype"]], threads=host_threads())


def noalloc(P, d, scale, partition):
    import torch
    got = torch.full_like(d["q"], float("nan"))
    P.paged_attention_decode_noalloc(got, d["q"], d["kc"], d["vc"], d["bt"], d["cl"], scale,
                                     partition_size=partition)
    assert P.get_device_error() == 0
    return got


def workspace_call(P, d, scale, partition, ws=None):
    import torch
    want = torch.full_like(d["q"], float("nan"))
    P.paged_attention_decode(want, d["q"], d["kc"], d["vc"], d["bt"], d["cl"], scale,
                             partition_size=partition, workspace=ws)
    assert P.get_device_error() == 0
    return want


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_noalloc_matches_workspace_entry_point_twice(pkv, dtype, D):
    from paged_kv_cache_05_gb300 import pagedkv as P
    rs = np.random.default_rng(4242 + D + (dtype == "bf16"))
    ctx = [1, 15, 16, 37, 0, 300, 1024, 513, 77, 2000]
    case = random_case(rs, len(ctx), 8, D, 16, ctx, dtype)
    d = device_case(case)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle_rows(case, scale)
    for partition in (0, 2048 // D):
        want = workspace_call(P, d, scale, partition).double().cpu().numpy()
        for call in range(2):
            got = noalloc(P, d, scale, partition)
            attn_check(got, want, "%s D=%d partition=%d no-alloc call %d vs workspace entry "
                       "point" % (dtype, D, partition, call))
            attn_check(got, ref, "%s D=%d partition=%d no-alloc call %d vs oracle" % (
                dtype, D, partition, call))


def test_noalloc_large_balanced_then_small_partitioned(pkv):
    """A balanced call large enough (about 57K steps) that its tail is split
    into chunks claimed at run time, three times in a row on the shared array;
    then a small call with a fixed split on the array the large one left
    behind; then the large call again.  Each result against the workspace
    entry point and the fp64 oracle."""
    import torch
    from paged_kv_cache_05_gb300 import pagedkv as P
    rs = np.random.default_rng(4343)
    S, H, D, B = 128, 16, 128, 16
    big = random_case(rs, S, H, D, B, [int(c) for c in rs.integers(1, 900, size=S)], "f16")
    small = random_case(rs, 10, 8, 64, 16, [1, 31, 32, 33, 0, 700, 64, 5, 1999, 129], "bf16")
    db, ds = device_case(big), device_case(small)
    sb = float(np.float32(1 / math.sqrt(D)))
    ss = float(np.float32(1 / math.sqrt(64)))
    ref_b, ref_s = oracle_rows(big, sb), oracle_rows(small, ss)
    # the workspace entry point on the same sizes claims dynamic chunks (the
    # grid, and so the split, is the same for both entry points)
    ws = pkv.alloc_workspace(S, H, D, B, db["bt"].shape[1], 0, db["q"].device)
    want_b = workspace_call(P, db, sb, 0, ws).double().cpu().numpy()
    assert int(ws[16:24].view(torch.int64).cpu()[0]) & 0xFFFFFF > 0
    want_s = workspace_call(P, ds, ss, 32).double().cpu().numpy()
    for what, d, scale, part, want, ref in (
            ("large balanced 1", db, sb, 0, want_b, ref_b),
            ("large balanced 2", db, sb, 0, want_b, ref_b),
            ("large balanced 3", db, sb, 0, want_b, ref_b),
            ("small partitioned", ds, ss, 32, want_s, ref_s),
            ("large balanced again", db, sb, 0, want_b, ref_b)):
        got = noalloc(P, d, scale, part)
        attn_check(got, want, what + " vs workspace entry point")
        attn_check(got, ref, what + " vs oracle")


def test_noalloc_rejects_sizes_beyond_the_static_array(pkv):
    from paged_kv_cache_05_gb300 import pagedkv as P
    L = P.lib()
    need = P.decode_workspace_size(8, 32, 128, 16, 2048, 16)
    assert need > P.NOALLOC_SCRATCH_BYTES
    f = 1 << 20          # never dereferenced: the size check comes first
    st = L.pkv_paged_attention_decode_noalloc(f, f, f, f, f, f, 0.1, 8, 32, 128, 16, 2048,
                                              1 << 20, 0, 16, None)
    assert st == P.PKV_ERR_INVALID
    assert "static array" in P.last_error()


def test_noalloc_empty_batch_checks_arguments_like_the_workspace_entry_point(pkv):
    """With no sequences both entry points still check num_blocks, dtype and
    scale, and answer the same arguments with the same status."""
    from paged_kv_cache_05_gb300 import pagedkv as P
    L = P.lib()
    for nb, dt, scale, want in ((0, 0, 0.1, P.PKV_ERR_INVALID), (16, 7, 0.1, P.PKV_ERR_INVALID),
                                (16, 0, float("inf"), P.PKV_ERR_INVALID),
                                (16, 0, 0.1, P.PKV_OK)):
        a = L.pkv_paged_attention_decode_noalloc(None, None, None, None, None, None, scale, 0, 8,
                                                 128, 16, 4, nb, dt, 0, None)
        b = L.pkv_paged_attention_decode(None, None, None, None, None, None, scale, 0, 8, 128,
                                         16, 4, nb, dt, 0, None, 0, None)
        assert a == b == want, (nb, dt, scale, a, b)
