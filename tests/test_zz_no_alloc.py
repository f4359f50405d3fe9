"""The decode entry point that allocates nothing (GPU).

For callers that cannot allocate device memory -- a serving loop whose memory
is planned once at start-up, or a plugin whose enqueue callback must not
allocate -- pkv_paged_attention_decode_noalloc keeps its scratch in the
library's static per-device array instead of a caller workspace.  Its output
must match the workspace entry point's, call after call, since the array keeps
whatever the previous call left in it.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import ctypes
import math

import numpy as np
import pytest

from helpers import attn_check, random_case, to_dev
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


@pytest.mark.parametrize("partition", [0, 16])
def test_noalloc_matches_workspace_entry_point_twice(pkv, partition):
    import torch
    from paged_kv_cache_05_gb300 import pagedkv as P
    rs = np.random.default_rng(4242 + partition)
    ctx = [1, 15, 16, 37, 0, 300, 1024, 513, 77, 2000]
    case = random_case(rs, len(ctx), 8, 128, 16, ctx, "f16")
    q = to_dev(case["q"], "f16")
    kc, vc = to_dev(case["kc"], "f16"), to_dev(case["vc"], "f16")
    bt = torch.from_numpy(case["bt"]).cuda()
    cl = torch.from_numpy(case["ctx"]).cuda()
    scale = float(np.float32(1 / math.sqrt(128)))
    want = torch.empty_like(q)
    P.paged_attention_decode(want, q, kc, vc, bt, cl, scale, partition_size=partition)
    want_np = want.double().cpu().numpy()
    for call in range(2):
        got = torch.full_like(q, float("nan"))
        P.paged_attention_decode_noalloc(got, q, kc, vc, bt, cl, scale, partition_size=partition)
        assert P.get_device_error() == 0
        attn_check(got, want_np, "no-alloc call %d vs workspace entry point" % call)
    # and both against the fp64 oracle
    ref = oracle.paged_attention_decode(case["q"], case["kc"], case["vc"], case["bt"],
                                        case["ctx"], scale, oracle.F16)
    attn_check(got, ref, "no-alloc vs oracle")


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
