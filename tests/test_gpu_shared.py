"""GPU parity of the shared-prefix decode entry point: sequences adjacent in
the batch whose block tables begin with the same full blocks are grouped and
their common prefix is read once.  Every row is compared with the fp64
oracle, on batches built by the oracle's block-manager model (prompts forked
into groups, suffixes appended with copy-on-write), with group sizes across
the limit of 8, prefixes at and below the minimum, members whose tokens all
lie in the prefix, sharers that are not adjacent, empty rows, every block
size and head dimension, both storage types and both splits."""
import math

import numpy as np
import pytest

import oracle
from helpers import ORC_DTYPE, attn_check, host_threads, to_dev, words
from oracle.block_manager import BlockManagerModel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def forked_batch(rs, B, layout, spare=16):
    """Tables and context lengths for a batch laid out as `layout`: a list of
    ("group", prompt_len, [suffix lengths]) and ("single", ctx) entries, in
    batch order; a group's members are forks of its first sequence, and their
    suffix tokens are appended round-robin (copy-on-write of a shared partial
    block, as the block manager does).  ("gap", ...) entries put a singleton
    between two sequences that share their prompt's blocks."""
    need = 0
    for e in layout:
        if e[0] == "group":
            need += -(-e[1] // B) + sum(-(-(e[1] % B + s) // B) + 1 for s in e[2])
        else:
            need += -(-e[1] // B) + 1
    m = BlockManagerModel(need + spare, B, int(rs.integers(1 << 30)))
    sid = 0
    appends = []
    order = []
    for e in layout:
        if e[0] == "group":
            lead = sid
            m.add_sequence(lead, e[1])
            order.append(lead)
            for k, suf in enumerate(e[2]):
                if k > 0:
                    m.fork(lead, sid)
                    order.append(sid)
                appends.append((sid, suf))
                sid += 1
            if not e[2]:
                sid += 1
        elif e[0] == "gap":
            # a forked pair with an unrelated sequence between them
            a, b = sid, sid + 2
            m.add_sequence(a, e[1])
            m.add_sequence(sid + 1, e[2])
            m.fork(a, b)
            order += [a, sid + 1, b]
            appends += [(a, 3), (b, 5)]
            sid += 3
        else:
            m.add_sequence(sid, e[1])
            order.append(sid)
            sid += 1
    left = dict(appends)
    while any(v > 0 for v in left.values()):
        for s in sorted(left):
            if left[s] > 0:
                m.append_slot(s)
                left[s] -= 1
    tables = [m.block_table(s) for s in order]
    ctx = np.array([m.context_len(s) for s in order], np.int32)
    mb = max(1, max(len(t) for t in tables))
    bt = np.full((len(order), mb), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    return bt, ctx, m.num_blocks


LAYOUT = [("group", 300, [17, 1, 200, 64, 5, 90]),     # six forks of one prompt
          ("single", 77),
          ("group", 64, [30, 12]),                     # a prefix of exactly 64 tokens
          ("group", 500, [int(x) for x in np.arange(11) * 7 + 1]),   # 11 forks: 8 + 3
          ("group", 40, [9, 3, 20]),                   # below the minimum prefix
          ("single", 0),
          ("group", 128, [0, 33, 0]),                  # members with every token shared
          ("gap", 256, 100),                           # sharers that are not adjacent
          ("group", 1100, [3, 400])]


def run_case(pkv, rs, dtype, D, B, partitions):
    import torch
    bt, ctx, nb = forked_batch(rs, B, LAYOUT)
    S, H = len(ctx), 4
    q_h = words((S, H, D), dtype, rs)
    kc_h = words((nb, H, B, D), dtype, rs)
    vc_h = words((nb, H, B, D), dtype, rs)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.paged_attention_decode_threaded(q_h, kc_h, vc_h, bt, ctx, scale,
                                                 ORC_DTYPE[dtype], threads=host_threads())
    q, kc, vc = to_dev(q_h, dtype), to_dev(kc_h, dtype), to_dev(vc_h, dtype)
    tb, cl = torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda()
    plain = pkv.decode_workspace_size(S, H, D, B, bt.shape[1], 0)
    for part in partitions:
        n = pkv.decode_shared_workspace_size(S, H, D, B, bt.shape[1], part)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode_shared(out, q, kc, vc, tb, cl, scale, partition_size=part,
                                          workspace=ws)
        assert pkv.get_device_error() == 0
        attn_check(out, ref, "shared %s D=%d B=%d partition=%d" % (dtype, D, B, part))
        # the group pass found the groups (units counted in the header that
        # follows the plain layout)
        units = int(ws[plain:plain + 4].view(torch.int32).cpu()[0]) if part == 0 else None
        if part == 0:
            assert units > 0
    zero = [s for s in range(S) if ctx[s] == 0]
    assert zero and (out[zero] == 0).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_shared_prefix_parity(pkv, dtype, D, B):
    rs = np.random.default_rng(3100 + 7 * D + B + (dtype == "bf16"))
    run_case(pkv, rs, dtype, D, B, (0, 2048 // D, 512))


def test_shared_equals_plain_without_sharing(pkv):
    """A batch with no shared blocks: the group pass finds nothing and the
    result is the plain entry point's, bit for bit (same kernels' arithmetic,
    fixed split)."""
    import torch
    from helpers import random_case
    rs = np.random.default_rng(3300)
    ctx = [int(c) for c in rs.integers(0, 600, size=40)]
    case = random_case(rs, len(ctx), 8, 128, 16, ctx, "f16")
    q = to_dev(case["q"], "f16")
    kc, vc = to_dev(case["kc"], "f16"), to_dev(case["vc"], "f16")
    bt, cl = torch.from_numpy(case["bt"]).cuda(), torch.from_numpy(case["ctx"]).cuda()
    a = torch.full_like(q, float("nan"))
    b = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode(a, q, kc, vc, bt, cl, 0.0883883, partition_size=512)
    pkv.paged_attention_decode_shared(b, q, kc, vc, bt, cl, 0.0883883, partition_size=512)
    assert pkv.get_device_error() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_repeated_calls_and_graph_replay(pkv):
    """Repeated calls on one workspace holding garbage beforehand, then CUDA
    graph replays: the group pass rewrites everything the later kernels read."""
    import torch
    rs = np.random.default_rng(3400)
    bt, ctx, nb = forked_batch(rs, 16, LAYOUT * 3)
    S, H, D = len(ctx), 8, 128
    q_h = words((S, H, D), "f16", rs)
    kc_h = words((nb, H, 16, D), "f16", rs)
    vc_h = words((nb, H, 16, D), "f16", rs)
    ref = oracle.paged_attention_decode_threaded(q_h, kc_h, vc_h, bt, ctx, 0.0883883,
                                                 oracle.F16, threads=host_threads())
    q, kc, vc = to_dev(q_h, "f16"), to_dev(kc_h, "f16"), to_dev(vc_h, "f16")
    tb, cl = torch.from_numpy(bt).cuda(), torch.from_numpy(ctx).cuda()
    ws = torch.empty(pkv.decode_shared_workspace_size(S, H, D, 16, bt.shape[1], 0),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    for i in range(3):
        ws.random_(0, 256)
        out.fill_(float("nan"))
        pkv.paged_attention_decode_shared(out, q, kc, vc, tb, cl, 0.0883883, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        attn_check(out, ref, "call %d" % i)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.paged_attention_decode_shared(out, q, kc, vc, tb, cl, 0.0883883, workspace=ws)
    for i in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        attn_check(out, ref, "replay %d" % i)
