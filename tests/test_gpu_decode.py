"""GPU parity of the decode attention against the fp64 oracle on small cases
that span several pipeline steps, chunks and ragged tails, plus the exact
properties the method fixes (context 1 returns V; placement is transparent)."""
import math

import numpy as np
import pytest

import oracle
from helpers import ORC_DTYPE, attn_check, random_case, to_dev
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def run_gpu(pkv, case, scale, partition=0):
    import torch
    dt = case["dtype"]
    q = to_dev(case["q"], dt)
    kc, vc = to_dev(case["kc"], dt), to_dev(case["vc"], dt)
    bt = torch.from_numpy(case["bt"]).cuda()
    cl = torch.from_numpy(case["ctx"]).cuda()
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode(out, q, kc, vc, bt, cl, scale, partition_size=partition)
    assert pkv.get_device_error() == 0
    return out


def run_oracle(case, scale):
    return oracle.paged_attention_decode(case["q"], case["kc"], case["vc"], case["bt"],
                                         case["ctx"], float(np.float32(scale)),
                                         ORC_DTYPE[case["dtype"]])


def step_tokens(D, B):
    return 2048 // D


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_parity_ragged_batch(pkv, dtype, D, B):
    rs = np.random.default_rng(1000 + D + B + (dtype == "bf16"))
    ctx = [1, 2, B - 1, B, B + 1, 0, 3 * B + 5, 257, int(rs.integers(300, 700)), 1000]
    case = random_case(rs, len(ctx), 3, D, B, ctx, dtype)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = run_oracle(case, scale)
    sub = step_tokens(D, B)
    for part in (0, sub, 4 * sub, 512):
        out = run_gpu(pkv, case, scale, part)
        attn_check(out, ref, "dtype=%s D=%d B=%d partition=%d" % (dtype, D, B, part))
        assert (out[5] == 0).all()          # context length 0: zero row


def test_context_one_returns_v_exactly(pkv):
    import torch
    rs = np.random.default_rng(11)
    for dtype in ("f16", "bf16"):
        case = random_case(rs, 7, 4, 128, 16, [1] * 7, dtype)
        out = run_gpu(pkv, case, 0.0883883)
        v = W.words_to_torch(case["vc"], dtype)[torch.from_numpy(case["bt"][:, 0]).long(), :, 0, :]
        assert torch.equal(out.cpu(), v)


def test_placement_is_transparent_bit_exact(pkv):
    """Permuting physical block ids (moving the pool rows with them) changes no bit."""
    import torch
    rs = np.random.default_rng(12)
    ctx = [5, 40, 333, 1024, 17, 600]
    case = random_case(rs, 6, 8, 128, 16, ctx, "f16", spare=30)
    a = run_gpu(pkv, case, 0.088)
    perm = rs.permutation(case["nb"])
    c2 = dict(case)
    c2["kc"], c2["vc"] = np.empty_like(case["kc"]), np.empty_like(case["vc"])
    c2["kc"][perm], c2["vc"][perm] = case["kc"], case["vc"]
    c2["bt"] = np.where(case["bt"] >= 0, perm[np.maximum(case["bt"], 0)], -1).astype(np.int32)
    b = run_gpu(pkv, c2, 0.088)
    assert torch.equal(a, b)


def test_masked_tail_contents_never_matter(pkv):
    """Unwritten slots of the last block (here NaN / Inf bit patterns) leave the
    result unchanged, bit for bit."""
    import torch
    rs = np.random.default_rng(13)
    ctx = [3, 17, 45, 100]
    case = random_case(rs, 4, 4, 128, 16, ctx, "f16")
    a = run_gpu(pkv, case, 0.088)
    c2 = dict(case)
    c2["kc"], c2["vc"] = case["kc"].copy(), case["vc"].copy()
    for s, n in enumerate(ctx):
        last = case["bt"][s, (n - 1) // 16]
        c2["kc"][last, :, n % 16 or 16:, :] = 0x7E00     # fp16 NaN
        c2["vc"][last, :, n % 16 or 16:, :] = 0x7C00     # fp16 +Inf
    b = run_gpu(pkv, c2, 0.088)
    assert torch.equal(a, b)


def test_shared_blocks_give_shared_results(pkv):
    """Sequences reading the same physical blocks with the same query agree exactly
    (garden section 5.1 diagram: tables [7,3,12] and [7,3,9])."""
    import torch
    rs = np.random.default_rng(14)
    case = random_case(rs, 2, 4, 128, 16, [32, 32], "f16", spare=14)
    case["bt"] = np.array([[7, 3, 12], [7, 3, 9]], np.int32)
    case["q"][1] = case["q"][0]
    out = run_gpu(pkv, case, 0.088)
    assert torch.equal(out[0], out[1])
    case["ctx"] = np.array([40, 40], np.int32)
    out = run_gpu(pkv, case, 0.088)
    assert not torch.equal(out[0], out[1])
    attn_check(out, run_oracle(case, 0.088), "diverged")


def test_bad_inputs_are_flagged_not_dereferenced(pkv):
    import torch
    from paged_kv_cache_05_gb300.pagedkv import DEVERR_BAD_BLOCK, DEVERR_BAD_CONTEXT
    rs = np.random.default_rng(15)
    case = random_case(rs, 3, 2, 64, 16, [20, 33, 5], "f16")
    q = to_dev(case["q"], "f16")
    kc, vc = to_dev(case["kc"], "f16"), to_dev(case["vc"], "f16")
    out = torch.empty_like(q)
    bt = case["bt"].copy()
    bt[1, 2] = case["nb"] + 1000
    pkv.paged_attention_decode(out, q, kc, vc, torch.from_numpy(bt).cuda(),
                               torch.from_numpy(case["ctx"]).cuda(), 0.125)
    assert pkv.get_device_error() == DEVERR_BAD_BLOCK
    ctx = case["ctx"].copy()
    ctx[2] = 16 * bt.shape[1] + 1                      # beyond the table
    pkv.paged_attention_decode(out, q, kc, vc, torch.from_numpy(case["bt"]).cuda(),
                               torch.from_numpy(ctx).cuda(), 0.125)
    # clamped to the table's capacity; the -1 entries past the real blocks are flagged too
    assert pkv.get_device_error() & DEVERR_BAD_CONTEXT


def test_tiny_workload_full_step(pkv):
    """The 4-sequence workload through the whole step: block manager (with a
    forked sibling so sequence 3's partial last block is shared) -> copy-on-write
    copy_blocks -> new-token reshape_and_cache -> decode; every stage against the
    oracle (manager model, oracle cache ops, fp64 attention)."""
    import torch
    spec = W.SPECS["tiny"]
    ctx = W.context_lens(spec)
    S, H, D, B, nb = spec.num_seqs, spec.num_heads, spec.head_dim, spec.block_size, 64
    kc = W.normal_words((nb, H, B, D), "f16", spec.seed, 10)
    vc = W.normal_words((nb, H, B, D), "f16", spec.seed, 11)
    knew = W.normal_words((S, H, D), "f16", spec.seed, 12)
    vnew = W.normal_words((S, H, D), "f16", spec.seed, 13)
    q = W.normal_words((S, H, D), "f16", spec.seed, 14)

    bm = pkv.BlockManager(nb, B, spec.seed)
    model = BlockManagerModel(nb, B, spec.seed)
    for s in range(S):
        bm.add_sequence(s, int(ctx[s]) - 1)
        model.add_sequence(s, int(ctx[s]) - 1)
    bm.fork(3, 4)
    model.fork(3, 4)
    slots, pairs = bm.append_slots(list(range(S)))
    ref = [model.append_slot(s) for s in range(S)]
    assert slots.tolist() == [r[0] for r in ref]
    assert pairs.tolist() == [[r[1], r[2]] for r in ref if r[1] >= 0] and len(pairs) == 1
    tables, ctx_now = bm.export(list(range(S)), 4)
    assert ctx_now.tolist() == ctx.tolist()
    for s in range(S):
        t = model.block_table(s)
        assert tables[s, :len(t)].tolist() == t

    dk, dv = to_dev(kc, "f16"), to_dev(vc, "f16")
    pkv.copy_blocks(dk, dv, torch.from_numpy(pairs).cuda())
    pkv.reshape_and_cache(to_dev(knew, "f16"), to_dev(vnew, "f16"), dk, dv,
                          torch.from_numpy(slots).cuda())
    oracle.copy_blocks(kc, vc, pairs)
    oracle.reshape_and_cache(knew, vnew, kc, vc, np.array([r[0] for r in ref]))
    assert np.array_equal(W.torch_to_words(dk), kc) and np.array_equal(W.torch_to_words(dv), vc)

    scale = spec.scale
    bt_model = np.full((S, 4), -1, np.int32)
    for s in range(S):
        t = model.block_table(s)
        bt_model[s, :len(t)] = t
    expect = oracle.paged_attention_decode(q, kc, vc, bt_model, ctx, scale)
    dq = to_dev(q, "f16")
    for part in (0, 32, 64):
        out = torch.empty_like(dq)
        pkv.paged_attention_decode(out, dq, dk, dv, torch.from_numpy(tables).cuda(),
                                   torch.from_numpy(ctx).cuda(), scale, partition_size=part)
        assert pkv.get_device_error() == 0
        attn_check(out, expect, "tiny partition=%d" % part)
        # the 1-token sequence sees only its new token: out == v exactly
        assert torch.equal(out[0].cpu(), W.words_to_torch(vnew[0], "f16"))


def test_alternating_batch_sizes(pkv):
    """Batches of different sizes (so different shared-memory sizes) in any order."""
    rs = np.random.default_rng(16)
    cases = {}
    for S in (3, 700, 40, 3, 700, 1500, 40):
        if S not in cases:
            ctx = list(rs.integers(0, 120, size=S))
            cases[S] = (random_case(rs, S, 2, 128, 16, ctx, "f16"), None)
        case, ref = cases[S]
        if ref is None:
            ref = run_oracle(case, 0.09)
            cases[S] = (case, ref)
        attn_check(run_gpu(pkv, case, 0.09), ref, "S=%d" % S)


def test_dynamic_tail_repeated_calls_and_graph_replay(pkv):
    """A batch large enough (about 57K steps) that the balanced split ends in
    chunks claimed at run time on any grid up to the largest.  Each call is
    checked against the oracle: repeated calls on one workspace that holds
    garbage beforehand (the call stamps its own claim word), then CUDA graph
    replays, where the call's arguments, its epoch included, are frozen."""
    import torch
    rs = np.random.default_rng(17)
    S, H, D, B = 128, 16, 128, 16
    ctx = [int(c) for c in rs.integers(1, 900, size=S)]
    case = random_case(rs, S, H, D, B, ctx, "f16")
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = run_oracle(case, scale)
    q = to_dev(case["q"], "f16")
    kc, vc = to_dev(case["kc"], "f16"), to_dev(case["vc"], "f16")
    bt = torch.from_numpy(case["bt"]).cuda()
    cl = torch.from_numpy(case["ctx"]).cuda()
    ws = pkv.alloc_workspace(S, H, D, B, bt.shape[1], 0, q.device)
    out = torch.empty_like(q)
    for i in range(3):
        ws.random_(0, 256)
        out.fill_(float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, scale, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        attn_check(out, ref, "call %d" % i)
        # header word 2 counts the claims of this call: the tail was dynamic
        claims = int(ws[16:24].view(torch.int64).cpu()[0]) & 0xFFFFFF
        assert claims > 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, scale, workspace=ws)
    for i in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        attn_check(out, ref, "replay %d" % i)


@pytest.mark.parametrize("partition", [0, 512])
def test_large_batch(pkv, partition):
    """4,000 short sequences (about 32 KiB of per-sequence lengths and step
    offsets in each CTA's shared memory, so fewer CTAs fit an SM), ragged
    lengths with empty rows, balanced and fixed splits."""
    rs = np.random.default_rng(1200 + partition)
    S = 4000
    ctx = [int(c) for c in rs.integers(0, 70, size=S)]
    case = random_case(rs, S, 2, 64, 16, ctx, "f16")
    scale = float(np.float32(1 / math.sqrt(64)))
    ref = oracle.paged_attention_decode_threaded(
        case["q"], case["kc"], case["vc"], case["bt"], case["ctx"], scale, ORC_DTYPE["f16"],
        threads=8)
    out = run_gpu(pkv, case, scale, partition)
    attn_check(out, ref, "large batch partition=%d" % partition)
    zero = [s for s in range(S) if ctx[s] == 0]
    assert zero and (out[zero] == 0).all()


def test_batch_size_limit(pkv):
    """The largest batch the ABI takes (16,384 sequences, whose per-sequence
    arrays fill most of a CTA's shared memory, one CTA per SM) matches the
    oracle; one more sequence is refused on the host, nothing launched."""
    import torch
    rs = np.random.default_rng(1300)
    S = 16384
    ctx = [int(c) for c in rs.integers(0, 40, size=S)]
    case = random_case(rs, S, 1, 64, 16, ctx, "f16")
    scale = 0.125
    ref = oracle.paged_attention_decode_threaded(
        case["q"], case["kc"], case["vc"], case["bt"], case["ctx"], scale, ORC_DTYPE["f16"],
        threads=8)
    out = run_gpu(pkv, case, scale)
    attn_check(out, ref, "16384 sequences")
    S1 = S + 1
    q = torch.zeros((S1, 1, 64), dtype=torch.float16, device="cuda")
    kc = torch.zeros((S1, 1, 16, 64), dtype=torch.float16, device="cuda")
    bt = torch.arange(S1, dtype=torch.int32, device="cuda").view(S1, 1)
    cl = torch.ones(S1, dtype=torch.int32, device="cuda")
    o1 = torch.full_like(q, float("nan"))
    with pytest.raises(pkv.PagedKVError) as ei:
        pkv.paged_attention_decode(o1, q, kc, kc, bt, cl, scale)
    assert ei.value.status == 1 and "num_seqs" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.isnan(o1).all() and pkv.get_device_error() == 0


@pytest.mark.parametrize("partition", [0, 512])
def test_pipeline_wait_timeout_is_reported_and_the_next_call_is_correct(pkv, partition):
    """The timeout path of the decode kernels, made to run out on purpose by
    a short wait bound (no wait is broken: with a 0 ns bound a pipeline wait
    gives up once its phase stays incomplete over 32 polls and a tick of the
    global timer, which on a batch of about 57K steps happens in some CTA
    within a few calls; how many depends on timing, so up to 40 are made).
    The call must return, set PKV_DEVERR_TIMEOUT and nothing else; a normal
    call on the same stream right after it must match the oracle."""
    import torch
    from paged_kv_cache_05_gb300 import pagedkv as P
    rs = np.random.default_rng(1400 + partition)
    S, H, D, B = 128, 16, 128, 16
    ctx = [int(c) for c in rs.integers(1, 900, size=S)]
    case = random_case(rs, S, H, D, B, ctx, "f16")
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = run_oracle(case, scale)
    q = to_dev(case["q"], "f16")
    kc, vc = to_dev(case["kc"], "f16"), to_dev(case["vc"], "f16")
    bt = torch.from_numpy(case["bt"]).cuda()
    cl = torch.from_numpy(case["ctx"]).cuda()
    ws = pkv.alloc_workspace(S, H, D, B, bt.shape[1], partition, q.device)
    out = torch.empty_like(q)
    assert pkv.get_device_error() == 0
    prev = P.set_decode_wait_limit(0)
    seen = []
    try:
        for _ in range(40):
            pkv.paged_attention_decode(out, q, kc, vc, bt, cl, scale, partition_size=partition,
                                       workspace=ws)
            torch.cuda.synchronize()
            bits = pkv.get_device_error()
            seen.append(bits)
            assert bits & ~P.DEVERR_TIMEOUT == 0, bits
            if bits:
                break
    finally:
        P.set_decode_wait_limit(prev)
    assert any(b & P.DEVERR_TIMEOUT for b in seen), seen
    for i in range(2):
        out.fill_(float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, scale, partition_size=partition,
                                   workspace=ws)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        attn_check(out, ref, "normal call %d after a timed-out call" % i)
