"""GPU parity of the one-call decode step (pkv_paged_attention_decode_append):
each sequence's newest token is written into its cache slot and attended.
Checked bit for bit against the two-call path (reshape_and_cache with the
table's slot, then paged_attention_decode) -- output and both pools -- and
against the fp64 oracle (the oracle's new-token write, then its attention)."""
import math

import numpy as np
import pytest

import oracle
from helpers import (ORC_DTYPE, attn_check, host_threads, random_case, to_dev, words)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def newest_slots(bt, ctx, B):
    """Slot of position ctx - 1 through the table (-1 for an empty sequence),
    walking the table as the address translation defines it."""
    out = np.full(len(ctx), -1, np.int64)
    for s, c in enumerate(ctx):
        if c > 0:
            out[s] = int(bt[s, (c - 1) // B]) * B + (c - 1) % B
    return out


def run_both(pkv, case, kn, vn, scale, partition):
    """Two-call path and one-call path on copies of the same pools."""
    import torch
    dt = case["dtype"]
    q = to_dev(case["q"], dt)
    bt = torch.from_numpy(case["bt"]).cuda()
    cl = torch.from_numpy(case["ctx"]).cuda()
    dkn, dvn = to_dev(kn, dt), to_dev(vn, dt)
    kc_a, vc_a = to_dev(case["kc"], dt), to_dev(case["vc"], dt)
    kc_b, vc_b = kc_a.clone(), vc_a.clone()
    slots = torch.from_numpy(newest_slots(case["bt"], case["ctx"], case["B"])).cuda()
    out_a = torch.full_like(q, float("nan"))
    out_b = torch.full_like(q, float("nan"))
    pkv.reshape_and_cache(dkn, dvn, kc_a, vc_a, slots)
    pkv.paged_attention_decode(out_a, q, kc_a, vc_a, bt, cl, scale, partition_size=partition)
    pkv.paged_attention_decode_append(out_b, q, dkn, dvn, kc_b, vc_b, bt, cl, scale,
                                      partition_size=partition)
    assert pkv.get_device_error() == 0
    return out_a, out_b, (kc_a, vc_a), (kc_b, vc_b)


def oracle_after_write(case, kn, vn, scale):
    kc, vc = case["kc"].copy(), case["vc"].copy()
    oracle.reshape_and_cache(kn, vn, kc, vc, newest_slots(case["bt"], case["ctx"], case["B"]))
    ref = oracle.paged_attention_decode_threaded(case["q"], kc, vc, case["bt"], case["ctx"], scale,
                                                 ORC_DTYPE[case["dtype"]], threads=host_threads())
    return ref, kc, vc


def check_case(pkv, rs, ctx, H, D, B, dtype, partition, bitwise=True):
    import torch
    from paged_kv_cache_05_gb300 import workloads as W
    case = random_case(rs, len(ctx), H, D, B, ctx, dtype)
    kn = words((len(ctx), H, D), dtype, rs)
    vn = words((len(ctx), H, D), dtype, rs)
    scale = float(np.float32(1 / math.sqrt(D)))
    out_a, out_b, pa, pb = run_both(pkv, case, kn, vn, scale, partition)
    what = "%s D=%d B=%d partition=%d" % (dtype, D, B, partition)
    if bitwise:
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16)), what + ": output"
    assert torch.equal(pa[0].view(torch.int16), pb[0].view(torch.int16)), what + ": k pool"
    assert torch.equal(pa[1].view(torch.int16), pb[1].view(torch.int16)), what + ": v pool"
    ref, kc, vc = oracle_after_write(case, kn, vn, scale)
    attn_check(out_b, ref, what + " vs oracle")
    attn_check(out_a, ref, what + " two-call path vs oracle")
    assert np.array_equal(W.torch_to_words(pb[0]), kc), what + ": k pool vs oracle"
    assert np.array_equal(W.torch_to_words(pb[1]), vc), what + ": v pool vs oracle"
    return out_b, kn, vn, case


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_append_matches_two_calls(pkv, dtype, D, B):
    """Ragged lengths: empty rows, one token (the new token alone), the newest
    token first / last in its block and in its step, long rows split over
    several pieces; both split modes."""
    rs = np.random.default_rng(900 + D + B + (dtype == "bf16"))
    ctx = [0, 1, 2, B - 1, B, B + 1, 15, 16, 17, 31, 32, 33, 300, 513, 1100, 2047]
    for partition in (0, 4 * (2048 // D)):
        check_case(pkv, rs, ctx, 4, D, B, dtype, partition)


def test_append_single_token_returns_v_new(pkv):
    """Context 1: the only key is the new token, so the output is v_new exactly."""
    import torch
    rs = np.random.default_rng(905)
    out, kn, vn, case = check_case(pkv, rs, [1, 1, 1], 8, 128, 16, "f16", 0)
    from paged_kv_cache_05_gb300 import workloads as W
    assert torch.equal(out.cpu().view(torch.int16),
                       W.words_to_torch(vn, "f16").view(torch.int16))


def test_append_dynamic_chunks(pkv):
    """A batch large enough that the balanced split hands the last quarter of
    its steps out as chunks claimed at run time, so rows end inside claimed
    chunks too.  Which warp of a CTA takes a claimed chunk's steps depends on
    the steps that CTA streamed before, which the claims decide at run time,
    so two calls may sum a row in a different order: the pools must be equal
    bit for bit, the outputs each within the tolerance of the oracle."""
    rs = np.random.default_rng(906)
    ctx = [int(c) for c in rs.integers(1, 900, size=128)]
    for _ in range(2):
        check_case(pkv, rs, ctx, 16, 128, 16, "f16", 0, bitwise=False)


def test_append_full_size_opt13b(pkv):
    """The OPT-13B-shaped decode layer: 64 sequences x 40 heads x 128, fp16,
    B = 16.  With a fixed 512-token split the work of every CTA and warp is
    fixed, so output and pools are bit-identical to the two-call path; with
    the balanced split (chunks claimed at run time) the pools are, and each
    output is within the tolerance of the oracle on every row."""
    import torch
    from paged_kv_cache_05_gb300 import workloads as W
    spec = W.SPECS["opt13b"]
    ctx = W.context_lens(spec)
    rs = np.random.default_rng(907)
    case = random_case(rs, spec.num_seqs, spec.num_heads, spec.head_dim, spec.block_size,
                       [int(c) for c in ctx], "f16")
    kn = words((spec.num_seqs, spec.num_heads, spec.head_dim), "f16", rs)
    vn = words((spec.num_seqs, spec.num_heads, spec.head_dim), "f16", rs)
    ref, _, _ = oracle_after_write(case, kn, vn, spec.scale)
    for partition in (512, 0):
        out_a, out_b, pa, pb = run_both(pkv, case, kn, vn, spec.scale, partition)
        if partition:
            assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
        assert torch.equal(pa[0].view(torch.int16), pb[0].view(torch.int16))
        assert torch.equal(pa[1].view(torch.int16), pb[1].view(torch.int16))
        attn_check(out_b, ref, "opt13b append, partition %d, vs oracle" % partition)
        attn_check(out_a, ref, "opt13b two calls, partition %d, vs oracle" % partition)


def test_append_bad_last_block_is_flagged_and_not_written(pkv):
    """A table entry out of range for the newest token's block: the device
    error word reports a bad block and no slot is written for that sequence
    (the others are)."""
    import torch
    rs = np.random.default_rng(908)
    ctx = [40, 17, 5]
    case = random_case(rs, 3, 4, 128, 16, ctx, "f16")
    bad = case["bt"].copy()
    bad[1, (ctx[1] - 1) // 16] = case["nb"] + 3          # out of the pool
    kn = words((3, 4, 128), "f16", rs)
    vn = words((3, 4, 128), "f16", rs)
    q = to_dev(case["q"], "f16")
    kc, vc = to_dev(case["kc"], "f16"), to_dev(case["vc"], "f16")
    out = torch.empty_like(q)
    pkv.paged_attention_decode_append(out, q, to_dev(kn, "f16"), to_dev(vn, "f16"), kc, vc,
                                      torch.from_numpy(bad).cuda(),
                                      torch.from_numpy(case["ctx"]).cuda(), 0.0883)
    assert pkv.get_device_error() & 1                   # PKV_DEVERR_BAD_BLOCK
    from paged_kv_cache_05_gb300 import workloads as W
    want_k, want_v = case["kc"].copy(), case["vc"].copy()
    good = newest_slots(case["bt"], case["ctx"], 16)
    good[1] = -1
    oracle.reshape_and_cache(kn, vn, want_k, want_v, good)
    assert np.array_equal(W.torch_to_words(kc), want_k)
    assert np.array_equal(W.torch_to_words(vc), want_v)

