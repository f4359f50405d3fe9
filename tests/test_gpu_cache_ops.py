"""GPU parity of the cache kernels against the oracle: bit-exact pools."""
import numpy as np
import pytest

import oracle
from helpers import to_dev, words
from paged_kv_cache_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,B", [(64, 16), (128, 8), (128, 16), (128, 64), (64, 32)])
def test_reshape_and_cache_bit_exact(pkv, dtype, D, B):
    import torch
    rs = np.random.default_rng(D * 100 + B + (dtype == "bf16"))
    H, nb = 5, 37
    T = min(300, nb * B)
    kc, vc = words((nb, H, B, D), dtype, rs), words((nb, H, B, D), dtype, rs)
    k, v = words((T, H, D), dtype, rs), words((T, H, D), dtype, rs)
    slots = rs.permutation(nb * B)[:T].astype(np.int64)
    slots[rs.random(T) < 0.1] = -1                       # "do not write" entries
    dk, dv = to_dev(kc, dtype), to_dev(vc, dtype)
    pkv.reshape_and_cache(to_dev(k, dtype), to_dev(v, dtype), dk, dv,
                          torch.from_numpy(slots).cuda())
    assert pkv.get_device_error() == 0
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    assert np.array_equal(W.torch_to_words(dk), kc)
    assert np.array_equal(W.torch_to_words(dv), vc)


@pytest.mark.parametrize("D,T", [(64, 20011), (128, 10007)])
def test_reshape_and_cache_many_rows(pkv, D, T):
    """Enough (token, head) rows that every CTA of the one-wave grid strides
    over them several times, the last pass partial."""
    import torch
    rs = np.random.default_rng(D + T)
    H, B = 8, 16
    nb = -(-T // B) + 3
    kc, vc = words((nb, H, B, D), "f16", rs), words((nb, H, B, D), "f16", rs)
    k, v = words((T, H, D), "f16", rs), words((T, H, D), "f16", rs)
    slots = rs.permutation(nb * B)[:T].astype(np.int64)
    slots[rs.random(T) < 0.05] = -1
    dk, dv = to_dev(kc, "f16"), to_dev(vc, "f16")
    pkv.reshape_and_cache(to_dev(k, "f16"), to_dev(v, "f16"), dk, dv,
                          torch.from_numpy(slots).cuda())
    assert pkv.get_device_error() == 0
    oracle.reshape_and_cache(k, v, kc, vc, slots)
    assert np.array_equal(W.torch_to_words(dk), kc)
    assert np.array_equal(W.torch_to_words(dv), vc)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("H,D,B", [(8, 64, 16), (40, 128, 16), (3, 128, 64), (2, 64, 8)])
def test_copy_blocks_bit_exact(pkv, dtype, H, D, B):
    import torch
    rs = np.random.default_rng(H * D + B)
    nb = 60
    kc, vc = words((nb, H, B, D), dtype, rs), words((nb, H, B, D), dtype, rs)
    perm = rs.permutation(nb)
    P = 17
    pairs = np.stack([perm[:P], perm[P:2 * P]], axis=1).astype(np.int32)   # dsts disjoint from srcs
    dk, dv = to_dev(kc, dtype), to_dev(vc, dtype)
    pkv.copy_blocks(dk, dv, torch.from_numpy(pairs).cuda())
    assert pkv.get_device_error() == 0
    oracle.copy_blocks(kc, vc, pairs)
    assert np.array_equal(W.torch_to_words(dk), kc)
    assert np.array_equal(W.torch_to_words(dv), vc)


def test_empty_calls_launch_nothing(pkv):
    import torch
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device="cuda")
    pkv.copy_blocks(kc, kc.clone(), torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    pkv.reshape_and_cache(torch.zeros((0, 2, 64), dtype=torch.float16, device="cuda"),
                          torch.zeros((0, 2, 64), dtype=torch.float16, device="cuda"),
                          kc, kc.clone(), torch.zeros(0, dtype=torch.int64, device="cuda"))
    assert pkv.get_device_error() == 0


def test_out_of_pool_ids_are_skipped_and_flagged(pkv):
    """Kernels validate ids before use: a bad slot or pair is skipped and flagged."""
    import torch
    from paged_kv_cache_05_gb300.pagedkv import DEVERR_BAD_BLOCK, DEVERR_BAD_SLOT
    rs = np.random.default_rng(5)
    nb, H, B, D = 8, 2, 16, 64
    kc = words((nb, H, B, D), "f16", rs)
    dk, dv = to_dev(kc, "f16"), to_dev(kc, "f16")
    k = to_dev(words((2, H, D), "f16", rs), "f16")
    slots = torch.tensor([nb * B, 3], dtype=torch.int64, device="cuda")   # first is past the pool
    pkv.reshape_and_cache(k, k, dk, dv, slots)
    assert pkv.get_device_error() == DEVERR_BAD_SLOT
    assert pkv.get_device_error() == 0                                   # cleared
    expect = kc.copy()
    expect[0, :, 3, :] = W.torch_to_words(k)[1]
    assert np.array_equal(W.torch_to_words(dk), expect)
    pairs = torch.tensor([[1, nb], [-1, 2]], dtype=torch.int32, device="cuda")
    pkv.copy_blocks(dk, dv, pairs)
    assert pkv.get_device_error() == DEVERR_BAD_BLOCK
    assert np.array_equal(W.torch_to_words(dk), expect)
