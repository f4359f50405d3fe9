"""The C ABI without a GPU: exports, host-side argument checks, the C++ block
manager against the oracle's independent model (bit-exact)."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, OutOfBlocks as ModelOOM

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_05_gb300 import build
    build.build()
    import paged_kv_cache_05_gb300 as m
    return m


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(pkv):
    names = declared_functions()
    assert len(names) >= 19
    L = ctypes.CDLL(pkv.pagedkv.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_workspace_size_checks(pkv):
    assert pkv.decode_workspace_size(64, 40, 128, 16, 128, 0) > 0
    assert pkv.decode_workspace_size(8, 32, 128, 16, 2048, 512) > \
        pkv.decode_workspace_size(8, 32, 128, 16, 2048, 0) // 2
    for bad in [(64, 40, 96, 16, 128, 0),      # head_dim
                (64, 40, 128, 12, 128, 0),     # block_size
                (64, 40, 128, 16, 0, 0),       # max_blocks
                (-1, 40, 128, 16, 8, 0),       # num_seqs
                (64, 40, 128, 16, 8, 24),      # partition not a multiple of the step
                (64, 0, 128, 16, 8, 0)]:       # heads
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.decode_workspace_size(*bad)
        assert e.value.status == 1


def test_decode_rejects_bad_arguments_before_touching_a_gpu(pkv):
    L = pkv.lib()
    ws = ctypes.c_size_t(0)
    assert L.pkv_decode_workspace_size(4, 8, 64, 16, 4, 0, ctypes.byref(ws)) == 0
    fake = 1 << 20   # never dereferenced: validation fails first
    base = [fake, fake, fake, fake, fake, fake, 0.125, 4, 8, 64, 16, 4, 64, 0, 0, fake * 256,
            ws.value, None]

    def call(**kw):
        args = list(base)
        names = ["out", "q", "k", "v", "bt", "cl", "scale", "S", "H", "D", "B", "maxb", "nb",
                 "dtype", "part", "ws", "wsb", "stream"]
        for k, v in kw.items():
            args[names.index(k)] = v
        return L.pkv_paged_attention_decode(*args)

    assert call(D=80) == 1
    assert call(B=4) == 1
    assert call(nb=0) == 1
    assert call(dtype=7) == 1
    assert call(scale=float("nan")) == 1
    assert call(out=0) == 1
    assert call(q=fake + 8) == 1            # misaligned
    assert call(ws=fake * 256 + 64) == 1    # workspace misaligned
    assert call(wsb=ws.value - 1) == 1      # workspace too small
    assert call(part=20) == 1
    assert "workspace" in pkv.pagedkv.last_error() or "partition" in pkv.pagedkv.last_error()
    assert call(S=0) == 0                   # empty batch: nothing to do


def test_decode_append_rejects_bad_arguments_before_touching_a_gpu(pkv):
    """The one-call decode step checks what pkv_paged_attention_decode checks,
    plus its k_new / v_new pointers, and launches nothing when a check fails."""
    L = pkv.lib()
    ws = ctypes.c_size_t(0)
    assert L.pkv_decode_workspace_size(4, 8, 64, 16, 4, 0, ctypes.byref(ws)) == 0
    fake = 1 << 20   # never dereferenced: validation fails first
    names = ["out", "q", "kn", "vn", "k", "v", "bt", "cl", "scale", "S", "H", "D", "B", "maxb",
             "nb", "dtype", "part", "ws", "wsb", "stream"]
    base = [fake, fake, fake, fake, fake, fake, fake, fake, 0.125, 4, 8, 64, 16, 4, 64, 0, 0,
            fake * 256, ws.value, None]

    def call(**kw):
        args = list(base)
        for k, v in kw.items():
            args[names.index(k)] = v
        return L.pkv_paged_attention_decode_append(*args)

    assert call(kn=None) == 1 and "NULL" in pkv.pagedkv.last_error()
    assert call(vn=None) == 1
    assert call(kn=fake + 8) == 1 and "aligned" in pkv.pagedkv.last_error()
    assert call(vn=fake + 4) == 1
    assert call(D=80) == 1
    assert call(B=4) == 1
    assert call(nb=0) == 1
    assert call(dtype=7) == 1
    assert call(scale=float("inf")) == 1
    assert call(out=0) == 1
    assert call(wsb=ws.value - 1) == 1 and "workspace" in pkv.pagedkv.last_error()
    assert call(S=0) == 0                   # empty batch: nothing to do


def test_cache_ops_reject_bad_arguments(pkv):
    L = pkv.lib()
    f = 1 << 20
    assert L.pkv_reshape_and_cache(f, f, f, f, f, 4, 8, 100, 16, 64, 0, None) == 1
    assert L.pkv_reshape_and_cache(f, f, f, f, f, -1, 8, 64, 16, 64, 0, None) == 1
    assert L.pkv_reshape_and_cache(f + 4, f, f, f, f, 4, 8, 64, 16, 64, 0, None) == 1
    assert L.pkv_reshape_and_cache(f, f, f, f, f, 0, 8, 64, 16, 64, 0, None) == 0
    assert L.pkv_copy_blocks(f, f, f, 2, 8, 64, 24, 64, 0, None) == 1
    assert L.pkv_copy_blocks(f, f, f, 70000, 8, 64, 16, 64, 0, None) == 1
    assert L.pkv_copy_blocks(f, f, f, 0, 8, 64, 16, 64, 0, None) == 0


# ---------------------------------------------------------------- block manager
def same_state(bm, model, seq_ids):
    for s in seq_ids:
        assert bm.block_table(s) == model.block_table(s)
        assert bm.context_len(s) == model.context_len(s)
    assert bm.num_free() == model.num_free()
    for b in range(model.num_blocks):
        assert bm.refcount(b) == model.refcount(b)


@pytest.mark.parametrize("seed", [0, 1, 1001, 2**63 + 5])
def test_manager_matches_model_on_random_churn(pkv, seed):
    rs = np.random.default_rng(seed % 1000)
    nb, B = 150, 16
    bm = pkv.BlockManager(nb, B, seed)
    model = BlockManagerModel(nb, B, seed)
    live, nxt = [], 0
    for step in range(1500):
        op = int(rs.integers(0, 10))
        if op < 2 or not live:
            n = int(rs.integers(0, 70))
            try:
                ref = model.add_sequence(nxt, n)
            except ModelOOM:
                with pytest.raises(pkv.OutOfBlocks):
                    bm.add_sequence(nxt, n)
                continue
            assert bm.add_sequence(nxt, n).tolist() == ref
            live.append(nxt)
            nxt += 1
        elif op < 3:
            parent = live[int(rs.integers(len(live)))]
            model.fork(parent, nxt)
            bm.fork(parent, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 4:
            sid = live.pop(int(rs.integers(len(live))))
            model.free_sequence(sid)
            bm.free_sequence(sid)
        else:
            sid = live[int(rs.integers(len(live)))]
            try:
                ref = model.append_slot(sid)
            except ModelOOM:
                with pytest.raises(pkv.OutOfBlocks):
                    bm.append_slot(sid)
                continue
            assert bm.append_slot(sid) == ref
        if step % 50 == 0:
            same_state(bm, model, live)
    same_state(bm, model, live)


@pytest.mark.parametrize("seed", [3, 44])
def test_manager_matches_model_with_swapping(pkv, seed):
    from oracle.block_manager import InvalidRequest

    def both(model_call, cpp_call):
        """Run one operation on both sides; failures must match in kind."""
        try:
            ref = model_call()
        except ModelOOM:
            with pytest.raises(pkv.OutOfBlocks):
                cpp_call()
            return None
        except InvalidRequest:
            with pytest.raises(pkv.PagedKVError) as e:
                cpp_call()
            assert e.value.status == 1
            return None
        return ref, cpp_call()

    rs = np.random.default_rng(seed)
    nb, ncpu, B = 120, 60, 8
    bm = pkv.BlockManager(nb, B, seed)
    model = BlockManagerModel(nb, B, seed)
    bm.add_cpu_pool(ncpu, seed + 1)
    model.add_cpu_pool(ncpu, seed + 1)
    live, nxt = [], 0
    for step in range(1200):
        op = int(rs.integers(0, 12))
        if op < 2 or not live:
            n = int(rs.integers(0, 50))
            r = both(lambda: model.add_sequence(nxt, n), lambda: bm.add_sequence(nxt, n))
            if r:
                assert r[1].tolist() == r[0]
                live.append(nxt)
                nxt += 1
        elif op < 3:
            parent = live[int(rs.integers(len(live)))]
            r = both(lambda: model.fork(parent, nxt), lambda: bm.fork(parent, nxt))
            if r:
                live.append(nxt)
                nxt += 1
        elif op < 4:
            sid = live.pop(int(rs.integers(len(live))))
            model.free_sequence(sid)
            bm.free_sequence(sid)
        elif op < 6:
            k = int(rs.integers(1, min(4, len(live)) + 1))
            group = [live[i] for i in rs.choice(len(live), k, replace=False)]
            if model.swapped[group[0]]:
                r = both(lambda: model.swap_in(group), lambda: bm.swap_in(group))
            else:
                r = both(lambda: model.swap_out(group), lambda: bm.swap_out(group))
            if r:
                assert r[1].tolist() == [list(p) for p in r[0]]
        else:
            sid = live[int(rs.integers(len(live)))]
            r = both(lambda: model.append_slot(sid), lambda: bm.append_slot(sid))
            if r:
                assert r[1] == r[0]
        if step % 40 == 0:
            for s_ in live:
                assert bm.block_table(s_) == model.block_table(s_)
                assert bm.is_swapped(s_) == model.swapped[s_]
            assert bm.num_free() == model.num_free()
            assert bm.num_free_cpu() == len(model.cpu_free)
            for b in range(ncpu):
                assert bm.cpu_refcount(b) == model.cpu_ref[b]


def test_swap_failures_match(pkv):
    bm = pkv.BlockManager(32, 16, 5)
    with pytest.raises(pkv.PagedKVError):
        bm.swap_out([0])                       # no CPU pool yet
    bm.add_cpu_pool(3, 6)
    bm.add_sequence(0, 64)                     # 4 blocks
    bm.add_sequence(1, 10)
    bm.fork(1, 2)
    with pytest.raises(pkv.OutOfBlocks):
        bm.swap_out([0])
    with pytest.raises(pkv.PagedKVError):
        bm.swap_out([1])                       # block shared with 2
    assert not bm.is_swapped(0) and bm.num_free_cpu() == 3
    bm.swap_out([1, 2])
    with pytest.raises(pkv.PagedKVError):
        bm.append_slot(1)
    with pytest.raises(pkv.PagedKVError):
        bm.export([1], 4)


def test_batched_append_matches_sequential_model(pkv):
    B = 16
    bm = pkv.BlockManager(400, B, 77)
    model = BlockManagerModel(400, B, 77)
    for g in range(4):                       # 4 prompts, each forked into 6 samples
        p = 100 + 37 * g
        bm.add_sequence(g * 10, p)
        model.add_sequence(g * 10, p)
        for c in range(1, 6):
            bm.fork(g * 10, g * 10 + c)
            model.fork(g * 10, g * 10 + c)
    ids = [g * 10 + c for g in range(4) for c in range(6)]
    for _ in range(40):
        slots, pairs = bm.append_slots(ids)
        ref = [model.append_slot(s) for s in ids]
        assert slots.tolist() == [r[0] for r in ref]
        assert pairs.tolist() == [[r[1], r[2]] for r in ref if r[1] >= 0]
    same_state(bm, model, ids)
    tables, ctx = bm.export(ids, 64)
    for i, s in enumerate(ids):
        t = model.block_table(s)
        assert tables[i, :len(t)].tolist() == t and (tables[i, len(t):] == -1).all()
        assert ctx[i] == model.context_len(s)


def test_batched_append_is_all_or_nothing(pkv):
    bm = pkv.BlockManager(6, 4, 3)
    bm.add_sequence(1, 4)
    bm.add_sequence(2, 4)
    bm.add_sequence(3, 13)                   # 4 blocks: 6 used, none free
    before = (bm.block_table(1), bm.block_table(2), bm.num_free())
    with pytest.raises(pkv.OutOfBlocks):
        bm.append_slots([1, 2])
    assert (bm.block_table(1), bm.block_table(2), bm.num_free()) == before
    with pytest.raises(pkv.PagedKVError):
        bm.append_slots([1, 1])              # repeated sequence
    with pytest.raises(pkv.PagedKVError):
        bm.append_slots([9])                 # unknown sequence
    assert bm.context_len(1) == 4


def test_swap_refuses_pageable_host_memory(pkv):
    """Pools the kernel could not dereference are refused before any launch."""
    L = pkv.lib()
    pool = np.zeros((4, 2, 16, 64), np.float16)            # ordinary (pageable) host memory
    pairs = np.array([[0, 1]], np.int32)
    p = pool.ctypes.data
    st = L.pkv_swap_blocks(p, p, p, p, pairs.ctypes.data, 1, 2, 64, 16, 4, 4, 0, None)
    assert st == 1 and "pinned" in pkv.pagedkv.last_error()
    assert L.pkv_swap_blocks(p, p, p, p, pairs.ctypes.data, 0, 2, 64, 16, 4, 4, 0, None) == 0


def test_documented_status_and_error_codes(pkv):
    """The status codes and device error bits the header documents, and the
    binding's copies of them, are the same numbers."""
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    enum = dict((n, int(v)) for n, v in re.findall(r"\b(PKV_(?:OK|ERR_\w+))\s*=\s*(\d+)", text))
    assert enum == {"PKV_OK": 0, "PKV_ERR_INVALID": 1, "PKV_ERR_CUDA": 2, "PKV_ERR_OOM": 3,
                    "PKV_ERR_DEVICE": 4}
    bits = dict((n, int(v)) for n, v in re.findall(r"#define\s+(PKV_DEVERR_\w+)\s+(\d+)", text))
    assert bits == {"PKV_DEVERR_BAD_BLOCK": 1, "PKV_DEVERR_BAD_SLOT": 2,
                    "PKV_DEVERR_BAD_CONTEXT": 4, "PKV_DEVERR_TIMEOUT": 8,
                    "PKV_DEVERR_WORKSPACE": 16}
    P = pkv.pagedkv
    assert (P.PKV_OK, P.PKV_ERR_INVALID, P.PKV_ERR_CUDA, P.PKV_ERR_OOM, P.PKV_ERR_DEVICE) == \
        (0, 1, 2, 3, 4)
    assert (P.DEVERR_BAD_BLOCK, P.DEVERR_BAD_SLOT, P.DEVERR_BAD_CONTEXT, P.DEVERR_TIMEOUT,
            P.DEVERR_WORKSPACE) == (1, 2, 4, 8, 16)
    # one status per outcome: a bad argument is INVALID and names the argument
    L = pkv.lib()
    out = ctypes.c_size_t(0)
    assert L.pkv_decode_workspace_size(4, 8, 96, 16, 4, 0, ctypes.byref(out)) == 1
    assert "head_dim" in P.last_error()
    assert L.pkv_decode_workspace_size(4, 8, 64, 16, 4, 0, None) == 1
    bm = P.BlockManager(4, 16, 1)
    bm.add_sequence(0, 64)
    with pytest.raises(P.OutOfBlocks) as e:
        bm.add_sequence(1, 1)
    assert e.value.status == 3


def test_decode_wait_limit_setter(pkv):
    """The bound of the decode kernels' pipeline waits: default 1 s, settable
    up to 10 s, returns the bound it replaces, a larger value is refused and
    leaves the bound unchanged."""
    P = pkv.pagedkv
    first = P.set_decode_wait_limit(5_000)
    try:
        assert first == 1_000_000_000
        assert P.set_decode_wait_limit(0) == 5_000
        with pytest.raises(P.PagedKVError) as e:
            P.set_decode_wait_limit(10_000_000_001)
        assert e.value.status == 1
        assert P.set_decode_wait_limit(10_000_000_000) == 0
    finally:
        P.set_decode_wait_limit(first)
    assert P.set_decode_wait_limit(first) == first


def test_prefill_rejects_bad_arguments_before_touching_a_gpu(pkv):
    """The prompt-phase calls check their sizes on the host and launch nothing
    when a check fails, including sizes whose work-schedule cost sums could
    overflow 64 bits."""
    L = pkv.lib()
    fake = 1 << 20   # never dereferenced: validation fails first
    names = ["out", "q", "k", "v", "bt", "cl", "qs", "scale", "S", "H", "D", "B", "maxb", "nb",
             "maxq", "T", "dtype", "stream"]
    base = [fake, fake, fake, fake, fake, fake, fake, 0.125, 4, 8, 128, 16, 8, 64, 100, 400, 0,
            None]

    def call(**kw):
        args = list(base)
        for k, v in kw.items():
            args[names.index(k)] = v
        return L.pkv_paged_attention_prefill(*args)

    assert call(D=96) == 1
    assert call(B=4) == 1
    assert call(maxq=-1) == 1
    assert call(dtype=3) == 1
    assert call(scale=float("nan")) == 1
    assert call(maxb=1 << 28) == 1 and "overflows" in pkv.pagedkv.last_error()
    assert call(nb=1 << 20, H=4096) == 1 and "32-bit" in pkv.pagedkv.last_error()
    # about 10^24 estimated cost: refused before anything is looked up on a device
    assert call(S=65535, H=65535, maxb=1 << 26, nb=1, maxq=1 << 30, T=1 << 30) == 1
    assert "too much work" in pkv.pagedkv.last_error()
    assert call(q=None) == 1 and "NULL" in pkv.pagedkv.last_error()
    assert call(S=0) == 0                   # empty batch: nothing to do
