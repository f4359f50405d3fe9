"""Oracle for the paged KV-cache decode path: plain, slow, obviously correct.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library (``paged_kv_cache_05_gb300``) never imports, links or calls it,
and this package imports nothing from the product.

Contents
  - ``oracle.c`` (built here into ``_liboracle.so`` with plain gcc, no fast-math):
    fp64 decode attention in two forms (contiguous textbook softmax and the
    block-indexed formula of the PagedAttention paper, section 4.1, as printed on
    the zhaifeiyue.github.io detail page), the new-token write and the
    block-granular copy.
  - ``block_manager.py``: the host block manager's policy (free list, reference
    counts, fork, copy-on-write of the last shared block), in plain Python.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against closed forms, library special cases
(numpy's float16, torch's bfloat16 and fp64 scaled-dot-product attention),
brute force and the worked examples the pages print.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lib = None
_lock = threading.Lock()

F16 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into _liboracle.so with gcc (no fast-math: exact fp64)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f64.restype = f64
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = f64
        attn_args = [P, P, P, P, P, P, f64, i32, i32, i32, i32, i32, i64, i32]
        lib.orc_paged_attention_decode.argtypes = attn_args + [i32, i32]
        lib.orc_paged_attention_decode.restype = i32
        lib.orc_paged_attention_decode_blockwise.argtypes = attn_args
        lib.orc_paged_attention_decode_blockwise.restype = i32
        lib.orc_reshape_and_cache.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64]
        lib.orc_reshape_and_cache.restype = i32
        lib.orc_copy_blocks.argtypes = [P, P, P, i32, i32, i32, i32, i64]
        lib.orc_copy_blocks.restype = i32
        lib.orc_swap_blocks.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, i64]
        lib.orc_swap_blocks.restype = i32
        lib.orc_paged_attention_prefill.argtypes = [P, P, P, P, P, P, P, f64, i32, i32, i32, i32,
                                                    i32, i64, i32]
        lib.orc_paged_attention_prefill.restype = i32
        _lib = lib
        return lib


def _words(a: np.ndarray) -> np.ndarray:
    """The raw 16-bit words of a float16/uint16/int16 array, C-contiguous."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16 or a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("expected 16-bit words, got %s" % a.dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f64(words: np.ndarray) -> np.ndarray:
    lib = _load()
    w = _words(words).ravel()
    return np.array([lib.orc_f16_to_f64(int(x)) for x in w], dtype=np.float64)


def bf16_to_f64(words: np.ndarray) -> np.ndarray:
    lib = _load()
    w = _words(words).ravel()
    return np.array([lib.orc_bf16_to_f64(int(x)) for x in w], dtype=np.float64)


def _attn_common(q, k_cache, v_cache, block_tables, context_lens):
    q = _words(q)
    k_cache = _words(k_cache)
    v_cache = _words(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, H, D = q.shape
    nb, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q and the caches")
    if bt.ndim != 2 or bt.shape[0] != S or cl.shape != (S,):
        raise ValueError("block_tables must be [S][max_blocks], context_lens [S]")
    return q, k_cache, v_cache, bt, cl, S, H, D, nb, B


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                           dtype=F16, seqs=None) -> np.ndarray:
    """fp64 decode attention, contiguous textbook form (gather then softmax).

    q: [S][H][D] 16-bit words; k_cache/v_cache: [num_blocks][H][B][D];
    block_tables: int32 [S][max_blocks]; context_lens: int32 [S];
    scale: the softmax scale as the kernel receives it (widen fp32 to fp64
    before passing it here).  ``seqs`` = (begin, end) restricts the computed
    sequences; the other rows of the result stay zero.
    """
    lib = _load()
    q, k_cache, v_cache, bt, cl, S, H, D, nb, B = _attn_common(
        q, k_cache, v_cache, block_tables, context_lens)
    out = np.zeros((S, H, D), dtype=np.float64)
    b, e = (0, S) if seqs is None else seqs
    rc = lib.orc_paged_attention_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(bt), _ptr(cl), float(scale), S, H, D, B,
                                        bt.shape[1], nb, int(dtype), int(b), int(e))
    if rc != 0:
        raise ValueError("oracle: invalid block table or context length (rc=%d)" % rc)
    return out


def paged_attention_decode_threaded(q, k_cache, v_cache, block_tables, context_lens, scale,
                                    dtype=F16, threads=1, seqs=None) -> np.ndarray:
    """The same oracle run over sequence ranges on ``threads`` host threads.

    The C routine releases the GIL (ctypes), so the ranges run concurrently;
    each range is the unchanged single-threaded oracle.
    """
    lib = _load()
    q, k_cache, v_cache, bt, cl, S, H, D, nb, B = _attn_common(
        q, k_cache, v_cache, block_tables, context_lens)
    out = np.zeros((S, H, D), dtype=np.float64)
    b, e = (0, S) if seqs is None else seqs
    todo = list(range(b, e))
    rcs = []

    def worker(idx):
        for s in todo[idx::threads]:
            rcs.append(lib.orc_paged_attention_decode(
                _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl),
                float(scale), S, H, D, B, bt.shape[1], nb, int(dtype), s, s + 1))

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(max(1, threads))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if any(rc != 0 for rc in rcs):
        raise ValueError("oracle: invalid block table or context length")
    return out


def paged_attention_decode_blockwise(q, k_cache, v_cache, block_tables, context_lens, scale,
                                     dtype=F16) -> np.ndarray:
    """fp64 decode attention in the block-indexed form of the paper's section 4.1."""
    lib = _load()
    q, k_cache, v_cache, bt, cl, S, H, D, nb, B = _attn_common(
        q, k_cache, v_cache, block_tables, context_lens)
    out = np.zeros((S, H, D), dtype=np.float64)
    rc = lib.orc_paged_attention_decode_blockwise(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl), float(scale),
        S, H, D, B, bt.shape[1], nb, int(dtype))
    if rc != 0:
        raise ValueError("oracle: invalid block table or context length (rc=%d)" % rc)
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping) -> None:
    """In place: write token t's K/V rows [H][D] into slot_mapping[t] (<0: skip)."""
    lib = _load()
    k, v = _words(k), _words(v)
    for c in (k_cache, v_cache):
        if not (c.flags.c_contiguous and c.dtype in (np.uint16, np.float16, np.int16)):
            raise TypeError("caches must be C-contiguous 16-bit arrays (written in place)")
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, H, D = k.shape
    nb, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or v.shape != k.shape or sm.shape != (T,):
        raise ValueError("shape mismatch")
    rc = lib.orc_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(sm),
                                   T, H, D, B, nb)
    if rc != 0:
        raise ValueError("oracle: slot out of the pool")


def copy_blocks(k_cache, v_cache, pairs) -> None:
    """In place: for each (src, dst) pair copy the whole block, K and V."""
    lib = _load()
    for c in (k_cache, v_cache):
        if not (c.flags.c_contiguous and c.dtype in (np.uint16, np.float16, np.int16)):
            raise TypeError("caches must be C-contiguous 16-bit arrays (written in place)")
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    nb, H, B, D = k_cache.shape
    rc = lib.orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pr), pr.shape[0], H, D, B, nb)
    if rc != 0:
        raise ValueError("oracle: block id out of the pool")


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs) -> None:
    """In place on dst: for each (src, dst) pair copy the whole block, K and V."""
    lib = _load()
    for c in (dst_k, dst_v):
        if not (c.flags.c_contiguous and c.dtype in (np.uint16, np.float16, np.int16)):
            raise TypeError("destination pools must be C-contiguous 16-bit arrays")
    sk, sv = _words(src_k), _words(src_v)
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    snb, H, B, D = sk.shape
    dnb = dst_k.shape[0]
    if tuple(dst_k.shape[1:]) != (H, B, D) or sv.shape != sk.shape or dst_v.shape != dst_k.shape:
        raise ValueError("pool shape mismatch")
    rc = lib.orc_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(sk), _ptr(sv), _ptr(pr), pr.shape[0],
                             H, D, B, snb, dnb)
    if rc != 0:
        raise ValueError("oracle: block id out of a pool")


def paged_attention_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                            dtype=F16) -> np.ndarray:
    """fp64 causal attention of each sequence's new tokens over its paged cache.

    q: [total_query_tokens][H][D]; query_start: int32 [S+1] (row offsets into q);
    the new tokens of sequence s occupy positions ctx-qlen .. ctx-1 and are
    already in the cache.  Returns [total_query_tokens][H][D] fp64.
    """
    lib = _load()
    q = _words(q)
    kc, vc = _words(k_cache), _words(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    T, H, D = q.shape
    nb, H2, B, D2 = kc.shape
    S = cl.shape[0]
    if (H2, D2) != (H, D) or qs.shape != (S + 1,) or qs[-1] != T or bt.shape[0] != S:
        raise ValueError("shape mismatch")
    out = np.zeros((T, H, D), dtype=np.float64)
    rc = lib.orc_paged_attention_prefill(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                         _ptr(cl), _ptr(qs), float(scale), S, H, D, B,
                                         bt.shape[1], nb, int(dtype))
    if rc != 0:
        raise ValueError("oracle: invalid table, context or query lengths (rc=%d)" % rc)
    return out
