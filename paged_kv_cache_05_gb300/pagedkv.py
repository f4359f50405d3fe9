"""Thin ctypes binding of libpagedkv.so (include/pagedkv.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and a non-OK status becomes an exception.
Every step of the computation runs in the library's CUDA kernels (or, for the
block manager, its C++ code).  There is no fallback: if the library is not
built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PKV_OK, PKV_ERR_INVALID, PKV_ERR_CUDA, PKV_ERR_OOM, PKV_ERR_DEVICE = range(5)
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID", 2: "PKV_ERR_CUDA", 3: "PKV_ERR_OOM",
                4: "PKV_ERR_DEVICE"}
PKV_F16, PKV_BF16 = 0, 1
DEVERR_BAD_BLOCK, DEVERR_BAD_SLOT, DEVERR_BAD_CONTEXT, DEVERR_TIMEOUT, DEVERR_WORKSPACE = (
    1, 2, 4, 8, 16)
MAX_GRID = 4096
MAX_SEQS = 16384

_lib = None
_lock = threading.Lock()


class PagedKVError(RuntimeError):
    def __init__(self, fn, status, message):
        super().__init__("%s: %s: %s" % (fn, STATUS_NAMES.get(status, status), message))
        self.status = status


class OutOfBlocks(PagedKVError):
    pass


def lib():
    """Load libpagedkv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libpagedkv.so is not built (%s); run "
                               "`python -m paged_kv_cache_05_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, u64, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                                 ctypes.c_float)
        sz = ctypes.c_size_t
        sig = {
            "pkv_decode_workspace_size": ([i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)], i32),
            "pkv_paged_attention_decode": ([P, P, P, P, P, P, f32, i32, i32, i32, i32, i32, i64,
                                            i32, i32, P, sz, P], i32),
            "pkv_paged_attention_decode_append": ([P, P, P, P, P, P, P, P, f32, i32, i32, i32,
                                                   i32, i32, i64, i32, i32, P, sz, P], i32),
            "pkv_decode_shared_workspace_size": ([i32, i32, i32, i32, i32, i32,
                                                  ctypes.POINTER(sz)], i32),
            "pkv_paged_attention_decode_shared": ([P, P, P, P, P, P, f32, i32, i32, i32, i32,
                                                   i32, i64, i32, i32, P, sz, P], i32),
            "pkv_contiguous_workspace_size": ([i32, i32, i32, i32, i32, ctypes.POINTER(sz)],
                                              i32),
            "pkv_contiguous_attention_decode": ([P, P, P, P, P, f32, i32, i32, i32, i32, i32,
                                                 i32, P, sz, P], i32),
            "pkv_paged_attention_decode_noalloc": ([P, P, P, P, P, P, f32, i32, i32, i32, i32,
                                                    i32, i64, i32, i32, P], i32),
            "pkv_paged_attention_prefill": ([P, P, P, P, P, P, P, f32, i32, i32, i32, i32,
                                             i32, i64, i32, i32, i32, P], i32),
            "pkv_paged_attention_prefill_write": ([P, P, P, P, P, P, P, P, P, f32, i32, i32, i32,
                                                   i32, i32, i64, i32, i32, i32, P], i32),
            "pkv_reshape_and_cache": ([P, P, P, P, P, i32, i32, i32, i32, i64, i32, P], i32),
            "pkv_copy_blocks": ([P, P, P, i32, i32, i32, i32, i64, i32, P], i32),
            "pkv_swap_blocks": ([P, P, P, P, P, i32, i32, i32, i32, i64, i64, i32, P], i32),
            "pkv_get_device_error": ([ctypes.POINTER(ctypes.c_int32), i32, P], i32),
            "pkv_set_decode_wait_limit": ([u64, ctypes.POINTER(u64)], i32),
            "pkv_last_error": ([], ctypes.c_char_p),
            "pkv_version": ([], ctypes.c_char_p),
            "pkv_bm_create": ([i64, i32, u64, ctypes.POINTER(P)], i32),
            "pkv_bm_destroy": ([P], None),
            "pkv_bm_add_sequence": ([P, i64, ctypes.c_int32, P], i32),
            "pkv_bm_fork": ([P, i64, i64], i32),
            "pkv_bm_append_slot": ([P, i64, ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_int32)], i32),
            "pkv_bm_append_slots": ([P, P, i32, P, P, ctypes.POINTER(ctypes.c_int32)], i32),
            "pkv_bm_free_sequence": ([P, i64], i32),
            "pkv_bm_block_table": ([P, i64, P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
                                   i32),
            "pkv_bm_context_len": ([P, i64, ctypes.POINTER(ctypes.c_int32)], i32),
            "pkv_bm_export": ([P, P, i32, P, ctypes.c_int32, P], i32),
            "pkv_bm_refcount": ([P, ctypes.c_int32], ctypes.c_int32),
            "pkv_bm_num_free": ([P], i64),
            "pkv_bm_add_cpu_pool": ([P, i64, u64], i32),
            "pkv_bm_swap_out": ([P, P, i32, P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
                                i32),
            "pkv_bm_swap_in": ([P, P, i32, P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
                               i32),
            "pkv_bm_is_swapped": ([P, i64], ctypes.c_int32),
            "pkv_bm_cpu_refcount": ([P, ctypes.c_int32], ctypes.c_int32),
            "pkv_bm_num_free_cpu": ([P], i64),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def last_error() -> str:
    return lib().pkv_last_error().decode()


def version() -> str:
    return lib().pkv_version().decode()


def _check(fn: str, status: int):
    if status != PKV_OK:
        cls = OutOfBlocks if status == PKV_ERR_OOM else PagedKVError
        raise cls(fn, status, last_error())


# ----------------------------------------------------------------- torch side
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t == torch.float16:
        return PKV_F16
    if t == torch.bfloat16:
        return PKV_BF16
    raise TypeError("fp16 or bf16 storage expected, got %s" % t)


def _stream(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t, name, dtype=None, ndim=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dimensions" % (name, ndim))
    return t.data_ptr()


def decode_workspace_size(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                          partition_size=0) -> int:
    out = ctypes.c_size_t(0)
    _check("pkv_decode_workspace_size",
           lib().pkv_decode_workspace_size(num_seqs, num_heads, head_dim, block_size,
                                           max_blocks_per_seq, partition_size,
                                           ctypes.byref(out)))
    return out.value


def alloc_workspace(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                    partition_size=0, device="cuda"):
    """A device buffer (torch uint8, 256-B aligned by torch's allocator) of the needed size."""
    torch = _torch()
    n = decode_workspace_size(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                              partition_size)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           partition_size=0, workspace=None, stream=None):
    """out[s,h] = softmax(scale q[s,h] . K_s) V_s over the sequence's paged K/V."""
    torch = _torch()
    S, H, D = q.shape
    nb, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shape mismatch")
    if tuple(out.shape) != (S, H, D) or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("out/q/cache dtype or shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    if workspace is None:
        workspace = alloc_workspace(S, H, D, B, block_tables.shape[1], partition_size,
                                    q.device)
    ptrs = [_dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32),
            _dev(context_lens, "context_lens", torch.int32, 1)]
    wsp = _dev(workspace, "workspace")
    _check("pkv_paged_attention_decode",
           lib().pkv_paged_attention_decode(*ptrs, float(scale), S, H, D, B,
                                            block_tables.shape[1], nb, _dtype_code(q.dtype),
                                            int(partition_size), wsp,
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream)))
    return out


def paged_attention_decode_append(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                  context_lens, scale, partition_size=0, workspace=None,
                                  stream=None):
    """One decode step: each sequence's newest token (position ctx - 1) is
    written into its cache slot from k_new / v_new [S, H, D] and attended
    (reshape_and_cache with the table's slot, then paged_attention_decode)."""
    torch = _torch()
    S, H, D = q.shape
    nb, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shape mismatch")
    if tuple(out.shape) != (S, H, D) or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("out/q/cache dtype or shape mismatch")
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        if tuple(t.shape) != (S, H, D) or t.dtype != q.dtype:
            raise ValueError("%s must be [num_seqs, num_heads, head_dim] of q's dtype" % n)
    if block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    if workspace is None:
        workspace = alloc_workspace(S, H, D, B, block_tables.shape[1], partition_size,
                                    q.device)
    ptrs = [_dev(out, "out"), _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32),
            _dev(context_lens, "context_lens", torch.int32, 1)]
    wsp = _dev(workspace, "workspace")
    _check("pkv_paged_attention_decode_append",
           lib().pkv_paged_attention_decode_append(*ptrs, float(scale), S, H, D, B,
                                                   block_tables.shape[1], nb,
                                                   _dtype_code(q.dtype), int(partition_size), wsp,
                                                   workspace.numel() * workspace.element_size(),
                                                   _stream(stream)))
    return out


def decode_shared_workspace_size(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                 partition_size=0) -> int:
    out = ctypes.c_size_t(0)
    _check("pkv_decode_shared_workspace_size",
           lib().pkv_decode_shared_workspace_size(num_seqs, num_heads, head_dim, block_size,
                                                  max_blocks_per_seq, partition_size,
                                                  ctypes.byref(out)))
    return out.value


def paged_attention_decode_shared(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                  partition_size=0, workspace=None, stream=None):
    """paged_attention_decode for batches whose adjacent sequences share prefix
    blocks: each group's common prefix is read once for all its members."""
    torch = _torch()
    S, H, D = q.shape
    nb, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shape mismatch")
    if tuple(out.shape) != (S, H, D) or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("out/q/cache dtype or shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    if workspace is None:
        n = decode_shared_workspace_size(S, H, D, B, block_tables.shape[1], partition_size)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    ptrs = [_dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32),
            _dev(context_lens, "context_lens", torch.int32, 1)]
    _check("pkv_paged_attention_decode_shared",
           lib().pkv_paged_attention_decode_shared(*ptrs, float(scale), S, H, D, B,
                                                   block_tables.shape[1], nb,
                                                   _dtype_code(q.dtype), int(partition_size),
                                                   _dev(workspace, "workspace"),
                                                   workspace.numel() * workspace.element_size(),
                                                   _stream(stream)))
    return out


def contiguous_workspace_size(num_seqs, num_heads, head_dim, max_context_len,
                              partition_size=0) -> int:
    out = ctypes.c_size_t(0)
    _check("pkv_contiguous_workspace_size",
           lib().pkv_contiguous_workspace_size(num_seqs, num_heads, head_dim, max_context_len,
                                               partition_size, ctypes.byref(out)))
    return out.value


def contiguous_attention_decode(out, q, k, v, context_lens, scale, partition_size=0,
                                workspace=None, stream=None):
    """The decode attention over a contiguous [S, H, max_context_len, D] K/V
    layout (no block table): the baseline layout paging is measured against."""
    torch = _torch()
    S, H, D = q.shape
    if k.dim() != 4 or tuple(k.shape[:2]) != (S, H) or k.shape[3] != D or \
            tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [num_seqs, num_heads, max_context_len, head_dim]")
    if tuple(out.shape) != (S, H, D) or out.dtype != q.dtype or k.dtype != q.dtype or \
            v.dtype != q.dtype:
        raise ValueError("out/q/k/v dtype or shape mismatch")
    T = k.shape[2]
    if workspace is None:
        n = contiguous_workspace_size(S, H, D, T, partition_size)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    _check("pkv_contiguous_attention_decode",
           lib().pkv_contiguous_attention_decode(
               _dev(out, "out"), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"),
               _dev(context_lens, "context_lens", torch.int32, 1), float(scale), S, H, D, T,
               _dtype_code(q.dtype), int(partition_size), _dev(workspace, "workspace"),
               workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def paged_attention_prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                            scale, max_query_len, stream=None):
    """Causal attention of each sequence's new tokens (rows query_start[s] ..
    query_start[s+1]-1 of q) over its paged cache, the new tokens included."""
    torch = _torch()
    T, H, D = q.shape
    nb, H2, B, D2 = k_cache.shape
    S = context_lens.shape[0]
    if (H2, D2) != (H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shape mismatch")
    if tuple(out.shape) != (T, H, D) or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("out/q/cache dtype or shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("block_tables [S, max_blocks], query_start [S+1] expected")
    _check("pkv_paged_attention_prefill",
           lib().pkv_paged_attention_prefill(
               _dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"),
               _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables", torch.int32),
               _dev(context_lens, "context_lens", torch.int32, 1),
               _dev(query_start, "query_start", torch.int32, 1), float(scale), S, H, D, B,
               block_tables.shape[1], nb, int(max_query_len), T, _dtype_code(q.dtype),
               _stream(stream)))
    return out


def paged_attention_prefill_write(out, q, k, v, k_cache, v_cache, block_tables, context_lens,
                                  query_start, scale, max_query_len, stream=None):
    """Whole prompts: writes every prompt token's K and V (rows of k, v) into the
    cache at its position and computes the causal attention of the prompts,
    reading K and V from k and v, in one kernel."""
    torch = _torch()
    T, H, D = q.shape
    nb, H2, B, D2 = k_cache.shape
    S = context_lens.shape[0]
    if (H2, D2) != (H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shape mismatch")
    if tuple(k.shape) != (T, H, D) or tuple(v.shape) != (T, H, D):
        raise ValueError("k and v must be [num_query_tokens, num_heads, head_dim]")
    if tuple(out.shape) != (T, H, D) or len({out.dtype, q.dtype, k.dtype, v.dtype,
                                             k_cache.dtype, v_cache.dtype}) != 1:
        raise ValueError("out/q/k/v/cache dtype or shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("block_tables [S, max_blocks], query_start [S+1] expected")
    _check("pkv_paged_attention_prefill_write",
           lib().pkv_paged_attention_prefill_write(
               _dev(out, "out"), _dev(q, "q"), _dev(k, "k"), _dev(v, "v"),
               _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
               _dev(block_tables, "block_tables", torch.int32),
               _dev(context_lens, "context_lens", torch.int32, 1),
               _dev(query_start, "query_start", torch.int32, 1), float(scale), S, H, D, B,
               block_tables.shape[1], nb, int(max_query_len), T, _dtype_code(q.dtype),
               _stream(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                   partition_size=0, stream=None):
    """paged_attention_decode without a workspace, for callers that cannot
    allocate device memory: the library's static per-device scratch array
    (NOALLOC_SCRATCH_BYTES) is used instead.  Calls that overlap on the GPU
    share that array and must not run concurrently."""
    torch = _torch()
    S, H, D = q.shape
    nb, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shape mismatch")
    if tuple(out.shape) != (S, H, D) or out.dtype != q.dtype or k_cache.dtype != q.dtype:
        raise ValueError("out/q/cache dtype or shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    ptrs = [_dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables", torch.int32),
            _dev(context_lens, "context_lens", torch.int32, 1)]
    _check("pkv_paged_attention_decode_noalloc",
           lib().pkv_paged_attention_decode_noalloc(*ptrs, float(scale), S, H, D, B,
                                                    block_tables.shape[1], nb,
                                                    _dtype_code(q.dtype), int(partition_size),
                                                    _stream(stream)))
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """k_cache[slot // B, h, slot % B] = k[t, h] (and v) for slot_mapping[t] >= 0."""
    torch = _torch()
    T, H, D = k.shape
    nb, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k/v/cache shape mismatch")
    if k.dtype != k_cache.dtype or v.dtype != k.dtype or v_cache.dtype != k.dtype:
        raise TypeError("k, v and the caches must share a dtype")
    _check("pkv_reshape_and_cache",
           lib().pkv_reshape_and_cache(_dev(k, "k"), _dev(v, "v"), _dev(k_cache, "k_cache"),
                                       _dev(v_cache, "v_cache"),
                                       _dev(slot_mapping, "slot_mapping", torch.int64, 1),
                                       T, H, D, B, nb, _dtype_code(k.dtype), _stream(stream)))


def copy_blocks(k_cache, v_cache, pairs, stream=None):
    """For each (src, dst) row of pairs: whole-block copy in both pools."""
    torch = _torch()
    nb, H, B, D = k_cache.shape
    P = pairs.shape[0] if pairs.numel() else 0
    if P == 0:
        return
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [num_pairs, 2]")
    _check("pkv_copy_blocks",
           lib().pkv_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                 _dev(pairs, "pairs", torch.int32), P, H, D, B, nb,
                                 _dtype_code(k_cache.dtype), _stream(stream)))


def _reachable(t, name):
    """A CUDA tensor or a pinned host tensor (the kernel dereferences it)."""
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("%s must be a CUDA tensor or pinned host memory" % name)
    return t.data_ptr()


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs, stream=None):
    """Whole-block copies between two pools (GPU <-> pinned CPU, either way):
    dst[pairs[p, 1]] = src[pairs[p, 0]] for K and V."""
    torch = _torch()
    snb, H, B, D = src_k.shape
    dnb = dst_k.shape[0]
    if tuple(dst_k.shape[1:]) != (H, B, D) or src_v.shape != src_k.shape or \
            dst_v.shape != dst_k.shape:
        raise ValueError("pool shape mismatch")
    if not (src_k.dtype == src_v.dtype == dst_k.dtype == dst_v.dtype):
        raise TypeError("the pools must share a dtype")
    P = pairs.shape[0] if pairs.numel() else 0
    if P == 0:
        return
    if pairs.dim() != 2 or pairs.shape[1] != 2 or pairs.dtype != torch.int32:
        raise ValueError("pairs must be int32 [num_pairs, 2]")
    _check("pkv_swap_blocks",
           lib().pkv_swap_blocks(_reachable(dst_k, "dst_k"), _reachable(dst_v, "dst_v"),
                                 _reachable(src_k, "src_k"), _reachable(src_v, "src_v"),
                                 _reachable(pairs, "pairs"), P, H, D, B, snb, dnb,
                                 _dtype_code(src_k.dtype), _stream(stream)))


def get_device_error(clear=True, stream=None) -> int:
    """Device error bits (PKV_DEVERR_*) of the current device; syncs the stream."""
    bits = ctypes.c_int32(0)
    st = lib().pkv_get_device_error(ctypes.byref(bits), int(bool(clear)), _stream(stream))
    if st not in (PKV_OK, PKV_ERR_DEVICE):
        _check("pkv_get_device_error", st)
    return bits.value


def set_decode_wait_limit(ns: int) -> int:
    """Bound (ns) of the decode kernels' pipeline waits for later launches;
    returns the bound it replaces (default 1 s).  Short bounds exist to
    exercise the timeout path."""
    prev = ctypes.c_uint64(0)
    _check("pkv_set_decode_wait_limit",
           lib().pkv_set_decode_wait_limit(int(ns), ctypes.byref(prev)))
    return prev.value


# ------------------------------------------------------------- block manager
class BlockManager:
    """Host KV block manager (C++ in libpagedkv.so)."""

    def __init__(self, num_blocks: int, block_size: int, seed: int):
        h = ctypes.c_void_p()
        _check("pkv_bm_create", lib().pkv_bm_create(int(num_blocks), int(block_size),
                                                    int(seed) & ((1 << 64) - 1),
                                                    ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pkv_bm_destroy(h)
            self._h = None

    def add_sequence(self, seq_id: int, prompt_len: int) -> np.ndarray:
        slots = np.empty(max(prompt_len, 1), dtype=np.int64)
        _check("pkv_bm_add_sequence",
               lib().pkv_bm_add_sequence(self._h, int(seq_id), int(prompt_len),
                                         slots.ctypes.data_as(ctypes.c_void_p)))
        return slots[:prompt_len]

    def fork(self, parent: int, child: int) -> None:
        _check("pkv_bm_fork", lib().pkv_bm_fork(self._h, int(parent), int(child)))

    def append_slot(self, seq_id: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_bm_append_slot",
               lib().pkv_bm_append_slot(self._h, int(seq_id), ctypes.byref(slot),
                                        ctypes.byref(src), ctypes.byref(dst)))
        return slot.value, src.value, dst.value

    def append_slots(self, seq_ids):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int32)
        npairs = ctypes.c_int32(0)
        _check("pkv_bm_append_slots",
               lib().pkv_bm_append_slots(self._h, ids.ctypes.data_as(ctypes.c_void_p), n,
                                         slots.ctypes.data_as(ctypes.c_void_p),
                                         pairs.ctypes.data_as(ctypes.c_void_p),
                                         ctypes.byref(npairs)))
        return slots[:n], pairs[:npairs.value]

    def free_sequence(self, seq_id: int) -> None:
        _check("pkv_bm_free_sequence", lib().pkv_bm_free_sequence(self._h, int(seq_id)))

    def block_table(self, seq_id: int) -> list:
        n = ctypes.c_int32(0)
        st = lib().pkv_bm_block_table(self._h, int(seq_id), None, 0, ctypes.byref(n))
        if st != PKV_OK and n.value == 0:
            _check("pkv_bm_block_table", st)
        buf = np.empty(max(n.value, 1), dtype=np.int32)
        _check("pkv_bm_block_table",
               lib().pkv_bm_block_table(self._h, int(seq_id), buf.ctypes.data_as(ctypes.c_void_p),
                                        n.value, ctypes.byref(n)))
        return buf[:n.value].tolist()

    def context_len(self, seq_id: int) -> int:
        n = ctypes.c_int32(0)
        _check("pkv_bm_context_len", lib().pkv_bm_context_len(self._h, int(seq_id),
                                                              ctypes.byref(n)))
        return n.value

    def export(self, seq_ids, max_blocks: int):
        """(block_tables int32 [n, max_blocks] with -1 padding, context_lens int32 [n])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        tables = np.empty((max(n, 1), max_blocks), dtype=np.int32)
        ctx = np.empty(max(n, 1), dtype=np.int32)
        _check("pkv_bm_export",
               lib().pkv_bm_export(self._h, ids.ctypes.data_as(ctypes.c_void_p), n,
                                   tables.ctypes.data_as(ctypes.c_void_p), int(max_blocks),
                                   ctx.ctypes.data_as(ctypes.c_void_p)))
        return tables[:n], ctx[:n]

    def refcount(self, block: int) -> int:
        return lib().pkv_bm_refcount(self._h, int(block))

    def num_free(self) -> int:
        return lib().pkv_bm_num_free(self._h)

    # -- swapping ------------------------------------------------------------
    def add_cpu_pool(self, num_cpu_blocks: int, seed: int) -> None:
        _check("pkv_bm_add_cpu_pool", lib().pkv_bm_add_cpu_pool(self._h, int(num_cpu_blocks),
                                                                int(seed) & ((1 << 64) - 1)))
        self.num_cpu_blocks = num_cpu_blocks

    def _swap(self, fn, seq_ids):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        cap = sum(len(self.block_table(int(s))) for s in ids)
        pairs = np.empty((max(cap, 1), 2), dtype=np.int32)
        n = ctypes.c_int32(0)
        _check(fn, getattr(lib(), fn)(self._h, ids.ctypes.data_as(ctypes.c_void_p), ids.shape[0],
                                      pairs.ctypes.data_as(ctypes.c_void_p), cap,
                                      ctypes.byref(n)))
        return pairs[:n.value]

    def swap_out(self, seq_ids) -> np.ndarray:
        """Move a group of resident sequences to the CPU pool; (gpu, cpu) pairs."""
        return self._swap("pkv_bm_swap_out", seq_ids)

    def swap_in(self, seq_ids) -> np.ndarray:
        """Move a group of swapped-out sequences back to the GPU pool; (cpu, gpu) pairs."""
        return self._swap("pkv_bm_swap_in", seq_ids)

    def is_swapped(self, seq_id: int) -> bool:
        r = lib().pkv_bm_is_swapped(self._h, int(seq_id))
        if r < 0:
            raise PagedKVError("pkv_bm_is_swapped", PKV_ERR_INVALID, "unknown sequence")
        return bool(r)

    def cpu_refcount(self, block: int) -> int:
        return lib().pkv_bm_cpu_refcount(self._h, int(block))

    def num_free_cpu(self) -> int:
        return lib().pkv_bm_num_free_cpu(self._h)
