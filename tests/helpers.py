"""Shared helpers of the GPU parity tests: tolerance check, random cases,
sampled oracle evaluation at full size.  Inputs come from the seeded
generators; expected values only from ``oracle``."""
from __future__ import annotations

import numpy as np

import oracle
from paged_kv_cache_05_gb300 import workloads as W

# Attention tolerance against the fp64 oracle: |gpu - ref| <= ABS + REL * |ref|
# element by element (max-abs error 2e-3 and relative error 1e-2, read as an
# allclose bound because a pure relative bound is unbounded near zero and the
# bf16 output rounding alone is up to 2^-9 relative).
TOL_ABS = 2e-3
TOL_REL = 1e-2

ORC_DTYPE = {"f16": oracle.F16, "bf16": oracle.BF16}


def attn_check(gpu_out, ref: np.ndarray, what: str = "") -> dict:
    """Element-wise tolerance check of a GPU result (torch, any device) against fp64."""
    import torch
    g = gpu_out.detach().to(torch.float64).cpu().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    err = np.abs(g - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = [tuple(int(i) for i in x) for x in np.argwhere(bad)[:5]]
        raise AssertionError("%s: %d elements out of tolerance, e.g. %s: gpu %s ref %s" % (
            what, int(bad.sum()), idx, [g[i] for i in idx], [ref[i] for i in idx]))
    big = np.abs(ref) >= 1e-2
    return dict(max_abs=float(err.max()),
                max_rel=float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0)


def words(shape, dtype, rs) -> np.ndarray:
    x = rs.standard_normal(size=shape).astype(np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    import torch
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def random_case(rs, S, H, D, B, ctx, dtype, spare=5, max_blocks=None):
    """Host words for q and the pools, and a random non-contiguous placement."""
    nblk = [-(-int(c) // B) for c in ctx]
    nb = sum(nblk) + spare
    mb = max_blocks or max(max(nblk), 1)
    perm = rs.permutation(nb)
    bt = np.full((S, mb), -1, dtype=np.int32)
    k = 0
    for s in range(S):
        bt[s, :nblk[s]] = perm[k:k + nblk[s]]
        k += nblk[s]
    return dict(q=words((S, H, D), dtype, rs), kc=words((nb, H, B, D), dtype, rs),
                vc=words((nb, H, B, D), dtype, rs), bt=bt, ctx=np.array(ctx, np.int32),
                S=S, H=H, D=D, B=B, nb=nb, dtype=dtype)


def to_dev(w: np.ndarray, dtype: str):
    return W.words_to_torch(w, dtype).cuda()


def compact_rows(kc: np.ndarray, vc: np.ndarray, tables: np.ndarray, ctx, seqs, B: int):
    """Host pools restricted to the blocks the selected sequences use, with their
    tables renumbered (placement does not change the result)."""
    used = []
    for s in seqs:
        n = -(-int(ctx[s]) // B)
        used.extend(int(b) for b in tables[s, :n])
    uniq = sorted(set(used)) or [0]
    remap = {b: i for i, b in enumerate(uniq)}
    mb = max(1, max(-(-int(ctx[s]) // B) for s in seqs))
    bt = np.full((len(seqs), mb), -1, np.int32)
    for i, s in enumerate(seqs):
        n = -(-int(ctx[s]) // B)
        bt[i, :n] = [remap[int(b)] for b in tables[s, :n]]
    idx = np.array(uniq)
    return kc[idx], vc[idx], bt, np.array([ctx[s] for s in seqs], np.int32), uniq


def host_threads() -> int:
    """Host cores this process may use (threads for the oracle's C routine)."""
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except Exception:
        return os.cpu_count() or 1


def sampled_oracle(q_host: np.ndarray, kc_host: np.ndarray, vc_host: np.ndarray,
                   tables: np.ndarray, ctx, seqs, scale, dtype: str) -> np.ndarray:
    """fp64 oracle rows [len(seqs), H, D] for selected sequences of a batch whose
    pools are given on the host (full pools or any superset of the used blocks)."""
    B = kc_host.shape[2]
    kc, vc, bt, cl, _ = compact_rows(kc_host, vc_host, tables, ctx, seqs, B)
    return oracle.paged_attention_decode_threaded(q_host[list(seqs)], kc, vc, bt, cl,
                                                  float(np.float32(scale)), ORC_DTYPE[dtype],
                                                  threads=host_threads())


def device_blocks_to_host(k_cache, v_cache, block_ids):
    """Host words of selected physical blocks of device pools: a dict-like pair
    of arrays indexed by position in ``block_ids``."""
    import torch
    idx = torch.tensor(list(block_ids), dtype=torch.long, device=k_cache.device)
    return (W.torch_to_words(k_cache.index_select(0, idx)),
            W.torch_to_words(v_cache.index_select(0, idx)))


def spread(ctx, n):
    """n sequence indices spread over the range of context lengths (shortest and
    longest included)."""
    order = np.argsort(ctx, kind="stable")
    pick = np.unique(np.linspace(0, len(ctx) - 1, n).round().astype(int))
    return sorted(int(order[i]) for i in pick)


def prefill_oracle_threaded(q, kc, vc, bt, ctx, qs, scale, dtype: str, threads: int = 8,
                            rows_per_call: int = 32):
    """The prompt-phase oracle on pieces of at most rows_per_call query rows,
    spread over host threads (the C routine runs without the GIL).  Each piece
    is the unchanged oracle on one sequence: rows a .. b-1 of a sequence with
    context n and qlen new tokens are the new tokens of the same sequence cut
    at context n - qlen + b (the rows attend positions up to their own)."""
    import threading
    T = int(qs[-1])
    H, D = kc.shape[1], kc.shape[3]
    out = np.zeros((T, H, D), np.float64)
    pieces = []
    for s in range(len(ctx)):
        q0, q1 = int(qs[s]), int(qs[s + 1])
        n, ql = int(ctx[s]), q1 - q0
        for a in range(0, ql, rows_per_call):
            b = min(a + rows_per_call, ql)
            pieces.append((s, q0 + a, q0 + b, n - ql + b))
    pieces.sort(key=lambda p: -(p[2] - p[1]) * p[3])
    errs = []

    def worker(i):
        try:
            for s, a, b, n_cut in pieces[i::threads]:
                out[a:b] = oracle.paged_attention_prefill(
                    q[a:b], kc, vc, bt[s:s + 1], np.array([n_cut], np.int32),
                    np.array([0, b - a], np.int32), scale, ORC_DTYPE[dtype])
        except Exception as e:  # surfaced below
            errs.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(max(1, threads))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errs:
        raise errs[0]
    return out
