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


def sampled_oracle(q, k_cache, v_cache, tables: np.ndarray, ctx: np.ndarray, seqs, scale,
                   dtype: str, heads=None) -> np.ndarray:
    """fp64 oracle for selected sequences (and heads) of a device-resident batch.

    The blocks those sequences use are copied to the host into a compact pool
    and their tables renumbered (placement does not change the result); the
    oracle then computes each selected row.  Returns [len(seqs), len(heads), D].
    """
    import torch
    H = q.shape[1]
    B = k_cache.shape[2]
    heads = list(range(H)) if heads is None else list(heads)
    used = []
    for s in seqs:
        n = -(-int(ctx[s]) // B)
        used.extend(int(b) for b in tables[s, :n])
    uniq = sorted(set(used)) or [0]
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.long, device=k_cache.device)
    hidx = torch.tensor(heads, dtype=torch.long, device=k_cache.device)
    kc = W.torch_to_words(k_cache.index_select(0, idx).index_select(1, hidx))
    vc = W.torch_to_words(v_cache.index_select(0, idx).index_select(1, hidx))
    sidx = torch.tensor(list(seqs), dtype=torch.long, device=q.device)
    qh = W.torch_to_words(q.index_select(0, sidx).index_select(1, hidx))
    mb = max(1, max(-(-int(ctx[s]) // B) for s in seqs))
    bt = np.full((len(seqs), mb), -1, np.int32)
    for i, s in enumerate(seqs):
        n = -(-int(ctx[s]) // B)
        bt[i, :n] = [remap[int(b)] for b in tables[s, :n]]
    cl = np.array([ctx[s] for s in seqs], np.int32)
    return oracle.paged_attention_decode_threaded(qh, kc, vc, bt, cl, float(np.float32(scale)),
                                                  ORC_DTYPE[dtype], threads=8)
