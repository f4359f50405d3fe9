"""Seeded synthetic inputs for the paged KV-cache decode path.

This module is the ONLY thing shared by the CUDA path's tests/benchmark and the
oracle's: it draws random numbers and sizes, and holds none of the method's
arithmetic (no address translation, no attention, no block management).  Block
tables and slot mappings are produced by the block manager (product side) and
by its independent model (oracle side), never here.

Workloads (shapes from the pages: OPT-13B is 40 heads x 128; the default block
size is 16; ShareGPT/Alpaca-like length mixes are replaced by seeded lognormal
and uniform draws because those traces are not available):

  tiny           seed 1001: 4 sequences, context lengths {1,15,16,37}, 8 heads,
                 head_dim 64, B 16, fp16, 64-block pool.
  opt13b         seed 1002: 64 sequences, 40 heads, head_dim 128, fp16, B 16,
                 lengths round(lognormal(ln 300, 1.0)) clipped to [1, 2048];
                 40 per-layer pools, each max(983, ceil(1.25 * needed)) blocks
                 (983 blocks = 12 GiB of KV over 40 layers, i.e. 15.7K slots).
  short          seed 1003: 256 sequences, lengths uniform [20, 300], 40 heads,
                 head_dim 128, bf16, B in {8, 16, 32, 64} with the same
                 per-token values for every B.
  shared_prefix  seed 1004: 32 prompts x 6 sequences, prompt uniform [128, 1024],
                 suffix uniform [1, 512] per sequence, 40 heads, head_dim 128,
                 fp16, B 16.
  long           seed 1005: 8 sequences, lengths uniform [8192, 32768], 32
                 heads, head_dim 128, fp16, B 16, an 80 GB (K+V) pool, split
                 length 512 tokens.
  prefill        seed 1006: 16 whole prompts, lengths uniform [512, 2048], 40
                 heads, head_dim 128, fp16, B 16 (the prompt phase).

Values are N(0, 1) rounded to the storage type.  Host arrays use numpy's
PCG64 (platform independent); device tensors use torch's CUDA generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

OPT13B_KV_BYTES_PER_TOKEN = 800 * 1024  # the detail page's "800 KB" per token (all layers)
GIB = 1 << 30


@dataclass
class Spec:
    name: str
    seed: int
    num_seqs: int
    num_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # "f16" or "bf16"
    partition_size: int = 0         # split length in tokens; 0 = balanced
    layers: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))

    @property
    def elem_bytes(self) -> int:
        return 2


SPECS = {
    "tiny": Spec("tiny", 1001, 4, 8, 64, 16, "f16",
                 extra=dict(context_lens=[1, 15, 16, 37], num_blocks=64)),
    "opt13b": Spec("opt13b", 1002, 64, 40, 128, 16, "f16", layers=40,
                   extra=dict(median=300.0, sigma=1.0, lo=1, hi=2048, kv_gib=12)),
    "short": Spec("short", 1003, 256, 40, 128, 16, "bf16",
                  extra=dict(lo=20, hi=300, block_sizes=(8, 16, 32, 64))),
    "shared_prefix": Spec("shared_prefix", 1004, 192, 40, 128, 16, "f16",
                          extra=dict(groups=32, per_group=6, prompt=(128, 1024),
                                     suffix=(1, 512))),
    "long": Spec("long", 1005, 8, 32, 128, 16, "f16", partition_size=512,
                 extra=dict(lo=8192, hi=32768, pool_bytes=80 * 10**9)),
    "prefill": Spec("prefill", 1006, 16, 40, 128, 16, "f16",
                    extra=dict(lo=512, hi=2048)),
}


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def context_lens(spec: Spec) -> np.ndarray:
    """Per-sequence context lengths (tokens attended, the new token included)."""
    r = rng(spec.seed, 1)
    e = spec.extra
    if spec.name == "tiny":
        return np.array(e["context_lens"], dtype=np.int32)
    if spec.name == "opt13b":
        x = r.lognormal(mean=math.log(e["median"]), sigma=e["sigma"], size=spec.num_seqs)
        return np.clip(np.rint(x), e["lo"], e["hi"]).astype(np.int32)
    if spec.name in ("short", "long", "prefill"):
        return r.integers(e["lo"], e["hi"], size=spec.num_seqs, endpoint=True).astype(np.int32)
    if spec.name == "shared_prefix":
        p, s = prompt_and_suffix_lens(spec)
        return (np.repeat(p, e["per_group"]) + s).astype(np.int32)
    raise KeyError(spec.name)


def prompt_and_suffix_lens(spec: Spec):
    """shared_prefix: per-group prompt lengths [G] and per-sequence suffix lengths [G*6]."""
    e = spec.extra
    r = rng(spec.seed, 2)
    p = r.integers(e["prompt"][0], e["prompt"][1], size=e["groups"], endpoint=True)
    s = r.integers(e["suffix"][0], e["suffix"][1], size=e["groups"] * e["per_group"],
                   endpoint=True)
    return p.astype(np.int32), s.astype(np.int32)


def blocks_needed(ctx: np.ndarray, block_size: int) -> int:
    return int(sum(-(-int(c) // block_size) for c in ctx))


def pool_blocks(spec: Spec, ctx: np.ndarray, block_size: int | None = None) -> int:
    """Physical blocks per pool (one pool per layer for K and one for V)."""
    B = block_size or spec.block_size
    need = blocks_needed(ctx, B)
    H, D = spec.num_heads, spec.head_dim
    if spec.name == "tiny":
        return spec.extra["num_blocks"]
    if spec.name == "opt13b":
        per_block = 2 * H * B * D * spec.elem_bytes          # K and V
        per_layer = spec.extra["kv_gib"] * GIB // spec.layers
        return max(per_layer // per_block, math.ceil(1.25 * need))
    if spec.name == "long":
        per_block = 2 * H * B * D * spec.elem_bytes
        return int(spec.extra["pool_bytes"] // per_block)
    if spec.name == "shared_prefix":
        p, s = prompt_and_suffix_lens(spec)
        g = spec.extra["per_group"]
        bound = sum(-(-int(x) // B) for x in p) + sum(-(-int(x) // B) + 1 for x in s)
        return math.ceil(1.25 * bound)
    return math.ceil(1.25 * need)


def normal_words(shape, dtype: str, seed: int, stream: int) -> np.ndarray:
    """N(0,1) samples rounded to fp16/bf16, returned as raw uint16 words (host)."""
    x = rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch
        return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def torch_dtype(dtype: str):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def device_normal(shape, dtype: str, seed: int, device="cuda", out=None):
    """N(0,1) samples of the storage type, drawn on the device (seeded)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if out is None:
        out = torch.empty(shape, dtype=torch_dtype(dtype), device=device)
    out.normal_(generator=g)
    return out


def words_to_torch(words: np.ndarray, dtype: str):
    """Host uint16 words -> torch tensor of the storage type (same bits)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(words).view(np.int16))
    return t.view(torch_dtype(dtype))


def torch_to_words(t) -> np.ndarray:
    """Torch fp16/bf16 tensor (any device) -> host uint16 words (same bits)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
