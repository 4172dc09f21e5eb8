"""Seeded synthetic inputs for causal varlen prefill attention.

This module only *builds inputs*: sequence lengths, cumulative offsets, cache
prefixes and N(0,1) bf16 tensors.  It holds none of the attention arithmetic,
so the CUDA path and the CPU oracle can both be fed from it without sharing any
of the method.

Shapes follow the flattened varlen layout of "大模型 Prompt Prefill 阶段的高效
Batching 与算子排布" (nxmr.cn, §2: prompts packed head-to-tail into one
[Total_Tokens, ...] stream indexed by cu_seqlens, e.g. lengths 5, 2, 3 give
cu_seqlens [0, 5, 7, 10]) and the per-sequence cache layout
(num_heads, seq_len, head_dim) of the worked example in "大语言模型推理核心：
Prefill与Decode原理及工程优化" (yfxerp.com, §2.1).  The first five named
workloads are the ones this library is measured on; long8k is the long32k
shape at a quarter of the length, used for profiling:

=================  ===========================================================
tiny_packed        lengths [5, 2, 3], 4/4 heads, head_dim 32, empty cache
layer512           one 512-token prompt, 32/32 heads, head_dim 128
varlen16           16 prompts, lengths ~ U{10..2048}, 32/32 heads, head_dim 128
chunked_decode     8192-token prompt as 16 chunks of 512, each step packed with
                   64 one-token decode rows over cached contexts ~ U{256..4096};
                   GQA 32/8 heads, head_dim 128 (16 launches)
long32k            one 32768-token prompt, 32/32 heads, head_dim 128
long8k             one 8192-token prompt, 32/32 heads, head_dim 128
chunk512           chunked_decode's chunk at launch 8 alone: 512 new tokens
                   over a 4096-token cached prefix, GQA 32/8, head_dim 128
decode64           chunked_decode's 64 decode rows at launch 8 alone
=================  ===========================================================
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

# bf16 pattern used to mark cache entries that no call may read or write
# (a quiet NaN with a recognisable payload).
CACHE_SENTINEL_BITS = 0x7FC5


@dataclasses.dataclass
class Step:
    """One launch: the sequences packed into one flattened batch."""

    seqlens_q: List[int]        # new tokens of each sequence in this launch
    cache_offsets: List[int]    # tokens already cached for each sequence

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    def cu_seqlens_q(self) -> List[int]:
        return [0] + list(np.cumsum(self.seqlens_q, dtype=np.int64).tolist())

    def cu_seqlens_k(self) -> List[int]:
        lk = [p + n for p, n in zip(self.cache_offsets, self.seqlens_q)]
        return [0] + list(np.cumsum(lk, dtype=np.int64).tolist())

    def visible_pairs(self, causal: bool = True, window: int = 0) -> int:
        """Number of (query, key) pairs the mask leaves visible (window: causal
        sliding window of that many most recent keys, 0 = none)."""
        tot = 0
        for n, p in zip(self.seqlens_q, self.cache_offsets):
            if causal and window > 0:
                # query i sees min(p + i + 1, window) keys
                full = max(0, min(n, window - p))          # rows with p + i + 1 <= window
                tot += full * p + full * (full + 1) // 2 + (n - full) * window
            else:
                tot += n * p + (n * (n + 1) // 2 if causal else n * n)
        return tot


@dataclasses.dataclass
class Workload:
    name: str
    n_heads: int
    n_kv_heads: int
    head_dim: int
    max_cache_len: int
    steps: List[Step]
    prefilled: List[int]        # cache tokens already present per slot before step 0
    seed: int
    causal: bool = True
    scale: Optional[float] = None

    def __post_init__(self):
        if self.scale is None:
            # 1/sqrt(d) rounded once to fp32, as the kernel receives it.
            self.scale = float(np.float32(1.0 / math.sqrt(self.head_dim)))

    @property
    def num_seqs(self) -> int:
        return self.steps[0].num_seqs

    def flops(self, window: int = 0) -> int:
        """Causal attention FLOPs: 4 * head_dim * n_heads per visible pair."""
        return 4 * self.head_dim * self.n_heads * sum(s.visible_pairs(self.causal, window) for s in self.steps)

    def tokens(self) -> int:
        return sum(s.total_q for s in self.steps)


def _tiny_packed() -> Workload:
    return Workload("tiny_packed", 4, 4, 32, 8, [Step([5, 2, 3], [0, 0, 0])], [0, 0, 0], seed=1)


def _layer512() -> Workload:
    return Workload("layer512", 32, 32, 128, 512, [Step([512], [0])], [0], seed=2)


def _varlen16() -> Workload:
    rng = np.random.default_rng(3)
    lens = rng.integers(10, 2048, size=16, endpoint=True).tolist()
    return Workload("varlen16", 32, 32, 128, 2048, [Step(lens, [0] * 16)], [0] * 16, seed=3)


def _chunked_decode(prompt: int = 8192, chunk: int = 512, n_decode: int = 64,
                    lo: int = 256, hi: int = 4096) -> Workload:
    rng = np.random.default_rng(4)
    ctx = rng.integers(lo, hi, size=n_decode, endpoint=True).tolist()
    n_chunks = prompt // chunk
    steps = []
    for s in range(n_chunks):
        steps.append(Step([chunk] + [1] * n_decode, [chunk * s] + [c + s for c in ctx]))
    cap = max(prompt, max(ctx) + n_chunks)
    return Workload("chunked_decode", 32, 8, 128, cap, steps, [0] + ctx, seed=4)


def _chunk512() -> Workload:
    # the chunk part of chunked_decode at its midpoint (launch 8): one 512-token
    # chunk over its 4096-token cached prefix, GQA 32/8
    return Workload("chunk512", 32, 8, 128, 4096 + 512, [Step([512], [4096])], [4096], seed=7)


def _decode64() -> Workload:
    # the decode part of chunked_decode at its midpoint (launch 8): its 64
    # one-token rows over their cached contexts, GQA 32/8
    ctx = np.random.default_rng(4).integers(256, 4096, size=64, endpoint=True).tolist()
    pref = [c + 8 for c in ctx]
    return Workload("decode64", 32, 8, 128, max(pref) + 1, [Step([1] * 64, pref)], pref, seed=8)


def _long32k() -> Workload:
    return Workload("long32k", 32, 32, 128, 32768, [Step([32768], [0])], [0], seed=5)


def _long8k() -> Workload:
    # the long32k shape family at a quarter of the length (profiling case: q/k/v
    # still exceed L2, device footprint under 1 GB)
    return Workload("long8k", 32, 32, 128, 8192, [Step([8192], [0])], [0], seed=6)


WORKLOADS = {
    "tiny_packed": _tiny_packed,
    "layer512": _layer512,
    "varlen16": _varlen16,
    "chunked_decode": _chunked_decode,
    "long32k": _long32k,
    "long8k": _long8k,
    "chunk512": _chunk512,
    "decode64": _decode64,
}


def get(name: str) -> Workload:
    return WORKLOADS[name]()


def random_workload(seed: int, *, head_dim: int, group: int, n_kv_heads: int = 2,
                    max_seqs: int = 5, max_len: int = 300, max_prefix: int = 300,
                    causal: bool = True, allow_empty: bool = True) -> Workload:
    """Small random varlen batch with random cached prefixes (parity tests)."""
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, max_seqs, endpoint=True))
    lens = rng.integers(0 if allow_empty else 1, max_len, size=b, endpoint=True).tolist()
    if sum(lens) == 0:
        lens[0] = 1
    pref = rng.integers(0, max_prefix, size=b, endpoint=True).tolist()
    cap = max(p + n for p, n in zip(pref, lens)) + int(rng.integers(0, 8))
    return Workload(f"random{seed}", n_kv_heads * group, n_kv_heads, head_dim, cap,
                    [Step(lens, pref)], pref, seed=1000 + seed, causal=causal)


def decode_workload(seed: int, *, head_dim: int, group: int, n_kv_heads: int = 2,
                    max_seqs: int = 24, max_prefix: int = 3000, causal: bool = True) -> Workload:
    """Decode-heavy random batch: mostly 1-4 new tokens over long cached
    prefixes (some on a tile edge), a few short chunks; the new tokens average
    well under 64 per sequence."""
    rng = np.random.default_rng(seed)
    b = int(rng.integers(4, max_seqs, endpoint=True))
    lens = [int(rng.integers(1, 4, endpoint=True)) if rng.random() < 0.85 else int(rng.integers(5, 120))
            for _ in range(b)]
    pref = []
    for _ in range(b):
        r = rng.random()
        if r < 0.1:
            pref.append(0)
        elif r < 0.25:
            pref.append(128 * int(rng.integers(1, max(2, max_prefix // 128))))
        else:
            pref.append(int(rng.integers(1, max_prefix, endpoint=True)))
    cap = max(p + n for p, n in zip(pref, lens)) + int(rng.integers(0, 8))
    return Workload(f"decode{seed}", n_kv_heads * group, n_kv_heads, head_dim, cap,
                    [Step(lens, pref)], pref, seed=2000 + seed, causal=causal)


# ---------------------------------------------------------------------------
# tensors
# ---------------------------------------------------------------------------

def _randn_bf16(g: torch.Generator, shape: Sequence[int]) -> torch.Tensor:
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_cache(wl: Workload, g: torch.Generator, sentinel: bool = True):
    """Cache [num_seqs, n_kv_heads, max_cache_len, head_dim] bf16 (CPU).

    Slot b holds ``wl.prefilled[b]`` seeded N(0,1) tokens; every other entry
    holds the NaN sentinel (or zero), so a read or a stray write is visible.
    """
    shape = (wl.num_seqs, wl.n_kv_heads, wl.max_cache_len, wl.head_dim)
    caches = []
    for _ in range(2):
        c = torch.empty(shape, dtype=torch.bfloat16)
        if sentinel:
            c.view(torch.int16).fill_(CACHE_SENTINEL_BITS)
        else:
            c.zero_()
        for b, p in enumerate(wl.prefilled):
            if p:
                c[b, :, :p] = _randn_bf16(g, (wl.n_kv_heads, p, wl.head_dim))
        caches.append(c)
    return caches[0], caches[1]


def make_paged_cache(wl: Workload, block_size: int, g: torch.Generator, extra_blocks: int = 3,
                     sentinel: bool = True):
    """A paged cache: (block_table [num_seqs, max_blocks] int32, pool_k, pool_v).

    The pools are [num_blocks, n_kv_heads, block_size, head_dim] bf16 (CPU)
    with num_blocks = num_seqs * max_blocks + extra_blocks, max_blocks =
    ceil(max_cache_len / block_size); each sequence gets max_blocks distinct
    physical blocks drawn by a seeded permutation.  Position p of sequence b
    is row p % block_size of block table[b][p // block_size]; the first
    ``wl.prefilled[b]`` positions hold seeded N(0,1) tokens, every other row
    the NaN sentinel (or zero).
    """
    B, Hk, d = wl.num_seqs, wl.n_kv_heads, wl.head_dim
    max_blocks = -(-wl.max_cache_len // block_size)
    num_blocks = B * max_blocks + extra_blocks
    perm = torch.randperm(num_blocks, generator=g)[: B * max_blocks]
    table = perm.to(torch.int32).reshape(B, max_blocks)
    pools = []
    for _ in range(2):
        c = torch.empty((num_blocks, Hk, block_size, d), dtype=torch.bfloat16)
        if sentinel:
            c.view(torch.int16).fill_(CACHE_SENTINEL_BITS)
        else:
            c.zero_()
        for b, p in enumerate(wl.prefilled):
            if p:
                vals = _randn_bf16(g, (Hk, p, d))
                for L in range(-(-p // block_size)):
                    rows = min(block_size, p - L * block_size)
                    c[int(table[b, L]), :, :rows] = vals[:, L * block_size: L * block_size + rows]
        pools.append(c)
    return table, pools[0], pools[1]


def make_q8_cache(wl: Workload, g: torch.Generator, sentinel: bool = True):
    """An int8 cache: (codes_k, scales_k, codes_v, scales_v) on the CPU.

    Codes int8 [num_seqs, n_kv_heads, max_cache_len, head_dim], scales fp32
    [num_seqs, n_kv_heads, max_cache_len].  The first ``wl.prefilled[b]`` rows of
    slot b hold what int8 rows of N(0,1)-like activations look like: codes drawn
    N(0, 36^2), rounded and clipped to [-127, 127], one code of each row set to
    +-127 (the row maximum), and scales uniform in [0.02, 0.035], so the values
    code * scale have about the spread of the bf16 tests' N(0,1) data.  Every
    other row holds random codes and a NaN scale (or zero codes and scale 0), so
    a read of it shows.
    """
    shape = (wl.num_seqs, wl.n_kv_heads, wl.max_cache_len, wl.head_dim)
    out = []
    for _ in range(2):
        codes = torch.randint(-127, 128, shape, generator=g, dtype=torch.int32).to(torch.int8)
        scales = torch.full(shape[:-1], float("nan") if sentinel else 0.0, dtype=torch.float32)
        if not sentinel:
            codes.zero_()
        for b, p in enumerate(wl.prefilled):
            if p:
                c = (torch.randn((wl.n_kv_heads, p, wl.head_dim), generator=g) * 36).round().clamp(-127, 127)
                col = torch.randint(0, wl.head_dim, (wl.n_kv_heads, p, 1), generator=g)
                sign = torch.randint(0, 2, (wl.n_kv_heads, p, 1), generator=g) * 2 - 1
                c.scatter_(2, col, (127 * sign).to(c.dtype))
                codes[b, :, :p] = c.to(torch.int8)
                scales[b, :, :p] = torch.rand((wl.n_kv_heads, p), generator=g) * 0.015 + 0.02
        out += [codes, scales]
    return tuple(out)


def make_paged_q8_cache(wl: Workload, block_size: int, g: torch.Generator, extra_blocks: int = 3,
                        sentinel: bool = True):
    """A paged int8 cache: (block_table, codes_k, scales_k, codes_v, scales_v).

    The table and block placement are drawn as in make_paged_cache; the pools
    are int8 [num_blocks, n_kv_heads, block_size, head_dim] and fp32
    [num_blocks, n_kv_heads, block_size], filled as make_q8_cache fills a slot:
    prefilled positions hold N(0, 36^2)-like codes (one +-127 per row) and
    scales in [0.02, 0.035], every other row random codes and a NaN scale.
    """
    B, Hk, d = wl.num_seqs, wl.n_kv_heads, wl.head_dim
    max_blocks = -(-wl.max_cache_len // block_size)
    num_blocks = B * max_blocks + extra_blocks
    perm = torch.randperm(num_blocks, generator=g)[: B * max_blocks]
    table = perm.to(torch.int32).reshape(B, max_blocks)
    out = [table]
    for _ in range(2):
        codes = torch.randint(-127, 128, (num_blocks, Hk, block_size, d), generator=g, dtype=torch.int32).to(torch.int8)
        scales = torch.full((num_blocks, Hk, block_size), float("nan") if sentinel else 0.0, dtype=torch.float32)
        if not sentinel:
            codes.zero_()
        for b, p in enumerate(wl.prefilled):
            if not p:
                continue
            c = (torch.randn((Hk, p, d), generator=g) * 36).round().clamp(-127, 127)
            col = torch.randint(0, d, (Hk, p, 1), generator=g)
            sign = torch.randint(0, 2, (Hk, p, 1), generator=g) * 2 - 1
            c.scatter_(2, col, (127 * sign).to(c.dtype))
            sc = torch.rand((Hk, p), generator=g) * 0.015 + 0.02
            for L in range(-(-p // block_size)):
                rows = min(block_size, p - L * block_size)
                blk = int(table[b, L])
                codes[blk, :, :rows] = c[:, L * block_size: L * block_size + rows].to(torch.int8)
                scales[blk, :, :rows] = sc[:, L * block_size: L * block_size + rows]
        out += [codes, scales]
    return tuple(out)


def make_step_inputs(wl: Workload, step: Step, g: torch.Generator):
    """q [T,H,d], k/v [T,Hk,d] bf16 and the int32 metadata of one launch (CPU)."""
    t = step.total_q
    q = _randn_bf16(g, (t, wl.n_heads, wl.head_dim))
    k = _randn_bf16(g, (t, wl.n_kv_heads, wl.head_dim))
    v = _randn_bf16(g, (t, wl.n_kv_heads, wl.head_dim))
    return dict(
        q=q, k=k, v=v,
        cu_seqlens_q=torch.tensor(step.cu_seqlens_q(), dtype=torch.int32),
        cu_seqlens_k=torch.tensor(step.cu_seqlens_k(), dtype=torch.int32),
        cache_offsets=torch.tensor(step.cache_offsets, dtype=torch.int32),
    )


def make_inputs(wl: Workload, sentinel: bool = True):
    """All inputs of a workload: (cache_k, cache_v, [per-step input dicts])."""
    g = torch.Generator().manual_seed(wl.seed)
    cache_k, cache_v = make_cache(wl, g, sentinel=sentinel)
    steps = [make_step_inputs(wl, s, g) for s in wl.steps]
    return cache_k, cache_v, steps


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a CPU tensor as a uint16 numpy array (no copy)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
