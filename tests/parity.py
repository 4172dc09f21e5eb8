"""Shared helpers of the parity tests: run a workload through the C ABI on the
GPU and through the CPU oracle on the same seeded inputs, then compare.

Tolerances (fp32 accumulation, bf16 output): out max-abs 2e-2 and mean-abs
1e-3, lse max-abs 5e-3; the KV cache must match bit for bit.
"""
import numpy as np
import torch

import oracle
from prefill_phase_attention_gb300 import binding
from prefill_phase_attention_gb300 import workloads as W

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 1e-3
LSE_MAX_ABS = 5e-3

# guard band (elements) around every GPU output buffer
GUARD = 4096
GUARD_BF16_BITS = 0x7FC7
GUARD_F32 = -12345.0


class Guarded:
    """A CUDA buffer with canary bands on both sides (catches stray writes)."""

    def __init__(self, shape, dtype, fill_bits=None, fill=None, device="cuda"):
        n = int(np.prod(shape))
        self.n = n
        self.buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
        if dtype == torch.bfloat16:
            self.buf.view(torch.int16).fill_(GUARD_BF16_BITS)
        else:
            self.buf.fill_(GUARD_F32)
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def guards_intact(self) -> bool:
        g = torch.cat([self.buf[:GUARD], self.buf[GUARD + self.n:]])
        if g.dtype == torch.bfloat16:
            return bool((g.view(torch.int16) == GUARD_BF16_BITS).all())
        return bool((g == GUARD_F32).all())


def run_step_gpu(wl, inp, cache_k_dev, cache_v_dev, guarded=True, window=0, block_table=None, rope_theta=0.0,
                 schedule=0):
    """One launch on the GPU; returns (out, lse) CUDA tensors (and checks guards).
    block_table (CUDA int32) selects the paged cache: the caches are then pools.
    schedule 1 .. 3 fixes the work schedule (pa_options.schedule; 0: the library's choice)."""
    dev = {k: v.cuda() for k, v in inp.items()}
    T = inp["q"].shape[0]
    out = Guarded((T, wl.n_heads, wl.head_dim), torch.bfloat16)
    lse = Guarded((T, wl.n_heads), torch.float32)
    if window or block_table is not None or rope_theta or schedule:
        binding.prefill_attn_varlen_ex(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"],
                                       cache_k_dev, cache_v_dev, dev["cache_offsets"], out.t, lse.t,
                                       scale=wl.scale, causal=wl.causal, window=window, block_table=block_table,
                                       rope_theta=rope_theta, schedule=schedule)
    else:
        binding.prefill_attn_varlen(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"],
                                    cache_k_dev, cache_v_dev, dev["cache_offsets"], out.t, lse.t,
                                    scale=wl.scale, causal=wl.causal)
    torch.cuda.synchronize()
    assert out.guards_intact(), "write outside out"
    assert lse.guards_intact(), "write outside lse"
    assert binding.prefill_attn_device_status() == 0
    return out.t, lse.t


def oracle_step(wl, inp, cache_k_bits, cache_v_bits, rows=None, want_cache=True, window=0, block_table=None,
                rope_theta=0.0):
    """The oracle on the same inputs; block_table (CPU int32 [B, max_blocks]) = paged pools."""
    cap, bs = wl.max_cache_len, 0
    if block_table is not None:
        bs = cache_k_bits.shape[2]
        cap = block_table.shape[1] * bs
        block_table = np.ascontiguousarray(block_table, np.int32)
    return oracle.prefill_attention(
        W.bf16_bits(inp["q"]), W.bf16_bits(inp["k"]), W.bf16_bits(inp["v"]),
        inp["cu_seqlens_q"].numpy(), inp["cu_seqlens_k"].numpy(), inp["cache_offsets"].numpy(),
        cache_k_bits, cache_v_bits, n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim,
        max_cache_len=cap, scale=wl.scale, causal=wl.causal, window=window, rows=rows,
        want_cache=want_cache, block_table=block_table, block_size=bs, rope_theta=rope_theta)


def compare(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, label=""):
    """Element-wise comparison on all rows, or on the flattened (t*H+h) rows given."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.cpu().numpy().astype(np.float64)
    H = o.shape[1]
    if rows is not None:
        t, h = rows // H, rows % H
        o, out_ref, l, lse_ref = o[t, h], out_ref[t, h], l[t, h], lse_ref[t, h]
    err = np.abs(o - out_ref)
    lerr = np.abs(l - lse_ref)
    assert np.isfinite(o).all(), f"{label}: non-finite output"
    assert err.max() <= OUT_MAX_ABS, f"{label}: out max-abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{label}: out mean-abs {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX_ABS, f"{label}: lse max-abs {lerr.max():.3e}"
    return float(err.max()), float(err.mean()), float(lerr.max())


def sample_rows(step, n_heads, n, seed):
    """Rows (t*H+h) spread over every sequence: first/last tokens, tile edges and random ones."""
    rng = np.random.default_rng(seed)
    cu = step.cu_seqlens_q()
    picks = []
    for b in range(step.num_seqs):
        lo, hi = cu[b], cu[b + 1]
        if hi <= lo:
            continue
        cand = {lo, hi - 1}
        for edge in range(lo + 127, hi, 128):
            cand.update({edge, min(edge + 1, hi - 1)})
        cand = sorted(cand)
        if len(cand) > n:
            cand = list(rng.choice(cand, n, replace=False))
        extra = rng.integers(lo, hi, size=max(1, n // 4)).tolist()
        for t in cand + extra:
            picks.append(int(t) * n_heads + int(rng.integers(0, n_heads)))
    return np.unique(np.array(picks, dtype=np.int64))


def compare_rotated_cache(got_bits, ref_bits, label=""):
    """Cache entries holding a rotated key: GPU (fp32 rotation rounded to bf16)
    and oracle (fp64 rotation rounded to bf16) may differ by one bf16 ulp where
    the exact value sits next to a rounding boundary, or, where x cos - y sin
    cancels, by the fp32 rotation's absolute error (a few 1e-7 * (|x| + |y|):
    2^-16 covers |x|, |y| up to 8); everything else is bit-identical."""
    as_f = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()
    diff = got_bits != ref_bits
    if not diff.any():
        return 0
    g, r = as_f(got_bits[diff]), as_f(ref_bits[diff])
    assert np.isfinite(g).all(), f"{label}: non-finite rotated key"
    tol = np.maximum(np.abs(g), np.abs(r)) * 2.0 ** -7 + 2.0 ** -16
    assert (np.abs(g - r) <= tol).all(), \
        f"{label}: rotated key off by {np.abs(g - r).max():.3e} (more than one bf16 ulp + 2^-16)"
    assert diff.mean() < 0.01, f"{label}: {diff.mean():.2%} of cache entries differ"
    return int(diff.sum())


def run_step_gpu_q8(wl, inp, ck, sk, cv, sv, window=0, rope_theta=0.0, block_table=None):
    """One launch over an int8 cache (codes + fp32 row scales, CUDA tensors);
    block_table (CUDA int32) selects paged pools."""
    dev = {k: v.cuda() for k, v in inp.items()}
    T = inp["q"].shape[0]
    out = Guarded((T, wl.n_heads, wl.head_dim), torch.bfloat16)
    lse = Guarded((T, wl.n_heads), torch.float32)
    binding.prefill_attn_varlen_ex(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"],
                                   ck, cv, dev["cache_offsets"], out.t, lse.t, scale=wl.scale, causal=wl.causal,
                                   window=window, rope_theta=rope_theta, cache_k_scale=sk, cache_v_scale=sv,
                                   block_table=block_table)
    torch.cuda.synchronize()
    assert out.guards_intact() and lse.guards_intact(), "write outside out/lse"
    assert binding.prefill_attn_device_status() == 0
    return out.t, lse.t


def oracle_step_q8(wl, inp, ck, sk, cv, sv, rows=None, window=0, rope_theta=0.0, want_cache=True,
                   block_table=None):
    """The oracle over an int8 cache (numpy codes/scales); cache images are (codes, scales).
    block_table (CPU int32 [B, max_blocks]): the codes/scales are paged pools."""
    cap, bs = wl.max_cache_len, 0
    if block_table is not None:
        bs = ck.shape[2]
        cap = block_table.shape[1] * bs
        block_table = np.ascontiguousarray(block_table, np.int32)
    return oracle.prefill_attention(
        W.bf16_bits(inp["q"]), W.bf16_bits(inp["k"]), W.bf16_bits(inp["v"]),
        inp["cu_seqlens_q"].numpy(), inp["cu_seqlens_k"].numpy(), inp["cache_offsets"].numpy(),
        ck, cv, n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim,
        max_cache_len=cap, scale=wl.scale, causal=wl.causal, window=window, rows=rows,
        rope_theta=rope_theta, kv_quant=1, cache_k_scale=sk, cache_v_scale=sv, want_cache=want_cache,
        block_table=block_table, block_size=bs)
