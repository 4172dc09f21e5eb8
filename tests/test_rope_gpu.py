"""GPU parity of the rotary position embedding (pa_options.rope_theta): the
CUDA path (rotary prologue kernel + attention) against the fp64 CPU oracle on
the same inputs.  out/lse within the stated tolerances; V cache bit-exact; the
rotated keys written to the cache within one bf16 ulp (or 2^-16 where the rotation cancels) of the oracle's (fp32
versus fp64 rotation, each rounded once to bf16), every other cache entry
bit-exact; q and k left unmodified."""
import numpy as np
import pytest
import torch

from prefill_phase_attention_gb300 import binding
from prefill_phase_attention_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(oracle_mod):
    from prefill_phase_attention_gb300 import build
    build.build()
    binding.load()
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


def _rotated_mask(shape, step, table=None, bs=0):
    """Cache entries (contiguous [B,Hk,cap,d] or pool [NB,Hk,bs,d]) that receive a new key."""
    m = np.zeros(shape, dtype=bool)
    for b, (n, P) in enumerate(zip(step.seqlens_q, step.cache_offsets)):
        for pos in range(P, P + n):
            if table is None:
                m[b, :, pos] = True
            else:
                m[int(table[b, pos // bs]), :, pos % bs] = True
    return m


def _check_caches(got_k, got_v, ref_k, ref_v, mask, label):
    assert np.array_equal(got_v, ref_v), f"{label}: cache_v differs"
    assert np.array_equal(got_k[~mask], ref_k[~mask]), f"{label}: cache_k differs outside the new rows"
    PT.compare_rotated_cache(got_k[mask], ref_k[mask], label)


def _run(wl, theta, window=0, bs=0, rows=None, seed=0, schedule=0):
    _, _, (inp,) = W.make_inputs(wl)
    table = None
    if bs:
        table, ck, cv = W.make_paged_cache(wl, bs, torch.Generator().manual_seed(seed))
    else:
        ck, cv, _ = W.make_inputs(wl)
    ck_d = PT.Guarded(ck.shape, torch.bfloat16, fill=ck)
    cv_d = PT.Guarded(cv.shape, torch.bfloat16, fill=cv)
    q0, k0 = inp["q"].clone(), inp["k"].clone()
    dev_inp = {kk: vv for kk, vv in inp.items()}
    out, lse = PT.run_step_gpu(wl, dev_inp, ck_d.t, cv_d.t, window=window,
                               block_table=None if table is None else table.cuda(), rope_theta=theta,
                               schedule=schedule)
    assert ck_d.guards_intact() and cv_d.guards_intact(), "write outside the cache"
    ref_out, ref_lse, ref_ck, ref_cv = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv), rows=rows,
                                                      window=window,
                                                      block_table=None if table is None else table.numpy(),
                                                      rope_theta=theta)
    PT.compare(out, lse, ref_out, ref_lse, rows=rows, label=f"{wl.name} rope {theta}")
    mask = _rotated_mask(ck.shape, wl.steps[0], table, bs)
    _check_caches(W.bf16_bits(ck_d.t.cpu()), W.bf16_bits(cv_d.t.cpu()), ref_ck, ref_cv, mask, wl.name)
    assert torch.equal(inp["q"], q0) and torch.equal(inp["k"], k0)


@pytest.mark.parametrize("seed", range(48))
def test_rope_random_shapes(seed):
    """Every head_dim x GQA group, two bases, with cached prefixes; some calls
    also use a sliding window, a paged cache or no causal mask."""
    d = [32, 64, 128][seed % 3]
    group = [1, 2, 4, 8][(seed // 3) % 4]
    theta = [10000.0, 500000.0][seed % 2]
    causal = seed % 11 != 10
    window = 150 if (causal and seed % 5 == 2) else 0
    bs = [0, 0, 16, 64][seed % 4]
    wl = W.random_workload(700 + seed, head_dim=d, group=group, n_kv_heads=2, causal=causal, max_prefix=500)
    _run(wl, theta, window=window, bs=bs, seed=seed, schedule=seed // 12)


def test_rope_long_prompt_sampled():
    """Positions up to 32767: the largest angles (m * inv_freq[0] = m radians)."""
    wl = W.get("long32k")
    rows = PT.sample_rows(wl.steps[0], wl.n_heads, 64, seed=3)
    _run(wl, 10000.0, rows=rows)


def test_rope_chunked_decode_all_steps():
    """16 launches of chunk + decode rows: each launch reads the rotated keys the
    earlier ones wrote, and rotates its own at positions 512 s + i and L_j + s."""
    wl = W.get("chunked_decode")
    ck, cv, steps = W.make_inputs(wl)
    ck_d, cv_d = ck.cuda(), cv.cuda()
    rk, rv = W.bf16_bits(ck).copy(), W.bf16_bits(cv).copy()
    mask = np.zeros(ck.shape, dtype=bool)  # every entry written so far with a rotated key
    for s, inp in enumerate(steps):
        out, lse = PT.run_step_gpu(wl, inp, ck_d, cv_d, rope_theta=10000.0)
        rows = PT.sample_rows(wl.steps[s], wl.n_heads, 16, seed=300 + s)
        dec = np.arange(512, 512 + 64, dtype=np.int64)
        rows = np.unique(np.concatenate([rows, dec * wl.n_heads + (s % wl.n_heads)]))
        # the oracle carries its own cache image from step to step
        ref_out, ref_lse, rk, rv = PT.oracle_step(wl, inp, rk, rv, rows=rows, rope_theta=10000.0)
        PT.compare(out, lse, ref_out, ref_lse, rows=rows, label=f"rope chunked step {s}")
        mask |= _rotated_mask(ck.shape, wl.steps[s])
    _check_caches(W.bf16_bits(ck_d.cpu()), W.bf16_bits(cv_d.cpu()), rk, rv, mask, "chunked_decode")


def test_rope_zero_is_the_plain_call():
    wl = W.random_workload(950, head_dim=128, group=4, n_kv_heads=2)
    ck, cv, (inp,) = W.make_inputs(wl)
    a_k, a_v, b_k, b_v = ck.cuda(), cv.cuda(), ck.cuda(), cv.cuda()
    o1, l1 = PT.run_step_gpu(wl, inp, a_k, a_v)
    d = {kk: vv.cuda() for kk, vv in inp.items()}
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    binding.prefill_attn_varlen_ex(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], b_k, b_v,
                                   d["cache_offsets"], o2, l2, scale=wl.scale, rope_theta=0.0)
    torch.cuda.synchronize()
    assert binding.prefill_attn_last_launch_count() == 2
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    assert torch.equal(a_k.view(torch.int16), b_k.view(torch.int16))


def test_rope_launch_count():
    wl = W.random_workload(951, head_dim=64, group=2, n_kv_heads=2)
    ck, cv, (inp,) = W.make_inputs(wl)
    PT.run_step_gpu(wl, inp, ck.cuda(), cv.cuda(), rope_theta=10000.0)
    assert binding.prefill_attn_last_launch_count() == 3
