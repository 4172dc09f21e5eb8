"""GPU parity of the int8 KV cache (pa_options.kv_quant = 1): the CUDA path
against the fp64 CPU oracle on the same codes and scales.  out/lse within the
stated tolerances; the codes and scales written for the new tokens bit-exact
(both sides decide them in fp32: scale = max|x| / 127, code = nearest-even of
x / scale), every other cache row untouched.  With RoPE on, the rotated key may
differ by one bf16 ulp before quantisation, so its rows are compared as
dequantised values within one quantisation step.

Rows of the cache that hold no cached token carry a NaN scale: a read of one
that reaches the result shows up as a non-finite output."""
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


def _new_rows(shape, steps):
    m = np.zeros(shape[:-1], dtype=bool)
    for step in steps:
        for b, (n, P) in enumerate(zip(step.seqlens_q, step.cache_offsets)):
            m[b, :, P:P + n] = True
    return m


def _check_cache(got, ref, new_rows, rope, label):
    (gk, gsk, gv, gsv), (rk, rsk, rv, rsv) = got, ref
    assert np.array_equal(gv, rv) and np.array_equal(gsv.view(np.int32), rsv.view(np.int32)), f"{label}: V cache"
    old = ~new_rows
    assert np.array_equal(gk[old], rk[old]) and np.array_equal(gsk[old].view(np.int32), rsk[old].view(np.int32)), \
        f"{label}: K cache rows outside the new tokens changed"
    if not rope:
        assert np.array_equal(gk, rk) and np.array_equal(gsk.view(np.int32), rsk.view(np.int32)), f"{label}: K cache"
        return
    gdq = gk[new_rows].astype(np.float64) * gsk[new_rows][:, None]
    rdq = rk[new_rows].astype(np.float64) * rsk[new_rows][:, None]
    step = np.maximum(gsk[new_rows], rsk[new_rows])[:, None]
    assert (np.abs(gdq - rdq) <= step * 1.01 + 1e-6).all(), f"{label}: rotated K rows differ by more than a step"


def _run(wl, window=0, rope=0.0, rows=None, seed=0):
    _, _, (inp,) = W.make_inputs(wl)
    ck, sk, cv, sv = W.make_q8_cache(wl, torch.Generator().manual_seed(seed))
    d = [PT.Guarded(t.shape, t.dtype, fill=t) if t.dtype == torch.float32 else None for t in (sk, sv)]
    ck_d, cv_d = ck.cuda(), cv.cuda()
    sk_d, sv_d = d[0], d[1]
    out, lse = PT.run_step_gpu_q8(wl, inp, ck_d, sk_d.t, cv_d, sv_d.t, window=window, rope_theta=rope)
    assert sk_d.guards_intact() and sv_d.guards_intact(), "write outside the scales"
    ro, rl, (rk, rsk), (rv, rsv) = PT.oracle_step_q8(wl, inp, ck.numpy(), sk.numpy(), cv.numpy(), sv.numpy(),
                                                     rows=rows, window=window, rope_theta=rope)
    PT.compare(out, lse, ro, rl, rows=rows, label=f"{wl.name} int8")
    got = (ck_d.cpu().numpy(), sk_d.t.cpu().numpy(), cv_d.cpu().numpy(), sv_d.t.cpu().numpy())
    _check_cache(got, (rk, rsk, rv, rsv), _new_rows(ck.shape, wl.steps), rope, wl.name)


@pytest.mark.parametrize("seed", range(48))
def test_quant_random_shapes(seed):
    """Every head_dim x GQA group over int8 prefixes; some with a window, RoPE,
    or no causal mask."""
    d = [32, 64, 128][seed % 3]
    group = [1, 2, 4, 8][(seed // 3) % 4]
    causal = seed % 7 != 6
    window = 120 if (causal and seed % 5 == 1) else 0
    rope = 10000.0 if seed % 4 == 3 else 0.0
    wl = W.random_workload(1100 + seed, head_dim=d, group=group, n_kv_heads=2, causal=causal, max_prefix=600)
    _run(wl, window=window, rope=rope, seed=seed)


def test_quant_long_prefix_sampled():
    """A 1024-token chunk over a 7000-token int8 prefix plus three short requests
    (GQA 32/8, d 128), on sampled rows."""
    wl = W.Workload("q8_long", 32, 8, 128, 8192, [W.Step([1024, 1, 37, 300], [7000, 4000, 129, 0])],
                    [7000, 4000, 129, 0], seed=41)
    rows = PT.sample_rows(wl.steps[0], wl.n_heads, 64, seed=9)
    _run(wl, rows=rows, seed=41)


def test_quant_chunked_decode_all_steps():
    """The chunked-prefill + decode mix (16 launches) over an int8 cache: each
    launch reads the codes the earlier ones wrote."""
    wl = W.get("chunked_decode")
    _, _, steps = W.make_inputs(wl)
    ck, sk, cv, sv = W.make_q8_cache(wl, torch.Generator().manual_seed(5))
    ck_d, sk_d, cv_d, sv_d = ck.cuda(), sk.cuda(), cv.cuda(), sv.cuda()
    rk, rsk, rv, rsv = ck.numpy(), sk.numpy(), cv.numpy(), sv.numpy()
    for s, inp in enumerate(steps):
        out, lse = PT.run_step_gpu_q8(wl, inp, ck_d, sk_d, cv_d, sv_d)
        rows = PT.sample_rows(wl.steps[s], wl.n_heads, 16, seed=400 + s)
        dec = np.arange(512, 512 + 64, dtype=np.int64)
        rows = np.unique(np.concatenate([rows, dec * wl.n_heads + (s % wl.n_heads)]))
        ro, rl, (rk, rsk), (rv, rsv) = PT.oracle_step_q8(wl, inp, rk, rsk, rv, rsv, rows=rows)
        PT.compare(out, lse, ro, rl, rows=rows, label=f"int8 chunked step {s}")
    got = (ck_d.cpu().numpy(), sk_d.cpu().numpy(), cv_d.cpu().numpy(), sv_d.cpu().numpy())
    _check_cache(got, (rk, rsk, rv, rsv), _new_rows(ck.shape, wl.steps), False, "int8 chunked_decode")


def test_quant_codes_of_special_rows():
    """Rows with max |x| = 127 (scale 1: codes are x rounded half to even), rows
    scaled by 1/8, all-zero rows: bit-exact against the oracle and the closed form."""
    d = 64
    wl = W.Workload("q8rows", 4, 2, d, 8, [W.Step([3], [0])], [0], seed=43)
    _, _, (inp,) = W.make_inputs(wl)
    vals = torch.zeros(d)
    vals[:7] = torch.tensor([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -127.0])
    k = torch.zeros(3, 2, d)
    k[0, 0] = vals
    k[1, 1] = vals / 8
    inp = dict(inp, k=k.to(torch.bfloat16), v=(k / 4).to(torch.bfloat16))
    ck, sk, cv, sv = (t.cuda() for t in W.make_q8_cache(wl, torch.Generator().manual_seed(0), sentinel=False))
    PT.run_step_gpu_q8(wl, inp, ck, sk, cv, sv)
    exp = np.zeros(d, np.int8)
    exp[:7] = [127, 2, 4, -2, 0, 2, -127]
    gk, gs = ck.cpu().numpy(), sk.cpu().numpy()
    assert np.array_equal(gk[0, 0, 0], exp) and gs[0, 0, 0] == 1.0
    assert np.array_equal(gk[0, 1, 1], exp) and gs[0, 1, 1] == np.float32(1 / 8)
    assert not gk[0, 1, 0].any() and gs[0, 1, 0] == 0.0 and not gk[0, :, 2].any()
    assert np.array_equal(cv.cpu().numpy()[0, 0, 0], exp) and sv.cpu().numpy()[0, 0, 0] == np.float32(0.25)



def _paged_new_rows(shape, step, table, bs):
    m = np.zeros(shape[:-1], dtype=bool)
    for b, (n, P) in enumerate(zip(step.seqlens_q, step.cache_offsets)):
        for pos in range(P, P + n):
            m[int(table[b, pos // bs]), :, pos % bs] = True
    return m


@pytest.mark.parametrize("seed", range(24))
def test_quant_paged_random_shapes(seed):
    """The int8 cache in block pools (block sizes 8 .. 256, random placement):
    partial last prefix blocks hold NaN-scaled rows that must expand to zeros."""
    d = [32, 64, 128][seed % 3]
    group = [1, 2, 4, 8][(seed // 3) % 4]
    bs = [8, 16, 32, 64, 128, 256][(seed // 2) % 6]
    window = 90 if seed % 5 == 3 else 0
    rope = 10000.0 if seed % 6 == 5 else 0.0
    wl = W.random_workload(1300 + seed, head_dim=d, group=group, n_kv_heads=2, max_prefix=500)
    _, _, (inp,) = W.make_inputs(wl)
    table, ck, sk, cv, sv = W.make_paged_q8_cache(wl, bs, torch.Generator().manual_seed(seed))
    sk_d = PT.Guarded(sk.shape, torch.float32, fill=sk)
    sv_d = PT.Guarded(sv.shape, torch.float32, fill=sv)
    ck_d, cv_d = ck.cuda(), cv.cuda()
    out, lse = PT.run_step_gpu_q8(wl, inp, ck_d, sk_d.t, cv_d, sv_d.t, window=window, rope_theta=rope,
                                  block_table=table.cuda())
    assert sk_d.guards_intact() and sv_d.guards_intact(), "write outside the scale pools"
    ro, rl, (rk, rsk), (rv, rsv) = PT.oracle_step_q8(wl, inp, ck.numpy(), sk.numpy(), cv.numpy(), sv.numpy(),
                                                     window=window, rope_theta=rope, block_table=table.numpy())
    PT.compare(out, lse, ro, rl, label=f"{wl.name} int8 paged bs={bs}")
    got = (ck_d.cpu().numpy(), sk_d.t.cpu().numpy(), cv_d.cpu().numpy(), sv_d.t.cpu().numpy())
    _check_cache(got, (rk, rsk, rv, rsv), _paged_new_rows(ck.shape, wl.steps[0], table, bs), bool(rope), wl.name)


def test_quant_paged_chunked_decode_sampled():
    """chunked_decode over 16-token int8 blocks, 16 launches, sampled rows."""
    wl = W.get("chunked_decode")
    _, _, steps = W.make_inputs(wl)
    bs = 16
    table, ck, sk, cv, sv = W.make_paged_q8_cache(wl, bs, torch.Generator().manual_seed(6))
    ck_d, sk_d, cv_d, sv_d, table_d = ck.cuda(), sk.cuda(), cv.cuda(), sv.cuda(), table.cuda()
    rk, rsk, rv, rsv = ck.numpy(), sk.numpy(), cv.numpy(), sv.numpy()
    for s, inp in enumerate(steps):
        out, lse = PT.run_step_gpu_q8(wl, inp, ck_d, sk_d, cv_d, sv_d, block_table=table_d)
        rows = PT.sample_rows(wl.steps[s], wl.n_heads, 12, seed=500 + s)
        ro, rl, (rk, rsk), (rv, rsv) = PT.oracle_step_q8(wl, inp, rk, rsk, rv, rsv, rows=rows,
                                                         block_table=table.numpy())
        PT.compare(out, lse, ro, rl, rows=rows, label=f"int8 paged chunked step {s}")
    got = (ck_d.cpu().numpy(), sk_d.cpu().numpy(), cv_d.cpu().numpy(), sv_d.cpu().numpy())
    new = np.zeros(ck.shape[:-1], dtype=bool)
    for st in wl.steps:
        new |= _paged_new_rows(ck.shape, st, table, bs)
    _check_cache(got, (rk, rsk, rv, rsv), new, False, "int8 paged chunked_decode")
