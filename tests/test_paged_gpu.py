"""GPU parity of the paged KV cache: the CUDA path with a block pool and a
per-sequence block table (prefill_attn_varlen_ex, block_table set) against the
fp64 CPU oracle on the same pool and table.  out/lse within the stated
tolerances; the whole pool bit-exact after the call (the new tokens in the
rows the table names, every other row untouched); no write outside any buffer.

The pools carry a NaN sentinel in every row that holds no cached token, so a
key or value read from past a sequence's prefix (the rest of its last prefix
block) that reaches the result shows up as a non-finite output.
"""
import numpy as np
import pytest
import torch

from prefill_phase_attention_gb300 import binding
from prefill_phase_attention_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu

BLOCK_SIZES = [8, 16, 32, 64, 128, 256]


@pytest.fixture(scope="module", autouse=True)
def _lib(oracle_mod):
    from prefill_phase_attention_gb300 import build
    build.build()
    binding.load()
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


def _run_paged(wl, bs, seed, window=0, rows=None, table=None, pools=None, schedule=0):
    g = torch.Generator().manual_seed(seed)
    _, _, (inp,) = W.make_inputs(wl)
    if table is None:
        table, pk, pv = W.make_paged_cache(wl, bs, g)
    else:
        pk, pv = pools
    pk_d = PT.Guarded(pk.shape, torch.bfloat16, fill=pk)
    pv_d = PT.Guarded(pv.shape, torch.bfloat16, fill=pv)
    out, lse = PT.run_step_gpu(wl, inp, pk_d.t, pv_d.t, window=window, block_table=table.cuda(),
                               schedule=schedule)
    assert pk_d.guards_intact() and pv_d.guards_intact(), "write outside the pool"
    ref_out, ref_lse, ref_pk, ref_pv = PT.oracle_step(wl, inp, W.bf16_bits(pk), W.bf16_bits(pv), rows=rows,
                                                      window=window, block_table=table.numpy())
    stats = PT.compare(out, lse, ref_out, ref_lse, rows=rows, label=f"{wl.name} bs={bs}")
    assert np.array_equal(W.bf16_bits(pk_d.t.cpu()), ref_pk), "pool_k differs"
    assert np.array_equal(W.bf16_bits(pv_d.t.cpu()), ref_pv), "pool_v differs"
    return stats


@pytest.mark.parametrize("seed", range(96))
def test_paged_random_shapes(seed):
    """Every head_dim x GQA group x block size, random prefixes (partial last
    blocks), empty sequences, some sliding windows and some non-causal calls."""
    d = [32, 64, 128][seed % 3]
    group = [1, 2, 4, 8][(seed // 3) % 4]
    bs = BLOCK_SIZES[(seed // 2) % 6]
    causal = seed % 7 != 6
    window = 0
    if causal and seed % 5 == 4:
        window = int(np.random.default_rng(seed).integers(1, 400))
    wl = W.random_workload(500 + seed, head_dim=d, group=group, n_kv_heads=2, causal=causal,
                           max_prefix=[300, 700][seed % 2])
    _run_paged(wl, bs, seed, window=window, schedule=(seed // 5) % 4)


@pytest.mark.parametrize("bs", [8, 64, 512, 1024])
def test_paged_d128_block_sizes(bs):
    """head_dim 128, where a prefix tile is one TMA box per cache block staged
    by 8-row groups, at the block sizes the random cases above leave out for
    d = 128: prefixes over many blocks (or many tiles of one block) with partial
    last blocks, GQA 4, every schedule."""
    for sched in (1, 2, 3):
        wl = W.random_workload(900 + bs + sched, head_dim=128, group=4, n_kv_heads=2, max_len=300,
                               max_prefix=2500)
        _run_paged(wl, bs, bs + sched, schedule=sched)


@pytest.mark.parametrize("bs", [16, 128])
def test_paged_long_prefix_sampled(bs):
    """A 1024-token chunk over a 7000-token cached prefix (GQA 32/8, d 128), plus
    three short requests, on sampled rows."""
    wl = W.Workload("paged_long", 32, 8, 128, 8192, [W.Step([1024, 1, 37, 300], [7000, 4000, 129, 0])],
                    [7000, 4000, 129, 0], seed=31)
    rows = PT.sample_rows(wl.steps[0], wl.n_heads, 64, seed=bs)
    for sched in (1, 2):
        _run_paged(wl, bs, 40 + bs, rows=rows, schedule=sched)


def test_paged_chunked_decode_all_steps():
    """The chunked-prefill + decode mix (16 launches, GQA 32/8) on a 16-token-block
    pool: each launch reads the blocks the previous ones wrote."""
    wl = W.get("chunked_decode")
    bs = 16
    _, _, steps = W.make_inputs(wl)
    table, pk, pv = W.make_paged_cache(wl, bs, torch.Generator().manual_seed(77))
    pk_d, pv_d, table_d = pk.cuda(), pv.cuda(), table.cuda()
    ok, ov = W.bf16_bits(pk).copy(), W.bf16_bits(pv).copy()
    for s, inp in enumerate(steps):
        out, lse = PT.run_step_gpu(wl, inp, pk_d, pv_d, block_table=table_d)
        rows = PT.sample_rows(wl.steps[s], wl.n_heads, 16, seed=200 + s)
        dec = np.arange(512, 512 + 64, dtype=np.int64)
        rows = np.unique(np.concatenate([rows, dec * wl.n_heads + (s % wl.n_heads)]))
        ref_out, ref_lse, ok, ov = PT.oracle_step(wl, inp, ok, ov, rows=rows, block_table=table.numpy())
        PT.compare(out, lse, ref_out, ref_lse, rows=rows, label=f"paged chunked step {s}")
    assert np.array_equal(W.bf16_bits(pk_d.cpu()), ok)
    assert np.array_equal(W.bf16_bits(pv_d.cpu()), ov)


def test_paged_shared_prefix_blocks():
    """Two requests map the same 3 physical blocks for a common 48-token prefix
    (prefix caching); each appends into blocks of its own."""
    bs, H, Hk, d = 16, 8, 2, 128
    wl = W.Workload("shared", H, Hk, d, 128, [W.Step([70, 33], [48, 48])], [48, 48], seed=12)
    g = torch.Generator().manual_seed(3)
    table, pk, pv = W.make_paged_cache(wl, bs, g)
    table[1, :3] = table[0, :3]
    _run_paged(wl, bs, 3, table=table, pools=(pk, pv))


def test_paged_bad_block_id_is_flagged_and_skipped():
    """A sequence naming a block outside the pool is rejected on the device: its
    rows of out and every pool row stay as they were; the others are computed."""
    bs = 16
    wl = W.Workload("badblk", 8, 2, 64, 256, [W.Step([40, 50], [30, 20])], [30, 20], seed=13)
    g = torch.Generator().manual_seed(4)
    table, pk, pv = W.make_paged_cache(wl, bs, g)
    _, _, (inp,) = W.make_inputs(wl)
    bad = table.clone()
    bad[0, 3] = pk.shape[0] + 5  # position 48..63 of sequence 0, inside [0, P + n)
    dev = {k: v.cuda() for k, v in inp.items()}
    pk_d, pv_d = pk.cuda(), pv.cuda()
    out = torch.full((90, 8, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((90, 8), -3.0, dtype=torch.float32, device="cuda")
    binding.prefill_attn_varlen_ex(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"],
                                   pk_d, pv_d, dev["cache_offsets"], out, lse, scale=wl.scale,
                                   block_table=bad.cuda())
    torch.cuda.synchronize()
    flags = binding.prefill_attn_device_status()
    assert flags & 1, "PA_DEVERR_METADATA expected"
    assert bool((out[:40] == 7.0).all()) and bool((lse[:40] == -3.0).all())
    ref_out, ref_lse, ref_pk, ref_pv = PT.oracle_step(wl, inp, W.bf16_bits(pk), W.bf16_bits(pv),
                                                      block_table=table.numpy())
    PT.compare(out[40:], lse[40:], ref_out[40:], ref_lse[40:], label="good sequence")
    # pool: sequence 1's new rows written, sequence 0's not
    got_k = W.bf16_bits(pk_d.cpu())
    b0_rows = [(int(table[0, p // bs]), p % bs) for p in range(30, 70)]
    for blk, r in b0_rows:
        assert np.array_equal(got_k[blk, :, r], W.bf16_bits(pk)[blk, :, r])
    for p in range(20, 70):
        blk, r = int(table[1, p // bs]), p % bs
        assert np.array_equal(got_k[blk, :, r], ref_pk[blk, :, r])


def test_paged_equals_contiguous_within_tolerance():
    """The same logical cache, contiguous and paged, gives results within the
    parity tolerance of each other (the tile boundaries differ, so not bitwise)."""
    wl = W.random_workload(900, head_dim=128, group=4, n_kv_heads=2, max_prefix=500, allow_empty=False)
    ck, cv, (inp,) = W.make_inputs(wl)
    bs = 32
    maxb = -(-wl.max_cache_len // bs)
    B = wl.num_seqs
    rng = np.random.default_rng(1)
    table = torch.from_numpy(rng.permutation(B * maxb).reshape(B, maxb).astype(np.int32))
    pk = torch.full((B * maxb, wl.n_kv_heads, bs, wl.head_dim), float("nan"), dtype=torch.bfloat16)
    pv = pk.clone()
    for b in range(B):
        for L in range(maxb):
            lo, hi = L * bs, min((L + 1) * bs, wl.max_cache_len)
            pk[int(table[b, L]), :, :hi - lo] = ck[b, :, lo:hi]
            pv[int(table[b, L]), :, :hi - lo] = cv[b, :, lo:hi]
    o1, l1 = PT.run_step_gpu(wl, inp, ck.cuda(), cv.cuda())
    o2, l2 = PT.run_step_gpu(wl, inp, pk.cuda(), pv.cuda(), block_table=table.cuda())
    PT.compare(o2, l2, o1.double().cpu().numpy(), l1.double().cpu().numpy(), label="paged vs contiguous")
