"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle on the
same seeded inputs.  out/lse within the stated tolerances, KV cache bit-exact,
no write outside any output buffer."""
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


def _run_single_step(wl, rows=None, window=0, schedule=0):
    ck, cv, (inp,) = W.make_inputs(wl)
    ck_d = PT.Guarded(ck.shape, torch.bfloat16, fill=ck)
    cv_d = PT.Guarded(cv.shape, torch.bfloat16, fill=cv)
    out, lse = PT.run_step_gpu(wl, inp, ck_d.t, cv_d.t, window=window, schedule=schedule)
    assert ck_d.guards_intact() and cv_d.guards_intact(), "write outside the cache"
    ref_out, ref_lse, ref_ck, ref_cv = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv), rows=rows,
                                                      window=window)
    stats = PT.compare(out, lse, ref_out, ref_lse, rows=rows, label=wl.name)
    assert np.array_equal(W.bf16_bits(ck_d.t.cpu()), ref_ck), "cache_k differs"
    assert np.array_equal(W.bf16_bits(cv_d.t.cpu()), ref_cv), "cache_v differs"
    return stats


@pytest.mark.parametrize("sched", [0, 1, 2, 3])
@pytest.mark.parametrize("name", ["tiny_packed", "layer512", "varlen16", "chunk512", "decode64"])
def test_named_workload_full(name, sched):
    """Every schedule (one-tile units splitting their KV tiles between the two
    slots; two-tile units; two-tile units with single-tile ones split) and
    the library's own choice."""
    _run_single_step(W.get(name), schedule=sched)


def test_long32k_sampled():
    """The headline configuration against the oracle on 6000+ of its 1,048,576
    (token, head) rows: every head of the last 128-token Q tile (the longest
    rows), the first and last row of every 128-row Q tile (the diagonal and
    the tile edges) with two heads each, and 1500 random rows; the cache in full."""
    wl = W.get("long32k")
    H, T = wl.n_heads, wl.steps[0].total_q
    rng = np.random.default_rng(5)
    last = np.arange(T - 128, T, dtype=np.int64)[:, None] * H + np.arange(H)[None, :]
    edges = np.concatenate([np.arange(0, T, 128), np.arange(127, T, 128)]).astype(np.int64)
    edge_rows = np.concatenate([edges * H + rng.integers(0, H, edges.size), edges * H + rng.integers(0, H, edges.size)])
    rand = rng.integers(0, T * H, size=1500)
    rows = np.unique(np.concatenate([last.ravel(), edge_rows, rand]))
    assert rows.size >= 6000
    _run_single_step(wl, rows=rows)


def test_chunked_decode_all_steps():
    """16 launches: each packs one 512-token chunk (prefix from the cache written by
    the previous launches) with 64 one-token decode rows, GQA 32/8."""
    wl = W.get("chunked_decode")
    ck, cv, steps = W.make_inputs(wl)
    ck_d, cv_d = ck.cuda(), cv.cuda()
    ok, ov = W.bf16_bits(ck).copy(), W.bf16_bits(cv).copy()
    for s, inp in enumerate(steps):
        out, lse = PT.run_step_gpu(wl, inp, ck_d, cv_d)
        st = wl.steps[s]
        rows = PT.sample_rows(st, wl.n_heads, 24, seed=100 + s)
        # every decode row of two heads as well
        dec = np.arange(512, 512 + 64, dtype=np.int64)
        rows = np.unique(np.concatenate([rows, dec * wl.n_heads + (s % wl.n_heads), dec * wl.n_heads + 31]))
        ref_out, ref_lse, ok, ov = PT.oracle_step(wl, inp, ok, ov, rows=rows)
        PT.compare(out, lse, ref_out, ref_lse, rows=rows, label=f"chunked step {s}")
    assert np.array_equal(W.bf16_bits(ck_d.cpu()), ok)
    assert np.array_equal(W.bf16_bits(cv_d.cpu()), ov)


@pytest.mark.parametrize("sched", [1, 2, 3])
@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_random_shapes(seed, d, group, sched):
    wl = W.random_workload(seed * 31 + d + group, head_dim=d, group=group, n_kv_heads=2,
                           causal=(seed % 4 != 3))
    _run_single_step(wl, schedule=sched)


def test_length_one_is_bit_exact():
    """One visible key: weight 1, so out must be exactly bf16(v) for every head."""
    wl = W.Workload("len1", 8, 2, 128, 4, [W.Step([1, 1, 1, 1], [0, 0, 0, 0])], [0, 0, 0, 0], seed=9)
    ck, cv, (inp,) = W.make_inputs(wl)
    out, _ = PT.run_step_gpu(wl, inp, ck.cuda(), cv.cuda())
    exp = inp["v"].repeat_interleave(4, dim=1)
    assert torch.equal(out.cpu().view(torch.int16), exp.view(torch.int16))


def test_chunked_equals_one_shot_on_gpu():
    H, Hk, d, n, c = 8, 2, 128, 1024, 256
    one = W.Workload("one", H, Hk, d, n, [W.Step([n], [0])], [0], seed=21)
    ck, cv, (inp,) = W.make_inputs(one)
    ck1, cv1 = ck.cuda(), cv.cuda()
    out1, lse1 = PT.run_step_gpu(one, inp, ck1, cv1)
    ck2, cv2 = ck.cuda(), cv.cuda()
    for s in range(n // c):
        sl = slice(s * c, (s + 1) * c)
        sub = dict(q=inp["q"][sl], k=inp["k"][sl], v=inp["v"][sl],
                   cu_seqlens_q=torch.tensor([0, c], dtype=torch.int32),
                   cu_seqlens_k=torch.tensor([0, s * c + c], dtype=torch.int32),
                   cache_offsets=torch.tensor([s * c], dtype=torch.int32))
        o, l = PT.run_step_gpu(one, sub, ck2, cv2)
        assert (o.float() - out1[sl].float()).abs().max().item() <= PT.OUT_MAX_ABS
        assert (l - lse1[sl]).abs().max().item() <= PT.LSE_MAX_ABS
    assert torch.equal(ck1.view(torch.int16), ck2.view(torch.int16))
    assert torch.equal(cv1.view(torch.int16), cv2.view(torch.int16))


def test_inconsistent_device_metadata_is_flagged_and_skipped():
    wl = W.get("tiny_packed")
    ck, cv, (inp,) = W.make_inputs(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    bad_k = dev["cu_seqlens_k"].clone()
    bad_k[2] += 1  # sequence 1 claims one key too many
    out = torch.zeros(10, 4, 32, dtype=torch.bfloat16, device="cuda")
    ck_d, cv_d = ck.cuda(), cv.cuda()
    binding.prefill_attn_varlen(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], bad_k, ck_d, cv_d,
                                dev["cache_offsets"], out, None, scale=wl.scale)
    flags = binding.prefill_attn_device_status()
    assert flags & binding.DEVERR_METADATA
    assert binding.prefill_attn_device_status() == 0  # read clears it
    # sequence 1 wrote nothing, sequences 0 and 2 were computed
    assert (out[5:7] == 0).all() and (out[0:5] != 0).any()
    assert (ck_d[1].view(torch.int16) == W.CACHE_SENTINEL_BITS).all()
    with pytest.raises(binding.PrefillAttnError, match="cu_seqlens_k"):
        binding.prefill_attn_varlen_validate(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], bad_k, ck_d,
                                             cv_d, dev["cache_offsets"], out, None, scale=wl.scale)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("d,group", [(32, 1), (64, 2), (128, 4), (128, 8)])
@pytest.mark.parametrize("window", [1, 17, 128, 200, 1000])
def test_sliding_window_random_shapes(seed, d, group, window):
    wl = W.random_workload(seed * 7 + d + group + window, head_dim=d, group=group, n_kv_heads=2)
    _run_single_step(wl, window=window, schedule=1 + seed % 3)


def test_sliding_window_long_prompt_sampled():
    """8192-token prompt with the page's window of 4096 tokens (sampled rows)."""
    wl = W.get("long8k")
    rows = PT.sample_rows(wl.steps[0], wl.n_heads, 96, seed=8)
    _run_single_step(wl, rows=rows, window=4096)


def test_sliding_window_chunk_over_cached_prefix():
    """Chunks over a long cached prefix with a window shorter than the prefix."""
    wl = W.Workload("winchunk", 16, 4, 128, 3000, [W.Step([300, 1, 700], [2000, 1500, 600])], [2000, 1500, 600],
                    seed=31)
    for window in (64, 333, 1024):
        for sched in (1, 2, 3):
            _run_single_step(wl, window=window, schedule=sched)


def test_many_sequences_sampled():
    """5000 sequences in one launch (more than one 1024-sequence pass of the
    scheduler): mostly one-token decode rows over cached contexts, some short
    prompts, some empty; GQA 16/2, d 64; sampled rows and the whole cache."""
    rng = np.random.default_rng(77)
    B = 5000
    lens = rng.choice([0, 1, 1, 1, 3, 17, 130], size=B).tolist()
    pref = rng.integers(0, 300, size=B).tolist()
    cap = max(p + n for p, n in zip(pref, lens)) + 1
    wl = W.Workload("many", 16, 2, 64, cap, [W.Step(lens, pref)], pref, seed=78)
    rows = PT.sample_rows(wl.steps[0], wl.n_heads, 2, seed=79)
    _run_single_step(wl, rows=rows)


@pytest.mark.parametrize("B", [1024, 1025])
def test_scheduler_table_boundary(B):
    """1024 sequences (the device scheduler keeps its per-sequence tables in
    shared memory) and 1025 (they go through the workspace): decode rows, short
    prompts and empty sequences over cached prefixes, every row checked under
    every schedule."""
    rng = np.random.default_rng(B)
    lens = rng.choice([0, 1, 1, 2, 9, 40], size=B).tolist()
    pref = rng.integers(0, 200, size=B).tolist()
    cap = max(p + n for p, n in zip(pref, lens)) + 1
    wl = W.Workload(f"seqs{B}", 8, 2, 64, cap, [W.Step(lens, pref)], pref, seed=B)
    for sched in (0, 1, 2, 3):
        _run_single_step(wl, schedule=sched)


def test_single_token_total():
    """total_q = 1: one decode row, nothing else."""
    wl = W.Workload("one_tok", 8, 2, 64, 70, [W.Step([1], [64])], [64], seed=80)
    _run_single_step(wl)


def test_query_block_edges():
    """Prompts whose lengths sit on and next to the 128-row tile and the 256-row
    work-unit edges, over prefixes on and next to tile edges."""
    lens = [127, 128, 129, 255, 256, 257]
    pref = [0, 127, 128, 129, 255, 256]
    wl = W.Workload("edges", 16, 4, 128, 600, [W.Step(lens, pref)], pref, seed=81)
    for sched in (1, 2, 3):
        _run_single_step(wl, schedule=sched)


def test_prompt_16_chunks_equals_one_launch_on_gpu():
    """The chunked workload's 8192-token prompt (GQA 32/8, d 128) as 16 launches of
    512 tokens over the cache they fill == one 8192-token launch: outputs within
    the tolerances of each other (and of the oracle on sampled rows), caches
    bit-exact."""
    H, Hk, d, n, c = 32, 8, 128, 8192, 512
    one = W.Workload("prompt8k", H, Hk, d, n, [W.Step([n], [0])], [0], seed=4)
    ck, cv, (inp,) = W.make_inputs(one)
    ck1, cv1 = ck.cuda(), cv.cuda()
    out1, lse1 = PT.run_step_gpu(one, inp, ck1, cv1)
    ck2, cv2 = ck.cuda(), cv.cuda()
    outs, lses = [], []
    for s in range(n // c):
        sl = slice(s * c, (s + 1) * c)
        sub = dict(q=inp["q"][sl], k=inp["k"][sl], v=inp["v"][sl],
                   cu_seqlens_q=torch.tensor([0, c], dtype=torch.int32),
                   cu_seqlens_k=torch.tensor([0, s * c + c], dtype=torch.int32),
                   cache_offsets=torch.tensor([s * c], dtype=torch.int32))
        o, l = PT.run_step_gpu(one, sub, ck2, cv2)
        outs.append(o.clone())
        lses.append(l.clone())
    out2, lse2 = torch.cat(outs), torch.cat(lses)
    PT.compare(out2, lse2, out1.double().cpu().numpy(), lse1.double().cpu().numpy(), label="16 chunks vs one")
    assert torch.equal(ck1.view(torch.int16), ck2.view(torch.int16))
    assert torch.equal(cv1.view(torch.int16), cv2.view(torch.int16))
    rows = PT.sample_rows(one.steps[0], H, 64, seed=11)
    ref_out, ref_lse, _, _ = PT.oracle_step(one, inp, W.bf16_bits(ck), W.bf16_bits(cv), rows=rows, want_cache=False)
    PT.compare(out2, lse2, ref_out, ref_lse, rows=rows, label="16 chunks vs oracle")


def test_two_streams_run_concurrently():
    """Calls on two streams at once keep separate workspaces: both match the oracle."""
    wa = W.random_workload(960, head_dim=128, group=4, n_kv_heads=2, max_prefix=400, allow_empty=False)
    wb = W.random_workload(961, head_dim=64, group=2, n_kv_heads=2, max_prefix=400, allow_empty=False)
    runs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for wl, st in zip((wa, wb), streams):
        ck, cv, (inp,) = W.make_inputs(wl)
        d = {k: v.cuda() for k, v in inp.items()}
        ck_d, cv_d = ck.cuda(), cv.cuda()
        out = torch.empty_like(d["q"])
        lse = torch.empty(d["q"].shape[0], wl.n_heads, device="cuda")
        runs.append((wl, inp, ck, cv, d, ck_d, cv_d, out, lse, st))
    torch.cuda.synchronize()
    for _ in range(5):  # several rounds so that the two streams' kernels overlap
        for wl, inp, ck, cv, d, ck_d, cv_d, out, lse, st in runs:
            with torch.cuda.stream(st):
                binding.prefill_attn_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], ck_d,
                                            cv_d, d["cache_offsets"], out, lse, scale=wl.scale, stream=st)
    torch.cuda.synchronize()
    for wl, inp, ck, cv, d, ck_d, cv_d, out, lse, st in runs:
        assert binding.prefill_attn_device_status(st) == 0
        ref_out, ref_lse, ref_ck, ref_cv = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv))
        PT.compare(out, lse, ref_out, ref_lse, label=f"{wl.name} on its own stream")
        assert np.array_equal(W.bf16_bits(ck_d.cpu()), ref_ck) and np.array_equal(W.bf16_bits(cv_d.cpu()), ref_cv)


@pytest.mark.parametrize("sched", [1, 2])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_out_16_byte_aligned(d, sched):
    """out at a 16-byte (not 32-byte) aligned address, the API's minimum: the
    epilogue then stores 16-byte pieces (in both softmax layouts: the plain
    schedule's and the splitting one's); results and guard bands as usual."""
    wl = W.random_workload(960 + d, head_dim=d, group=2, n_kv_heads=2, allow_empty=False)
    ck, cv, (inp,) = W.make_inputs(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    T = inp["q"].shape[0]
    n = T * wl.n_heads * d
    buf = torch.full((n + 64,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[8:8 + n].view(T, wl.n_heads, d)  # 16 bytes past a 256-byte aligned base
    assert out.data_ptr() % 32 == 16
    lse = torch.empty(T, wl.n_heads, device="cuda")
    ck_d, cv_d = ck.cuda(), cv.cuda()
    binding.prefill_attn_varlen_ex(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"], ck_d, cv_d,
                                   dev["cache_offsets"], out, lse, scale=wl.scale, causal=wl.causal, schedule=sched)
    torch.cuda.synchronize()
    assert binding.prefill_attn_device_status() == 0
    assert binding.prefill_attn_last_schedule() == sched
    assert bool((buf[:8] == 7.0).all()) and bool((buf[8 + n:] == 7.0).all()), "write outside out"
    ref_out, ref_lse, _, _ = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv), want_cache=False)
    PT.compare(out, lse, ref_out, ref_lse, label=f"out +16 B d={d} schedule {sched}")
