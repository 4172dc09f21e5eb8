"""GPU parity of decode-heavy launches: many sequences of a few new tokens over
long cached prefixes.  Such launches (new tokens averaging under 64 per
sequence) take the kernel variant whose single-slot units split their key
tiles between both slots (even / odd) and merge the two partial results; the
paged and windowed forms included; some calls fix another schedule (one-tile
units, or two-tile units that never split).  out/lse within the stated tolerances, the
cache (or pool) bit-exact, no write outside any buffer."""
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


def _check(wl, window=0, bs=0, seed=0, schedule=0):
    step = wl.steps[0]
    assert step.total_q < 64 * step.num_seqs
    _, _, (inp,) = W.make_inputs(wl)
    table = None
    if bs:
        table, ck, cv = W.make_paged_cache(wl, bs, torch.Generator().manual_seed(seed))
    else:
        ck, cv, _ = W.make_inputs(wl)
    ck_d = PT.Guarded(ck.shape, torch.bfloat16, fill=ck)
    cv_d = PT.Guarded(cv.shape, torch.bfloat16, fill=cv)
    out, lse = PT.run_step_gpu(wl, inp, ck_d.t, cv_d.t, window=window,
                               block_table=None if table is None else table.cuda(), schedule=schedule)
    assert ck_d.guards_intact() and cv_d.guards_intact(), "write outside the cache"
    ref_out, ref_lse, ref_k, ref_v = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv), window=window,
                                                    block_table=None if table is None else table.numpy())
    PT.compare(out, lse, ref_out, ref_lse, label=f"{wl.name} window={window} bs={bs}")
    assert np.array_equal(W.bf16_bits(ck_d.t.cpu()), ref_k), "cache_k differs"
    assert np.array_equal(W.bf16_bits(cv_d.t.cpu()), ref_v), "cache_v differs"


@pytest.mark.parametrize("seed", range(36))
def test_decode_batches(seed):
    """Every head_dim x GQA group; contiguous and paged caches; some sliding
    windows (a window shorter than a tile leaves rows with no visible key in one
    of the two halves) and some non-causal calls."""
    d = [32, 64, 128][seed % 3]
    group = [1, 2, 4, 8][(seed // 3) % 4]
    causal = seed % 9 != 8
    window = [0, 0, 0, 37, 700][seed % 5] if causal else 0
    bs = [0, 0, 16, 128][seed % 4]
    wl = W.decode_workload(3100 + seed, head_dim=d, group=group, causal=causal)
    _check(wl, window=window, bs=bs, seed=seed, schedule=[0, 1, 2][seed % 3])


@pytest.mark.parametrize("prefix", [127, 128, 129, 255, 256, 383])
def test_decode_tile_counts(prefix):
    """One new token over prefixes that give 2, 3 and 4 key tiles (the two
    halves of equal and unequal length)."""
    wl = W.Workload("decode_edges", 32, 8, 128, prefix + 9, [W.Step([1, 2, 1, 1], [prefix, prefix, 5, prefix])],
                    [prefix, prefix, 5, prefix], seed=prefix)
    _check(wl)


def test_decode_mixed_with_chunk():
    """A 200-token chunk among 40 decode rows: the chunk's units keep the plain
    schedule, its last unit and the decode rows split their tiles."""
    lens = [200] + [1] * 40
    pref = [300] + [int(x) for x in np.random.default_rng(5).integers(100, 2500, size=40)]
    wl = W.Workload("decode_chunk", 32, 8, 128, max(p + n for p, n in zip(pref, lens)), [W.Step(lens, pref)],
                    pref, seed=41)
    _check(wl)
