"""The allocation-free entry point, called through the C ABI.

prefill_attn_varlen_noalloc serves callers that cannot allocate device memory
when they call in (an engine that gave nearly all HBM to its own KV-cache
arena, or a request path where an allocation's implicit synchronisation is not
allowed).  It keeps the scheduler scratch in a fixed array inside the library,
shared by every call.

Each case runs the same inputs through prefill_attn_varlen and through the
allocation-free call, and checks both against the fp64 oracle (every row for
the small cases, sampled rows for the long prompt); the two GPU results must
also agree with each other and the caches must be bit-exact.  Calls follow one
another, so every call after the first runs over the previous call's leftover
scratch contents.

This file sorts last in collection order on purpose: its subject is a
fixed-size array that lives as long as the process, and a run that stops at
the first failure (pytest -x) should have run every other GPU test before it
gets here.  It does not depend on running last: every case builds its own
inputs, and the array is cleared where it must be at every call.
"""
import ctypes

import numpy as np
import pytest
import torch

from prefill_phase_attention_gb300 import binding, build
from prefill_phase_attention_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu

# the limits stated in include/prefill_attn.h
MAX_SEQS, MAX_UNITS = 4096, 61440


@pytest.fixture(scope="module")
def lib(oracle_mod):
    build.build()
    return binding.load()


def _args(wl, dev, ck, cv, out, lse):
    T, H, d = dev["q"].shape
    return (dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), dev["cu_seqlens_q"].data_ptr(),
            dev["cu_seqlens_k"].data_ptr(), ck.data_ptr(), cv.data_ptr(), dev["cache_offsets"].data_ptr(),
            out.data_ptr(), lse.data_ptr(), len(wl.steps[0].seqlens_q), T, wl.max_cache_len, H, wl.n_kv_heads, d,
            ctypes.c_float(wl.scale), int(wl.causal), torch.cuda.current_stream().cuda_stream)


def _run(lib, fn, wl, dev, ck0, cv0):
    T = dev["q"].shape[0]
    ck, cv = ck0.cuda(), cv0.cuda()
    out = torch.empty(T, wl.n_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, wl.n_heads, dtype=torch.float32, device="cuda")
    status = fn(*_args(wl, dev, ck, cv, out, lse))
    assert status == 0, lib.prefill_attn_last_error().decode()
    torch.cuda.synchronize()
    flags = ctypes.c_int32(0)
    assert lib.prefill_attn_device_status(torch.cuda.current_stream().cuda_stream, ctypes.byref(flags)) == 0, \
        flags.value
    return out, lse, ck, cv


def _check_case(lib, wl, rows=None):
    ck, cv, (inp,) = W.make_inputs(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    ref_out, ref_lse, ref_ck, ref_cv = _run(lib, lib.prefill_attn_varlen, wl, dev, ck, cv)
    out, lse, ck2, cv2 = _run(lib, lib.prefill_attn_varlen_noalloc, wl, dev, ck, cv)
    # against the allocating entry point
    err = (out.float() - ref_out.float()).abs()
    assert err.max().item() <= PT.OUT_MAX_ABS and err.mean().item() <= PT.OUT_MEAN_ABS
    assert (lse - ref_lse).abs().max().item() <= PT.LSE_MAX_ABS
    assert torch.equal(ck2.view(torch.int16), ref_ck.view(torch.int16))
    assert torch.equal(cv2.view(torch.int16), ref_cv.view(torch.int16))
    # against the oracle
    o_out, o_lse, o_ck, o_cv = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv), rows=rows)
    PT.compare(out, lse, o_out, o_lse, rows=rows, label=f"noalloc {wl.name}")
    assert np.array_equal(W.bf16_bits(ck2.cpu()), o_ck), "cache_k differs from the oracle"
    assert np.array_equal(W.bf16_bits(cv2.cpu()), o_cv), "cache_v differs from the oracle"


def test_noalloc_matches_oracle_and_allocating_entry_point_on_calls_in_a_row(lib):
    # different batches one after the other: a chunked varlen batch with cached
    # prefixes and GQA, the packed example of the pages, a decode-heavy batch
    cases = [W.random_workload(7, head_dim=128, group=4, n_kv_heads=2, max_len=300, max_prefix=300),
             W.get("tiny_packed"),
             W.decode_workload(11, head_dim=64, group=4, n_kv_heads=2)]
    for wl in cases:
        _check_case(lib, wl)


def test_noalloc_long_prompt_schedule(lib):
    # one 4096-token MHA prompt: two-tile units on the plain kernel (the
    # long-prompt schedule), 512 units over the fixed array
    wl = W.Workload("noalloc4096", 32, 32, 128, 4096, [W.Step([4096], [0])], [0], seed=21)
    T = wl.steps[0].total_q
    assert lib.prefill_attn_auto_schedule(T, 1, 32, 32, 0, torch.cuda.get_device_properties(0).multi_processor_count) \
        == 2
    rows = PT.sample_rows(wl.steps[0], wl.n_heads, 200, seed=21)
    _check_case(lib, wl, rows=rows)


def _many_decode_rows(n_seqs, seed):
    # n_seqs one-token sequences over cached prefixes of 0..64 tokens, 15/15
    # heads, head_dim 32: the host bounds the units at 15 * (ceil(n/256) + n)
    rng = np.random.default_rng(seed)
    pref = rng.integers(0, 64, size=n_seqs, endpoint=True).tolist()
    return W.Workload(f"noalloc_decode{n_seqs}", 15, 15, 32, 66, [W.Step([1] * n_seqs, pref)], pref, seed=seed)


def test_noalloc_at_its_unit_limit_and_one_past_it(lib):
    # 4080 one-token sequences: 15 * (16 + 4080) = 61440 units, exactly the limit
    wl = _many_decode_rows(4080, seed=22)
    assert 15 * (-(-4080 // 256) + 4080) == MAX_UNITS
    _check_case(lib, wl)
    # 4081 sequences bound 61455 units: refused before any launch
    wl = _many_decode_rows(4081, seed=23)
    ck, cv, (inp,) = W.make_inputs(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    T = dev["q"].shape[0]
    ckd, cvd = ck.cuda(), cv.cuda()
    out = torch.empty(T, wl.n_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, wl.n_heads, dtype=torch.float32, device="cuda")
    assert lib.prefill_attn_varlen_noalloc(*_args(wl, dev, ckd, cvd, out, lse)) == 2
    assert "allocation-free limit" in lib.prefill_attn_last_error().decode()
    assert lib.prefill_attn_last_launch_count() == 0


def test_noalloc_reports_rejected_metadata(lib):
    # a sequence whose cu_seqlens_k disagrees with cache_offsets + seqlen_q is
    # skipped by the device scheduler; the error word of the fixed scratch says so
    wl = W.random_workload(5, head_dim=64, group=2, n_kv_heads=2, allow_empty=False)
    ck, cv, (inp,) = W.make_inputs(wl)
    dev = {k: v.cuda() for k, v in inp.items()}
    dev["cu_seqlens_k"][1:] += 1  # every sequence now claims one key too many
    T = dev["q"].shape[0]
    ckd, cvd = ck.cuda(), cv.cuda()
    out = torch.zeros(T, wl.n_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(T, wl.n_heads, dtype=torch.float32, device="cuda")
    assert lib.prefill_attn_varlen_noalloc(*_args(wl, dev, ckd, cvd, out, lse)) == 0
    flags = ctypes.c_int32(0)
    st = lib.prefill_attn_device_status(torch.cuda.current_stream().cuda_stream, ctypes.byref(flags))
    assert st == 5 and flags.value & binding.DEVERR_METADATA, (st, flags.value)
    # read and cleared: the next status read is clean
    assert lib.prefill_attn_device_status(torch.cuda.current_stream().cuda_stream, ctypes.byref(flags)) == 0


def test_noalloc_rejects_sizes_beyond_its_limit(lib):
    # 5000 sequences exceed the 4096-sequence limit: refused before any launch
    fake = 1 << 20
    st = lib.prefill_attn_varlen_noalloc(fake, fake, fake, fake, fake, fake * 2, fake * 3, fake, fake * 4, None,
                                         5000, 5000, 8, 4, 4, 64, ctypes.c_float(0.125), 1, None)
    assert st == 2 and "allocation-free limit" in lib.prefill_attn_last_error().decode()
