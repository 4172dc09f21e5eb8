"""The allocation-free entry point, called through the C ABI.

prefill_attn_varlen_noalloc serves callers that cannot allocate device memory
when they call in (an engine that gave nearly all HBM to its own KV-cache
arena, or a request path where an allocation's implicit synchronisation is not
allowed).  It keeps the scheduler scratch in a fixed array inside the library.
This file checks it against prefill_attn_varlen on two calls in a row: the
second call runs over the first call's leftover scratch contents.  It sits in
a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

from prefill_phase_attention_gb300 import binding, build
from prefill_phase_attention_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu


def _args(wl, dev, ck, cv, out, lse):
    T, H, d = dev["q"].shape
    return (dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), dev["cu_seqlens_q"].data_ptr(),
            dev["cu_seqlens_k"].data_ptr(), ck.data_ptr(), cv.data_ptr(), dev["cache_offsets"].data_ptr(),
            out.data_ptr(), lse.data_ptr(), len(wl.steps[0].seqlens_q), T, wl.max_cache_len, H, wl.n_kv_heads, d,
            ctypes.c_float(wl.scale), int(wl.causal), torch.cuda.current_stream().cuda_stream)


def _run(fn, wl, inp, ck0, cv0):
    dev = {k: v.cuda() for k, v in inp.items()}
    T = inp["q"].shape[0]
    ck, cv = ck0.cuda(), cv0.cuda()
    out = torch.empty(T, wl.n_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, wl.n_heads, dtype=torch.float32, device="cuda")
    status = fn(*_args(wl, dev, ck, cv, out, lse))
    assert status == 0, binding.load().prefill_attn_last_error().decode()
    torch.cuda.synchronize()
    return out, lse, ck, cv


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    build.build()
    lib = binding.load()
    # two different batches, one after the other: a chunked varlen batch with
    # cached prefixes and GQA, then the packed example of the pages
    cases = [W.random_workload(7, head_dim=128, group=4, n_kv_heads=2, max_len=300, max_prefix=300),
             W.get("tiny_packed")]
    for wl in cases:
        ck, cv, (inp,) = W.make_inputs(wl)
        ref_out, ref_lse, ref_ck, ref_cv = _run(lib.prefill_attn_varlen, wl, inp, ck, cv)
        out, lse, ck2, cv2 = _run(lib.prefill_attn_varlen_noalloc, wl, inp, ck, cv)
        err = (out.float() - ref_out.float()).abs()
        assert err.max().item() <= PT.OUT_MAX_ABS and err.mean().item() <= PT.OUT_MEAN_ABS
        assert (lse - ref_lse).abs().max().item() <= PT.LSE_MAX_ABS
        assert torch.equal(ck2.view(torch.int16), ref_ck.view(torch.int16))
        assert torch.equal(cv2.view(torch.int16), ref_cv.view(torch.int16))


def test_noalloc_rejects_sizes_beyond_its_limit():
    lib = binding.load()
    # 5000 sequences exceed the 4096-sequence limit: refused before any launch
    fake = 1 << 20
    st = lib.prefill_attn_varlen_noalloc(fake, fake, fake, fake, fake, fake * 2, fake * 3, fake, fake * 4, None,
                                         5000, 5000, 8, 4, 4, 64, ctypes.c_float(0.125), 1, None)
    assert st == 2 and "allocation-free limit" in lib.prefill_attn_last_error().decode()
