"""The device-side timeout path on a healthy GPU (no fault, no trap, no hang).

With the test hook pa_options.wait_timeout_test = 1 the producer thread of the
first CTA waits on a barrier that nothing completes.  The bounded wait gives up
after 2 s; that CTA records PA_DEVERR_TIMEOUT, drains its copies, frees its
tensor memory and exits while the other CTAs finish.  The host then reads the
status through prefill_attn_device_status, and the same context runs a normal
call that matches the oracle."""
import time

import numpy as np
import pytest
import torch

from prefill_phase_attention_gb300 import binding
from prefill_phase_attention_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu

PA_ERR_DEVICE_TIMEOUT = 4
PA_DEVERR_TIMEOUT = 2


@pytest.fixture(scope="module", autouse=True)
def _lib(oracle_mod):
    from prefill_phase_attention_gb300 import build
    build.build()
    binding.load()
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")


def test_wait_timeout_is_reported_and_the_context_survives():
    wl = W.get("varlen16")
    ck, cv, (inp,) = W.make_inputs(wl)
    d = {k: v.cuda() for k, v in inp.items()}
    out = torch.zeros_like(d["q"])
    lse = torch.zeros(d["q"].shape[0], wl.n_heads, device="cuda")
    assert binding.prefill_attn_device_status() == 0
    t0 = time.time()
    binding.prefill_attn_varlen_ex(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], ck.cuda(),
                                   cv.cuda(), d["cache_offsets"], out, lse, scale=wl.scale, wait_timeout_test=True)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    # the status call reads and clears the error word
    import ctypes
    flags = ctypes.c_int32(0)
    st = binding.load().prefill_attn_device_status(binding._stream_handle(None), ctypes.byref(flags))
    assert st == PA_ERR_DEVICE_TIMEOUT and flags.value & PA_DEVERR_TIMEOUT, (st, flags.value)
    assert 1.5 < elapsed < 30, elapsed  # one bounded wait (2 s), then the CTA exits
    assert binding.prefill_attn_device_status() == 0  # cleared
    # most rows were still computed by the other CTAs
    ref_out, ref_lse, _, _ = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv), want_cache=False,
                                            rows=np.arange(0, inp["q"].shape[0] * wl.n_heads, 97, dtype=np.int64))
    # and the context is healthy: the same call without the hook matches the oracle
    ck2, cv2 = ck.cuda(), cv.cuda()
    o2, l2 = PT.run_step_gpu(wl, inp, ck2, cv2)
    rows = np.arange(0, inp["q"].shape[0] * wl.n_heads, 97, dtype=np.int64)
    PT.compare(o2, l2, ref_out, ref_lse, rows=rows, label="after the timeout")
