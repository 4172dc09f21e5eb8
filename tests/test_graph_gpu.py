"""prefill_attn_varlen captured into a CUDA graph and replayed.

A serving loop captures its per-step launches once and replays them.  The
library's calls enqueue only kernels (the device scheduler reads cu_seqlens
and cache_offsets when it runs), so one captured call can be replayed for
every step of a chunked-prefill + decode workload whose sizes stay the same
while the metadata and the data in the buffers change.  Under capture the
library allocates nothing: a stream whose workspace would have to grow is
refused with PA_ERR_UNSUPPORTED.
"""
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


def test_graph_replays_every_step_of_chunked_decode():
    """One captured call replayed for the 16 launches of the chunked-prefill +
    decode mix (same num_seqs and total_q at every launch, new q/k/v and new
    cache offsets copied into the captured buffers before each replay): each
    launch matches the oracle on sampled rows (every decode row of one head
    included) and the cache the launches fill matches bit for bit."""
    wl = W.get("chunked_decode")
    ck, cv, steps = W.make_inputs(wl)
    dev = {k: v.cuda() for k, v in steps[0].items()}  # the captured buffers
    ck_d, cv_d = ck.cuda(), cv.cuda()
    out = torch.empty_like(dev["q"])
    lse = torch.empty(dev["q"].shape[0], wl.n_heads, device="cuda")
    st = torch.cuda.Stream()

    def call():
        binding.prefill_attn_varlen(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"], ck_d,
                                    cv_d, dev["cache_offsets"], out, lse, scale=wl.scale, stream=st)

    # a call outside the capture sizes the stream's workspace; it writes step 0's
    # rows into a scratch copy of the cache, which the replays then overwrite
    scratch_k, scratch_v = ck_d.clone(), cv_d.clone()
    with torch.cuda.stream(st):
        binding.prefill_attn_varlen(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"],
                                    scratch_k, scratch_v, dev["cache_offsets"], out, lse, scale=wl.scale, stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        call()
    ok, ov = W.bf16_bits(ck).copy(), W.bf16_bits(cv).copy()
    for s, inp in enumerate(steps):
        for key, t in inp.items():
            dev[key].copy_(t)  # same shapes at every step
        g.replay()
        torch.cuda.synchronize()
        assert binding.prefill_attn_device_status() == 0
        rows = PT.sample_rows(wl.steps[s], wl.n_heads, 16, seed=300 + s)
        dec = np.arange(512, 512 + 64, dtype=np.int64)
        rows = np.unique(np.concatenate([rows, dec * wl.n_heads + (s % wl.n_heads)]))
        ref_out, ref_lse, ok, ov = PT.oracle_step(wl, inp, ok, ov, rows=rows)
        PT.compare(out, lse, ref_out, ref_lse, rows=rows, label=f"graph replay, step {s}")
    assert np.array_equal(W.bf16_bits(ck_d.cpu()), ok), "cache_k differs after the replays"
    assert np.array_equal(W.bf16_bits(cv_d.cpu()), ov), "cache_v differs after the replays"


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_graph_capture_refuses_to_grow_the_workspace():
    """A stream that never ran a call has no workspace: capturing a call on it
    is refused before anything is enqueued, and the stream still works after."""
    wl = W.random_workload(970, head_dim=64, group=2, n_kv_heads=2, allow_empty=False)
    ck, cv, (inp,) = W.make_inputs(wl)
    d = {k: v.cuda() for k, v in inp.items()}
    ck_d, cv_d = ck.cuda(), cv.cuda()
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[0], wl.n_heads, device="cuda")
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(binding.PrefillAttnError) as err:
        with torch.cuda.graph(g, stream=st):
            binding.prefill_attn_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], ck_d, cv_d,
                                        d["cache_offsets"], out, lse, scale=wl.scale, stream=st)
    assert err.value.status == 2 and "graph capture" in str(err.value)
    # outside the capture the same call runs and matches the oracle
    with torch.cuda.stream(st):
        binding.prefill_attn_varlen(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], ck_d, cv_d,
                                    d["cache_offsets"], out, lse, scale=wl.scale, stream=st)
    torch.cuda.synchronize()
    ref_out, ref_lse, ref_ck, ref_cv = PT.oracle_step(wl, inp, W.bf16_bits(ck), W.bf16_bits(cv))
    PT.compare(out, lse, ref_out, ref_lse, label="after the refused capture")
    assert np.array_equal(W.bf16_bits(ck_d.cpu()), ref_ck) and np.array_equal(W.bf16_bits(cv_d.cpu()), ref_cv)
