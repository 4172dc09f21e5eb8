"""Host-side pieces of bench.py: the algorithmic bytes and FLOPs a line is
judged against, the mixed roofline, the choice of peak, and the code hash that
ties stored ncu counters to a kernel version.  No GPU needed."""
import os
import shutil

import pytest

import bench
from prefill_phase_attention_gb300 import workloads as W


def test_algorithmic_bytes_and_flops_of_the_packed_example():
    # 10 tokens of 3 prompts (5, 2, 3), 4/4 heads, d 32, empty cache:
    # q, k, v read + out written = 10 * (4 + 4 + 4 + 4) * 32 * 2 B, lse 10 * 4 * 4 B,
    # K and V rows into the cache 2 * 10 * 4 * 32 * 2 B
    wl = W.get("tiny_packed")
    assert bench.algorithmic_bytes(wl) == 10240 + 160 + 5120
    # causal pairs 5*6/2 + 2*3/2 + 3*4/2 = 24, 4 * d * H FLOPs per pair
    assert wl.flops() == 4 * 32 * 4 * 24


def test_algorithmic_bytes_count_the_cached_prefix_once():
    # one 10-token chunk over a 100-token prefix, 8/2 heads, d 64
    wl = W.Workload("chunk", 8, 2, 64, 200, [W.Step([10], [100])], [100], seed=1)
    new = 10 * (8 + 2 + 2 + 8) * 64 * 2 + 4 * 10 * 8  # q, k, v, out; lse
    kv_row = 2 * 64 * 2  # one token's K (or V) row over the KV heads, bf16
    assert bench.algorithmic_bytes(wl) == new + 2 * 10 * kv_row + 2 * 100 * kv_row
    # int8 cache: codes (1 byte) + one fp32 scale per (token, KV head)
    kv_row8 = 2 * 64 + 4 * 2
    assert bench.algorithmic_bytes(wl, kv_quant=True) == new + 2 * 10 * kv_row8 + 2 * 100 * kv_row8


def test_mixed_roofline_takes_the_larger_bound():
    wl = W.get("layer512")
    flops, byt = wl.flops(), bench.algorithmic_bytes(wl)
    r = bench.mixed_roofline(wl, 1.0, 1000.0, 5000.0)
    t_tensor = flops / 1000e12 * 1e3
    t_hbm = byt / 5000e9 * 1e3
    assert r["bound"] == ("tensor" if t_tensor >= t_hbm else "hbm")
    assert r["frac"] == pytest.approx(max(t_tensor, t_hbm) / 1.0, abs=1e-4)
    # a slow enough tensor peak makes the same step tensor-bound
    assert bench.mixed_roofline(wl, 1.0, 1e-3, 5000.0)["bound"] == "tensor"


def test_peak_for_uses_burst_below_three_seconds():
    peaks = {"bf16_tflops": 1945.7, "bf16_tflops_sustained": 1721.8}
    assert bench.peak_for(0.11, peaks) == (1945.7, "bf16_tflops")
    assert bench.peak_for(bench.SUSTAINED_AFTER_S, peaks) == (1721.8, "bf16_tflops_sustained")


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "prefill_phase_attention_gb300", "csrc")
    dst = tmp_path / "prefill_phase_attention_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in ("attn_fwd.cu", "ptx.cuh", "common.cuh"):
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_sha256()
    kern = dst / "attn_fwd.cu"
    text = kern.read_text(encoding="utf-8")
    kern.write_text("// a new comment line\n" + text.replace("// ", "//  ", 5) + "\n/* block\ncomment */\n\n",
                    encoding="utf-8")
    assert bench.kernel_sha256() == h0
    kern.write_text(text.replace("constexpr int kThreads = 384;", "constexpr int kThreads = 385;"), encoding="utf-8")
    assert bench.kernel_sha256() != h0
