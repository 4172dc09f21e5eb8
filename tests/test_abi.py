"""The C ABI: the library loads, exports every declared entry point, and
rejects host-checkable argument errors before touching a GPU."""
import ctypes
import os
import re

import pytest

from prefill_phase_attention_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(prefill_attn_\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "prefill_attn_varlen" in names and len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(binding.SIGNATURES) >= set(names), "binding lacks a declared entry point"


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert lib.prefill_attn_status_string(code).decode() == name


def _call(lib, **kw):
    a = dict(q=16, k=32, v=48, cu_q=64, cu_k=80, ck=96, cv=112, off=128, out=144, lse=None,
             num_seqs=1, total_q=4, cap=8, H=4, Hk=2, d=64, scale=0.125, causal=1, stream=None)
    a.update(kw)
    return lib.prefill_attn_varlen(a["q"], a["k"], a["v"], a["cu_q"], a["cu_k"], a["ck"], a["cv"], a["off"],
                                   a["out"], a["lse"], a["num_seqs"], a["total_q"], a["cap"], a["H"], a["Hk"],
                                   a["d"], a["scale"], a["causal"], a["stream"])


@pytest.mark.parametrize("kw,status,msg", [
    (dict(d=48), 2, "head_dim"),
    (dict(H=6, Hk=4), 1, "multiple"),
    (dict(H=258, Hk=1), 2, "exceeds"),
    (dict(scale=0.0), 1, "scale"),
    (dict(scale=float("inf")), 1, "scale"),
    (dict(causal=2), 1, "causal"),
    (dict(num_seqs=-1), 1, "num_seqs"),
    (dict(cap=0), 1, "max_cache_len"),
    (dict(q=None), 1, "q is NULL"),
    (dict(k=33), 1, "aligned"),
    (dict(out=16), 1, "alias"),
    (dict(ck=32), 1, "alias"),
])
def test_host_checks_reject_before_launch(lib, kw, status, msg):
    assert _call(lib, **kw) == status
    assert msg in lib.prefill_attn_last_error().decode()


def test_empty_batch_is_a_no_op(lib):
    assert _call(lib, num_seqs=0, q=None, k=None, v=None) == 0
    assert lib.prefill_attn_last_launch_count() == 0
    assert _call(lib, total_q=0) == 0


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    t = torch.zeros(4, 2, 32, dtype=torch.bfloat16)
    i = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError):
        binding.prefill_attn_varlen(t, t, t, i, i, t[None], t[None], i[:1], t)


def _call_ex(lib, window=0, causal=1, struct_size=None, block_table=None, block_size=0, max_blocks=0,
             num_blocks=0, reserved=0, rope_theta=0.0, reserved2=0, kv_quant=0, reserved3=0, sk=None, sv=None,
             wait_timeout_test=0, schedule=0):
    opts = binding.PaOptions(ctypes.sizeof(binding.PaOptions) if struct_size is None else struct_size, window,
                             block_table, block_size, max_blocks, num_blocks, reserved, rope_theta, reserved2,
                             kv_quant, reserved3, sk, sv, wait_timeout_test, schedule)
    return lib.prefill_attn_varlen_ex(16, 32, 48, 64, 80, 96, 112, 128, 144, None, 1, 4, 8, 4, 2, 64,
                                      0.125, causal, ctypes.byref(opts), None)


_PAGED = dict(block_table=256, block_size=8, max_blocks=1, num_blocks=4)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(window=-1), 1, "window"),
    (dict(window=8, causal=0), 1, "causal"),
    (dict(struct_size=2), 1, "struct_size"),
    (dict(reserved=1), 1, "reserved"),
    (dict(_PAGED, struct_size=16), 1, "paged"),  # covers the pointer but not the sizes
    (dict(_PAGED, block_size=12), 2, "power of two"),
    (dict(_PAGED, block_size=4, max_blocks=2), 2, "power of two"),
    (dict(_PAGED, block_size=16), 1, "max_cache_len"),
    (dict(_PAGED, num_blocks=0), 1, "num_blocks"),
    (dict(_PAGED, block_table=258), 1, "aligned"),
    (dict(_PAGED, num_blocks=1 << 30), 2, "num_blocks"),
    (dict(rope_theta=-1.0), 1, "rope_theta"),
    (dict(rope_theta=float("nan")), 1, "rope_theta"),
    (dict(rope_theta=float("inf")), 1, "rope_theta"),
    (dict(reserved2=3), 1, "reserved2"),
    (dict(kv_quant=2, sk=512, sv=1024), 1, "kv_quant"),
    (dict(kv_quant=1), 1, "cache_k_scale"),
    (dict(kv_quant=1, sk=514, sv=1024), 1, "aligned"),
    (dict(kv_quant=1, sk=512, sv=1024, reserved3=1), 1, "reserved3"),
    (dict(kv_quant=1, sk=512, sv=1024, struct_size=48), 1, "scale pointers"),
    (dict(wait_timeout_test=2), 1, "wait_timeout_test"),
    (dict(schedule=4), 1, "schedule"),
    (dict(schedule=-1), 1, "schedule"),
    (dict(schedule=1, kv_quant=1, sk=512, sv=1024), 1, "schedule 1 needs"),
    (dict(schedule=3, kv_quant=1, sk=512, sv=1024), 1, "schedule 3 needs"),
    (dict(schedule=1, wait_timeout_test=1), 1, "schedule 1 needs"),
])
def test_options_are_checked_before_launch(lib, kw, status, msg):
    assert _call_ex(lib, **kw) == status
    assert msg in lib.prefill_attn_last_error().decode()


def test_options_layout_matches_header():
    """The binding's pa_options has the header's field offsets (x86-64 and aarch64 LP64)."""
    P = binding.PaOptions
    assert [(n, getattr(P, n).offset) for n, _ in P._fields_] == [
        ("struct_size", 0), ("window", 4), ("block_table", 8), ("block_size", 16),
        ("max_blocks_per_seq", 20), ("num_blocks", 24), ("reserved", 28), ("rope_theta", 32),
        ("reserved2", 36), ("kv_quant", 40), ("reserved3", 44), ("cache_k_scale", 48), ("cache_v_scale", 56),
        ("wait_timeout_test", 64), ("schedule", 68)]
    assert ctypes.sizeof(P) == 72


@pytest.mark.parametrize("args,expect", [
    # (total_q, num_seqs, n_heads, n_kv_heads, kv_quant, num_sms) -> schedule
    ((32768, 1, 32, 32, 0, 152), 2),   # one long prompt: 4096 two-tile units
    ((512, 1, 32, 32, 0, 152), 1),     # a 512-token MHA prompt: 64 two-tile units <= 152
    ((1024, 1, 32, 32, 0, 152), 1),    # 128 two-tile units <= 152
    ((1536, 1, 32, 32, 0, 152), 2),    # 192 two-tile units > 152
    ((512, 1, 32, 8, 0, 152), 1),      # GQA-4: 64-token units, 8 x 8 = 64 units
    ((576, 65, 32, 8, 0, 152), 3),     # a chunk and 64 decode rows: 8.9 new tokens per sequence
    ((64, 64, 32, 8, 0, 152), 3),      # decode rows only
    ((64, 64, 32, 8, 1, 152), 2),      # int8 cache: always two-tile units, no splitting
    ((4096, 64, 32, 8, 0, 152), 2),    # exactly 64 tokens per sequence is not decode-heavy
    ((4095, 64, 32, 8, 0, 152), 3),
    ((0, 1, 32, 32, 0, 152), -1),
    ((512, 1, 30, 8, 0, 152), -1),     # n_heads not a multiple of n_kv_heads
    ((512, 1, 32, 32, 0, 0), -1),
])
def test_auto_schedule_policy(lib, args, expect):
    """The schedule the library picks when pa_options.schedule is 0 (host-only)."""
    assert binding.prefill_attn_auto_schedule(*args) == expect


def test_last_schedule_is_zero_without_a_launch(lib):
    # an empty batch returns PA_OK without launching anything
    assert lib.prefill_attn_varlen(16, 32, 48, 64, 80, 96, 112, 128, 144, None, 0, 0, 8, 4, 2, 64, 0.125, 1,
                                   None) == 0
    assert lib.prefill_attn_last_launch_count() == 0
    assert lib.prefill_attn_last_schedule() == 0


def test_device_error_bits_are_distinct_and_match_the_binding():
    """Each PA_DEVERR_* bit of the header is its own bit, the binding's constants
    match, and the misaligned shared-memory window has a bit of its own
    (reported as PA_ERR_DEVICE_LAYOUT, not as a wait timeout)."""
    src = open(os.path.join(ROOT, "include", "prefill_attn.h")).read()
    bits = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define PA_DEVERR_(\w+) 0x([0-9a-fA-F]+)", src)}
    assert bits == {"METADATA": 0x1, "TIMEOUT": 0x2, "OVERFLOW": 0x4, "SMEM_ALIGN": 0x8}
    assert binding.DEVERR_METADATA == bits["METADATA"] and binding.DEVERR_TIMEOUT == bits["TIMEOUT"]
    assert binding.DEVERR_OVERFLOW == bits["OVERFLOW"] and binding.DEVERR_SMEM_ALIGN == bits["SMEM_ALIGN"]
    assert re.search(r"PA_ERR_DEVICE_LAYOUT = 6", src)
    assert binding.STATUS[6] == "PA_ERR_DEVICE_LAYOUT"
    # the kernel raises the alignment bit, never the timeout bit, for a misaligned window
    kern = open(os.path.join(ROOT, "prefill_phase_attention_gb300", "csrc", "attn_fwd.cu")).read()
    assert re.search(r"const bool misaligned = \(smem_u32\(smem_raw\) & 1023u\) != 0;", kern)
    i = kern.index("if (misaligned) {")
    assert "PA_DEVERR_SMEM_ALIGN" in kern[i:i + 200] and "PA_DEVERR_TIMEOUT" not in kern[i:i + 200]
