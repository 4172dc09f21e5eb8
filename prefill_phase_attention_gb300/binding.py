"""ctypes binding of include/prefill_attn.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors are
PyTorch CUDA tensors; their data pointers, sizes and the current CUDA stream
are passed straight to the library, which does all of the work on the GPU.
There is no fallback: if the compiled library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

PA_OK = 0
STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
          4: "PA_ERR_DEVICE_TIMEOUT", 5: "PA_ERR_DEVICE_METADATA", 6: "PA_ERR_DEVICE_LAYOUT"}
DEVERR_METADATA, DEVERR_TIMEOUT, DEVERR_OVERFLOW, DEVERR_SMEM_ALIGN = 0x1, 0x2, 0x4, 0x8

class PaOptions(ctypes.Structure):
    """pa_options of include/prefill_attn.h."""
    _fields_ = [("struct_size", ctypes.c_uint32), ("window", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("block_size", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("reserved2", ctypes.c_int32),
                ("kv_quant", ctypes.c_int32), ("reserved3", ctypes.c_int32),
                ("cache_k_scale", ctypes.c_void_p), ("cache_v_scale", ctypes.c_void_p),
                ("wait_timeout_test", ctypes.c_int32), ("schedule", ctypes.c_int32)]


# Entry points declared in include/prefill_attn.h: name -> (restype, argtypes)
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_VARLEN_ARGS = [_P] * 10 + [_I] * 6 + [_F, _I, _P]
_VARLEN_EX_ARGS = [_P] * 10 + [_I] * 6 + [_F, _I, ctypes.POINTER(PaOptions), _P]
SIGNATURES = {
    "prefill_attn_varlen": (_I, _VARLEN_ARGS),
    "prefill_attn_varlen_validate": (_I, _VARLEN_ARGS),
    "prefill_attn_varlen_noalloc": (_I, _VARLEN_ARGS),
    "prefill_attn_varlen_ex": (_I, _VARLEN_EX_ARGS),
    "prefill_attn_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "prefill_attn_release": (None, []),
    "prefill_attn_status_string": (ctypes.c_char_p, [_I]),
    "prefill_attn_last_error": (ctypes.c_char_p, []),
    "prefill_attn_last_launch_count": (_I, []),
    "prefill_attn_last_schedule": (_I, []),
    "prefill_attn_auto_schedule": (_I, [_I, _I, _I, _I, _I, _I]),
}

_lib = None


class PrefillAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load (once) the compiled library and bind every declared entry point."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"prefill_attn library not built: {p} is missing "
                           "(run prefill_phase_attention_gb300.build.build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(status: int):
    if status != PA_OK:
        raise PrefillAttnError(status, load().prefill_attn_last_error().decode())


# The current stream's raw handle: torch's own accessor costs ~0.1 us, building
# a torch.cuda.Stream object for it ~3 us (a quarter of a small call's host time).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device_index: Optional[int] = None) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and device_index is not None:
        return _raw_stream(device_index)
    return torch.cuda.current_stream().cuda_stream


def _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                 scale, causal, stream, max_cache_len=None, cache_dtype=torch.bfloat16):
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("cache_k", cache_k, cache_dtype), ("cache_v", cache_v, cache_dtype),
                        ("out", out, torch.bfloat16), ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("cu_seqlens_k", cu_seqlens_k, torch.int32), ("cache_offsets", cache_offsets, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous CUDA float32 tensor")
    if q.dim() != 3 or k.dim() != 3 or cache_k.dim() != 4:
        raise ValueError("q/k/v are [total_q, heads, head_dim]; caches are [num_seqs, kv_heads, cap, head_dim]")
    total_q, n_heads, head_dim = q.shape
    n_kv_heads = k.shape[1]
    num_seqs = cache_offsets.numel()
    if scale is None:
        scale = head_dim ** -0.5
    return (q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
            cache_k.data_ptr(), cache_v.data_ptr(), cache_offsets.data_ptr(), out.data_ptr(),
            None if lse is None else lse.data_ptr(),
            num_seqs, total_q, cache_k.shape[2] if max_cache_len is None else max_cache_len,
            n_heads, n_kv_heads, head_dim,
            float(scale), int(bool(causal)), _stream_handle(stream, q.get_device()))


def prefill_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out,
                        lse=None, *, scale: Optional[float] = None, causal: bool = True, stream=None) -> None:
    """Enqueue causal varlen prefill attention + the KV-cache write on `stream`.

    Shapes: q/out [total_q, n_heads, head_dim], k/v [total_q, n_kv_heads, head_dim] (bf16),
    cache_k/v [num_seqs, n_kv_heads, max_cache_len, head_dim] (bf16), cu_seqlens_q/k
    [num_seqs+1], cache_offsets [num_seqs] (int32), lse [total_q, n_heads] fp32 or None.
    """
    args = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                        scale, causal, stream)
    _check(load().prefill_attn_varlen(*args))


def make_options(window: int = 0, block_table=None, block_size: int = 0, num_blocks: int = 0,
                 rope_theta: float = 0.0, cache_k_scale=None, cache_v_scale=None,
                 wait_timeout_test: bool = False, schedule: int = 0) -> PaOptions:
    o = PaOptions()
    o.struct_size = ctypes.sizeof(PaOptions)
    o.window = int(window)
    o.rope_theta = float(rope_theta)
    o.wait_timeout_test = int(bool(wait_timeout_test))
    o.schedule = int(schedule)
    if cache_k_scale is not None:
        o.kv_quant = 1
        o.cache_k_scale = cache_k_scale.data_ptr()
        o.cache_v_scale = cache_v_scale.data_ptr()
    if block_table is not None:
        o.block_table = block_table.data_ptr()
        o.block_size = int(block_size)
        o.max_blocks_per_seq = int(block_table.shape[1])
        o.num_blocks = int(num_blocks)
    return o


def prefill_attn_varlen_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse=None, *,
                           scale: Optional[float] = None, causal: bool = True, window: int = 0,
                           block_table=None, rope_theta: float = 0.0, cache_k_scale=None, cache_v_scale=None,
                           wait_timeout_test: bool = False, schedule: int = 0, stream=None) -> None:
    """prefill_attn_varlen with options.

    window > 0 restricts each query to its `window` most recent keys (causal only).
    block_table (int32 CUDA [num_seqs, max_blocks_per_seq]) selects the paged cache:
    cache_k/v are then block pools [num_blocks, n_kv_heads, block_size, head_dim]
    and position p of sequence b lives in row p % block_size of block
    block_table[b, p // block_size].
    rope_theta > 0 rotates every new q/k to its absolute position (rotary
    embedding, rotate-half pairing) before attention and the cache write.
    cache_k_scale / cache_v_scale (fp32 CUDA [num_seqs, n_kv_heads, max_cache_len])
    select the int8 cache: cache_k/v are then int8 codes and row (b, h, p) stands
    for code * scale.
    schedule fixes the work schedule (pa_options.schedule: 1 one-tile units
    splitting their KV tiles between the two slots, 2 two-tile units, 3
    two-tile units with single-tile ones split; 0 = the library's choice).
    """
    cap = None
    if block_table is not None:
        if block_table.dtype != torch.int32 or not block_table.is_cuda or not block_table.is_contiguous() \
                or block_table.dim() != 2:
            raise ValueError("block_table must be a contiguous 2-D CUDA int32 tensor")
        cap = block_table.shape[1] * cache_k.shape[2]
    quant = cache_k_scale is not None or cache_v_scale is not None
    if quant:
        for name, t in (("cache_k_scale", cache_k_scale), ("cache_v_scale", cache_v_scale)):
            if t is None or t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() \
                    or tuple(t.shape) != tuple(cache_k.shape[:-1]):
                raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of shape cache.shape[:-1]")
    args = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                        scale, causal, stream, max_cache_len=cap,
                        cache_dtype=torch.int8 if quant else torch.bfloat16)
    opts = make_options(window, block_table, cache_k.shape[2], cache_k.shape[0], rope_theta,
                        cache_k_scale, cache_v_scale, wait_timeout_test, schedule)
    _check(load().prefill_attn_varlen_ex(*args[:-1], ctypes.byref(opts), args[-1]))


def prefill_attn_varlen_noalloc(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out,
                                lse=None, *, scale: Optional[float] = None, causal: bool = True,
                                stream=None) -> None:
    """Same as prefill_attn_varlen, with the scheduler scratch in the library's fixed
    device array instead of an allocated workspace (see include/prefill_attn.h)."""
    args = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                        scale, causal, stream)
    _check(load().prefill_attn_varlen_noalloc(*args))


def prefill_attn_varlen_validate(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets,
                                 out, lse=None, *, scale: Optional[float] = None, causal: bool = True,
                                 stream=None) -> None:
    """Strict (host-synchronising) check of the same arguments; raises on failure."""
    args = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_k, cache_v, cache_offsets, out, lse,
                        scale, causal, stream)
    _check(load().prefill_attn_varlen_validate(*args))


def prefill_attn_device_status(stream=None) -> int:
    """Synchronise, read and clear the device error word; returns its PA_DEVERR_* bits."""
    flags = ctypes.c_int32(0)
    st = load().prefill_attn_device_status(_stream_handle(stream), ctypes.byref(flags))
    if st not in (PA_OK, 4, 5, 6):
        _check(st)
    return flags.value


def prefill_attn_release() -> None:
    load().prefill_attn_release()


def prefill_attn_last_launch_count() -> int:
    return load().prefill_attn_last_launch_count()


def prefill_attn_last_schedule() -> int:
    """The schedule (pa_options.schedule 1, 2 or 3) the last call on this thread ran."""
    return load().prefill_attn_last_schedule()


def prefill_attn_auto_schedule(total_q: int, num_seqs: int, n_heads: int, n_kv_heads: int, kv_quant: bool,
                               num_sms: int) -> int:
    """The schedule the library picks for these sizes (host-only; -1 for rejected sizes)."""
    return load().prefill_attn_auto_schedule(total_q, num_seqs, n_heads, n_kv_heads, int(bool(kv_quant)), num_sms)
