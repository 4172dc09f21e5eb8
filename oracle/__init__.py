"""CPU oracle for causal varlen prefill attention (fp64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The library's
product path never imports, links or executes anything here, and this package
imports nothing from the library.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over query rows);
this module compiles it with gcc and marshals numpy arrays into it.  Every
floating-point input is a bf16 bit pattern (``numpy.uint16``); outputs are
float64.  See ``oracle.c`` for the definition and the passages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

ERRORS = {
    -1: "bad sizes",
    -2: "cu_seqlens_q does not start at 0 or decreases",
    -3: "cu_seqlens_k != cumulative (cache_offsets + seqlen_q)",
    -4: "a sequence does not fit its cache slot",
    -5: "selected row out of range",
    -6: "out of memory",
    -7: "a window needs the causal mask",
    -8: "bad block table",
}


def build_command():
    return ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", _LIB_PATH, "-lm"]


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        subprocess.check_call(build_command())
    return _LIB_PATH


def load_library(path: str):
    """Bind oracle_prefill_attention from a compiled oracle library."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_prefill_attention
    P = ctypes.c_void_p
    I = ctypes.c_int
    f.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                  ctypes.c_double, I, I, P, I, I, I, ctypes.c_double, I, P, P, P, P, P, ctypes.c_int64, I]
    f.restype = I
    g = lib.oracle_rope_rotate
    g.argtypes = [P, ctypes.c_int64, I, P, I, ctypes.c_double, P]
    g.restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def prefill_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, cache_offsets, cache_k, cache_v, *,
                      n_heads: int, n_kv_heads: int, head_dim: int, max_cache_len: int,
                      scale: float, causal: bool = True, window: int = 0, block_table=None, block_size: int = 0,
                      rope_theta: float = 0.0, kv_quant: int = 0, cache_k_scale=None, cache_v_scale=None,
                      rows: Optional[np.ndarray] = None, want_cache: bool = True, threads: int = 0, lib=None):
    """Run the oracle.

    q [T,H,d], k/v [T,Hk,d], cache_k/v [B,Hk,cap,d]: uint16 bf16 bit patterns.
    cu_seqlens_q/k [B+1], cache_offsets [B]: int32.
    rows: optional int64 array of flattened (token * n_heads + head) rows.
    window: 0, or W > 0 (causal only): each query sees its W most recent keys.
    block_table: optional int32 [B, max_blocks]; then cache_k/v are block pools
    [num_blocks, Hk, block_size, d] and max_cache_len = max_blocks * block_size.
    rope_theta > 0: rotary embedding of the new q/k at their absolute positions.
    kv_quant = 1: cache_k/v are int8 codes (same shapes) and cache_k_scale /
    cache_v_scale float32 arrays of shape cache.shape[:-1]; the returned cache
    images are then (codes, scales) pairs.

    Returns (out float64 [T,H,d], lse float64 [T,H], cache_k', cache_v') where
    unselected rows of out/lse are NaN and the cache images are None when
    ``want_cache`` is false.
    """
    lib = lib or _load()
    u16 = lambda a: np.ascontiguousarray(a, dtype=np.uint16)
    i32 = lambda a: np.ascontiguousarray(a, dtype=np.int32)
    q, k, v = map(u16, (q, k, v))
    if kv_quant:
        cache_k = np.ascontiguousarray(cache_k, dtype=np.int8)
        cache_v = np.ascontiguousarray(cache_v, dtype=np.int8)
        sk = np.ascontiguousarray(cache_k_scale, dtype=np.float32)
        sv = np.ascontiguousarray(cache_v_scale, dtype=np.float32)
        assert sk.shape == cache_k.shape[:-1] == sv.shape
    else:
        cache_k, cache_v = map(u16, (cache_k, cache_v))
        sk = sv = None
    cu_q, cu_k, off = map(i32, (cu_seqlens_q, cu_seqlens_k, cache_offsets))
    num_seqs = off.shape[0]
    total_q = int(cu_q[-1]) if num_seqs else 0
    assert q.size == total_q * n_heads * head_dim, "q size disagrees with cu_seqlens_q"
    assert k.size == total_q * n_kv_heads * head_dim and v.size == k.size
    if block_table is None:
        assert cache_k.size == num_seqs * n_kv_heads * max_cache_len * head_dim == cache_v.size
        bt, max_blocks, num_blocks = None, 0, 0
    else:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        max_blocks = bt.shape[1]
        num_blocks = cache_k.shape[0]
        assert cache_k.shape == (num_blocks, n_kv_heads, block_size, head_dim) == cache_v.shape
    out = np.full((total_q, n_heads, head_dim), np.nan, dtype=np.float64)
    lse = np.full((total_q, n_heads), np.nan, dtype=np.float64)
    ck = np.empty_like(cache_k) if want_cache else None
    cv = np.empty_like(cache_v) if want_cache else None
    sk_out = np.empty_like(sk) if (want_cache and kv_quant) else None
    sv_out = np.empty_like(sv) if (want_cache and kv_quant) else None
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    rc = lib.oracle_prefill_attention(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_q), _ptr(cu_k), _ptr(off), _ptr(cache_k), _ptr(cache_v),
        _ptr(ck), _ptr(cv), _ptr(out), _ptr(lse),
        num_seqs, max_cache_len, n_heads, n_kv_heads, head_dim, float(scale), int(bool(causal)), int(window),
        _ptr(bt), int(block_size), int(max_blocks), int(num_blocks), float(rope_theta),
        int(kv_quant), _ptr(sk), _ptr(sv), _ptr(sk_out), _ptr(sv_out), _ptr(sel), 0 if sel is None else sel.shape[0], int(threads))
    if rc != 0:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")
    if want_cache:
        ck = ck.reshape(cache_k.shape)
        cv = cv.reshape(cache_v.shape)
        if kv_quant:
            ck, cv = (ck, sk_out), (cv, sv_out)
    return out, lse, ck, cv


def rope_rotate(x, positions, *, rope_theta: float, max_pos: Optional[int] = None, lib=None):
    """The oracle's rotary rotation alone, before any rounding.

    x [n, d]: uint16 bf16 bit patterns; positions [n]: int32 absolute positions.
    Returns float64 [n, d]: each vector rotated to its position (rotate-half
    pairing, fp32 inv_freq and angles, fp64 cos/sin and rotation).
    """
    lib = lib or _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    n, d = x.shape
    assert pos.shape == (n,)
    mp = int(max_pos if max_pos is not None else (int(pos.max()) + 1 if n else 1))
    out = np.empty((n, d), dtype=np.float64)
    rc = lib.oracle_rope_rotate(_ptr(x), n, d, _ptr(pos), mp, float(rope_theta), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")
    return out
