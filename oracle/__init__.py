"""Plain CPU oracle for the paged variable-length attention forward.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product path (the CUDA library
and its binding) never does, and the two share no code.

The arithmetic lives in ``pva_oracle.c`` (plain C, fp32, one request and one
head at a time).  This module compiles it with gcc, marshals numpy arrays to
it, and adds the host-side metadata helpers the pages define:

* ``batch_layout`` -- "Variable-length batching and one mixed forward pass",
  sections "Layout and metadata" and "Implementation" (``build_batch``):
  per-request (new tokens, tokens already computed) -> query_start_loc,
  seq_lens, positions, logits_indices.
* ``last_indices`` -- "The attention backend and a reference implementation",
  section "The interface" (``get_last_indices``: each request's last query
  index in the flat q).
* ``e4m3_encode`` / ``e4m3_decode`` and the ``*_fp8`` functions -- an FP8 (E4M3,
  OCP 8-bit floating-point format) KV pool with a per-kv-head scale, the
  KV-cache dtype choice of "Attention backends: ..." (the backend interface's
  kv_cache_dtype): stored e4m3(x / scale), read back as e4m3 * scale.

Parity pins for everything here are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Iterable, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pva_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.oracle_slot_mapping.argtypes = [i32, P, P, P, i64, i32, P]
        lib.oracle_slot_mapping.restype = i32
        lib.oracle_store_kvcache.argtypes = [i64, i32, i32, P, P, P, i64, P, P]
        lib.oracle_store_kvcache.restype = i32
        lib.oracle_causal_mask.argtypes = [i32, i32, P]
        lib.oracle_causal_mask.restype = None
        lib.oracle_attention.argtypes = [i32, P, P, P, i64, i32, i64, i32, i32, i32, f32,
                                         P, P, P, P, P, P]
        lib.oracle_attention.restype = i32
        lib.oracle_attention_fp8.argtypes = [i32, P, P, P, i64, i32, i64, i32, i32, i32, f32,
                                             P, P, P, P, P, P, P, P]
        lib.oracle_attention_fp8.restype = i32
        lib.oracle_store_kvcache_fp8.argtypes = [i64, i32, i32, P, P, P, i64, P, P, P, P]
        lib.oracle_store_kvcache_fp8.restype = i32
        lib.oracle_e4m3_encode_array.argtypes = [i64, P, P]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [i64, P, P]
        lib.oracle_e4m3_decode_array.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


class OracleError(ValueError):
    pass


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """bf16 storage as uint16 bit patterns (accepts a torch bf16 tensor or uint16 array)."""
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("expected bf16 bit patterns as uint16")
        return np.ascontiguousarray(a)
    import torch  # local import: numpy-only callers never need torch

    if a.dtype != torch.bfloat16:
        raise TypeError("expected a torch.bfloat16 tensor")
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# --------------------------------------------------------------------------- metadata

def slot_mapping(cu_seqlens_q, cache_seqlens, page_table, page_size: int) -> np.ndarray:
    """Destination slot of every new token: the last n_i positions of request i."""
    cu = _c(cu_seqlens_q, np.int32)
    lens = _c(cache_seqlens, np.int32)
    pt = _c(page_table, np.int32)
    B = lens.shape[0]
    T = int(cu[B])
    out = np.zeros(T, dtype=np.int64)
    rc = _load().oracle_slot_mapping(B, _ptr(cu), _ptr(lens), _ptr(pt), pt.shape[1], page_size, _ptr(out))
    if rc != 0:
        raise OracleError(f"request {-rc - 1}: q_len must satisfy 0 <= q_len <= kv_len")
    return out


def causal_mask(n: int, kv_len: int) -> np.ndarray:
    """[n, kv_len] bool, True where query r may see key j (bottom-right aligned)."""
    m = np.zeros((n, kv_len), dtype=np.uint8)
    _load().oracle_causal_mask(n, kv_len, _ptr(m))
    return m.astype(bool)


def last_indices(cu_seqlens_q) -> np.ndarray:
    """Index of each request's last query in the flat q (``get_last_indices``)."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    return cu[1:] - 1


def batch_layout(items: Iterable[tuple[int, int, bool]]):
    """Flat-batch metadata from per-request (new_tokens, already_computed, needs_logits).

    Mirrors what ``build_batch`` assembles: request i's new tokens sit at
    positions computed .. computed+new-1; query_start_loc is their prefix sum;
    seq_lens is computed+new (the KV length after this step); logits_indices
    holds the flat index of the last new token of each request that samples.
    """
    qsl, seq_lens, positions, logits = [0], [], [], []
    for new, computed, need_logits in items:
        positions.extend(range(computed, computed + new))
        qsl.append(qsl[-1] + new)
        seq_lens.append(computed + new)
        if need_logits:
            logits.append(qsl[-1] - 1)
    return {
        "query_start_loc": qsl,
        "seq_lens": seq_lens,
        "positions": positions,
        "logits_indices": logits,
    }


# --------------------------------------------------------------------------- store + attention

def store_kvcache(k, v, slots, k_pool, v_pool) -> tuple[np.ndarray, np.ndarray]:
    """Return copies of the pools with this step's K/V written at their slots (raw bf16 bits)."""
    kb, vb = _bits(k), _bits(v)
    kp, vp = _bits(k_pool).copy(), _bits(v_pool).copy()
    T, Hkv, D = kb.shape
    s = _c(slots, np.int64)
    num_slots = kp.shape[0]
    rc = _load().oracle_store_kvcache(T, Hkv, D, _ptr(kb), _ptr(vb), _ptr(s), num_slots, _ptr(kp), _ptr(vp))
    if rc != 0:
        raise OracleError(f"token {-rc - 1}: slot out of range")
    return kp, vp


def attention(q, k_pool, v_pool, cu_seqlens_q, cache_seqlens, page_table, page_size: int,
              scale: float | None = None, row_select: np.ndarray | None = None):
    """fp32 attention output [T, Hq, D] and LSE [T, Hq] over an already-written pool.

    ``row_select`` ([T, Hq] bool) restricts the work to the marked rows; the
    others are returned as NaN.
    """
    qb, kp, vp = _bits(q), _bits(k_pool), _bits(v_pool)
    T, Hq, D = qb.shape
    Hkv = kp.shape[1]
    if Hq % Hkv != 0:
        raise OracleError("Hq must be a multiple of Hkv")
    cu = _c(cu_seqlens_q, np.int32)
    lens = _c(cache_seqlens, np.int32)
    pt = _c(page_table, np.int32)
    B = lens.shape[0]
    num_pages = kp.shape[0] // page_size
    if scale is None:
        scale = float(D) ** -0.5
    out = np.full((T, Hq, D), np.nan, dtype=np.float32)
    lse = np.full((T, Hq), np.nan, dtype=np.float32)
    sel = None if row_select is None else _c(row_select, np.uint8)
    rc = _load().oracle_attention(B, _ptr(cu), _ptr(lens), _ptr(pt), pt.shape[1], page_size, num_pages,
                                  Hq, Hkv, D, float(scale), _ptr(qb), _ptr(kp), _ptr(vp), _ptr(sel),
                                  _ptr(out), _ptr(lse))
    if rc != 0:
        raise OracleError(f"request {-rc - 1}: q_len > kv_len or page id out of range" if rc > -1000000
                          else "out of host memory")
    return out, lse


def forward(q, k, v, k_pool, v_pool, cu_seqlens_q, cache_seqlens, page_table, page_size: int,
            slots: Sequence[int] | np.ndarray | None = None, scale: float | None = None,
            row_select: np.ndarray | None = None):
    """The whole step: store this step's K/V first, then attention.

    Returns (out fp32 [T,Hq,D], lse fp32 [T,Hq], k_pool bits, v_pool bits).
    ``slots`` defaults to the slot mapping derived from the page table.
    """
    if slots is None:
        slots = slot_mapping(cu_seqlens_q, cache_seqlens, page_table, page_size)
    kp, vp = store_kvcache(k, v, slots, k_pool, v_pool)
    out, lse = attention(q, kp, vp, cu_seqlens_q, cache_seqlens, page_table, page_size, scale, row_select)
    return out, lse, kp, vp


# --------------------------------------------------------------------------- FP8 (E4M3) KV pool

def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, |x| > 448 saturates, NaN -> NaN code) of fp32 values."""
    a = _c(np.asarray(x, dtype=np.float32), np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(a.size, _ptr(a), _ptr(out))
    return out


def e4m3_decode(b) -> np.ndarray:
    """fp32 values of E4M3 codes."""
    a = _c(np.asarray(b, dtype=np.uint8), np.uint8)
    out = np.empty(a.shape, dtype=np.float32)
    _load().oracle_e4m3_decode_array(a.size, _ptr(a), _ptr(out))
    return out


def _u8(a) -> np.ndarray:
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint8:
            raise TypeError("expected an FP8 pool as uint8 codes")
        return np.ascontiguousarray(a)
    import torch

    if a.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise TypeError("expected a torch uint8 (or float8_e4m3fn) tensor")
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.uint8).numpy())


def _scales(x, Hkv: int) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    a = _c(np.asarray(x, dtype=np.float32).reshape(-1), np.float32)
    if a.shape[0] != Hkv:
        raise OracleError("one scale per kv head expected")
    return a


def store_kvcache_fp8(k, v, slots, k_pool, v_pool, k_scale, v_scale) -> tuple[np.ndarray, np.ndarray]:
    """Copies of the FP8 pools with this step's K/V quantised into their slots."""
    kb, vb = _bits(k), _bits(v)
    kp, vp = _u8(k_pool).copy(), _u8(v_pool).copy()
    T, Hkv, D = kb.shape
    s = _c(slots, np.int64)
    ks, vs = _scales(k_scale, Hkv), _scales(v_scale, Hkv)
    rc = _load().oracle_store_kvcache_fp8(T, Hkv, D, _ptr(kb), _ptr(vb), _ptr(s), kp.shape[0], _ptr(ks), _ptr(vs),
                                         _ptr(kp), _ptr(vp))
    if rc != 0:
        raise OracleError(f"token {-rc - 1}: slot out of range")
    return kp, vp


def attention_fp8(q, k_pool, v_pool, k_scale, v_scale, cu_seqlens_q, cache_seqlens, page_table, page_size: int,
                  scale: float | None = None, row_select: np.ndarray | None = None):
    """``attention`` over FP8 pools ([slots, Hkv, D] uint8 codes, one scale per kv head)."""
    qb, kp, vp = _bits(q), _u8(k_pool), _u8(v_pool)
    T, Hq, D = qb.shape
    Hkv = kp.shape[1]
    if Hq % Hkv != 0:
        raise OracleError("Hq must be a multiple of Hkv")
    ks, vs = _scales(k_scale, Hkv), _scales(v_scale, Hkv)
    cu = _c(cu_seqlens_q, np.int32)
    lens = _c(cache_seqlens, np.int32)
    pt = _c(page_table, np.int32)
    B = lens.shape[0]
    num_pages = kp.shape[0] // page_size
    if scale is None:
        scale = float(D) ** -0.5
    out = np.full((T, Hq, D), np.nan, dtype=np.float32)
    lse = np.full((T, Hq), np.nan, dtype=np.float32)
    sel = None if row_select is None else _c(row_select, np.uint8)
    rc = _load().oracle_attention_fp8(B, _ptr(cu), _ptr(lens), _ptr(pt), pt.shape[1], page_size, num_pages,
                                      Hq, Hkv, D, float(scale), _ptr(qb), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs),
                                      _ptr(sel), _ptr(out), _ptr(lse))
    if rc != 0:
        raise OracleError(f"request {-rc - 1}: q_len > kv_len or page id out of range" if rc > -1000000
                          else "out of host memory")
    return out, lse


def forward_fp8(q, k, v, k_pool, v_pool, k_scale, v_scale, cu_seqlens_q, cache_seqlens, page_table,
                page_size: int, slots=None, scale: float | None = None, row_select: np.ndarray | None = None):
    """The whole step over FP8 pools: quantised store first, then attention.

    Returns (out fp32 [T,Hq,D], lse fp32 [T,Hq], k_pool codes, v_pool codes).
    """
    if slots is None:
        slots = slot_mapping(cu_seqlens_q, cache_seqlens, page_table, page_size)
    kp, vp = store_kvcache_fp8(k, v, slots, k_pool, v_pool, k_scale, v_scale)
    out, lse = attention_fp8(q, kp, vp, k_scale, v_scale, cu_seqlens_q, cache_seqlens, page_table, page_size,
                             scale, row_select)
    return out, lse, kp, vp

