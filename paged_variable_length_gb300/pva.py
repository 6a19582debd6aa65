"""Thin ctypes binding of libpva.so (the C ABI in include/pva.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  torch is used for device memory and the current stream.  The
library is loaded on first use; if it is missing this raises -- there is no
other code path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpva.so")

PVA_OK = 0
STATUS_NAMES = {
    0: "PVA_OK", 1: "PVA_ERR_INVALID_ARG", 2: "PVA_ERR_UNSUPPORTED", 3: "PVA_ERR_WORKSPACE_TOO_SMALL",
    4: "PVA_ERR_CUDA", 5: "PVA_ERR_DEVICE_CHECK", 6: "PVA_ERR_NOT_PREPARED",
}
DEVERR = {
    0x01: "PVA_DEVERR_CU_SEQLENS", 0x02: "PVA_DEVERR_Q_GT_KV", 0x04: "PVA_DEVERR_PAGE_ID",
    0x08: "PVA_DEVERR_SLOT", 0x10: "PVA_DEVERR_LIMITS", 0x20: "PVA_DEVERR_TIMEOUT",
}
# Every function include/pva.h declares; the CPU tests check the library exports each one.
EXPORTS = ("attn_abi_version", "attn_status_string", "attn_workspace_size", "attn_prepare_metadata",
           "attn_forward", "attn_store_kvcache", "attn_get_device_status", "attn_debug_plan_counts",
           "attn_set_timing_events", "attn_prepare_metadata_static", "attn_forward_fp8kv", "attn_store_kvcache_fp8kv",
           "attn_debug_set_wait_limit")


class PvaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class Config(ctypes.Structure):
    """Mirror of pva_config."""
    _fields_ = [
        ("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int64), ("sm_scale", ctypes.c_float),
        ("max_batch", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("max_kv_len", ctypes.c_int32),
        ("enable_split_kv", ctypes.c_int32), ("enable_cascade", ctypes.c_int32),
        ("min_cascade_pages", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
    ]


class Meta(ctypes.Structure):
    """Mirror of pva_meta (opaque, caller-owned, host memory)."""
    _fields_ = [("opaque", ctypes.c_uint64 * 64)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libpva.so (once).  Raises FileNotFoundError when it was not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise FileNotFoundError(f"{path} is missing: build it with paged_variable_length_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        CP, MP = ctypes.POINTER(Config), ctypes.POINTER(Meta)
        lib.attn_abi_version.argtypes, lib.attn_abi_version.restype = [], i32
        lib.attn_status_string.argtypes, lib.attn_status_string.restype = [ctypes.c_int], ctypes.c_char_p
        lib.attn_workspace_size.argtypes, lib.attn_workspace_size.restype = [CP], sz
        lib.attn_prepare_metadata.argtypes = [CP, P, P, P, i64, P, i32, i32, i32, P, sz, P, MP]
        lib.attn_prepare_metadata.restype = ctypes.c_int
        lib.attn_prepare_metadata_static.argtypes = [CP, P, P, P, i64, P, i32, i32, i32, P, MP]
        lib.attn_prepare_metadata_static.restype = ctypes.c_int
        lib.attn_forward.argtypes = [MP, P, P, P, P, P, P, P, P]
        lib.attn_forward.restype = ctypes.c_int
        lib.attn_store_kvcache.argtypes = [MP, P, P, P, P, P]
        lib.attn_store_kvcache.restype = ctypes.c_int
        lib.attn_forward_fp8kv.argtypes = [MP, P, P, P, P, P, P, P, P, P, P]
        lib.attn_forward_fp8kv.restype = ctypes.c_int
        lib.attn_store_kvcache_fp8kv.argtypes = [MP, P, P, P, P, P, P, P]
        lib.attn_store_kvcache_fp8kv.restype = ctypes.c_int
        lib.attn_get_device_status.argtypes = [MP, ctypes.POINTER(ctypes.c_uint32)]
        lib.attn_get_device_status.restype = ctypes.c_int
        lib.attn_set_timing_events.argtypes = [MP, ctypes.POINTER(ctypes.c_void_p), i32]
        lib.attn_set_timing_events.restype = ctypes.c_int
        lib.attn_debug_set_wait_limit.argtypes = [MP, i64]
        lib.attn_debug_set_wait_limit.restype = ctypes.c_int
        lib.attn_debug_plan_counts.argtypes = [MP, ctypes.POINTER(ctypes.c_int64), i32]
        lib.attn_debug_plan_counts.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def abi_version() -> int:
    return int(load().attn_abi_version())


def _check(status: int, where: str) -> None:
    if status != PVA_OK:
        raise PvaError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


KV_BF16, KV_E4M3 = 0, 1


def make_config(num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, max_batch, max_tokens, max_kv_len,
                sm_scale: float = 0.0, enable_split_kv: bool = True, enable_cascade: bool = True,
                min_cascade_pages: int = 8, kv_dtype: int = KV_BF16) -> Config:
    return Config(num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale, max_batch, max_tokens,
                  max_kv_len, int(enable_split_kv), int(enable_cascade), int(min_cascade_pages), int(kv_dtype))


def attn_workspace_size(cfg: Config) -> int:
    return int(load().attn_workspace_size(ctypes.byref(cfg)))


def attn_prepare_metadata(cfg: Config, cu_seqlens_q, cache_seqlens, page_table, slot_mapping, batch: int,
                          total_tokens: int, max_q_len: int, workspace, stream=None) -> Meta:
    meta = Meta()
    st = load().attn_prepare_metadata(
        ctypes.byref(cfg), _ptr(cu_seqlens_q), _ptr(cache_seqlens), _ptr(page_table), int(page_table.stride(0)),
        _ptr(slot_mapping), int(batch), int(total_tokens), int(max_q_len), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream(stream), ctypes.byref(meta))
    _check(st, "attn_prepare_metadata")
    return meta


def attn_prepare_metadata_static(cfg: Config, cu_seqlens_q, cache_seqlens, page_table, slot_mapping, batch: int,
                                 total_tokens: int, max_q_len: int, stream=None) -> Meta:
    """attn_prepare_metadata with the plan in the library's built-in scratch area (no workspace)."""
    meta = Meta()
    st = load().attn_prepare_metadata_static(
        ctypes.byref(cfg), _ptr(cu_seqlens_q), _ptr(cache_seqlens), _ptr(page_table), int(page_table.stride(0)),
        _ptr(slot_mapping), int(batch), int(total_tokens), int(max_q_len), _stream(stream), ctypes.byref(meta))
    _check(st, "attn_prepare_metadata_static")
    return meta


def attn_forward(meta: Meta, q, k, v, k_pool, v_pool, out, lse=None, stream=None) -> None:
    st = load().attn_forward(ctypes.byref(meta), _ptr(q), _ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(out),
                             _ptr(lse), _stream(stream))
    _check(st, "attn_forward")


def attn_store_kvcache(meta: Meta, k, v, k_pool, v_pool, stream=None) -> None:
    st = load().attn_store_kvcache(ctypes.byref(meta), _ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool),
                                   _stream(stream))
    _check(st, "attn_store_kvcache")


def attn_forward_fp8kv(meta: Meta, q, k, v, k_pool, v_pool, k_scale, v_scale, out, lse=None, stream=None) -> None:
    """attn_forward over E4M3 pools (uint8 tensors) with per-kv-head fp32 scales (device tensors)."""
    st = load().attn_forward_fp8kv(ctypes.byref(meta), _ptr(q), _ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool),
                                   _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "attn_forward_fp8kv")


def attn_store_kvcache_fp8kv(meta: Meta, k, v, k_pool, v_pool, k_scale, v_scale, stream=None) -> None:
    st = load().attn_store_kvcache_fp8kv(ctypes.byref(meta), _ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool),
                                         _ptr(k_scale), _ptr(v_scale), _stream(stream))
    _check(st, "attn_store_kvcache_fp8kv")


def attn_get_device_status(meta: Meta) -> int:
    """Synchronises; returns the device error word (0 = clean)."""
    bits = ctypes.c_uint32(0)
    st = load().attn_get_device_status(ctypes.byref(meta), ctypes.byref(bits))
    if st not in (PVA_OK, 5):
        _check(st, "attn_get_device_status")
    return int(bits.value)


def attn_debug_plan_counts(meta: Meta) -> dict:
    arr = (ctypes.c_int64 * 9)()
    n = load().attn_debug_plan_counts(ctypes.byref(meta), arr, 9)
    keys = ("dec_units", "dec_groups", "pre_tiles", "casc_groups", "casc_tiles", "split_chunk", "partial_slots",
            "kernels_per_forward", "casc_levels")
    return {keys[i]: int(arr[i]) for i in range(n)}


def attn_debug_set_wait_limit(meta: Meta, limit_ns: int) -> None:
    """Tests only: the forward kernels' wait limit for this meta (ns; 0 = give up at once,
    negative = the default 2 s).  Synchronises; the next prepare restores the default."""
    _check(load().attn_debug_set_wait_limit(ctypes.byref(meta), int(limit_ns)), "attn_debug_set_wait_limit")


def attn_set_timing_events(meta: Meta, events) -> None:
    """events: five torch.cuda.Event(enable_timing=True) already recorded once, or None to turn off."""
    if not events:
        _check(load().attn_set_timing_events(ctypes.byref(meta), None, 0), "attn_set_timing_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().attn_set_timing_events(ctypes.byref(meta), arr, len(events)), "attn_set_timing_events")


def deverr_names(bits: int) -> list[str]:
    return [name for b, name in DEVERR.items() if bits & b]


def ragged_layout(cu_seqlens_q, cu_seqlens_kv, device=None):
    """Page table and slot mapping that make contiguous (ragged) K/V an ordinary batch.

    With K/V given as [total_kv, Hkv, D] tensors whose rows cu_seqlens_kv[i] ..
    cu_seqlens_kv[i+1]-1 are request i's keys (its cached part, if any, followed by its
    new tokens), a config with page_size 1 and num_pages >= total_kv, and
    page_table[i][j] = cu_seqlens_kv[i] + j address them in place: pass k / v themselves
    as the pools, kv lengths cu_seqlens_kv[i+1] - cu_seqlens_kv[i] as cache_seqlens, and
    this slot mapping (-1 for every new token: nothing is stored, the keys already sit
    where the table points).  Returns (page_table int32 [B, max_kv], slot_mapping int64
    [total_q]) on ``device``.  Host-side arithmetic, once per batch.
    """
    import torch

    cu = torch.as_tensor(cu_seqlens_kv, dtype=torch.int64).cpu()
    lens = cu[1:] - cu[:-1]
    B = int(lens.numel())
    width = max(int(lens.max()) if B else 1, 1)
    j = torch.arange(width, dtype=torch.int64)
    table = torch.where(j[None, :] < lens[:, None], cu[:-1, None] + j[None, :], torch.zeros(1, dtype=torch.int64))
    total_q = int(torch.as_tensor(cu_seqlens_q)[-1])
    dev = device if device is not None else "cpu"
    return table.to(torch.int32).to(dev), torch.full((total_q,), -1, dtype=torch.int64, device=dev)


class PagedAttention:
    """Owns a config and a torch-allocated workspace; one prepare per batch, one forward per layer."""

    def __init__(self, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, max_batch, max_tokens,
                 max_kv_len, sm_scale: float = 0.0, enable_split_kv: bool = True, enable_cascade: bool = True,
                 min_cascade_pages: int = 8, device="cuda", kv_dtype: int = KV_BF16):
        import torch

        self.cfg = make_config(num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, max_batch, max_tokens,
                               max_kv_len, sm_scale, enable_split_kv, enable_cascade, min_cascade_pages, kv_dtype)
        nbytes = attn_workspace_size(self.cfg)
        if nbytes == 0:
            raise PvaError(2, "attn_workspace_size")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.meta = None
        self._keep = None

    def prepare(self, cu_seqlens_q, cache_seqlens, page_table, total_tokens: int, slot_mapping=None,
                max_q_len: int = 0, stream=None) -> Meta:
        """Once per batch.  The index tensors are kept referenced until the next prepare."""
        batch = int(cache_seqlens.numel())
        self._keep = (cu_seqlens_q, cache_seqlens, page_table, slot_mapping)
        self.meta = attn_prepare_metadata(self.cfg, cu_seqlens_q, cache_seqlens, page_table, slot_mapping, batch,
                                          total_tokens, max_q_len, self.workspace, stream)
        return self.meta

    def forward(self, q, k, v, k_pool, v_pool, out=None, lse=None, stream=None, k_scale=None, v_scale=None):
        """One layer.  With an E4M3 config the pools are uint8 and k_scale / v_scale (fp32 [Hkv],
        on the device) are required."""
        import torch

        if out is None:
            out = torch.empty_like(q)
        if self.cfg.kv_dtype == KV_E4M3:
            attn_forward_fp8kv(self.meta, q, k, v, k_pool, v_pool, k_scale, v_scale, out, lse, stream)
        else:
            attn_forward(self.meta, q, k, v, k_pool, v_pool, out, lse, stream)
        return out
