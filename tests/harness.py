"""Shared test helpers: run a workload through the CUDA library and the oracle,
and compare them with the tolerances the parity bar states.

Tolerances: the KV pool after the write is bit-exact; the bf16 output must
satisfy |gpu - ref| <= 2e-2 + 1e-2 * |ref| elementwise against the fp32
oracle (max-abs 2e-2 with a 1e-2 relative allowance); LSE within 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_variable_length_gb300 import pva
from paged_variable_length_gb300 import workloads as W

ATOL = 2e-2
RTOL = 1e-2
LSE_ATOL = 1e-3


def make_engine(wl: W.Workload, enable_split_kv=True, enable_cascade=True, min_cascade_pages=8, sm_scale=0.0,
                max_tokens=None, max_batch=None, max_kv_len=None, kv_dtype=pva.KV_BF16):
    return pva.PagedAttention(
        wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages,
        max_batch=max_batch or max(wl.batch, 1), max_tokens=max_tokens or max(wl.total_tokens, 1),
        max_kv_len=max_kv_len or max(max(wl.kv_lens) if wl.kv_lens else 1, 1), sm_scale=sm_scale,
        enable_split_kv=enable_split_kv, enable_cascade=enable_cascade, min_cascade_pages=min_cascade_pages,
        kv_dtype=kv_dtype)


def run_cuda(wl: W.Workload, t: dict, engine=None, slot_mapping=None, max_q_len=0, with_lse=True):
    """Prepare + forward on the GPU; the pools in `t` are updated in place."""
    eng = engine or make_engine(wl)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, slot_mapping, max_q_len)
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[0], t["q"].shape[1], dtype=torch.float32, device=t["q"].device) if with_lse else None
    eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out, lse)
    torch.cuda.synchronize()
    return out, lse, eng


def host_copy(t: dict) -> dict:
    return {k: v.detach().cpu().clone() for k, v in t.items()}


def run_oracle(wl: W.Workload, h: dict, slots=None, row_select=None, scale=None):
    return oracle.forward(h["q"], h["k"], h["v"], h["k_pool"], h["v_pool"], h["cu_seqlens_q"].numpy(),
                          h["cache_seqlens"].numpy(), h["page_table"].numpy(), wl.page_size, slots=slots,
                          scale=scale, row_select=row_select)


def pool_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(gpu_out, gpu_lse, ref_out, ref_lse, mask=None):
    g = gpu_out.float().cpu().numpy()
    ref = ref_out
    if mask is not None:
        g, ref = g[mask], ref[mask]
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside |d| <= {ATOL} + {RTOL}|ref|; "
                           f"max abs {err.max():.3e}")
    if gpu_lse is not None:
        gl = gpu_lse.cpu().numpy()
        rl = ref_lse
        if mask is not None:
            m2 = mask.any(axis=-1) if mask.ndim == 3 else mask
            gl, rl = gl[m2], rl[m2]
        lerr = np.abs(gl - rl)
        assert lerr.max() <= LSE_ATOL, f"LSE max abs err {lerr.max():.3e}"
    return float(err.max())
