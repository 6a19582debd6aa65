"""Shared test helpers: run a workload through the CUDA library and the oracle,
and compare them with the tolerances the parity bar states.

Tolerances: the KV pool after the write is bit-exact; against the fp32 oracle the
bf16 output must have max-abs error <= 2e-2 and max-rel error <= 1e-2, the relative
error of an element taken against max(|ref|, 1) (so below |ref| = 1 it is the absolute
error, and no element near zero can fail on rounding alone); LSE within 1e-3 absolute.
Every comparison is recorded (test, max-abs, max-rel, LSE) and listed at the end of
the session.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_variable_length_gb300 import pva
from paged_variable_length_gb300 import workloads as W

MAX_ABS = 2e-2
MAX_REL = 1e-2
LSE_ATOL = 1e-3

# (test id, compared elements, max-abs, max-rel, LSE max-abs) of every assert_close call
RECORDS: list = []


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


def error_figures(g: np.ndarray, ref: np.ndarray):
    """(max-abs, max-rel) of g against ref; the relative error is taken against max(|ref|, 1)."""
    if g.size == 0:
        return 0.0, 0.0
    err = np.abs(g.astype(np.float64) - ref.astype(np.float64))
    rel = err / np.maximum(np.abs(ref.astype(np.float64)), 1.0)
    return float(err.max()), float(rel.max())


def assert_close(gpu_out, gpu_lse, ref_out, ref_lse, mask=None):
    """Assert the stated bar (max-abs <= 2e-2, max-rel <= 1e-2, LSE <= 1e-3) and
    return the max-abs error.  `mask` selects the compared rows (sampled checks)."""
    import os

    g = gpu_out.float().cpu().numpy()
    ref = ref_out
    if mask is not None:
        g, ref = g[mask], ref[mask]
    assert np.isfinite(g).all(), "non-finite output"
    max_abs, max_rel = error_figures(g, ref)
    lerr = None
    if gpu_lse is not None:
        gl = gpu_lse.cpu().numpy()
        rl = ref_lse
        if mask is not None:
            m2 = mask.any(axis=-1) if mask.ndim == 3 else mask
            gl, rl = gl[m2], rl[m2]
        lerr = float(np.abs(gl - rl).max()) if gl.size else 0.0
    RECORDS.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], int(g.size), max_abs, max_rel, lerr))
    assert max_abs <= MAX_ABS, f"max-abs error {max_abs:.3e} > {MAX_ABS} (max-rel {max_rel:.3e})"
    assert max_rel <= MAX_REL, f"max-rel error {max_rel:.3e} > {MAX_REL} (max-abs {max_abs:.3e})"
    if lerr is not None:
        assert lerr <= LSE_ATOL, f"LSE max abs err {lerr:.3e}"
    return max_abs
