"""The kernels' bounded waits, made to run out on healthy batches (GPU).

Every wait inside the forward kernels (pipeline stages, the tensor core, the work queue)
gives up after a time limit, sets PVA_DEVERR_TIMEOUT, waits for its CTA's own copies and
MMAs, frees what it holds and returns: a wedged kernel ends with a status instead of
hanging the device.  attn_debug_set_wait_limit(meta, 0) makes every such wait give up as
soon as it would have to wait at all, so these tests run ordinary batches -- decode only,
prefill tiles on the tensor-core kernel, a shared-prefix pass, an FP8 pool -- with waits
that do run out, and check that the forward returns (no trap), that the status reports
the timeout, and that the next prepare + forward on the same device, at the default
limit, matches the oracle (KV pool bit-exact, output within the parity bar).
"""
import numpy as np
import pytest
import torch

import oracle
from harness import assert_close, host_copy, make_engine, pool_bits, run_oracle
from paged_variable_length_gb300 import pva
from paged_variable_length_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
TIMEOUT = 0x20

CASES = {
    "decode-only": lambda: W.custom([1, 1, 1, 1, 1, 1], [700, 33, 1500, 2500, 90, 300], 32, 8, 128, 16, seed=11),
    "prefill-and-decode": lambda: W.custom([300, 1, 1, 40], [300, 2000, 900, 700], 32, 8, 128, 16, seed=12),
    "shared-prefix": lambda: W.custom([1] * 6, [300, 310, 290, 400, 333, 301], 32, 8, 128, 16, seed=13,
                                      shared_prefix_pages=16),
}


def _prepare(eng, wl, t):
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, None, max(wl.q_lens))


@pytest.mark.parametrize("name", list(CASES))
def test_expired_waits_report_timeout_then_the_next_forward_is_correct(name):
    wl = CASES[name]()
    t = W.make_tensors(wl, DEV, poison_unused=True)
    h = host_copy(t)
    eng = make_engine(wl)
    _prepare(eng, wl, t)
    pva.attn_debug_set_wait_limit(eng.meta, 0)
    out = torch.zeros_like(t["q"])
    eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out)
    torch.cuda.synchronize()  # the forward returns: the kernels gave up instead of hanging
    bits = pva.attn_get_device_status(eng.meta)
    assert bits & TIMEOUT, f"no wait ran out (error bits {bits:#x})"
    # a new prepare restores the default limit and clears the error word
    _prepare(eng, wl, t)
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=DEV)
    eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out, lse)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    ref_o, ref_l, ref_kp, ref_vp = run_oracle(wl, h)
    assert np.array_equal(pool_bits(t["k_pool"]), ref_kp) and np.array_equal(pool_bits(t["v_pool"]), ref_vp)
    assert_close(out, lse, ref_o, ref_l)


def test_fp8_pool_expired_waits_then_correct():
    wl = W.custom([40, 1, 130], [40, 2000, 300], 32, 8, 128, 16, seed=14)  # tensor-core and decode kernels
    t = W.make_tensors(wl, DEV)
    kp, vp, ks, vs = W.make_fp8_pools(wl, DEV, poison_unused=True)
    h = {n: x.detach().cpu().clone() for n, x in dict(t, kp=kp, vp=vp, ks=ks, vs=vs).items()}
    eng = make_engine(wl, kv_dtype=pva.KV_E4M3)
    _prepare(eng, wl, t)
    pva.attn_debug_set_wait_limit(eng.meta, 0)
    out = torch.zeros_like(t["q"])
    eng.forward(t["q"], t["k"], t["v"], kp, vp, out, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) & TIMEOUT
    _prepare(eng, wl, t)
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=DEV)
    eng.forward(t["q"], t["k"], t["v"], kp, vp, out, lse, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    ref_o, ref_l, ref_kp, ref_vp = oracle.forward_fp8(
        h["q"], h["k"], h["v"], h["kp"], h["vp"], h["ks"], h["vs"], h["cu_seqlens_q"].numpy(),
        h["cache_seqlens"].numpy(), h["page_table"].numpy(), wl.page_size)
    assert np.array_equal(kp.cpu().numpy(), ref_kp) and np.array_equal(vp.cpu().numpy(), ref_vp)
    assert_close(out, lse, ref_o, ref_l)


def test_default_limit_is_restored_by_a_negative_limit():
    wl = CASES["decode-only"]()
    t = W.make_tensors(wl, DEV)
    h = host_copy(t)
    eng = make_engine(wl)
    _prepare(eng, wl, t)
    pva.attn_debug_set_wait_limit(eng.meta, 0)
    pva.attn_debug_set_wait_limit(eng.meta, -1)
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=DEV)
    eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out, lse)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    ref_o, ref_l, _, _ = run_oracle(wl, h)
    assert_close(out, lse, ref_o, ref_l)
