"""attn_prepare_metadata_static -- the plan in the library's built-in scratch area, no
workspace allocated -- against the workspace entry point on the same batch: the KV
pool bit-exact, the bf16 output within the parity bar of the other tests (max-abs 2e-2,
max-rel 1e-2 against max(|ref|, 1)) and the LSE within 1e-3 of the workspace path's, on
two calls in a row.  Collected last so that it also runs
after every other GPU test in one session.
"""
import pytest
import torch

from paged_variable_length_gb300 import pva
from paged_variable_length_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
MAX_ABS, MAX_REL, LSE_ATOL = 2e-2, 1e-2, 1e-3

CASES = {
    "worked": lambda: W.worked_example(0),
    "decode-splits": lambda: W.custom([1, 1, 3, 1, 1], [700, 33, 40, 2500, 1], 32, 8, 128, 16, seed=3),
    "prefill-and-decode": lambda: W.custom([40, 1, 130], [40, 2000, 300], 32, 8, 128, 16, seed=4),
    "shared-prefix": lambda: W.custom([1] * 6, [300, 310, 290, 400, 333, 301], 32, 8, 128, 16, seed=5,
                                      shared_prefix_pages=16),
    "decode-full-size": lambda: W.decode_only(0),
}


def _config(wl, **kw):
    limits = dict(max_batch=wl.batch, max_tokens=wl.total_tokens, max_kv_len=max(wl.kv_lens))
    limits.update(kw)
    return pva.make_config(wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages, **limits)


def _compare(wl, cfg):
    t = W.make_tensors(wl, DEV)
    pools = (t["k_pool"].clone(), t["v_pool"].clone())
    args = (t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], None, wl.batch, wl.total_tokens,
            max(wl.q_lens))
    ws = torch.empty(pva.attn_workspace_size(cfg), dtype=torch.uint8, device=DEV)
    ref_out, ref_lse, ref_kp, ref_vp = _forward(pva.attn_prepare_metadata(cfg, *args, ws), t, pools)
    for _ in range(2):
        out, lse, kp, vp = _forward(pva.attn_prepare_metadata_static(cfg, *args), t, pools)
        assert torch.equal(kp, ref_kp) and torch.equal(vp, ref_vp)
        d = (out.float() - ref_out.float()).abs()
        assert float(d.max()) <= MAX_ABS
        assert float((d / ref_out.float().abs().clamp(min=1.0)).max()) <= MAX_REL
        assert float((lse - ref_lse).abs().max()) <= LSE_ATOL


def _forward(meta, t, pools):
    k_pool, v_pool = pools[0].clone(), pools[1].clone()
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=DEV)
    pva.attn_forward(meta, t["q"], t["k"], t["v"], k_pool, v_pool, out, lse)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(meta) == 0
    return out, lse, k_pool, v_pool


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_workspace_path(name):
    wl = CASES[name]()
    _compare(wl, _config(wl))


def test_static_scratch_with_fewer_units_than_decode_ctas():
    # Two kv heads: four decode CTAs per SM.  Limits whose default plan needs more than the
    # scratch area, so the static call plans fewer split-KV units than decode CTAs; the
    # decode-only batch must then take the unit queue, not the balanced split (whose cuts
    # need more partial slots than such a plan holds).
    wl = W.custom([1] * 40, [1000 + 50 * i for i in range(40)], 16, 2, 128, 16, seed=6)
    cfg = _config(wl, max_batch=64, max_tokens=700_000, enable_cascade=False)
    assert pva.attn_workspace_size(cfg) > 64 << 20
    _compare(wl, cfg)


def test_plan_too_large_for_the_scratch_area_is_refused():
    wl = W.worked_example(0)
    t = W.make_tensors(wl, DEV)
    cfg = pva.make_config(wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages,
                          max_batch=wl.batch, max_tokens=8_000_000, max_kv_len=max(wl.kv_lens))
    with pytest.raises(pva.PvaError) as e:
        pva.attn_prepare_metadata_static(cfg, t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], None,
                                         wl.batch, wl.total_tokens, max(wl.q_lens))
    assert e.value.status == 3  # PVA_ERR_WORKSPACE_TOO_SMALL
