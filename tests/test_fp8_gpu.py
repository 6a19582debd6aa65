"""GPU parity of the FP8 (E4M3) KV pool path against the CPU oracle.

The pool after the quantising store is compared byte for byte (the quantisation is
integer-valued work: one E4M3 code per element); the output against the oracle's
fp32 attention over e4m3 * scale within the same bar as the bf16 path (max-abs 2e-2,
max-rel 1e-2 relative to max(|ref|, 1)) (the kernels' f16 operands hold every E4M3 value, the activations' bf16 values
and P more finely than the bf16 path does); LSE within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from harness import assert_close, make_engine
from paged_variable_length_gb300 import pva
from paged_variable_length_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _fp8_case(wl, slot_mapping=False, max_q_len=0, **eng_kw):
    t = W.make_tensors(wl, DEV)
    kp, vp, ks, vs = W.make_fp8_pools(wl, DEV, poison_unused=True)
    h = {name: x.detach().cpu().clone() for name, x in dict(t, kp=kp, vp=vp, ks=ks, vs=vs).items()}
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
    sm = torch.as_tensor(slots, device=DEV) if slot_mapping else None
    eng = make_engine(wl, kv_dtype=pva.KV_E4M3, **eng_kw)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, sm, max_q_len)
    out = torch.empty_like(t["q"])
    lse = torch.empty(wl.total_tokens, wl.num_qo_heads, dtype=torch.float32, device=DEV)
    eng.forward(t["q"], t["k"], t["v"], kp, vp, out, lse, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    ref_o, ref_l, ref_kp, ref_vp = oracle.forward_fp8(
        h["q"], h["k"], h["v"], h["kp"], h["vp"], h["ks"], h["vs"], h["cu_seqlens_q"].numpy(),
        h["cache_seqlens"].numpy(), h["page_table"].numpy(), wl.page_size, slots=slots)
    assert np.array_equal(kp.cpu().numpy(), ref_kp), "K pool codes differ from the oracle's"
    assert np.array_equal(vp.cpu().numpy(), ref_vp), "V pool codes differ from the oracle's"
    return assert_close(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("seed", [0, 1])
def test_fp8_worked_example(seed):
    _fp8_case(W.worked_example(seed))


CASES = [
    # (Hq, Hkv, D, ps, q_lens, kv_lens)
    (32, 8, 128, 16, [1, 1, 1, 1, 3], [1, 16, 17, 700, 33]),
    (28, 4, 128, 1, [1, 2, 1, 1], [5, 2, 1000, 257]),
    (8, 8, 64, 4, [1, 9, 0, 16, 1], [3, 20, 5, 16, 77]),
    (32, 8, 128, 16, [40, 1, 130], [40, 2000, 300]),      # prefills and a chunk (tensor-core kernel)
    (16, 1, 128, 32, [1, 5, 1], [4096, 5, 31]),            # MQA
    (16, 16, 64, 2, [1, 1, 7], [9, 1, 7]),                 # MHA
    (32, 2, 128, 8, [1, 1], [3000, 5]),                    # group 16
    (32, 8, 128, 64, [1, 200, 1, 3], [5000, 260, 64, 3]),  # pages of 64 slots
    (32, 16, 128, 128, [1, 1, 70], [3000, 129, 200]),      # pages of 128 slots, two head blocks
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[1]}-{c[2]}-ps{c[3]}-{i}" for i, c in enumerate(CASES)])
def test_fp8_random_batches(case):
    Hq, Hkv, D, ps, ql, kl = case
    wl = W.custom(ql, kl, Hq, Hkv, D, ps, seed=len(ql) + D + 1)
    _fp8_case(wl)


def test_fp8_explicit_slots_and_no_split():
    wl = W.custom([1, 1, 4], [3000, 700, 2500], 32, 8, 128, 16, seed=5)
    _fp8_case(wl, slot_mapping=True)
    _fp8_case(wl, enable_split_kv=False)


def test_fp8_entry_points_refuse_the_other_pool_type():
    wl = W.custom([1, 3], [40, 9], 8, 2, 64, 4, seed=3)
    t = W.make_tensors(wl, DEV)
    kp, vp, ks, vs = W.make_fp8_pools(wl, DEV)
    out = torch.empty_like(t["q"])
    e8 = make_engine(wl, kv_dtype=pva.KV_E4M3)
    e8.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens)
    with pytest.raises(pva.PvaError):
        pva.attn_forward(e8.meta, t["q"], t["k"], t["v"], kp, vp, out)
    with pytest.raises(pva.PvaError):
        pva.attn_forward_fp8kv(e8.meta, t["q"], t["k"], t["v"], kp, vp, None, vs, out)
    e16 = make_engine(wl)
    e16.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens)
    with pytest.raises(pva.PvaError):
        pva.attn_forward_fp8kv(e16.meta, t["q"], t["k"], t["v"], kp, vp, ks, vs, out)
    # the config check: only the two pool types exist
    assert pva.attn_workspace_size(pva.make_config(8, 2, 64, 4, 100, 4, 16, 64, kv_dtype=pva.KV_E4M3)) > 0
    assert pva.attn_workspace_size(pva.make_config(8, 2, 64, 4, 100, 4, 16, 64, kv_dtype=7)) == 0


def test_fp8_full_size_decode_workload_sampled_rows():
    """The bench's decode workload (64 requests, kv_len U[512, 4096], 32/8/128, ps 16) over an
    FP8 pool: written slots bit-exact, 3000 sampled rows (and every request's last token)
    against the oracle."""
    wl = W.WORKLOADS["decode"](0)
    t = W.make_tensors(wl, DEV)
    kp, vp, ks, vs = W.make_fp8_pools(wl, DEV)
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
    eng = make_engine(wl, kv_dtype=pva.KV_E4M3)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, None, max(wl.q_lens))
    out = torch.empty_like(t["q"])
    lse = torch.empty(wl.total_tokens, wl.num_qo_heads, dtype=torch.float32, device=DEV)
    eng.forward(t["q"], t["k"], t["v"], kp, vp, out, lse, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    sl = torch.as_tensor(slots, device=DEV)
    ref_k = oracle.e4m3_encode(t["k"].float().cpu().numpy() / ks.cpu().numpy()[None, :, None])
    ref_v = oracle.e4m3_encode(t["v"].float().cpu().numpy() / vs.cpu().numpy()[None, :, None])
    assert np.array_equal(kp[sl].cpu().numpy(), ref_k) and np.array_equal(vp[sl].cpu().numpy(), ref_v)
    rng = np.random.default_rng(0)
    T, Hq = wl.total_tokens, wl.num_qo_heads
    sel = np.zeros((T, Hq), bool)
    sel.reshape(-1)[rng.choice(T * Hq, size=min(1000, T * Hq), replace=False)] = True
    sel[np.asarray(wl.cu_seqlens_q[1:]) - 1, :] = True
    ref_o, ref_l = oracle.attention_fp8(t["q"].cpu(), kp.cpu(), vp.cpu(), ks.cpu(), vs.cpu(), wl.cu_seqlens_q,
                                        wl.cache_seqlens, wl.page_table, wl.page_size, row_select=sel)
    assert_close(out, lse, ref_o, ref_l, mask=sel)


def _fp8_sampled(wl, n_rows=1500, seed=0):
    """Full-size FP8 workload: written slots byte-exact, sampled rows (and every request's
    last token) against the oracle over the written pool."""
    t = W.make_tensors(wl, DEV)
    kp, vp, ks, vs = W.make_fp8_pools(wl, DEV)
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
    eng = make_engine(wl, kv_dtype=pva.KV_E4M3)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, None, max(wl.q_lens))
    out = torch.empty_like(t["q"])
    lse = torch.empty(wl.total_tokens, wl.num_qo_heads, dtype=torch.float32, device=DEV)
    eng.forward(t["q"], t["k"], t["v"], kp, vp, out, lse, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    sl = torch.as_tensor(slots, device=DEV)
    ref_k = oracle.e4m3_encode(t["k"].float().cpu().numpy() / ks.cpu().numpy()[None, :, None])
    ref_v = oracle.e4m3_encode(t["v"].float().cpu().numpy() / vs.cpu().numpy()[None, :, None])
    assert np.array_equal(kp[sl].cpu().numpy(), ref_k) and np.array_equal(vp[sl].cpu().numpy(), ref_v)
    rng = np.random.default_rng(seed)
    T, Hq = wl.total_tokens, wl.num_qo_heads
    sel = np.zeros((T, Hq), bool)
    sel.reshape(-1)[rng.choice(T * Hq, size=min(n_rows, T * Hq), replace=False)] = True
    sel[np.asarray(wl.cu_seqlens_q[1:]) - 1, :] = True
    ref_o, ref_l = oracle.attention_fp8(t["q"].cpu(), kp.cpu(), vp.cpu(), ks.cpu(), vs.cpu(), wl.cu_seqlens_q,
                                        wl.cache_seqlens, wl.page_table, wl.page_size, row_select=sel)
    assert_close(out, lse, ref_o, ref_l, mask=sel)
    return pva.attn_debug_plan_counts(eng.meta)


@pytest.mark.parametrize("name", ["prefill", "mixed", "cascade", "cascade_tree", "cascade_tree3", "cascade_deep",
                                  "specdec"])
def test_fp8_full_size_workloads(name):
    counts = _fp8_sampled(W.WORKLOADS[name](0))
    if name == "cascade":
        assert counts["casc_groups"] >= 1, "the shared prefix should run as a prefix pass"
    if name == "cascade_tree":
        assert counts["casc_groups"] == 9, "a root group and 8 branch sub-groups"
    if name == "cascade_tree3":
        assert counts["casc_groups"] == 21, "a root group, 4 branches and 16 twigs"
    if name == "cascade_deep":
        assert counts["casc_levels"] == 6, "a binary tree six levels deep"
    if name in ("prefill", "mixed"):
        assert counts["pre_tiles"] > 0, "prefills should run on the tensor-core kernel"


def test_fp8_shared_prefix_groups():
    """Two prefix groups, a member sharing only part of its group's prefix, an unrelated
    decode, a too-short request and a prefill in one FP8 batch (prefix pass + merge)."""
    from test_parity_gpu import _cascade_batch

    wl = _cascade_batch(seed=4)
    _fp8_case(wl)
    _fp8_case(wl, enable_cascade=False)


def test_fp8_three_level_prefix_tree():
    """Three levels of shared prefixes (two twigs under one branch, a partial sharer, a
    member a level deeper than any group) in one FP8 batch."""
    from test_parity_gpu import _tree3_batch

    _fp8_case(_tree3_batch(seed=4))


def test_fp8_two_level_prefix_tree():
    """Two groups with three sub-groups beneath them (partial sharers, members without a
    sub-group, a prefill) in one FP8 batch."""
    from test_parity_gpu import _tree_batch

    wl = _tree_batch(seed=2)
    _fp8_case(wl)


def test_fp8_deep_prefix_tree():
    """Six levels of shared prefixes (two child runs under every node) in one FP8 batch."""
    from test_parity_gpu import _deep_tree

    wl = _deep_tree(31, 6, 2)
    t = W.make_tensors(wl, DEV)
    eng = make_engine(wl, kv_dtype=pva.KV_E4M3)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_levels"] == 6
    _fp8_case(wl)
