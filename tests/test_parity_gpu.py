"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on the
same seeded inputs.  KV pool bit-exact after the write; bf16 output within max-abs
2e-2 and max-rel 1e-2 (relative to max(|ref|, 1)); LSE within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from harness import assert_close, host_copy, make_engine, pool_bits, run_cuda, run_oracle
from paged_variable_length_gb300 import pva
from paged_variable_length_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _full_check(wl, poison=True, slot_mapping=False, max_q_len=0, engine=None, **eng_kw):
    t = W.make_tensors(wl, DEV, poison_unused=poison)
    h = host_copy(t)
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
    sm = torch.as_tensor(slots, device=DEV) if slot_mapping else None
    eng = engine or make_engine(wl, **eng_kw)
    out, lse, eng = run_cuda(wl, t, engine=eng, slot_mapping=sm, max_q_len=max_q_len)
    ref_o, ref_l, ref_kp, ref_vp = run_oracle(wl, h, slots=slots)
    assert np.array_equal(pool_bits(t["k_pool"]), ref_kp), "K pool differs from the oracle's"
    assert np.array_equal(pool_bits(t["v_pool"]), ref_vp), "V pool differs from the oracle's"
    err = assert_close(out, lse, ref_o, ref_l)
    assert pva.attn_get_device_status(eng.meta) == 0
    return err, eng


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_worked_example(seed):
    _full_check(W.worked_example(seed))


def test_pages_literal_layout():
    """The ch. 5 example layout: H 16, Hkv 8, D 128, page rows 0-5 / 40-43,20-22 / 50-58."""
    table = np.zeros((3, 16), np.int32)
    table[0, :6] = np.arange(6)
    table[1, :7] = [40, 41, 42, 43, 20, 21, 22]
    table[2, :9] = np.arange(50, 59)
    wl = W.Workload("literal", [6, 3, 1], [6, 7, 9], 16, 8, 128, 1, 64, table)
    _full_check(wl, poison=False)
    _full_check(wl, poison=False, slot_mapping=True)


CASES = [
    # (Hq, Hkv, D, ps, q_lens, kv_lens)
    (4, 2, 64, 1, [6, 3, 1], [6, 7, 9]),
    (32, 8, 128, 16, [1, 1, 1, 1, 3], [1, 16, 17, 700, 33]),
    (28, 4, 128, 1, [1, 2, 1, 1], [5, 2, 1000, 257]),
    (8, 8, 64, 4, [1, 9, 0, 16, 1], [3, 20, 5, 16, 77]),
    (32, 8, 128, 16, [40, 1, 130], [40, 2000, 300]),          # prefills and a long decode in one batch
    (16, 1, 128, 32, [1, 5, 1], [4096, 5, 31]),                # MQA
    (16, 16, 64, 2, [1, 1, 7], [9, 1, 7]),                     # MHA (group 1)
    (32, 2, 128, 8, [1, 1], [3000, 5]),                        # group 16
    (32, 16, 128, 128, [1, 1, 70], [3000, 129, 200]),          # two head blocks (Hkv 16), 128-slot pages
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[1]}-{c[2]}-ps{c[3]}-{i}" for i, c in enumerate(CASES)])
@pytest.mark.parametrize("explicit_slots", [False, True])
def test_random_batches(case, explicit_slots):
    Hq, Hkv, D, ps, ql, kl = case
    wl = W.custom(ql, kl, Hq, Hkv, D, ps, seed=len(ql) + D)
    _full_check(wl, slot_mapping=explicit_slots)


def test_split_kv_off_matches_on():
    wl = W.custom([1, 1, 4], [3000, 700, 2500], 32, 8, 128, 16, seed=5)
    e1, _ = _full_check(wl, enable_split_kv=True)
    e2, _ = _full_check(wl, enable_split_kv=False)


def test_many_layers_reuse_one_plan():
    """prepare once, forward per layer (different pools and activations)."""
    wl = W.custom([1, 5, 1, 12], [900, 5, 64, 40], 32, 8, 128, 16, seed=11)
    eng = make_engine(wl)
    t0 = W.make_tensors(wl, DEV)
    eng.prepare(t0["cu_seqlens_q"], t0["cache_seqlens"], t0["page_table"], wl.total_tokens)
    for layer in range(3):
        wl.seed = 100 + layer
        t = W.make_tensors(wl, DEV)
        h = host_copy(t)
        out = torch.empty_like(t["q"])
        lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=DEV)
        eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out, lse)
        torch.cuda.synchronize()
        ref_o, ref_l, ref_kp, _ = run_oracle(wl, h)
        assert np.array_equal(pool_bits(t["k_pool"]), ref_kp)
        assert_close(out, lse, ref_o, ref_l)


def test_deterministic():
    wl = W.custom([1, 1, 3], [5000, 1200, 800], 32, 8, 128, 16, seed=9)
    t = W.make_tensors(wl, DEV)
    outs = []
    for _ in range(2):
        tt = {k: v.clone() for k, v in t.items()}
        out, lse, _ = run_cuda(wl, tt)
        outs.append((out.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_store_only_is_bit_exact():
    wl = W.custom([3, 1, 7], [3, 9, 20], 8, 2, 128, 4, seed=4)
    t = W.make_tensors(wl, DEV)
    h = host_copy(t)
    eng = make_engine(wl)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens)
    pva.attn_store_kvcache(eng.meta, t["k"], t["v"], t["k_pool"], t["v_pool"])
    torch.cuda.synchronize()
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
    kp, vp = oracle.store_kvcache(h["k"], h["v"], slots, h["k_pool"], h["v_pool"])
    assert np.array_equal(pool_bits(t["k_pool"]), kp) and np.array_equal(pool_bits(t["v_pool"]), vp)


def test_padding_slots_are_skipped():
    wl = W.custom([2, 1], [2, 6], 8, 2, 64, 1, seed=6)
    t = W.make_tensors(wl, DEV)
    h = host_copy(t)
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
    slots[1] = -1  # a padding token: not stored
    eng = make_engine(wl)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens,
                torch.as_tensor(slots, device=DEV))
    out = torch.empty_like(t["q"])
    eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out)
    torch.cuda.synchronize()
    kp, _ = oracle.store_kvcache(h["k"], h["v"], slots, h["k_pool"], h["v_pool"])
    assert np.array_equal(pool_bits(t["k_pool"]), kp)


# ------------------------------------------------------------------ device-checked errors


def _error_bits(wl, t, slot_mapping=None, max_q_len=0):
    eng = make_engine(wl)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, slot_mapping, max_q_len)
    out = torch.zeros_like(t["q"])
    eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out)
    return pva.attn_get_device_status(eng.meta), out


def test_q_len_above_kv_len_is_flagged_not_run():
    wl = W.custom([3, 1], [3, 4], 8, 2, 64, 1, seed=1)
    t = W.make_tensors(wl, DEV)
    t["cache_seqlens"][0] = 2  # 3 new tokens but a KV length of 2
    bits, out = _error_bits(wl, t)
    assert bits & 0x02
    assert torch.count_nonzero(out) == 0


def test_decreasing_cu_seqlens_is_flagged():
    wl = W.custom([3, 1], [3, 4], 8, 2, 64, 1, seed=1)
    t = W.make_tensors(wl, DEV)
    t["cu_seqlens_q"][1] = 5
    bits, _ = _error_bits(wl, t)
    assert bits & 0x01


def test_page_id_outside_pool_is_flagged():
    wl = W.custom([1], [40], 8, 2, 64, 4, seed=2)
    t = W.make_tensors(wl, DEV)
    t["page_table"][0, 3] = wl.num_pages + 7
    bits, _ = _error_bits(wl, t)
    assert bits & 0x04


def test_slot_outside_pool_is_flagged():
    wl = W.custom([2], [2], 8, 2, 64, 1, seed=3)
    t = W.make_tensors(wl, DEV)
    sm = torch.tensor([0, wl.num_slots + 3], dtype=torch.int64, device=DEV)
    bits, _ = _error_bits(wl, t, slot_mapping=sm)
    assert bits & 0x08


def test_q_len_above_hint_is_flagged():
    wl = W.custom([5, 1], [9, 4], 8, 2, 64, 1, seed=3)
    t = W.make_tensors(wl, DEV)
    bits, _ = _error_bits(wl, t, max_q_len=2)
    assert bits & 0x10


# ------------------------------------------------------------------ full-size workloads (sampled rows)


def _sampled_check(wl, n_rows=3000, seed=0):
    t = W.make_tensors(wl, DEV)
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
    written = np.unique(slots)
    k_in = t["k"].cpu()
    v_in = t["v"].cpu()
    q_h = t["q"].cpu()
    eng = make_engine(wl)
    out, lse, eng = run_cuda(wl, t, engine=eng, max_q_len=max(wl.q_lens))
    assert pva.attn_get_device_status(eng.meta) == 0
    # pool: the written rows are bit-exact copies of this step's K/V
    kp = t["k_pool"][torch.as_tensor(slots, device=DEV)].cpu()
    vp = t["v_pool"][torch.as_tensor(slots, device=DEV)].cpu()
    assert torch.equal(kp, k_in) and torch.equal(vp, v_in)
    assert written.size == slots.size
    # output: sampled rows recomputed by the oracle over the written pool
    rng = np.random.default_rng(seed)
    T, Hq = wl.total_tokens, wl.num_qo_heads
    sel = np.zeros((T, Hq), bool)
    if T * Hq <= n_rows:
        sel[:] = True
    else:
        idx = rng.choice(T * Hq, size=n_rows, replace=False)
        sel.reshape(-1)[idx] = True
        sel[np.asarray(wl.cu_seqlens_q[1:]) - 1, :] = True  # every request's last token, all heads
    ref_o, ref_l = oracle.attention(q_h, t["k_pool"].cpu(), t["v_pool"].cpu(), wl.cu_seqlens_q, wl.cache_seqlens,
                                    wl.page_table, wl.page_size, row_select=sel)
    return assert_close(out, lse, ref_o, ref_l, mask=sel)


@pytest.mark.parametrize("name", ["decode", "mixed", "cascade", "prefill"])
def test_full_size_workload(name):
    _sampled_check(W.WORKLOADS[name](0))


def test_full_size_prefix_tree():
    """128 decodes: a 2048-token root, 8 branches of 16 sharing 1024 more tokens each."""
    wl = W.cascade_tree(0)
    t = W.make_tensors(wl, DEV)
    eng = make_engine(wl)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] == 9
    _sampled_check(wl)


# ------------------------------------------------------------------ shared-prefix (cascade) path


def _table_workload(q_lens, kv_lens, rows, Hq, Hkv, D, ps, num_pages, seed):
    """A workload with explicit page-table rows (lists of page ids)."""
    width = max(len(r) for r in rows)
    table = np.zeros((len(rows), width), np.int32)
    for i, r in enumerate(rows):
        table[i, :len(r)] = r
    return W.Workload("table", list(q_lens), list(kv_lens), Hq, Hkv, D, ps, num_pages, table, 1.0, seed)


def _cascade_batch(seed=0, Hq=32, Hkv=8, D=128, ps=16):
    """Two prefix groups (12 and 9 shared pages), a member sharing only part of its
    group's prefix, an unrelated decode, a decode too short for a prefix, a prefill."""
    rng = np.random.default_rng(seed)
    P = 400
    perm = list(rng.permutation(P))
    take = lambda k: [int(perm.pop()) for _ in range(k)]
    pre_a, pre_b = take(12), take(9)
    rows, q_lens, kv_lens = [], [], []
    for tail in (1, 5, 16, 40, 17):            # group A: prefix 12 pages, tails of 1..40 keys
        L = 12 * ps + tail
        rows.append(pre_a + take((L + ps - 1) // ps - 12)); q_lens.append(1); kv_lens.append(L)
    for tail in (3, 30, 64):                    # group B
        L = 9 * ps + tail
        rows.append(pre_b + take((L + ps - 1) // ps - 9)); q_lens.append(1); kv_lens.append(L)
    L = 12 * ps + 7                             # shares only 10 of group A's pages
    rows.append(pre_a[:10] + take((L + ps - 1) // ps - 10)); q_lens.append(1); kv_lens.append(L)
    L = 300                                     # unrelated decode
    rows.append(take((L + ps - 1) // ps)); q_lens.append(1); kv_lens.append(L)
    L = 5 * ps                                  # group A's first pages but too short a prefix
    rows.append(pre_a[:5]); q_lens.append(1); kv_lens.append(L)
    L = 200                                     # a prefill in the same batch
    rows.append(take((L + ps - 1) // ps)); q_lens.append(L); kv_lens.append(L)
    return _table_workload(q_lens, kv_lens, rows, Hq, Hkv, D, ps, P, seed)


@pytest.mark.parametrize("seed", [0, 1])
def test_cascade_groups_match_the_oracle(seed):
    wl = _cascade_batch(seed)
    err, eng = _full_check(wl)
    counts = pva.attn_debug_plan_counts(eng.meta)
    assert counts["casc_groups"] == 2 and counts["casc_tiles"] > 0


def test_cascade_on_equals_off_within_tolerance():
    wl = _cascade_batch(3)
    _, eng_on = _full_check(wl, enable_cascade=True)
    _, eng_off = _full_check(wl, enable_cascade=False)
    assert pva.attn_debug_plan_counts(eng_off.meta)["casc_groups"] == 0


def test_cascade_group_size_and_tile_edges():
    """A group larger than one member tile pair (G 4: 32 members per tile) with ragged
    member counts and a prefix that is not a multiple of 128 keys."""
    ps = 16
    rng = np.random.default_rng(7)
    P = 3000
    perm = list(rng.permutation(P))
    take = lambda k: [int(perm.pop()) for _ in range(k)]
    pre = take(27)  # 432 keys
    rows, ql, kl = [], [], []
    for m in range(70):
        tail = int(rng.integers(1, 80))
        L = 27 * ps + tail
        rows.append(pre + take((L + ps - 1) // ps - 27)); ql.append(1); kl.append(L)
    wl = _table_workload(ql, kl, rows, 32, 8, 128, ps, P, 7)
    _, eng = _full_check(wl, poison=True)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] == 1


def test_cascade_with_group_of_seven_heads():
    wl = _cascade_batch(4, Hq=28, Hkv=4, D=128, ps=16)
    _full_check(wl)


def _tree_batch(seed=0, Hq=32, Hkv=8, D=128, ps=16):
    """Two levels of shared prefixes.  Group A (10 root pages) holds sub-group A1 (9 more
    shared pages; one member's query sits right after them), sub-group A2 (12 more pages,
    one member sharing only 8 of them), three members with private pages after the root
    and two sharing only 5 more pages (too short for a sub-group).  Group B (8 root pages)
    holds sub-group B1 (10 more) and one private member.  Plus an unrelated decode and a
    prefill: 2 groups and 3 sub-groups."""
    rng = np.random.default_rng(seed)
    P = 900
    perm = list(rng.permutation(P))
    take = lambda k: [int(perm.pop()) for _ in range(k)]
    rows, q_lens, kv_lens = [], [], []

    def add(shared, tail):
        L = len(shared) * ps + tail
        rows.append(shared + take((L + ps - 1) // ps - len(shared)))
        q_lens.append(1)
        kv_lens.append(L)

    root_a, a1, a2, a5 = take(10), take(9), take(12), take(5)
    for tail in (1, 7, 16, 40, 23):
        add(root_a + a1, tail)
    for tail in (3, 30, 64):
        add(root_a + a2, tail)
    add(root_a + a2[:8], 17)
    for tail in (5, 90, 33):
        add(root_a, tail)
    for tail in (2, 19):
        add(root_a + a5, tail)
    root_b, b1 = take(8), take(10)
    for tail in (11, 48, 1):
        add(root_b + b1, tail)
    add(root_b, 70)
    add([], 300)                                # unrelated decode
    L = 200                                     # a prefill in the same batch
    rows.append(take((L + ps - 1) // ps)); q_lens.append(L); kv_lens.append(L)
    return _table_workload(q_lens, kv_lens, rows, Hq, Hkv, D, ps, P, seed)


@pytest.mark.parametrize("seed", [0, 1])
def test_two_level_prefix_tree_matches_the_oracle(seed):
    wl = _tree_batch(seed)
    _, eng = _full_check(wl)
    counts = pva.attn_debug_plan_counts(eng.meta)
    assert counts["casc_groups"] == 5, counts
    _, eng_off = _full_check(wl, enable_cascade=False)
    assert pva.attn_debug_plan_counts(eng_off.meta)["casc_groups"] == 0


@pytest.mark.parametrize("Hq,Hkv,D", [(28, 4, 128), (16, 4, 64), (32, 32, 128)])
def test_two_level_prefix_tree_head_layouts(Hq, Hkv, D):
    wl = _tree_batch(5, Hq=Hq, Hkv=Hkv, D=D)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] == 5


def _tree3_batch(seed=0, Hq=32, Hkv=8, D=128, ps=16):
    """Three levels of shared prefixes.  Root R (9 pages) holds branch R1 (8 more shared
    pages), in which twig R1a shares 10 more pages (5 members, one cut short after 8 of
    them: the twig's prefix stops at the shortest) and twig R1b 8 more (2 members); R1 also
    has members with private pages after it, and one member goes a fourth level deeper
    (shared with nobody: its tail).  Branch R2 (12 more pages) has 3 members and no twig.
    Plus a member of R alone, an unrelated decode and a prefill: 1 root group, 2 branches,
    2 twigs."""
    rng = np.random.default_rng(seed)
    P = 1200
    perm = list(rng.permutation(P))
    take = lambda k: [int(perm.pop()) for _ in range(k)]
    rows, q_lens, kv_lens = [], [], []

    def add(shared, tail):
        L = len(shared) * ps + tail
        rows.append(shared + take((L + ps - 1) // ps - len(shared)))
        q_lens.append(1)
        kv_lens.append(L)

    root = take(9)
    r1, r2 = root + take(8), root + take(12)
    r1a, r1b = r1 + take(10), r1 + take(8)
    for tail in (1, 17, 40):
        add(r1a, tail)
    add(r1a[:len(r1) + 8], 33)                  # in the twig for 8 of its 10 pages
    for tail in (5, 61):
        add(r1b, tail)
    for tail in (2, 29):
        add(r1, tail)
    add(r1a + take(9), 3)                      # a fourth shared level would start here: nobody shares it
    for tail in (8, 44, 90):
        add(r2, tail)
    add(root, 70)
    add([], 300)                                # unrelated decode
    L = 180                                     # a prefill in the same batch
    rows.append(take((L + ps - 1) // ps)); q_lens.append(L); kv_lens.append(L)
    return _table_workload(q_lens, kv_lens, rows, Hq, Hkv, D, ps, P, seed)


@pytest.mark.parametrize("seed", [0, 1])
def test_three_level_prefix_tree_matches_the_oracle(seed):
    wl = _tree3_batch(seed)
    _, eng = _full_check(wl)
    counts = pva.attn_debug_plan_counts(eng.meta)
    assert counts["casc_groups"] == 5, counts
    _full_check(wl, enable_cascade=False)


@pytest.mark.parametrize("Hq,Hkv,D", [(28, 4, 128), (16, 4, 64)])
def test_three_level_prefix_tree_head_layouts(Hq, Hkv, D):
    wl = _tree3_batch(3, Hq=Hq, Hkv=Hkv, D=D)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] == 5


def test_full_size_three_level_prefix_tree():
    """128 decodes: 1024 shared tokens, 4 branches of 1024 more, 4 twigs of 1024 more each."""
    wl = W.cascade_tree3(0)
    t = W.make_tensors(wl, DEV)
    eng = make_engine(wl)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] == 1 + 4 + 16
    _sampled_check(wl)


def test_full_size_six_level_prefix_tree():
    """128 decodes in a binary prefix tree six levels deep, 512 shared tokens a level."""
    wl = W.cascade_deep(0)
    t = W.make_tensors(wl, DEV)
    eng = make_engine(wl)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens)
    counts = pva.attn_debug_plan_counts(eng.meta)
    assert counts["casc_levels"] == 6 and counts["casc_groups"] == 1 + 2 + 4 + 8 + 16 + 32, counts
    _sampled_check(wl)


def _deep_tree(seed, depth, fanout=2, Hq=32, Hkv=8, D=128, ps=16, min_pages=8):
    """A shared-prefix tree `depth` levels deep: every node extends its parent's pages by a
    run of min_pages to min_pages + 3 pages and has `fanout` child nodes (the deepest
    nodes three single-token decodes each, with private tails); about half of the inner
    nodes (all of them in a chain, fanout 1, where otherwise two levels would share one
    prefix) also have a decode that ends there.  Plus an unrelated decode and a prefill."""
    rng = np.random.default_rng(7000 + seed)
    P = 1500 if ps > 1 else 8000
    perm = [int(x) for x in rng.permutation(P)]
    take = lambda k: [perm.pop() for _ in range(int(k))]
    rows, q_lens, kv_lens = [], [], []

    def add(shared, tail, n=1):
        L = len(shared) * ps + tail
        rows.append(shared + take((L + ps - 1) // ps - len(shared)))
        q_lens.append(n)
        kv_lens.append(L)

    def node(shared, level):
        run = shared + take(rng.integers(min_pages, min_pages + 4))
        if level == depth:
            for _ in range(3):
                add(run, int(rng.integers(1, 60)))
            return
        for _ in range(fanout):
            node(run, level + 1)
        if fanout == 1 or rng.random() < 0.5:
            add(run, int(rng.integers(1, 60)))

    node([], 1)
    add([], 400)                                # unrelated decode
    L = 150                                     # a prefill in the same batch
    rows.append(take((L + ps - 1) // ps)); q_lens.append(L); kv_lens.append(L)
    order = rng.permutation(len(rows))          # requests in any order
    rows = [rows[i] for i in order]
    return _table_workload([q_lens[i] for i in order], [kv_lens[i] for i in order], rows, Hq, Hkv, D, ps, P, seed)


@pytest.mark.parametrize("depth,fanout", [(4, 2), (6, 2), (8, 1)])
def test_deep_prefix_trees(depth, fanout):
    """Trees of 4, 6 and 8 levels: every level is found, and each member merges one
    partial per level with its tail."""
    wl = _deep_tree(depth, depth, fanout)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_levels"] == depth
    _full_check(wl, enable_cascade=False)


def test_prefix_tree_deeper_than_the_levels_found():
    """A chain of 11 nested shared runs: the first eight are prefix levels, the rest are
    read as part of each member's own keys."""
    wl = _deep_tree(11, 11, fanout=1)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_levels"] == 8


@pytest.mark.parametrize("Hq,Hkv,D,ps", [(28, 4, 128, 16), (16, 4, 64, 16), (32, 8, 128, 64), (32, 8, 128, 1)])
def test_deep_prefix_tree_layouts(Hq, Hkv, D, ps):
    wl = _deep_tree(20 + ps, 5, 2, Hq=Hq, Hkv=Hkv, D=D, ps=ps)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_levels"] == 5


def test_sub_group_larger_than_a_tile_pair():
    """A sub-group of 70 members (G 4: 32 member rows per tile) under a 27-page root
    (432 keys: the sub-group's keys start off a 128-key boundary), a second sub-group of
    3, and root members without one."""
    ps = 16
    rng = np.random.default_rng(8)
    P = 4000
    perm = list(rng.permutation(P))
    take = lambda k: [int(perm.pop()) for _ in range(k)]
    root, s1, s2 = take(27), take(13), take(20)
    rows, ql, kl = [], [], []
    for shared, count in ((root + s1, 70), (root + s2, 3), (root, 4)):
        for _ in range(count):
            L = len(shared) * ps + int(rng.integers(1, 80))
            rows.append(shared + take((L + ps - 1) // ps - len(shared))); ql.append(1); kl.append(L)
    wl = _table_workload(ql, kl, rows, 32, 8, 128, ps, P, 8)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] == 3


# ------------------------------------------------------------------ head_dim 64 on the tensor-core path

D64_CASES = [
    # (Hq, Hkv, ps, q_lens, kv_lens): every batch has a request with q_len * G > 16 rows
    (8, 8, 16, [40, 1, 300], [40, 700, 300]),          # MHA: prefills, a decode
    (16, 8, 4, [100, 3, 17], [228, 3, 50]),            # G = 2: chunked prefill on a cached prefix
    (32, 8, 1, [260, 1, 9], [260, 1500, 100]),         # G = 4, token slots
    (28, 4, 16, [129, 255], [1000, 255]),              # G = 7, ragged tiles
]


@pytest.mark.parametrize("case", D64_CASES, ids=[f"d64-{c[0]}-{c[1]}-ps{c[2]}" for c in D64_CASES])
def test_head_dim_64_tensor_core_path(case):
    Hq, Hkv, ps, ql, kl = case
    wl = W.custom(ql, kl, Hq, Hkv, 64, ps, seed=sum(ql))
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["pre_tiles"] > 0


def test_head_dim_64_cascade():
    wl = _cascade_batch(6, Hq=16, Hkv=4, D=64, ps=16)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] > 0


# ------------------------------------------------------------------ speculative-decoding verify batches


@pytest.mark.parametrize("draft,Hq,Hkv", [(1, 32, 8), (3, 32, 8), (7, 32, 8), (3, 28, 4), (3, 64, 8)])
def test_spec_decode_uniform_batches(draft, Hq, Hkv):
    """Every request appends 1 + draft tokens that see the cache and each other causally
    (the decode kernel's groups hold up to 16 / G of them; larger groups split)."""
    rng = np.random.default_rng(draft * 100 + Hq)
    n = 1 + draft
    kl = [int(x) for x in rng.integers(n, 1500, size=12)] + [n, n + 1]  # two with (almost) no cache
    wl = W.custom([n] * len(kl), kl, Hq, Hkv, 128, 16, seed=draft + Hq)
    _full_check(wl, max_q_len=n)
    _full_check(wl)  # without the max_q_len hint


def test_spec_decode_full_size_workload():
    _sampled_check(W.WORKLOADS["specdec"](0))


# ------------------------------------------------------------------ ragged (contiguous) K/V


@pytest.mark.parametrize("case", [
    # (Hq, Hkv, D, q_lens, kv_lens): keys of request i are rows cu_kv[i] .. of k / v
    (32, 8, 128, [300, 1, 77, 1000], [300, 40, 77, 1500]),   # fresh prefills, a decode, a chunk on cache
    (8, 2, 64, [5, 1, 16], [9, 1, 16]),
    (28, 4, 128, [2000, 512], [2000, 512]),
])
def test_ragged_kv_through_the_identity_table(case):
    """FlashInfer's ragged layout: K/V contiguous per request, no pool.  The identity page
    table (page_size 1) and slot -1 for every token address them in place."""
    Hq, Hkv, D, ql, kl = case
    rng = np.random.default_rng(len(ql) + D)
    cu_q = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    cu_kv = np.concatenate([[0], np.cumsum(kl)]).astype(np.int64)
    T, TK = int(cu_q[-1]), int(cu_kv[-1])
    g = torch.Generator(device="cpu").manual_seed(11)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(TK, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(TK, Hkv, D, generator=g).to(torch.bfloat16)
    table, slots = pva.ragged_layout(cu_q, cu_kv, DEV)
    eng = pva.PagedAttention(Hq, Hkv, D, 1, TK, len(ql), T, max(kl))
    dq, dk, dv = q.to(DEV), k.to(DEV), v.to(DEV)
    lens = torch.as_tensor(kl, dtype=torch.int32, device=DEV)
    eng.prepare(torch.as_tensor(cu_q, device=DEV), lens, table, T, slots, max(ql))
    out = torch.empty_like(dq)
    lse = torch.empty(T, Hq, dtype=torch.float32, device=DEV)
    eng.forward(dq, dk, dv, dk, dv, out, lse)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    assert torch.equal(dk.cpu(), k) and torch.equal(dv.cpu(), v), "nothing may be stored"
    ref_o, ref_l = oracle.attention(q, k, v, cu_q, np.asarray(kl, np.int32), table.cpu().numpy(), 1)
    assert_close(out, lse, ref_o, ref_l)


def test_ragged_full_size_workload():
    wl = W.WORKLOADS["ragged"](0)
    t = W.make_tensors(wl, DEV)
    t["k_pool"], t["v_pool"] = t["k"], t["v"]
    eng = make_engine(wl)
    slots = torch.full((wl.total_tokens,), -1, dtype=torch.int64, device=DEV)
    eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, slots, max(wl.q_lens))
    out = torch.empty_like(t["q"])
    lse = torch.empty(wl.total_tokens, wl.num_qo_heads, dtype=torch.float32, device=DEV)
    eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out, lse)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    rng = np.random.default_rng(0)
    T, Hq = wl.total_tokens, wl.num_qo_heads
    sel = np.zeros((T, Hq), bool)
    sel.reshape(-1)[rng.choice(T * Hq, size=2000, replace=False)] = True
    sel[np.asarray(wl.cu_seqlens_q[1:]) - 1, :] = True
    ref_o, ref_l = oracle.attention(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), wl.cu_seqlens_q, wl.cache_seqlens,
                                    wl.page_table, 1, row_select=sel)
    assert_close(out, lse, ref_o, ref_l, mask=sel)


def _random_forest(seed, Hq=32, Hkv=8, D=128, ps=16, min_pages=8, P=4000):
    """Random shared-prefix forests: 1-3 roots of min_pages-1 .. min_pages+5 pages (some too
    short for a group), each with 1-3 branches of min_pages-1 .. min_pages+3 further
    pages, leaves that sometimes share a third run (a third level when long enough) and
    a fourth (a fourth level when long enough), leaves cut short inside a shared run,
    multi-token decodes
    (never prefix members), unrelated decodes and a prefill."""
    rng = np.random.default_rng(1000 + seed)
    rng4 = np.random.default_rng(3000 + seed)
    perm = [int(x) for x in rng.permutation(P)]
    take = lambda k: [perm.pop() for _ in range(int(k))]
    rows, ql, kl = [], [], []

    def add(shared, tail, n=1):
        L = len(shared) * ps + tail
        rows.append(shared + take((L + ps - 1) // ps - len(shared)))
        ql.append(n)
        kl.append(L)

    for _ in range(int(rng.integers(1, 4))):
        root = take(rng.integers(min_pages - 1, min_pages + 6))
        for _ in range(int(rng.integers(1, 5))):
            branch = root + take(rng.integers(min_pages - 1, min_pages + 4))
            third = branch + take(rng.integers(1, 12)) if rng.random() < 0.4 else None
            # (the fourth runs draw from a generator of their own: the forests of the other
            # draws stay what they were)
            fourth = third + take(rng4.integers(1, 12)) if third is not None and rng4.random() < 0.5 else None
            for _ in range(int(rng.integers(2, 7))):
                shared = third if third is not None and rng.random() < 0.6 else branch
                if fourth is not None and shared is third and rng4.random() < 0.5:
                    shared = fourth
                if rng.random() < 0.2:  # shares only part of the run
                    shared = shared[:int(rng.integers(1, len(shared) + 1))]
                n = 1 if rng.random() < 0.85 else int(rng.integers(2, 4))
                add(shared, int(rng.integers(n, 60)), n)
    for _ in range(int(rng.integers(0, 4))):  # unrelated decodes
        add([], int(rng.integers(1, 700)))
    L = int(rng.integers(20, 300))             # a prefill
    rows.append(take((L + ps - 1) // ps)); ql.append(L); kl.append(L)
    order = rng.permutation(len(rows))          # requests in any order
    rows = [rows[i] for i in order]
    ql = [ql[i] for i in order]
    kl = [kl[i] for i in order]
    return _table_workload(ql, kl, rows, Hq, Hkv, D, ps, P, seed)


@pytest.mark.parametrize("seed", range(8))
def test_random_prefix_forests(seed):
    layouts = [(32, 8, 128), (28, 4, 128), (16, 4, 64), (32, 32, 128)]
    Hq, Hkv, D = layouts[seed % len(layouts)]
    wl = _random_forest(seed, Hq=Hq, Hkv=Hkv, D=D)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] >= 1
    _full_check(wl, enable_cascade=False)


@pytest.mark.parametrize("ps,P,seed", [(1, 40000, 0), (1, 40000, 3), (64, 2000, 1), (128, 1000, 2)])
def test_random_prefix_forests_other_page_sizes(ps, P, seed):
    """The same forests over token slots (shared runs of 7 to 30 slots: prefix chunks far
    shorter than a 128-key tile) and over pages of 64 and 128 slots (a shared page holds
    half a tile or a whole one)."""
    wl = _random_forest(seed, ps=ps, P=P)
    _, eng = _full_check(wl)
    assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] >= 1
    _full_check(wl, enable_cascade=False)


# ------------------------------------------------------------------ edge cases


@pytest.mark.parametrize("case", [
    (32, 8, 128, 64, [1, 200, 1, 3], [5000, 260, 64, 3]),   # pages of 64 slots
    (16, 4, 64, 128, [1, 1, 130], [9000, 255, 700]),          # pages of 128 slots, the largest built
])
def test_large_pages(case):
    Hq, Hkv, D, ps, ql, kl = case
    _full_check(W.custom(ql, kl, Hq, Hkv, D, ps, seed=ps))


def test_batch_at_capacity():
    """A batch exactly at the configured max_batch, max_tokens and max_kv_len (the plan's
    capacities at their smallest)."""
    rng = np.random.default_rng(5)
    ql = [1] * 30 + [64, 33]
    kl = [int(x) for x in rng.integers(1, 3000, size=30)] + [64, 3000]
    wl = W.custom(ql, kl, 32, 8, 128, 16, seed=5)
    _full_check(wl, max_batch=wl.batch, max_tokens=wl.total_tokens, max_kv_len=max(kl))


def test_empty_batch_and_no_new_tokens():
    """No request at all, and requests that all bring zero new tokens: prepare and forward
    succeed, write nothing and leave the status clean."""
    wl = W.custom([1, 2], [10, 40], 32, 8, 128, 16, seed=3)
    eng = make_engine(wl)
    t = W.make_tensors(wl, DEV)
    k0, v0 = t["k_pool"].clone(), t["v_pool"].clone()
    out = torch.full_like(t["q"], 7.0)
    none = lambda x: x[:0]  # empty views that keep a valid address
    cu0 = torch.zeros(1, dtype=torch.int32, device=DEV)
    eng.prepare(cu0, none(t["cache_seqlens"]), none(t["page_table"]), 0, None, 0)
    eng.forward(none(t["q"]), none(t["k"]), none(t["v"]), t["k_pool"], t["v_pool"], none(out), None)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    cu = torch.zeros(3, dtype=torch.int32, device=DEV)
    eng.prepare(cu, t["cache_seqlens"], t["page_table"], 0, None, 0)
    eng.forward(none(t["q"]), none(t["k"]), none(t["v"]), t["k_pool"], t["v_pool"], none(out), None)
    torch.cuda.synchronize()
    assert pva.attn_get_device_status(eng.meta) == 0
    assert torch.equal(t["k_pool"], k0) and torch.equal(t["v_pool"], v0)
    assert torch.all(out == 7.0)
