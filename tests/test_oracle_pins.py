"""Pins for the CPU oracle: values the pages print, closed forms, library special
cases and invariants.  None of these retypes the oracle's own formula; each is
chosen so that a plausible slip in the oracle (a dropped scale, a top-left
instead of bottom-right mask, a wrong GQA head map, a swapped page/offset
index, a missing store, a wrong LSE) fails at least one of them.

Runs on the CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _logical_batch(q_lens, cached, Hq, Hkv, D, page_size, seed=0, num_pages=None, junk=float("nan"),
                   qzero=False, const_v=None):
    """Per-request full sequences (as in the ch. 5 example) placed in a paged pool.

    The cached prefix of each request is placed by reshaping the pool to
    [pages, page_size, Hkv, D] and assigning whole pages -- not through any
    slot formula -- so the oracle's own slot arithmetic is checked, not reused.
    The positions of this step's new tokens are left holding ``junk`` until the
    oracle's store writes them.
    """
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    lens = [n + c for n, c in zip(q_lens, cached)]
    need = [math.ceil(L / page_size) for L in lens]
    if num_pages is None:
        num_pages = sum(need) + 5
    perm = rng.permutation(num_pages)
    width = max(need) + 2
    table = np.zeros((len(lens), width), dtype=np.int32)
    off = 0
    for i, p in enumerate(need):
        table[i, :p] = perm[off:off + p]
        off += p
    k_pool = torch.full((num_pages, page_size, Hkv, D), junk, dtype=torch.bfloat16)
    v_pool = torch.full((num_pages, page_size, Hkv, D), junk, dtype=torch.bfloat16)
    full, qs, ks, vs = [], [], [], []
    for i, (n, c) in enumerate(zip(q_lens, cached)):
        L = n + c
        fq = torch.randn(L, Hq, D, generator=g).to(torch.bfloat16)
        fk = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
        fv = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
        if qzero:
            fq.zero_()
        if const_v is not None:
            fv[:] = const_v[None, :, :]
        full.append((fq, fk, fv))
        # place the cached prefix page by page
        pages = table[i, :need[i]]
        padded_k = torch.full((need[i] * page_size, Hkv, D), junk, dtype=torch.bfloat16)
        padded_v = torch.full((need[i] * page_size, Hkv, D), junk, dtype=torch.bfloat16)
        padded_k[:c] = fk[:c]
        padded_v[:c] = fv[:c]
        for p_idx, pid in enumerate(pages):
            k_pool[int(pid)] = padded_k[p_idx * page_size:(p_idx + 1) * page_size]
            v_pool[int(pid)] = padded_v[p_idx * page_size:(p_idx + 1) * page_size]
        qs.append(fq[c:])
        ks.append(fk[c:])
        vs.append(fv[c:])
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return {
        "full": full, "q": torch.cat(qs), "k": torch.cat(ks), "v": torch.cat(vs),
        "k_pool": k_pool.view(-1, Hkv, D), "v_pool": v_pool.view(-1, Hkv, D),
        "cu": cu, "lens": np.asarray(lens, np.int32), "table": table, "page_size": page_size,
        "cached": list(cached), "q_lens": list(q_lens),
    }


def _run(b, scale=None, skip_store=False):
    if skip_store:
        out, lse = oracle.attention(b["q"], b["k_pool"], b["v_pool"], b["cu"], b["lens"], b["table"],
                                    b["page_size"], scale)
        return out, lse
    out, lse, _, _ = oracle.forward(b["q"], b["k"], b["v"], b["k_pool"], b["v_pool"], b["cu"], b["lens"],
                                    b["table"], b["page_size"], scale=scale)
    return out, lse


def _dense_reference(b, D):
    """Complete causal attention per request with torch's SDPA, sliced to the new rows."""
    outs, lses = [], []
    scale = D ** -0.5
    for (fq, fk, fv), c in zip(b["full"], b["cached"]):
        qf, kf, vf = (x.float().transpose(0, 1) for x in (fq, fk, fv))
        o = F.scaled_dot_product_attention(qf, kf, vf, is_causal=True, scale=scale, enable_gqa=True)
        outs.append(o.transpose(0, 1)[c:])
        # LSE from a library reduction over the dense scores, masked with a plain lower triangle
        G = qf.shape[0] // kf.shape[0]
        kr = kf.repeat_interleave(G, dim=0)
        s = torch.matmul(qf.double(), kr.double().transpose(1, 2)) * scale
        L = s.shape[-1]
        tri = torch.ones(L, L, dtype=torch.bool).tril()
        s = s.masked_fill(~tri, float("-inf"))
        lses.append(torch.logsumexp(s, dim=-1).transpose(0, 1)[c:])
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


# ---------------------------------------------------------------- printed values


def test_worked_example_metadata_matches_printout():
    gold = _golden("ch5_worked_example.json")
    st, pr = gold["setup"], gold["printed"]
    table = np.zeros((3, st["page_table_width"]), dtype=np.int32)
    for i, row in enumerate(st["page_table_rows"]):
        table[i, :len(row)] = row
    q_lens, cached = st["q_lens"], st["cached_lens"]
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    lens = np.asarray([n + c for n, c in zip(q_lens, cached)], np.int32)
    assert cu.tolist() == pr["cu_seqlens_q"]
    assert lens.tolist() == pr["cache_seqlens"]
    assert table[:, :lens.max()].tolist() == pr["page_table_cut_to_max_seqlen_k"]
    slots = oracle.slot_mapping(cu, lens, table, st["page_size"])
    assert slots.tolist() == pr["out_loc"]
    assert oracle.last_indices(cu).tolist() == pr["last_indices"]


def test_self_test_mask_example():
    gold = _golden("ch5_worked_example.json")["self_test_mask"]
    m = oracle.causal_mask(gold["q_len"], gold["kv_len"])
    assert np.flatnonzero(m[0]).tolist() == gold["first_query_visible_keys"]
    # the diagonal lands in the bottom-right corner: the last query sees every key
    assert m[-1].all()
    # each later query sees exactly one more key
    assert m.sum(axis=1).tolist() == [5, 6, 7]


def test_mask_special_cases():
    # no prefix (n == L): plain lower triangle; decode (n == 1): all true
    for L in (1, 2, 5, 9):
        assert np.array_equal(oracle.causal_mask(L, L), np.tril(np.ones((L, L), bool)))
        assert oracle.causal_mask(1, L).all()


def test_batch_layout_examples():
    gold = _golden("batch_layout_examples.json")
    for case in gold["cases"]:
        got = oracle.batch_layout([tuple(x) for x in case["items"]])
        for key in ("query_start_loc", "seq_lens", "positions", "logits_indices"):
            assert got[key] == case[key], (case["section"], key)


def test_exercise_3_cu_seqlens():
    # no prefix hit: q lens == kv lens, so cu_q == cu_k; pure decode: [0, 1, ..., bs]
    lens = [5, 3, 8]
    got = oracle.batch_layout([(n, 0, True) for n in lens])
    cu_k = np.concatenate([[0], np.cumsum(got["seq_lens"])]).tolist()
    assert got["query_start_loc"] == cu_k
    dec = oracle.batch_layout([(1, c, True) for c in (4, 9, 2, 7)])
    assert dec["query_start_loc"] == [0, 1, 2, 3, 4]


# ---------------------------------------------------------------- library special cases


@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_pages_literal_layout_vs_dense_causal(page_size):
    """The ch. 5 example (H 16, Hkv 8, D 128, lens 6/7/9 with 0/4/8 cached) against
    complete causal attention; the pages' tolerance is atol 1e-5 in fp32."""
    gold = _golden("ch5_worked_example.json")
    atol = gold["test_tolerance"]["atol"]
    b = _logical_batch([6, 3, 1], [0, 4, 8], 16, 8, 128, page_size, seed=0)
    out, lse = _run(b)
    ref_o, ref_lse = _dense_reference(b, 128)
    assert np.abs(out - ref_o).max() <= atol
    assert np.abs(lse - ref_lse).max() <= 1e-5


@pytest.mark.parametrize("Hq,Hkv,D,ps", [(4, 2, 64, 1), (28, 4, 128, 1), (32, 8, 128, 16), (6, 6, 64, 2)])
def test_random_batches_vs_dense_causal(Hq, Hkv, D, ps):
    """Prefill, chunked prefill and decode in one batch, several GQA group sizes."""
    q_lens = [9, 1, 17, 1, 4]
    cached = [0, 30, 12, 0, 3]
    b = _logical_batch(q_lens, cached, Hq, Hkv, D, ps, seed=3)
    out, lse = _run(b)
    ref_o, ref_lse = _dense_reference(b, D)
    assert np.abs(out - ref_o).max() <= 1e-5
    assert np.abs(lse - ref_lse).max() <= 1e-5


def test_scale_is_used():
    b = _logical_batch([3, 1], [2, 5], 4, 2, 32, 1, seed=5)
    o1, l1 = _run(b)
    o2, l2 = _run(b, scale=0.05)
    assert not np.allclose(o1, o2)
    # with q scaled by s and scale/s the scores are the same (up to rounding of q*s, which is exact here)
    b2 = dict(b)
    b2["q"] = (b["q"].float() * 2.0).to(torch.bfloat16)
    o3, l3 = _run(b2, scale=(32 ** -0.5) / 2.0)
    np.testing.assert_allclose(o3, o1, atol=1e-6)
    np.testing.assert_allclose(l3, l1, atol=1e-6)


def test_fp64_brute_force_tiny():
    """Tiny cases against a float64 numpy evaluation that repeats K/V per q head
    and builds the dense full-sequence softmax, then keeps the new rows."""
    for seed, (ql, cl) in enumerate([([1], [0]), ([2, 1], [3, 6]), ([5, 3], [0, 2])]):
        b = _logical_batch(ql, cl, 4, 2, 8, 2, seed=seed)
        out, lse = _run(b)
        row = 0
        for (fq, fk, fv), c in zip(b["full"], b["cached"]):
            q = fq.double().numpy()
            k = np.repeat(fk.double().numpy(), 2, axis=1)
            v = np.repeat(fv.double().numpy(), 2, axis=1)
            L = q.shape[0]
            for t in range(c, L):
                for h in range(4):
                    s = np.array([(q[t, h] * k[j, h]).sum() / math.sqrt(8) for j in range(t + 1)])
                    w = np.exp(s - s.max())
                    o = (w[:, None] * v[:t + 1, h]).sum(0) / w.sum()
                    assert np.abs(out[row, h] - o).max() < 1e-5
                    assert abs(lse[row, h] - (s.max() + math.log(w.sum()))) < 1e-5
                row += 1


# ---------------------------------------------------------------- closed forms


def test_single_key_returns_its_value():
    b = _logical_batch([1], [0], 4, 2, 16, 1, seed=1)
    out, lse = _run(b)
    fq, fk, fv = b["full"][0]
    # one visible key: p = 1, so O = V_0 exactly and LSE = the single score
    np.testing.assert_array_equal(out[0], np.repeat(fv[0].float().numpy(), 2, axis=0))
    s = (fq[0].double().numpy() * np.repeat(fk[0].double().numpy(), 2, axis=0)).sum(-1) / 4.0
    np.testing.assert_allclose(lse[0], s, atol=1e-5)


def test_zero_query_gives_mean_of_visible_values_and_log_count():
    q_lens, cached = [4, 1, 3], [0, 6, 5]
    b = _logical_batch(q_lens, cached, 4, 2, 16, 2, seed=2, qzero=True)
    out, lse = _run(b)
    row = 0
    for (fq, fk, fv), n, c in zip(b["full"], q_lens, cached):
        L = n + c
        for r in range(n):
            visible = L - n + r + 1
            mean = fv[:visible].double().numpy().mean(axis=0)  # [Hkv, D]
            for h in range(4):
                np.testing.assert_allclose(out[row, h], mean[h // 2], atol=1e-6)
                assert abs(lse[row, h] - math.log(visible)) < 1e-6
            row += 1


def test_constant_values_pass_through():
    const = torch.randn(2, 16, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    b = _logical_batch([5, 1], [3, 7], 6, 2, 16, 4, seed=4, const_v=const)
    b["v"][:] = const[None]
    out, _ = _run(b)
    for h in range(6):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(const[h // 3].float().numpy(), out[:, h].shape),
                                   atol=1e-6)


# ---------------------------------------------------------------- invariants


def test_write_before_read():
    """Skipping the store leaves this step's keys stale (here NaN junk, or a
    different random draw): every request's output changes."""
    b = _logical_batch([6, 3, 1], [0, 4, 8], 4, 2, 64, 1, seed=0, junk=0.0)
    good, _ = _run(b)
    stale, _ = _run(b, skip_store=True)
    cu = b["cu"]
    for i in range(3):
        assert not np.allclose(good[cu[i]:cu[i + 1]], stale[cu[i]:cu[i + 1]])


def test_mixed_batch_equals_each_request_alone():
    q_lens, cached = [7, 1, 12], [0, 5, 10]
    b = _logical_batch(q_lens, cached, 8, 2, 32, 4, seed=6)
    mixed, mixed_lse = _run(b)
    for i in range(3):
        sub = {
            "q": b["q"][b["cu"][i]:b["cu"][i + 1]], "k": b["k"][b["cu"][i]:b["cu"][i + 1]],
            "v": b["v"][b["cu"][i]:b["cu"][i + 1]], "k_pool": b["k_pool"], "v_pool": b["v_pool"],
            "cu": np.array([0, q_lens[i]], np.int32), "lens": b["lens"][i:i + 1],
            "table": b["table"][i:i + 1], "page_size": 4,
        }
        alone, alone_lse = _run(sub)
        np.testing.assert_array_equal(alone, mixed[b["cu"][i]:b["cu"][i + 1]])
        np.testing.assert_array_equal(alone_lse, mixed_lse[b["cu"][i]:b["cu"][i + 1]])


def test_page_placement_does_not_matter():
    """Moving every page to another id (and rewriting the table) changes nothing."""
    b = _logical_batch([4, 2], [8, 3], 4, 2, 16, 4, seed=7)
    out, lse = _run(b)
    P = b["k_pool"].shape[0] // 4
    perm = np.random.default_rng(11).permutation(P)
    kp = torch.empty_like(b["k_pool"]).view(P, 4, 2, 16)
    vp = torch.empty_like(b["v_pool"]).view(P, 4, 2, 16)
    kp[torch.as_tensor(perm)] = b["k_pool"].view(P, 4, 2, 16)
    vp[torch.as_tensor(perm)] = b["v_pool"].view(P, 4, 2, 16)
    moved = dict(b, k_pool=kp.view(-1, 2, 16), v_pool=vp.view(-1, 2, 16), table=perm[b["table"]].astype(np.int32))
    out2, lse2 = _run(moved)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_row_select_computes_only_marked_rows():
    b = _logical_batch([5, 2], [1, 4], 4, 2, 16, 2, seed=8)
    full, full_lse = _run(b)
    sel = np.zeros((7, 4), bool)
    sel[1, 2] = sel[6, 0] = True
    kp, vp = oracle.store_kvcache(b["k"], b["v"], oracle.slot_mapping(b["cu"], b["lens"], b["table"], 2),
                                  b["k_pool"], b["v_pool"])
    part, part_lse = oracle.attention(b["q"], kp, vp, b["cu"], b["lens"], b["table"], 2, row_select=sel)
    np.testing.assert_array_equal(part[sel], full[sel])
    np.testing.assert_array_equal(part_lse[sel], full_lse[sel])
    assert np.isnan(part[~sel]).all()


def test_split_and_merge_by_lse_equals_full():
    """The LSE merge reading: attention over keys [0,a) and [a,L) combined as
    lse = logaddexp(lse_1, lse_2), o = e^(lse_1-lse) o_1 + e^(lse_2-lse) o_2,
    equals attention over [0,L).  Checked with single-request decode batches
    whose page tables cover the two key ranges separately."""
    Hq, Hkv, D, ps = 4, 2, 16, 1
    g = torch.Generator().manual_seed(12)
    L, a = 11, 4
    q = torch.randn(1, Hq, D, generator=g).to(torch.bfloat16)
    k_pool = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    v_pool = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    cu = np.array([0, 1], np.int32)
    full_o, full_l = oracle.attention(q, k_pool, v_pool, cu, np.array([L], np.int32),
                                      np.arange(L, dtype=np.int32)[None], ps)
    o1, l1 = oracle.attention(q, k_pool, v_pool, cu, np.array([a], np.int32),
                              np.arange(a, dtype=np.int32)[None], ps)
    o2, l2 = oracle.attention(q, k_pool, v_pool, cu, np.array([L - a], np.int32),
                              np.arange(a, L, dtype=np.int32)[None], ps)
    lse = np.logaddexp(l1.astype(np.float64), l2.astype(np.float64))
    o = np.exp(l1 - lse)[..., None] * o1 + np.exp(l2 - lse)[..., None] * o2
    np.testing.assert_allclose(o, full_o, atol=1e-5)
    np.testing.assert_allclose(lse, full_l, atol=1e-5)


# ---------------------------------------------------------------- store + validation


def test_store_is_a_bit_exact_scatter():
    rng = np.random.default_rng(0)
    T, Hkv, D, S = 9, 2, 8, 40
    k = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
    kp0 = rng.integers(0, 65536, size=(S, Hkv, D), dtype=np.uint16)
    vp0 = rng.integers(0, 65536, size=(S, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(S)[:T].astype(np.int64)
    slots[3] = -1  # padding token: no write
    kp, vp = oracle.store_kvcache(k, v, slots, kp0, vp0)
    for t in range(T):
        if slots[t] >= 0:
            assert np.array_equal(kp[slots[t]], k[t]) and np.array_equal(vp[slots[t]], v[t])
    untouched = np.setdiff1d(np.arange(S), slots[slots >= 0])
    assert np.array_equal(kp[untouched], kp0[untouched]) and np.array_equal(vp[untouched], vp0[untouched])
    bad = slots.copy()
    bad[0] = S
    with pytest.raises(oracle.OracleError):
        oracle.store_kvcache(k, v, bad, kp0, vp0)


def test_rejects_more_queries_than_keys():
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(np.array([0, 5], np.int32), np.array([4], np.int32), np.zeros((1, 4), np.int32), 1)
    q = torch.zeros(5, 2, 8, dtype=torch.bfloat16)
    pool = torch.zeros(8, 1, 8, dtype=torch.bfloat16)
    with pytest.raises(oracle.OracleError):
        oracle.attention(q, pool, pool, np.array([0, 5], np.int32), np.array([4], np.int32),
                         np.zeros((1, 8), np.int32), 1)


def test_rejects_page_ids_outside_the_pool():
    q = torch.zeros(1, 2, 8, dtype=torch.bfloat16)
    pool = torch.zeros(8, 1, 8, dtype=torch.bfloat16)
    table = np.array([[0, 1, 9]], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.attention(q, pool, pool, np.array([0, 1], np.int32), np.array([3], np.int32), table, 1)
    # junk columns beyond kv_len are never read, even if out of range
    out, _ = oracle.attention(q, pool, pool, np.array([0, 1], np.int32), np.array([2], np.int32), table, 1)
    assert np.isfinite(out).all()


def test_empty_requests_are_skipped():
    b = _logical_batch([3, 2], [1, 2], 4, 2, 16, 1, seed=10)
    # insert a request with no new tokens (n = 0) between the two
    cu = np.array([0, 3, 3, 5], np.int32)
    lens = np.array([4, 5, 4], np.int32)
    table = np.stack([b["table"][0], b["table"][0], b["table"][1]])
    out, _, _, _ = oracle.forward(b["q"], b["k"], b["v"], b["k_pool"], b["v_pool"], cu, lens, table, 1)
    ref, _ = _run(b)
    np.testing.assert_array_equal(out, ref)


def test_padding_waste_example():
    gold = _golden("batch_layout_examples.json")["padding_waste"]
    ql = gold["query_lens"]
    padded, real = len(ql) * max(ql), sum(ql)
    assert (padded, real) == (gold["padded"], gold["real"])
    assert round(100 * (1 - real / padded)) == gold["waste_percent"]


# --------------------------------------------------------------------------- FP8 (E4M3) pool

E4M3_POINTS = [
    # (code, value) straight from the format definition: bias 7, 3 mantissa bits,
    # subnormals m * 2^-9, S.1111.111 the only NaN, largest finite 1.75 * 2^8
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x0F, 1.875 * 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x77, 1.875 * 2.0 ** 7), (0x7E, 448.0),
    (0x80, -0.0), (0xB8, -1.0), (0xFE, -448.0),
]


def test_e4m3_decode_format_points():
    codes = np.array([c for c, _ in E4M3_POINTS], np.uint8)
    got = oracle.e4m3_decode(codes)
    for (c, v), g in zip(E4M3_POINTS, got):
        assert g == v and math.copysign(1.0, g) == math.copysign(1.0, v), hex(c)
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_encode_rounding_and_saturation():
    cases = [
        (1.0, 0x38), (448.0, 0x7E), (449.0, 0x7E), (1e6, 0x7E), (np.inf, 0x7E), (-np.inf, 0xFE),
        (2.0 ** -10, 0x00),          # half the smallest subnormal: tie, to the even code 0
        (3 * 2.0 ** -10, 0x02),      # 1.5 quanta: tie between codes 1 and 2, to the even 2
        (2.0 ** -10 * 1.01, 0x01),   # just above the tie
        (1.0625, 0x38),              # halfway 1.0 / 1.125: even mantissa 0
        (1.1875, 0x3A),              # halfway 1.125 / 1.25: even mantissa 2
        (-0.0, 0x80), (-1e-30, 0x80),
        (15.5, 0x58),                # quantum 1 in [8, 16): a tie between 15 (0x57) and 16 (0x58), even 16
    ]
    got = oracle.e4m3_encode(np.array([x for x, _ in cases], np.float32))
    for (x, c), g in zip(cases, got):
        assert g == c, (x, hex(c), hex(g))
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_e4m3_round_trip_every_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_e4m3_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-460, 460, 3000), rng.normal(0, 1, 3000), rng.normal(0, 0.01, 3000)])
    x = x.astype(np.float32)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(finite).astype(np.float64)
    got = oracle.e4m3_decode(oracle.e4m3_encode(x)).astype(np.float64)
    clipped = np.clip(x.astype(np.float64), -448, 448)
    best = np.min(np.abs(vals[None, :] - clipped[:, None]), axis=1)
    assert np.array_equal(np.abs(got - clipped), best)


def test_e4m3_encode_matches_torch_in_range():
    """torch's float8_e4m3fn conversion (round to nearest even) is an independent
    implementation for values inside the finite range."""
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None:
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.uniform(-440, 440, 5000), rng.normal(0, 1, 5000), rng.normal(0, 0.003, 5000)])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(f8).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_fp8_store_quantises_each_head_with_its_scale():
    rng = np.random.default_rng(5)
    T, Hkv, D = 3, 2, 8
    k = torch.from_numpy(rng.normal(0, 3, (T, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.normal(0, 3, (T, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    ks, vs = np.array([0.5, 2.0], np.float32), np.array([4.0, 0.25], np.float32)
    kp = np.full((10, Hkv, D), 0x7F, np.uint8)
    vp = np.full((10, Hkv, D), 0x7F, np.uint8)
    slots = np.array([7, -1, 2], np.int64)
    kq, vq = oracle.store_kvcache_fp8(k, v, slots, kp, vp, ks, vs)
    # untouched slots keep their bytes; slot -1 writes nothing
    untouched = [s for s in range(10) if s not in (7, 2)]
    assert (kq[untouched] == 0x7F).all() and (vq[untouched] == 0x7F).all()
    # the written rows decode to the inputs within half a quantum (scales are powers of
    # two, so the quotient is exact), and each head uses its own scale
    for t, s in ((0, 7), (2, 2)):
        for h in range(Hkv):
            kx = k[t, h].float().numpy() / ks[h]
            back = oracle.e4m3_decode(kq[s, h])
            q = np.where(np.abs(kx) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(kx), 1e-30))) - 3))
            assert (np.abs(back - kx) <= q / 2 + 1e-12).all()
            assert (np.abs(oracle.e4m3_decode(vq[s, h]) * vs[h] - v[t, h].float().numpy()) <=
                    np.abs(v[t, h].float().numpy()) * 2.0 ** -4 + 2.0 ** -9 * vs[h]).all()


def test_fp8_attention_reduces_to_bf16_attention_on_exact_values():
    """K/V values that are E4M3 values times power-of-two scales are stored exactly, so
    the FP8 step must equal the (pinned) bf16 step on the same values."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, ps = 3, 4, 2, 16, 4
    q_lens, kv_lens = [3, 1, 5], [9, 13, 5]
    pages = [math.ceil(L / ps) for L in kv_lens]
    P = sum(pages) + 2
    pt = np.zeros((B, max(pages)), np.int32)
    perm = rng.permutation(P)
    off = 0
    for i, n in enumerate(pages):
        pt[i, :n] = perm[off:off + n]
        off += n
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    lens = np.array(kv_lens, np.int32)
    T = int(cu[-1])
    ks, vs = np.array([0.5, 4.0], np.float32), np.array([2.0, 0.125], np.float32)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)

    def exact(shape, scale_per_head):
        codes = rng.choice(finite, size=shape)
        return oracle.e4m3_decode(codes) * scale_per_head[None, :, None]

    q = torch.from_numpy(rng.normal(0, 1, (T, Hq, D)).astype(np.float32)).to(torch.bfloat16)
    # e4m3 values times a power-of-two scale: exact in bf16 and exact after division by the scale
    k = exact((T, Hkv, D), ks)
    v = exact((T, Hkv, D), vs)
    kp0, vp0 = exact((P * ps, Hkv, D), ks), exact((P * ps, Hkv, D), vs)
    kb, vb = (torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16) for a in (k, v))
    kpb, vpb = (torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16) for a in (kp0, vp0))
    # the same values as bf16 (exact: e4m3 has 3 mantissa bits) and as FP8 codes
    assert np.array_equal(kb.float().numpy(), k) and np.array_equal(kpb.float().numpy(), kp0)
    kp8 = oracle.e4m3_encode(kp0 / ks[None, :, None])
    vp8 = oracle.e4m3_encode(vp0 / vs[None, :, None])
    o8, l8, kq, vq = oracle.forward_fp8(q, kb, vb, kp8, vp8, ks, vs, cu, lens, pt, ps)
    o16, l16, kq16, vq16 = oracle.forward(q, kb, vb, kpb, vpb, cu, lens, pt, ps)
    assert np.array_equal(oracle.e4m3_decode(kq) * ks[None, :, None],
                          torch.from_numpy(kq16.view(np.int16)).view(torch.bfloat16).float().numpy())
    np.testing.assert_allclose(o8, o16, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(l8, l16, rtol=1e-6, atol=1e-6)
