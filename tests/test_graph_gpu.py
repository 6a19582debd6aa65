"""CUDA-graph capture and replay of a whole step (prepare + forward).

The library allocates nothing, never synchronises the stream and reads no device
value on the host inside either call, so one step captured into a graph replays
with whatever the captured buffers hold at replay time: new batch indices (same
shapes), new activations and new pools.  After each replay the pools must match the
oracle's bit for bit and the output must be within the parity tolerance.
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
FIELDS = ["cu_seqlens_q", "cache_seqlens", "page_table", "q", "k", "v", "k_pool", "v_pool"]

SHAPES = [
    # (q_lens, kv_lens, Hq, Hkv, D, ps, shared_prefix_pages)
    ([1, 1, 40, 1, 130], [700, 33, 40, 2000, 300], 32, 8, 128, 16, 0),   # decodes, prefills, a chunk
    ([1] * 24, [300 + 7 * i for i in range(24)], 32, 8, 128, 16, 16),    # shared 256-token prefix
    ([1, 2, 1, 9], [5, 2, 1000, 257], 28, 4, 128, 1, 0),                  # token-slot pool
]


@pytest.mark.parametrize("shape", SHAPES, ids=["mixed-ps16", "cascade", "mixed-ps1"])
def test_graph_replay_with_new_inputs(shape):
    ql, kl, Hq, Hkv, D, ps, spp = shape
    wl0 = W.custom(ql, kl, Hq, Hkv, D, ps, seed=100, shared_prefix_pages=spp)
    t = W.make_tensors(wl0, DEV, poison_unused=True)
    eng = make_engine(wl0)
    out = torch.empty_like(t["q"])
    lse = torch.empty(wl0.total_tokens, Hq, dtype=torch.float32, device=DEV)

    def step():
        eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl0.total_tokens, None, 0)
        eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out, lse)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture (module loading, first-launch attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed in (101, 102):
        wl = W.custom(ql, kl, Hq, Hkv, D, ps, seed=seed, shared_prefix_pages=spp)
        assert wl.num_pages == wl0.num_pages and wl.page_table.shape == wl0.page_table.shape
        fresh = W.make_tensors(wl, DEV, poison_unused=True)
        for f in FIELDS:
            t[f].copy_(fresh[f])
        h = host_copy(fresh)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.cache_seqlens, wl.page_table, wl.page_size)
        ref_o, ref_l, ref_kp, ref_vp = run_oracle(wl, h, slots=slots)
        assert np.array_equal(pool_bits(t["k_pool"]), ref_kp), "K pool differs from the oracle's"
        assert np.array_equal(pool_bits(t["v_pool"]), ref_vp), "V pool differs from the oracle's"
        assert_close(out, lse, ref_o, ref_l)
        assert pva.attn_get_device_status(eng.meta) == 0
        if spp:
            assert pva.attn_debug_plan_counts(eng.meta)["casc_groups"] >= 1, "no shared-prefix group under replay"


def test_graph_replay_is_idempotent():
    """Replaying the same step twice leaves the pools and the output unchanged: the
    store writes the same rows, and attention reads them after the write."""
    wl = W.custom([1, 5, 1, 12], [900, 5, 64, 40], 32, 8, 128, 16, seed=7)
    t = W.make_tensors(wl, DEV)
    eng = make_engine(wl)
    out = torch.empty_like(t["q"])

    def step():
        eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], wl.total_tokens, None, 0)
        eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    first = (out.clone(), t["k_pool"].clone(), t["v_pool"].clone())
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), first[0].view(torch.int16))
    assert torch.equal(t["k_pool"].view(torch.int16), first[1].view(torch.int16))
    assert torch.equal(t["v_pool"].view(torch.int16), first[2].view(torch.int16))
