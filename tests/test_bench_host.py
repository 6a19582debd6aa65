"""Host-side logic of bench.py that needs no GPU: the multi-rank aggregation (two gloo
ranks on CPU), the reference arm's behaviour under torchrun, and the algorithmic work
model behind the roofline figures."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from paged_variable_length_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 1.25 + 0.5 * rank  # each rank's own step time
    slowest = bench.max_over_ranks(ms, dist, "cpu")
    out[rank] = (slowest, bench.job_tokens_per_s(64, world, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, value = res[rank]
        assert slowest == pytest.approx(1.75)
        # both replicas' tokens over the slowest rank's time
        assert value == pytest.approx(2 * 64 / 1.75e-3)


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tokens_per_s(100, 1, 2.0) == pytest.approx(50000.0)


def _run_bench(args, env_extra=None, timeout=300):
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          env=env, timeout=timeout)


def test_reference_arm_prints_one_line_on_rank_zero_only():
    r1 = _run_bench(["--impl", "reference", "--workload", "worked", "--steps", "1", "--warmup", "0", "--gpus", "2"],
                    {"RANK": "1", "WORLD_SIZE": "2"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_bench(["--impl", "reference", "--workload", "worked", "--steps", "2", "--warmup", "1"],
                    {"RANK": "0", "WORLD_SIZE": "1"})
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == W.worked_example(0).description


def test_work_model_counts_every_visible_pair_once():
    wl = W.worked_example(0)
    work = bench.algorithmic_work(wl)
    pairs = 0
    for n, L in zip(wl.q_lens, wl.kv_lens):
        mask = np.arange(L)[None, :] <= (L - n + np.arange(n))[:, None]  # bottom-right causal
        pairs += int(mask.sum())
    assert work["flops"] == 4 * wl.head_dim * wl.num_qo_heads * pairs
    row = wl.num_kv_heads * wl.head_dim * 2
    assert work["kv_bytes"] == 2 * sum(wl.kv_lens) * row  # no page shared: every row once


def test_work_model_counts_a_shared_prefix_once():
    wl = W.cascade(0, batch=4, prefix=256, lo=16, hi=32)
    work = bench.algorithmic_work(wl)
    row = wl.num_kv_heads * wl.head_dim * 2
    tails = [L - 256 for L in wl.kv_lens]
    assert work["kv_bytes"] == 2 * (256 + sum(tails)) * row
    assert work["kv_bytes_without_sharing"] == 2 * sum(wl.kv_lens) * row


def test_work_model_counts_a_prefix_tree_once():
    """Two levels: the root run once, each branch run once, every private tail once."""
    root, branch, branches, per = 256, 128, 3, 4
    wl = W.cascade_tree(0, branches=branches, per_branch=per, root=root, branch=branch, lo=16, hi=40,
                        num_pages=400)
    work = bench.algorithmic_work(wl)
    row = wl.num_kv_heads * wl.head_dim * 2
    tails = [L - root - branch for L in wl.kv_lens]
    assert len(tails) == branches * per and min(tails) >= 16
    assert work["kv_bytes"] == 2 * (root + branches * branch + sum(tails)) * row
    assert work["kv_bytes_without_sharing"] == 2 * sum(wl.kv_lens) * row
    # the page table has the tree's structure: one root run, `branches` distinct branch runs
    rp, bp = root // wl.page_size, branch // wl.page_size
    assert len({tuple(r[:rp]) for r in wl.page_table}) == 1
    assert len({tuple(r[rp:rp + bp]) for r in wl.page_table}) == branches


def test_work_model_counts_a_deep_prefix_tree_once():
    """Six binary levels: every node's run once, every private tail once."""
    levels, run, per_leaf = 6, 64, 2
    wl = W.cascade_deep(0, levels=levels, run=run, per_leaf=per_leaf, lo=16, hi=40, num_pages=2000)
    work = bench.algorithmic_work(wl)
    row = wl.num_kv_heads * wl.head_dim * 2
    nodes = 2 ** levels - 1
    tails = [L - levels * run for L in wl.kv_lens]
    assert len(tails) == 2 ** (levels - 1) * per_leaf and min(tails) >= 16
    assert work["kv_bytes"] == 2 * (nodes * run + sum(tails)) * row
    # the page table has the tree's structure: 2^(l-1) distinct runs at level l
    rp = run // wl.page_size
    for lv in range(levels):
        assert len({tuple(r[lv * rp:(lv + 1) * rp]) for r in wl.page_table}) == 2 ** lv
