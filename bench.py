"""Benchmark: one step = prepare_metadata + one attn_forward (store + attention)
over one synthetic batch, through the C ABI of libpva.so.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|prefill|mixed|cascade|worked|...]
    python bench.py --impl reference ...     # the CPU oracle on a bounded sample

Prints ONE JSON line: the headline workload (decode by default) and, at N = 1, under
"configs" the other workloads (worked example, prefill, mixed, shared-prefix cascade
with and without the prefix pass, decode on an E4M3 pool) timed the same way.  Multi-GPU (torchrun, one process per GPU): every rank
runs an independent replica of the workload (requests are independent; no
collective in the data path), timing is max over ranks, `value` is the
whole-job tokens/s (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged varlen attention tokens/s and % roofline (HBM for decode, TC for prefill)"
L2_FLUSH_BYTES = 512 << 20  # > 4x the 129 MB L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode",
                    choices=["worked", "decode", "prefill", "mixed", "cascade", "cascade_tree", "cascade_tree3",
                             "cascade_deep", "specdec", "ragged"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--clocks-dir", default=None,
                    help="where the nvidia-smi clock samples are written (default: a temporary directory)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only --workload (skip the other workloads' entries under 'configs')")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "e4m3"],
                    help="pool element type (e4m3: one byte per element, a scale per kv head)")
    return ap.parse_args()


# ------------------------------------------------------------------------------ ncu traffic

# DRAM bytes (read + write) per launch from the committed ncu captures, keyed by
# (kernel phase, workload).  A figure is used only while the kernel's sources hash to
# what they were at capture time; after any change the roofline reports null.
NCU_TRAFFIC = {
    ("decode", "decode"): {
        "bytes": 617.539328e6,
        "sources": ['paged_variable_length_gb300/csrc/decode.cu', 'paged_variable_length_gb300/csrc/device_utils.cuh', 'paged_variable_length_gb300/csrc/pva_internal.h'],
        "sha256_16": "613cd1f6c6e4c52d",
        "summary": "profiles/decode_kernel_decode_workload.md",
    },
    ("tensor_core", "prefill"): {
        "bytes": 220.163328e6,
        "sources": ['paged_variable_length_gb300/csrc/prefill_tc.cu', 'paged_variable_length_gb300/csrc/device_utils.cuh', 'paged_variable_length_gb300/csrc/tc_utils.cuh', 'paged_variable_length_gb300/csrc/pva_internal.h'],
        "sha256_16": "8f5604412ac531c8",
        "summary": "profiles/prefill_kernel_prefill_workload.md",
    },
}


def ncu_traffic(phase: str, workload: str):
    import hashlib

    entry = NCU_TRAFFIC.get((phase, workload))
    if entry is None:
        return None
    h = hashlib.sha256()
    for f in entry["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return entry["bytes"] if h.hexdigest()[:16] == entry["sha256_16"] else None


# ------------------------------------------------------------------------------ multi-rank helpers

def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the batch (weak scaling)."""
    return world * tokens_per_rank / (ms / 1e3)


def job_config(wl, args, world: int) -> dict:
    return {
        "workload": wl.description, "seed": args.seed, "batch": wl.batch, "new_tokens": wl.total_tokens,
        "kv_dtype": args.kv_dtype,
        "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write, outside the timed events)",
        "step": "attn_prepare_metadata + attn_forward (store_kvcache + attention), one layer",
        "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
    }


# ------------------------------------------------------------------------------ algorithmic work

def algorithmic_work(wl, kv_elem_bytes: int = 2):
    """Bytes and FLOPs the step must move / compute, independent of the kernels.

    bytes: every visible KV row once (unique pages), this step's Q read and O
    write, the new K/V read (bf16) and their pool write (kv_elem_bytes per element).
    FLOPs: 4*D per visible (query, key) pair per q head (QK^T and PV), causal pairs only.
    """
    import numpy as np

    Hq, Hkv, D, ps = wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
    row_kv = Hkv * D * kv_elem_bytes  # bytes of one slot's K (or V) row in the pool, all kv heads
    # unique KV rows read: positions < kv_len of each request, shared prefix pages counted once
    seen = set()
    kv_rows = 0
    for i, L in enumerate(wl.kv_lens):
        if wl.q_lens[i] == 0:
            continue
        full, rem = divmod(L, ps)
        for p in range(full + (1 if rem else 0)):
            pid = int(wl.page_table[i, p])
            rows = ps if p < full else rem
            key = (pid, rows)
            if pid in seen:
                continue
            seen.add(pid)
            kv_rows += rows
    T = wl.total_tokens
    kv_bytes = 2 * kv_rows * row_kv
    q_bytes = T * Hq * D * 2
    o_bytes = T * Hq * D * 2
    new_kv_bytes = 2 * T * Hkv * D * 2
    store_bytes = new_kv_bytes + 2 * T * row_kv  # read k,v (bf16) + write the pool rows
    if wl.name == "ragged":
        store_bytes = 0  # contiguous K/V: nothing is stored
    pairs = 0
    for n, L in zip(wl.q_lens, wl.kv_lens):
        # query r sees L - n + r + 1 keys
        pairs += n * (L - n) + n * (n + 1) // 2
    flops = 4 * D * Hq * pairs
    no_share_kv = 2 * sum(L for n, L in zip(wl.q_lens, wl.kv_lens) if n) * row_kv
    return {
        "kv_bytes": kv_bytes, "q_bytes": q_bytes, "o_bytes": o_bytes, "store_bytes": store_bytes,
        "attn_bytes": kv_bytes + q_bytes + o_bytes, "step_bytes": kv_bytes + q_bytes + o_bytes + store_bytes,
        "flops": flops, "pairs": pairs, "kv_bytes_without_sharing": no_share_kv,
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True, directory: str | None = None):
        self.proc = None
        self.path = None
        if not enabled:
            return
        try:
            import tempfile

            directory = directory or tempfile.mkdtemp(prefix="pva_clocks_")
            os.makedirs(directory, exist_ok=True)
            self.path = os.path.join(directory, f"clocks_rank{gpu_index}.csv")
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_first_sample(self, timeout_s: float = 3.0):
        if self.proc is None:
            return
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < timeout_s:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ CPU oracle baseline

def _oracle_sample(wl, tensors_cpu, chosen):
    """The sampled requests' inputs in the oracle's form."""
    import numpy as np

    cu = wl.cu_seqlens_q
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in chosen]) if chosen else np.zeros(0, np.int64)
    sub_cu = np.concatenate([[0], np.cumsum([wl.q_lens[i] for i in chosen])]).astype(np.int32)
    return {"q": tensors_cpu["q"][rows], "k": tensors_cpu["k"][rows], "v": tensors_cpu["v"][rows], "cu": sub_cu,
            "lens": np.asarray([wl.kv_lens[i] for i in chosen], np.int32), "table": wl.page_table[chosen]}


def _oracle_pass(wl, tensors_cpu, s) -> float:
    """One store + attention pass of the oracle over a sample; returns its seconds."""
    import oracle

    t0 = time.perf_counter()
    if "k_scale" in tensors_cpu:
        oracle.forward_fp8(s["q"], s["k"], s["v"], tensors_cpu["k_pool"], tensors_cpu["v_pool"],
                           tensors_cpu["k_scale"], tensors_cpu["v_scale"], s["cu"], s["lens"], s["table"],
                           wl.page_size)
    else:
        oracle.forward(s["q"], s["k"], s["v"], tensors_cpu["k_pool"], tensors_cpu["v_pool"], s["cu"], s["lens"],
                       s["table"], wl.page_size)
    return time.perf_counter() - t0


def _sample_by_rate(wl, rate_flops: float, budget_s: float):
    """Requests in order until the estimated oracle time reaches the budget (at least one)."""
    chosen, est = [], 0.0
    for i, (n, L) in enumerate(zip(wl.q_lens, wl.kv_lens)):
        cost = 4.0 * wl.head_dim * wl.num_qo_heads * (n * L) + 1e6
        if chosen and est + cost / rate_flops > budget_s:
            break
        chosen.append(i)
        est += cost / rate_flops
    return chosen


def cpu_baseline(wl, tensors_cpu, budget_s: float, single_thread: bool = True):
    """The oracle as it stands, timed on this host over bounded samples of the workload's
    requests (in order): with OpenMP on all the cores it gets (passes repeated for about
    half the budget), and single-threaded on a sample sized from the first leg's rate for
    the other half.  When even one request would take the single-threaded leg past its
    budget, its rate is that of the OpenMP leg divided by the thread count, labelled as
    extrapolated."""
    import oracle

    oracle.build()
    threads = oracle.num_threads()
    half = budget_s / 2 if single_thread else budget_s
    # ~0.5 GFLOP/s per thread on the plain loops: only sizes the first sample
    chosen = _sample_by_rate(wl, 0.5e9 * max(threads, 1), half)
    s = _oracle_sample(wl, tensors_cpu, chosen)
    tokens = int(s["cu"][-1])
    flops = sum(4.0 * wl.head_dim * wl.num_qo_heads * wl.q_lens[i] * wl.kv_lens[i] for i in chosen)
    secs, passes = 0.0, 0
    while passes < 1 or (secs < half and passes < 50):
        secs += _oracle_pass(wl, tensors_cpu, s)
        passes += 1
    value = tokens * passes / secs if secs > 0 else None
    out = {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "sample": f"{len(chosen)} of {wl.batch} requests ({tokens} of {wl.total_tokens} new tokens), "
                     f"{passes} store+attention passes with {threads} OpenMP threads, {secs:.2f} s"}
    if not single_thread:
        return out
    rate1 = flops * passes / secs / max(threads, 1)  # FLOP/s of one thread, from the first leg
    chosen1 = _sample_by_rate(wl, rate1, half)
    first_cost = 4.0 * wl.head_dim * wl.num_qo_heads * wl.q_lens[0] * wl.kv_lens[0] / rate1
    try:
        oracle.set_num_threads(1)
        if first_cost > 2 * half:
            v1, how = value / max(threads, 1), "extrapolated: the OpenMP rate / thread count (one request exceeds the budget)"
        else:
            s1 = _oracle_sample(wl, tensors_cpu, chosen1)
            dt = _oracle_pass(wl, tensors_cpu, s1)
            v1 = int(s1["cu"][-1]) / dt if dt > 0 else None
            how = f"{len(chosen1)} of {wl.batch} requests, one pass, {dt:.2f} s"
    finally:
        oracle.set_num_threads(threads)
    out["single_thread"] = {"value": v1, "unit": "tokens/s", "cores": 1, "sample": how}
    return out


# ------------------------------------------------------------------------------ reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from paged_variable_length_gb300 import workloads as W

    wl = W.WORKLOADS[args.workload](args.seed)
    t = W.make_tensors(wl, "cpu")
    if args.kv_dtype == "e4m3":
        t["k_pool"], t["v_pool"], t["k_scale"], t["v_scale"] = W.make_fp8_pools(wl, "cpu")
    vals = []
    base = None
    # each step a bounded sample (about a minute in all); the single-threaded leg on the last
    budget = min(args.cpu_budget_s, 60.0 / max(args.steps + args.warmup, 1))
    for i in range(args.warmup + args.steps):
        last = i == args.warmup + args.steps - 1
        base = cpu_baseline(wl, t, budget_s=2 * budget if last else budget, single_thread=last)
        if i >= args.warmup:
            vals.append(base["value"])
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": job_config(wl, args, args.gpus),
        "cpu_baseline": dict(base, value=value),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------------------------------ our arm

class Bench:
    """One workload on the GPU: its tensors, an engine, and the timed graph-replayed step."""

    def __init__(self, name, args, dev, rank=0, fp8=False, enable_cascade=True):
        import torch

        from paged_variable_length_gb300 import pva
        from paged_variable_length_gb300 import workloads as W

        self.pva, self.torch = pva, torch
        self.name, self.args, self.dev, self.fp8 = name, args, dev, fp8
        self.wl = wl = W.WORKLOADS[name](args.seed + rank)
        self.work = algorithmic_work(wl, 1 if fp8 else 2)
        self.t = t = W.make_tensors(wl, dev)
        self.scales = {}
        if fp8:
            t["k_pool"], t["v_pool"], ks, vs = W.make_fp8_pools(wl, dev)
            self.scales = {"k_scale": ks, "v_scale": vs}
        self.slots = None
        if wl.name == "ragged":
            # contiguous K/V: the batch's own k / v rows are the keys, nothing is stored
            t["k_pool"], t["v_pool"] = t["k"], t["v"]
            self.slots = torch.full((wl.total_tokens,), -1, dtype=torch.int64, device=dev)
        self.max_q = max(wl.q_lens)
        self.eng = pva.PagedAttention(wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages,
                                      max_batch=wl.batch, max_tokens=wl.total_tokens, max_kv_len=max(wl.kv_lens),
                                      device=dev, kv_dtype=pva.KV_E4M3 if fp8 else pva.KV_BF16,
                                      enable_cascade=enable_cascade)
        self.out = torch.empty_like(t["q"])
        self.lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device=dev)

    def step(self):
        t = self.t
        self.eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], self.wl.total_tokens, self.slots,
                         self.max_q)
        self.eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], self.out, self.lse, **self.scales)

    def warm_and_capture(self, flush):
        """Warm-up steps, the device status check, and the step captured as a CUDA graph
        (the library makes no host-device synchronisation and allocates nothing, so the
        whole prepare + forward is capturable and the timed replays carry no Python gaps)."""
        torch, pva = self.torch, self.pva
        for _ in range(self.args.warmup):
            flush.fill_(1.0)
            self.step()
        torch.cuda.synchronize()
        bits = pva.attn_get_device_status(self.eng.meta)
        if bits:
            raise RuntimeError(f"{self.name}: device error bits: {pva.deverr_names(bits)}")
        self.plan = pva.attn_debug_plan_counts(self.eng.meta)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        self.graph.replay()
        torch.cuda.synchronize()

    def time_steps(self, flush, stream):
        """K graph replays, L2 flushed before each (outside the events); mean ms per step."""
        torch = self.torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(self.args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(self.args.steps)]
        for i in range(self.args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            self.graph.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        times = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        return sum(times) / len(times)

    def phases(self, flush, stream):
        """Per-kernel durations: the same step replayed from a second graph with the
        library's timing events between its kernels (they break the kernels' launch
        overlap, so the phases add up to more than the step)."""
        torch, pva, t = self.torch, self.pva, self.t
        kev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
        pev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        for e in kev + pev:
            e.record(stream)
        phase = {"prepare": [], "store": [], "tensor_core": [], "decode": [], "merge": []}
        pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pgraph):
            pev[0].record()
            self.eng.prepare(t["cu_seqlens_q"], t["cache_seqlens"], t["page_table"], self.wl.total_tokens,
                             self.slots, self.max_q)
            pev[1].record()
            pva.attn_set_timing_events(self.eng.meta, kev)
            self.eng.forward(t["q"], t["k"], t["v"], t["k_pool"], t["v_pool"], self.out, self.lse, **self.scales)
        pva.attn_set_timing_events(self.eng.meta, None)
        for i in range(self.args.steps):
            flush.fill_(float(i))
            pgraph.replay()
            torch.cuda.synchronize()
            phase["prepare"].append(pev[0].elapsed_time(pev[1]))
            for j, nm in enumerate(["store", "tensor_core", "decode", "merge"]):
                phase[nm].append(kev[j].elapsed_time(kev[j + 1]))
        return {k: (sum(v) / len(v) if v else 0.0) for k, v in phase.items()}

    def rooflines(self, ms, phase_ms, peaks):
        """The dominant kernel's roofline and the whole step's."""
        work = self.work
        dom = max(("tensor_core", "decode"), key=lambda k: phase_ms[k])
        if dom == "tensor_core" and work["flops"] > 0:
            roof = {"bound": "tensor", "achieved": work["flops"] / (phase_ms[dom] / 1e3) / 1e12,
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
        else:
            roof = {"bound": "hbm", "achieved": work["attn_bytes"] / (phase_ms[dom] / 1e3) / 1e9,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["traffic"] = ncu_traffic(dom, self.name if not self.fp8 else self.name + "-e4m3")
        roof["kernel"] = dom
        roof["peak_source"] = peaks["source"]
        roof_time_s = max(work["flops"] / (peaks["bf16_tflops"] * 1e12),
                          work["step_bytes"] / (peaks["hbm_gbs"] * 1e9))
        step = {"roofline_time_us": roof_time_s * 1e6, "frac_of_step": roof_time_s / (ms / 1e3),
                "bytes": work["step_bytes"], "flops": work["flops"]}
        return roof, step

    def e2e(self, flush, stream):
        """The same step through the eager public API with host buffers: the step's inputs
        staged in one pinned host buffer and copied to the device in one transfer (a
        serving loop stages a step's inputs together; one copy per tensor would add a
        copy launch each), and a device -> host copy of the output, inside the timed
        region."""
        torch, t, wl = self.torch, self.t, self.wl
        names = ("q", "k", "v", "cu_seqlens_q", "cache_seqlens", "page_table")
        offs, total = {}, 0
        for k in names:  # each input at a 256-byte boundary of the staging buffers
            offs[k] = total
            total += (t[k].numel() * t[k].element_size() + 255) // 256 * 256
        host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        dev_buf = torch.empty(total, dtype=torch.uint8, device=t["q"].device)
        dev_in = {}
        for k in names:
            nb = t[k].numel() * t[k].element_size()
            host_buf[offs[k]:offs[k] + nb].copy_(t[k].cpu().contiguous().view(-1).view(torch.uint8))
            dev_in[k] = dev_buf[offs[k]:offs[k] + nb].view(t[k].dtype).view(t[k].shape)
        host_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        h2d = sum(t[k].numel() * t[k].element_size() for k in names)
        d2h = host_out.numel() * host_out.element_size()

        def e2e_step():
            dev_buf.copy_(host_buf, non_blocking=True)
            self.eng.prepare(dev_in["cu_seqlens_q"], dev_in["cache_seqlens"], dev_in["page_table"], wl.total_tokens,
                             self.slots, self.max_q)
            kp_e, vp_e = (dev_in["k"], dev_in["v"]) if wl.name == "ragged" else (t["k_pool"], t["v_pool"])
            self.eng.forward(dev_in["q"], dev_in["k"], dev_in["v"], kp_e, vp_e, self.out, None, **self.scales)
            host_out.copy_(self.out, non_blocking=True)

        for _ in range(max(1, self.args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(self.args.steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(self.args.steps)]
        for i in range(self.args.steps):
            flush.fill_(float(i))
            e_s[i].record(stream)
            e2e_step()
            e_e[i].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in zip(e_s, e_e)) / self.args.steps, h2d, d2h

    def summary(self, ms, phase_ms, peaks):
        roof, step = self.rooflines(ms, phase_ms, peaks)
        return {"workload": self.wl.description, "kv_dtype": "e4m3" if self.fp8 else "bf16",
                "new_tokens": self.wl.total_tokens, "value": self.wl.total_tokens / (ms / 1e3),
                "unit": "tokens/s", "ms_per_step": ms, "phases_ms": phase_ms, "roofline": roof,
                "step_roofline": step, "plan": self.plan}


# the other BASELINE workloads (and variants) timed beside the headline one
CONFIGS = [
    ("worked", "worked", {}),
    ("decode", "decode", {}),
    ("prefill", "prefill", {}),
    ("mixed", "mixed", {}),
    ("cascade", "cascade", {}),
    ("cascade_off", "cascade", {"enable_cascade": False}),
    ("cascade_tree", "cascade_tree", {}),
    ("cascade_tree3", "cascade_tree3", {}),
    ("cascade_deep", "cascade_deep", {}),
    ("decode_e4m3", "decode", {"fp8": True}),
]


def run_configs(args, dev, flush, stream, peaks, headline_key):
    """Every entry of CONFIGS but the headline one: the same timed step (K graph replays,
    L2 flushed before each) and phases, one workload at a time."""
    import torch

    out = {}
    for key, name, kw in CONFIGS:
        if key == headline_key:
            continue
        b = Bench(name, args, dev, **kw)
        b.warm_and_capture(flush)
        ms = b.time_steps(flush, stream)
        out[key] = b.summary(ms, b.phases(flush, stream), peaks)
        del b
        torch.cuda.empty_cache()
    if "cascade" in out and "cascade_off" in out:
        on, off = out["cascade"], out["cascade_off"]
        out["cascade"]["vs_no_cascade"] = {
            "speedup": off["ms_per_step"] / on["ms_per_step"],
            "ms_per_step_without_prefix_pass": off["ms_per_step"],
            "kv_bytes_prefix_once": on["step_roofline"]["bytes"],
            "kv_bytes_without_sharing": algorithmic_work(W_of("cascade", args.seed))["kv_bytes_without_sharing"],
        }
    return out


def W_of(name, seed):
    from paged_variable_length_gb300 import workloads as W

    return W.WORKLOADS[name](seed)


def run_ours(args):
    import torch

    from paged_variable_length_gb300 import build as libbuild
    from paged_variable_length_gb300 import pva

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    if rank == 0:
        libbuild.build()
    if dist is not None:
        dist.barrier()
    pva.load()

    fp8 = args.kv_dtype == "e4m3"
    dev = torch.device("cuda", local)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    b = Bench(args.workload, args, dev, rank=rank, fp8=fp8)
    wl = b.wl
    b.warm_and_capture(flush)

    # ---- timed region: K steps, L2 flushed before each (outside the events)
    clocks = ClockSampler(local, enabled=not args.no_clocks, directory=args.clocks_dir)
    clocks.wait_first_sample()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ms = b.time_steps(flush, stream)
    if dist is not None:
        dist.barrier()
    # the timed region is short next to the sampler's period: keep the same step
    # running (no flush) for ~1 s more so the clock record covers the load
    t_end = time.perf_counter() + 1.0
    while time.perf_counter() < t_end:
        for _ in range(50):
            b.graph.replay()
        torch.cuda.synchronize()
    clock_info = clocks.stop()
    ms = max_over_ranks(ms, dist, dev)
    value = job_tokens_per_s(wl.total_tokens, world, ms)

    phase_ms = b.phases(flush, stream)
    roof, step_roof = b.rooflines(ms, phase_ms, peaks)
    e2e_ms, h2d, d2h = b.e2e(flush, stream)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    plan = b.plan

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(wl, {k: v.cpu() for k, v in dict(b.t, **b.scales).items()}, args.cpu_budget_s)
    del b
    torch.cuda.empty_cache()
    configs = None
    if world == 1 and not args.no_configs:
        configs = run_configs(args, dev, flush, stream, peaks, args.workload + ("_e4m3" if fp8 else ""))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 MMA on e4m3 KV" if fp8 else "bf16", "data": "synthetic",
            "config": job_config(wl, args, world),
            "roofline": roof,
            "step_roofline": step_roof,
            "phases_ms": phase_ms,
            "plan": plan,
            "gpu_launches": int(args.steps * (1 + plan.get("kernels_per_forward", 2))),
            "e2e": {"value": job_tokens_per_s(wl.total_tokens, world, e2e_ms), "unit": "tokens/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "clocks": clock_info,
            "cpu_baseline": base,
            "configs": configs,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
