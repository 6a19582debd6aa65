"""Host check of the prefix-pass sizing rule (CPU, no GPU).

The prepare kernel aims the shared-prefix pass at the share of the SMs its tensor-core
time takes beside the decode tails' streaming time, from per-SM rates measured on GB300
(prefix_pass_target in csrc/pva_internal.h; only the speed depends on it).  This test
restates the rule, checks that it stays within [1, casc_target] for random batches and
SM counts, grows with the prefix and shrinks with the tails, and gives the targets the
kernel comment quotes for the 128-member cascade batch, seed 0 (36 for bf16, 76 for FP8 pools).
"""
import os
import random
import re

import pytest

from paged_variable_length_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "paged_variable_length_gb300", "csrc", "pva_internal.h")


def _rates():
    text = open(HDR).read()
    get = lambda name: float(re.search(name + r"\s*=\s*([0-9.]+)f", text).group(1))
    return get("kTuneTcGflopsPerSm"), get("kTuneFp8TcSlowdown"), get("kTuneDecodeGbsPerSm")


def _target(pair16, tail_keys, group, fp8, casc_target):
    tc, slow, dec = _rates()
    if tail_keys == 0:
        return casc_target
    pre = pair16 * 16.0 * group * 2.0 * dec * (slow if fp8 else 1.0)
    tail = tail_keys * (1.0 if fp8 else 2.0) * tc
    r = pre / tail
    return max(1, min(casc_target, int(casc_target * r / (1.0 + r))))


def _cascade_inputs(wl):
    prefix = wl.shared_prefix_pages * wl.page_size
    pair16 = wl.batch * (prefix // 16)  # one group: every member x the prefix's 16-key stages
    tail_keys = sum(L - prefix for L in wl.kv_lens)
    return pair16, tail_keys, wl.num_qo_heads // wl.num_kv_heads


def test_cascade_batch_targets():
    pair16, tail_keys, g = _cascade_inputs(W.cascade(0))
    assert _target(pair16, tail_keys, g, False, 152) == 36
    assert _target(pair16, tail_keys, g, True, 152) == 76


def test_target_range_and_monotonicity():
    rng = random.Random(0)
    for _ in range(2000):
        sms = rng.choice([1, 2, 8, 60, 132, 148, 152, 160])
        g = rng.choice([1, 2, 4, 7, 8, 16])
        fp8 = rng.random() < 0.5
        pair16 = rng.randint(0, 1 << 22)
        tail = rng.randint(0, 1 << 24)
        t = _target(pair16, tail, g, fp8, sms)
        assert 1 <= t <= sms
        assert _target(pair16 * 2, tail, g, fp8, sms) >= t
        assert _target(pair16, tail * 2 + 1, g, fp8, sms) <= t or tail == 0
