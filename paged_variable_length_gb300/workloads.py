"""Seeded synthetic batches shaped like the pages' workloads.

This module only draws inputs: lengths, page allocations and random values.
It holds none of the attention arithmetic, and it imports nothing from the
rest of the package, so the CUDA path and the CPU oracle can both be fed
from it.

Each workload is a flat, mixed batch as described in "The attention backend
and a reference implementation" (mini-sglang from Scratch, ch. 5, section
"Variable-length, paged attention with prefixes") and "Variable-length
batching and one mixed forward pass" (section "Layout and metadata"):
``q_lens[i]`` new tokens after ``kv_lens[i] - q_lens[i]`` cached ones, the
KV addressed through a page table of page ids.

Integer draws are inclusive at both ends (``rng.integers(lo, hi + 1)``).
Lengths and page allocations come from ``numpy.random.default_rng(seed)``;
values come from a ``torch.Generator`` on the target device seeded with the
same seed, so a workload is reproducible per device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16_NAN_BITS = 0x7FC0


@dataclass
class Workload:
    name: str
    q_lens: list
    kv_lens: list
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    page_table: np.ndarray            # int32 [B, max_pages], junk columns filled with `junk_page`
    value_scale: float = 1.0
    seed: int = 0
    junk_page: int = 0
    shared_prefix_pages: int = 0      # pages every row shares at its start (cascade workload)
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.q_lens)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.q_lens))

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cache_seqlens(self) -> np.ndarray:
        return np.asarray(self.kv_lens, dtype=np.int32)

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.page_size

    def used_pages(self) -> np.ndarray:
        """Sorted unique page ids that hold some request's positions < kv_len."""
        ids = []
        for i, L in enumerate(self.kv_lens):
            ids.append(self.page_table[i, : math.ceil(L / self.page_size)])
        return np.unique(np.concatenate(ids)) if ids else np.zeros(0, np.int32)


def _allocate_rows(rng, kv_lens, page_size, num_pages, shared_prefix_pages=0):
    """Give every request ceil(kv_len/page_size) distinct pages of a shuffled pool.

    With ``shared_prefix_pages`` > 0 the first that many pages are one common
    run shared by every row; the remaining pages of each row are private.
    """
    perm = rng.permutation(num_pages).astype(np.int32)
    need = [math.ceil(L / page_size) for L in kv_lens]
    ld = max(need) if need else 1
    table = np.zeros((len(kv_lens), max(ld, 1)), dtype=np.int32)
    shared = perm[:shared_prefix_pages]
    off = shared_prefix_pages
    for i, p in enumerate(need):
        private = p - shared_prefix_pages
        if private < 0:
            raise ValueError("request shorter than the shared prefix")
        if off + private > num_pages:
            raise ValueError("page pool too small for this batch")
        table[i, :shared_prefix_pages] = shared
        table[i, shared_prefix_pages:p] = perm[off: off + private]
        off += private
    return table


def worked_example(seed: int = 0) -> Workload:
    """3 requests, q_lens [6,3,1], kv_lens [6,7,9] (0, 4 and 8 cached); Hq 4, Hkv 2, D 64;
    page_size 1 over a 64-slot pool, each request's slots a seeded permutation."""
    rng = np.random.default_rng(seed)
    q_lens, kv_lens = [6, 3, 1], [6, 7, 9]
    table = _allocate_rows(rng, kv_lens, 1, 64)
    return Workload("worked", q_lens, kv_lens, 4, 2, 64, 1, 64, table, 1.0, seed,
                    description="worked example: q_lens [6,3,1], kv_lens [6,7,9], Hq4/Hkv2/D64, ps1, 64 slots")


def decode_only(seed: int = 0, batch: int = 64, lo: int = 512, hi: int = 4096) -> Workload:
    """64 single-token decodes, kv_len ~ U[512,4096]; Hq 32, Hkv 8, D 128; page_size 16,
    pages drawn without replacement from a shuffled 20000-page pool."""
    rng = np.random.default_rng(seed)
    kv_lens = [int(x) for x in rng.integers(lo, hi + 1, size=batch)]
    table = _allocate_rows(rng, kv_lens, 16, 20000)
    return Workload("decode", [1] * batch, kv_lens, 32, 8, 128, 16, 20000, table, 1.0, seed,
                    description=f"decode-only: {batch} requests x 1 query, kv_len U[{lo},{hi}], "
                                "Hq32/Hkv8/D128, ps16, 20000-page pool")


def prefill_only(seed: int = 0, batch: int = 8, lo: int = 256, hi: int = 4096) -> Workload:
    """8 fresh prefills, q_len = kv_len ~ U[256,4096]; Hq 32, Hkv 8, D 128; page_size 16,
    random non-contiguous pages of a 20000-page pool; values N(0,1) * 0.5."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(lo, hi + 1, size=batch)]
    table = _allocate_rows(rng, lens, 16, 20000)
    return Workload("prefill", list(lens), list(lens), 32, 8, 128, 16, 20000, table, 0.5, seed,
                    description=f"prefill-only: {batch} fresh prefills, len U[{lo},{hi}], "
                                "Hq32/Hkv8/D128, ps16, 20000-page pool, values 0.5*N(0,1)")


def mixed(seed: int = 0, num_decodes: int = 61, decode_hi: int = 8192) -> Workload:
    """Fresh prefills of 2000 and 512 tokens, a 1024-token chunk on 3072 cached, and 61
    decodes with kv_len ~ U[1,8192]; Hq 28, Hkv 4, D 128; page_size 1 over a 600000-slot
    pool whose slots are a random permutation."""
    rng = np.random.default_rng(seed)
    dec = [int(x) for x in rng.integers(1, decode_hi + 1, size=num_decodes)]
    q_lens = [2000, 512, 1024] + [1] * num_decodes
    kv_lens = [2000, 512, 4096] + dec
    table = _allocate_rows(rng, kv_lens, 1, 600000)
    return Workload("mixed", q_lens, kv_lens, 28, 4, 128, 1, 600000, table, 1.0, seed,
                    description=f"mixed: prefills 2000+512, chunk 1024 on 3072 cached, {num_decodes} "
                                f"decodes kv_len U[1,{decode_hi}], Hq28/Hkv4/D128, ps1, 600000 slots")


def cascade(seed: int = 0, batch: int = 128, prefix: int = 4096, lo: int = 16, hi: int = 512) -> Workload:
    """128 single-token decodes whose page tables share the same 4096-token prefix pages,
    then private tails of U[16,512] tokens; Hq 32, Hkv 8, D 128; page_size 16."""
    rng = np.random.default_rng(seed)
    if prefix % 16:
        raise ValueError("the shared prefix is whole pages")
    tails = [int(x) for x in rng.integers(lo, hi + 1, size=batch)]
    kv_lens = [prefix + t for t in tails]
    table = _allocate_rows(rng, kv_lens, 16, 20000, shared_prefix_pages=prefix // 16)
    return Workload("cascade", [1] * batch, kv_lens, 32, 8, 128, 16, 20000, table, 1.0, seed,
                    shared_prefix_pages=prefix // 16,
                    description=f"cascade: {batch} decodes sharing a {prefix}-token prefix, tails "
                                f"U[{lo},{hi}], Hq32/Hkv8/D128, ps16, 20000-page pool")


def cascade_tree(seed: int = 0, branches: int = 8, per_branch: int = 16, root: int = 2048, branch: int = 1024,
                 lo: int = 16, hi: int = 512, page_size: int = 16, num_pages: int = 20000) -> Workload:
    """A two-level prefix tree of single-token decodes: every row starts with the same
    ``root``-token run of pages, each of ``branches`` groups of ``per_branch`` rows then
    shares a further ``branch``-token run of its own, and each row ends in a private tail
    of U[lo, hi] tokens; Hq 32, Hkv 8, D 128; page_size 16 over a 20000-page pool."""
    rng = np.random.default_rng(seed)
    if root % page_size or branch % page_size:
        raise ValueError("the shared runs are whole pages")
    perm = [int(x) for x in rng.permutation(num_pages)]
    take = lambda k: [perm.pop() for _ in range(k)]
    root_pages = take(root // page_size)
    rows, kv_lens = [], []
    for _ in range(branches):
        branch_pages = take(branch // page_size)
        for _ in range(per_branch):
            tail = int(rng.integers(lo, hi + 1))
            L = root + branch + tail
            rows.append(root_pages + branch_pages + take(math.ceil(L / page_size) - len(root_pages) - len(branch_pages)))
            kv_lens.append(L)
    table = np.zeros((len(rows), max(len(r) for r in rows)), np.int32)
    for i, r in enumerate(rows):
        table[i, :len(r)] = r
    return Workload("cascade_tree", [1] * len(rows), kv_lens, 32, 8, 128, page_size, num_pages, table, 1.0, seed,
                    shared_prefix_pages=root // page_size,
                    extra={"branch_pages": branch // page_size, "per_branch": per_branch},
                    description=f"cascade tree: {branches}x{per_branch} decodes, a {root}-token root prefix, "
                                f"{branch}-token branch prefixes, tails U[{lo},{hi}], Hq32/Hkv8/D128, "
                                f"ps{page_size}, {num_pages}-page pool")


def cascade_tree3(seed: int = 0, fanout=(4, 4), per_leaf: int = 8, runs=(1024, 1024, 1024), lo: int = 16,
                  hi: int = 512, page_size: int = 16, num_pages: int = 20000) -> Workload:
    """A three-level prefix tree of single-token decodes: every row starts with the same
    ``runs[0]``-token run of pages; ``fanout[0]`` branches each add a ``runs[1]``-token run
    of their own; inside each branch ``fanout[1]`` twigs add a ``runs[2]``-token run; each
    twig holds ``per_leaf`` rows, which end in private tails of U[lo, hi] tokens.  Default:
    4 x 4 twigs of 8 rows (128 decodes), 1024 tokens a level; Hq 32, Hkv 8, D 128;
    page_size 16 over a 20000-page pool."""
    rng = np.random.default_rng(seed)
    if any(r % page_size for r in runs):
        raise ValueError("the shared runs are whole pages")
    perm = [int(x) for x in rng.permutation(num_pages)]
    take = lambda k: [perm.pop() for _ in range(k)]
    root_pages = take(runs[0] // page_size)
    rows, kv_lens = [], []
    for _ in range(fanout[0]):
        branch_pages = root_pages + take(runs[1] // page_size)
        for _ in range(fanout[1]):
            twig_pages = branch_pages + take(runs[2] // page_size)
            for _ in range(per_leaf):
                L = sum(runs) + int(rng.integers(lo, hi + 1))
                rows.append(twig_pages + take(math.ceil(L / page_size) - len(twig_pages)))
                kv_lens.append(L)
    table = np.zeros((len(rows), max(len(r) for r in rows)), np.int32)
    for i, r in enumerate(rows):
        table[i, :len(r)] = r
    return Workload("cascade_tree3", [1] * len(rows), kv_lens, 32, 8, 128, page_size, num_pages, table, 1.0, seed,
                    shared_prefix_pages=runs[0] // page_size,
                    extra={"fanout": tuple(fanout), "runs": tuple(runs), "per_leaf": per_leaf},
                    description=f"cascade tree, three levels: {fanout[0]}x{fanout[1]}x{per_leaf} decodes, "
                                f"{runs[0]}/{runs[1]}/{runs[2]}-token shared runs, tails U[{lo},{hi}], "
                                f"Hq32/Hkv8/D128, ps{page_size}, {num_pages}-page pool")


def cascade_deep(seed: int = 0, levels: int = 6, run: int = 512, per_leaf: int = 4, lo: int = 16, hi: int = 512,
                 page_size: int = 16, num_pages: int = 20000) -> Workload:
    """A binary prefix tree ``levels`` deep of single-token decodes: every row starts with
    the same ``run``-token run of pages, and at each further level the rows of a node split
    into two halves that each add a ``run``-token run of their own; each of the
    2^(levels-1) leaves holds ``per_leaf`` rows, which end in private tails of U[lo, hi]
    tokens.  Default: six levels of 512 tokens, 32 leaves of 4 rows (128 decodes); Hq 32,
    Hkv 8, D 128; page_size 16 over a 20000-page pool."""
    rng = np.random.default_rng(seed)
    if run % page_size:
        raise ValueError("the shared runs are whole pages")
    perm = [int(x) for x in rng.permutation(num_pages)]
    take = lambda k: [perm.pop() for _ in range(k)]
    rows, kv_lens = [], []

    def node(pages, level):
        pages = pages + take(run // page_size)
        if level == levels:
            for _ in range(per_leaf):
                L = levels * run + int(rng.integers(lo, hi + 1))
                rows.append(pages + take(math.ceil(L / page_size) - len(pages)))
                kv_lens.append(L)
            return
        for _ in range(2):
            node(pages, level + 1)

    node([], 1)
    table = np.zeros((len(rows), max(len(r) for r in rows)), np.int32)
    for i, r in enumerate(rows):
        table[i, :len(r)] = r
    return Workload("cascade_deep", [1] * len(rows), kv_lens, 32, 8, 128, page_size, num_pages, table, 1.0, seed,
                    shared_prefix_pages=run // page_size,
                    extra={"levels": levels, "run": run, "per_leaf": per_leaf},
                    description=f"cascade tree, {levels} levels: binary, {2 ** (levels - 1)}x{per_leaf} decodes, "
                                f"{run}-token shared run a level, tails U[{lo},{hi}], Hq32/Hkv8/D128, "
                                f"ps{page_size}, {num_pages}-page pool")


def ragged_prefill(seed: int = 0, batch: int = 8, lo: int = 256, hi: int = 4096) -> Workload:
    """The prefill workload's requests (8 fresh prefills, len U[256,4096], Hq 32, Hkv 8,
    D 128) over contiguous K/V: page_size 1, the "pool" is the batch's own k / v rows and
    page_table[i][j] = cu_seqlens[i] + j (request i's keys are its new tokens)."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(lo, hi + 1, size=batch)]
    cu = np.concatenate([[0], np.cumsum(lens)])
    table = np.zeros((batch, max(lens)), np.int32)
    for i, L in enumerate(lens):
        table[i, :L] = np.arange(cu[i], cu[i] + L)
    return Workload("ragged", list(lens), list(lens), 32, 8, 128, 1, int(cu[-1]), table, 0.5, seed,
                    description=f"ragged prefill: {batch} fresh prefills, len U[{lo},{hi}], Hq32/Hkv8/D128, "
                                "contiguous K/V (no pool, no store)")


def spec_decode(seed: int = 0, batch: int = 64, draft: int = 3, lo: int = 512, hi: int = 4096) -> Workload:
    """A uniform speculative-decoding verify step: every request appends 1 + draft tokens
    (the last accepted token and the drafted ones), causally masked among themselves;
    kv_len ~ U[lo, hi] including them; Hq 32, Hkv 8, D 128; page_size 16 over a 20000-page pool."""
    rng = np.random.default_rng(seed)
    n = 1 + draft
    kv_lens = [int(x) for x in rng.integers(max(lo, n), hi + 1, size=batch)]
    table = _allocate_rows(rng, kv_lens, 16, 20000)
    return Workload("specdec", [n] * batch, kv_lens, 32, 8, 128, 16, 20000, table, 1.0, seed,
                    description=f"speculative verify: {batch} requests x {n} queries (1 + {draft} drafted), "
                                f"kv_len U[{lo},{hi}], Hq32/Hkv8/D128, ps16, 20000-page pool")


def custom(q_lens, kv_lens, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages=None,
           seed: int = 0, value_scale: float = 1.0, shared_prefix_pages: int = 0, slack_pages: int = 8,
           name: str = "custom") -> Workload:
    """Any (q_len, kv_len) list; pages drawn from a shuffled pool (default: just large enough)."""
    rng = np.random.default_rng(seed)
    need = sum(math.ceil(L / page_size) for L in kv_lens) - shared_prefix_pages * max(len(kv_lens) - 1, 0)
    if num_pages is None:
        num_pages = max(need + slack_pages, 1)
    table = _allocate_rows(rng, list(kv_lens), page_size, num_pages, shared_prefix_pages)
    return Workload(name, list(q_lens), list(kv_lens), num_qo_heads, num_kv_heads, head_dim, page_size,
                    num_pages, table, value_scale, seed, shared_prefix_pages=shared_prefix_pages)


WORKLOADS = {
    "worked": worked_example,
    "decode": decode_only,
    "prefill": prefill_only,
    "mixed": mixed,
    "cascade": cascade,
    "cascade_tree": cascade_tree,
    "cascade_tree3": cascade_tree3,
    "cascade_deep": cascade_deep,
    "specdec": spec_decode,
    "ragged": ragged_prefill,
}


def make_tensors(wl: Workload, device="cpu", poison_unused: bool = False, fill_all_pages: bool = False):
    """Draw q, k, v (this step's new tokens) and the two pools, all bf16 on ``device``.

    Pages that some request uses get N(0,1) * value_scale.  Other pages are
    zero, or NaN when ``poison_unused`` (a stray read then shows up as NaN in
    the output without ever leaving the pool).  With ``poison_unused`` the
    slots of a request's last page past its kv_len are NaN too.
    Returns a dict of torch tensors plus the integer metadata.
    """
    import torch

    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(wl.seed) * 7919 + 17)
    T, Hq, Hkv, D, ps = wl.total_tokens, wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
    s = float(wl.value_scale)

    def randn(*shape):
        x = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        if s != 1.0:
            x.mul_(s)
        return x.to(torch.bfloat16)

    q = randn(T, Hq, D)
    k = randn(T, Hkv, D)
    v = randn(T, Hkv, D)
    fill = torch.full((), float("nan") if poison_unused else 0.0, dtype=torch.bfloat16)
    k_pool = torch.empty(wl.num_pages, ps, Hkv, D, dtype=torch.bfloat16, device=dev)
    v_pool = torch.empty_like(k_pool)
    if fill_all_pages:
        k_pool.copy_(randn(wl.num_pages, ps, Hkv, D))
        v_pool.copy_(randn(wl.num_pages, ps, Hkv, D))
    else:
        k_pool.fill_(fill.item())
        v_pool.fill_(fill.item())
        used = torch.as_tensor(wl.used_pages(), dtype=torch.long, device=dev)
        if used.numel():
            k_pool[used] = randn(used.numel(), ps, Hkv, D)
            v_pool[used] = randn(used.numel(), ps, Hkv, D)
    if poison_unused:
        for i, L in enumerate(wl.kv_lens):
            if L % ps:
                last = int(wl.page_table[i, L // ps])
                k_pool[last, L % ps:] = float("nan")
                v_pool[last, L % ps:] = float("nan")
    k_pool = k_pool.view(wl.num_pages * ps, Hkv, D)
    v_pool = v_pool.view(wl.num_pages * ps, Hkv, D)
    return {
        "q": q, "k": k, "v": v, "k_pool": k_pool, "v_pool": v_pool,
        "cu_seqlens_q": torch.as_tensor(wl.cu_seqlens_q, dtype=torch.int32, device=dev),
        "cache_seqlens": torch.as_tensor(wl.cache_seqlens, dtype=torch.int32, device=dev),
        "page_table": torch.as_tensor(wl.page_table, dtype=torch.int32, device=dev),
    }


def make_fp8_pools(wl: Workload, device="cpu", poison_unused: bool = False):
    """E4M3 pools (uint8 codes) and one fp32 scale per kv head for K and for V.

    Codes are drawn directly (random sign, exponent field 0..10, random mantissa:
    magnitudes up to ~15 times the scale), so no conversion arithmetic is involved.
    Pages no request uses, and with ``poison_unused`` the slots of a request's last page
    past its kv_len, hold the NaN code 0x7F instead (zero codes without poisoning).
    Scales are drawn in [0.02, 0.1) (not powers of two, so quantising divides inexactly).
    Returns (k_pool, v_pool, k_scale, v_scale), torch tensors on ``device``.
    """
    import torch

    rng = np.random.default_rng(int(wl.seed) * 104729 + 3)
    Hkv, D, ps, P = wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages

    def codes(n_pages):
        sign = rng.integers(0, 2, size=(n_pages, ps, Hkv, D), dtype=np.uint8) << 7
        expo = rng.integers(0, 11, size=(n_pages, ps, Hkv, D), dtype=np.uint8) << 3
        mant = rng.integers(0, 8, size=(n_pages, ps, Hkv, D), dtype=np.uint8)
        return sign | expo | mant

    fill = 0x7F if poison_unused else 0x00
    pools = []
    used = np.asarray(wl.used_pages(), dtype=np.int64)
    for _ in range(2):
        pool = np.full((P, ps, Hkv, D), fill, dtype=np.uint8)
        if used.size:
            pool[used] = codes(used.size)
        if poison_unused:
            for i, L in enumerate(wl.kv_lens):
                if L % ps:
                    pool[int(wl.page_table[i, L // ps]), L % ps:] = 0x7F
        pools.append(torch.from_numpy(pool.reshape(P * ps, Hkv, D)).to(device))
    k_scale = torch.from_numpy(rng.uniform(0.02, 0.1, Hkv).astype(np.float32)).to(device)
    v_scale = torch.from_numpy(rng.uniform(0.02, 0.1, Hkv).astype(np.float32)).to(device)
    return pools[0], pools[1], k_scale, v_scale


def set_junk_columns(wl: Workload, page_id: int) -> None:
    """Point every page-table column past a request's last page at ``page_id``."""
    for i, L in enumerate(wl.kv_lens):
        wl.page_table[i, math.ceil(L / wl.page_size):] = page_id
    wl.junk_page = page_id

