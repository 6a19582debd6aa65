// K0: prepare_metadata -- once per batch, on the device, one CTA.
//
// Turns (cu_seqlens_q, cache_seqlens, page_table, slot_mapping) into the work
// lists the forward kernels walk, as "The attention backend and a reference
// implementation" (section "The interface") asks of prepare_metadata: done once
// per batch because every layer sees the same batch structure.  It runs on the
// device so that the step needs no host round trip ("Variable-length batching
// and one mixed forward pass", section "Inference view": metadata building is
// CPU work that can rival the GPU's compute time).
//
//   0. shared-prefix (cascade) groups: single-token decodes whose page tables start
//      with the same run of pages ("Source walkthrough: Attention backends",
//      section 3.3: the shared part is computed once and merged by log-sum-exp), and
//      inside each group sub-groups whose rows continue with a further shared run, and
//      so on inside those, up to kMaxCascLevels levels of the prefix tree the page
//      describes its multi-level form over;
//   1. validate cu_seqlens_q / cache_seqlens (error word, never a trap) and
//      classify each request: q_len * G <= 16 rows -> decode groups (the
//      warp-MMA streaming kernel), otherwise -> 128-row tensor-core tiles;
//   2. split-KV plan: one chunk length so that the decode work fills the GPU;
//      each group's visible key range (after the prefix, for cascade members) is
//      cut into near-equal chunks;
//   3. work lists, longest item first: decode units, prefill tile pairs with
//      their causal KV extents, and the prefix-pass units of the cascade groups;
//   4. when the caller passed no slot_mapping: the request of every new token, from
//      which the store kernel derives each token's slot through the page table.
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "pva_internal.h"

namespace pva {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 256;  // cost classes for the longest-first ordering of work items
constexpr int kCmpPages = 8;         // page ids a lane compares per step of the shared-prefix search
constexpr int kLineLimit = 1 << 29;  // the balanced decode split is used below this many keys

// Per-request shared-memory arrays (dynamic shared memory, batch <= smem_batch), followed
// by the open-addressing table of the shared-prefix search when cascade detection runs.
enum SmemArray {
    kCu = 0, kLen, kToff, kFirst, kLeader, kLcp, kCnt, kCgid, kGoff, kMpos, kCUoff, kLeader2, kCgid2, kNumArrays
};

// Write a plan record as whole 16-byte words (a record is 32, 48 or 64 bytes, and the
// record arrays start on 256-byte boundaries): one 16-byte store per word instead of
// one 4-byte store per field keeps the single CTA's store traffic in few L2
// transactions.
template <class T>
__device__ __forceinline__ void store_record(T* dst, const T& v) {
    static_assert(sizeof(T) % 16 == 0, "records are whole 16-byte words");
    int4 w[sizeof(T) / 16];
    memcpy(w, &v, sizeof(T));
    int4* d = reinterpret_cast<int4*>(dst);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(T) / 16); ++k) d[k] = w[k];
}

// Fibonacci hashing of a page id into a table of 2^bits entries.
__device__ __forceinline__ uint32_t page_hash(int32_t page, int bits) {
    return ((uint32_t)page * 2654435761u) >> (32 - bits);
}

// Exclusive scan of N counters across the block; each thread contributes v[k].
template <int N>
__device__ void block_scan(int (&v)[N], int (&total)[N], int (*warp_tmp)[N]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
        int x = v[k];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        incl[k] = x;
    }
    if (lane == 31) {
#pragma unroll
        for (int k = 0; k < N; ++k) warp_tmp[warp][k] = incl[k];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) {
            int x = lane < kWarps ? warp_tmp[lane][k] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane < kWarps) warp_tmp[lane][k] = x;  // inclusive warp prefix
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < N; ++k) {
        const int before = warp > 0 ? warp_tmp[warp - 1][k] : 0;
        total[k] = warp_tmp[kWarps - 1][k];
        v[k] = before + incl[k] - v[k];
    }
    __syncthreads();
}

// block_scan of two counters, out of line: one copy of the code serves the shared-prefix
// steps (where the kernel's cold instruction fetch dominates) and pass 2.  Returns this
// thread's exclusive offsets (x, y) and the block totals (z, w).
__device__ __noinline__ int4 block_scan2(int a, int b, int (*warp_tmp)[2]) {
    int v[2] = {a, b}, total[2];
    block_scan<2>(v, total, warp_tmp);
    return make_int4(v[0], v[1], total[0], total[1]);
}

// Index i with off[i] <= x < off[i+1] (off ascending, off[0] <= x); among equal offsets
// the last one, so that entries of width zero are passed over.
__device__ __forceinline__ int find_bucket(const int32_t* off, int count, int x) {
    int lo = 0, hi = count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int cost_bucket(int cost) { return kBuckets - 1 - min(kBuckets - 1, cost); }

__device__ __forceinline__ bool is_group_leader(const int32_t* leader, const int32_t* cnt, const int32_t* lcp,
                                                int i, int min_pages) {
    return leader[i] == i && cnt[i] >= 2 && lcp[i] >= min_pages;
}

// Prefix-pass units of a group with m members: pairs of member tiles x kv heads.
__device__ __forceinline__ int casc_pair_units(int members, int TM, int Hkv) {
    return (((members + TM - 1) / TM) + 1) / 2 * Hkv;
}

// Per-request arrays of shared-prefix level L >= 3 in the workspace (a = 0: the request's
// leader at that level, later its member-list slot; 1: its group id, -1 for none; 2:
// member counts, then member-list cursors, indexed by leader).  Levels 1 and 2 keep theirs
// in shared memory.
__device__ __forceinline__ int32_t* deep_level(const PrepareParams& p, int L, int a) {
    return reinterpret_cast<int32_t*>(p.ws + p.lay.casc_deep) + ((L - 3) * 3 + a) * (p.batch + 1);
}

// What the shared-prefix search of every level needs besides its own arrays (set once, in
// shared memory: passed as one pointer, so that the calls below keep few values live in
// the 64-register kernel).
struct SearchCtx {
    int32_t* dyn;
    int32_t* hkey;
    int32_t* hval;
    CascGroup* scg;
    CascGroup* cgroups;
    const int32_t* page_table;
    int64_t ld_table;
    int64_t num_pages;
    int stride, hbits, min_pages, B, ps, max_groups;
};

// First index k in [start, l) at which two page-table rows differ, one warp: lanes read
// consecutive ids, kCmpPages each per step.  The search stops after the step that finds
// one, and never reads past *bound, the group's prefix as far as the other warps have
// found it (it only falls, and a mismatch at or past it changes no minimum).  Returns a
// value >= min(l, *bound) when the rows agree up to there.  Warp-uniform.
__device__ __forceinline__ int first_mismatch(const int32_t* ri, const int32_t* rl, int start, int l,
                                              const volatile int32_t* bound, int lane) {
    int mis = l;
    #pragma unroll 1
    for (int k0 = start;; k0 += 32 * kCmpPages) {
        l = min(l, __shfl_sync(0xffffffffu, *bound, 0));
        if (k0 >= l) break;
        int va[kCmpPages], vb[kCmpPages];
#pragma unroll
        for (int u = 0; u < kCmpPages; ++u) {
            const int k = k0 + u * 32 + lane;
            va[u] = k < l ? ri[k] : 0;
            vb[u] = k < l ? rl[k] : 0;
        }
#pragma unroll
        for (int u = 0; u < kCmpPages; ++u) {
            const int k = k0 + u * 32 + lane;
            if (k < l && va[u] != vb[u]) mis = min(mis, k);
        }
        mis = __reduce_min_sync(0xffffffffu, mis);
        if (mis < l) break;
    }
    return mis;
}

// One level deeper in the shared-prefix tree (pass 0 of the kernel below; level 2 inside
// the top-level groups, level 3 inside level 2's, and so on): inside a parent group,
// members keyed by
// the page right after the parent's prefix; the lowest-numbered one leads its sub-group,
// whose prefix extends the parent's by the run of pages every sub-member shares with it
// (again at least min_pages, again whole pages before each member's query).  Its prefix
// pass covers keys [parent prefix, sub-group prefix) only.  parent[i]: request i's group
// at the parent level (-1: none).  Scratch arrays: the page after the parent's prefix
// (page2), pages before the query then the sub-prefix (pg2), counts then next free member
// slots (cnt2, kept for the member lists); outputs: the sub-leader (lead2) and sub-group
// id (cgid2, -1: none) of each request; the hash table is reused.  Sub-group records are
// numbered after the n_groups already found, their member lists after `members0` entries;
// a level whose groups would exceed max_groups records in all is not formed (its requests
// run the rest as tails).  Returns how many there are and their member entries in
// *members_total.  A function of its own (not inlined), so that its registers do not
// weigh on the rest of the kernel, which runs 1024 threads and so has 64 registers each.
__device__ __noinline__ int find_next_level(const SearchCtx* cx, const int32_t* parent, int32_t* page2, int32_t* pg2,
                                            int32_t* cnt2, int32_t* lead2, int32_t* cgid2, int n_groups,
                                            int members0, int (*s_tmp2)[2], int* members_total) {
    const int tid = threadIdx.x, lane = tid & 31;
    int32_t* dyn = cx->dyn;
    int32_t* hkey = cx->hkey;
    int32_t* hval = cx->hval;
    CascGroup* scg = cx->scg;
    CascGroup* cgroups = cx->cgroups;
    const int32_t* page_table = cx->page_table;
    const int64_t ld_table = cx->ld_table, num_pages = cx->num_pages;
    const int stride = cx->stride, hbits = cx->hbits, min_pages = cx->min_pages, B = cx->B, ps = cx->ps;
    const int max_groups = cx->max_groups;
    const int chunk_req = (B + kThreads - 1) / kThreads;
    const int r0 = min(B, tid * chunk_req), r1 = min(B, r0 + chunk_req);
    const int HT = 1 << hbits;
    auto sa = [&](int a) { return dyn + a * stride; };
    const int32_t* cu = sa(kCu);
    const int32_t* lens = sa(kLen);
    *members_total = 0;
    #pragma unroll 1
    for (int h = tid; h < HT; h += kThreads) {
        hkey[h] = -1;
        hval[h] = 0x7fffffff;
    }
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads) {
        const int g = parent[i];
        int pg = -1, pages = 0;
        if (g >= 0) {
            const int n = cu[i + 1] - cu[i], L = lens[i];
            pages = (L - n) / ps;
            const int P1 = scg[g].prefix_len / ps;
            if (pages - P1 >= min_pages) {
                const int32_t x = page_table[(int64_t)i * ld_table + P1];
                pg = (x >= 0 && x < num_pages) ? x : -1;
            }
        }
        page2[i] = pg;
        pg2[i] = pages;
        cnt2[i] = 0;
        lead2[i] = -1;
        cgid2[i] = 0;
    }
    __syncthreads();
    // hash key: the page mixed with the group id (two different pairs meeting on one
    // key would only lose sharing: a member whose pair differs from its sub-leader's
    // is dropped below)
    auto key2 = [&](int i) -> int {
        return page2[i] < 0 ? -1
                            : (int)(((uint32_t)page2[i] * 2654435761u ^ (uint32_t)parent[i] * 0x9E3779B9u) &
                                    0x7fffffffu);
    };
    int dup = 0;  // some key met twice (in a warp, or already in the table)
    #pragma unroll 1
    for (int i0 = 0; i0 < B; i0 += kThreads) {
        const int i = i0 + tid;
        const int f = i < B ? key2(i) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, f);
        const int lead = __ffs(peers) - 1;
        int h = 0;
        if (f >= 0 && __popc(peers) > 1) dup = 1;
        if (f >= 0 && lane == lead) {
            uint32_t hh = page_hash(f, hbits);
            while (true) {
                const int prev = atomicCAS(&hkey[hh], -1, f);
                if (prev == f) dup = 1;
                if (prev == -1 || prev == f) break;
                hh = (hh + 1) & (HT - 1);
            }
            atomicMin(&hval[hh], i);
            h = (int)hh;
        }
        h = __shfl_sync(0xffffffffu, h, lead);
        if (f >= 0) lead2[i] = h;
    }
    // no two members of a group continue with the same page: no sub-group (the usual
    // case; the rest of the search is skipped)
    if (!__syncthreads_or(dup)) {
        #pragma unroll 1
        for (int i = tid; i < B; i += kThreads) cgid2[i] = -1;
        __syncthreads();
        return 0;
    }
    #pragma unroll 1
    for (int i0 = 0; i0 < B; i0 += kThreads) {
        const int i = i0 + tid;
        int ld = (i < B && page2[i] >= 0) ? hval[lead2[i]] : -1;
        if (ld >= 0 && (parent[ld] != parent[i] || page2[ld] != page2[i])) ld = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, ld);
        if (i < B) lead2[i] = ld;
        if (ld >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt2[ld], __popc(peers));
    }
    __syncthreads();
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads) {
        const int ld = lead2[i];
        cgid2[i] = (ld >= 0 && ld != i) ? min(pg2[i], pg2[ld]) : 0;
    }
    __syncthreads();
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads)
        if (cgid2[i] > 0) atomicMin(&pg2[lead2[i]], cgid2[i]);
    {
        const int warp = tid >> 5;
        #pragma unroll 1
        for (int i = warp; i < B; i += kWarps) {
            const int l = cgid2[i];
            const int g = parent[i];
            if (l <= 0 || g < 0) continue;  // warp-uniform
            const int start = scg[g].prefix_len / ps + 1;  // page start - 1 matched by the key
            if (l <= start) continue;
            const int ld = lead2[i];
            const int32_t* ri = page_table + (int64_t)i * ld_table;
            const int32_t* rl = page_table + (int64_t)ld * ld_table;
            int mis = l;
            #pragma unroll 1
            for (int k0 = start; k0 < l; k0 += 32 * kCmpPages) {
                int va[kCmpPages], vb[kCmpPages];
#pragma unroll
                for (int u = 0; u < kCmpPages; ++u) {
                    const int k = k0 + u * 32 + lane;
                    va[u] = k < l ? ri[k] : 0;
                    vb[u] = k < l ? rl[k] : 0;
                }
#pragma unroll
                for (int u = 0; u < kCmpPages; ++u) {
                    const int k = k0 + u * 32 + lane;
                    if (k < l && va[u] != vb[u]) mis = min(mis, k);
                }
            }
            mis = __reduce_min_sync(0xffffffffu, mis);
            if (lane == 0 && mis < l) atomicMin(&pg2[ld], mis);
        }
    }
    __syncthreads();
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads) cgid2[i] = -1;
    __syncthreads();
    auto is_sub_leader = [&](int i) {
        if (lead2[i] != i || cnt2[i] < 2) return false;
        return pg2[i] - scg[parent[i]].prefix_len / ps >= min_pages;
    };
    int hv[2] = {0, 0};
    #pragma unroll 1
    for (int i = r0; i < r1; ++i)
        if (is_sub_leader(i)) {
            hv[0] += 1;
            hv[1] += cnt2[i];
        }
    int ht[2];
    {
        const int4 r = block_scan2(hv[0], hv[1], s_tmp2);
        hv[0] = r.x, hv[1] = r.y, ht[0] = r.z, ht[1] = r.w;
    }
    if (n_groups + ht[0] > max_groups) {  // no room for this level's records: not formed
        #pragma unroll 1
        for (int i = tid; i < B; i += kThreads) cgid2[i] = -1;
        __syncthreads();
        return 0;
    }
    {
        int gid = n_groups + hv[0], moff = members0 + hv[1];
        #pragma unroll 1
        for (int i = r0; i < r1; ++i) {
            if (!is_sub_leader(i)) continue;
            CascGroup cg;
            cg.leader = i;
            cg.key_base = scg[parent[i]].prefix_len;
            cg.prefix_len = pg2[i] * ps;
            cg.n_members = cnt2[i];
            cg.member_off = moff;
            cg.n_chunks = 0;
            cg.chunk_keys = 0;
            cg.unit_off = 0;
            cg.n_units = 0;
            cg.level = scg[parent[i]].level + 1;
            cg.pad0 = cg.pad1 = 0;
            store_record(&cgroups[gid], cg);
            scg[gid] = cg;
            cgid2[i] = gid;
            cnt2[i] = moff;  // next free member slot of the sub-group
            moff += cg.n_members;
            ++gid;
        }
    }
    const int n_new = ht[0];
    *members_total = ht[1];
    __syncthreads();
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads) {
        const int ld = lead2[i];
        if (ld >= 0 && ld != i) cgid2[i] = cgid2[ld];
    }
    __syncthreads();
    return n_new;
}

// Pass 0 of the kernel below once some candidates share a first page: each member's
// prefix with its leader (page-id compare), the top-level group records and each
// member's group id.  Out of line, like the chunk planning below and the deeper levels
// (find_next_level): most batches have no shared first page, and this code, inlined, lay
// between the passes every batch runs, where the instruction fetch streamed through it
// (3 to 8 us more per prepare, measured with the forward's kernels queued behind it).
// Returns the number of groups and of their member-list entries.
__device__ __noinline__ int2 build_prefix_groups(const PrepareParams& p, int32_t* dyn, int (*s_tmp2)[2]) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int B = p.batch, ps = p.page_size, stride = p.smem_batch + 1;
    const int chunk_req = (B + kThreads - 1) / kThreads;
    const int r0 = min(B, tid * chunk_req), r1 = min(B, r0 + chunk_req);
    auto sa = [&](int a) { return dyn + a * stride; };
    const int hbits = casc_hash_bits(p.smem_batch);
    int32_t* hkey = dyn + kNumArrays * stride;
    int32_t* hval = hkey + (1 << hbits);
    CascGroup* scg = reinterpret_cast<CascGroup*>(hval + (1 << hbits));
    CascGroup* cgroups = reinterpret_cast<CascGroup*>(p.ws + p.lay.casc_groups);
    int32_t* first = sa(kFirst);
    int32_t* leader = sa(kLeader);
    int32_t* lcp = sa(kLcp);
    int32_t* cnt = sa(kCnt);
    int32_t* lim = sa(kMpos);
    int n_cgroups = 0;
    // Every member compares pages 1 .. lim-1 of its row with the leader's (page 0
    // matched by construction), one warp per member: lanes read consecutive page ids,
    // so each load instruction is one line of each row, 256 ids per step, up to the
    // first mismatch or the group's prefix as found so far.  The group prefix is the
    // smallest mismatch, or the smallest member's page count.
    // The rows about to be compared (members' and leaders' page ids up to the pages
    // compared) are requested into L2 here, all at once, so that the warps' compare steps
    // below, one member after another, mostly find them there.  Only rows of requests
    // that share a first page are touched: a batch without such requests reads no row.
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads) {
        const int ld = leader[i];
        const int l = (ld >= 0 && ld != i) ? min(lcp[i], lcp[ld]) : 0;
        lim[i] = l;
        const int pf = l > 0 ? l : ((ld == i && cnt[i] >= 2) ? lcp[i] : 0);
        const char* row = reinterpret_cast<const char*>(p.page_table + (int64_t)i * p.ld);
        for (int off = 4; off < pf * 4; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
    }
    __syncthreads();
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads)
        if (lim[i] > 0) atomicMin(&lcp[leader[i]], lim[i]);
    {
        const int warp = tid >> 5;
        #pragma unroll 1
        for (int i = warp; i < B; i += kWarps) {
            const int l = lim[i];
            if (l <= 1) continue;  // warp-uniform: i is the same for the whole warp
            const int ld = leader[i];
            const int mis = first_mismatch(p.page_table + (int64_t)i * p.ld, p.page_table + (int64_t)ld * p.ld, 1,
                                           l, &lcp[ld], lane);
            if (lane == 0 && mis < l) atomicMin(&lcp[ld], mis);
        }
    }
    __syncthreads();
    // group ids in leader order (a deterministic plan) and member slot ranges
    int gv[2] = {0, 0};
    #pragma unroll 1
    for (int i = r0; i < r1; ++i)
        if (is_group_leader(leader, cnt, lcp, i, p.min_cascade_pages)) {
            gv[0] += 1;
            gv[1] += cnt[i];
        }
    int gt[2];
    {
        const int4 r = block_scan2(gv[0], gv[1], s_tmp2);
        gv[0] = r.x, gv[1] = r.y, gt[0] = r.z, gt[1] = r.w;
    }
    {
        int gid = gv[0], moff = gv[1];
        #pragma unroll 1
        for (int i = r0; i < r1; ++i) {
            if (!is_group_leader(leader, cnt, lcp, i, p.min_cascade_pages)) continue;
            sa(kCgid)[i] = gid;
            CascGroup cg;
            cg.leader = i;
            cg.prefix_len = lcp[i] * ps;
            cg.n_members = cnt[i];
            cg.member_off = moff;
            cg.n_chunks = 0;
            cg.chunk_keys = 0;
            cg.unit_off = 0;
            cg.n_units = 0;
            cg.key_base = 0;
            cg.level = 0;
            cg.pad0 = cg.pad1 = 0;
            store_record(&cgroups[gid], cg);
            scg[gid] = cg;
            sa(kMpos)[i] = moff;  // next free member slot of the group
            moff += cnt[i];
            ++gid;
        }
    }
    n_cgroups = gt[0];
    __syncthreads();
    // members take the group id of their leader (-1 when the leader leads no group)
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads) {
        const int ld = leader[i];
        if (ld >= 0 && ld != i)
            sa(kCgid)[i] = is_group_leader(leader, cnt, lcp, ld, p.min_cascade_pages) ? sa(kCgid)[ld] : -1;
    }
    __syncthreads();
    return make_int2(n_cgroups, gt[1]);  // groups, member-list entries
}

// Key chunks of each group's prefix (about `target` prefix-pass units in total, see
// below), unit ranges, member lists.  A member takes one partial slot per chunk of each
// of its groups; with n levels in the batch each level gets at most 1/n of the chunks,
// so no member needs more than kMaxCascChunks.  Out of line for the reason given above.
__device__ __noinline__ void plan_prefix_chunks(const PrepareParams& p, int32_t* dyn, int n_cgroups,
                                                int n_levels, unsigned long long work, int (*s_tmp2)[2],
                                                int* s_casc_units) {
    const int tid = threadIdx.x;
    const int B = p.batch, stride = p.smem_batch + 1, TM = p.pre_tokens, Hkv = p.num_kv_heads;
    auto sa = [&](int a) { return dyn + a * stride; };
    const int hbits = casc_hash_bits(p.smem_batch);
    CascGroup* scg = reinterpret_cast<CascGroup*>(dyn + kNumArrays * stride + 2 * (1 << hbits));
    CascGroup* cgroups = reinterpret_cast<CascGroup*>(p.ws + p.lay.casc_groups);
    const int ng = n_cgroups;
    const int nc_cap = kMaxCascChunks / max(n_levels, 1);
    const int gch = (ng + kThreads - 1) / kThreads;
    const int g0 = min(ng, tid * gch), g1 = min(ng, g0 + gch);
    int pv[2] = {0, 0};  // pair units; (member, 16 prefix keys) pairs
    #pragma unroll 1
    for (int g = g0; g < g1; ++g) {
        pv[0] += casc_pair_units(scg[g].n_members, TM, Hkv);
        pv[1] += scg[g].n_members * ((scg[g].prefix_len - scg[g].key_base) / 16);
    }
    int pt[2];
    {
        const int4 r = block_scan2(pv[0], pv[1], s_tmp2);
        pv[0] = r.x, pv[1] = r.y, pt[0] = r.z, pt[1] = r.w;
    }
    const int pair_units = max(pt[0], 1);
    // Units aimed for: the decode tails start on the SMs the prefix pass leaves free, so
    // the pass gets about the share of the SMs its tensor-core time takes beside the
    // tails' HBM time (prefix_pass_target, with the per-SM rates measured on GB300).
    const int target = prefix_pass_target(pt[1], work, p.group, p.kv_fp8, p.lay.casc_target);
    int uv[1] = {0};
    #pragma unroll 1
    for (int g = g0; g < g1; ++g) {
        const CascGroup cg = scg[g];
        const int span = cg.prefix_len - cg.key_base;
        int nc = (target + pair_units - 1) / pair_units;
        nc = max(1, min(nc, min(nc_cap, (span + kPreKeys - 1) / kPreKeys)));
        const int ck = ((span + nc - 1) / nc + kPreKeys - 1) / kPreKeys * kPreKeys;
        uv[0] += (span + ck - 1) / ck * casc_pair_units(cg.n_members, TM, Hkv);
    }
    int ut[1];
    {
        const int4 r = block_scan2(uv[0], 0, s_tmp2);
        uv[0] = r.x, ut[0] = r.z;
    }
    int uoff = uv[0];
    #pragma unroll 1
    for (int g = g0; g < g1; ++g) {
        CascGroup cg = scg[g];
        const int span = cg.prefix_len - cg.key_base;
        int nc = (target + pair_units - 1) / pair_units;
        nc = max(1, min(nc, min(nc_cap, (span + kPreKeys - 1) / kPreKeys)));
        const int ck = ((span + nc - 1) / nc + kPreKeys - 1) / kPreKeys * kPreKeys;
        cg.chunk_keys = ck;
        cg.n_chunks = (span + ck - 1) / ck;
        cg.unit_off = uoff;
        cg.n_units = cg.n_chunks * casc_pair_units(cg.n_members, TM, Hkv);
        sa(kCUoff)[g] = uoff;
        uoff += cg.n_units;
        store_record(&cgroups[g], cg);
        scg[g] = cg;
    }
    if (tid == 0) *s_casc_units = ut[0];
    // each member takes a slot of its group's member list at every level it belongs to
    // (filled when its decode group is written below): level 1's goes to the first-page
    // array, free again; level 2's to kLcp, free since the searches ended; a deeper level's
    // replaces the request's own leader entry at that level, read only by itself
    #pragma unroll 1
    for (int i = tid; i < B; i += kThreads) {
        if (sa(kCgid)[i] < 0) continue;
        sa(kFirst)[i] = atomicAdd(&sa(kMpos)[sa(kLeader)[i]], 1);
        if (n_levels < 2 || sa(kCgid2)[i] < 0) continue;
        sa(kLcp)[i] = atomicAdd(&sa(kCnt)[sa(kLeader2)[i]], 1);
        #pragma unroll 1
        for (int L = 3; L <= n_levels; ++L) {
            if (deep_level(p, L, 1)[i] < 0) break;
            int32_t* lead = deep_level(p, L, 0);
            lead[i] = atomicAdd(&deep_level(p, L, 2)[lead[i]], 1);
        }
    }
}

// Pass 3 of the balanced decode split (see the kernel below): the decode groups of this
// thread's requests with their start on the key line (g0) and their pieces (one, plus one
// per CTA share boundary inside the group), and dec_first: for every CTA whose share
// starts inside a group's stretch of the line, that group.  No unit records: the decode
// kernel cuts the pieces.  Inlined: it is on the path of every decode batch, and with the
// shared-prefix steps out of line the kernel spills less with it inlined than with it a
// function of its own (12 against 40 bytes; decode step 126.1 -> 124.1 us).  (A balanced
// plan has no tensor-core unit, hence no shared-prefix group.)
__device__ __forceinline__ void emit_balanced_groups(const PrepareParams& p, const int32_t* cu, const int32_t* lens,
                                                  int r0, int r1, int TB, int gi, int pi, int g0, int share,
                                                  int line, int n_groups, DecGroup* groups) {
    int32_t* dec_first = reinterpret_cast<int32_t*>(p.ws + p.lay.dec_first);
    if (threadIdx.x == 0)  // CTAs whose share starts past the line: no group
        #pragma unroll 1
        for (int c = (line + share - 1) / share; c <= p.lay.dec_ctas; ++c) dec_first[c] = n_groups;
    #pragma unroll 1
    for (int i = r0; i < r1; ++i) {
        const int c0 = cu[i], n = cu[i + 1] - c0, L = lens[i];
        if (n <= 0 || (p.use_prefill && n > TB)) continue;
        const int ng = (n + TB - 1) / TB;
        #pragma unroll 1
        for (int g = 0; g < ng; ++g) {
            const int a0 = g * TB, na = min(TB, n - a0);
            const int kv_end = L - n + a0 + na;
            const int pieces = 1 + (g0 + kv_end - 1) / share - g0 / share;
            DecGroup dg;
            dg.req = i;
            dg.tok0 = c0 + a0;
            dg.ntok = na;
            dg.qpos0 = L - n + a0;
            dg.nsplit = pieces;
            dg.pbase = pieces > 1 ? pi : -1;
            dg.kv_end = kv_end;
            dg.casc = -1;
            dg.nparts = pieces;
            dg.tail0 = 0;
            dg.g0 = g0;
            dg.pad1 = dg.pad2 = dg.pad3 = dg.pad4 = dg.pad5 = 0;
            store_record(&groups[gi], dg);
            const int e16 = g0 + (kv_end + kDecKeysPerStage - 1) / kDecKeysPerStage * kDecKeysPerStage + kDecPieceCost;
            #pragma unroll 1
            for (int c = (g0 + share - 1) / share; c * share < e16 && c <= p.lay.dec_ctas; ++c) dec_first[c] = gi;
            g0 = e16;
            if (pieces > 1) pi += pieces;
            ++gi;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) prepare_kernel(PrepareParams p) {
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.lay.header);
    DecUnit* units = reinterpret_cast<DecUnit*>(p.ws + p.lay.dec_units);
    DecGroup* groups = reinterpret_cast<DecGroup*>(p.ws + p.lay.dec_groups);
    PreTile* tiles = reinterpret_cast<PreTile*>(p.ws + p.lay.pre_tiles);
    CascGroup* cgroups = reinterpret_cast<CascGroup*>(p.ws + p.lay.casc_groups);
    int2* cmembers = reinterpret_cast<int2*>(p.ws + p.lay.casc_members);

    extern __shared__ int32_t dyn[];
    __shared__ uint32_t s_err;
    __shared__ unsigned long long s_work;
    __shared__ int s_tmp3[kWarps][3];
    __shared__ int s_tmp2[kWarps][2];
    __shared__ int s_hist_u[kBuckets];
    __shared__ int s_hist_t[kBuckets];
    __shared__ int s_casc_units;
    __shared__ int s_max_ntok;
    __shared__ int s_share;  // balanced decode split: keys per CTA (0: the unit queue)
    __shared__ int s_line;   // balanced decode split: length of the key line
    __shared__ SearchCtx s_cx;  // the deeper levels' shared-prefix search

    // the store kernel that follows may set up its CTAs now: it reads nothing this kernel
    // writes before its grid_dep_wait
    dev::grid_dep_launch();
    const int tid = threadIdx.x;
    const int B = p.batch;
    const int TB = p.dec_tokens, TM = p.pre_tokens, Hkv = p.num_kv_heads, ps = p.page_size;
    const bool small = p.smem_batch >= B;  // per-request arrays fit in shared memory
    const int stride = p.smem_batch + 1;
    // per-request array a (computed where used: a table of 13 pointers would hold 26 of
    // the kernel's 64 registers)
    auto sa = [&](int a) { return dyn + a * stride; };
    if (tid == 0) {
        s_err = 0;
        s_work = 0;
        s_casc_units = 0;
        s_max_ntok = 0;
    }
    const bool casc = p.use_cascade && small && B >= 2;
    // One round trip for everything that depends on the request index alone: cu, the
    // lengths and (for the shared-prefix search) each row's first page id.  Every later
    // pass works from shared memory; the step runs with cold caches, so each dependent
    // global round trip costs a DRAM latency.
    if (small) {
        #pragma unroll 1
        for (int i = tid; i <= B; i += kThreads) {
            sa(kCu)[i] = p.cu[i];
            if (i < B) sa(kLen)[i] = p.seqlens[i];
            if (casc && i < B) sa(kFirst)[i] = p.page_table[(int64_t)i * p.ld];
            sa(kCgid)[i] = -1;
        }
    }
    __syncthreads();
    const int32_t* cu = small ? sa(kCu) : p.cu;
    const int32_t* lens = small ? sa(kLen) : p.seqlens;
    auto valid_req = [&](int n, int L) { return n >= 0 && n <= L && L <= p.max_kv_len && n <= p.max_q_len; };
    // each thread owns a contiguous run of requests for the counting passes
    const int chunk_req = (B + kThreads - 1) / kThreads;
    const int r0 = min(B, tid * chunk_req), r1 = min(B, r0 + chunk_req);
    // ---- pass 0: shared-prefix groups among single-token decodes.  Requests are keyed
    // by their first page; the lowest-numbered request with a key leads its group; the
    // group's prefix is the run of pages every member shares with the leader (whole pages
    // that lie strictly before each member's query, so no causal mask ever applies to it).
    int n_cgroups = 0;
    int n_levels = 0;  // deepest level with a group (0: none)
    // shared-memory copy of the cascade group records (after the hash table)
    CascGroup* scg = reinterpret_cast<CascGroup*>(dyn + kNumArrays * stride +
                                                  2 * (casc ? (1 << casc_hash_bits(p.smem_batch)) : 0));
    if (casc) {
        int32_t* first = sa(kFirst);
        int32_t* leader = sa(kLeader);
        int32_t* lcp = sa(kLcp);
        int32_t* cnt = sa(kCnt);
        int32_t* lim = sa(kMpos);   // pages compared per member (until the groups are numbered)
        const int hbits = casc_hash_bits(p.smem_batch);
        const int HT = 1 << hbits;  // > 2 * batch: the probe below always meets a free entry
        int32_t* hkey = dyn + kNumArrays * stride;
        int32_t* hval = hkey + HT;
        #pragma unroll 1
        for (int h = tid; h < HT; h += kThreads) {
            hkey[h] = -1;
            hval[h] = 0x7fffffff;
        }
        #pragma unroll 1
        for (int i = tid; i < B; i += kThreads) {
            const int n = cu[i + 1] - cu[i], L = lens[i];
            const bool ok = n == 1 && valid_req(n, L);
            const int pages = ok ? (L - n) / ps : 0;  // whole pages strictly before the query
            const int f = (ok && pages >= p.min_cascade_pages) ? first[i] : -1;
            first[i] = (f >= 0 && f < p.num_pages) ? f : -1;
            lcp[i] = pages;
            cnt[i] = 0;
            leader[i] = -1;
        }
        __syncthreads();
        // Requests sharing a first page mostly sit in the same warps: the lanes of a warp
        // with equal keys act once (lowest lane, which holds the lowest request index), so
        // a group of many requests does not serialise on one shared-memory address.
        const int lane = tid & 31;
        #pragma unroll 1
        for (int i0 = 0; i0 < B; i0 += kThreads) {  // uniform trip count: whole warps take part
            const int i = i0 + tid;
            const int f = i < B ? first[i] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, f);
            const int lead = __ffs(peers) - 1;
            int h = 0;
            if (f >= 0 && lane == lead) {
                uint32_t hh = page_hash(f, hbits);
                while (true) {
                    const int prev = atomicCAS(&hkey[hh], -1, f);
                    if (prev == -1 || prev == f) break;
                    hh = (hh + 1) & (HT - 1);
                }
                atomicMin(&hval[hh], i);
                h = (int)hh;
            }
            h = __shfl_sync(0xffffffffu, h, lead);
            if (f >= 0) leader[i] = h;
        }
        __syncthreads();
        int has_member = 0;
        #pragma unroll 1
        for (int i0 = 0; i0 < B; i0 += kThreads) {
            const int i = i0 + tid;
            const int ld = (i < B && first[i] >= 0) ? hval[leader[i]] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, ld);
            if (ld >= 0) {
                leader[i] = ld;
                if (lane == __ffs(peers) - 1) atomicAdd(&cnt[ld], __popc(peers));
                has_member |= ld != i;
            }
        }
        // no two candidates share a first page (the usual decode batch): no groups
        if (__syncthreads_or(has_member)) {
            const int2 c = build_prefix_groups(p, dyn, s_tmp2);
            n_cgroups = c.x;
            const int members1 = c.y;
            // ---- level 2: sub-groups inside each group, then level 3 inside those, and so
            // on (the level-1 scratch arrays kFirst / kLcp serve every search in turn)
            if (n_cgroups > 0) {
                n_levels = 1;
                if (tid == 0) {
                    s_cx.dyn = dyn;
                    s_cx.hkey = hkey;
                    s_cx.hval = hval;
                    s_cx.scg = scg;
                    s_cx.cgroups = cgroups;
                    s_cx.page_table = p.page_table;
                    s_cx.ld_table = p.ld;
                    s_cx.num_pages = p.num_pages;
                    s_cx.stride = stride;
                    s_cx.hbits = hbits;
                    s_cx.min_pages = p.min_cascade_pages;
                    s_cx.B = B;
                    s_cx.ps = ps;
                    // records the searches may number in all: the shared-memory copy holds smem_batch + 1
                    s_cx.max_groups = min(p.smem_batch + 1, p.lay.max_casc_groups);
                }
                __syncthreads();
                // level 2 inside the top-level groups, then (while the last level found any)
                // each next level inside the one before, through one call site (a second one
                // cost the kernel registers)
                int members = members1;
                #pragma unroll 1
                for (int level = 2; level <= kMaxCascLevels; ++level) {
                    const bool l2 = level == 2;
                    int m_new = 0;
                    const int n_new = find_next_level(
                        &s_cx, l2 ? sa(kCgid) : level == 3 ? sa(kCgid2) : deep_level(p, level - 1, 1), sa(kFirst),
                        sa(kLcp), l2 ? sa(kCnt) : deep_level(p, level, 2), l2 ? sa(kLeader2) : deep_level(p, level, 0),
                        l2 ? sa(kCgid2) : deep_level(p, level, 1), n_cgroups, members, s_tmp2, &m_new);
                    n_cgroups += n_new;
                    members += m_new;
                    if (n_new == 0) break;
                    n_levels = level;
                }
            }
        }
    }
    // request i's group at level L (-1: none; a member at level L is one at every level
    // above it)
    auto casc_at = [&](int i, int L) {
        if (L > n_levels) return -1;
        return L == 1 ? sa(kCgid)[i] : L == 2 ? sa(kCgid2)[i] : deep_level(p, L, 1)[i];
    };
    auto casc_of = [&](int i) { return casc_at(i, 1); };
    // keys before request i's decode tail: its deepest shared prefix (0 for no group)
    auto prefix_of = [&](int i) {
        int lp = 0;
        #pragma unroll 1
        for (int L = 1; L <= n_levels; ++L) {
            const int g = casc_at(i, L);
            if (g < 0) break;
            lp = scg[g].prefix_len;
        }
        return lp;
    };
    // prefix partial slots of request i (its groups' chunks)
    auto prefix_parts = [&](int i) {
        int np = 0;
        #pragma unroll 1
        for (int L = 1; L <= n_levels; ++L) {
            const int g = casc_at(i, L);
            if (g < 0) break;
            np += scg[g].n_chunks;
        }
        return np;
    };

    // ---- pass 1: validate, count decode groups and prefill tiles, sum decode key extents
    uint32_t err = 0;
    int cnt[3] = {0, 0, 0};  // decode groups, prefill tile pairs x kv heads, decode key line
    unsigned long long work = 0, line = 0;
    int max_ntok = 0;
    if (tid == 0 && cu[0] != 0) err |= kErrCu;
    if (tid == 0 && B > p.max_batch) err |= kErrLimits;
    if (tid == 0 && p.total_tokens > p.max_tokens) err |= kErrLimits;
    #pragma unroll 1
    for (int i = r0; i < r1; ++i) {
        const int c0 = cu[i], c1 = cu[i + 1], L = lens[i];
        const int n = c1 - c0;
        if (n < 0) err |= kErrCu;
        if (i == B - 1 && c1 != p.total_tokens) err |= kErrCu;
        if (L < 0 || n > L) err |= kErrQgtKv;
        if (L > p.max_kv_len || n > p.max_q_len) err |= kErrLimits;
        if (n <= 0 || !valid_req(n, L)) continue;
        if (p.use_prefill && n > TB) {
            cnt[1] += (int)((((n + TM - 1) / TM) + 1) / 2) * Hkv;  // units of two Q tiles
        } else {
            const int ng = (n + TB - 1) / TB;
            cnt[0] += ng;
            max_ntok = max(max_ntok, min(n, TB));
            const int lp = prefix_of(i);
            #pragma unroll 1
            for (int g = 0; g < ng; ++g) {
                const int ext = L - n + min((g + 1) * TB, n) - lp;
                work += (unsigned long long)ext;
                line += (unsigned long long)((ext + kDecKeysPerStage - 1) / kDecKeysPerStage * kDecKeysPerStage +
                                             kDecPieceCost);
            }
        }
    }
    cnt[2] = (int)min(line, (unsigned long long)kLineLimit);
    if (err) atomicOr(&s_err, err);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) work += __shfl_xor_sync(0xffffffffu, work, o);
    if ((tid & 31) == 0 && work) atomicAdd(&s_work, work);
    max_ntok = __reduce_max_sync(0xffffffffu, max_ntok);
    if ((tid & 31) == 0 && max_ntok) atomicMax(&s_max_ntok, max_ntok);
    int tot3[3];
    block_scan<3>(cnt, tot3, s_tmp3);  // cnt now holds this thread's exclusive offsets
    // first prefill unit and first decode group of each request: the emission below runs
    // in parallel over units and finds a unit's request by binary search
    int32_t* tile_off = small ? sa(kToff) : reinterpret_cast<int32_t*>(p.ws + p.lay.req_scratch);
    {
        int toff = cnt[1], goff = cnt[0];
        #pragma unroll 1
        for (int i = r0; i < r1; ++i) {
            tile_off[i] = toff;
            if (small) sa(kGoff)[i] = goff;
            const int n = cu[i + 1] - cu[i], L = lens[i];
            if (n > 0 && valid_req(n, L)) {
                if (p.use_prefill && n > TB) toff += (int)((((n + TM - 1) / TM) + 1) / 2) * Hkv;
                else goff += (n + TB - 1) / TB;
            }
        }
        if (tid == 0) tile_off[B] = tot3[1];
    }

    // ---- shared-prefix groups: key chunks, unit ranges, member lists (out of line)
    if (casc && n_cgroups > 0)
        plan_prefix_chunks(p, dyn, n_cgroups, n_levels, s_work, s_tmp2, &s_casc_units);
    __syncthreads();
    const int tiles_total = tot3[1] + s_casc_units;
    if (tot3[0] > p.lay.max_dec_groups || tiles_total > p.lay.max_pre_tiles) {
        if (tid == 0) atomicOr(&s_err, kErrLimits);
    }
    __syncthreads();
    const uint32_t fatal = s_err & kErrFatal;

    // ---- split-KV chunk: the decode work spread over ~target_units CTAs
    int chunk = 0x3fffffff;
    if (p.split_kv && s_work > 0) {
        unsigned long long c = (s_work + p.lay.target_units - 1) / p.lay.target_units;
        c = (c + kDecKeysPerStage - 1) / kDecKeysPerStage * kDecKeysPerStage;
        chunk = (int)(c > (unsigned long long)kMinSplitChunk ? c : (unsigned long long)kMinSplitChunk);
    }
    // ---- balanced split: with no tensor-core unit every decode CTA starts at once, so the
    // decode groups' keys (each group padded to whole 16-key stages and followed by a gap of
    // kDecPieceCost keys, the cost of starting a piece) are laid end to end on one line and
    // CTA c takes the line's keys [c * share, (c + 1) * share): equal work per CTA, and a
    // group is cut only where a CTA's share ends (fewer partials than queued
    // units of one chunk each, which also left the grid's last units as a tail).  The
    // decode kernel cuts its pieces from the group records (g0: the group's start on the
    // line) and dec_first (the group the CTA's share starts in).
    // (kept in shared memory and read where used: this kernel has 64 registers a thread)
    // (the line is cut at most once per decode CTA: that many more units than groups, and
    // at most two partial slots per cut; a workspace planned for fewer split-KV units than
    // decode CTAs takes the unit queue instead)
    if (tid == 0) {
        int share = 0;
        const bool fits = p.lay.max_dec_units >= tot3[0] + p.lay.dec_ctas + 1 &&
                          p.lay.max_partial >= 2 * p.lay.dec_ctas + 2;
        if (p.split_kv && tiles_total == 0 && Hkv <= kDecHeadBlock && s_work > 0 && s_work < kLineLimit / 2 &&
            fits) {
            const int per_cta = (tot3[2] + p.lay.dec_ctas - 1) / p.lay.dec_ctas;
            share = max(kMinDecShare, (per_cta + kDecKeysPerStage - 1) / kDecKeysPerStage * kDecKeysPerStage);
        }
        s_share = share;
        s_line = tot3[2];
    }

    // ---- pass 2: units and partial slots per thread's requests, and the unit cost
    // histogram (a group's units all have length `per` but the last)
    #pragma unroll 1
    for (int b = tid; b < kBuckets; b += kThreads) {
        s_hist_u[b] = 0;
        s_hist_t[b] = 0;
    }
    __syncthreads();
    int cnt2[2] = {0, 0};  // units, partial slots
    if (!fatal) {
        const int share = s_share;
        int g0 = cnt[2];  // balanced split: this thread's first group's start on the line
        #pragma unroll 1
        for (int i = r0; i < r1; ++i) {
            const int n = cu[i + 1] - cu[i], L = lens[i];
            if (n <= 0 || (p.use_prefill && n > TB)) continue;
            const int ng = (n + TB - 1) / TB;
            const int lp = prefix_of(i);
            const int npre = prefix_parts(i);
            #pragma unroll 1
            for (int g = 0; g < ng; ++g) {
                const int ext = L - n + min((g + 1) * TB, n) - lp;
                if (share > 0) {  // pieces: one, plus one per CTA share boundary inside the group
                    const int pieces = 1 + (g0 + ext - 1) / share - g0 / share;
                    cnt2[0] += pieces;
                    if (pieces > 1) cnt2[1] += pieces;
                    g0 += (ext + kDecKeysPerStage - 1) / kDecKeysPerStage * kDecKeysPerStage + kDecPieceCost;
                    continue;
                }
                int per;
                const int s = split_ranges(ext, chunk, &per);
                const int nparts = s + npre;
                cnt2[0] += s;
                if (nparts > 1) cnt2[1] += nparts;
                const int last = max(0, ext - (s - 1) * per);
                if (s <= 0) continue;
                if (s > 1) atomicAdd(&s_hist_u[cost_bucket(per / kDecKeysPerStage)], s - 1);
                atomicAdd(&s_hist_u[cost_bucket((last + kDecKeysPerStage - 1) / kDecKeysPerStage)], 1);
            }
        }
    }
    int tot2[2];
    {
        const int4 r = block_scan2(cnt2[0], cnt2[1], s_tmp2);
        cnt2[0] = r.x, cnt2[1] = r.y, tot2[0] = r.z, tot2[1] = r.w;
    }
    const bool over = tot2[0] > p.lay.max_dec_units || tot2[1] > p.lay.max_partial;
    if (over && tid == 0) atomicOr(&s_err, kErrLimits);
    const bool run = !fatal && !over;

    // tile pair / prefix-pass unit x -> its record and cost
    auto make_tile = [&](int x, PreTile& pt) -> int {
        if (x < tot3[1]) {  // (request, pair of Q tiles, kv head)
            const int i = find_bucket(tile_off, B, x);
            const int lx = x - tile_off[i];
            const int c0 = cu[i], n = cu[i + 1] - c0, L = lens[i];
            const int nt = (n + TM - 1) / TM;
            const int t = 2 * (lx / Hkv), h = lx % Hkv;  // Q tiles t and t+1
            const int a0 = t * TM, na0 = min(TM, n - a0);
            const int na1 = t + 1 < nt ? min(TM, n - a0 - TM) : 0;
            pt.req = i;
            pt.kvh = h;
            pt.tok0 = c0 + a0;
            pt.ntok0 = na0;
            pt.ntok1 = na1;
            pt.qpos0 = L - n + a0;
            pt.kv_end0 = L - n + a0 + na0;
            pt.kv_end1 = na1 > 0 ? pt.kv_end0 + na1 : pt.kv_end0;
            return (pt.kv_end1 + kPreKeys - 1) / kPreKeys;
        }
        // (cascade group, key chunk, pair of member tiles, kv head)
        const int y = x - tot3[1];
        const int g = find_bucket(sa(kCUoff), n_cgroups, y);
        const CascGroup cgr = scg[g];
        const int ly = y - cgr.unit_off;
        const int pu = casc_pair_units(cgr.n_members, TM, Hkv);
        const int c = ly / pu, rest = ly % pu;
        const int pair = rest / Hkv, h = rest % Hkv;
        const int m0 = pair * 2 * TM;
        pt.req = -1 - g;
        pt.kvh = h;
        pt.tok0 = cgr.member_off + m0;
        pt.ntok0 = min(TM, cgr.n_members - m0);
        pt.ntok1 = max(0, min(TM, cgr.n_members - m0 - TM));
        pt.qpos0 = c;
        pt.kv_end0 = cgr.key_base + c * cgr.chunk_keys;
        pt.kv_end1 = min(cgr.prefix_len, cgr.key_base + (c + 1) * cgr.chunk_keys);
        return (pt.kv_end1 - pt.kv_end0 + kPreKeys - 1) / kPreKeys;
    };
    if (run) {
        #pragma unroll 1
        for (int x = tid; x < tiles_total; x += kThreads) {
            PreTile pt;
            atomicAdd(&s_hist_t[cost_bucket(make_tile(x, pt))], 1);
        }
    }
    __syncthreads();

    // ---- pass 3: write groups; units and tiles go out longest first (a counting sort on
    // their cost), so that the kernels' in-order work fetch ends with the short items and
    // the grid finishes together (longest-processing-time-first).  The position of a
    // unit in the list never changes a result: each split writes its own partial slot and
    // the merge walks the slots in split order.
    if (tid < 32) {  // bucket counts -> first position of each bucket (bucket 0 = costliest)
        constexpr int kPer = kBuckets / 32;
        int su = 0, st = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            su += s_hist_u[tid * kPer + k];
            st += s_hist_t[tid * kPer + k];
        }
        int iu = su, itt = st;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yu = __shfl_up_sync(0xffffffffu, iu, o), yt = __shfl_up_sync(0xffffffffu, itt, o);
            if (tid >= o) {
                iu += yu;
                itt += yt;
            }
        }
        int au = iu - su, at = itt - st;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int cu_ = s_hist_u[tid * kPer + k], ct = s_hist_t[tid * kPer + k];
            s_hist_u[tid * kPer + k] = au;
            s_hist_t[tid * kPer + k] = at;
            au += cu_;
            at += ct;
        }
    }
    __syncthreads();
    if (run && s_share > 0) {
        emit_balanced_groups(p, cu, lens, r0, r1, TB, cnt[0], cnt2[1], cnt[2], s_share, s_line, tot3[0], groups);
    } else if (run) {
        int gi = cnt[0], pi = cnt2[1];
        #pragma unroll 1
        for (int i = r0; i < r1; ++i) {
            const int c0 = cu[i], n = cu[i + 1] - c0, L = lens[i];
            if (n <= 0) continue;
            if (p.use_prefill && n > TB) continue;  // prefill units: emitted below
            const int ng = (n + TB - 1) / TB;
            const int lp = prefix_of(i);
            const int cg = casc_of(i);
            const int npre = prefix_parts(i);
            #pragma unroll 1
            for (int g = 0; g < ng; ++g) {
                const int a0 = g * TB, na = min(TB, n - a0);
                const int kv_end = L - n + a0 + na;
                int per;
                const int s = split_ranges(kv_end - lp, chunk, &per);
                const int nparts = s + npre;
                DecGroup dg;
                dg.req = i;
                dg.tok0 = c0 + a0;
                dg.ntok = na;
                dg.qpos0 = L - n + a0;
                dg.nsplit = s;
                dg.pbase = nparts > 1 ? pi : -1;
                dg.kv_end = kv_end;
                dg.casc = cg;
                dg.nparts = nparts;
                dg.tail0 = lp;
                dg.g0 = 0;
                dg.pad1 = dg.pad2 = dg.pad3 = dg.pad4 = dg.pad5 = 0;
                store_record(&groups[gi], dg);
                // member list entries of a shared-prefix member (one new token): its q row and
                // the partial slot of chunk 0 of each of its groups, level by level (each
                // level's chunks after those of the level above)
                if (cg >= 0) {
                    int slot = pi + s;
                    cmembers[sa(kFirst)[i]] = make_int2(dg.tok0, slot);
                    slot += scg[cg].n_chunks;
                    #pragma unroll 1
                    for (int lv = 2; lv <= n_levels; ++lv) {
                        const int gl = casc_at(i, lv);
                        if (gl < 0) break;
                        cmembers[lv == 2 ? sa(kLcp)[i] : deep_level(p, lv, 0)[i]] = make_int2(dg.tok0, slot);
                        slot += scg[gl].n_chunks;
                    }
                }
                for (int u = 0; u < s; ++u) {
                    DecUnit du;
                    du.group = gi;
                    du.k0 = min(kv_end, lp + u * per);
                    du.k1 = min(kv_end, lp + (u + 1) * per);
                    du.split = u;
                    du.req = i;
                    du.tok0 = dg.tok0;
                    du.ntok = dg.ntok;
                    du.qpos0 = dg.qpos0;
                    du.nsplit = s;
                    du.pbase = dg.pbase;
                    du.nparts = nparts;
                    du.pad1 = 0;
                    const int b = cost_bucket((du.k1 - du.k0 + kDecKeysPerStage - 1) / kDecKeysPerStage);
                    store_record(&units[atomicAdd(&s_hist_u[b], 1)], du);
                }
                if (nparts > 1) pi += nparts;
                ++gi;
            }
        }
        // prefill tile pairs, then cascade prefix units, in parallel over the unit index
        #pragma unroll 1
        for (int x = tid; x < tiles_total; x += kThreads) {
            PreTile pt;
            const int b = cost_bucket(make_tile(x, pt));
            store_record(&tiles[atomicAdd(&s_hist_t[b], 1)], pt);
        }
    }

    // ---- the request of every new token, from which the store kernel derives the slot
    // mapping when the caller passed none (its many warps then load the page ids side by
    // side; here, one thread per token would wait for them one after another)
    if (run && p.tok_req != nullptr) {
        // each thread a contiguous run of tokens: one search for its first token's request
        // (request i with cu[i] <= t < cu[i+1]), then a walk
        const int per = (p.total_tokens + kThreads - 1) / kThreads;
        const int t0 = min(p.total_tokens, tid * per), t1 = min(p.total_tokens, t0 + per);
        int i = t0 < t1 ? find_bucket(cu, B, t0) : 0;
        #pragma unroll 1
        for (int t = t0; t < t1; ++t) {
            while (cu[i + 1] <= t) ++i;
            p.tok_req[t] = i;
        }
    }
    __syncthreads();
    if (tid == 0) {
        const bool ok = (s_err & kErrFatal) == 0;
        hdr->error_bits = s_err;
        hdr->n_dec_groups = ok ? tot3[0] : 0;
        hdr->n_pre_tiles = ok ? tiles_total : 0;
        hdr->n_dec_units = ok ? tot2[0] : 0;
        hdr->n_partial_slots = ok ? tot2[1] : 0;
        hdr->split_chunk = chunk;
        hdr->n_casc_groups = ok ? n_cgroups : 0;
        hdr->n_casc_levels = ok ? n_levels : 0;
        hdr->n_casc_tiles = ok ? s_casc_units : 0;
        hdr->n_casc_units = ok ? s_casc_units : 0;
        hdr->max_group_tokens = ok ? s_max_ntok : 0;
        hdr->dec_share = ok ? s_share : 0;
        hdr->wait_override = 0;
    }
}

}  // namespace

size_t prepare_smem_bytes(int smem_batch, bool cascade) {
    size_t words = (size_t)kNumArrays * (smem_batch + 1);
    // hash table, then group records (top level and sub-groups: one per pair of requests each)
    if (cascade) words += 2 * ((size_t)1 << casc_hash_bits(smem_batch)) + (smem_batch + 1) * (sizeof(CascGroup) / 4);
    return words * sizeof(int32_t);
}

cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t s) {
    const size_t smem = prepare_smem_bytes(p.smem_batch, p.use_cascade != 0);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    prepare_kernel<<<1, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pva
