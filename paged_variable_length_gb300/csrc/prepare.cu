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
//   1. validate cu_seqlens_q / cache_seqlens (error word, never a trap);
//   2. classify each request: q_len * G <= 16 rows -> decode groups (the
//      warp-MMA streaming kernel), otherwise -> 128-row tensor-core tiles;
//   3. split-KV plan: choose one chunk length so that the decode work fills the
//      GPU, split each group's visible key range into near-equal chunks;
//   4. prefill tiles: causal KV extent of each tile (keys past the tile's last
//      query are never loaded);
//   5. derive slot_mapping from the page table when the caller passed none.
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "pva_internal.h"

namespace pva {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 256;  // cost classes for the longest-first ordering of work items

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

__global__ void __launch_bounds__(kThreads, 1) prepare_kernel(PrepareParams p) {
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.lay.header);
    DecUnit* units = reinterpret_cast<DecUnit*>(p.ws + p.lay.dec_units);
    DecGroup* groups = reinterpret_cast<DecGroup*>(p.ws + p.lay.dec_groups);
    PreTile* tiles = reinterpret_cast<PreTile*>(p.ws + p.lay.pre_tiles);
    uint32_t* counters = reinterpret_cast<uint32_t*>(p.ws + p.lay.counters);

    __shared__ uint32_t s_err;
    __shared__ unsigned long long s_work;
    __shared__ int s_tmp3[kWarps][3];
    __shared__ int s_tmp2[kWarps][2];
    __shared__ int s_hist_u[kBuckets];
    __shared__ int s_hist_t[kBuckets];
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_err = 0;
        s_work = 0;
    }
    __syncthreads();

    const int B = p.batch;
    const int TB = p.dec_tokens, TM = p.pre_tokens, Hkv = p.num_kv_heads;
    const int chunk_req = (B + kThreads - 1) / kThreads;
    const int r0 = min(B, tid * chunk_req), r1 = min(B, r0 + chunk_req);

    // ---- pass 1: validate, count decode groups and prefill tiles, sum decode key extents
    uint32_t err = 0;
    int cnt[3] = {0, 0, 0};  // groups, tiles, (unused)
    unsigned long long work = 0;
    if (tid == 0 && p.cu[0] != 0) err |= kErrCu;
    if (tid == 0 && B > p.max_batch) err |= kErrLimits;
    if (tid == 0 && p.total_tokens > p.max_tokens) err |= kErrLimits;
    for (int i = r0; i < r1; ++i) {
        const int c0 = p.cu[i], c1 = p.cu[i + 1], L = p.seqlens[i];
        const int n = c1 - c0;
        if (n < 0) err |= kErrCu;
        if (i == B - 1 && c1 != p.total_tokens) err |= kErrCu;
        if (L < 0 || n > L) err |= kErrQgtKv;
        if (L > p.max_kv_len || n > p.max_q_len) err |= kErrLimits;
        if (n <= 0 || n > L || L > p.max_kv_len || n > p.max_q_len) continue;
        if (p.use_prefill && n > TB) {
            cnt[1] += (int)((((n + TM - 1) / TM) + 1) / 2) * Hkv;  // units of two Q tiles
        } else {
            const int ng = (n + TB - 1) / TB;
            cnt[0] += ng;
            for (int g = 0; g < ng; ++g) work += (unsigned long long)(L - n + min((g + 1) * TB, n));
        }
    }
    if (err) atomicOr(&s_err, err);
    if (work) atomicAdd(&s_work, work);
    int tot3[3];
    block_scan<3>(cnt, tot3, s_tmp3);  // cnt now holds this thread's exclusive offsets
    if (tot3[0] > p.lay.max_dec_groups || tot3[1] > p.lay.max_pre_tiles) {
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

    // ---- pass 2: units and partial slots per thread's requests
    int cnt2[2] = {0, 0};  // units, partial slots
    if (!fatal) {
        for (int i = r0; i < r1; ++i) {
            const int n = p.cu[i + 1] - p.cu[i], L = p.seqlens[i];
            if (n <= 0 || (p.use_prefill && n > TB)) continue;
            const int ng = (n + TB - 1) / TB;
            for (int g = 0; g < ng; ++g) {
                const int ext = L - n + min((g + 1) * TB, n);
                int per;
                const int s = split_ranges(ext, chunk, &per);
                cnt2[0] += s;
                if (s > 1) cnt2[1] += s;
            }
        }
    }
    int tot2[2];
    block_scan<2>(cnt2, tot2, s_tmp2);
    if (tot2[0] > p.lay.max_dec_units || tot2[1] > p.lay.max_partial) {
        if (tid == 0) atomicOr(&s_err, kErrLimits);
    }
    __syncthreads();
    const bool run = (s_err & kErrFatal) == 0;

    // ---- pass 3: write groups; units and tiles go out longest first (a counting sort on
    // their cost), so that the kernels' in-order work fetch ends with the short items and
    // the grid finishes together (longest-processing-time-first).  The position of a
    // unit in the list never changes a result: each split writes its own partial slot and
    // the merge walks the slots in split order.
    for (int b = tid; b < kBuckets; b += kThreads) {
        s_hist_u[b] = 0;
        s_hist_t[b] = 0;
    }
    __syncthreads();
    for (int emit = 0; emit < 2; ++emit) {
        if (run) {
            int gi = cnt[0], pi = cnt2[1];
            for (int i = r0; i < r1; ++i) {
                const int c0 = p.cu[i], n = p.cu[i + 1] - c0, L = p.seqlens[i];
                if (n <= 0) continue;
                if (p.use_prefill && n > TB) {
                    const int nt = (n + TM - 1) / TM;
                    for (int t = 0; t < nt; t += 2) {  // a unit: Q tiles t and t+1
                        const int a0 = t * TM, na0 = min(TM, n - a0);
                        const int na1 = t + 1 < nt ? min(TM, n - a0 - TM) : 0;
                        const int kv_end0 = L - n + a0 + na0;
                        const int kv_end1 = na1 > 0 ? kv_end0 + na1 : kv_end0;
                        const int b = kBuckets - 1 - min(kBuckets - 1, (kv_end1 + kPreKeys - 1) / kPreKeys);
                        for (int h = 0; h < Hkv; ++h) {
                            if (!emit) {
                                atomicAdd(&s_hist_t[b], 1);
                                continue;
                            }
                            PreTile pt;
                            pt.req = i;
                            pt.kvh = h;
                            pt.tok0 = c0 + a0;
                            pt.ntok0 = na0;
                            pt.ntok1 = na1;
                            pt.qpos0 = L - n + a0;
                            pt.kv_end0 = kv_end0;
                            pt.kv_end1 = kv_end1;
                            tiles[atomicAdd(&s_hist_t[b], 1)] = pt;
                        }
                    }
                    continue;
                }
                const int ng = (n + TB - 1) / TB;
                for (int g = 0; g < ng; ++g) {
                    const int a0 = g * TB, na = min(TB, n - a0);
                    const int ext = L - n + a0 + na;
                    int per;
                    const int s = split_ranges(ext, chunk, &per);
                    DecGroup dg;
                    dg.req = i;
                    dg.tok0 = c0 + a0;
                    dg.ntok = na;
                    dg.qpos0 = L - n + a0;
                    dg.nsplit = s;
                    dg.pbase = s > 1 ? pi : -1;
                    dg.kv_end = ext;
                    dg.casc = -1;
                    if (emit) {
                        groups[gi] = dg;
                        counters[gi] = 0;
                    }
                    for (int u = 0; u < s; ++u) {
                        DecUnit du;
                        du.group = gi;
                        du.k0 = min(ext, u * per);
                        du.k1 = min(ext, (u + 1) * per);
                        const int b = kBuckets - 1 - min(kBuckets - 1, (du.k1 - du.k0 + kDecKeysPerStage - 1) /
                                                                           kDecKeysPerStage);
                        if (!emit) {
                            atomicAdd(&s_hist_u[b], 1);
                            continue;
                        }
                        du.split = u;
                        du.req = i;
                        du.tok0 = dg.tok0;
                        du.ntok = dg.ntok;
                        du.qpos0 = dg.qpos0;
                        du.nsplit = dg.nsplit;
                        du.pbase = dg.pbase;
                        du.pad0 = du.pad1 = 0;
                        units[atomicAdd(&s_hist_u[b], 1)] = du;
                    }
                    if (s > 1) pi += s;
                    ++gi;
                }
            }
        }
        __syncthreads();
        if (!emit && tid == 0) {  // bucket counts -> first position of each bucket (bucket 0 = costliest)
            int au = 0, at = 0;
            for (int b = 0; b < kBuckets; ++b) {
                const int cu_ = s_hist_u[b], ct = s_hist_t[b];
                s_hist_u[b] = au;
                s_hist_t[b] = at;
                au += cu_;
                at += ct;
            }
        }
        __syncthreads();
    }

    // ---- derived slot mapping: the new tokens are each request's last q_len positions
    if (run && p.derived_slots != nullptr) {
        uint32_t perr = 0;
        for (int t = tid; t < p.total_tokens; t += kThreads) {
            int lo = 0, hi = B - 1;  // request i with cu[i] <= t < cu[i+1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.cu[mid] <= t) lo = mid;
                else hi = mid - 1;
            }
            const int i = lo;
            const int n = p.cu[i + 1] - p.cu[i], L = p.seqlens[i];
            const int pos = L - n + (t - p.cu[i]);
            const int64_t page = p.page_table[(int64_t)i * p.ld + pos / p.page_size];
            int64_t slot = -1;
            if (page < 0 || page >= p.num_pages) perr |= kErrPage;
            else slot = page * p.page_size + pos % p.page_size;
            p.derived_slots[t] = slot;
        }
        if (perr) atomicOr(&s_err, perr);
    }
    __syncthreads();
    if (tid == 0) {
        const bool ok = (s_err & kErrFatal) == 0;
        hdr->error_bits = s_err;
        hdr->n_dec_groups = ok ? tot3[0] : 0;
        hdr->n_pre_tiles = ok ? tot3[1] : 0;
        hdr->n_dec_units = ok ? tot2[0] : 0;
        hdr->n_partial_slots = ok ? tot2[1] : 0;
        hdr->split_chunk = chunk;
        hdr->n_casc_groups = 0;
        hdr->n_casc_tiles = 0;
        hdr->n_casc_units = 0;
    }
}

}  // namespace

cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t s) {
    prepare_kernel<<<1, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pva
