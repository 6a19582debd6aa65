// K3 + K4: decode / small-row attention streaming the paged KV pool, and the
// split-KV log-sum-exp combine as a small kernel right after it.
//
// What it computes is the ch. 5 reference forward ("The attention backend and
// a reference implementation", section "Variable-length, paged attention with
// prefixes") for requests with few new tokens: for every q head h of kv head
// g, softmax(scale * q K^T) V over the request's keys 0..kv_len-1 gathered
// through the page table, with the bottom-right causal mask.  Long KV ranges
// are split over CTAs and recombined by LSE, the split-KV / Flash-Decoding
// scheme "Variable-length batching and one mixed forward pass" (Exercises,
// answer 2) names for decode batches.
//
// GB300 design (one CTA per SM-slot, persistent):
//   * a work unit is (decode group, key range); a group is up to floor(16/G)
//     consecutive new tokens of one request, all q heads;
//   * work distribution: when no tensor-core pass precedes the grid (every CTA starts
//     at once), a balanced split -- the groups' keys on one line, each CTA an equal
//     share, the pieces cut from the group records; otherwise a queue of split-KV
//     chunks, longest first, taken with an atomic counter by CTAs as they start;
//   * producer warp: takes its pieces or units, and for every
//     16-key stage issues one bulk async copy (TMA, 1-D) per key row --
//     Hkv*D bf16 = all kv heads of one slot, 1-2 KiB contiguous in the pool --
//     for K and for V into a ring of shared-memory stages (mbarrier
//     complete_tx).  Rows land 16 bytes apart from a multiple of 128 so the
//     per-head reads below are bank-conflict free;
//   * consumer warp w owns kv head w: its G*ntok (<= 16) query rows are one
//     m16 operand held in registers; S = Q K^T and O += P V run as
//     m16n8k16 warp MMAs (fp32 accumulate) on the staged rows, with an online
//     softmax in registers.  The tcgen05 tensor core's smallest M (64) would
//     leave >= 87% of its rows idle here; the warp MMA keeps the CUDA cores
//     free so the kernel stays bound by HBM, not by issue slots;
//   * split groups write fp32 partial (O, LSE) to the workspace and the CTA
//     moves straight on (no fence, no arrival count, no waiting); the merge
//     kernel then combines every group: lse = log sum_s exp(lse_s),
//     o = sum_s exp(lse_s - lse) o_s.  For a member of a shared-prefix group the
//     units cover only the keys after the prefix, and the merge also takes the
//     prefix-pass partials that the tensor-core kernel wrote.  A merge inside the
//     decode kernel (by the CTA finishing a group last) kept that CTA's
//     consumers from the ring for the whole combine, and the arrival protocol
//     stalled every split unit on a fence and an atomic round trip.
// FP8 pools (F8): the staged rows are E4M3 bytes (half the bytes per key), and the warp
// MMAs take f16 operands: an E4M3 pair becomes an f16 pair with one exact conversion,
// where bf16 would need several instructions per pair.  Q is converted to f16 once per
// unit (exact for 2^-17 <= |q| <= 65504), P is packed as f16.  The dot products may run
// over the head dimension in any order, so each lane reads its K fragments from one
// contiguous run of its key's row (Q uses the same order); for P V each lane owns a
// run of output columns of its four key rows, and the epilogue writes the columns back
// in place.  The per-head scales: k_scale folds into the softmax scale, v_scale into
// the final 1/l.
// Every wait is bounded (PVA_DEVERR_TIMEOUT, then the CTA drains its copies
// and leaves); nothing traps.
#include <cuda_runtime.h>

#include <cfloat>

#include "device_utils.cuh"
#include "pva_internal.h"

namespace pva {
namespace {

constexpr int kMaxKvHeads = kDecHeadBlock;
constexpr int kStageKeys = kDecKeysPerStage;  // 16
constexpr int kRowPad = 16;                    // bytes between consecutive staged rows beyond Hkv*D*2
constexpr float kLn2 = 0.69314718055994530942f;

struct StageInfo {
    int32_t unit, group, k, k1;
    int32_t tok0, ntok, qpos0, nsplit;
    int32_t pbase, split, flags, hb;
    int32_t nparts, pad0, pad1, pad2;
};
constexpr int kFirst = 1, kLast = 2, kEnd = 4;

struct DecSmemHead {
    uint64_t full[8];
    uint64_t empty[8];
    StageInfo info[8];
    int32_t abort_flag;
};

__device__ __forceinline__ void abort_cta(DecSmemHead* sh, uint32_t* err) {
    sh->abort_flag = 1;
    dev::set_error(err, kErrTimeout);
}

// A work wait of one whole warp (every lane calls it, converged): the lanes' results are
// voted, so the warp leaves together or not at all (its next steps -- warp MMAs, fragment
// loads, warp syncs -- need every lane); lane 0 records the abort.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit, DecSmemHead* sh,
                                          uint32_t* err) {
    if (__all_sync(0xffffffffu, dev::mbar_wait(bar, parity, limit))) return true;
    if ((threadIdx.x & 31) == 0) abort_cta(sh, err);
    __syncwarp();
    return false;
}

template <int D, bool F8>
__global__ void __launch_bounds__(32 * (kMaxKvHeads + 1), 1)
    decode_kernel(ForwardParams p, int stages, int row_stride) {
    constexpr int ES = F8 ? 1 : 2;  // bytes per pool element
    extern __shared__ __align__(128) uint8_t smem[];
    DecSmemHead* sh = reinterpret_cast<DecSmemHead*>(smem);
    uint8_t* ring = smem + ((sizeof(DecSmemHead) + 127) / 128) * 128;
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.lay.header);
    uint32_t* err = &hdr->error_bits;
    const uint64_t wlim = dev::wait_limit(hdr->wait_override);  // work waits (drains: the default)

    // a CTA serves HB = min(Hkv, 8) kv heads ("head block"); work item = (unit, head block)
    const int Hkv = p.num_kv_heads, G = p.group, Hq = p.num_qo_heads;
    const int HB = Hkv < kMaxKvHeads ? Hkv : kMaxKvHeads;
    const int n_hb = Hkv / HB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_bytes = HB * D * ES;
    // rows staged back to back (no padding): one copy per stage and pool (see launch_d)
    const bool runs = row_stride == row_bytes;
    const int stage_bytes = 2 * kStageKeys * row_stride;
    // Plan from the prepare kernel (complete before the store kernel released this grid);
    // pool rows, the work counter and the prefix-pass partials only after grid_dep_wait.
    dev::grid_dep_launch();
    const int n_units = hdr->n_dec_units * n_hb;
    // after a tensor-core kernel with units the store kernel has already finished (see
    // ForwardParams::dec_wait_late); the producer warp waits for that grid before it
    // returns (a CTA cannot exit before it), so this grid (and the merge after it)
    // completes after it.  With no unit the tensor-core kernel released this grid at
    // once, and it waits before its work.
    const bool wait_late = p.dec_wait_late && hdr->n_pre_tiles > 0;
    if ((hdr->error_bits & kErrFatal) || n_units == 0) {
        dev::grid_dep_wait();
        return;
    }

    const DecUnit* units = reinterpret_cast<const DecUnit*>(p.ws + p.lay.dec_units);
    const DecGroup* dgroups = reinterpret_cast<const DecGroup*>(p.ws + p.lay.dec_groups);
    // Balanced split (share > 0, planned only when no tensor-core unit precedes this grid):
    // the decode groups' keys lie end to end on one line, each group padded to whole
    // stages and followed by a gap (kDecPieceCost keys, charged for a piece start, that
    // nobody processes), and this CTA takes the line's keys [line_lo, line_hi).  Its pieces are cut
    // from the group records; a piece that starts at a share boundary inside a group is
    // that group's split (boundary index - index of the boundary before the group).
    const int share = hdr->dec_share;
    const int n_groups = hdr->n_dec_groups;
    const int line_lo = (int)blockIdx.x * share, line_hi = line_lo + share;
    auto piece = [&](int g, const DecGroup& dg, DecUnit& du) -> bool {
        const int ext = dg.kv_end - dg.tail0;
        const int a = max(dg.g0, line_lo), e = min(dg.g0 + ext, line_hi);
        if (a >= e) return false;
        du.group = g;
        du.k0 = dg.tail0 + (a - dg.g0);
        du.k1 = dg.tail0 + (e - dg.g0);
        du.split = a == dg.g0 ? 0 : (int)blockIdx.x - dg.g0 / share;
        du.req = dg.req;
        du.tok0 = dg.tok0;
        du.ntok = dg.ntok;
        du.qpos0 = dg.qpos0;
        du.nsplit = dg.nsplit;
        du.pbase = dg.pbase;
        du.nparts = dg.nparts;
        du.pad1 = 0;
        return true;
    };
    // When every CTA of the grid starts at once (not after a tensor-core kernel, whose
    // CTAs release SMs one by one), this CTA's first piece -- unit b of the queue, or the
    // start of its share of the line -- and its first page ids (plan and page table,
    // complete before this grid) are requested now, before the set-up and the wait below;
    // the work counter serves the queue's units after the first gridDim.x.  After a
    // tensor-core kernel the first unit comes from the counter too, so the longest units
    // go to the CTAs that start first.
    const bool static_first = !wait_late || share > 0;  // (a balanced plan has no tensor-core unit)
    DecUnit du_first{};
    bool have_first = false;
    int g_first = -1;
    int32_t page_first_raw = 0;
    if (static_first && warp == HB) {
        if (share > 0) {
            int g = reinterpret_cast<const int32_t*>(p.ws + p.lay.dec_first)[blockIdx.x];
            if (g < n_groups) {
                have_first = piece(g, dgroups[g], du_first);
                // the share starts in the group's padding: the next group
                if (!have_first && ++g < n_groups) have_first = piece(g, dgroups[g], du_first);
            }
            g_first = g;
        } else if ((int)blockIdx.x < n_units) {
            du_first = units[blockIdx.x / n_hb];
            have_first = true;
        }
        const int key = du_first.k0 + (lane & 15);
        if (have_first && key < du_first.k1)
            page_first_raw = p.page_table[(int64_t)du_first.req * p.ld + (key >> p.page_shift)];
    }

    // zero the ring once so rows past a range's end are finite (they are masked,
    // and 0 * finite stays 0 in the P V product)
    for (int i = threadIdx.x * 16; i < stages * stage_bytes; i += blockDim.x * 16)
        *reinterpret_cast<int4*>(ring + i) = make_int4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            dev::mbar_init(&sh->full[s], 1);
            dev::mbar_init(&sh->empty[s], HB);
        }
        sh->abort_flag = 0;
        dev::fence_barrier_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (!wait_late) dev::grid_dep_wait();

    int32_t* sched = &hdr->pad[0];
    const int sched_base = static_first ? (int)gridDim.x : 0;  // units taken statically

    if (warp == HB) {
        // ================================================================ producer
        int stage = 0;
        uint32_t phase = 0;
        const uint64_t policy = dev::policy_evict_first();
        const int ps_mask = p.page_size - 1;
        uint32_t armed = 0, armed_par = 0;  // stages with copies issued, and the parity of that phase
        // Dynamic work fetch, one unit ahead but late: the ticket for the next unit is
        // taken four stages before the current unit ends, its record read two stages
        // before, its first page id one stage before.  A CTA so holds a unit in
        // reserve only briefly (a long reservation starves the tail of the grid), and
        // no global round trip sits between a freed ring slot and the copies that
        // refill it.  Page ids inside a unit are read one stage ahead.
        auto page_of = [&](const int32_t* prow, int key) -> int64_t {
            int64_t page = prow[key >> p.page_shift];
            if (page < 0 || page >= p.num_pages) {
                dev::set_error(err, kErrPage);
                page = 0;  // keep the transaction count; the result is flagged
            }
            return page;
        };
        const int r = lane & 15;
        int u;
        DecUnit du{};
        int64_t page_first = -1;  // page of the unit's first stage, when already fetched
        int g_cur = g_first;  // balanced split: the group of the current piece
        if (static_first) {
            u = have_first ? (share > 0 ? 0 : (int)blockIdx.x) : n_units;
            if (u < n_units) {
                du = du_first;
                if (du.k0 + r < du.k1) {
                    page_first = page_first_raw;
                    if (page_first < 0 || page_first >= p.num_pages) {
                        dev::set_error(err, kErrPage);
                        page_first = 0;  // keep the transaction count; the result is flagged
                    }
                }
            }
        } else {
            u = __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(sched, 1) : 0, 0);
            if (u < n_units) du = units[u / n_hb];
        }
        while (true) {
            if (!warp_wait(&sh->empty[stage], phase ^ 1, wlim, sh, err)) break;
            if (u >= n_units) {
                if (lane == 0) {
                    sh->info[stage].flags = kEnd;
                    dev::mbar_arrive(&sh->full[stage]);
                }
                armed &= ~(1u << stage);  // the end marker carries no copies (earlier ones were consumed)
                break;
            }
            const int hb = u % n_hb;
            const int32_t* prow = p.page_table + (int64_t)du.req * p.ld;
            // warm L2 with this unit's query rows (read by the consumers at unit start)
            {
                const char* qbase = reinterpret_cast<const char*>(p.q + (int64_t)du.tok0 * Hq * D);
                const int qbytes = du.ntok * Hq * D * 2;
                for (int off = lane * 128; off < qbytes; off += 32 * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(qbase + off));
            }
            int64_t page_next = page_first >= 0 ? page_first : ((du.k0 + r < du.k1) ? page_of(prow, du.k0 + r) : 0);
            page_first = -1;
            const int nst = (du.k1 - du.k0 + kStageKeys - 1) / kStageKeys;
            int ticket = 0, u_next = n_units, g_next = g_cur;
            DecUnit du_next{};
            for (int si_ = 0; si_ < nst; ++si_) {
                const int k = du.k0 + si_ * kStageKeys;
                if (share == 0 && si_ == max(nst - 4, 0) && lane == 0) ticket = sched_base + atomicAdd(sched, 1);
                if (si_ == max(nst - 2, 0)) {
                    if (share > 0) {  // the next group's piece of this CTA's share, if any
                        const int gn = g_cur + 1;
                        if (gn < n_groups && piece(gn, dgroups[gn], du_next)) {
                            u_next = 0;
                            g_next = gn;
                        }
                    } else {
                        u_next = __shfl_sync(0xffffffffu, ticket, 0);
                        if (u_next < n_units) du_next = units[u_next / n_hb];
                    }
                }
                const int64_t page = page_next;
                if (k + kStageKeys + r < du.k1) {
                    page_next = page_of(prow, k + kStageKeys + r);
                } else if (si_ == nst - 1 && u_next < n_units && du_next.k0 + r < du_next.k1) {
                    page_first = page_of(p.page_table + (int64_t)du_next.req * p.ld, du_next.k0 + r);
                }
                if (si_ != 0 && !warp_wait(&sh->empty[stage], phase ^ 1, wlim, sh, err)) goto producer_done;
                const int nk = min(kStageKeys, du.k1 - k);
                if (lane == 0) {
                    StageInfo& si = sh->info[stage];
                    si.unit = u;
                    si.group = du.group;
                    si.k = k;
                    si.k1 = du.k1;
                    si.tok0 = du.tok0;
                    si.ntok = du.ntok;
                    si.qpos0 = du.qpos0;
                    si.nsplit = du.nsplit;
                    si.pbase = du.pbase;
                    si.split = du.split;
                    si.hb = hb;
                    si.nparts = du.nparts;
                    si.flags = (si_ == 0 ? kFirst : 0) | (si_ == nst - 1 ? kLast : 0);
                    dev::mbar_arrive_expect_tx(&sh->full[stage], (uint32_t)(2 * nk * row_bytes));
                }
                armed |= 1u << stage;
                armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                __syncwarp();
                if (runs && (k & (kStageKeys - 1)) == 0) {
                    // the stage's rows are consecutive slots of one page (a 16-aligned run of
                    // keys inside a page of >= 16 slots): one copy for K, one for V
                    if (r == 0) {
                        const int64_t slot = (page << p.page_shift) + (k & ps_mask);
                        const uint8_t* src = reinterpret_cast<const uint8_t*>(lane < 16 ? p.k_pool : p.v_pool) +
                                             slot * (int64_t)(Hkv * D) * ES;
                        uint8_t* dst = ring + stage * stage_bytes + (lane < 16 ? 0 : kStageKeys * row_stride);
                        dev::bulk_g2s_hint(dst, src, (uint32_t)(nk * row_bytes), &sh->full[stage], policy);
                    }
                } else if (r < nk) {
                    const int64_t slot = (page << p.page_shift) + ((k + r) & ps_mask);
                    const uint8_t* src = reinterpret_cast<const uint8_t*>(lane < 16 ? p.k_pool : p.v_pool) +
                                         (slot * (int64_t)(Hkv * D) + hb * HB * D) * ES;
                    uint8_t* dst = ring + stage * stage_bytes + (lane < 16 ? 0 : kStageKeys * row_stride) +
                                   r * row_stride;
                    dev::bulk_g2s_hint(dst, src, (uint32_t)row_bytes, &sh->full[stage], policy);
                }
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            u = u_next;
            du = du_next;
            g_cur = g_next;
        }
    producer_done:
        // drain: every copy this warp issued must land before the CTA may exit -- also when
        // it ends normally, since a consumer may still give up on a stage in flight (a stage
        // the consumers already took has completed and returns at once)
        for (int s = 0; s < stages; ++s)
            if (armed & (1u << s)) (void)dev::mbar_wait(&sh->full[s], (armed_par >> s) & 1u);
        if (wait_late) dev::grid_dep_wait();
        return;
    }

    // ==================================================================== consumers
    const int gl = warp;           // kv head within the head block
    const int gq = lane >> 2;      // fragment row group
    const int cq = lane & 3;       // fragment column pair
    constexpr int KS = D / 16;     // k-steps over the head dim
    constexpr int NT = D / 8;      // n-tiles of the output
    uint32_t qa[KS][4];
    float o[NT][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int lim0 = 0, lim1 = 0;
    float ks = 1.f, vs = 1.f;  // per-head scales of an FP8 pool
    const int r0 = gq, r1 = gq + 8;
    int stage = 0;
    uint32_t phase = 0;

    while (true) {
        if (!warp_wait(&sh->full[stage], phase, wlim, sh, err)) return;
        const StageInfo si = sh->info[stage];
        if (si.flags & kEnd) break;
        const int rows = si.ntok * G;
        const int g = si.hb * HB + gl;  // kv head
        if (si.flags & kFirst) {
            // load this head's query rows as m16k16 A fragments (rows >= rows are zero)
            const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
            const int64_t qrow0 = r0 < rows ? ((int64_t)(si.tok0 + r0 / G) * Hq + g * G + r0 % G) * D : -1;
            const int64_t qrow1 = r1 < rows ? ((int64_t)(si.tok0 + r1 / G) * Hq + g * G + r1 % G) * D : -1;
            if constexpr (F8) {
                // k-step kk, fragment columns (2cq, 2cq+1 | 2cq+8, 2cq+9) <- head dims
                // cq*D/4 + 4kk + (0, 1 | 2, 3): the order the K fragments use below
                auto f16pair = [](uint32_t bf2) {
                    return dev::pack_f16x2(__uint_as_float(bf2 << 16), __uint_as_float(bf2 & 0xFFFF0000u));
                };
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const int c = cq * (D / 4) + 4 * kk;
                    qa[kk][0] = qrow0 >= 0 ? f16pair(q32[(qrow0 + c) >> 1]) : 0u;
                    qa[kk][1] = qrow1 >= 0 ? f16pair(q32[(qrow1 + c) >> 1]) : 0u;
                    qa[kk][2] = qrow0 >= 0 ? f16pair(q32[(qrow0 + c + 2) >> 1]) : 0u;
                    qa[kk][3] = qrow1 >= 0 ? f16pair(q32[(qrow1 + c + 2) >> 1]) : 0u;
                }
                ks = p.k_scale[g];
                vs = p.v_scale[g];
            } else {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const int c = kk * 16 + 2 * cq;
                    qa[kk][0] = qrow0 >= 0 ? q32[(qrow0 + c) >> 1] : 0u;
                    qa[kk][1] = qrow1 >= 0 ? q32[(qrow1 + c) >> 1] : 0u;
                    qa[kk][2] = qrow0 >= 0 ? q32[(qrow0 + c + 8) >> 1] : 0u;
                    qa[kk][3] = qrow1 >= 0 ? q32[(qrow1 + c + 8) >> 1] : 0u;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            // causal limit of each fragment row (rows past `rows` see nothing)
            lim0 = r0 < rows ? si.qpos0 + r0 / G : -1;
            lim1 = r1 < rows ? si.qpos0 + r1 / G : -1;
        }

        const uint8_t* Ks = ring + stage * stage_bytes + gl * D * ES;
        const uint8_t* Vs = Ks + kStageKeys * row_stride;
        const uint32_t ks_base = dev::smem_u32(Ks);
        const uint32_t vs_base = dev::smem_u32(Vs);

        // ---- S = Q K^T over the stage's 16 keys (two n8 tiles)
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        if constexpr (F8) {
            // key nt*8 + gq: the lane's D/4 bytes of the row, four per k-step
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const uint8_t* krow = Ks + (nt * 8 + gq) * row_stride + cq * (D / 4);
                uint32_t kw[KS];
#pragma unroll
                for (int i = 0; i < KS / 4; ++i) {
                    const int4 w = *reinterpret_cast<const int4*>(krow + 16 * i);
                    kw[4 * i] = (uint32_t)w.x;
                    kw[4 * i + 1] = (uint32_t)w.y;
                    kw[4 * i + 2] = (uint32_t)w.z;
                    kw[4 * i + 3] = (uint32_t)w.w;
                }
#pragma unroll
                for (int kk = 0; kk < KS; ++kk)
                    dev::mma_f16_16816(s[nt], qa[kk], dev::e4m3x2_to_f16x2(kw[kk]), dev::e4m3x2_to_f16x2(kw[kk] >> 16));
            }
        } else {
#pragma unroll
            for (int kk2 = 0; kk2 < KS / 2; ++kk2) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t addr =
                        ks_base + (nt * 8 + (lane & 7)) * row_stride + (kk2 * 32 + (lane >> 3) * 8) * 2;
                    uint32_t b0, b1, b2, b3;
                    dev::ldsm_x4(addr, b0, b1, b2, b3);
                    dev::mma_bf16_16816(s[nt], qa[2 * kk2], b0, b1);
                    dev::mma_bf16_16816(s[nt], qa[2 * kk2 + 1], b2, b3);
                }
            }
        }

        // ---- scale, mask (range end and causal diagonal), online softmax
        const float sl = p.scale_log2 * ks;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = si.k + nt * 8 + 2 * cq + (e & 1);
                const int lim = e < 2 ? lim0 : lim1;
                float x = s[nt][e] * sl;
                if (key >= si.k1 || key > lim) x = -INFINITY;
                s[nt][e] = x;
            }
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = dev::fast_exp2(m0 - mu0);  // m0 = -inf -> 0
        const float al1 = dev::fast_exp2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = dev::fast_exp2(s[nt][0] - mu0);
            s[nt][1] = dev::fast_exp2(s[nt][1] - mu0);
            s[nt][2] = dev::fast_exp2(s[nt][2] - mu1);
            s[nt][3] = dev::fast_exp2(s[nt][3] - mu1);
            ps0 += s[nt][0] + s[nt][1];
            ps1 += s[nt][2] + s[nt][3];
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            o[nt][0] *= al0;
            o[nt][1] *= al0;
            o[nt][2] *= al1;
            o[nt][3] *= al1;
        }
        uint32_t pa[4];
        if constexpr (F8) {
            pa[0] = dev::pack_f16x2(s[0][0], s[0][1]);
            pa[1] = dev::pack_f16x2(s[0][2], s[0][3]);
            pa[2] = dev::pack_f16x2(s[1][0], s[1][1]);
            pa[3] = dev::pack_f16x2(s[1][2], s[1][3]);
            // ---- O += P V: the lane's keys 2cq, 2cq+1 | 2cq+8, 2cq+9 (its k rows), its run of
            // D/8 output columns gq*D/8 .. (gq+1)*D/8 - 1; output tile nt, column n holds head
            // dim n*D/8 + nt.  A byte permute pairs the two keys of a column for the conversion.
            constexpr int VW = D / 32;  // words of a lane's run
            uint32_t vw[4][VW];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint8_t* vrow = Vs + (2 * cq + (i & 1) + (i >> 1) * 8) * row_stride + gq * (D / 8);
                if constexpr (VW == 4) {
                    const int4 w = *reinterpret_cast<const int4*>(vrow);
                    vw[i][0] = (uint32_t)w.x;
                    vw[i][1] = (uint32_t)w.y;
                    vw[i][2] = (uint32_t)w.z;
                    vw[i][3] = (uint32_t)w.w;
                } else {
                    const uint2 w = *reinterpret_cast<const uint2*>(vrow);
                    vw[i][0] = w.x;
                    vw[i][1] = w.y;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt += 2) {
                const int wi = nt >> 2, j = nt & 3;  // word and byte of columns nt, nt + 1
                const uint32_t sel = (uint32_t)(j | ((4 + j) << 4) | ((j + 1) << 8) | ((5 + j) << 12));
                const uint32_t x01 = dev::prmt(vw[0][wi], vw[1][wi], sel);  // k rows 2cq, 2cq+1
                const uint32_t x89 = dev::prmt(vw[2][wi], vw[3][wi], sel);  // k rows 2cq+8, 2cq+9
                dev::mma_f16_16816(o[nt], pa, dev::e4m3x2_to_f16x2(x01), dev::e4m3x2_to_f16x2(x89));
                dev::mma_f16_16816(o[nt + 1], pa, dev::e4m3x2_to_f16x2(x01 >> 16), dev::e4m3x2_to_f16x2(x89 >> 16));
            }
        } else {
            pa[0] = dev::pack_bf16x2(s[0][0], s[0][1]);
            pa[1] = dev::pack_bf16x2(s[0][2], s[0][3]);
            pa[2] = dev::pack_bf16x2(s[1][0], s[1][1]);
            pa[3] = dev::pack_bf16x2(s[1][2], s[1][3]);
            // ---- O += P V (V rows are the k dimension: transposed fragment loads)
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
                const uint32_t addr =
                    vs_base + ((lane & 7) + ((lane >> 3) & 1) * 8) * row_stride + (dt * 16 + (lane >> 4) * 8) * 2;
                uint32_t v0, v1, v2, v3;
                dev::ldsm_x4_t(addr, v0, v1, v2, v3);
                dev::mma_bf16_16816(o[2 * dt], pa, v0, v1);
                dev::mma_bf16_16816(o[2 * dt + 1], pa, v2, v3);
            }
        }

        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&sh->empty[stage]);
        if (++stage == stages) {
            stage = 0;
            phase ^= 1;
        }
        if (!(si.flags & kLast)) continue;

        // ================================================================ unit epilogue
        float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
        float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
        const float inv0 = lt0 > 0.f ? vs / lt0 : 0.f;
        const float inv1 = lt1 > 0.f ? vs / lt1 : 0.f;
        const float lse0 = lt0 > 0.f ? m0 + __log2f(lt0) : -INFINITY;  // log2 domain
        const float lse1 = lt1 > 0.f ? m1 + __log2f(lt1) : -INFINITY;

        if (si.nparts == 1) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = half ? r1 : r0;
                if (r >= rows) continue;
                const int64_t orow = (int64_t)(si.tok0 + r / G) * Hq + g * G + r % G;
                uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + orow * D);
                const float inv = half ? inv1 : inv0;
                if constexpr (F8) {
                    // columns (2cq + e) * D/8 + nt of o[nt][2 half + e]: two runs of D/8
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        uint32_t w[NT / 2];
#pragma unroll
                        for (int nt = 0; nt < NT; nt += 2)
                            w[nt / 2] = dev::pack_bf16x2(o[nt][2 * half + e] * inv, o[nt + 1][2 * half + e] * inv);
                        uint4* d4 = reinterpret_cast<uint4*>(dst + (2 * cq + e) * (D / 16));
#pragma unroll
                        for (int i = 0; i < NT / 8; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        dst[(nt * 8 + 2 * cq) >> 1] =
                            dev::pack_bf16x2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
                }
                if (p.lse != nullptr && cq == 0) p.lse[orow] = (half ? lse1 : lse0) * kLn2;
            }
            continue;
        }

        // split group: fp32 partial (normalised O, log2-domain LSE) into its slot; the
        // merge kernel that follows combines the group's slots.  Plain stores: nothing
        // in this kernel reads them back, so the consumers move on to the next unit.
        const int slot = si.pbase + si.split;
        float* po = reinterpret_cast<float*>(p.ws + p.lay.partial_o) + (int64_t)slot * p.lay.rows_per_slot * D;
        float* pl = reinterpret_cast<float*>(p.ws + p.lay.partial_lse) + (int64_t)slot * p.lay.rows_per_slot;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = half ? r1 : r0;
            if (r >= rows) continue;
            const int prow = (r / G) * Hq + g * G + r % G;  // (token, q head) within the group
            const float inv = half ? inv1 : inv0;
            if constexpr (F8) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float4* d4 = reinterpret_cast<float4*>(po + (int64_t)prow * D + (2 * cq + e) * (D / 8));
#pragma unroll
                    for (int i = 0; i < NT / 4; ++i)
                        d4[i] = make_float4(o[4 * i][2 * half + e] * inv, o[4 * i + 1][2 * half + e] * inv,
                                            o[4 * i + 2][2 * half + e] * inv, o[4 * i + 3][2 * half + e] * inv);
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    *reinterpret_cast<float2*>(po + (int64_t)prow * D + nt * 8 + 2 * cq) =
                        make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
            }
            if (cq == 0) pl[prow] = half ? lse1 : lse0;
        }
    }
}

// K4: log-sum-exp combine of the split groups (and of the prefix-pass partials of
// shared-prefix members): for every row (token, q head) of a group with nparts > 1,
// lse = log2 sum_s 2^lse_s, o = sum_s 2^(lse_s - lse) o_s over the group's slots
// pbase .. pbase + nparts - 1, in slot order (deterministic).  One warp per row: lane s
// holds part s's LSE, so the maximum and the normaliser are two warp reductions, and
// lane c accumulates columns [c * D/32, (c+1) * D/32) of every part with independent
// loads (the partials are L2-resident: written by the kernels just before).  A work
// item is one group's rows [32c, 32c + 32) (c < rows_per_slot / 32), one row per warp,
// items numbered chunk-major (chunk 0 of every group first, so single-token groups,
// whose rows are all in chunk 0, each go to their own CTA), so the rows of a group
// with several tokens spread over several SMs (a CTA per group
// left each warp four rows in sequence in a speculative-verify batch: merge 23.6 ->
// 14 us there).  Smaller CTAs with fewer rows each cost more in launch and record
// reads than they saved (merge of the cascade batch 10.2 -> 16.4 us at 8 warps).
// Launched programmatically after the decode kernel, whose grid it waits for.
constexpr int kMergeThreads = 1024;
constexpr int kHoist = 2;  // parts whose columns each lane loads before the LSE reductions

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(ForwardParams p) {
    constexpr int kPer = D / 32;  // output columns per lane
    constexpr int kWarps = kMergeThreads / 32;
    dev::grid_dep_launch();
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.lay.header);
    const int n_groups = hdr->n_dec_groups;
    if ((hdr->error_bits & kErrFatal) || n_groups == 0 || hdr->n_partial_slots == 0) {
        dev::grid_dep_wait();
        return;
    }
    const DecGroup* groups = reinterpret_cast<const DecGroup*>(p.ws + p.lay.dec_groups);
    const float* plse = reinterpret_cast<const float*>(p.ws + p.lay.partial_lse);
    const float* pout = reinterpret_cast<const float*>(p.ws + p.lay.partial_o);
    const int rps = p.lay.rows_per_slot, Hq = p.num_qo_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // row chunks of a group: its rows are at most max_group_tokens * Hq (<= rps)
    const int chunks = (min(rps, max(hdr->max_group_tokens, 1) * Hq) + kWarps - 1) / kWarps;
    const int n_items = n_groups * chunks;
    // the group records come from the plan (complete before the forward began): the first
    // one is read before the wait for the decode grid, only the partials after it
    DecGroup dg_next{};
    if ((int)blockIdx.x < n_items) dg_next = groups[blockIdx.x % n_groups];
    dev::grid_dep_wait();
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const DecGroup dg = dg_next;
        if (it + (int)gridDim.x < n_items) dg_next = groups[(it + gridDim.x) % n_groups];
        const int np = dg.nparts;
        if (np <= 1) continue;
        const int rows = dg.ntok * Hq;
        const float* plb = plse + (int64_t)dg.pbase * rps;
        const float* pob = pout + (int64_t)dg.pbase * rps * D;
        {
            const int row = (it / n_groups) * kWarps + warp;
            if (row >= rows) continue;
            // the first kHoist parts' columns are requested together with the LSEs, so that
            // the usual split counts take one round trip to L2, not two
            float hv[kHoist][kPer];
#pragma unroll
            for (int k = 0; k < kHoist; ++k) {
                const float* sp = pob + ((int64_t)k * rps + row) * D + lane * kPer;
                if constexpr (kPer == 4) {
                    const float4 v = k < np ? __ldcg(reinterpret_cast<const float4*>(sp)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    hv[k][0] = v.x, hv[k][1] = v.y, hv[k][2] = v.z, hv[k][3] = v.w;
                } else {
                    const float2 v = k < np ? __ldcg(reinterpret_cast<const float2*>(sp)) : make_float2(0.f, 0.f);
                    hv[k][0] = v.x, hv[k][1] = v.y;
                }
            }
            const float lfirst = lane < np ? __ldcg(plb + (int64_t)lane * rps + row) : -INFINITY;
            float mx = lfirst;
            for (int s0 = 32; s0 < np; s0 += 32)
                if (s0 + lane < np) mx = fmaxf(mx, __ldcg(plb + (int64_t)(s0 + lane) * rps + row));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mu = mx == -INFINITY ? 0.f : mx;
            float acc[kPer];
#pragma unroll
            for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
            float wsum = 0.f;
            for (int s0 = 0; s0 < np; s0 += 32) {
                const float l = s0 == 0 ? lfirst : (s0 + lane < np ? __ldcg(plb + (int64_t)(s0 + lane) * rps + row)
                                                                    : -INFINITY);
                const float w = dev::fast_exp2(l - mu);  // 0 for an empty part (lse -inf)
                wsum += w;
                const int cnt = min(32, np - s0);
                const float* src = pob + ((int64_t)s0 * rps + row) * D + lane * kPer;
                int k = 0;
                if (s0 == 0) {
#pragma unroll
                    for (int h = 0; h < kHoist; ++h) {
                        const float wk = __shfl_sync(0xffffffffu, w, h);
                        if (h < cnt) {
#pragma unroll
                            for (int c = 0; c < kPer; ++c) acc[c] += wk * hv[h][c];
                        }
                    }
                    k = kHoist;
                }
#pragma unroll 4
                for (; k < cnt; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, w, k);
                    const float* sp = src + (int64_t)k * rps * D;
                    if constexpr (kPer == 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(sp));
                        acc[0] += wk * v.x;
                        acc[1] += wk * v.y;
                        acc[2] += wk * v.z;
                        acc[3] += wk * v.w;
                    } else {
                        const float2 v = __ldcg(reinterpret_cast<const float2*>(sp));
                        acc[0] += wk * v.x;
                        acc[1] += wk * v.y;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
            const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
            const int64_t orow = (int64_t)(dg.tok0 + row / Hq) * Hq + row % Hq;
            uint16_t* dst = p.out + orow * D + lane * kPer;
            if constexpr (kPer == 4) {
                uint2 packed;
                packed.x = dev::pack_bf16x2(acc[0] * inv, acc[1] * inv);
                packed.y = dev::pack_bf16x2(acc[2] * inv, acc[3] * inv);
                *reinterpret_cast<uint2*>(dst) = packed;
            } else {
                *reinterpret_cast<uint32_t*>(dst) = dev::pack_bf16x2(acc[0] * inv, acc[1] * inv);
            }
            if (p.lse != nullptr && lane == 0) p.lse[orow] = wsum > 0.f ? (mu + __log2f(wsum)) * kLn2 : -INFINITY;
        }
    }
}

template <int D>
int stage_count(int num_kv_heads, int ctas_per_sm, int es, int pad) {
    const int hb = num_kv_heads < kMaxKvHeads ? num_kv_heads : kMaxKvHeads;
    const int row_stride = hb * D * es + pad;
    const int stage_bytes = 2 * kStageKeys * row_stride;
    const int budget = 220 * 1024 / ctas_per_sm - 1024;
    int st = budget / stage_bytes;
    return st < 2 ? 2 : (st > 8 ? 8 : st);
}

template <int D>
size_t smem_bytes(int num_kv_heads, int stages, int es, int pad) {
    const int hb = num_kv_heads < kMaxKvHeads ? num_kv_heads : kMaxKvHeads;
    const int row_stride = hb * D * es + pad;
    return ((sizeof(DecSmemHead) + 127) / 128) * 128 + (size_t)stages * 2 * kStageKeys * row_stride;
}

// FP8 rows are half as long as bf16 ones, and one bulk copy per 1 KiB row left the copy
// engine, not HBM, the limit (ncu: DRAM at a third of its peak, consumers waiting on the
// stages).  So with pages of at least a stage (16 slots) and every kv head in the CTA, a
// stage's rows -- consecutive slots of one page, contiguous in the pool -- come as one
// copy per pool and sit back to back.  The K fragment reads then meet 2-way shared-memory
// bank conflicts (a lane's run sits at the same bank offset in every row); the padded
// per-row layout stays for the other cases and for bf16, whose ldmatrix reads need it.
template <int D, bool F8>
cudaError_t launch_d(const ForwardParams& p, int ctas, cudaStream_t s) {
    constexpr int es = F8 ? 1 : 2;
    const int cps = decode_ctas_per_sm(p.num_kv_heads, D);
    const bool runs = F8 && p.page_size >= kStageKeys && p.num_kv_heads <= kMaxKvHeads;
    const int stages = stage_count<D>(p.num_kv_heads, cps, es, runs ? 0 : kRowPad);
    const size_t smem = smem_bytes<D>(p.num_kv_heads, stages, es, runs ? 0 : kRowPad);
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int hb = p.num_kv_heads < kMaxKvHeads ? p.num_kv_heads : kMaxKvHeads;
    const int row_stride = hb * D * es + (runs ? 0 : kRowPad);
    return launch_programmatic(decode_kernel<D, F8>, (unsigned)ctas, 32u * (hb + 1), smem, s, p, stages,
                               row_stride);
}

template <int D>
cudaError_t launch_m(const ForwardParams& p, int ctas, cudaStream_t s) {
    return launch_programmatic(merge_kernel<D>, (unsigned)ctas, (unsigned)kMergeThreads, 0, s, p);
}

}  // namespace

int decode_ctas_per_sm(int num_kv_heads, int head_dim) {
    (void)head_dim;
    const int hb = num_kv_heads < kMaxKvHeads ? num_kv_heads : kMaxKvHeads;
    int c = 8 / (hb > 0 ? hb : 1);
    return c < 1 ? 1 : (c > 4 ? 4 : c);
}

bool decode_supported(int num_qo_heads, int num_kv_heads, int head_dim) {
    if (num_kv_heads < 1) return false;
    if (num_kv_heads > kMaxKvHeads && num_kv_heads % kMaxKvHeads != 0) return false;
    if (num_qo_heads % num_kv_heads != 0) return false;
    if (num_qo_heads / num_kv_heads > kDecRows) return false;
    return head_dim == 64 || head_dim == 128;
}

cudaError_t launch_decode(const ForwardParams& p, int head_dim, int ctas, cudaStream_t s) {
    if (head_dim == 128) return p.kv_fp8 ? launch_d<128, true>(p, ctas, s) : launch_d<128, false>(p, ctas, s);
    if (head_dim == 64) return p.kv_fp8 ? launch_d<64, true>(p, ctas, s) : launch_d<64, false>(p, ctas, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge(const ForwardParams& p, int head_dim, int ctas, cudaStream_t s) {
    if (head_dim == 128) return launch_m<128>(p, ctas, s);
    if (head_dim == 64) return launch_m<64>(p, ctas, s);
    return cudaErrorInvalidValue;
}

}  // namespace pva
