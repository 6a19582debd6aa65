// K2: prefill / chunked-prefill attention on the 5th-generation tensor cores.
//
// What it computes is the reference forward of "The attention backend and a
// reference implementation" (section "Variable-length, paged attention with
// prefixes") for requests with many new tokens: S = scale * Q K^T over the
// request's keys gathered through the page table, the bottom-right causal mask
// (query r of n sees keys j <= kv_len - n + r), softmax, O = P V.  It is the
// dense contraction of the path, so it runs as tcgen05 MMAs:
//
//   * a tile is 128 rows = floor(128/G) consecutive new tokens x the G q heads
//     of one kv head (GQA packing: every K/V tile loaded serves all G heads);
//     keys run in 128-key tiles up to the tile's causal end (later keys are
//     never loaded: causal tile skipping), only tiles crossing the diagonal
//     get an elementwise mask;
//   * warp 0 (producer) loads Q once per tile and K/V tiles through TMA from
//     the paged pool: one 3-D box per page (rows of one kv head, 128-byte
//     swizzle) and single-row boxes for the valid rows of a partial last page,
//     so no slot past kv_len is read; two K and two V stages;
//   * warp 1 issues the MMAs from one thread: S_j = Q K_j^T into one of two
//     TMEM buffers (fp32, 128 lanes x 128 columns), then O += P_{j-1} V_{j-1}
//     into a TMEM accumulator, so the next S overlaps the current softmax;
//   * warps 2-5 (one TMEM lane = one row per thread) run the online softmax:
//     tcgen05.ld of S, mask, running max, exp2, P as bf16 into shared memory
//     (the A operand of the P V product); O in TMEM is rescaled only when a
//     row's max grows by more than 2^8, and normalised once at the end.
// Every wait is bounded; a timeout sets PVA_DEVERR_TIMEOUT and the CTA winds
// down (outstanding copies and MMAs waited for, TMEM freed) without trapping.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "device_utils.cuh"
#include "pva_internal.h"
#include "tc_utils.cuh"

namespace pva {
namespace {

constexpr int kThreads = 192;
constexpr int kRegion = 128 * 128;  // one 128-row x 128-byte swizzled region (64 bf16 columns)
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Layout2 {
    static constexpr int kHalves = D / 64;
    static constexpr int kTile = kRegion * kHalves;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTile;
    static constexpr int kV = kK + 2 * kTile;
    static constexpr int kP = kV + 2 * kTile;
    static constexpr int kBytes = kP + 2 * kRegion;
};

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2];
    uint64_t p_full, pv_done, o_free, drain;
    uint32_t tmem_base;
    int32_t abort_flag;
};

__device__ __forceinline__ uint32_t sw128(int row, int col16) {  // byte offset of 16-byte chunk col16 of a row
    return row * 128 + (((col16 ^ (row & 7)) & 7) << 4);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* b, uint32_t* err) {
    if (dev::mbar_wait(bar, parity)) return true;
    b->abort_flag = 1;
    dev::set_error(err, kErrTimeout);
    return false;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const ForwardParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k_page, const __grid_constant__ CUtensorMap tm_v_page,
                   const __grid_constant__ CUtensorMap tm_k_row, const __grid_constant__ CUtensorMap tm_v_row,
                   int rows_page) {
    using L = Layout2<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Bars bars;
    Bars* b = &bars;
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.lay.header);
    uint32_t* err = &hdr->error_bits;
    const int n_tiles = hdr->n_pre_tiles;
    if ((hdr->error_bits & kErrFatal) || n_tiles == 0 || (int)blockIdx.x >= n_tiles) return;
    const PreTile* tiles = reinterpret_cast<const PreTile*>(p.ws + p.lay.pre_tiles);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group, Hq = p.num_qo_heads;
    const int TM = kPreRows / G;

    for (int i = threadIdx.x * 16; i < L::kBytes; i += kThreads * 16)
        *reinterpret_cast<int4*>(smem + i) = make_int4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        dev::mbar_init(&b->q_full, 1);
        dev::mbar_init(&b->q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            dev::mbar_init(&b->k_full[s], 1);
            dev::mbar_init(&b->k_empty[s], 1);
            dev::mbar_init(&b->v_full[s], 1);
            dev::mbar_init(&b->v_empty[s], 1);
            dev::mbar_init(&b->s_full[s], 1);
        }
        dev::mbar_init(&b->p_full, 4);
        dev::mbar_init(&b->pv_done, 1);
        dev::mbar_init(&b->o_free, 4);
        dev::mbar_init(&b->drain, 1);
        b->abort_flag = 0;
        dev::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&b->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = b->tmem_base;
    const uint32_t t_s[2] = {tmem, tmem + 128};
    const uint32_t t_o = tmem + 256;

    if (warp == 0) {
        // ============================================================== producer (TMA)
        if (lane == 0) {
            tc::prefetch_tmap(&tm_q);
            tc::prefetch_tmap(&tm_k_page);
            tc::prefetch_tmap(&tm_v_page);
        }
        const uint64_t pol_kv = dev::policy_evict_last();  // K/V tiles are re-read by the request's other tiles
        uint32_t it = 0;
        int uc = 0;
        // barriers this warp armed with copies, and the parity of the phase each last armed
        uint32_t armed = 0, armed_par = 0;  // bit 0: q, bits 1-2: k stages, bits 3-4: v stages
        auto arm = [&](int bit, uint32_t par) {
            armed |= 1u << bit;
            armed_par = (armed_par & ~(1u << bit)) | (par << bit);
        };
        const int ps = p.page_size, ps_mask = p.page_size - 1;
        for (int u = blockIdx.x; u < n_tiles && !b->abort_flag; u += gridDim.x, ++uc) {
            const PreTile pt = tiles[u];
            const int32_t* prow = p.page_table + (int64_t)pt.req * p.ld;
            if (uc > 0 && !wait_or_abort(&b->q_empty, (uc - 1) & 1, b, err)) break;
            if (lane == 0) {
                dev::mbar_arrive_expect_tx(&b->q_full, (uint32_t)(L::kHalves * 128 * G * TM));
                for (int h = 0; h < L::kHalves; ++h)
                    tc::tma_load_3d(smem + L::kQ + h * kRegion, &tm_q, h * 64, pt.kvh * G, pt.tok0, &b->q_full);
            }
            arm(0, uc & 1);
            const int nkt = (pt.kv_end + kPreKeys - 1) / kPreKeys;
            for (int j = 0; j < nkt; ++j, ++it) {
                const int st = it & 1;
                const uint32_t ph = (it >> 1) & 1;
                const int key0 = j * kPreKeys;
                const int nkeys = min(kPreKeys, pt.kv_end - key0);
                const int nfull = nkeys / rows_page;              // whole boxes of rows_page rows
                const int npart = nkeys - nfull * rows_page;     // valid rows of a partial last page
                // slots of this lane's boxes/rows (ops lane, lane+32, ...; at most 128 ops)
                int64_t slot[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int op = lane + 32 * i;
                    slot[i] = -1;
                    int key = -1;
                    if (op < nfull) key = key0 + op * rows_page;
                    else if (op < nfull + npart) key = key0 + nfull * rows_page + (op - nfull);
                    if (key >= 0) {
                        int64_t page = prow[key / ps];
                        if (page < 0 || page >= p.num_pages) {
                            dev::set_error(err, kErrPage);
                            page = 0;
                        }
                        slot[i] = page * ps + (key & ps_mask);
                    }
                }
                const uint32_t bytes = (uint32_t)(nkeys * 128 * L::kHalves);
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    uint64_t* full = kv ? &b->v_full[st] : &b->k_full[st];
                    uint64_t* empty = kv ? &b->v_empty[st] : &b->k_empty[st];
                    const CUtensorMap* tm_page = kv ? &tm_v_page : &tm_k_page;
                    const CUtensorMap* tm_row = kv ? &tm_v_row : &tm_k_row;
                    uint8_t* base = smem + (kv ? L::kV : L::kK) + st * L::kTile;
                    if (!wait_or_abort(empty, ph ^ 1, b, err)) goto producer_out;
                    if (lane == 0) dev::mbar_arrive_expect_tx(full, bytes);
                    __syncwarp();
                    arm(kv ? 3 + st : 1 + st, ph);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int op = lane + 32 * i;
                        if (slot[i] < 0) continue;
                        const bool whole = op < nfull;
                        const int row = whole ? op * rows_page : nfull * rows_page + (op - nfull);
                        for (int h = 0; h < L::kHalves; ++h)
                            tc::tma_load_3d_hint(base + h * kRegion + row * 128, whole ? tm_page : tm_row, h * 64,
                                                 pt.kvh, (int)slot[i], full, pol_kv);
                    }
                }
            }
        }
    producer_out:
        // copies still in flight must land before the CTA may leave
        if (b->abort_flag) {
            uint64_t* bars_armed[5] = {&b->q_full, &b->k_full[0], &b->k_full[1], &b->v_full[0], &b->v_full[1]};
            for (int i = 0; i < 5; ++i)
                if (armed & (1u << i)) (void)dev::mbar_wait(bars_armed[i], (armed_par >> i) & 1u);
        }
    } else if (warp == 1) {
        // ============================================================== MMA issuer (one thread)
        const uint32_t id_qk = tc::idesc_bf16_f32(128, 128, 0, 0);
        const uint32_t id_pv = tc::idesc_bf16_f32(128, D, 0, 1);
        const uint32_t sq = dev::smem_u32(smem + L::kQ);
        const uint32_t sp = dev::smem_u32(smem + L::kP);
        uint32_t it = 0;
        int uc = 0;
        bool ok = true;
        auto pv = [&](uint32_t t, bool first_of_unit, int ucount) -> bool {
            if (!wait_or_abort(&b->p_full, t & 1, b, err)) return false;
            if (!wait_or_abort(&b->v_full[t & 1], (t >> 1) & 1, b, err)) return false;
            if (first_of_unit && ucount > 0 && !wait_or_abort(&b->o_free, (ucount - 1) & 1, b, err)) return false;
            tc::fence_after_sync();
            const uint32_t sv = dev::smem_u32(smem + L::kV + (t & 1) * L::kTile);
#pragma unroll
            for (int kk = 0; kk < kPreKeys / 16; ++kk) {
                const uint64_t ad = tc::smem_desc(sp + (kk >> 2) * kRegion + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B);
                const uint64_t bd = tc::smem_desc(sv + kk * 2048, kRegion, 1024, tc::kSwizzle128B);
                tc::mma_ss(t_o, ad, bd, id_pv, (first_of_unit && kk == 0) ? 0u : 1u);
            }
            tc::mma_commit(&b->pv_done);
            tc::mma_commit(&b->v_empty[t & 1]);
            return true;
        };
        if (lane == 0) {
            for (int u = blockIdx.x; u < n_tiles && ok; u += gridDim.x, ++uc) {
                const PreTile pt = tiles[u];
                const int nkt = (pt.kv_end + kPreKeys - 1) / kPreKeys;
                if (!wait_or_abort(&b->q_full, uc & 1, b, err)) {
                    ok = false;
                    break;
                }
                for (int j = 0; j < nkt && ok; ++j) {
                    const uint32_t t = it + j;
                    const int st = t & 1;
                    if (!wait_or_abort(&b->k_full[st], (t >> 1) & 1, b, err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t sk = dev::smem_u32(smem + L::kK + st * L::kTile);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t ad =
                            tc::smem_desc(sq + (kk >> 2) * kRegion + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B);
                        const uint64_t bd =
                            tc::smem_desc(sk + (kk >> 2) * kRegion + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B);
                        tc::mma_ss(t_s[st], ad, bd, id_qk, kk > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&b->s_full[st]);
                    tc::mma_commit(&b->k_empty[st]);
                    if (j == nkt - 1) tc::mma_commit(&b->q_empty);
                    if (j > 0) ok = pv(t - 1, j - 1 == 0, uc);
                }
                if (ok) ok = pv(it + nkt - 1, nkt == 1, uc);
                it += nkt;
            }
            // every MMA issued must complete before TMEM is released
            tc::mma_commit(&b->drain);
            (void)dev::mbar_wait(&b->drain, 0);
        }
        __syncwarp();
    } else {
        // ============================================================== softmax (one row per thread)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float sl = p.scale_log2;
        uint32_t it = 0;
        int uc = 0;
        for (int u = blockIdx.x; u < n_tiles && !b->abort_flag; u += gridDim.x, ++uc) {
            const PreTile pt = tiles[u];
            const int nkt = (pt.kv_end + kPreKeys - 1) / kPreKeys;
            const bool valid = row < pt.ntok * G;
            const int limit = valid ? pt.qpos0 + row / G : -1;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < nkt; ++j) {
                const uint32_t t = it + j;
                const int st = t & 1;
                if (!wait_or_abort(&b->s_full[st], (t >> 1) & 1, b, err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                float s[kPreKeys];
#pragma unroll
                for (int c = 0; c < kPreKeys / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(t_s[st] + lane_base + c * 32, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = v[i];
                }
                const int key0 = j * kPreKeys;
                const bool need_mask = key0 + kPreKeys - 1 > pt.qpos0;
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < kPreKeys; ++c) {
                    float x = s[c] * sl;
                    if (need_mask && key0 + c > limit) x = -INFINITY;
                    s[c] = x;
                    mx = fmaxf(mx, x);
                }
                const float m_new = fmaxf(m, mx);
                bool waited = false;
                if (j == 0) {
                    m = m_new;
                } else {
                    const bool resc = m_new > m + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, resc)) {
                        if (!wait_or_abort(&b->pv_done, (t - 1) & 1, b, err)) {
                            ok = false;
                            break;
                        }
                        waited = true;
                        tc::fence_after_sync();
                        const float alpha = resc ? dev::fast_exp2(m - m_new) : 1.f;
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            float v[32];
                            tc::tmem_ld32(t_o + lane_base + c * 32, v);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] *= alpha;
                            tc::tmem_st32(t_o + lane_base + c * 32, v);
                        }
                        tc::tmem_wait_st();
                        if (resc) {
                            l *= alpha;
                            m = m_new;
                        }
                    }
                }
                const float mu = m == -INFINITY ? 0.f : m;
                float ls = 0.f;
#pragma unroll
                for (int c = 0; c < kPreKeys; ++c) {
                    s[c] = dev::fast_exp2(s[c] - mu);
                    ls += s[c];
                }
                l += ls;
                if (j > 0 && !waited) {
                    if (!wait_or_abort(&b->pv_done, (t - 1) & 1, b, err)) {
                        ok = false;
                        break;
                    }
                }
                // P row -> shared memory, bf16, 128-byte swizzle (A operand of P V, K-major)
                uint8_t* prow_s = smem + L::kP;
#pragma unroll
                for (int c16 = 0; c16 < kPreKeys / 8; ++c16) {
                    uint4 w;
                    w.x = dev::pack_bf16x2(s[c16 * 8 + 0], s[c16 * 8 + 1]);
                    w.y = dev::pack_bf16x2(s[c16 * 8 + 2], s[c16 * 8 + 3]);
                    w.z = dev::pack_bf16x2(s[c16 * 8 + 4], s[c16 * 8 + 5]);
                    w.w = dev::pack_bf16x2(s[c16 * 8 + 6], s[c16 * 8 + 7]);
                    *reinterpret_cast<uint4*>(prow_s + (c16 >> 3) * kRegion + sw128(row, c16 & 7)) = w;
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&b->p_full);
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16 rows of out, LSE
            const uint32_t t_last = it + nkt - 1;
            if (!wait_or_abort(&b->pv_done, t_last & 1, b, err)) break;
            tc::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t orow = valid ? ((int64_t)(pt.tok0 + row / G) * Hq + pt.kvh * G + row % G) : 0;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                tc::tmem_ld32(t_o + lane_base + c * 32, v);
                tc::tmem_wait_ld();
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D + c * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = dev::pack_bf16x2(v[q4 * 8 + 0] * inv, v[q4 * 8 + 1] * inv);
                        w.y = dev::pack_bf16x2(v[q4 * 8 + 2] * inv, v[q4 * 8 + 3] * inv);
                        w.z = dev::pack_bf16x2(v[q4 * 8 + 4] * inv, v[q4 * 8 + 5] * inv);
                        w.w = dev::pack_bf16x2(v[q4 * 8 + 6] * inv, v[q4 * 8 + 7] * inv);
                        dst[q4] = w;
                    }
                }
            }
            if (valid && p.lse != nullptr) p.lse[orow] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&b->o_free);
            it += nkt;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side: tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// 3-D bf16 map over [outer][mid][D] with a box of {64, box_mid, box_outer} and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t D, uint64_t mid, uint64_t outer, uint32_t box_mid,
              uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {D, mid, outer};
    cuuint64_t strides[2] = {D * 2, mid * D * 2};
    cuuint32_t box[3] = {64, box_mid, box_outer};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_p(const ForwardParams& p, int ctas, cudaStream_t s) {
    const int G = p.group;
    const int TM = kPreRows / G;
    const int rows_page = p.page_size < kPreKeys ? p.page_size : kPreKeys;
    CUtensorMap tq, tkp, tvp, tkr, tvr;
    if (!make_map(&tq, p.q, D, p.num_qo_heads, (uint64_t)p.total_tokens, (uint32_t)G, (uint32_t)TM) ||
        !make_map(&tkp, p.k_pool, D, p.num_kv_heads, (uint64_t)p.num_slots, 1, (uint32_t)rows_page) ||
        !make_map(&tvp, p.v_pool, D, p.num_kv_heads, (uint64_t)p.num_slots, 1, (uint32_t)rows_page) ||
        !make_map(&tkr, p.k_pool, D, p.num_kv_heads, (uint64_t)p.num_slots, 1, 1) ||
        !make_map(&tvr, p.v_pool, D, p.num_kv_heads, (uint64_t)p.num_slots, 1, 1))
        return cudaErrorInvalidValue;
    const size_t smem = Layout2<D>::kBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<D><<<ctas, kThreads, smem, s>>>(p, tq, tkp, tvp, tkr, tvr, rows_page);
    return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int num_qo_heads, int num_kv_heads, int head_dim) {
    if (head_dim != 64 && head_dim != 128) return false;
    const int G = num_qo_heads / num_kv_heads;
    return G >= 1 && G <= 16 && encode_fn() != nullptr;
}

cudaError_t launch_prefill(const ForwardParams& p, int head_dim, int ctas, cudaStream_t s) {
    if (ctas <= 0) return cudaSuccess;
    if (head_dim == 128) return launch_p<128>(p, ctas, s);
    if (head_dim == 64) return launch_p<64>(p, ctas, s);
    return cudaErrorInvalidValue;
}

}  // namespace pva
