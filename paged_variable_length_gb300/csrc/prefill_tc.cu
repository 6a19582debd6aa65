// K2: prefill / chunked-prefill attention on the 5th-generation tensor cores.
//
// What it computes is the reference forward of "The attention backend and a
// reference implementation" (section "Variable-length, paged attention with
// prefixes") for requests with many new tokens: S = scale * Q K^T over the
// request's keys gathered through the page table, the bottom-right causal mask
// (query r of n sees keys j <= kv_len - n + r), softmax, O = P V.  It is the
// dense contraction of the path, so it runs as tcgen05 MMAs:
//
//   * a Q tile is 128 rows = floor(128/G) consecutive new tokens x the G q
//     heads of one kv head (GQA packing: every K/V tile loaded serves all G
//     heads); a CTA work unit holds two consecutive Q tiles of one request and
//     kv head, which share every K/V tile;
//   * keys run in 128-key tiles up to each Q tile's causal end (later keys
//     are never loaded or multiplied: causal tile skipping); only tiles that
//     cross the diagonal get an elementwise mask;
//   * warps 9-11 (producers) gather Q and K/V tiles row by row from the paged
//     pool with 16-byte async copies into the 128-byte-swizzled layout of the
//     MMA operands (rows past kv_len are not read); two K and two V stages;
//   * warp 8 issues the MMAs (one elected lane of the converged warp), in the order
//     PV0(j), S0(j+1), PV1(j), S1(j+1): while one softmax warpgroup works on
//     its S tile the tensor core runs the other tile's products;
//   * warps 0-3 / 4-7 are the softmax warpgroups of Q tile 0 / 1, one row per
//     thread (TMEM lane = row): tcgen05.ld of S, mask, running max, exp2, and
//     P as packed bf16 written back into the S columns of TMEM, where the
//     P V MMA reads it as its A operand.  O (fp32, TMEM) is rescaled only when
//     a row's max grows by more than 2^8, and normalised once at the end.
// TMEM: per Q tile h, S_h at columns 256h .. 256h+127 (P_h aliases its first
// 64 columns) and O_h at 256h+128 .. 256h+255.
// FP8 pools (F8): the MMAs take f16 operands (kind::f16 needs one type for both): each
// producer lane async-copies its rows' E4M3 bytes of a K and a V tile into a
// shared-memory staging area (kStage8), and once its own copies have landed converts
// exactly those bytes to f16 (exact: every E4M3 value is an f16 value) into the
// swizzled operand tiles; Q lands as bf16 and each softmax thread converts its own row
// in place at the start of a unit (exact inside f16's range); P is packed as f16.
// k_scale of the unit's kv head folds into the softmax scale, v_scale into 1/l.
// Every wait is bounded; a timeout sets PVA_DEVERR_TIMEOUT and the CTA winds
// down (outstanding copies and MMAs waited for, TMEM freed) without trapping.
#include <cuda.h>  // CUtensorMap and the tensor-map encoder's types (resolved through the runtime)
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "device_utils.cuh"
#include "pva_internal.h"
#include "tc_utils.cuh"

namespace pva {
namespace {

// 12 warps = three warpgroups: softmax of Q tile 0 (warps 0-3), of Q tile 1 (4-7), and
// the control group (warp 8: MMA issuer, warps 9-11: producers).  Registers move from
// the control group to the softmax groups with setmaxnreg: launched at kRegsLaunch
// each, the control warps drop to kRegsCtrl and the softmax warps rise to kRegsSoftmax
// (8 x kRegsSoftmax + 4 x kRegsCtrl == 12 x kRegsLaunch, so the increase never waits
// for registers that are not there).
constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsCtrl = 104;
static_assert(8 * kRegsSoftmax + 4 * kRegsCtrl == 12 * kRegsLaunch, "register split must balance");
constexpr int kMmaWarp = 8;
constexpr int kProducerWarp0 = 9;
constexpr int kProducerThreads = 96;
// Readers of every work-queue entry: 3 producer warps, the MMA warp, 8 softmax warps.
constexpr int kQueueReaders = 3 + 1 + 8;
constexpr int kRegion = 128 * 128;  // one 128-row x 128-byte swizzled region (64 bf16 columns)
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, bool F8 = false>
struct SmemMap {
    static constexpr int kHalves = D / 64;
    static constexpr int kTile = kRegion * kHalves;
    static constexpr int kQ = 0;                 // two Q tiles
    static constexpr int kK = kQ + 2 * kTile;    // two K stages
    static constexpr int kV = kK + 2 * kTile;    // two V stages
    static constexpr int kOff = kV + 2 * kTile;  // per producer warp: source offsets of its rows (64 x int64)
    // FP8: the raw E4M3 rows of one K tile and one V tile (row r at r * D)
    static constexpr int kStage8 = kOff + 3 * 64 * 8;
    static constexpr int kBytes = kStage8 + (F8 ? 2 * kPreRows * D : 0);
};

struct Bars {
    // q_full: both Q tiles in operand form (F8: q_raw when the bf16 rows have landed,
    // q_full once the softmax warps have converted them)
    uint64_t q_full, q_empty, q_raw;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2], o_ready[2], o_free[2];
    uint64_t drain;
    uint64_t uq_full[4], uq_empty[4];  // work queue: unit indices fetched from the global counter
    int32_t uq[4];
    uint32_t tmem_base;
    int32_t abort_flag;
    uint64_t wait_limit;  // of the work waits (the drains before the CTA leaves: the default)
};

// A work wait of one whole warp (every lane calls it, converged): the lanes' results are
// voted, so the warp leaves together or not at all -- its next steps (warp-wide tensor-core
// loads, warp syncs) need every lane.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t wlim, Bars* b,
                                              uint32_t* err) {
    if (__all_sync(0xffffffffu, dev::mbar_wait(bar, parity, wlim))) return true;
    if ((threadIdx.x & 31) == 0) {
        b->abort_flag = 1;
        dev::set_error(err, kErrTimeout);
    }
    __syncwarp();
    return false;
}

// Work queue.  Units are handed out dynamically, longest first (the plan lists them in
// that order), one at a time: entry k is filled by one producer thread when the CTA
// starts its unit k-1, so a CTA never holds more than one unit in reserve and the
// grid finishes together.  Every role reads every entry; -1 ends the kernel.
__device__ __forceinline__ void queue_push(Bars* b, int k, int32_t* counter, int n_units, uint64_t wlim,
                                           uint32_t* err) {
    if (k >= 4 && !dev::mbar_wait(&b->uq_empty[k & 3], ((k >> 2) & 1) ^ 1, wlim)) {
        b->abort_flag = 1;
        dev::set_error(err, kErrTimeout);
    }
    const int v = b->abort_flag ? n_units : atomicAdd(counter, 1);
    b->uq[k & 3] = v < n_units ? v : -1;
    dev::mbar_arrive(&b->uq_full[k & 3]);
}

// All lanes of the calling warp (converged) read entry k and lane 0 releases it; the wait
// is voted, so every lane gets the same entry (or -1).
__device__ __forceinline__ int queue_read(Bars* b, int k, int lane, uint64_t wlim, uint32_t* err) {
    int v = -1;
    if (__all_sync(0xffffffffu, dev::mbar_wait(&b->uq_full[k & 3], (k >> 2) & 1, wlim))) {
        v = b->uq[k & 3];
    } else if (lane == 0) {
        b->abort_flag = 1;
        dev::set_error(err, kErrTimeout);
    }
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(&b->uq_empty[k & 3]);
    return v;
}

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// What a unit asks for, for either kind: a prefill tile pair (keys [0, kv_end_h) of Q
// tile h, causal) or a cascade prefix-pass unit (keys [k0, k1) of the shared prefix for
// both member tiles, no causal mask).
struct UnitView {
    bool casc;
    int key_base;   // first key of the unit (on a page boundary)
    int key_end;    // keys [key_base, key_end) are loaded
    int end[2];     // keys visible to tile h end here
    int nk[2];      // 128-key tiles tile h walks (0: tile absent)
};

__device__ __forceinline__ UnitView unit_view(const PreTile& pt) {
    UnitView v;
    v.casc = pt.req < 0;
    v.key_base = v.casc ? pt.kv_end0 : 0;
    v.end[0] = v.casc ? pt.kv_end1 : pt.kv_end0;
    v.end[1] = pt.kv_end1;
    v.key_end = pt.ntok1 > 0 ? v.end[1] : v.end[0];
    v.nk[0] = pt.ntok0 > 0 ? (v.end[0] - v.key_base + kPreKeys - 1) / kPreKeys : 0;
    v.nk[1] = pt.ntok1 > 0 ? (v.end[1] - v.key_base + kPreKeys - 1) / kPreKeys : 0;
    return v;
}

// q_map: Q as a 3-D tensor (D, Hq, T) whose box is one 64-column half of a Q tile (64
// columns x G heads x TM tokens, rows in tile order); used when q_tma is nonzero.
template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const ForwardParams p, const __grid_constant__ CUtensorMap q_map, const int q_tma) {
    using L = SmemMap<D, F8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Bars bars;
    Bars* b = &bars;
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.lay.header);
    uint32_t* err = &hdr->error_bits;
    // The plan was written by the prepare kernel, which finished before the store
    // kernel released this grid; the pool rows and the work counter come from the store
    // kernel, which may still run (programmatic launch): they are read only after
    // grid_dep_wait.  An idle CTA waits too, so that this grid never completes before its
    // predecessor.  The dependents (the decode kernel) are released only after that wait,
    // so that when they start the store kernel has finished: decode does not wait for
    // this grid before its own work, only before it exits.
    const int n_units = hdr->n_pre_tiles;
    if ((hdr->error_bits & kErrFatal) || n_units == 0 || (int)blockIdx.x >= n_units) {
        // an idle CTA releases the dependents at once: with no unit at all the decode
        // kernel then waits for this grid at its start (see ForwardParams::dec_wait_late)
        dev::grid_dep_launch();
        dev::grid_dep_wait();
        return;
    }
    const PreTile* units = reinterpret_cast<const PreTile*>(p.ws + p.lay.pre_tiles);
    int32_t* counter = &hdr->pad[1];  // zeroed by the store kernel of this forward
    const CascGroup* cgroups = reinterpret_cast<const CascGroup*>(p.ws + p.lay.casc_groups);
    const int2* cmembers = reinterpret_cast<const int2*>(p.ws + p.lay.casc_members);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group, Hq = p.num_qo_heads;
    const int TM = kPreRows / G;

    for (int i = threadIdx.x * 16; i < L::kBytes; i += kThreads * 16)
        *reinterpret_cast<int4*>(smem + i) = make_int4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        dev::mbar_init(&b->q_full, F8 ? 8 : kProducerThreads);
        dev::mbar_init(&b->q_raw, kProducerThreads);
        dev::mbar_init(&b->q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            dev::mbar_init(&b->k_full[s], kProducerThreads);
            dev::mbar_init(&b->k_empty[s], 1);
            dev::mbar_init(&b->v_full[s], kProducerThreads);
            dev::mbar_init(&b->v_empty[s], 1);
            dev::mbar_init(&b->s_full[s], 1);
            dev::mbar_init(&b->p_full[s], 4);
            dev::mbar_init(&b->o_ready[s], 1);
            dev::mbar_init(&b->o_free[s], 4);
        }
        dev::mbar_init(&b->drain, 1);
        for (int s = 0; s < 4; ++s) {
            dev::mbar_init(&b->uq_full[s], 1);
            dev::mbar_init(&b->uq_empty[s], kQueueReaders);
        }
        b->abort_flag = 0;
        b->wait_limit = dev::wait_limit(hdr->wait_override);
        dev::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(&b->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = b->tmem_base;
    const uint64_t wlim = b->wait_limit;  // of the work waits, in a register for every role
    dev::grid_dep_wait();
    dev::grid_dep_launch();

    if (warp >= 8) {
        // control warpgroups: give registers to the softmax warpgroups
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
    if (warp >= kProducerWarp0) {
        // ============================================================== producer (cp.async gathers)
        // The three producer warps move the rows of every Q / K / V tile: a row is one kv
        // head of one slot (or one q head of one token), D*2 bytes, copied as 16-byte async
        // copies into the 128-byte-swizzled layout the MMA descriptors expect.  Q rows that
        // are gathered (shared-prefix members, or Q without a tensor map): the lanes of a
        // copy instruction take consecutive 16-byte chunks of kRowsPerCopy whole rows, so
        // every instruction touches whole 128-byte lines on both sides (one lane per row
        // made each instruction touch 32 lines, eight times the shared-memory wavefronts the
        // data needs, and those bursts slowed the tensor core's operand reads).  Each lane
        // computes the source offsets of two of its warp's rows into the warp's own table in
        // shared memory, which the copy loop reads back (one broadcast load per copy).
        // K and V rows (any page size) are copied by 8 lanes per 128-byte half row instead:
        // 4 rows per instruction, the offsets of a lane's 11 rows kept in registers, no
        // table round trip.  With a token-slot pool (page size 1) this form also beat the
        // table form: 255 against 327 us for the tensor-core pass of 8 contiguous prefills,
        // 108 against 142 us for the mixed batch.  A page of a few rows per kv head is too
        // small a box for TMA to stream efficiently (about 270 cycles per box measured), and
        // rows past kv_len are not copied.  The MMA thread orders these generic-proxy writes
        // before its tensor-core reads with a proxy fence after it has waited on the tile's
        // barrier.
        constexpr int kChunks = D / 8;              // 16-byte chunks per row
        constexpr int kRowsPerCopy = 32 / kChunks;  // rows one copy instruction moves
        constexpr int kStride = 3 * kRowsPerCopy;   // rows the three warps move per step
        constexpr int kCopyIters = (kPreRows + kStride - 1) / kStride;
        static_assert(kCopyIters * kRowsPerCopy <= 64, "two row offsets per lane");
        const int pwarp = warp - kProducerWarp0;  // 0..2
        const int chunk = lane % kChunks, sub = lane / kChunks;
        const int ps_mask = p.page_size - 1;
        // row of a tile held by this warp's row index k (k = copy step * kRowsPerCopy + sub)
        auto row_of = [&](int k) { return pwarp * kRowsPerCopy + (k % kRowsPerCopy) + (k / kRowsPerCopy) * kStride; };
        // every producer thread arrives on a tile's barrier when its own copies of that
        // tile have landed (hardware-tracked: the producer never waits for its loads)
        auto issue = [&](uint64_t* full) {
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(dev::smem_u32(full))
                         : "memory");
        };
        // the warp's rows of a tile; o0 / o1: element offsets (from base) of row indices lane
        // and lane + 32, -1 for a row that is not copied
        // table entry of row index k: the rows one lane copies (k = i * kRowsPerCopy + sub)
        // sit next to each other, so that the unrolled copy loop reads them as vectors
        int64_t* offs = reinterpret_cast<int64_t*>(smem + L::kOff) + pwarp * 64;
        auto slot_of = [](int k) { return (k % kRowsPerCopy) * kCopyIters + k / kRowsPerCopy; };
        auto copy_tile = [&](uint8_t* tile, int64_t o0, int64_t o1, const uint16_t* base) {
            __syncwarp();  // the previous tile's copy loop has read the table
            if (lane < kCopyIters * kRowsPerCopy) offs[slot_of(lane)] = o0;
            if (lane + 32 < kCopyIters * kRowsPerCopy) offs[slot_of(lane + 32)] = o1;
            __syncwarp();
            const uint32_t t0 = dev::smem_u32(tile) + (chunk >> 3) * kRegion;
            const uint16_t* src0 = base + chunk * 8;
            const int64_t* mine = offs + sub * kCopyIters;
#pragma unroll
            for (int i = 0; i < kCopyIters; ++i) {
                const int r = pwarp * kRowsPerCopy + sub + i * kStride;
                const int64_t o = mine[i];
                if (r < kPreRows && o >= 0) {
                    const uint32_t dst = t0 + r * 128 + (((chunk & 7) ^ (r & 7)) << 4);
                    // no memory clobber: the table reads above may then be hoisted and batched;
                    // the copies are ordered by the __syncwarp before the table is rewritten and
                    // by the mbarrier arrive that follows every tile
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src0 + o));
                }
            }
        };
        uint32_t it = 0;
        const bool fetcher = pwarp == 0 && lane == 0;
        uint64_t* q_land = F8 ? &b->q_raw : &b->q_full;
        // Leaving early (a wait that gave up) must not strand a Q tile loaded by TMA: the
        // thread that loads one remembers its phase's parity until a later unit's q_empty wait
        // shows it consumed, and waits for it before the CTA leaves; every producer arrives on
        // the Q phase of the unit it leaves in, so that the phase can complete.
        int tma_pending = -1;  // parity of this thread's TMA-loaded Q phase not yet seen consumed
        int q_arrived = 0;     // Q phases this thread has arrived on
        int uc = 0;
        if (fetcher) queue_push(b, 0, counter, n_units, wlim, err);
        for (;; ++uc) {
            const int u = queue_read(b, uc, lane, wlim, err);
            if (u < 0 || b->abort_flag) break;
            if (fetcher) queue_push(b, uc + 1, counter, n_units, wlim, err);
            const PreTile pt = units[u];
            const UnitView uv = unit_view(pt);
            const int32_t* prow =
                p.page_table + (int64_t)(uv.casc ? cgroups[-1 - pt.req].leader : pt.req) * p.ld;
            // ---- Q: row r = token (or cascade member) r / G, head r % G of each tile
            if (uc > 0 && !wait_or_abort(&b->q_empty, (uc - 1) & 1, wlim, b, err)) break;
            tma_pending = -1;  // the Q tiles of every earlier unit have been consumed
            if (q_tma && !uv.casc) {
                // consecutive tokens: the G heads of a kv head are adjacent rows of q, so a tile
                // half is one tensor box (tokens past the batch read as zeros; rows of tokens
                // past the unit's are never used).  The producers' arrivals below still count,
                // and the phase also waits for the boxes' bytes.
                if (pwarp == 0 && lane == 0) {
                    tc::fence_proxy_async_smem();  // earlier gathers into these tiles -> async-proxy writes
                    const uint32_t box = 128u * (uint32_t)(G * TM);
                    dev::mbar_expect_tx(q_land, box * (D / 64) * ((pt.ntok0 > 0) + (pt.ntok1 > 0)));
                    for (int h = 0; h < 2; ++h) {
                        if ((h ? pt.ntok1 : pt.ntok0) <= 0) continue;
                        for (int x = 0; x < D / 64; ++x)
                            tc::tma_load_3d(smem + L::kQ + h * L::kTile + x * kRegion, &q_map, x * 64, pt.kvh * G,
                                            pt.tok0 + h * TM, q_land);
                    }
                    tma_pending = uc & 1;
                }
            } else
            for (int h = 0; h < 2; ++h) {
                const int ntok = h ? pt.ntok1 : pt.ntok0;
                int64_t oq[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = row_of(lane + 32 * i);
                    const int t = r / G;
                    oq[i] = -1;
                    if (r < kPreRows && t < ntok) {
                        const int token =
                            uv.casc ? cmembers[pt.tok0 + h * TM + t].x : pt.tok0 + h * TM + t;
                        oq[i] = ((int64_t)token * Hq + pt.kvh * G + (r - t * G)) * D;
                    }
                }
                copy_tile(smem + L::kQ + h * L::kTile, oq[0], oq[1], p.q);
            }
            issue(q_land);
            ++q_arrived;
            // ---- K and V tiles
            const int kv_end = uv.key_end;
            const int nkt = (kv_end - uv.key_base + kPreKeys - 1) / kPreKeys;
            bool ok = true;
            if constexpr (F8) {
                // E4M3 rows: each lane async-copies 16 bytes (16 elements) of its rows of a tile's
                // K and V into a staging area, and once its own copies have landed converts
                // exactly those bytes to f16 (exact) into the swizzled operand tiles -- no
                // registers hold rows in flight, and the copies of a tile go out together (one
                // round trip per tile).  LPR lanes cover a row, so one copy instruction takes RPI
                // whole rows.  The next tile's page ids are read while this one is converted.
                constexpr int LPR = D / 16, RPI = 32 / LPR, RPS = 3 * RPI;
                constexpr int NS = (kPreRows + RPS - 1) / RPS;
                static_assert(NS <= 32, "one validity bit per row");
                const int sub = lane / LPR, e0 = (lane % LPR) * 16;
                const int c0 = (e0 % 64) / 8;  // first chunk of the lane's pair in its region
                const uint32_t region = (uint32_t)(e0 / 64) * kRegion;
                const int64_t ld_row = (int64_t)p.num_kv_heads * D;  // pool bytes per slot
                const uint32_t stage8 = dev::smem_u32(smem + L::kStage8);
                auto row_of8 = [&](int m) { return pwarp * RPI + sub + RPS * m; };
                auto tile_pages = [&](int j, int32_t (&pg)[NS]) {
#pragma unroll
                    for (int m = 0; m < NS; ++m) {
                        const int key = uv.key_base + j * kPreKeys + row_of8(m);
                        pg[m] = (j < nkt && row_of8(m) < kPreRows && key < kv_end) ? prow[key >> p.page_shift] : 0;
                    }
                };
                // the copies of tile j (page ids pg); returns the rows this lane copied
                auto load_tile = [&](int j, int32_t (&pg)[NS]) -> uint32_t {
                    uint32_t valid = 0;
                    bool bad = false;
#pragma unroll
                    for (int m = 0; m < NS; ++m) {
                        const int r = row_of8(m);
                        const int key = uv.key_base + j * kPreKeys + r;
                        if (r >= kPreRows || key >= kv_end) continue;
                        valid |= 1u << m;
                        int64_t page = pg[m];
                        if (page < 0 || page >= p.num_pages) {
                            bad = true;
                            page = 0;
                        }
                        const int64_t off = ((page << p.page_shift) + (key & ps_mask)) * ld_row + (int64_t)pt.kvh * D + e0;
                        const uint32_t dk = stage8 + r * D + e0, dv = dk + kPreRows * D;
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dk),
                                     "l"(reinterpret_cast<const uint8_t*>(p.k_pool) + off));
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dv),
                                     "l"(reinterpret_cast<const uint8_t*>(p.v_pool) + off));
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    if (bad) dev::set_error(err, kErrPage);
                    return valid;
                };
                // staged rows (K at 0, V at kPreRows * D) -> f16 tile, then the tile's barrier
                auto convert = [&](uint32_t valid, uint32_t src0, uint8_t* tile, uint64_t* full) {
                    const uint32_t t0 = dev::smem_u32(tile) + region;
#pragma unroll
                    for (int m = 0; m < NS; ++m) {
                        if (!(valid >> m & 1)) continue;
                        const int r = row_of8(m);
                        uint32_t x, y, z, q;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(x), "=r"(y), "=r"(z), "=r"(q)
                                     : "r"(src0 + r * D + e0));
                        const uint32_t row = t0 + r * 128;
                        dev::st_shared_v4(row + ((c0 ^ (r & 7)) << 4), dev::e4m3x2_to_f16x2(x),
                                          dev::e4m3x2_to_f16x2(x >> 16), dev::e4m3x2_to_f16x2(y),
                                          dev::e4m3x2_to_f16x2(y >> 16));
                        dev::st_shared_v4(row + (((c0 + 1) ^ (r & 7)) << 4), dev::e4m3x2_to_f16x2(z),
                                          dev::e4m3x2_to_f16x2(z >> 16), dev::e4m3x2_to_f16x2(q),
                                          dev::e4m3x2_to_f16x2(q >> 16));
                    }
                    // these generic-proxy stores -> the tensor core's operand reads
                    tc::fence_proxy_async_smem();
                    dev::mbar_arrive(full);
                };
                int32_t pg[NS];
                tile_pages(0, pg);
                uint32_t valid = nkt > 0 ? load_tile(0, pg) : 0u;
                for (int j = 0; j < nkt && ok; ++j, ++it) {
                    const int st = it & 1;
                    const uint32_t ph = (it >> 1) & 1;
                    tile_pages(j + 1, pg);
                    asm volatile("cp.async.wait_group 0;" ::: "memory");  // this lane's copies of tile j
                    if (!(ok = wait_or_abort(&b->k_empty[st], ph ^ 1, wlim, b, err))) break;
                    convert(valid, stage8, smem + L::kK + st * L::kTile, &b->k_full[st]);
                    if (!(ok = wait_or_abort(&b->v_empty[st], ph ^ 1, wlim, b, err))) break;
                    convert(valid, stage8 + kPreRows * D, smem + L::kV + st * L::kTile, &b->v_full[st]);
                    if (j + 1 < nkt) valid = load_tile(j + 1, pg);
                }
            } else {
                // 8 lanes per 128-byte half row, 4 rows per copy instruction; each lane keeps
                // the source offsets of its kG8 rows (pwarp * 4 + lane / 8 + 12 m) in registers
                constexpr int kG8 = (kPreRows + 11) / 12;
                const int grp = lane >> 3, c8 = lane & 7;
                // specialised for token slots (page size 1: the page id is the slot) and for
                // pages of several slots
                auto gather = [&](auto token_slots) {
                    constexpr bool kTok = decltype(token_slots)::value;
                    for (int j = 0; j < nkt && ok; ++j, ++it) {
                        const int st = it & 1;
                        const uint32_t ph = (it >> 1) & 1;
                        // all page ids first (independent loads in flight together), then the checks:
                        // an error report between the loads would order them one after another
                        int32_t pg[kG8];
#pragma unroll
                        for (int m = 0; m < kG8; ++m) {
                            const int r = pwarp * 4 + grp + 12 * m;
                            const int key = uv.key_base + j * kPreKeys + r;
                            pg[m] = (r < kPreRows && key < kv_end) ? prow[kTok ? key : key >> p.page_shift] : 0;
                        }
                        // each row's slot as 32 bits (a pool that fits in HBM has fewer than 2^32
                        // slots; kNoSlot: the row is not copied), the address formed at the copy:
                        // the producer warps run in 104 registers
                        constexpr uint32_t kNoSlot = 0xFFFFFFFFu;
                        uint32_t sl[kG8];
                        bool bad = false;
#pragma unroll
                        for (int m = 0; m < kG8; ++m) {
                            const int r = pwarp * 4 + grp + 12 * m;
                            const int key = uv.key_base + j * kPreKeys + r;
                            sl[m] = kNoSlot;
                            if (r < kPreRows && key < kv_end) {
                                int64_t page = pg[m];
                                if (page < 0 || page >= p.num_pages) {
                                    bad = true;
                                    page = 0;
                                }
                                sl[m] = (uint32_t)(kTok ? page : (page << p.page_shift) + (key & ps_mask));
                            }
                        }
                        if (bad) dev::set_error(err, kErrPage);
                        const int64_t slot_elems = (int64_t)p.num_kv_heads * D;
                        auto copy_g8 = [&](uint8_t* tile, const uint16_t* base) {
                            const uint32_t t0 = dev::smem_u32(tile);
                            const uint16_t* b0 = base + (int64_t)pt.kvh * D + c8 * 8;
#pragma unroll
                            for (int m = 0; m < kG8; ++m) {
                                const int r = pwarp * 4 + grp + 12 * m;
                                if (sl[m] == kNoSlot) continue;
                                const uint16_t* src = b0 + (int64_t)sl[m] * slot_elems;
                                const uint32_t d = t0 + r * 128 + ((c8 ^ (r & 7)) << 4);
                                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src));
                                if (D == 128)
                                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + kRegion),
                                                 "l"(src + 64));
                            }
                        };
                        if (!wait_or_abort(&b->k_empty[st], ph ^ 1, wlim, b, err)) {
                            ok = false;
                            break;
                        }
                        copy_g8(smem + L::kK + st * L::kTile, p.k_pool);
                        issue(&b->k_full[st]);
                        if (!wait_or_abort(&b->v_empty[st], ph ^ 1, wlim, b, err)) {
                            ok = false;
                            break;
                        }
                        copy_g8(smem + L::kV + st * L::kTile, p.v_pool);
                        issue(&b->v_full[st]);
                    }
                };
                if (p.page_size == 1)
                    gather(BoolTag<true>{});
                else
                    gather(BoolTag<false>{});
            }
            if (!ok) break;
        }
        // After an abort, this thread arrives on the Q phase of the unit it left in (so that
        // the phase can complete); then its TMA-loaded Q tile and its async copies must land
        // before the CTA may leave.  (Not at a normal end: a phase completed by those
        // arrivals would put the barrier two phases ahead of a warp still waiting on the
        // one before, which shares its parity.)
        if (b->abort_flag && q_arrived == uc) issue(q_land);
        if (tma_pending >= 0) (void)dev::mbar_wait(q_land, (uint32_t)tma_pending);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else if (warp == kMmaWarp) {
        // ============================================================== MMA issuer (one warp)
        // The whole warp runs this role with warp-uniform control flow (every wait is voted
        // across the warp); each MMA and commit is issued by one elected lane.
        const uint32_t id_qk = F8 ? tc::idesc_f16_f32(128, 128, 0, 0) : tc::idesc_bf16_f32(128, 128, 0, 0);
        const uint32_t id_pv = F8 ? tc::idesc_f16_f32(128, D, 0, 1) : tc::idesc_bf16_f32(128, D, 0, 1);
        constexpr uint32_t kDescHi = tc::smem_desc_hi(1024, tc::kSwizzle128B);
        constexpr uint32_t kTileLo = L::kTile >> 4;  // one tile, in descriptor address units
        // descriptor low words: Q tiles and K stages K-major, V stages MN-major (the leading
        // byte offset of V steps from one 64-column region to the next)
        const uint32_t q_lo = tc::smem_desc_lo(dev::smem_u32(smem + L::kQ), 16);
        const uint32_t k_lo = tc::smem_desc_lo(dev::smem_u32(smem + L::kK), 16);
        const uint32_t v_lo = tc::smem_desc_lo(dev::smem_u32(smem + L::kV), kRegion);
        auto wait = [&](uint64_t* bar, uint32_t parity) -> bool { return wait_or_abort(bar, parity, wlim, b, err); };
        uint32_t it = 0;                      // KV tiles across units
        uint32_t n_p[2] = {0, 0};             // P tiles consumed per Q tile
        uint32_t n_units_h[2] = {0, 0};       // units that had Q tile h
        bool ok = true;
        // S_h = Q_h K(st)^T: K-steps of 16 columns inside a 128-byte swizzle row, then the
        // next 64-column region
        // `mid` runs after the first half of the MMAs, when the tensor core's queue is full:
        // work placed there overlaps the queued products instead of leaving the queue empty
        auto issue_s = [&](int h, int st, auto&& mid) {
            const uint32_t a0 = q_lo + h * kTileLo, b0 = k_lo + st * kTileLo;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if (kk == D / 32) mid();
                const uint32_t off = (uint32_t)((kk >> 2) * kRegion + (kk & 3) * 32) >> 4;
                tc::mma_ss_warp(tmem + 256 * h, a0 + off, b0 + off, kDescHi, id_qk, kk > 0 ? 1u : 0u);
            }
            tc::mma_commit_warp(&b->s_full[h]);
        };
        auto nothing = [] {};
        // O_h += P_h V(st); P_h is read from TMEM (the first 64 columns of S_h), V in K-steps
        // of 16 rows (2048 bytes)
        auto issue_pv = [&](int h, int st, bool first) -> bool {
            if (!wait(&b->p_full[h], n_p[h] & 1)) return false;
            ++n_p[h];
            if (first && n_units_h[h] > 0 && !wait(&b->o_free[h], (n_units_h[h] - 1) & 1)) return false;
            tc::fence_after_sync();
            const uint32_t b0 = v_lo + st * kTileLo;
#pragma unroll
            for (int kk = 0; kk < kPreKeys / 16; ++kk)
                tc::mma_ts_warp(tmem + 256 * h + 128, tmem + 256 * h + kk * 8, b0 + kk * (2048 >> 4), kDescHi, id_pv,
                                (first && kk == 0) ? 0u : 1u);
            return true;
        };
        for (int uc = 0; ok; ++uc) {
            const int u = __shfl_sync(0xffffffffu, queue_read(b, uc, lane, wlim, err), 0);
            if (u < 0) break;
            const UnitView uv = unit_view(units[u]);
            const int nkt0 = uv.nk[0];
            const int nkt1 = uv.nk[1];
            const int nkt = nkt1 > nkt0 ? nkt1 : nkt0;
            if (!wait(&b->q_full, uc & 1)) break;
            // prologue: S_h(0) for both tiles
            if (!wait(&b->k_full[it & 1], (it >> 1) & 1)) break;
            tc::fence_after_sync();
            tc::fence_proxy_async_smem();  // the producers' generic-proxy copies -> MMA operand reads
            if (nkt0 > 0) issue_s(0, it & 1, nothing);
            if (nkt1 > 0) issue_s(1, it & 1, nothing);
            tc::mma_commit_warp(&b->k_empty[it & 1]);
            if (nkt == 1) tc::mma_commit_warp(&b->q_empty);
            // inputs of the coming step (V(t), K(t + 1)) already seen complete
            bool inputs_seen = false;
            for (int j = 0; j < nkt && ok; ++j) {
                const uint32_t t = it + j;
                const int st = t & 1, st1 = (t + 1) & 1;
                const bool next = j + 1 < nkt;
                if (!inputs_seen &&
                    !(ok = wait(&b->v_full[st], (t >> 1) & 1) && (!next || wait(&b->k_full[st1], ((t + 1) >> 1) & 1))))
                    break;
                inputs_seen = false;
                tc::fence_after_sync();
                tc::fence_proxy_async_smem();
                // the last product of this step that reads V(t), and the last S
                const int last_pv = j < nkt1 ? 1 : 0;
                const int last_s = j + 1 < nkt1 ? 1 : 0;
                // in the middle of the last S: a look (no wait) at the next step's inputs, and the
                // release of V(t)'s stage
                auto probe = [&] {
                    if (j + 1 < nkt) {
                        const uint32_t t1 = t + 1;
                        inputs_seen = __all_sync(0xffffffffu, dev::mbar_test_wait(&b->v_full[st1], (t1 >> 1) & 1) &&
                                                                  (j + 2 >= nkt || dev::mbar_test_wait(&b->k_full[st],
                                                                                                       ((t1 + 1) >> 1) & 1)));
                    }
                };
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int nk = h ? nkt1 : nkt0;
                    if (j >= nk) continue;
                    if (!(ok = issue_pv(h, st, j == 0))) break;
                    if (j == nk - 1) tc::mma_commit_warp(&b->o_ready[h]);
                    if (h == last_pv) tc::mma_commit_warp(&b->v_empty[st]);
                    if (j + 1 < nk) {
                        if (h == last_s) issue_s(h, st1, probe);
                        else issue_s(h, st1, nothing);
                    }
                }
                if (!ok) break;
                if (next) {
                    tc::mma_commit_warp(&b->k_empty[st1]);
                    if (j + 1 == nkt - 1) tc::mma_commit_warp(&b->q_empty);
                }
            }
            if (nkt0 > 0) ++n_units_h[0];
            if (nkt1 > 0) ++n_units_h[1];
            it += nkt;
        }
        // every MMA issued must complete before TMEM is released
        tc::mma_commit_warp(&b->drain);
        (void)dev::mbar_wait(&b->drain, 0);
        __syncwarp();
    }  // warps 10-11: idle
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ============================================================== softmax (one row per thread)
        const int h = warp >> 2;  // Q tile of this warpgroup
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + 256 * h + lane_base;
        const uint32_t t_o = t_s + 128;
        const float sl_base = p.scale_log2;
        uint32_t n_s = 0;   // S tiles seen by this warpgroup
        uint32_t n_u = 0;   // units with this Q tile
        for (int k = 0;; ++k) {
            const int u = queue_read(b, k, lane, wlim, err);
            if (u < 0 || b->abort_flag) break;
            const PreTile pt = units[u];
            const UnitView uv = unit_view(pt);
            const int ntok = h ? pt.ntok1 : pt.ntok0;
            const int nk = uv.nk[h];
            if constexpr (F8) {
                // this thread's row of Q tile h, bf16 -> f16 in place (both regions; every
                // warp takes part in every unit: q_full counts the eight softmax warps)
                if (!wait_or_abort(&b->q_raw, k & 1, wlim, b, err)) break;
#pragma unroll
                for (int x = 0; x < D / 64; ++x) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4* q16 = reinterpret_cast<uint4*>(smem + L::kQ + h * L::kTile + x * kRegion + row * 128 +
                                                              c * 16);
                        const uint4 v = *q16;
                        *q16 = make_uint4(dev::bf16x2_to_f16x2(v.x), dev::bf16x2_to_f16x2(v.y),
                                          dev::bf16x2_to_f16x2(v.z), dev::bf16x2_to_f16x2(v.w));
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&b->q_full);
            }
            if (nk == 0) continue;
            const float sl = F8 ? sl_base * p.k_scale[pt.kvh] : sl_base;
            const bool valid = row < ntok * G;
            // last visible key of this row, and the first key some row may not see
            const int qpos = pt.qpos0 + h * TM;
            const int limit = !valid ? -1 : (uv.casc ? uv.end[h] - 1 : qpos + row / G);
            const int mask_from = uv.casc ? uv.end[h] : qpos + 1;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < nk; ++j, ++n_s) {
                if (!wait_or_abort(&b->s_full[h], n_s & 1, wlim, b, err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                // the whole S row: four 32-column TMEM loads in flight, one wait
                float s[kPreKeys / 32][32];
#pragma unroll
                for (int c = 0; c < kPreKeys / 32; ++c) tc::tmem_ld32_async(t_s + c * 32, s[c]);
#pragma unroll
                for (int c = 0; c < kPreKeys / 32; ++c) tc::tmem_wait_ld_regs(s[c]);
                const int key0 = uv.key_base + j * kPreKeys;
                const bool need_mask = key0 + kPreKeys - 1 >= mask_from;
                if (need_mask) {  // a tile crossing the diagonal (or the end of the keys)
#pragma unroll
                    for (int c = 0; c < kPreKeys; ++c)
                        if (key0 + c > limit) s[c >> 5][c & 31] = -INFINITY;
                }
                // row maximum: three-input max over 8 independent chains
                float mxa[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mxa[i] = fmaxf(s[0][2 * i], s[0][2 * i + 1]);
#pragma unroll
                for (int c = 16; c < kPreKeys; c += 2) {
                    const int i = (c >> 1) & 7;
                    mxa[i] = dev::fmax3(mxa[i], s[c >> 5][c & 31], s[(c + 1) >> 5][(c + 1) & 31]);
                }
                const float mx = dev::fmax3(dev::fmax3(mxa[0], mxa[1], mxa[2]), dev::fmax3(mxa[3], mxa[4], mxa[5]),
                                            fmaxf(mxa[6], mxa[7]));
                const float m_new = fmaxf(m, mx * sl);  // log2 units (sl = scale * log2 e > 0)
                // rescale decision: the row maximum grew by more than the threshold; O itself is
                // rescaled after P is written (the S registers are dead by then), before P is
                // signalled, so the PV product of this tile adds to the rescaled O
                float alpha = 1.f;
                bool resc = false;
                if (j == 0) {
                    m = m_new;
                } else {
                    resc = m_new > m + kRescaleThreshold;
                    if (resc) {
                        alpha = dev::fast_exp2(m - m_new);
                        l *= alpha;
                        m = m_new;
                    }
                }
                const float nmu = m == -INFINITY ? 0.f : -m;
                float lsa[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) lsa[i] = 0.f;
                // P = exp2(s * sl - m) as packed bf16 pairs, 16 columns (32 keys) per TMEM store
                // (a quarter of the row at a time keeps fewer registers live); the
                // scale-and-shift and the row sum run as packed fp32 pairs
#pragma unroll
                for (int c2 = 0; c2 < kPreKeys / 32; ++c2) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int c = c2 * 32 + 2 * i;
                        float x0, x1;
                        dev::ffma2(x0, x1, s[c >> 5][c & 31], s[(c + 1) >> 5][(c + 1) & 31], sl, sl, nmu, nmu);
                        const float e0 = dev::fast_exp2(x0);
                        const float e1 = dev::fast_exp2(x1);
                        dev::fadd2(lsa[2 * (i & 3)], lsa[2 * (i & 3) + 1], e0, e1);
                        pk[i] = F8 ? dev::pack_f16x2(e0, e1) : dev::pack_bf16x2(e0, e1);
                    }
                    tc::tmem_st16u(t_s + c2 * 16, pk);
                }
                l += ((lsa[0] + lsa[1]) + (lsa[2] + lsa[3])) + ((lsa[4] + lsa[5]) + (lsa[6] + lsa[7]));
                if (__any_sync(0xffffffffu, resc)) {
                    // O_h is stable here: P_h(j-1) V was issued before S_h(j), whose
                    // completion this thread has observed
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float v[32];
                        tc::tmem_ld32_async(t_o + c * 32, v);
                        tc::tmem_wait_ld_regs(v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= alpha;
                        tc::tmem_st32(t_o + c * 32, v);
                    }
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(&b->p_full[h]);
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16 rows of out, LSE
            if (!wait_or_abort(&b->o_ready[h], n_u & 1, wlim, b, err)) break;
            tc::fence_after_sync();
            const float inv = l > 0.f ? (F8 ? p.v_scale[pt.kvh] : 1.f) / l : 0.f;
            const int64_t orow = (valid && !uv.casc)
                                     ? ((int64_t)(pt.tok0 + h * TM + row / G) * Hq + pt.kvh * G + row % G)
                                     : 0;
            float o[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tc::tmem_ld32_async(t_o + c * 32, o[c]);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tc::tmem_wait_ld_regs(o[c]);
            // O is in registers: the accumulator may be overwritten by the next unit
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&b->o_free[h]);
            ++n_u;
            if (valid && uv.casc) {
                // prefix-pass partial of a cascade member: normalised O and the log2-domain
                // LSE into the member's slot for this key chunk (combined by the merge kernel)
                const int slot = cmembers[pt.tok0 + h * TM + row / G].y + pt.qpos0;
                const int prow = pt.kvh * G + row % G;  // one new token: row = q head
                float* po = reinterpret_cast<float*>(p.ws + p.lay.partial_o) +
                            ((int64_t)slot * p.lay.rows_per_slot + prow) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        reinterpret_cast<float4*>(po + c * 32)[q4] =
                            make_float4(o[c][q4 * 4] * inv, o[c][q4 * 4 + 1] * inv, o[c][q4 * 4 + 2] * inv,
                                        o[c][q4 * 4 + 3] * inv);
                }
                reinterpret_cast<float*>(p.ws + p.lay.partial_lse)[(int64_t)slot * p.lay.rows_per_slot + prow] =
                    l > 0.f ? m + __log2f(l) : -INFINITY;
            } else if (valid) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D + c * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = dev::pack_bf16x2(o[c][q4 * 8 + 0] * inv, o[c][q4 * 8 + 1] * inv);
                        w.y = dev::pack_bf16x2(o[c][q4 * 8 + 2] * inv, o[c][q4 * 8 + 3] * inv);
                        w.z = dev::pack_bf16x2(o[c][q4 * 8 + 4] * inv, o[c][q4 * 8 + 5] * inv);
                        w.w = dev::pack_bf16x2(o[c][q4 * 8 + 6] * inv, o[c][q4 * 8 + 7] * inv);
                        dst[q4] = w;
                    }
                }
                if (p.lse != nullptr) p.lse[orow] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// The Q tensor map of the kernel; false when it cannot be built (the kernel then gathers
// Q rows with async copies, as it does for cascade members).
bool encode_q_map(const ForwardParams& p, int D, CUtensorMap* m) {
    const EncodeTiledFn enc = tensor_map_encoder();
    if (enc == nullptr || p.total_tokens <= 0 || (reinterpret_cast<uintptr_t>(p.q) & 15) != 0) return false;
    const int G = p.group, TM = kPreRows / G;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.num_qo_heads, (cuuint64_t)p.total_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.num_qo_heads * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TM};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(p.q), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool F8>
cudaError_t launch_p(const ForwardParams& p, int ctas, cudaStream_t s) {
    const size_t smem = SmemMap<D, F8>::kBytes + 1024;
    static_assert(SmemMap<D, F8>::kBytes + 1024 + 512 <= 227 * 1024, "shared memory per block");
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // The register split inside the kernel assumes the launch allocates exactly
    // kRegsLaunch registers per thread; with fewer, the softmax warps' increase
    // could not be satisfied.  Refuse to launch rather than risk that.
    static int launch_regs = -1;
    if (launch_regs < 0) {
        cudaFuncAttributes attr{};
        e = cudaFuncGetAttributes(&attr, prefill_kernel<D, F8>);
        if (e != cudaSuccess) return e;
        launch_regs = attr.numRegs;
    }
    if (launch_regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
    CUtensorMap q_map;
    memset(&q_map, 0, sizeof(q_map));
    const int q_tma = encode_q_map(p, D, &q_map) ? 1 : 0;
    return launch_programmatic(prefill_kernel<D, F8>, (unsigned)ctas, (unsigned)kThreads, smem, s, p, q_map,
                               q_tma);
}

}  // namespace

bool prefill_supported(int num_qo_heads, int num_kv_heads, int head_dim) {
    if (head_dim != 64 && head_dim != 128) return false;
    const int G = num_qo_heads / num_kv_heads;
    return G >= 1 && G <= 16;
}

cudaError_t launch_prefill(const ForwardParams& p, int head_dim, int ctas, cudaStream_t s) {
    if (ctas <= 0) return cudaSuccess;
    if (head_dim == 128) return p.kv_fp8 ? launch_p<128, true>(p, ctas, s) : launch_p<128, false>(p, ctas, s);
    if (head_dim == 64) return p.kv_fp8 ? launch_p<64, true>(p, ctas, s) : launch_p<64, false>(p, ctas, s);
    return cudaErrorInvalidValue;
}

}  // namespace pva
