// K1: store_kvcache -- this step's K and V rows scattered into the paged pool.
//
// "The attention backend and a reference implementation" (section
// "Variable-length, paged attention with prefixes"): the forward writes this
// step's K/V into the pool before reading any of it back; "Attention backends:
// backend, metadata builder and implementation" (step 2) describes the same
// update as a scatter by slot.  A slot row holds all kv heads of one token,
// Hkv * D bf16 = 1-2 KiB contiguous in both the source and the pool, so one
// warp moves one token's K row (or V row) with 16-byte vector accesses: reads
// stream past L1, writes stay in L2 for the attention kernels that follow.  Into an
// FP8 pool each element is quantised on the way (x / scale of its kv head, to E4M3).
// Without a caller slot_mapping each warp derives its token's slot from the page table
// (the token's request comes from the plan): the new tokens are the request's last
// q_len positions.
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "pva_internal.h"

namespace pva {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) store_kernel(ForwardParams p, int row_vecs) {
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.lay.header);
    // Launched programmatically: the kernel before it (the prepare kernel, or the previous
    // forward's last kernel, which may still read the pool) must have finished before the
    // plan, the slots or the pool are touched.  Only then may the attention kernel that
    // follows set up its CTAs: it reads the plan before its own grid_dep_wait, so the plan
    // must be complete when it starts, and it reads nothing this kernel writes before that
    // wait.
    dev::grid_dep_wait();
    dev::grid_dep_launch();
    // the attention kernels that follow fetch their work from these counters
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->pad[0] = 0;  // decode kernel work counter
        hdr->pad[1] = 0;  // prefill kernel work counter
    }
    if (hdr->error_bits & kErrFatal) return;
    const int lane = threadIdx.x & 31;
    const int64_t job = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);  // (token, K|V)
    if (job >= 2 * (int64_t)p.total_tokens) return;
    const int64_t t = job >> 1;
    const bool is_v = job & 1;
    int64_t slot;
    if (p.slots != nullptr) {
        slot = p.slots[t];
    } else {
        // slot mapping derived from the page table: the new tokens of request i are its last
        // q_len positions (prepare recorded each token's request)
        const int i = p.tok_req[t];
        const int c0 = p.cu[i], n = p.cu[i + 1] - c0, L = p.seqlens[i];
        const int pos = L - n + (int)(t - c0);
        const int64_t page = p.page_table[(int64_t)i * p.ld + (pos >> p.page_shift)];
        if (page < 0 || page >= p.num_pages) {
            if (lane == 0 && !is_v) dev::set_error(&hdr->error_bits, kErrPage);
            return;
        }
        slot = (page << p.page_shift) + (pos & (p.page_size - 1));
    }
    if (slot == -1) return;
    if (slot < 0 || slot >= p.num_slots) {
        if (lane == 0 && !is_v) dev::set_error(&hdr->error_bits, kErrSlot);
        return;
    }
    const int4* src = reinterpret_cast<const int4*>(is_v ? p.v : p.k) + t * row_vecs;
    if (!p.kv_fp8) {
        int4* dst = reinterpret_cast<int4*>(is_v ? p.v_pool : p.k_pool) + slot * row_vecs;
        for (int i = lane; i < row_vecs; i += 32) dst[i] = dev::ld_stream_v4(src + i);
        return;
    }
    // FP8 pool: element (h, d) becomes e4m3(x / scale[h]) (IEEE division, nearest even,
    // saturating); a lane turns 16 elements (two source vectors, one head) into one
    // 16-byte pool vector
    const float* scale = is_v ? p.v_scale : p.k_scale;
    int4* dst = reinterpret_cast<int4*>(is_v ? p.v_pool : p.k_pool) + slot * (row_vecs / 2);
    const int D = row_vecs * 8 / p.num_kv_heads;
    for (int i = lane; i < row_vecs / 2; i += 32) {
        const float sc = scale[(16 * i) / D];
        const int4 a = dev::ld_stream_v4(src + 2 * i), b = dev::ld_stream_v4(src + 2 * i + 1);
        const uint32_t w[8] = {(uint32_t)a.x, (uint32_t)a.y, (uint32_t)a.z, (uint32_t)a.w,
                               (uint32_t)b.x, (uint32_t)b.y, (uint32_t)b.z, (uint32_t)b.w};
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float x0 = __fdiv_rn(__uint_as_float(w[2 * j] << 16), sc);
            const float x1 = __fdiv_rn(__uint_as_float(w[2 * j] & 0xFFFF0000u), sc);
            const float x2 = __fdiv_rn(__uint_as_float(w[2 * j + 1] << 16), sc);
            const float x3 = __fdiv_rn(__uint_as_float(w[2 * j + 1] & 0xFFFF0000u), sc);
            q[j] = dev::f32x2_to_e4m3x2(x0, x1) | (dev::f32x2_to_e4m3x2(x2, x3) << 16);
        }
        dst[i] = make_int4((int)q[0], (int)q[1], (int)q[2], (int)q[3]);
    }
}

}  // namespace

cudaError_t launch_store(const ForwardParams& p, int head_dim, cudaStream_t s) {
    if (p.total_tokens <= 0) return cudaSuccess;
    const int row_vecs = p.num_kv_heads * head_dim * 2 / 16;
    const int64_t jobs = 2 * (int64_t)p.total_tokens;
    const int64_t blocks = (jobs + kThreads / 32 - 1) / (kThreads / 32);
    return launch_programmatic(store_kernel, (unsigned)blocks, (unsigned)kThreads, 0, s, p, row_vecs);
}

}  // namespace pva
