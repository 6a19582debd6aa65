// Internal plan layout shared by the host API and the kernels of libpva.so.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/pva.h"

namespace pva {

// ---------------------------------------------------------------- tiling constants

// Decode/row-block kernel: keys per pipeline stage and maximum rows (q tokens x
// q heads of one kv head) one warp holds -- the M of one m16n8k16 tile.
constexpr int kDecKeysPerStage = 16;
constexpr int kDecRows = 16;
// Tensor-core prefill kernel: rows per tile (M of tcgen05.mma) and keys per KV tile.
constexpr int kPreRows = 128;
constexpr int kPreKeys = 128;
// Smallest split-KV chunk (keys) worth a separate CTA.
constexpr int kMinSplitChunk = 256;
// Most key chunks one shared prefix is cut into for the cascade prefix pass.
constexpr int kMaxCascChunks = 8;
// Deepest level of the shared-prefix tree detected (level 1: a run of leading pages shared
// by a group; level L + 1: a further run shared by some members of a level-L group).
// With n levels in a batch each level's prefixes are cut into at most kMaxCascChunks / n
// chunks, so every level keeps at least one.
constexpr int kMaxCascLevels = 8;
static_assert(kMaxCascLevels <= kMaxCascChunks, "every level keeps one prefix chunk");
constexpr int kDecHeadBlock = 8;     // kv heads one decode CTA serves (more: several CTAs per unit)
constexpr int kMinDecShare = 128;    // fewest keys a decode CTA gets in the balanced split
// Keys the balanced split charges for starting a group's piece: on the key line each group is
// followed by a gap of this many keys that no CTA processes, so a CTA whose share holds more
// group starts gets fewer keys (a piece start cost ~0.9 us on the decode workload, about the
// time of 9 keys of 4 KiB at one SM's streaming rate; measured per CTA: one piece 111.0 us,
// two 112.1, three 113.0).
constexpr int kDecPieceCost = 16;

// Error bits the kernels OR into the plan's error word (same values as pva.h).
constexpr uint32_t kErrCu = PVA_DEVERR_CU_SEQLENS;
constexpr uint32_t kErrQgtKv = PVA_DEVERR_Q_GT_KV;
constexpr uint32_t kErrPage = PVA_DEVERR_PAGE_ID;
constexpr uint32_t kErrSlot = PVA_DEVERR_SLOT;
constexpr uint32_t kErrLimits = PVA_DEVERR_LIMITS;
constexpr uint32_t kErrTimeout = PVA_DEVERR_TIMEOUT;
// Errors that make the whole batch description untrustworthy: nothing runs.
constexpr uint32_t kErrFatal = kErrCu | kErrQgtKv | kErrLimits;

// ---------------------------------------------------------------- device plan records

// Header at offset 0 of the workspace, written by the prepare kernel.
struct PlanHeader {
    uint32_t error_bits;
    int32_t n_dec_units;
    int32_t n_dec_groups;
    int32_t n_pre_tiles;
    int32_t n_casc_groups;
    int32_t n_casc_tiles;
    int32_t split_chunk;
    int32_t n_partial_slots;
    int32_t n_casc_units;
    int32_t max_group_tokens;  // most tokens in one decode group (bounds the merge's rows)
    int32_t dec_share;         // keys per decode CTA of the balanced split; 0: the work queue
    uint32_t wait_override;    // tests only: wait limit in ns + 1 for the forward kernels' work
                               // waits (attn_debug_set_wait_limit); 0 (set by prepare): default
    int32_t n_casc_levels;     // deepest shared-prefix level with a group (0: none)
    int32_t pad[51];           // pad[0] / pad[1]: decode / tensor-core work counters
};
static_assert(sizeof(PlanHeader) == 256, "header is one 256-byte line");

// A decode group: up to floor(16 / G) consecutive new tokens of one request,
// all q heads.  One merge (LSE combine) per group when it is split.
struct DecGroup {
    int32_t req;
    int32_t tok0;        // global index of the first token (row of q)
    int32_t ntok;        // tokens in the group (>= 1)
    int32_t qpos0;       // absolute position of the first token: kv_len - q_len + (tok0 - cu[req])
    int32_t nsplit;      // number of units (key ranges) covering the group
    int32_t pbase;       // first partial slot (valid when nsplit > 1)
    int32_t kv_end;      // keys [0, kv_end) are visible to some token of the group
    int32_t casc;        // cascade group id feeding prefix partials, or -1
    int32_t nparts;      // partial slots of the group (see DecUnit::nparts)
    int32_t tail0;       // first key the decode units cover (the prefix length of a cascade member)
    int32_t g0;          // balanced split: first key of the group in the batch's key line
    int32_t pad1, pad2, pad3, pad4, pad5;
};
static_assert(sizeof(DecGroup) == 64, "DecGroup is one 64-byte record");

// One CTA work item of the decode kernel: keys [k0, k1) of a group.  The group's
// fields are repeated here so that one load brings everything a unit needs.
struct DecUnit {
    int32_t group;
    int32_t k0;
    int32_t k1;
    int32_t split;       // index among the group's units (partial slot pbase + split)
    int32_t req;
    int32_t tok0;
    int32_t ntok;
    int32_t qpos0;
    int32_t nsplit;      // units (CTAs) that arrive on the group's counter
    int32_t pbase;
    int32_t nparts;      // partial slots merged: nsplit, plus the prefix chunks of a cascade member
    int32_t pad1;
};

// A shared-prefix (cascade) group: decode requests whose page tables start with the
// same prefix_len / page_size pages.  The prefix pass attends every member's query
// rows to the prefix keys once per chunk of keys; the members' decode units cover only
// the keys after the prefix, and the merge combines both by log-sum-exp.
struct CascGroup {
    int32_t leader;       // request whose page-table row addresses the prefix
    int32_t prefix_len;   // keys [key_base, prefix_len) are shared by the members
    int32_t n_members;
    int32_t member_off;   // members[member_off ..]: (token, first prefix partial slot) per member
    int32_t n_chunks;     // prefix pass key chunks
    int32_t chunk_keys;   // keys per chunk (multiple of kPreKeys)
    int32_t unit_off;     // first prefix-pass unit of the group (relative to the cascade units)
    int32_t n_units;
    int32_t key_base;     // 0 for a top-level group; a sub-group's: its parent's prefix_len
    int32_t level;        // 0 top level, 1 sub-group
    int32_t pad0, pad1;
};
static_assert(sizeof(CascGroup) % 16 == 0, "CascGroup is whole 16-byte words");

// One work unit of the tensor-core prefill kernel: two consecutive Q tiles of one
// request and kv head.  A Q tile is kPreRows rows = floor(kPreRows / G) tokens x the
// G q heads; tile h covers tokens tok0 + h*TM ..; it sees keys [0, kv_end_h) with the
// causal diagonal.  ntok1 == 0 when the request has no second tile here.
struct PreTile {
    int32_t req;
    int32_t kvh;
    int32_t tok0;        // global index of the first token of tile 0
    int32_t ntok0;       // tokens in tile 0 (>= 1)
    int32_t ntok1;       // tokens in tile 1 (0: absent)
    int32_t qpos0;       // absolute position of the first token of tile 0
    int32_t kv_end0;     // keys [0, kv_end0) for tile 0
    int32_t kv_end1;     // keys [0, kv_end1) for tile 1
};
// A cascade prefix-pass unit reuses PreTile: req = -1 - cascade group, tok0 = first
// member (index into the member list), ntok0 / ntok1 = members in Q tile 0 / 1, qpos0 =
// key chunk, kv_end0 / kv_end1 = the chunk's keys [k0, k1).  No causal mask applies:
// the prefix lies before every member's query.

// Workspace carve-up (byte offsets from the workspace base); computed on the host.
struct Layout {
    size_t header;
    size_t dec_units;
    size_t dec_groups;
    size_t pre_tiles;
    size_t slots;        // int32 [max_tokens]: request of each new token (the slot mapping is derived from it)
    size_t partial_o;    // fp32 [max_partial][rows_per_slot][D]
    size_t partial_lse;  // fp32 [max_partial][rows_per_slot]
    size_t req_scratch;  // int32 [max_batch * 4] prepare scratch
    size_t casc_groups;  // CascGroup [max_casc_groups]
    size_t casc_members; // int2 [kMaxCascLevels * max_batch]: member's token, partial slot of its prefix chunk 0
    size_t casc_deep;    // int32 [3 * (kMaxCascLevels - 2) * (max_batch + 1)]: levels 3 and deeper, per request
    size_t dec_first;    // int32 [dec_ctas + 1]: balanced split, first group of each CTA's keys
    size_t total;
    int32_t max_dec_units;
    int32_t max_dec_groups;
    int32_t max_pre_tiles;
    int32_t max_partial;
    int32_t rows_per_slot;
    int32_t target_units;
    int32_t max_casc_groups;
    int32_t casc_target;  // most prefix-pass units aimed for (one per SM; prepare aims lower)
    int32_t dec_ctas;     // CTAs of the decode grid
};

// Parameters of the prepare kernel (by value).
struct PrepareParams {
    const int32_t* cu;
    const int32_t* seqlens;
    const int32_t* page_table;
    int64_t ld;
    const int64_t* user_slots;   // may be null
    int32_t* tok_req;            // request of each new token, written when user_slots is null
    int32_t batch;
    int32_t total_tokens;
    int32_t max_q_len;
    int32_t page_size;
    int64_t num_pages;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t group;               // Hq / Hkv
    int32_t dec_tokens;          // tokens per decode group = 16 / group
    int32_t pre_tokens;          // tokens per prefill tile = 128 / group
    int32_t use_prefill;         // 1: requests with q_len > dec_tokens go to the prefill kernel
    int32_t use_cascade;         // 1: detect shared prefixes among decodes
    int32_t min_cascade_pages;
    int32_t smem_batch;          // per-request arrays live in shared memory when batch <= this
    int32_t split_kv;
    int32_t kv_fp8;              // 1: E4M3 pools (weighs the prefix pass against the tails)
    int32_t max_kv_len;
    int32_t max_tokens;
    int32_t max_batch;
    uint8_t* ws;
    Layout lay;
};

// Parameters common to the forward kernels (by value).
struct ForwardParams {
    const uint16_t* q;           // bf16 bits [T, Hq, D]
    const uint16_t* k;           // [T, Hkv, D]
    const uint16_t* v;
    uint16_t* k_pool;            // [slots, Hkv, D]
    uint16_t* v_pool;
    uint16_t* out;               // [T, Hq, D]
    float* lse;                  // [T, Hq] or null
    const int32_t* cu;
    const int32_t* seqlens;
    const int32_t* page_table;
    int64_t ld;
    const int64_t* slots;        // the caller's slot mapping, or null: derived from tok_req
    const int32_t* tok_req;      // request of each new token (when slots is null)
    int32_t total_tokens;
    int32_t page_size;
    int32_t page_shift;          // log2(page_size)
    int64_t num_pages;
    int64_t num_slots;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t group;
    float scale_log2;            // sm_scale * log2(e)
    uint8_t* ws;
    Layout lay;
    // FP8 (E4M3) pools: k_pool / v_pool hold one byte per element and each kv head h
    // has the scales k_scale[h], v_scale[h] (device fp32); zero for bf16 pools
    int32_t kv_fp8;
    const float* k_scale;
    const float* v_scale;
    // the decode kernel follows the tensor-core kernel; when that kernel has units it
    // signals its dependents only after its own wait for the store kernel, and decode
    // then starts on SMs the tensor-core kernel has left and waits for that grid only
    // before it exits
    int32_t dec_wait_late;
};

// Host view of a prepared batch, stored inside pva_meta::opaque.
struct MetaHost {
    uint64_t magic;
    pva_config cfg;
    int32_t batch;
    int32_t total_tokens;
    int32_t max_q_len;
    int32_t sm_count;
    int32_t use_prefill;
    int32_t use_cascade;
    int32_t use_merge;
    int32_t dec_ctas;
    int32_t pre_ctas;
    const int32_t* cu;
    const int32_t* seqlens;
    const int32_t* page_table;
    int64_t ld;
    const int64_t* slots;        // the caller's slot mapping or null
    const int32_t* tok_req;      // per-token request index in the workspace (slots null)
    uint8_t* ws;
    void* stream;
    void* events[5];           // optional timing events (attn_set_timing_events)
    int32_t n_events;
    int32_t kernels_per_forward;
    Layout lay;
};
static_assert(sizeof(MetaHost) <= sizeof(pva_meta), "MetaHost must fit in pva_meta");
constexpr uint64_t kMetaMagic = 0x5056414d45544131ull;  // "PVAMETA1"

// ---------------------------------------------------------------- host helpers

inline int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split a key range of `ext` keys into near-equal chunks of whole 16-key stages,
// about `chunk` keys each; returns the number of (non-empty) chunks and their length.
#ifdef __CUDACC__
__host__ __device__
#endif
inline int split_ranges(int ext, int chunk, int* per_out) {
    int s = (ext + chunk - 1) / chunk;
    if (s < 1) s = 1;
    int per = ((ext + s - 1) / s + kDecKeysPerStage - 1) / kDecKeysPerStage * kDecKeysPerStage;
    if (per < kDecKeysPerStage) per = kDecKeysPerStage;
    *per_out = per;
    return (ext + per - 1) / per;
}

// ---------------------------------------------------------------- GB300 tuning: prefix-pass size
//
// Rates of one GB300 SM measured in this library's kernels, used only to size the
// shared-prefix pass against the decode tails that run beside it (no result depends on
// them): the tensor-core kernel's prefix pass does ~6.9 TFLOP/s per SM (1/1.6 of that
// with FP8 pools, whose operands it converts), the decode kernel streams ~36 GB/s per SM.
// A (member, prefix key) pair costs 4 D Hq = 4 D G Hkv FLOPs and a tail key 2 Hkv D es
// bytes, so prefix time / tail time = pairs * G * 2 * 36 / (tail keys * es * 6900)
// (es = bytes per pool element), and the pass aims for that share of the SMs:
// units = casc_target * r / (1 + r), at least 1.  On the 128-member cascade batch (4096
// shared keys, tails U[16, 512], G 4; seed 0: 34 480 tail keys) this gives 36 units for
// bf16 and 76 for FP8 pools on 152 SMs, next to the best targets measured there (38 and
// 76); one unit per SM took 101 / 99 us against 86 / 87 us.
constexpr float kTuneTcGflopsPerSm = 6900.f;  // tensor-core prefix pass, bf16, per SM (GFLOP/s)
constexpr float kTuneFp8TcSlowdown = 1.6f;    // the same with FP8 pools is this much slower
constexpr float kTuneDecodeGbsPerSm = 36.f;   // decode streaming per SM (GB/s)

// Prefix-pass units to aim for: pair16 = (member, 16 prefix keys) pairs over all groups,
// tail_keys = keys of the decode tails, group = G; at most casc_target, at least 1.
#ifdef __CUDACC__
__host__ __device__
#endif
inline int prefix_pass_target(long long pair16, unsigned long long tail_keys, int group, int kv_fp8,
                              int casc_target) {
    if (tail_keys == 0) return casc_target;
    const float pre = (float)pair16 * 16.f * (float)group * 2.f * kTuneDecodeGbsPerSm *
                      (kv_fp8 ? kTuneFp8TcSlowdown : 1.f);
    const float tail = (float)tail_keys * (kv_fp8 ? 1.f : 2.f) * kTuneTcGflopsPerSm;
    const float r = pre / tail;
    const int t = (int)((float)casc_target * r / (1.f + r));
    return t < 1 ? 1 : (t > casc_target ? casc_target : t);
}

// Entries (log2) of the prepare kernel's shared-memory hash table for shared-prefix
// detection: more than twice the batch, so that open addressing always finds a free entry.
#ifdef __CUDACC__
__host__ __device__
#endif
inline int casc_hash_bits(int batch) {
    int b = 6;
    while ((1 << b) < 2 * (batch + 1)) ++b;
    return b;
}

// Launch with programmatic stream serialization: the kernel's CTAs may start while the
// previous kernel of the stream is still running (that kernel lets them with
// grid_dep_launch); the kernel reads nothing the previous one writes before its
// grid_dep_wait.  This hides the launch and set-up of the attention kernels behind the
// kernel before them.
template <class... Params, class... Args>
cudaError_t launch_programmatic(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                                cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Launchers (defined in the .cu files).
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t s);
size_t prepare_smem_bytes(int smem_batch, bool cascade);
cudaError_t launch_store(const ForwardParams& p, int head_dim, cudaStream_t s);
cudaError_t launch_decode(const ForwardParams& p, int head_dim, int ctas, cudaStream_t s);
cudaError_t launch_merge(const ForwardParams& p, int head_dim, int ctas, cudaStream_t s);
cudaError_t launch_prefill(const ForwardParams& p, int head_dim, int ctas, cudaStream_t s);
bool prefill_supported(int num_qo_heads, int num_kv_heads, int head_dim);
int decode_ctas_per_sm(int num_kv_heads, int head_dim);
bool decode_supported(int num_qo_heads, int num_kv_heads, int head_dim);

}  // namespace pva
