// The C ABI of libpva.so (declared in include/pva.h): argument checks that need
// no GPU, workspace planning, and kernel launches.  The host never reads device
// data here except in the two documented debug helpers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "pva_internal.h"

namespace pva {
namespace {

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

// Batches up to this size keep their per-request arrays in the prepare kernel's shared
// memory; shared-prefix detection needs them there, with its hash table beside them,
// which bounds it to smaller batches.
constexpr int kPrepareSmemBatch = 4096;
constexpr int kCascadeMaxBatch = 1536;

// Host-side validation of the static configuration.
pva_status check_config(const pva_config* c) {
    if (c == nullptr) return PVA_ERR_INVALID_ARG;
    if (c->num_qo_heads <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0 || c->page_size <= 0 ||
        c->num_pages <= 0 || c->max_batch <= 0 || c->max_tokens < 0 || c->max_kv_len < 0)
        return PVA_ERR_INVALID_ARG;
    if (c->num_qo_heads % c->num_kv_heads != 0) return PVA_ERR_INVALID_ARG;
    if (!is_pow2(c->page_size) || c->page_size > 128) return PVA_ERR_UNSUPPORTED;
    if (!decode_supported(c->num_qo_heads, c->num_kv_heads, c->head_dim)) return PVA_ERR_UNSUPPORTED;
    // the tensor-core kernel's gathers keep a slot in 32 bits (all ones marks a row not copied)
    if ((int64_t)c->num_pages * c->page_size >= ((int64_t)1 << 32)) return PVA_ERR_UNSUPPORTED;
    if (c->kv_dtype != PVA_KV_BF16 && c->kv_dtype != PVA_KV_E4M3) return PVA_ERR_UNSUPPORTED;
    return PVA_OK;
}

// target_units > 0 replaces the number of split-KV units the plan aims for (and with
// it the unit and partial-slot capacity); 0 keeps the default of four per decode CTA.
// The default leaves room for the balanced split too (it cuts the key line at most once
// per decode CTA: one more unit per cut, at most two partial slots per cut); with fewer
// units the prepare kernel plans the queue of split-KV chunks instead.
Layout make_layout(const pva_config* c, int sm_count, int target_units = 0) {
    Layout L{};
    const int G = c->num_qo_heads / c->num_kv_heads;
    const int TB = kDecRows / G;
    const int TM = kPreRows / G;
    const int cps = decode_ctas_per_sm(c->num_kv_heads, c->head_dim);
    L.dec_ctas = sm_count * cps;
    L.target_units = target_units > 0 ? target_units : 4 * L.dec_ctas;
    L.max_dec_groups = (int32_t)(c->max_tokens / TB + c->max_batch + 1);
    L.max_dec_units = L.max_dec_groups + L.target_units + 1;
    L.max_partial = 2 * L.target_units + 2;
    L.max_pre_tiles = (int32_t)((c->max_tokens / TM + c->max_batch + 1) * (int64_t)c->num_kv_heads);
    // up to kMaxCascLevels levels of groups, each at most one per two requests; the prepare kernel
    // numbers no more than max_batch + 1 records in all (a deeper level that would need
    // more is not formed: its requests read those keys as tails)
    L.max_casc_groups = c->enable_cascade ? c->max_batch + 1 : 1;
    // at most one prefix-pass unit per SM; the prepare kernel aims for fewer, weighing the
    // prefix pass against the decode tails that run beside it
    L.casc_target = sm_count;
    if (c->enable_cascade) {
        // every member of a group takes one partial slot per prefix chunk of each of its
        // groups (one a level), at most kMaxCascChunks in all (with n levels in a batch each
        // level takes at most 1/n of them); the prefix pass has at most (member tiles / 2 +
        // groups) x kv heads x chunks units per level
        L.max_partial += c->max_batch * kMaxCascChunks;
        L.max_pre_tiles += (int32_t)((2 * (c->max_batch / (2 * TM)) + L.max_casc_groups + 2) *
                                     (int64_t)c->num_kv_heads * kMaxCascChunks);
    }
    L.rows_per_slot = kDecRows * c->num_kv_heads;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.header = take(sizeof(PlanHeader));
    L.dec_units = take(sizeof(DecUnit) * (size_t)L.max_dec_units);
    L.dec_groups = take(sizeof(DecGroup) * (size_t)L.max_dec_groups);
    L.pre_tiles = take(sizeof(PreTile) * (size_t)L.max_pre_tiles);
    L.slots = take(sizeof(int64_t) * (size_t)(c->max_tokens + 1));
    L.partial_o = take(sizeof(float) * (size_t)L.max_partial * L.rows_per_slot * c->head_dim);
    L.partial_lse = take(sizeof(float) * (size_t)L.max_partial * L.rows_per_slot);
    L.req_scratch = take(sizeof(int32_t) * 4 * (size_t)(c->max_batch + 1));
    L.casc_groups = take(sizeof(CascGroup) * (size_t)L.max_casc_groups);
    L.casc_members = take(sizeof(int32_t) * 2 * kMaxCascLevels * (size_t)c->max_batch);  // (token, slot) per member per level
    L.casc_deep = take(sizeof(int32_t) * 3 * (kMaxCascLevels - 2) * (size_t)(c->max_batch + 1));
    L.dec_first = take(sizeof(int32_t) * ((size_t)L.dec_ctas + 1));
    L.total = off;
    return L;
}

const MetaHost* meta_of(const pva_meta* m) {
    if (m == nullptr) return nullptr;
    const MetaHost* h = reinterpret_cast<const MetaHost*>(m->opaque);
    return h->magic == kMetaMagic ? h : nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ForwardParams forward_params(const MetaHost* h, const void* q, const void* k, const void* v, void* k_pool,
                             void* v_pool, void* out, float* lse) {
    ForwardParams fp{};
    fp.q = static_cast<const uint16_t*>(q);
    fp.k = static_cast<const uint16_t*>(k);
    fp.v = static_cast<const uint16_t*>(v);
    fp.k_pool = static_cast<uint16_t*>(k_pool);
    fp.v_pool = static_cast<uint16_t*>(v_pool);
    fp.out = static_cast<uint16_t*>(out);
    fp.lse = lse;
    fp.cu = h->cu;
    fp.seqlens = h->seqlens;
    fp.page_table = h->page_table;
    fp.ld = h->ld;
    fp.slots = h->slots;
    fp.tok_req = h->tok_req;
    fp.total_tokens = h->total_tokens;
    fp.page_size = h->cfg.page_size;
    fp.page_shift = ilog2(h->cfg.page_size);
    fp.num_pages = h->cfg.num_pages;
    fp.num_slots = h->cfg.num_pages * (int64_t)h->cfg.page_size;
    fp.num_qo_heads = h->cfg.num_qo_heads;
    fp.num_kv_heads = h->cfg.num_kv_heads;
    fp.group = h->cfg.num_qo_heads / h->cfg.num_kv_heads;
    const float scale = h->cfg.sm_scale > 0.f ? h->cfg.sm_scale : 1.0f / std::sqrt((float)h->cfg.head_dim);
    fp.scale_log2 = scale * 1.4426950408889634f;
    fp.ws = h->ws;
    fp.lay = h->lay;
    return fp;
}

}  // namespace
}  // namespace pva

using namespace pva;

extern "C" {

int32_t attn_abi_version(void) { return PVA_ABI_VERSION; }

const char* attn_status_string(pva_status s) {
    switch (s) {
        case PVA_OK: return "PVA_OK";
        case PVA_ERR_INVALID_ARG: return "PVA_ERR_INVALID_ARG: null pointer, bad size or bad layout";
        case PVA_ERR_UNSUPPORTED: return "PVA_ERR_UNSUPPORTED: head_dim, group size or page_size not built";
        case PVA_ERR_WORKSPACE_TOO_SMALL: return "PVA_ERR_WORKSPACE_TOO_SMALL";
        case PVA_ERR_CUDA: return "PVA_ERR_CUDA: a CUDA runtime call failed";
        case PVA_ERR_DEVICE_CHECK: return "PVA_ERR_DEVICE_CHECK: the device error word is nonzero";
        case PVA_ERR_NOT_PREPARED: return "PVA_ERR_NOT_PREPARED: meta was not filled by attn_prepare_metadata";
    }
    return "unknown pva_status";
}

size_t attn_workspace_size(const pva_config* cfg) {
    if (check_config(cfg) != PVA_OK) return 0;
    const int sms = device_sm_count();
    if (sms <= 0) return 0;
    return make_layout(cfg, sms).total;
}

namespace {

// Scratch area of attn_prepare_metadata_static: a plan workspace that exists in every
// device's copy of this module, for callers that cannot allocate one.
static __device__ __align__(256) uint8_t g_static_workspace[PVA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
// Device address of g_static_workspace per device, with the CUDA context it was looked up
// in: a context created anew (after cudaDeviceReset) has its own copy of the module.
struct StaticArea {
    unsigned long long ctx_id;
    void* ptr;
};
StaticArea g_static_area[kMaxDevices];

// Identifier of the calling thread's current CUDA context (0 when it cannot be read; the
// address is then looked up on every call).  Through the driver's entry points, resolved
// once.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Host checks of attn_prepare_metadata's arguments other than the workspace.
pva_status check_prepare_args(const pva_config* cfg, const int32_t* cu_seqlens_q, const int32_t* cache_seqlens,
                              const int32_t* page_table, int64_t ld_page_table, int32_t batch, int32_t total_tokens,
                              pva_meta* meta) {
    pva_status st = check_config(cfg);
    if (st != PVA_OK) return st;
    if (meta == nullptr || cu_seqlens_q == nullptr) return PVA_ERR_INVALID_ARG;
    // an empty batch reads neither the lengths nor the page table
    if (batch > 0 && (cache_seqlens == nullptr || page_table == nullptr || ld_page_table <= 0))
        return PVA_ERR_INVALID_ARG;
    if (batch < 0 || total_tokens < 0 || (batch == 0 && total_tokens != 0)) return PVA_ERR_INVALID_ARG;
    if (batch > cfg->max_batch || total_tokens > cfg->max_tokens) return PVA_ERR_INVALID_ARG;
    return PVA_OK;
}

// The plan for one batch in `workspace` (carved up by `lay`); arguments already checked.
pva_status prepare_in_workspace(const pva_config* cfg, const int32_t* cu_seqlens_q, const int32_t* cache_seqlens,
                                const int32_t* page_table, int64_t ld_page_table, const int64_t* slot_mapping,
                                int32_t batch, int32_t total_tokens, int32_t max_q_len, void* workspace,
                                const Layout& lay, int sms, void* stream, pva_meta* meta) {
    const int G = cfg->num_qo_heads / cfg->num_kv_heads;
    const int TB = kDecRows / G;
    const int mq = max_q_len > 0 ? max_q_len : (total_tokens > 0 ? total_tokens : 1);

    MetaHost h{};
    h.magic = kMetaMagic;
    h.cfg = *cfg;
    if (h.cfg.min_cascade_pages <= 0) h.cfg.min_cascade_pages = 8;
    h.batch = batch;
    h.total_tokens = total_tokens;
    h.max_q_len = mq;
    h.sm_count = sms;
    // requests with more than TB new tokens run on the tensor-core prefill kernel, which
    // also runs the prefix pass of shared-prefix groups
    const bool tc_ok = prefill_supported(cfg->num_qo_heads, cfg->num_kv_heads, cfg->head_dim);
    h.use_prefill = (mq > TB && tc_ok) ? 1 : 0;
    h.use_cascade = (cfg->enable_cascade && tc_ok && batch >= 2 && batch <= kCascadeMaxBatch) ? 1 : 0;
    h.dec_ctas = lay.dec_ctas;  // sms x decode CTAs per SM; the plan's balanced split assumes it
    {
        const int64_t TM = kPreRows / G;
        const int64_t bound = ((int64_t)total_tokens / TM + batch + 1) * cfg->num_kv_heads;
        h.pre_ctas = h.use_prefill ? (int32_t)(bound < sms ? bound : sms) : 0;
        if (h.use_cascade) h.pre_ctas = sms;
    }
    h.cu = cu_seqlens_q;
    h.seqlens = cache_seqlens;
    h.page_table = page_table;
    h.ld = ld_page_table;
    h.ws = static_cast<uint8_t*>(workspace);
    h.slots = slot_mapping;
    h.tok_req = slot_mapping != nullptr ? nullptr : reinterpret_cast<const int32_t*>(h.ws + lay.slots);
    h.stream = stream;
    h.lay = lay;
    h.n_events = 0;
    // groups can have partial slots to combine only with split-KV or shared prefixes
    h.use_merge = (cfg->enable_split_kv || h.use_cascade) ? 1 : 0;
    // store, [prefill / prefix pass], decode, [combine]
    h.kernels_per_forward = 2 + ((h.use_prefill || h.use_cascade) ? 1 : 0) + h.use_merge;

    PrepareParams pp{};
    pp.cu = cu_seqlens_q;
    pp.seqlens = cache_seqlens;
    pp.page_table = page_table;
    pp.ld = ld_page_table;
    pp.user_slots = slot_mapping;
    pp.tok_req = slot_mapping != nullptr ? nullptr : reinterpret_cast<int32_t*>(h.ws + lay.slots);
    pp.batch = batch;
    pp.total_tokens = total_tokens;
    pp.max_q_len = mq;
    pp.page_size = cfg->page_size;
    pp.num_pages = cfg->num_pages;
    pp.num_qo_heads = cfg->num_qo_heads;
    pp.num_kv_heads = cfg->num_kv_heads;
    pp.group = G;
    pp.dec_tokens = kDecRows / G;
    pp.pre_tokens = kPreRows / G;
    pp.use_prefill = h.use_prefill;
    pp.use_cascade = h.use_cascade;
    pp.kv_fp8 = cfg->kv_dtype == PVA_KV_E4M3 ? 1 : 0;
    pp.min_cascade_pages = h.cfg.min_cascade_pages;
    pp.smem_batch = batch <= kPrepareSmemBatch ? batch : 0;
    pp.split_kv = cfg->enable_split_kv ? 1 : 0;
    pp.max_kv_len = cfg->max_kv_len;
    pp.max_tokens = cfg->max_tokens;
    pp.max_batch = cfg->max_batch;
    pp.ws = h.ws;
    pp.lay = lay;
    if (launch_prepare(pp, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PVA_ERR_CUDA;
    std::memset(meta, 0, sizeof(*meta));
    std::memcpy(meta->opaque, &h, sizeof(h));
    return PVA_OK;
}

}  // namespace

pva_status attn_prepare_metadata(const pva_config* cfg, const int32_t* cu_seqlens_q, const int32_t* cache_seqlens,
                                 const int32_t* page_table, int64_t ld_page_table, const int64_t* slot_mapping,
                                 int32_t batch, int32_t total_tokens, int32_t max_q_len, void* workspace,
                                 size_t workspace_bytes, void* stream, pva_meta* meta) {
    pva_status st = check_prepare_args(cfg, cu_seqlens_q, cache_seqlens, page_table, ld_page_table, batch,
                                       total_tokens, meta);
    if (st != PVA_OK) return st;
    if (workspace == nullptr) return PVA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PVA_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return PVA_ERR_CUDA;
    const Layout lay = make_layout(cfg, sms);
    if (workspace_bytes < lay.total) return PVA_ERR_WORKSPACE_TOO_SMALL;
    return prepare_in_workspace(cfg, cu_seqlens_q, cache_seqlens, page_table, ld_page_table, slot_mapping, batch,
                                total_tokens, max_q_len, workspace, lay, sms, stream, meta);
}

namespace pva {
namespace {

pva_status store_impl(const MetaHost* h, const void* k, const void* v, void* k_pool, void* v_pool,
                      const float* k_scale, const float* v_scale, void* stream) {
    if (h->total_tokens > 0 && (k == nullptr || v == nullptr)) return PVA_ERR_INVALID_ARG;
    if (k_pool == nullptr || v_pool == nullptr) return PVA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool)) return PVA_ERR_INVALID_ARG;
    ForwardParams fp = forward_params(h, nullptr, k, v, k_pool, v_pool, nullptr, nullptr);
    fp.kv_fp8 = h->cfg.kv_dtype == PVA_KV_E4M3 ? 1 : 0;
    fp.k_scale = k_scale;
    fp.v_scale = v_scale;
    if (launch_store(fp, h->cfg.head_dim, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PVA_ERR_CUDA;
    return PVA_OK;
}

}  // namespace
}  // namespace pva

pva_status attn_store_kvcache(const pva_meta* meta, const void* k, const void* v, void* k_pool, void* v_pool,
                              void* stream) {
    const MetaHost* h = meta_of(meta);
    if (h == nullptr) return PVA_ERR_NOT_PREPARED;
    if (h->cfg.kv_dtype != PVA_KV_BF16) return PVA_ERR_INVALID_ARG;
    return store_impl(h, k, v, k_pool, v_pool, nullptr, nullptr, stream);
}

pva_status attn_store_kvcache_fp8kv(const pva_meta* meta, const void* k, const void* v, void* k_pool,
                                    void* v_pool, const float* k_scale, const float* v_scale, void* stream) {
    const MetaHost* h = meta_of(meta);
    if (h == nullptr) return PVA_ERR_NOT_PREPARED;
    if (h->cfg.kv_dtype != PVA_KV_E4M3 || k_scale == nullptr || v_scale == nullptr) return PVA_ERR_INVALID_ARG;
    return store_impl(h, k, v, k_pool, v_pool, k_scale, v_scale, stream);
}

pva_status attn_prepare_metadata_static(const pva_config* cfg, const int32_t* cu_seqlens_q,
                                        const int32_t* cache_seqlens, const int32_t* page_table,
                                        int64_t ld_page_table, const int64_t* slot_mapping, int32_t batch,
                                        int32_t total_tokens, int32_t max_q_len, void* stream, pva_meta* meta) {
    pva_status st = check_prepare_args(cfg, cu_seqlens_q, cache_seqlens, page_table, ld_page_table, batch,
                                       total_tokens, meta);
    if (st != PVA_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PVA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PVA_ERR_UNSUPPORTED;
    void* ws = nullptr;
    {
        // host code only knows the array by a host-side stand-in: its device address comes
        // from the runtime, once per device and context (with that device current)
        std::lock_guard<std::mutex> lock(g_static_mu);
        const unsigned long long ctx = current_context_id();
        StaticArea& a = g_static_area[dev];
        if (a.ptr == nullptr || ctx == 0 || a.ctx_id != ctx) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return PVA_ERR_CUDA;
            a.ptr = p;
            a.ctx_id = ctx;
        }
        ws = a.ptr;
    }
    const int sms = device_sm_count();
    if (sms <= 0) return PVA_ERR_CUDA;
    // the default plan, or one aiming for fewer split-KV units when that does not fit
    // (below one unit per decode CTA the prepare kernel plans the unit queue, whose
    // capacity follows the target, instead of the balanced split)
    Layout lay = make_layout(cfg, sms);
    for (int t = lay.target_units; lay.total > PVA_STATIC_WORKSPACE_BYTES && t > sms;) {
        t = t / 2 > sms ? t / 2 : sms;
        lay = make_layout(cfg, sms, t);
    }
    if (lay.total > PVA_STATIC_WORKSPACE_BYTES) return PVA_ERR_WORKSPACE_TOO_SMALL;
    return prepare_in_workspace(cfg, cu_seqlens_q, cache_seqlens, page_table, ld_page_table, slot_mapping, batch,
                                total_tokens, max_q_len, ws, lay, sms, stream, meta);
}

namespace pva {
namespace {

pva_status forward_impl(const MetaHost* h, const void* q, const void* k, const void* v, void* k_pool, void* v_pool,
                        const float* k_scale, const float* v_scale, void* out, float* lse, void* stream) {
    if (h->total_tokens > 0 && (q == nullptr || k == nullptr || v == nullptr || out == nullptr))
        return PVA_ERR_INVALID_ARG;
    if (k_pool == nullptr || v_pool == nullptr) return PVA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(k_pool) ||
        !aligned16(v_pool) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return PVA_ERR_INVALID_ARG;
    if (h->total_tokens == 0) return PVA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ForwardParams fp = forward_params(h, q, k, v, k_pool, v_pool, out, lse);
    fp.kv_fp8 = h->cfg.kv_dtype == PVA_KV_E4M3 ? 1 : 0;
    fp.k_scale = k_scale;
    fp.v_scale = v_scale;
    fp.dec_wait_late = (h->use_prefill || h->use_cascade) ? 1 : 0;
    // inside a stream capture the events become graph nodes that still time the replay
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (h->n_events == 5 && cudaStreamIsCapturing(s, &capture) != cudaSuccess) return PVA_ERR_CUDA;
    auto mark = [&](int i) {
        if (h->n_events != 5) return cudaSuccess;
        cudaEvent_t ev = static_cast<cudaEvent_t>(h->events[i]);
        return capture == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                                        : cudaEventRecord(ev, s);
    };
    if (mark(0) != cudaSuccess) return PVA_ERR_CUDA;
    if (launch_store(fp, h->cfg.head_dim, s) != cudaSuccess) return PVA_ERR_CUDA;
    if (mark(1) != cudaSuccess) return PVA_ERR_CUDA;
    if ((h->use_prefill || h->use_cascade) && launch_prefill(fp, h->cfg.head_dim, h->pre_ctas, s) != cudaSuccess)
        return PVA_ERR_CUDA;
    if (mark(2) != cudaSuccess) return PVA_ERR_CUDA;
    if (launch_decode(fp, h->cfg.head_dim, h->dec_ctas, s) != cudaSuccess) return PVA_ERR_CUDA;
    if (mark(3) != cudaSuccess) return PVA_ERR_CUDA;
    if (h->use_merge && launch_merge(fp, h->cfg.head_dim, h->sm_count, s) != cudaSuccess) return PVA_ERR_CUDA;
    if (mark(4) != cudaSuccess) return PVA_ERR_CUDA;
    return PVA_OK;
}

}  // namespace
}  // namespace pva

pva_status attn_forward(const pva_meta* meta, const void* q, const void* k, const void* v, void* k_pool,
                        void* v_pool, void* out, float* lse, void* stream) {
    const MetaHost* h = meta_of(meta);
    if (h == nullptr) return PVA_ERR_NOT_PREPARED;
    if (h->cfg.kv_dtype != PVA_KV_BF16) return PVA_ERR_INVALID_ARG;
    return forward_impl(h, q, k, v, k_pool, v_pool, nullptr, nullptr, out, lse, stream);
}

pva_status attn_forward_fp8kv(const pva_meta* meta, const void* q, const void* k, const void* v, void* k_pool,
                              void* v_pool, const float* k_scale, const float* v_scale, void* out, float* lse,
                              void* stream) {
    const MetaHost* h = meta_of(meta);
    if (h == nullptr) return PVA_ERR_NOT_PREPARED;
    if (h->cfg.kv_dtype != PVA_KV_E4M3 || k_scale == nullptr || v_scale == nullptr) return PVA_ERR_INVALID_ARG;
    return forward_impl(h, q, k, v, k_pool, v_pool, k_scale, v_scale, out, lse, stream);
}

pva_status attn_get_device_status(const pva_meta* meta, uint32_t* error_bits) {
    const MetaHost* h = meta_of(meta);
    if (h == nullptr) return PVA_ERR_NOT_PREPARED;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(h->stream)) != cudaSuccess) return PVA_ERR_CUDA;
    PlanHeader hdr{};
    if (cudaMemcpy(&hdr, h->ws + h->lay.header, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PVA_ERR_CUDA;
    if (error_bits) *error_bits = hdr.error_bits;
    return hdr.error_bits ? PVA_ERR_DEVICE_CHECK : PVA_OK;
}

pva_status attn_set_timing_events(pva_meta* meta, void* const* events, int32_t n) {
    if (meta == nullptr) return PVA_ERR_NOT_PREPARED;
    MetaHost* h = reinterpret_cast<MetaHost*>(meta->opaque);
    if (h->magic != kMetaMagic) return PVA_ERR_NOT_PREPARED;
    if (n != 0 && n != 5) return PVA_ERR_INVALID_ARG;
    if (n == 5 && events == nullptr) return PVA_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i) {
        if (n == 5 && events[i] == nullptr) return PVA_ERR_INVALID_ARG;
        h->events[i] = n == 5 ? events[i] : nullptr;
    }
    h->n_events = n;
    return PVA_OK;
}

pva_status attn_debug_set_wait_limit(const pva_meta* meta, int64_t limit_ns) {
    const MetaHost* h = meta_of(meta);
    if (h == nullptr) return PVA_ERR_NOT_PREPARED;
    // the header holds limit + 1 (0: the default); limits above ~4.29 s are capped
    uint32_t v = 0;
    if (limit_ns >= 0) v = (uint32_t)((limit_ns < 0xFFFFFFFEll ? limit_ns : 0xFFFFFFFEll) + 1);
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(h->stream)) != cudaSuccess) return PVA_ERR_CUDA;
    if (cudaMemcpy(h->ws + h->lay.header + offsetof(PlanHeader, wait_override), &v, sizeof(v),
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return PVA_ERR_CUDA;
    return PVA_OK;
}

int32_t attn_debug_plan_counts(const pva_meta* meta, int64_t* counts, int32_t n) {
    const MetaHost* h = meta_of(meta);
    if (h == nullptr || counts == nullptr || n <= 0) return 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(h->stream)) != cudaSuccess) return 0;
    PlanHeader hdr{};
    if (cudaMemcpy(&hdr, h->ws + h->lay.header, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess) return 0;
    const int64_t vals[9] = {hdr.n_dec_units, hdr.n_dec_groups,     hdr.n_pre_tiles,        hdr.n_casc_groups,
                             hdr.n_casc_tiles, hdr.split_chunk,      hdr.n_partial_slots,    h->kernels_per_forward,
                             hdr.n_casc_levels};
    const int m = n < 9 ? n : 9;
    for (int i = 0; i < m; ++i) counts[i] = vals[i];
    return m;
}

}  // extern "C"
