/*
 * pva.h -- C ABI of libpva.so: the paged variable-length attention forward
 * of an LLM serving engine, for NVIDIA GB300 (sm_103a).
 *
 * The operation (one flat, mixed batch of prefill, chunked-prefill and decode
 * requests; all requests' new tokens packed end to end without padding):
 *
 *   once per batch   attn_prepare_metadata(...)  -> pva_meta
 *   once per layer   attn_forward(q, k, v, k_pool, v_pool, out, lse, meta)
 *                      = store this step's K/V into the paged pool, then
 *                        causal, bottom-right-aligned GQA attention of every
 *                        request over its cached prefix plus its new tokens.
 *
 * Where each piece is defined:
 *   - "The attention backend and a reference implementation" (mini-sglang
 *     from Scratch, ch. 5), section "The interface": prepare_metadata once
 *     per batch (the metadata is the same for every layer), forward once per
 *     layer, write-before-read.
 *   - same page, section "Variable-length, paged attention with prefixes":
 *     cu_seqlens_q, cache_seqlens (KV length INCLUDING this step's tokens),
 *     the page table, and the bottom-right causal mask (query r of n sits at
 *     absolute position kv_len - n + r and sees keys j <= kv_len - n + r).
 *   - "Attention backends: backend, metadata builder and implementation"
 *     (explain vLLM), step 2: the implementation writes into a caller-given
 *     output, and the KV update is a scatter by slot (slot_mapping).
 *   - "Source walkthrough: Attention backends" (SGLang learning notes),
 *     sections 3.1 and 7: plan once into a preallocated workspace, run per
 *     layer; section 3.3: shared-prefix (cascade) attention merged by
 *     log-sum-exp.
 *   - "Variable-length batching and one mixed forward pass", sections
 *     "Layout and metadata" and "Exercises" (answer 2): prefill, chunked
 *     prefill and decode differ only in (cached, new) lengths; long decodes
 *     are split over the KV sequence and combined (split-KV).
 *
 * Conventions (all calls):
 *   - Every pointer to batch data or pools is a DEVICE pointer on the current
 *     CUDA device unless stated otherwise; the caller owns all memory.  The
 *     library allocates no device memory and never synchronises a stream
 *     (except attn_get_device_status, which is documented as syncing).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - bf16 tensors are row-major and contiguous:
 *       q   [total_tokens, num_qo_heads, head_dim]
 *       k,v [total_tokens, num_kv_heads, head_dim]   (this step's new tokens)
 *       k_pool, v_pool [num_pages * page_size, num_kv_heads, head_dim]
 *       out [total_tokens, num_qo_heads, head_dim]
 *     lse is fp32 [total_tokens, num_qo_heads] (natural log of the sum of
 *     exp of the scaled scores), or NULL.
 *   - Index tensors are int32 except slot_mapping (int64).
 *   - q head h reads kv head h / (num_qo_heads / num_kv_heads).
 *   - Pool slot of position j of request i:
 *       page_table[i * ld_page_table + j / page_size] * page_size + j % page_size.
 *     Page-table columns past ceil(kv_len / page_size) are never read.
 *   - Errors the host can see (null pointers, unsupported shapes, workspace
 *     too small) return a status and launch nothing.  Errors that depend on
 *     device data (non-monotone cu_seqlens_q, q_len > kv_len, page ids or
 *     slots outside the pool, a batch larger than the planned limits) set
 *     bits of a device error word in the workspace; the kernels then skip
 *     the offending work and never trap.  attn_get_device_status reads it.
 */
#ifndef PVA_H
#define PVA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PVA_ABI_VERSION 2

#if defined(__GNUC__)
#define PVA_API __attribute__((visibility("default")))
#else
#define PVA_API
#endif

typedef enum pva_status {
    PVA_OK = 0,
    PVA_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad layout */
    PVA_ERR_UNSUPPORTED = 2,          /* head_dim, group size or page_size outside the built set */
    PVA_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < attn_workspace_size(cfg) */
    PVA_ERR_CUDA = 4,                 /* a CUDA runtime call failed (launch, attribute, ...) */
    PVA_ERR_DEVICE_CHECK = 5,         /* attn_get_device_status found device error bits set */
    PVA_ERR_NOT_PREPARED = 6          /* meta was not filled by attn_prepare_metadata */
} pva_status;

/* Bits of the device error word (attn_get_device_status). */
#define PVA_DEVERR_CU_SEQLENS 0x01u  /* cu_seqlens_q[0] != 0, decreasing, or cu[batch] != total_tokens */
#define PVA_DEVERR_Q_GT_KV    0x02u  /* some request has q_len > kv_len (or kv_len < 0) */
#define PVA_DEVERR_PAGE_ID    0x04u  /* a page id read for a position < kv_len lies outside [0, num_pages) */
#define PVA_DEVERR_SLOT       0x08u  /* a slot_mapping entry lies outside [-1, num_pages * page_size) */
#define PVA_DEVERR_LIMITS     0x10u  /* batch exceeds cfg.max_batch / max_tokens / max_kv_len or the max_q_len hint */
#define PVA_DEVERR_TIMEOUT    0x20u  /* a bounded wait inside a kernel gave up (internal error) */

/*
 * Element type of the paged KV pool (pva_config.kv_dtype).  The pages name the
 * pool's dtype as a backend choice ("Attention backends: backend, metadata builder
 * and implementation", the kv_cache_dtype of the backend interface) without fixing
 * a format; the 8-bit one here is E4M3 of the OCP 8-bit floating-point
 * specification (bias 7, 3 mantissa bits, no infinities, largest finite 448) with
 * one fp32 scale per kv head for K and one for V.
 */
#define PVA_KV_BF16 0
#define PVA_KV_E4M3 1

/*
 * Static description of the model's attention layer and of the largest batch
 * the workspace is planned for.  Plain data; the caller fills every field.
 */
typedef struct pva_config {
    int32_t num_qo_heads;       /* Hq */
    int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0 and Hq / Hkv <= 16 */
    int32_t head_dim;           /* D: 64 or 128 */
    int32_t page_size;          /* 1, 2, 4, ..., 128 (a power of two) */
    int64_t num_pages;          /* pool capacity in pages; num_pages * page_size < 2^32 */
    float sm_scale;             /* softmax scale; <= 0 selects 1/sqrt(head_dim) */
    int32_t max_batch;          /* upper bound on requests per batch */
    int32_t max_tokens;         /* upper bound on new tokens per batch */
    int32_t max_kv_len;         /* upper bound on any request's kv_len */
    int32_t enable_split_kv;    /* nonzero: split long KV ranges over several CTAs (LSE combine) */
    int32_t enable_cascade;     /* nonzero: read prefixes shared by several decodes once */
    int32_t min_cascade_pages;  /* shortest shared prefix (in pages) worth a cascade pass; <= 0 -> 8 */
    int32_t kv_dtype;           /* PVA_KV_BF16 (0) or PVA_KV_E4M3: the pool element type */
} pva_config;

/*
 * The prepared batch.  Host-side, caller-owned, filled by
 * attn_prepare_metadata; it refers to device memory inside the workspace and
 * stays valid until the next attn_prepare_metadata on the same workspace.
 * Treat it as opaque.
 */
typedef struct pva_meta {
    uint64_t opaque[64];
} pva_meta;

/* Version of this header the library was built from (PVA_ABI_VERSION). */
PVA_API int32_t attn_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
PVA_API const char* attn_status_string(pva_status status);

/*
 * Device bytes the workspace must hold for batches within cfg's limits on the
 * current device (the plan is sized by its SM count).  Returns 0 when cfg is
 * invalid or unsupported.  Host-only: makes no CUDA call other than a device
 * attribute query.
 */
PVA_API size_t attn_workspace_size(const pva_config* cfg);

/*
 * Once per batch: validate the batch on the device and build the plan inside
 * `workspace` -- the slot mapping (derived when slot_mapping is NULL), the
 * classification of each request (decode rows vs. prefill tiles), the
 * per-tile work list with causal KV extents, the split-KV plan and the
 * shared-prefix (cascade) groups.  One kernel launch on `stream`, no sync.
 * Shared prefixes are found among single-token decodes whose page-table rows start
 * with the same run of at least min_cascade_pages pages lying before their query, and
 * inside such a group among members whose rows continue with a further such run, and
 * so on inside those (up to eight levels of the prefix tree; runs below the eighth are
 * read as part of each member's own keys); each shared run is read once per group by
 * the forward.
 * Detection runs for batches of 2 to 1536 requests.
 *
 *   cu_seqlens_q   int32 [batch+1]  request i's new tokens are q[cu[i] : cu[i+1]]
 *   cache_seqlens  int32 [batch]    kv_len of request i, including its new tokens
 *   page_table     int32 [batch, ld_page_table]  page ids, row i = request i
 *   slot_mapping   int64 [total_tokens] pool slot of each new token, -1 = do not
 *                  store; or NULL to derive it from the page table (the new
 *                  tokens are positions kv_len - q_len .. kv_len - 1)
 *   batch, total_tokens   host values; total_tokens must equal cu[batch].  With
 *                  batch 0, cache_seqlens and page_table are not read and may be
 *                  NULL (ld_page_table is then ignored)
 *   max_q_len      host upper bound on any request's q_len (<= 0: unknown,
 *                  taken as total_tokens); lets the forward skip the prefill
 *                  kernel for decode-only batches.  A request above it sets
 *                  PVA_DEVERR_LIMITS and is skipped.
 *   workspace      device buffer of at least attn_workspace_size(cfg) bytes,
 *                  256-byte aligned, owned by the caller, not used
 *                  concurrently by another prepare/forward.
 * The arrays must stay unchanged until the last attn_forward using `meta`
 * (the forward kernels read them: the page table, the lengths, and slot_mapping
 * or, without one, the derived slots through the page table).  A page id of a
 * derived slot outside the pool is flagged (PVA_DEVERR_PAGE_ID) by the forward.
 */
PVA_API pva_status attn_prepare_metadata(const pva_config* cfg, const int32_t* cu_seqlens_q,
                                 const int32_t* cache_seqlens, const int32_t* page_table,
                                 int64_t ld_page_table, const int64_t* slot_mapping, int32_t batch,
                                 int32_t total_tokens, int32_t max_q_len, void* workspace,
                                 size_t workspace_bytes, void* stream, pva_meta* meta);

/* Bytes of the scratch area built into the library for attn_prepare_metadata_static. */
#define PVA_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)

/*
 * attn_prepare_metadata without a caller workspace: the plan is built in a
 * fixed scratch area of PVA_STATIC_WORKSPACE_BYTES compiled into this
 * library (one per device), so the call allocates no device memory at all.
 * It is meant for callers that cannot hand the library a device buffer: a
 * host program whose device memory belongs to an allocator it may not call on
 * this path, or a plugin inside a framework that exposes no allocation hook.
 * None of the pages this library follows describes such a call; it is an
 * addition for those callers.
 *
 * Arguments and results are those of attn_prepare_metadata minus workspace /
 * workspace_bytes; the returned meta is used with attn_forward as usual.
 * Limits and behaviour:
 *   - The first call on a device looks up that device's copy of the scratch
 *     area (with that device current), and so does the first call after the
 *     device's context was created anew (cudaDeviceReset); make that first call
 *     before any stream capture on the device.
 *   - When the plan for cfg does not fit, the number of split-KV units is
 *     lowered (down to one per SM) until it does; when it still does not fit,
 *     the call returns PVA_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 *     attn_workspace_size(cfg) above PVA_STATIC_WORKSPACE_BYTES is the sign
 *     that this can happen.
 *   - Nothing in the scratch area has to start at zero: every plan record is
 *     written by the prepare kernel before the forward reads it, and the work
 *     counters are reset by each forward's first kernel.
 *   - There is one scratch area per device, shared by every caller in the
 *     process: a prepare or forward using it that overlaps another one on the
 *     same device (another stream, another thread) races with it, and each
 *     call invalidates the meta of the previous one on that device.
 */
PVA_API pva_status attn_prepare_metadata_static(const pva_config* cfg, const int32_t* cu_seqlens_q,
                                        const int32_t* cache_seqlens, const int32_t* page_table,
                                        int64_t ld_page_table, const int64_t* slot_mapping, int32_t batch,
                                        int32_t total_tokens, int32_t max_q_len, void* stream, pva_meta* meta);

/*
 * Once per layer: store_kvcache, then attention, in stream order on `stream`.
 * k_pool / v_pool are updated in place (bit-exact copies of k / v rows at
 * their slots) and then read; out (and lse when not NULL) are fully written
 * for every new token.  Requests with q_len == 0 write nothing.  q, k, v, out
 * must be 16-byte aligned.  Several forwards may reuse one meta (one per
 * layer); they must not run concurrently on the same workspace.
 */
PVA_API pva_status attn_forward(const pva_meta* meta, const void* q, const void* k, const void* v,
                        void* k_pool, void* v_pool, void* out, float* lse, void* stream);

/*
 * store_kvcache alone: k_pool[slot[t], h, :] = k[t, h, :] and the same for v,
 * for every new token t with slot != -1.  attn_forward already includes it.
 */
PVA_API pva_status attn_store_kvcache(const pva_meta* meta, const void* k, const void* v, void* k_pool,
                              void* v_pool, void* stream);

/*
 * attn_forward for a pool of E4M3 bytes (the meta must come from a config with
 * kv_dtype = PVA_KV_E4M3; attn_forward refuses such a meta and this call refuses a
 * bf16 one, with PVA_ERR_INVALID_ARG).
 *   k_pool, v_pool  uint8 [num_pages * page_size, Hkv, D], updated in place, 16-byte aligned
 *   k_scale, v_scale  DEVICE fp32 [Hkv], the scale of each kv head
 *   q, k, v, out, lse as for attn_forward (bf16 activations)
 * The store writes e4m3(k[t, h, d] / k_scale[h]) (IEEE fp32 division, round to
 * nearest even, magnitudes beyond 448 saturate to 448, NaN stays NaN), likewise for
 * v; attention reads each element as e4m3 * scale of its head, otherwise exactly as
 * attn_forward (same kernels and plan: the tensor cores and the warp MMAs then take
 * f16 operands, every E4M3 value being an f16 value).  q enters as f16, exact for
 * 2^-17 <= |q| <= 65504; q outside f16's range gives undefined results.  Scales must
 * be finite and nonzero.
 */
PVA_API pva_status attn_forward_fp8kv(const pva_meta* meta, const void* q, const void* k, const void* v,
                              void* k_pool, void* v_pool, const float* k_scale, const float* v_scale,
                              void* out, float* lse, void* stream);

/* store_kvcache alone into an E4M3 pool (the quantisation of attn_forward_fp8kv). */
PVA_API pva_status attn_store_kvcache_fp8kv(const pva_meta* meta, const void* k, const void* v, void* k_pool,
                                    void* v_pool, const float* k_scale, const float* v_scale, void* stream);

/*
 * Debug/test helper: synchronises the stream of the last prepare/forward on
 * meta's workspace, then reads the device error word into *error_bits
 * (PVA_DEVERR_*).  Returns PVA_ERR_DEVICE_CHECK when any bit is set.
 */
PVA_API pva_status attn_get_device_status(const pva_meta* meta, uint32_t* error_bits);

/*
 * Profiling helper: with n > 0, every later attn_forward on this meta records
 * caller-created events (cudaEvent_t passed as void*) on its stream:
 * events[0] before its first kernel, then one after each phase --
 * [1] store_kvcache, [2] tensor-core pass (prefill tiles and the
 * shared-prefix pass), [3] decode / split-KV units, [4] LSE combine of the
 * split groups.  A phase that launches nothing records at the same point as
 * the previous one; recording the events also keeps the kernels from
 * overlapping their launch with the kernel before them.  n must be 0 (off)
 * or 5; the handles must outlive the forwards.  Timing only; it changes no
 * result.
 */
PVA_API pva_status attn_set_timing_events(pva_meta* meta, void* const* events, int32_t n);

/*
 * Test helper for the kernels' bounded waits: every wait inside the forward kernels
 * (on a pipeline stage, the tensor core, the work queue) gives up after 2 s, sets
 * PVA_DEVERR_TIMEOUT, waits (with the 2 s limit) for its CTA's own copies and MMAs,
 * frees what it holds and returns, so a wedged kernel ends with a status instead of
 * hanging the device.  This call shortens that limit for the forwards that use meta,
 * so a test can make the waits run out on a healthy batch: limit_ns >= 0 is the new
 * limit in ns (0: a wait gives up at once if its condition does not already hold);
 * limit_ns < 0 restores the default.  The waits that drain a CTA's copies and MMAs
 * before it leaves keep the default.  The next attn_prepare_metadata on the workspace
 * also restores it, and clears the error word.  Synchronises the meta's stream, then
 * writes the plan header; not for use inside a stream capture.
 */
PVA_API pva_status attn_debug_set_wait_limit(const pva_meta* meta, int64_t limit_ns);

/*
 * Debug/test helper: copies plan counters to host (synchronising): counts[0]
 * decode units, [1] decode merge groups, [2] prefill tiles, [3] cascade
 * groups, [4] cascade prefix tiles, [5] split-KV chunk (keys), [6] partial
 * slots used, [7] kernels one attn_forward launches, [8] levels of the shared-prefix
 * tree found (0: none).  Returns the number of entries written (<= n).
 */
PVA_API int32_t attn_debug_plan_counts(const pva_meta* meta, int64_t* counts, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* PVA_H */
