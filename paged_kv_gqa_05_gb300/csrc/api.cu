// C ABI of the library: argument checks, the plan (split heuristic + work list
// upload into persistent device buffers), TMA descriptor set-up and launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"

namespace pgqa {
using DecodeLauncher = cudaError_t (*)(int, int, int, const CUtensorMap &, const CUtensorMap &,
                                        const DecodeParams &, int, bool, cudaStream_t);
cudaError_t launch_decode_bf16_d64(int, int, int, const CUtensorMap &, const CUtensorMap &, const DecodeParams &, int, bool, cudaStream_t);
cudaError_t launch_decode_bf16_d128(int, int, int, const CUtensorMap &, const CUtensorMap &, const DecodeParams &, int, bool, cudaStream_t);
cudaError_t launch_decode_fp16_d64(int, int, int, const CUtensorMap &, const CUtensorMap &, const DecodeParams &, int, bool, cudaStream_t);
cudaError_t launch_decode_fp16_d128(int, int, int, const CUtensorMap &, const CUtensorMap &, const DecodeParams &, int, bool, cudaStream_t);

cudaError_t launch_decode(int kind, int stages, int head_dim, int group, pgqa_dtype dtype, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, const DecodeParams &p, int num_items, bool pdl,
                          cudaStream_t stream) {
    DecodeLauncher f = dtype == PGQA_BF16 ? (head_dim == 64 ? launch_decode_bf16_d64 : launch_decode_bf16_d128)
                                          : (head_dim == 64 ? launch_decode_fp16_d64 : launch_decode_fp16_d128);
    return f(kind, stages, group, tm_k, tm_v, p, num_items, pdl, stream);
}
cudaError_t decode_blocks_per_sm_bf16_d64(int, int, int *);
cudaError_t decode_blocks_per_sm_bf16_d128(int, int, int *);
cudaError_t decode_blocks_per_sm_fp16_d64(int, int, int *);
cudaError_t decode_blocks_per_sm_fp16_d128(int, int, int *);

// Resident CTAs per SM of the per-item tensor-core decode kernel for (stages, group).
cudaError_t decode_blocks_per_sm(int stages, int head_dim, int group, pgqa_dtype dtype, int *blocks) {
    auto f = dtype == PGQA_BF16 ? (head_dim == 64 ? decode_blocks_per_sm_bf16_d64 : decode_blocks_per_sm_bf16_d128)
                                : (head_dim == 64 ? decode_blocks_per_sm_fp16_d64 : decode_blocks_per_sm_fp16_d128);
    return f(stages, group, blocks);
}
using PrefillLauncher = cudaError_t (*)(int, int, const CUtensorMap &, const CUtensorMap &, const PrefillParams &,
                                         int, bool, cudaStream_t);
cudaError_t launch_prefill_bf16_d64(int, int, const CUtensorMap &, const CUtensorMap &, const PrefillParams &, int, bool, cudaStream_t);
cudaError_t launch_prefill_bf16_d128(int, int, const CUtensorMap &, const CUtensorMap &, const PrefillParams &, int, bool, cudaStream_t);
cudaError_t launch_prefill_fp16_d64(int, int, const CUtensorMap &, const CUtensorMap &, const PrefillParams &, int, bool, cudaStream_t);
cudaError_t launch_prefill_fp16_d128(int, int, const CUtensorMap &, const CUtensorMap &, const PrefillParams &, int, bool, cudaStream_t);

cudaError_t launch_prefill(int kind, int head_dim, int group, pgqa_dtype dtype, const CUtensorMap &tm_k,
                           const CUtensorMap &tm_v, const PrefillParams &p, int num_items, bool pdl,
                           cudaStream_t stream) {
    PrefillLauncher f = dtype == PGQA_BF16 ? (head_dim == 64 ? launch_prefill_bf16_d64 : launch_prefill_bf16_d128)
                                           : (head_dim == 64 ? launch_prefill_fp16_d64 : launch_prefill_fp16_d128);
    return f(kind, group, tm_k, tm_v, p, num_items, pdl, stream);
}
}  // namespace pgqa

using namespace pgqa;

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
static thread_local char g_last_error[512] = "";

static pgqa_status fail(pgqa_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

static pgqa_status cuda_fail(cudaError_t e, const char *what) {
    return fail(PGQA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------
// per-device flag word
// ---------------------------------------------------------------------------
static __device__ unsigned int g_device_flags;

static pgqa_status device_flags(unsigned int **out) {
    static std::mutex mu;
    static unsigned int *ptrs[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 256) return fail(PGQA_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_flags);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(flags)");
        ptrs[dev] = static_cast<unsigned int *>(p);
    }
    *out = ptrs[dev];
    return PGQA_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The pool [num_pages, page_size, Hkv, D] as the 3-D tensor {D, Hkv, rows};
// one box is `box_rows` consecutive rows of one kv head.
static pgqa_status make_pool_map(CUtensorMap *map, const void *pool, int64_t num_pages, int page_size,
                                 int num_kv_heads, int head_dim, pgqa_dtype dt, int box_rows, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return fail(PGQA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_kv_heads),
                                static_cast<cuuint64_t>(num_pages) * page_size};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                   static_cast<cuuint64_t>(num_kv_heads) * head_dim * 2};
    // The tensor-core kernel takes 64-channel (128-byte) boxes with 128-byte swizzle; the
    // CUDA-core kernel takes whole rows unswizzled.
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(swizzle128 ? 64 : head_dim), 1u,
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, dt == PGQA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PGQA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return PGQA_OK;
}

// ---------------------------------------------------------------------------
// helpers
// ---------------------------------------------------------------------------
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool supported_page_size(int ps) {
    return ps == 16 || ps == 32 || ps == 64 || ps == 128 || ps == 256;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------
struct MapCacheEntry {
    const void *ptr = nullptr;
    int64_t num_pages = 0;
    int box_rows = 0;
    bool swizzle128 = false;
    CUtensorMap map;
};

struct pgqa_plan {
    pgqa_plan_config cfg{};
    int device = 0;
    int num_sms = 0;
    int group = 0;
    int tile = 0;       // decode warp tile (tokens)
    int box_rows = 0;
    int ctas_per_sm = 0;     // CTA slots per SM for 2-stage plans (the most of any variant)
    int slots_per_sm[4] = {0, 0, 0, 0};  // by pipeline depth (1 = the wide form, 2 or 3): resident decode
                                         // CTAs per SM
    int kernel = PGQA_DECODE_TENSOR_CORE;
    int prefill_kind = PGQA_PREFILL_TCGEN05;  // prefill-segment kernel
    int prefill_pairs = 128;                  // (row, head) pairs per prefill tile of that kernel
    int stages = 2;     // per-warp pipeline depth of the tensor-core kernel (chosen per plan_update)
    int max_items = 0;  // capacity of the work list and of the partial slots
    int max_tasks = 0;
    int max_prefill = 0;     // capacity of the prefill-tile list
    int max_slots = 0;       // capacity of the split partials (slots of G x head_dim floats)
    float2 *rope_cs = nullptr;  // rotary (cos, sin) table [rope_max_position][head_dim / 2], or null

    void *d_meta = nullptr;  // [max_items] WorkItem, [max_tasks] MergeTask, [max_prefill] PrefillItem
    float *d_partial_o = nullptr;
    float *d_partial_lse = nullptr;
    void *h_meta[2] = {nullptr, nullptr};
    cudaEvent_t staged[2] = {nullptr, nullptr};
    bool staged_used[2] = {false, false};
    int cur = 0;

    bool valid = false;
    int n_items = 0, n_tasks = 0, split_tokens = 0, max_splits_used = 0, total_q_rows = 0;
    int max_task_splits = 0;
    int n_prefill = 0;
    bool causal = false;
    bool fusable = false;  // every request has at least as many keys as query rows
    int64_t kv_tokens = 0, num_pages = 0;
    const int32_t *kv_indices = nullptr;

    static constexpr int kMapCache = 64;
    MapCacheEntry maps[kMapCache];
    int map_next = 0;

    WorkItem *items() { return static_cast<WorkItem *>(d_meta); }
    MergeTask *tasks() {
        return reinterpret_cast<MergeTask *>(static_cast<char *>(d_meta) + sizeof(WorkItem) * max_items);
    }
    size_t prefill_offset() const { return sizeof(WorkItem) * max_items + sizeof(MergeTask) * max_tasks; }
    PrefillItem *prefill_items() { return reinterpret_cast<PrefillItem *>(static_cast<char *>(d_meta) + prefill_offset()); }
};

static pgqa_status pool_map(pgqa_plan *plan, const void *pool, int box_rows, bool swizzle128,
                            const CUtensorMap **out) {
    for (auto &e : plan->maps)
        if (e.ptr == pool && e.num_pages == plan->num_pages && e.box_rows == box_rows && e.swizzle128 == swizzle128) {
            *out = &e.map;
            return PGQA_OK;
        }
    MapCacheEntry &e = plan->maps[plan->map_next];
    plan->map_next = (plan->map_next + 1) % pgqa_plan::kMapCache;
    pgqa_status s = make_pool_map(&e.map, pool, plan->num_pages, plan->cfg.page_size, plan->cfg.num_kv_heads,
                                  plan->cfg.head_dim, plan->cfg.dtype, box_rows, swizzle128);
    if (s != PGQA_OK) {
        e.ptr = nullptr;
        return s;
    }
    e.ptr = pool;
    e.num_pages = plan->num_pages;
    e.box_rows = box_rows;
    e.swizzle128 = swizzle128;
    *out = &e.map;
    return PGQA_OK;
}

static void plan_free(pgqa_plan *p) {
    if (!p) return;
    for (int i = 0; i < 2; ++i) {
        if (p->staged[i]) {
            cudaEventSynchronize(p->staged[i]);
            cudaEventDestroy(p->staged[i]);
        }
        if (p->h_meta[i]) cudaFreeHost(p->h_meta[i]);
    }
    if (p->d_meta) cudaFree(p->d_meta);
    if (p->d_partial_o) cudaFree(p->d_partial_o);
    if (p->d_partial_lse) cudaFree(p->d_partial_lse);
    if (p->rope_cs) cudaFree(p->rope_cs);
    delete p;
}

// Helpers shared with the other entry-point translation units.
namespace pgqa {
pgqa_status report(pgqa_status s, const char *msg) { return fail(s, "%s", msg); }
pgqa_status report_cuda(cudaError_t e, const char *what) { return cuda_fail(e, what); }
pgqa_status current_device_flags(unsigned int **out) { return device_flags(out); }
pgqa_status encode_pool_map(CUtensorMap *map, const void *pool, int64_t num_pages, int page_size, int num_kv_heads,
                            int head_dim, pgqa_dtype dt, int box_rows, bool swizzle128) {
    return make_pool_map(map, pool, num_pages, page_size, num_kv_heads, head_dim, dt, box_rows, swizzle128);
}
}  // namespace pgqa

extern "C" {

int pgqa_abi_version(void) { return PGQA_ABI_VERSION; }

const char *pgqa_status_string(pgqa_status s) {
    switch (s) {
        case PGQA_OK: return "ok";
        case PGQA_ERR_INVALID_ARG: return "invalid argument";
        case PGQA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PGQA_ERR_BAD_PAGE_TABLE: return "malformed page table";
        case PGQA_ERR_CUDA: return "CUDA error";
        case PGQA_ERR_CAPACITY: return "plan capacity exceeded";
        case PGQA_ERR_DEVICE_CHECK: return "device-side check fired";
    }
    return "unknown status";
}

const char *pgqa_last_error(void) { return g_last_error; }

pgqa_status pgqa_read_device_flags(uint32_t *flags_host, int clear) {
    if (!flags_host) return fail(PGQA_ERR_INVALID_ARG, "flags_host is NULL");
    unsigned int *d = nullptr;
    pgqa_status s = device_flags(&d);
    if (s != PGQA_OK) return s;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    e = cudaMemcpy(flags_host, d, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device flags");
    if (clear) {
        e = cudaMemset(d, 0, sizeof(uint32_t));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "clear device flags");
    }
    if (*flags_host) return fail(PGQA_ERR_DEVICE_CHECK, "device flags 0x%x", *flags_host);
    return PGQA_OK;
}

pgqa_status pgqa_kv_append(void *k_pool, void *v_pool, int64_t num_pages, int page_size, int num_kv_heads,
                           int head_dim, pgqa_dtype dtype, const void *k, const void *v,
                           const int64_t *slot_mapping, int64_t num_tokens, pgqa_stream_t stream) {
    if (num_tokens < 0 || num_pages < 0) return fail(PGQA_ERR_INVALID_ARG, "negative size");
    if (dtype != PGQA_BF16 && dtype != PGQA_FP16) return fail(PGQA_ERR_UNSUPPORTED, "append dtype must be bf16/fp16");
    if (head_dim != 64 && head_dim != 128) return fail(PGQA_ERR_UNSUPPORTED, "head_dim %d", head_dim);
    if (!supported_page_size(page_size)) return fail(PGQA_ERR_UNSUPPORTED, "page_size %d", page_size);
    if (num_kv_heads < 1) return fail(PGQA_ERR_INVALID_ARG, "num_kv_heads %d", num_kv_heads);
    if (num_kv_heads > (1 << 20)) return fail(PGQA_ERR_UNSUPPORTED, "num_kv_heads %d > 2^20", num_kv_heads);
    if (num_tokens == 0) return PGQA_OK;
    if (!k_pool || !v_pool || !k || !v || !slot_mapping) return fail(PGQA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k) || !aligned16(v))
        return fail(PGQA_ERR_INVALID_ARG, "pool and row pointers must be 16-byte aligned");
    unsigned int *flags = nullptr;
    pgqa_status s = device_flags(&flags);
    if (s != PGQA_OK) return s;
    const int row_bytes = num_kv_heads * head_dim * 2;
    cudaError_t e = launch_kv_append(k_pool, v_pool, k, v, slot_mapping, num_tokens, num_pages * page_size,
                                     row_bytes, flags, true, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    return PGQA_OK;
}

pgqa_status pgqa_kv_append_rope(const pgqa_plan *plan, void *k_pool, void *v_pool, int64_t num_pages, const void *k,
                                const void *v, const int64_t *slot_mapping, const int32_t *positions,
                                int64_t num_tokens, pgqa_stream_t stream) {
    if (!plan) return fail(PGQA_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->rope_cs) return fail(PGQA_ERR_INVALID_ARG, "the plan was created without RoPE (rope_theta 0)");
    if (num_tokens < 0 || num_pages < 0) return fail(PGQA_ERR_INVALID_ARG, "negative size");
    if (num_tokens == 0) return PGQA_OK;
    if (!k_pool || !v_pool || !k || !v || !slot_mapping || !positions)
        return fail(PGQA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k) || !aligned16(v))
        return fail(PGQA_ERR_INVALID_ARG, "pool and row pointers must be 16-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != plan->device) return fail(PGQA_ERR_INVALID_ARG, "plan belongs to device %d, current is %d", plan->device, dev);
    unsigned int *flags = nullptr;
    pgqa_status s = device_flags(&flags);
    if (s != PGQA_OK) return s;
    const pgqa_plan_config &c = plan->cfg;
    e = launch_kv_append_rope(k_pool, v_pool, k, v, slot_mapping, positions, num_tokens, num_pages * c.page_size,
                              c.num_kv_heads, c.head_dim, c.dtype, plan->rope_cs, c.rope_max_position, flags, true,
                              reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_append_rope launch");
    return PGQA_OK;
}

// Plan options that plan_create accepts (all host-side).
static pgqa_status check_config(const pgqa_plan_config &c) {
    if (c.num_kv_heads < 1 || c.num_qo_heads < 1 || c.num_qo_heads % c.num_kv_heads != 0)
        return fail(PGQA_ERR_INVALID_ARG, "num_qo_heads %d must be a positive multiple of num_kv_heads %d",
                    c.num_qo_heads, c.num_kv_heads);
    const int group = c.num_qo_heads / c.num_kv_heads;
    // The tensor-core decode tile holds 16 heads (two n tiles); the CUDA-core kernel 8.
    const int max_group = c.decode_kernel == PGQA_DECODE_CUDA_CORE ? 8 : 16;
    if (group > max_group)
        return fail(PGQA_ERR_UNSUPPORTED, "query heads per kv head %d > %d", group, max_group);
    if (c.head_dim != 64 && c.head_dim != 128) return fail(PGQA_ERR_UNSUPPORTED, "head_dim %d", c.head_dim);
    if (!supported_page_size(c.page_size)) return fail(PGQA_ERR_UNSUPPORTED, "page_size %d", c.page_size);
    if (c.dtype != PGQA_BF16 && c.dtype != PGQA_FP16) return fail(PGQA_ERR_UNSUPPORTED, "dtype must be bf16/fp16");
    if (c.max_batch < 1 || c.max_q_rows < 1 || c.max_q_rows > (1 << 24))
        return fail(PGQA_ERR_INVALID_ARG, "max_batch/max_q_rows out of range");
    if (c.max_splits < 0 || c.split_tokens < 0 || c.ctas_per_sm < 0)
        return fail(PGQA_ERR_INVALID_ARG, "negative plan option");
    if (c.decode_kernel < PGQA_DECODE_AUTO || c.decode_kernel > PGQA_DECODE_CUDA_CORE)
        return fail(PGQA_ERR_INVALID_ARG, "decode_kernel %d", c.decode_kernel);
    if (c.prefill_kernel < PGQA_PREFILL_AUTO || c.prefill_kernel > PGQA_PREFILL_MMA_SYNC)
        return fail(PGQA_ERR_INVALID_ARG, "prefill_kernel %d", c.prefill_kernel);
    if (c.prefill_splits < 0 || c.prefill_splits > 8)
        return fail(PGQA_ERR_INVALID_ARG, "prefill_splits %d (0..8)", c.prefill_splits);
    if (c.test_stall_wait_us < 0 || c.test_stall_wait_us > 1000000)
        return fail(PGQA_ERR_INVALID_ARG, "test_stall_wait_us %d outside [0, 1000000]", c.test_stall_wait_us);
    if (c.pipeline_stages < 0 || c.pipeline_stages > 3)
        return fail(PGQA_ERR_UNSUPPORTED, "pipeline_stages %d (0, 1, 2 or 3)", c.pipeline_stages);
    if (c.pipeline_stages == 1 && (c.decode_kernel == PGQA_DECODE_CUDA_CORE || group > 8))
        return fail(PGQA_ERR_UNSUPPORTED, "the wide decode form (pipeline_stages 1) runs groups of up to 8 heads "
                    "on the per-item tensor-core kernel");
    if (c.rope_theta < 0.0 || std::isnan(c.rope_theta)) return fail(PGQA_ERR_INVALID_ARG, "rope_theta %g", c.rope_theta);
    if (c.rope_theta > 0.0) {
        if (c.rope_max_position < 1 || c.rope_max_position > (1 << 24))
            return fail(PGQA_ERR_INVALID_ARG, "rope_max_position %d outside [1, 2^24]", c.rope_max_position);
        if (c.decode_kernel == PGQA_DECODE_CUDA_CORE)
            return fail(PGQA_ERR_UNSUPPORTED, "RoPE runs on the tensor-core kernels");
    }
    return PGQA_OK;
}

// The plan's host-side shape: kernel choices and tile sizes that follow from the options.
static void plan_shape(pgqa_plan *p, const pgqa_plan_config &c) {
    p->cfg = c;
    p->group = c.num_qo_heads / c.num_kv_heads;
    p->tile = decode_warp_tile(c.head_dim);
    p->box_rows = std::min(c.page_size, p->tile);
    p->kernel = c.decode_kernel == PGQA_DECODE_CUDA_CORE ? PGQA_DECODE_CUDA_CORE : PGQA_DECODE_TENSOR_CORE;
    p->stages = c.pipeline_stages == 0 ? 2 : c.pipeline_stages;
    // AUTO takes the tcgen05 kernel, measured faster on GB300 for 512-row causal chunks over
    // 1536 keys at every shape tried: d 64 g 7 19.5 against 26.1 us, d 64 g 4 (page 16) 25.8
    // against 36.4, d 128 g 6 25.5 against 28.1, d 128 g 16 39.4 against 60.0; beside a ragged
    // call's 127 decode rows 42.1 against 42.5 us.
    p->prefill_kind = c.prefill_kernel == PGQA_PREFILL_MMA_SYNC ? PGQA_PREFILL_MMA_SYNC : PGQA_PREFILL_TCGEN05;
    p->prefill_pairs = p->prefill_kind == PGQA_PREFILL_MMA_SYNC ? 64 : 128;
}

// Capacities of the plan's lists, from its options, SM count and CTA slots per SM.
static pgqa_status plan_capacity(pgqa_plan *p) {
    const pgqa_plan_config &c = p->cfg;
    p->ctas_per_sm = std::max(p->slots_per_sm[2], p->slots_per_sm[3]);
    // Slices never exceed 8 waves of CTAs + one per row and kv head; forced short slices may need more.
    const int64_t items = c.max_q_rows * c.num_kv_heads + 8LL * p->num_sms * p->ctas_per_sm + 64;
    const int64_t prefill = (c.max_q_rows * p->group / 64 + c.max_batch + 1) * c.num_kv_heads * 8;
    if (items > (1 << 26) || prefill > (1 << 26)) return fail(PGQA_ERR_CAPACITY, "plan capacity too large");
    p->max_items = static_cast<int>(items);
    p->max_tasks = static_cast<int>(c.max_q_rows * c.num_kv_heads);
    p->max_prefill = static_cast<int>(prefill);
    // partial slots: split decode slices, plus up to 8 key slices per prefill row and kv head
    p->max_slots = p->max_items + static_cast<int>(c.max_q_rows * c.num_kv_heads * 8);
    return PGQA_OK;
}

pgqa_status pgqa_plan_create(pgqa_plan **out, const pgqa_plan_config *cfg) {
    if (!out || !cfg) return fail(PGQA_ERR_INVALID_ARG, "NULL argument");
    *out = nullptr;
    const pgqa_plan_config &c = *cfg;
    const pgqa_status cs = check_config(c);
    if (cs != PGQA_OK) return cs;
    const int group = c.num_qo_heads / c.num_kv_heads;
    pgqa_plan *p = new (std::nothrow) pgqa_plan();
    if (!p) return fail(PGQA_ERR_CAPACITY, "out of host memory");
    plan_shape(p, c);
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    // CTA slots of the split heuristic, unless the caller fixes them: the resident CTAs
    // per SM of the kernel that will run (registers and shared memory decide), at most
    // two.  Timed on GB300, a third resident CTA adds no bandwidth once HBM is saturated
    // and only shortens every slice (uniform 4 x 32768-token batch, d 128: 304 slices
    // 26.3 us, 456 slices 28.8 us).
    for (int st = 1; st <= 3 && e == cudaSuccess; ++st) {
        int b = 2;  // the CUDA-core kernel's launch bound
        if (c.ctas_per_sm > 0) {
            b = c.ctas_per_sm;
        } else if (p->kernel == PGQA_DECODE_TENSOR_CORE && (st > 1 || group <= 8)) {
            e = decode_blocks_per_sm(st, c.head_dim, group, c.dtype, &b);
            b = std::min(b, 2);
        }
        p->slots_per_sm[st] = std::max(1, b);
    }
    if (e != cudaSuccess) {
        plan_free(p);
        return cuda_fail(e, "device query");
    }
    const pgqa_status ps = plan_capacity(p);
    if (ps != PGQA_OK) {
        plan_free(p);
        return ps;
    }
    const size_t meta = sizeof(WorkItem) * p->max_items + sizeof(MergeTask) * p->max_tasks +
                        sizeof(PrefillItem) * p->max_prefill;
    e = cudaMalloc(&p->d_meta, meta);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&p->d_partial_o),
                       sizeof(float) * static_cast<size_t>(p->max_slots) * group * c.head_dim);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&p->d_partial_lse), sizeof(float) * static_cast<size_t>(p->max_slots) * group);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaMallocHost(&p->h_meta[i], meta);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->staged[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess && c.rope_theta > 0.0) {
        // built once on the device (fp64 angles), complete before plan_create returns
        const size_t bytes = sizeof(float2) * static_cast<size_t>(c.rope_max_position) * (c.head_dim / 2);
        e = cudaMalloc(reinterpret_cast<void **>(&p->rope_cs), bytes);
        if (e == cudaSuccess) e = launch_rope_table(p->rope_cs, c.rope_max_position, c.head_dim, c.rope_theta, 0);
        if (e == cudaSuccess) e = cudaStreamSynchronize(0);
    }
    if (e != cudaSuccess) {
        plan_free(p);
        return cuda_fail(e, "plan allocation");
    }
    *out = p;
    return PGQA_OK;
}

pgqa_status pgqa_plan_destroy(pgqa_plan *plan) {
    plan_free(plan);
    return PGQA_OK;
}

pgqa_status pgqa_plan_get_info(const pgqa_plan *plan, pgqa_plan_info *info) {
    if (!plan || !info) return fail(PGQA_ERR_INVALID_ARG, "NULL argument");
    info->num_items = plan->n_items;
    info->num_merge_tasks = plan->n_tasks;
    info->split_tokens = plan->split_tokens;
    info->max_splits_used = plan->max_splits_used;
    info->total_q_rows = plan->total_q_rows;
    info->num_sms = plan->num_sms;
    info->kv_tokens = plan->kv_tokens;
    info->num_prefill_tiles = plan->n_prefill;
    return PGQA_OK;
}

// Admissible keys of one query row and where its new K/V rows go.
struct Row {
    int32_t q_row, page_base, n;  // n: admissible keys of the row
    int32_t new_begin, new_row_base, own_pos;
};

// Streaming rate model of the per-item decode kernel on GB300, fitted to timed
// launches of uniform and mixed batches (bytes per ns, i.e. GB/s):
//   one CTA alone streams at kCtaRate (latency-bound: ~64 KB in flight per CTA with
//   two stages, 1.4x that with three); n CTAs together at n c / (1 + (n c / P)^3)^(1/3),
//   which saturates at P, the rate the kernel reaches with every slot busy.
static double cta_rate(int head_dim, int group, int stages) {
    const double c = head_dim == 64 ? 30.0 : (group <= 8 ? 40.0 : 35.0);
    return stages == 3 ? 1.4 * c : c;
}
static constexpr double kSaturatedRate = 5300.0;  // bytes / ns
static constexpr double kWaveCostNs = 1500.0;     // CTA set-up + epilogue, per wave of CTAs
static constexpr double kMergeCostNs = 2000.0;    // the merge launch, once any row is split

// Pipeline depth of the tensor-core decode kernel: three stages when every warp's tiles
// of the longest slice can be requested at once (the whole slice in flight from the
// start), or when the grid is less than one full wave at two CTAs per SM (so some SMs
// run a single CTA), its slices are long (every warp's share at least one warp tile past
// what its three stages hold) and no prefill grid shares the GPU.  Measured on GB300:
// 32 mixed d 128 (292 CTAs) -4 %, 64 x 2049 at g = 16 (256 CTAs) -6 %; a full wave
// (4 x 32k, 304 CTAs) ran its launch 6 % slower, and a ragged call, whose decode rows then
// went unsplit, 9 %.  Otherwise two, so that three CTAs fit on an SM and overlap each
// other's set-up and epilogue.
//
// Slices of at most kDecodeWideWarps warp tiles take the wide form instead (reported as
// depth 1): one warp per tile, the whole slice requested at once, so no warp of the CTA
// runs more than one tile's chain of dependent steps.  On GB300 that chain, not the copy,
// paced the 128 x 301 step: its busiest warps ran three tiles at ~0.55 us each.
static int pick_stages(const pgqa_plan *plan, int64_t max_slice, int64_t n_items, bool with_prefill) {
    if (plan->kernel == PGQA_DECODE_TENSOR_CORE && plan->group <= 8 &&
        max_slice <= static_cast<int64_t>(kDecodeWideWarps) * plan->tile)
        return 1;
    const int64_t held = 3LL * kDecodeWarps * plan->tile;  // keys three stages hold
    if (max_slice <= held) return 3;
    // Long slices (a warp tile past what three stages hold) in a grid short of one full
    // wave: SMs with one CTA have the shared memory for the deeper ring (timed on GB300
    // for 1 x 32k: 256-key slices at three stages 9.9 us, 224-key slices at two 10.35).
    if (!with_prefill && max_slice >= held + kDecodeWarps * plan->tile &&
        n_items < static_cast<int64_t>(plan->num_sms) * plan->slots_per_sm[3])
        return 3;
    return 2;
}

// Slice length (whole warp tiles, at least one tile per warp) for the decode rows that
// minimises the estimated launch time.  The hardware runs `slots` CTAs at once and
// starts the rest (longest first) as slots free up, so the estimate walks waves of
// `slots` items: each wave takes max(its bytes / rate(CTAs in it), its longest slice /
// one CTA's rate), plus kWaveCostNs; splitting adds kMergeCostNs.
static int64_t choose_slice(const pgqa_plan *plan, const Row *rows, int64_t n_rows, int64_t longest,
                            int64_t prefill_ctas) {
    const bool with_prefill = prefill_ctas > 0;
    const pgqa_plan_config &c = plan->cfg;
    const int64_t tile = plan->tile;
    const int64_t min_split = static_cast<int64_t>(kDecodeWarps) * tile;
    const double row_bytes = 4.0 * c.head_dim;  // K + V of one token of one kv head
    // distinct admissible-key counts, longest first, with their multiplicity
    std::vector<int64_t> lens(static_cast<size_t>(n_rows));
    for (int64_t i = 0; i < n_rows; ++i) lens[i] = rows[i].n;
    std::sort(lens.begin(), lens.end(), std::greater<int64_t>());
    std::vector<std::pair<int64_t, int64_t>> hist;  // (n, rows)
    for (int64_t n : lens) {
        if (!hist.empty() && hist.back().first == n)
            ++hist.back().second;
        else
            hist.push_back({n, 1});
    }
    std::vector<std::pair<int64_t, int64_t>> slices;  // (slice length, items)
    slices.reserve(2 * hist.size());
    std::vector<uint64_t> order;  // slices, longest first (see below)
    order.reserve(2 * hist.size());
    int64_t best_len = round_up(std::max<int64_t>(longest, min_split), tile), prev_len = -1;
    double best = 0.0;
    bool have = false;
    for (int64_t parts = 1;; ++parts) {
        const int64_t len = round_up(ceil_div(std::max<int64_t>(1, longest), parts), tile);
        if (len < min_split && have) break;
        if (len == prev_len) continue;
        prev_len = len;
        slices.clear();
        int64_t n_items = 0, max_slice = 0;
        bool split = false;
        for (const auto &h : hist) {
            const int64_t n = h.first, cnt = h.second * c.num_kv_heads;
            if (n == 0) {
                slices.push_back({0, cnt});
                n_items += cnt;
                continue;
            }
            int64_t ns = ceil_div(n, std::max(len, min_split));
            if (c.max_splits > 0) ns = std::min<int64_t>(ns, c.max_splits);
            const int64_t sl = round_up(ceil_div(n, ns), tile);
            ns = ceil_div(n, sl);
            if (ns > 1) slices.push_back({sl, (ns - 1) * cnt});
            slices.push_back({n - (ns - 1) * sl, cnt});
            n_items += ns * cnt;
            max_slice = std::max(max_slice, std::min(sl, n));
            split = split || ns > 1;
        }
        const int stages =
            c.pipeline_stages != 0 ? c.pipeline_stages : pick_stages(plan, max_slice, n_items, with_prefill);
        // A prefill CTA beside decode rows leaves its SM room for one decode CTA fewer
        // (its ~104 KB of shared memory), so those slots are not the decode rows'.
        const int64_t slots = std::max<int64_t>(
            plan->num_sms, static_cast<int64_t>(plan->num_sms) * plan->slots_per_sm[stages] - prefill_ctas);
        if (have && (n_items > 8 * slots || n_items > plan->max_items)) break;
        const double cr = cta_rate(c.head_dim, plan->group, stages);
        // Longest slices first: sort packed keys (length, then the entry's index, which only
        // orders slices of equal length, and those are interchangeable in the walk below) --
        // a fraction of the cost of sorting the pairs, which dominated plan_update's host time.
        order.resize(slices.size());
        for (size_t i = 0; i < slices.size(); ++i)
            order[i] = (static_cast<uint64_t>(slices[i].first) << 33) | static_cast<uint64_t>(i);
        std::sort(order.begin(), order.end(), std::greater<uint64_t>());
        double t = 0.0, wave_bytes = 0.0;
        int64_t free_slots = slots, in_wave = 0, first = -1;
        auto close_wave = [&]() {
            const double nc = static_cast<double>(in_wave) * cr;
            const double rate = nc / std::cbrt(1.0 + std::pow(nc / kSaturatedRate, 3.0));
            t += std::max(wave_bytes / rate, static_cast<double>(first) * row_bytes / cr) + kWaveCostNs;
        };
        for (const uint64_t key : order) {
            const auto &sl = slices[key & ((uint64_t(1) << 33) - 1)];
            int64_t cnt = sl.second;
            while (cnt > 0) {
                const int64_t take = std::min(cnt, free_slots);
                if (first < 0) first = sl.first;
                wave_bytes += static_cast<double>(take) * sl.first * row_bytes;
                in_wave += take;
                cnt -= take;
                free_slots -= take;
                if (free_slots == 0) {
                    close_wave();
                    free_slots = slots;
                    wave_bytes = 0.0;
                    in_wave = 0;
                    first = -1;
                }
            }
        }
        if (in_wave > 0) close_wave();
        if (split) t += kMergeCostNs;
        if (!have || t < best) {
            best = t;
            best_len = len;
            have = true;
        }
        if (len <= min_split) break;
    }
    return best_len;
}

// What plan_update builds, computed on the host alone: the table's checks, the
// decode work list (slices of every (row, kv head)), the merge list, the prefill
// tiles and the decode kernel's pipeline depth.
struct Schedule {
    std::vector<WorkItem> items;
    std::vector<MergeTask> tasks;
    std::vector<PrefillItem> prefill;
    int64_t split_tokens = 0, rows = 0, kv_tokens = 0;
    int max_used = 1, max_task_splits = 0, stages = 2;
    bool fusable = true;
};

static pgqa_status build_schedule(const pgqa_plan *plan, const int32_t *kv_indptr, const int32_t *last_page_len,
                                  const int32_t *qo_indptr, int batch, bool have_indices,
                                  const int32_t *kv_indices_host, int64_t num_pages, int causal, Schedule *out) {
    const pgqa_plan_config &c = plan->cfg;
    if (batch < 0 || num_pages < 0) return fail(PGQA_ERR_INVALID_ARG, "negative batch or num_pages");
    if (batch > c.max_batch) return fail(PGQA_ERR_CAPACITY, "batch %d > max_batch %d", batch, c.max_batch);
    if (num_pages * static_cast<int64_t>(c.page_size) >= (int64_t(1) << 31))
        return fail(PGQA_ERR_UNSUPPORTED, "pool rows must stay below 2^31");
    if (!kv_indptr || (batch > 0 && !last_page_len)) return fail(PGQA_ERR_INVALID_ARG, "NULL page table");
    if (kv_indptr[0] != 0) return fail(PGQA_ERR_BAD_PAGE_TABLE, "kv_indptr[0] = %d", kv_indptr[0]);
    for (int b = 0; b < batch; ++b) {
        const int64_t np = static_cast<int64_t>(kv_indptr[b + 1]) - kv_indptr[b];
        if (np < 0) return fail(PGQA_ERR_BAD_PAGE_TABLE, "kv_indptr decreases at request %d", b);
        if (np == 0 && last_page_len[b] != 0)
            return fail(PGQA_ERR_BAD_PAGE_TABLE, "request %d has no pages but last_page_len %d", b, last_page_len[b]);
        if (np > 0 && (last_page_len[b] < 1 || last_page_len[b] > c.page_size))
            return fail(PGQA_ERR_BAD_PAGE_TABLE, "last_page_len[%d] = %d outside [1, %d]", b, last_page_len[b],
                        c.page_size);
        if (np * c.page_size >= (int64_t(1) << 30)) return fail(PGQA_ERR_UNSUPPORTED, "request %d too long", b);
    }
    const int64_t nnz = batch > 0 ? kv_indptr[batch] : 0;
    if (nnz > 0 && !have_indices) return fail(PGQA_ERR_INVALID_ARG, "kv_indices is NULL");
    if (kv_indices_host)
        for (int64_t i = 0; i < nnz; ++i)
            if (kv_indices_host[i] < 0 || kv_indices_host[i] >= num_pages)
                return fail(PGQA_ERR_BAD_PAGE_TABLE, "kv_indices[%lld] = %d outside [0, %lld)",
                            static_cast<long long>(i), kv_indices_host[i], static_cast<long long>(num_pages));
    int64_t rows = batch;
    if (qo_indptr) {
        if (qo_indptr[0] != 0) return fail(PGQA_ERR_BAD_PAGE_TABLE, "qo_indptr[0] = %d", qo_indptr[0]);
        for (int b = 0; b < batch; ++b)
            if (qo_indptr[b + 1] < qo_indptr[b]) return fail(PGQA_ERR_BAD_PAGE_TABLE, "qo_indptr decreases at %d", b);
        rows = batch > 0 ? qo_indptr[batch] : 0;
    }
    if (rows > c.max_q_rows)
        return fail(PGQA_ERR_CAPACITY, "%lld query rows > max_q_rows %lld", static_cast<long long>(rows),
                    static_cast<long long>(c.max_q_rows));

    // Admissible keys per query row (bottom-right causal for multi-row requests).
    std::vector<Row> rowv;
    rowv.reserve(static_cast<size_t>(rows));
    int64_t kv_tokens = 0;
    bool fusable = true;
    std::vector<PrefillItem> prefill;
    for (int b = 0; b < batch; ++b) {
        const int64_t np = static_cast<int64_t>(kv_indptr[b + 1]) - kv_indptr[b];
        const int64_t n = np == 0 ? 0 : (np - 1) * c.page_size + last_page_len[b];
        kv_tokens += n;
        const int64_t r0 = qo_indptr ? qo_indptr[b] : b, r1 = qo_indptr ? qo_indptr[b + 1] : b + 1;
        const int64_t L = r1 - r0;
        // A fused append writes the request's last L key positions from the L new rows.
        if (L > n) fusable = false;
        if (c.rope_theta > 0.0 && L > 0) {
            // query rows sit at the request's last L key positions, all in the table
            if (L > n)
                return fail(PGQA_ERR_INVALID_ARG, "request %d: %lld query rows over %lld keys have no rotary position",
                            b, static_cast<long long>(L), static_cast<long long>(n));
            if (n > c.rope_max_position)
                return fail(PGQA_ERR_INVALID_ARG, "request %d: key positions up to %lld exceed rope_max_position %d", b,
                            static_cast<long long>(n - 1), c.rope_max_position);
        }
        const int64_t nb = L <= n ? n - L : INT32_MAX;
        // (Rows of tensor-core decode items therefore come from single-row requests: the
        // decode kernel's fused append relies on at most one new row per item.)
        if (L > 1 && plan->kernel == PGQA_DECODE_TENSOR_CORE) {
            // A chunk of rows: tensor-core prefill tiles of prefill_pairs (row, head) pairs per
            // kv head (key slices are assigned below, once all tiles are known).
            const int G = plan->group;
            const int mp = plan->prefill_pairs;
            for (int kvh = 0; kvh < c.num_kv_heads; ++kvh)
                for (int64_t m0 = 0; m0 < L * G; m0 += mp) {
                    const int64_t i_last = std::min<int64_t>(L - 1, (m0 + mp - 1) / G);
                    int64_t kend = causal ? n - L + i_last + 1 : n;
                    kend = std::max<int64_t>(0, std::min<int64_t>(n, kend));
                    prefill.push_back({kv_indptr[b], 0, static_cast<int32_t>(kend), static_cast<int32_t>(r0),
                                       static_cast<int32_t>(L), static_cast<int32_t>(n), kvh,
                                       static_cast<int32_t>(m0), -1, 0, 1, 0});
                }
            continue;
        }
        for (int64_t r = r0; r < r1; ++r) {
            int64_t a = n;
            if (causal) a = std::min<int64_t>(n, std::max<int64_t>(0, n - L + (r - r0) + 1));
            rowv.push_back({static_cast<int32_t>(r), kv_indptr[b], static_cast<int32_t>(a),
                            static_cast<int32_t>(nb), static_cast<int32_t>(L <= n ? r0 - nb : 0),
                            static_cast<int32_t>(L <= n ? nb + (r - r0) : -1)});
        }
    }

    // Prefill key slices (each >= 256 keys, at most 8), partials merged per (row, kv head)
    // like split decode rows.  Alone, a chunk takes the most slices that still fit one wave
    // of two CTAs per SM.  Beside decode rows it takes about one CTA per SM, leaving each
    // SM room for decode CTAs: measured on GB300 for a 512-row chunk over 1536 keys with
    // 127 decode rows, 2 slices (112 prefill CTAs) ran the call in 35.2 us against 41.3
    // with 5 (280 CTAs, which filled every slot until they finished); 3 and 4 gave 36.6
    // and 38.1.
    int pf_splits = 1;
    if (!prefill.empty()) {
        int64_t kmax = 0;
        for (const PrefillItem &t : prefill) kmax = std::max<int64_t>(kmax, t.key_end);
        const int64_t ctas_per_sm = rowv.empty() ? 2 : 1;  // decode rows give at least one item each
        if (c.prefill_splits > 0)
            pf_splits = std::min(8, c.prefill_splits);
        else
            pf_splits = static_cast<int>(std::min<int64_t>(
                {8, std::max<int64_t>(1, ctas_per_sm * plan->num_sms / static_cast<int64_t>(prefill.size())),
                 std::max<int64_t>(1, kmax / 256)}));
    }

    const int tile = plan->tile;
    int64_t longest = 0;
    for (const Row &rw : rowv) longest = std::max<int64_t>(longest, rw.n);
    const int64_t ls = c.split_tokens > 0
                           ? round_up(c.split_tokens, tile)
                           : choose_slice(plan, rowv.data(), static_cast<int64_t>(rowv.size()), longest,
                                          static_cast<int64_t>(prefill.size()) * pf_splits);

    std::vector<WorkItem> items;
    std::vector<MergeTask> tasks;
    items.reserve(static_cast<size_t>(rows) * c.num_kv_heads);
    int slot = 0, max_used = 1, max_task_splits = 0;
    for (const Row &rw : rowv) {
        for (int kvh = 0; kvh < c.num_kv_heads; ++kvh) {
            const int64_t n = rw.n;
            int64_t ns = n == 0 ? 1 : ceil_div(n, ls);
            if (c.max_splits > 0) ns = std::min<int64_t>(ns, c.max_splits);
            const int64_t len = n == 0 ? 0 : round_up(ceil_div(n, ns), tile);
            ns = n == 0 ? 1 : ceil_div(n, len);
            if (ns == 1) {
                items.push_back({rw.page_base, 0, static_cast<int32_t>(n), rw.q_row, kvh, -1, rw.new_begin,
                                 rw.new_row_base, rw.own_pos, rw.own_pos, 0, 0});
                continue;
            }
            if (static_cast<int64_t>(tasks.size()) >= plan->max_tasks || slot + ns > plan->max_slots)
                return fail(PGQA_ERR_CAPACITY, "split partials exceed the plan capacity");
            for (int64_t s = 0; s < ns; ++s)
                items.push_back({rw.page_base, static_cast<int32_t>(s * len),
                                 static_cast<int32_t>(std::min<int64_t>(n, (s + 1) * len)), rw.q_row, kvh,
                                 slot + static_cast<int32_t>(s), rw.new_begin, rw.new_row_base,
                                 s == ns - 1 ? rw.own_pos : -1, rw.own_pos, 0, 0});
            tasks.push_back({rw.q_row, kvh, slot, static_cast<int32_t>(ns)});
            slot += static_cast<int>(ns);
            max_used = std::max<int>(max_used, static_cast<int>(ns));
            max_task_splits = std::max<int>(max_task_splits, static_cast<int>(ns));
        }
        if (static_cast<int64_t>(items.size()) > plan->max_items)
            return fail(PGQA_ERR_CAPACITY, "work items exceed the plan capacity %d", plan->max_items);
    }
    // Longest slices first, so that they start in the first wave.
    std::stable_sort(items.begin(), items.end(), [](const WorkItem &a, const WorkItem &b) {
        return (a.tok_end - a.tok_begin) > (b.tok_end - b.tok_begin);
    });

    // The prefill key slices chosen above, each tile cut into pf_splits CTAs.
    if (pf_splits > 1) {
        // partial slots per (request, kv head): rows x splits, after the decode slots
        std::vector<PrefillItem> split_items;
        split_items.reserve(prefill.size() * pf_splits);
        int32_t prev_row0 = -1, prev_head = -1;
        int64_t base = 0;
        for (const PrefillItem &t : prefill) {
            if (t.q_row0 != prev_row0 || t.kv_head != prev_head) {  // a new (request, kv head)
                base = slot;
                slot += t.rows * pf_splits;
                if (slot > plan->max_slots) return fail(PGQA_ERR_CAPACITY, "split partials exceed the plan capacity");
                for (int i = 0; i < t.rows; ++i) {
                    if (static_cast<int64_t>(tasks.size()) >= plan->max_tasks)
                        return fail(PGQA_ERR_CAPACITY, "merge tasks exceed the plan capacity");
                    tasks.push_back({t.q_row0 + i, t.kv_head, static_cast<int32_t>(base + i * pf_splits), pf_splits});
                }
                prev_row0 = t.q_row0;
                prev_head = t.kv_head;
            }
            const int64_t len = round_up(ceil_div(std::max<int32_t>(1, t.key_end), pf_splits), 64);
            for (int sidx = 0; sidx < pf_splits; ++sidx) {
                PrefillItem u = t;
                u.key_begin = static_cast<int32_t>(std::min<int64_t>(t.key_end, sidx * len));
                u.key_end = static_cast<int32_t>(std::min<int64_t>(t.key_end, (sidx + 1) * len));
                u.part_base = static_cast<int32_t>(base);
                u.split = sidx;
                u.num_splits = pf_splits;
                split_items.push_back(u);
            }
        }
        prefill.swap(split_items);
        max_task_splits = std::max(max_task_splits, pf_splits);
    }
    if (static_cast<int64_t>(prefill.size()) > plan->max_prefill)
        return fail(PGQA_ERR_CAPACITY, "prefill tiles exceed the plan capacity %d", plan->max_prefill);
    // Longest prefill slices first.
    std::stable_sort(prefill.begin(), prefill.end(), [](const PrefillItem &a, const PrefillItem &b) {
        return a.key_end - a.key_begin > b.key_end - b.key_begin;
    });

    int stages = c.pipeline_stages;
    if (stages == 0) {
        int64_t longest_item = 0;
        for (const WorkItem &w : items) longest_item = std::max<int64_t>(longest_item, w.tok_end - w.tok_begin);
        stages = pick_stages(plan, longest_item, static_cast<int64_t>(items.size()), !prefill.empty());
    }
    out->items.swap(items);
    out->tasks.swap(tasks);
    out->prefill.swap(prefill);
    out->split_tokens = ls;
    out->rows = rows;
    out->kv_tokens = kv_tokens;
    out->max_used = max_used;
    out->max_task_splits = max_task_splits;
    out->stages = stages;
    out->fusable = fusable;
    return PGQA_OK;
}

pgqa_status pgqa_plan_update(pgqa_plan *plan, const int32_t *kv_indptr, const int32_t *last_page_len,
                             const int32_t *qo_indptr, int batch, const int32_t *kv_indices,
                             const int32_t *kv_indices_host, int64_t num_pages, int causal,
                             pgqa_stream_t stream) {
    if (!plan) return fail(PGQA_ERR_INVALID_ARG, "plan is NULL");
    plan->valid = false;
    Schedule sc;
    const pgqa_status ss = build_schedule(plan, kv_indptr, last_page_len, qo_indptr, batch, kv_indices != nullptr,
                                          kv_indices_host, num_pages, causal, &sc);
    if (ss != PGQA_OK) return ss;
    const std::vector<WorkItem> &items = sc.items;
    const std::vector<MergeTask> &tasks = sc.tasks;
    const std::vector<PrefillItem> &prefill = sc.prefill;

    // Stage in pinned memory (double-buffered) and copy into the persistent buffer.
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int buf = plan->cur;
    cudaError_t e = cudaSuccess;
    if (plan->staged_used[buf]) {
        e = cudaEventSynchronize(plan->staged[buf]);
        if (e != cudaSuccess) return cuda_fail(e, "staging buffer wait");
    }
    char *h = static_cast<char *>(plan->h_meta[buf]);
    const size_t items_bytes = sizeof(WorkItem) * items.size();
    const size_t tasks_off = sizeof(WorkItem) * plan->max_items;
    const size_t tasks_bytes = sizeof(MergeTask) * tasks.size();
    const size_t prefill_off = plan->prefill_offset();
    const size_t prefill_bytes = sizeof(PrefillItem) * prefill.size();
    if (items_bytes) std::memcpy(h, items.data(), items_bytes);
    if (tasks_bytes) std::memcpy(h + tasks_off, tasks.data(), tasks_bytes);
    if (prefill_bytes) std::memcpy(h + prefill_off, prefill.data(), prefill_bytes);
    if (items_bytes) e = cudaMemcpyAsync(plan->d_meta, h, items_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && tasks_bytes)
        e = cudaMemcpyAsync(static_cast<char *>(plan->d_meta) + tasks_off, h + tasks_off, tasks_bytes,
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && prefill_bytes)
        e = cudaMemcpyAsync(static_cast<char *>(plan->d_meta) + prefill_off, h + prefill_off, prefill_bytes,
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(plan->staged[buf], st);
    if (e != cudaSuccess) return cuda_fail(e, "work list upload");
    plan->staged_used[buf] = true;
    plan->cur ^= 1;

    plan->stages = sc.stages;
    plan->n_items = static_cast<int>(items.size());
    plan->n_prefill = static_cast<int>(prefill.size());
    plan->causal = causal != 0;
    plan->n_tasks = static_cast<int>(tasks.size());
    plan->split_tokens = static_cast<int>(sc.split_tokens);
    plan->max_splits_used = sc.max_used;
    plan->max_task_splits = sc.max_task_splits;
    plan->total_q_rows = static_cast<int>(sc.rows);
    plan->kv_tokens = sc.kv_tokens;
    plan->num_pages = num_pages;
    plan->kv_indices = kv_indices;
    plan->fusable = sc.fusable;
    plan->valid = true;
    return PGQA_OK;
}

pgqa_status pgqa_plan_schedule(const pgqa_plan_config *cfg, int num_sms, const int32_t *kv_indptr,
                               const int32_t *last_page_len, const int32_t *qo_indptr, int batch,
                               const int32_t *kv_indices, int64_t num_pages, int causal, pgqa_slice *slices,
                               int max_slices, pgqa_merge *merges, int max_merges, pgqa_prefill_tile *tiles,
                               int max_tiles, pgqa_schedule_info *info) {
    if (!cfg || !info) return fail(PGQA_ERR_INVALID_ARG, "NULL argument");
    if (num_sms < 1) return fail(PGQA_ERR_INVALID_ARG, "num_sms %d", num_sms);
    if (max_slices < 0 || max_merges < 0 || max_tiles < 0) return fail(PGQA_ERR_INVALID_ARG, "negative array size");
    const pgqa_status cs = check_config(*cfg);
    if (cs != PGQA_OK) return cs;
    // A host-only plan: its shape and capacities as pgqa_plan_create sets them on a GPU
    // with num_sms SMs, where every decode variant keeps two CTAs resident per SM.
    pgqa_plan *p = new (std::nothrow) pgqa_plan();
    if (!p) return fail(PGQA_ERR_CAPACITY, "out of host memory");
    plan_shape(p, *cfg);
    p->num_sms = num_sms;
    p->slots_per_sm[1] = p->slots_per_sm[2] = p->slots_per_sm[3] = cfg->ctas_per_sm > 0 ? cfg->ctas_per_sm : 2;
    Schedule sc;
    pgqa_status st = plan_capacity(p);
    if (st == PGQA_OK)
        st = build_schedule(p, kv_indptr, last_page_len, qo_indptr, batch, kv_indices != nullptr, kv_indices,
                            num_pages, causal, &sc);
    const int pairs = p->prefill_pairs;
    delete p;
    if (st != PGQA_OK) return st;

    info->num_items = static_cast<int>(sc.items.size());
    info->num_merge_tasks = static_cast<int>(sc.tasks.size());
    info->num_prefill_tiles = static_cast<int>(sc.prefill.size());
    info->split_tokens = static_cast<int>(sc.split_tokens);
    info->max_splits_used = sc.max_used;
    info->pipeline_stages = sc.stages;
    info->total_q_rows = static_cast<int>(sc.rows);
    info->kv_tokens = sc.kv_tokens;
    if ((slices && max_slices < info->num_items) || (merges && max_merges < info->num_merge_tasks) ||
        (tiles && max_tiles < info->num_prefill_tiles))
        return fail(PGQA_ERR_CAPACITY, "output arrays hold %d / %d / %d entries, the schedule has %d / %d / %d",
                    max_slices, max_merges, max_tiles, info->num_items, info->num_merge_tasks,
                    info->num_prefill_tiles);
    if (slices)
        for (size_t i = 0; i < sc.items.size(); ++i) {
            const WorkItem &w = sc.items[i];
            slices[i] = {w.q_row, w.kv_head, w.tok_begin, w.tok_end, w.out_slot < 0 ? -1 : w.out_slot,
                         w.write_pos};
        }
    if (merges)
        for (size_t i = 0; i < sc.tasks.size(); ++i) {
            const MergeTask &t = sc.tasks[i];
            merges[i] = {t.q_row, t.kv_head, t.slot_base, t.num_splits};
        }
    if (tiles)
        for (size_t i = 0; i < sc.prefill.size(); ++i) {
            const PrefillItem &t = sc.prefill[i];
            tiles[i] = {t.q_row0, t.rows, t.n_keys, t.kv_head, t.pair0, pairs, t.key_begin, t.key_end,
                        t.part_base < 0 ? -1 : t.part_base, t.split, t.num_splits};
        }
    return PGQA_OK;
}

static pgqa_status run_impl(pgqa_plan *plan, const void *k_new, const void *v_new, const void *q, void *k_pool,
                            void *v_pool, void *out, pgqa_dtype out_dtype, float *lse, float sm_scale, int flags,
                            pgqa_stream_t stream) {
    if (!plan) return fail(PGQA_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->valid) return fail(PGQA_ERR_INVALID_ARG, "run() before a successful plan_update()");
    const pgqa_plan_config &c = plan->cfg;
    if (out_dtype != PGQA_FP32 && out_dtype != c.dtype)
        return fail(PGQA_ERR_UNSUPPORTED, "out_dtype must be fp32 or the plan's dtype");
    if (flags & ~PGQA_RUN_POOL_STABLE) return fail(PGQA_ERR_INVALID_ARG, "unknown run flags 0x%x", flags);
    const bool fused = k_new != nullptr || v_new != nullptr;
    if (fused) {
        if (!k_new || !v_new) return fail(PGQA_ERR_INVALID_ARG, "k_new and v_new go together");
        if (plan->kernel != PGQA_DECODE_TENSOR_CORE)
            return fail(PGQA_ERR_UNSUPPORTED, "the fused append runs on the tensor-core decode kernel");
        if (!plan->fusable)
            return fail(PGQA_ERR_INVALID_ARG, "a request has more query rows than keys: nothing to append them to");
        if (!aligned16(k_new) || !aligned16(v_new))
            return fail(PGQA_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    }
    if (plan->n_items == 0 && plan->n_prefill == 0) return PGQA_OK;
    if (!q || !k_pool || !v_pool || !out) return fail(PGQA_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PGQA_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != plan->device) return fail(PGQA_ERR_INVALID_ARG, "plan belongs to device %d, current is %d", plan->device, dev);
    unsigned int *dflags = nullptr;
    pgqa_status s = device_flags(&dflags);
    if (s != PGQA_OK) return s;
    const bool swz = plan->kernel == PGQA_DECODE_TENSOR_CORE;
    const CUtensorMap *mk = nullptr, *mv = nullptr;
    s = pool_map(plan, k_pool, plan->box_rows, swz, &mk);
    if (s == PGQA_OK) s = pool_map(plan, v_pool, plan->box_rows, swz, &mv);
    if (s != PGQA_OK) return s;

    const float scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(c.head_dim));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (plan->n_prefill > 0) {
        const int prows = std::min(c.page_size, 64);
        const CUtensorMap *pk = nullptr, *pv = nullptr;
        s = pool_map(plan, k_pool, prows, true, &pk);
        if (s == PGQA_OK) s = pool_map(plan, v_pool, prows, true, &pv);
        if (s != PGQA_OK) return s;
        PrefillParams pp{};
        pp.q = q;
        pp.items = plan->prefill_items();
        pp.kv_indices = plan->kv_indices;
        pp.num_pages = plan->num_pages;
        pp.page_size = c.page_size;
        pp.box_rows = prows;
        pp.num_qo_heads = c.num_qo_heads;
        pp.num_kv_heads = c.num_kv_heads;
        pp.causal = plan->causal ? 1 : 0;
        pp.scale_log2 = scale * 1.4426950408889634f;
        pp.out = out;
        pp.out_dtype = out_dtype;
        pp.lse = lse;
        pp.flags = dflags;
        pp.k_new = k_new;
        pp.v_new = v_new;
        pp.k_pool = k_pool;
        pp.v_pool = v_pool;
        pp.prefetch_pool = (flags & PGQA_RUN_POOL_STABLE) ? 1 : 0;
        pp.partial_o = plan->d_partial_o;
        pp.partial_lse = plan->d_partial_lse;
        pp.rope_cs = plan->rope_cs;
        e = launch_prefill(plan->prefill_kind, c.head_dim, plan->group, c.dtype, *pk, *pv, pp, plan->n_prefill, true,
                           st);
        if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    }
    if (plan->n_items > 0) {
    DecodeParams p{};
    p.q = q;
    p.items = plan->items();
    p.kv_indices = plan->kv_indices;
    p.num_pages = plan->num_pages;
    p.page_size = c.page_size;
    p.box_rows = plan->box_rows;
    p.num_qo_heads = c.num_qo_heads;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.out_dtype = out_dtype;
    p.lse = lse;
    p.partial_o = plan->d_partial_o;
    p.partial_lse = plan->d_partial_lse;
    p.flags = dflags;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.num_kv_heads = c.num_kv_heads;
    p.prefetch_pool = (flags & PGQA_RUN_POOL_STABLE) ? 1 : 0;
    // With a prefill grid just launched, the decode grid runs beside it.
    p.defer_wait = plan->n_prefill > 0 ? 1 : 0;
    p.rope_cs = plan->rope_cs;
    p.stall_wait_us = static_cast<uint32_t>(c.test_stall_wait_us);
    e = launch_decode(plan->kernel, plan->stages, c.head_dim, plan->group, c.dtype, *mk, *mv, p, plan->n_items,
                      true, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    }
    if (plan->n_tasks > 0) {
        MergeParams mp{};
        mp.tasks = plan->tasks();
        mp.partial_o = plan->d_partial_o;
        mp.partial_lse = plan->d_partial_lse;
        mp.out = out;
        mp.out_dtype = out_dtype;
        mp.lse = lse;
        mp.num_qo_heads = c.num_qo_heads;
        mp.group = plan->group;
        mp.head_dim = c.head_dim;
        e = launch_merge(mp, plan->n_tasks, plan->max_task_splits, true, st);
        if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    }
    return PGQA_OK;
}

pgqa_status pgqa_run(pgqa_plan *plan, const void *q, const void *k_pool, const void *v_pool, void *out,
                     pgqa_dtype out_dtype, float *lse, float sm_scale, pgqa_stream_t stream) {
    return run_impl(plan, nullptr, nullptr, q, const_cast<void *>(k_pool), const_cast<void *>(v_pool), out,
                    out_dtype, lse, sm_scale, 0, stream);
}

pgqa_status pgqa_append_run(pgqa_plan *plan, const void *k_new, const void *v_new, const void *q, void *k_pool,
                            void *v_pool, void *out, pgqa_dtype out_dtype, float *lse, float sm_scale, int flags,
                            pgqa_stream_t stream) {
    // both NULL: no new rows, a run() that honours the flags
    if (!k_new != !v_new) return fail(PGQA_ERR_INVALID_ARG, "k_new and v_new go together");
    return run_impl(plan, k_new, v_new, q, k_pool, v_pool, out, out_dtype, lse, sm_scale, flags, stream);
}

}  // extern "C"
