// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through the runtime)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedgqa.h"

namespace pgqa {

// ---------------------------------------------------------------------------
// Work description produced by plan_update (host) and read by the kernels.
// ---------------------------------------------------------------------------

// One CTA of the split-KV partial kernel: one (query row, kv head, key slice).
struct alignas(16) WorkItem {
    int32_t page_base;     // kv_indptr[request]: first entry of the request's pages in kv_indices
    int32_t tok_begin;     // key slice [tok_begin, tok_end), tok_begin a multiple of the warp tile
    int32_t tok_end;       // <= the row's admissible key count
    int32_t q_row;         // query row
    int32_t kv_head;
    int32_t out_slot;      // < 0: write the final output of (q_row, kv_head);
                           // >= 0: write partial slot out_slot (merged later)
    int32_t new_begin;     // first key position of the request holding one of the call's new rows
                           // (the request's last qo_len positions); INT32_MAX when it has none
    int32_t new_row_base;  // the new row of key position p is k_new[p + new_row_base]
    int32_t write_pos;     // key position whose new row this item stores into the pool, or -1
    int32_t q_pos;         // key position of the query row's own key: its rotary position
    int32_t pad1, pad2;
};
static_assert(sizeof(WorkItem) == 48, "WorkItem is 48 bytes");

// One merge: the partial slots [slot_base, slot_base + num_splits) of (q_row, kv_head).
struct alignas(16) MergeTask {
    int32_t q_row;
    int32_t kv_head;
    int32_t slot_base;
    int32_t num_splits;
};
static_assert(sizeof(MergeTask) == 16, "MergeTask is 16 bytes");

// One CTA of the prefill-segment kernel: 64 (row, head) pairs of one kv head of
// a multi-row request, pairs numbered m = i * G + h (i: row within the request).
struct alignas(16) PrefillItem {
    int32_t page_base;   // kv_indptr[request]
    int32_t key_begin;   // key slice [key_begin, key_end) of this CTA (key_begin a multiple of 64)
    int32_t key_end;
    int32_t q_row0;      // first query row of the request
    int32_t rows;        // L: query rows of the request
    int32_t n_keys;      // N: keys of the request
    int32_t kv_head;
    int32_t pair0;       // first pair of the CTA
    int32_t part_base;   // < 0: write final rows; else partial slot of (row i, split s) is
                         // part_base + i * num_splits + s
    int32_t split;       // s
    int32_t num_splits;
    int32_t pad;
};
static_assert(sizeof(PrefillItem) == 48, "PrefillItem is 48 bytes");

// Warp tile (tokens one warp owns per pipeline stage) of the decode kernel.
__host__ __device__ constexpr int decode_warp_tile(int head_dim) { return head_dim == 64 ? 32 : 16; }
constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 3;
// The wide form of the tensor-core decode kernel: this many warps, one stage each, for
// slices of at most kDecodeWideWarps warp tiles (320 keys at head_dim 64, 160 at 128).
constexpr int kDecodeWideWarps = 10;

struct DecodeParams {
    const void *q;             // [rows, Hq, D]
    const WorkItem *items;
    const int32_t *kv_indices;
    int64_t num_pages;
    int page_size;
    int box_rows;              // rows per TMA box: min(page_size, warp tile)
    int num_qo_heads;
    float scale_log2;          // sm_scale * log2(e)
    void *out;                 // [rows, Hq, D] of out_dtype
    int out_dtype;             // pgqa_dtype
    float *lse;                // [rows, Hq] natural log, nullable
    float *partial_o;          // [slots, G, D]
    float *partial_lse;        // [slots, G] log2 domain
    unsigned int *flags;       // device flag word
    // fused append (all null for a plain run): new rows [rows, Hkv, D], one per query
    // row, and the pools as plain pointers for storing them
    const void *k_new;
    const void *v_new;
    void *k_pool;
    void *v_pool;
    int num_kv_heads;
    int prefetch_pool;         // 1: the pool rows (other than the new ones) are stable, so
                               // K/V loads may start before the grid-dependency wait
    int defer_wait;            // 1: launched right after an independent prefill grid of the same
                               // call; every older kernel is complete, so the dependency wait
                               // moves to the end (it only keeps completion order)
    const float2 *rope_cs;     // rotary (cos, sin) table [positions][D/2]; null: q and new rows
                               // are used as given
    uint32_t stall_wait_us;    // test hook of the per-item tensor-core kernel (0 = off): warp 0
                               // of every CTA withholds its first tile's copies and gives up
                               // waiting for them after this many microseconds
};

struct PrefillParams {
    const void *q;
    const PrefillItem *items;
    const int32_t *kv_indices;
    int64_t num_pages;
    int page_size;
    int box_rows;              // rows per TMA box: min(page_size, 64)
    int num_qo_heads;
    int num_kv_heads;
    int causal;                // bottom-right causal bound per row
    float scale_log2;
    void *out;
    int out_dtype;
    float *lse;
    unsigned int *flags;
    const void *k_new;         // fused append (nullable), as in DecodeParams
    const void *v_new;
    void *k_pool;
    void *v_pool;
    int prefetch_pool;
    float *partial_o;          // split prefill rows: [slots, G, D]
    float *partial_lse;        // [slots, G] log2 domain
    const float2 *rope_cs;     // as in DecodeParams
};

struct MergeParams {
    const MergeTask *tasks;
    const float *partial_o;    // [slots, G, D]
    const float *partial_lse;  // [slots, G] log2 domain
    void *out;
    int out_dtype;
    float *lse;
    int num_qo_heads;
    int group;                 // G
    int head_dim;
};

// Launchers (defined in the kernel translation units).  Decode: one CTA per work item.
cudaError_t launch_decode(int kind, int stages, int head_dim, int group, pgqa_dtype dtype, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, const DecodeParams &p, int num_items, bool pdl,
                          cudaStream_t stream);
cudaError_t launch_prefill(int kind, int head_dim, int group, pgqa_dtype dtype, const CUtensorMap &tm_k,
                           const CUtensorMap &tm_v, const PrefillParams &p, int num_items, bool pdl,
                           cudaStream_t stream);
cudaError_t launch_merge(const MergeParams &p, int num_tasks, int max_splits, bool pdl,
                         cudaStream_t stream);
cudaError_t launch_kv_append(void *k_pool, void *v_pool, const void *k, const void *v,
                             const int64_t *slot_mapping, int64_t num_tokens, int64_t num_slots,
                             int row_bytes, unsigned int *flags, bool pdl, cudaStream_t stream);
cudaError_t launch_rope_table(float2 *cs, int max_position, int head_dim, double theta, cudaStream_t stream);
cudaError_t launch_kv_append_rope(void *k_pool, void *v_pool, const void *k, const void *v,
                                  const int64_t *slot_mapping, const int32_t *positions, int64_t num_tokens,
                                  int64_t num_slots, int num_kv_heads, int head_dim, pgqa_dtype dtype,
                                  const float2 *cs, int max_position, unsigned int *flags, bool pdl,
                                  cudaStream_t stream);

// Host helpers defined in api.cu.
pgqa_status report(pgqa_status s, const char *msg);
pgqa_status report_cuda(cudaError_t e, const char *what);
pgqa_status current_device_flags(unsigned int **out);
pgqa_status encode_pool_map(CUtensorMap *map, const void *pool, int64_t num_pages, int page_size, int num_kv_heads,
                            int head_dim, pgqa_dtype dt, int box_rows, bool swizzle128);

// ---------------------------------------------------------------------------
// Device helpers (inline PTX)
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// One bounded probe of the barrier phase; the thread may sleep up to ~10 us inside
// it (suspend-time hint) instead of spinning, and wakes when the phase completes.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(10000u)
        : "memory");
    return ok != 0;
}

// Waits for the barrier phase with the given parity; gives up after about
// limit_ns nanoseconds and returns false (the caller raises
// PGQA_FLAG_WAIT_TIMEOUT instead of hanging).
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// The wait every pipeline barrier uses: ~2 s, far beyond any copy or product.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    return mbar_wait_limit(bar, parity, 2000000000ull);
}

// 3-D tiled TMA load into CTA shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// Same, with an L2 cache policy (K/V are streamed once per call: evict first).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                                 int c2, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// 3-D tiled box of a tensor map requested into L2 (no destination, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Page indices of a key slice, staged in shared memory by the whole CTA in one
// round trip so that TMA issue never waits on a dependent global load.
constexpr int kSlicePageCap = 512;

struct SlicePages {
    const int32_t *smem;       // [min(count, kSlicePageCap)]
    const int32_t *global;     // kv_indices + page_base
    int first;                 // page number (within the request) of smem[0]
    __device__ __forceinline__ int64_t operator()(int tok, int page_size) const {
        const int i = tok / page_size - first;
        return i < kSlicePageCap ? smem[i] : global[first + i];
    }
};

__device__ __forceinline__ SlicePages stage_slice_pages(int32_t *buf, const int32_t *kv_indices, int page_base,
                                                       int tok_begin, int tok_end, int page_size) {
    SlicePages sp;
    sp.first = tok_begin / page_size;
    sp.global = kv_indices + page_base;
    sp.smem = buf;
    const int n = tok_end > tok_begin ? (tok_end - 1) / page_size - sp.first + 1 : 0;
    const int m = n < kSlicePageCap ? n : kSlicePageCap;
    for (int i = threadIdx.x; i < m; i += blockDim.x) buf[i] = __ldg(sp.global + sp.first + i);
    return sp;  // caller synchronises the CTA before use
}

// Bulk prefetch of [ptr, ptr + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void *ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(ptr)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's memory, and let
// the next grid start its prologue early.  No-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Hardware approximations (PTX ex2/lg2/rcp .approx): a few ulp, ample for the
// softmax weights and the log-sum-exp.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Named barrier 1 over `count` threads: producers arrive, the consumer waits.
__device__ __forceinline__ void named_bar_arrive(int count) {
    asm volatile("bar.arrive 1, %0;" ::"r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_sync(int count) {
    asm volatile("bar.sync 1, %0;" ::"r"(count) : "memory");
}
// Named barrier with a compile-time id (a runtime id would reserve all sixteen).
template <int ID>
__device__ __forceinline__ void named_bar_arrive_c(int count) {
    asm volatile("bar.arrive %0, %1;" ::"n"(ID), "r"(count) : "memory");
}
template <int ID>
__device__ __forceinline__ void named_bar_sync_c(int count) {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_arrive_id(int id, int count) {
    switch (id) {
        case 1: named_bar_arrive_c<1>(count); break;
        case 2: named_bar_arrive_c<2>(count); break;
        case 3: named_bar_arrive_c<3>(count); break;
        default: named_bar_arrive_c<4>(count); break;
    }
}
__device__ __forceinline__ void named_bar_sync_id(int id, int count) {
    switch (id) {
        case 1: named_bar_sync_c<1>(count); break;
        case 2: named_bar_sync_c<2>(count); break;
        case 3: named_bar_sync_c<3>(count); break;
        default: named_bar_sync_c<4>(count); break;
    }
}

// 16-byte shared-memory load through a plain C++ access, so the compiler orders
// it against __syncwarp and the barrier waits (which clobber memory).
__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// The work item of this CTA into registers with three 16-byte loads that stay where
// they are written.  A plain struct copy lets the compiler read each field at its first
// use; a field first used after griddepcontrol.wait (a memory clobber) is then read
// from global memory again there, putting a dependent load on the critical path.
__device__ __forceinline__ WorkItem load_work_item(const WorkItem *src) {
    static_assert(sizeof(WorkItem) == 48, "three 16-byte loads");
    int32_t w[12];
    const char *b = reinterpret_cast<const char *>(src);
#pragma unroll
    for (int k = 0; k < 3; ++k)
        asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[4 * k]), "=r"(w[4 * k + 1]), "=r"(w[4 * k + 2]), "=r"(w[4 * k + 3])
                     : "l"(b + 16 * k));
    WorkItem it;
    it.page_base = w[0];
    it.tok_begin = w[1];
    it.tok_end = w[2];
    it.q_row = w[3];
    it.kv_head = w[4];
    it.out_slot = w[5];
    it.new_begin = w[6];
    it.new_row_base = w[7];
    it.write_pos = w[8];
    it.q_pos = w[9];
    it.pad1 = w[10];
    it.pad2 = w[11];
    return it;
}

// A 16-byte shared-memory load the compiler keeps where it is written (not hoisted out
// of the branch or loop that holds it).
__device__ __forceinline__ float4 lds128_pinned(const void *p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Two packed 16-bit floats -> two fp32 (exact widening).
template <typename T>
__device__ __forceinline__ float2 widen2(uint32_t packed);

template <>
__device__ __forceinline__ float2 widen2<__nv_bfloat16>(uint32_t packed) {
    // bf16 is the upper half of an fp32: shift the low element up, mask the high one.
    return make_float2(__uint_as_float(packed << 16), __uint_as_float(packed & 0xffff0000u));
}

template <>
__device__ __forceinline__ float2 widen2<__half>(uint32_t packed) {
    __half2 h = *reinterpret_cast<__half2 *>(&packed);
    return __half22float2(h);
}

template <typename T>
__device__ __forceinline__ T narrow(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 narrow<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half narrow<__half>(float x) { return __float2half_rn(x); }

// Two values rounded to T (nearest, ties to even) and packed, the first in the low half.
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
           (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
}

// Rotary embedding, rotate-half form: channel i < D/2 pairs with channel i + D/2 and
// both turn by the angle whose (cos, sin) is entry i of the position's table row:
//     lo' = lo cos - hi sin,   hi' = hi cos + lo sin,
// in fp32 and rounded once to T.  lo packs channels i, i + 1; hi packs i + D/2,
// i + D/2 + 1; cs = (cos_i, sin_i, cos_i+1, sin_i+1).  Every path that rotates a row
// (q in registers, new K rows patched into tiles or stored into the pool) goes
// through this one function, so a stored key matches the one attended bit for bit.
template <typename T>
__device__ __forceinline__ void rope_rotate2(uint32_t &lo, uint32_t &hi, float4 cs) {
    const float2 a = widen2<T>(lo), b = widen2<T>(hi);
    const float a0 = fmaf(a.x, cs.x, -__fmul_rn(b.x, cs.y));
    const float a1 = fmaf(a.y, cs.z, -__fmul_rn(b.y, cs.w));
    const float b0 = fmaf(b.x, cs.x, __fmul_rn(a.x, cs.y));
    const float b1 = fmaf(b.y, cs.z, __fmul_rn(a.y, cs.w));
    lo = pack2<T>(a0, a1);
    hi = pack2<T>(b0, b1);
}

// 16-byte chunk `ch` (channels 8 ch .. 8 ch + 7) of the D-channel row at `row` with the
// rotary embedding of table row `cs` applied; reads the chunk and its partner in the
// other half.
template <typename T, int D>
__device__ __forceinline__ uint4 rope_chunk(const T *row, int ch, const float2 *cs) {
    constexpr int HC = D / 16;  // chunks per half
    const bool second = ch >= HC;
    const int first = second ? ch - HC : ch;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(row + first * 8));
    const uint4 y = __ldg(reinterpret_cast<const uint4 *>(row + (first + HC) * 8));
    const float4 *c = reinterpret_cast<const float4 *>(cs + first * 8);
    uint32_t lo[4] = {x.x, x.y, x.z, x.w}, hi[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) rope_rotate2<T>(lo[j], hi[j], __ldg(c + j));
    return second ? make_uint4(hi[0], hi[1], hi[2], hi[3]) : make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

#endif  // __CUDACC__

}  // namespace pgqa
