// Split-KV decode for callers that cannot allocate device memory.
//
// Some callers of this code cannot call cudaMalloc: processes whose device memory
// is reserved up front and handed out by another allocator (a framework's caching
// allocator or an arena sized at start-up), where an allocation outside it fails
// or fragments that reserve; and embedded or real-time hosts that forbid
// allocation after initialisation, because cudaMalloc and cudaFree may block or
// synchronise the device at unpredictable times.  For them,
// pgqa_decode_static_scratch runs the same decode path (the tensor-core partial
// kernel and the log-sum-exp merge) with every intermediate buffer -- the work
// list, the merge list and the split partials -- carved out of one file-scope
// device array.  The caller passes only inputs and outputs.
//
// The array lives as long as the library is loaded, on every device that loads
// it.  Its device address is looked up once per device (cudaGetSymbolAddress,
// with that device current) on the first call there; that first call should
// therefore happen before any stream capture.  Every call shares the array, so
// two calls whose kernels overlap on the GPU (different streams, no ordering)
// race on it.  Nothing in it has to start at zero: each call writes its work
// list and partials before reading them.
#include <climits>
#include <mutex>

#include <cmath>

#include "common.cuh"

namespace pgqa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch for the current device (looked up once).
pgqa_status static_scratch_ptr(unsigned char **out) {
    static std::mutex mu;
    static unsigned char *ptrs[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= 256) return report(PGQA_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return report_cuda(e, "cudaGetSymbolAddress(static scratch)");
        ptrs[dev] = static_cast<unsigned char *>(p);
    }
    *out = ptrs[dev];
    return PGQA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// One thread per (request, kv head, slice): an even cut of the request's keys
// into `splits` slices of whole warp tiles, read from the device page table.
// The table is checked here, where it is first read: a request whose page range
// [kv_indptr[b], kv_indptr[b+1]) is negative, decreasing or reaches past the
// num_indices entries of kv_indices, or that has no pages but a non-zero
// last_page_len, raises PGQA_FLAG_PAGE_INDEX and gets no keys, so no kernel reads
// kv_indices outside [0, num_indices).  A last_page_len outside [1, page_size]
// for a request with pages is clamped and raises the same flag.
__global__ void build_static_work(const int32_t *__restrict__ kv_indptr, const int32_t *__restrict__ last_page_len,
                                  int64_t num_indices, int batch, int num_kv_heads, int splits, int page_size,
                                  int tile, WorkItem *items, MergeTask *tasks, unsigned int *flags) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int total = batch * num_kv_heads * splits;
    if (i >= total) return;
    const int s = i % splits;
    const int t = i / splits;
    const int kvh = t % num_kv_heads;
    const int b = t / num_kv_heads;
    const int p0 = kv_indptr[b], p1 = kv_indptr[b + 1];
    int last = last_page_len[b];
    bool bad = p0 < 0 || p1 < p0 || static_cast<int64_t>(p1) > num_indices;
    const int np = bad ? 0 : p1 - p0;
    if (np == 0 && last != 0) bad = true;  // no pages means no keys: last_page_len must be 0
    int n = 0;
    if (!bad && np > 0) {
        if (last < 1 || last > page_size) {
            if (s == 0 && kvh == 0) atomicOr(flags, PGQA_FLAG_PAGE_INDEX);
            last = last < 1 ? 1 : page_size;
        }
        const int64_t n64 = static_cast<int64_t>(np - 1) * page_size + last;
        if (n64 > INT_MAX / 2)
            bad = true;  // a key count the 32-bit slice bounds cannot hold
        else
            n = static_cast<int>(n64);
    }
    if (bad && s == 0 && kvh == 0) atomicOr(flags, PGQA_FLAG_PAGE_INDEX);
    const int per = (n + splits - 1) / splits;
    const int len = ((per + tile - 1) / tile) * tile;
    const int tb = min(n, s * len);
    const int te = min(n, (s + 1) * len);
    WorkItem w;
    w.page_base = bad ? 0 : p0;
    w.tok_begin = tb;
    w.tok_end = te;
    w.q_row = b;
    w.kv_head = kvh;
    w.out_slot = splits == 1 ? -1 : i;
    w.new_begin = INT_MAX;
    w.new_row_base = 0;
    w.write_pos = -1;
    w.q_pos = n > 0 ? n - 1 : 0;  // unused: this entry point has no rotary embedding
    w.pad1 = w.pad2 = 0;
    items[i] = w;
    if (s == 0 && splits > 1) tasks[t] = MergeTask{b, kvh, t * splits, splits};
}

}  // namespace
}  // namespace pgqa

using namespace pgqa;

extern "C" PGQA_API pgqa_status pgqa_decode_static_scratch(const void *q, const void *k_pool, const void *v_pool,
                                                  const int32_t *kv_indptr, const int32_t *kv_indices,
                                                  int64_t num_indices, const int32_t *last_page_len, int batch,
                                                  int64_t num_pages,
                                                  int page_size, int num_qo_heads, int num_kv_heads, int head_dim,
                                                  pgqa_dtype dtype, int splits, void *out, pgqa_dtype out_dtype,
                                                  float *lse, float sm_scale, pgqa_stream_t stream) {
    if (batch < 0 || num_pages < 0 || num_indices < 0)
        return report(PGQA_ERR_INVALID_ARG, "negative batch, num_pages or num_indices");
    if (num_kv_heads < 1 || num_qo_heads < 1 || num_qo_heads % num_kv_heads != 0)
        return report(PGQA_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads");
    const int group = num_qo_heads / num_kv_heads;
    if (group > 8) return report(PGQA_ERR_UNSUPPORTED, "more than 8 query heads per kv head");
    if (head_dim != 64 && head_dim != 128) return report(PGQA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128 && page_size != 256)
        return report(PGQA_ERR_UNSUPPORTED, "page_size must be 16, 32, 64, 128 or 256");
    if (dtype != PGQA_BF16 && dtype != PGQA_FP16) return report(PGQA_ERR_UNSUPPORTED, "dtype must be bf16 or fp16");
    if (out_dtype != PGQA_FP32 && out_dtype != dtype)
        return report(PGQA_ERR_UNSUPPORTED, "out_dtype must be fp32 or the input dtype");
    if (splits < 1 || splits > 256) return report(PGQA_ERR_INVALID_ARG, "splits must be in [1, 256]");
    if (num_pages * static_cast<int64_t>(page_size) >= (int64_t(1) << 31))
        return report(PGQA_ERR_UNSUPPORTED, "pool rows must stay below 2^31");
    if (batch == 0) return PGQA_OK;
    // kv_indices may be NULL only when it has no entries (every request then has no keys).
    if (!q || !k_pool || !v_pool || !kv_indptr || !last_page_len || !out || (!kv_indices && num_indices > 0))
        return report(PGQA_ERR_INVALID_ARG, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool) |
         reinterpret_cast<uintptr_t>(out)) & 15u)
        return report(PGQA_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned");

    // Scratch layout: work items | merge tasks | partial outputs | partial lse.  The
    // request count is bounded first, so that the sizes below cannot wrap.
    const uint64_t max_items = kStaticScratchBytes / sizeof(WorkItem);
    const uint64_t pairs = static_cast<uint64_t>(batch) * static_cast<uint64_t>(num_kv_heads);  // < 2^62
    if (pairs > max_items || pairs * static_cast<uint64_t>(splits) > max_items)
        return report(PGQA_ERR_CAPACITY,
                      "batch x kv heads x splits needs more than the 8 MiB static scratch; lower splits or batch");
    const size_t n_items = static_cast<size_t>(batch) * num_kv_heads * splits;
    const size_t n_tasks = static_cast<size_t>(batch) * num_kv_heads;
    const size_t items_bytes = align256(n_items * sizeof(WorkItem));
    const size_t tasks_bytes = align256(n_tasks * sizeof(MergeTask));
    const size_t po_bytes = align256(n_items * group * head_dim * sizeof(float));
    const size_t pl_bytes = align256(n_items * group * sizeof(float));
    if (items_bytes + tasks_bytes + po_bytes + pl_bytes > kStaticScratchBytes)
        return report(PGQA_ERR_CAPACITY,
                      "batch x kv heads x splits needs more than the 8 MiB static scratch; lower splits or batch");

    unsigned char *scratch = nullptr;
    pgqa_status st = static_scratch_ptr(&scratch);
    if (st != PGQA_OK) return st;
    unsigned int *flags = nullptr;
    st = current_device_flags(&flags);
    if (st != PGQA_OK) return st;
    WorkItem *items = reinterpret_cast<WorkItem *>(scratch);
    MergeTask *tasks = reinterpret_cast<MergeTask *>(scratch + items_bytes);
    float *partial_o = reinterpret_cast<float *>(scratch + items_bytes + tasks_bytes);
    float *partial_lse = reinterpret_cast<float *>(scratch + items_bytes + tasks_bytes + po_bytes);

    const int tile = decode_warp_tile(head_dim);
    const int box_rows = page_size < tile ? page_size : tile;
    CUtensorMap mk, mv;
    st = encode_pool_map(&mk, k_pool, num_pages, page_size, num_kv_heads, head_dim, dtype, box_rows, true);
    if (st == PGQA_OK) st = encode_pool_map(&mv, v_pool, num_pages, page_size, num_kv_heads, head_dim, dtype, box_rows, true);
    if (st != PGQA_OK) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int total = static_cast<int>(n_items);
    build_static_work<<<(total + 127) / 128, 128, 0, s>>>(kv_indptr, last_page_len, num_indices, batch, num_kv_heads,
                                                          splits, page_size, tile, items, tasks, flags);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return report_cuda(e, "static work-list launch");

    DecodeParams p{};
    p.q = q;
    p.items = items;
    p.kv_indices = kv_indices;
    p.num_pages = num_pages;
    p.page_size = page_size;
    p.box_rows = box_rows;
    p.num_qo_heads = num_qo_heads;
    p.scale_log2 = (sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(head_dim))) * 1.4426950408889634f;
    p.out = out;
    p.out_dtype = out_dtype;
    p.lse = lse;
    p.partial_o = partial_o;
    p.partial_lse = partial_lse;
    p.flags = flags;
    p.num_kv_heads = num_kv_heads;
    // The work list was just written by a kernel: launch without programmatic
    // overlap so the decode kernel starts only after it is complete.
    e = launch_decode(PGQA_DECODE_TENSOR_CORE, 2, head_dim, group, dtype, mk, mv, p, total, false, s);
    if (e != cudaSuccess) return report_cuda(e, "decode launch");
    if (splits > 1) {
        MergeParams mp{};
        mp.tasks = tasks;
        mp.partial_o = partial_o;
        mp.partial_lse = partial_lse;
        mp.out = out;
        mp.out_dtype = out_dtype;
        mp.lse = lse;
        mp.num_qo_heads = num_qo_heads;
        mp.group = group;
        mp.head_dim = head_dim;
        e = launch_merge(mp, static_cast<int>(n_tasks), splits, false, s);
        if (e != cudaSuccess) return report_cuda(e, "merge launch");
    }
    return PGQA_OK;
}
