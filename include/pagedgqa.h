/*
 * pagedgqa.h -- C ABI of the GB300 (sm_103a) paged GQA split-KV decode library.
 *
 * Decode attention over a paged KV cache with grouped-query heads: each query
 * row (Hq heads, Hq/Hkv of them sharing each KV head) attends over its
 * request's cached keys/values, which sit in fixed-size pages of a pool and are
 * found through a CSR page table.  Work is split along each request's history
 * ("split-KV"); a partial (output, log-sum-exp) is computed per slice in
 * parallel and the partials are merged.  A paged KV append writes new tokens'
 * rows into the pool.  A ragged call also serves requests with several query
 * rows (a chunked prefill): their rows attend causally, bottom-right aligned.
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless the parameter name ends in _host.
 *     The caller owns every buffer it passes; the library never frees them.
 *   - All work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream).  No entry point synchronises the device unless it says so.
 *   - Errors are returned as pgqa_status; nothing traps or aborts.  A failed
 *     call enqueues no work.  pgqa_last_error() gives a one-line reason
 *     (thread-local, valid until the next failing call on the same thread).
 *   - Layouts are row-major and contiguous:
 *       KV pool   [num_pages, page_size, num_kv_heads, head_dim]  (one for K, one for V)
 *       q, out    [total_q_rows, num_qo_heads, head_dim]
 *       lse       [total_q_rows, num_qo_heads]  fp32, natural log
 *   - Query head h reads KV head h / (num_qo_heads / num_kv_heads).
 *   - Supported shapes: head_dim 64 or 128; page_size 16, 32, 64, 128 or 256;
 *     num_qo_heads / num_kv_heads between 1 and 16 (1 and 8 for the CUDA-core
 *     decode kernel and pgqa_decode_static_scratch); bf16 or fp16 q/k/v.
 *     Anything else returns PGQA_ERR_UNSUPPORTED.
 *   - Pool, q, k, v and out pointers must be 16-byte aligned.
 */
#ifndef PAGEDGQA_H
#define PAGEDGQA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PGQA_ABI_VERSION 5

#if defined(__GNUC__)
#define PGQA_API __attribute__((visibility("default")))
#else
#define PGQA_API
#endif

/* Same object as cudaStream_t; declared here so callers need no CUDA headers. */
typedef struct CUstream_st *pgqa_stream_t;

typedef enum pgqa_status {
    PGQA_OK = 0,
    PGQA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, negative size, ... */
    PGQA_ERR_UNSUPPORTED = 2,    /* shape or dtype outside the supported set */
    PGQA_ERR_BAD_PAGE_TABLE = 3, /* page table rejected by the host-side check */
    PGQA_ERR_CUDA = 4,           /* a CUDA runtime call failed */
    PGQA_ERR_CAPACITY = 5,       /* request exceeds the plan's configured capacity */
    PGQA_ERR_DEVICE_CHECK = 6    /* a device-side bounds check fired (see pgqa_read_device_flags) */
} pgqa_status;

typedef enum pgqa_dtype { PGQA_BF16 = 0, PGQA_FP16 = 1, PGQA_FP32 = 2 } pgqa_dtype;

/* Bits of the per-device flag word that kernels set instead of trapping. */
#define PGQA_FLAG_PAGE_INDEX 1u   /* a page index >= num_pages was skipped */
#define PGQA_FLAG_SLOT_RANGE 2u   /* an append slot >= num_pages * page_size was skipped */
#define PGQA_FLAG_WAIT_TIMEOUT 4u /* a pipeline barrier wait gave up (bounded spin) */
#define PGQA_FLAG_SMEM_ALIGN 8u   /* shared memory too coarsely aligned for the TMA layout; CTA skipped */
#define PGQA_FLAG_ROPE_POSITION 16u /* a rotary position outside [0, rope_max_position) was skipped */

PGQA_API int pgqa_abi_version(void);
PGQA_API const char *pgqa_status_string(pgqa_status status);
PGQA_API const char *pgqa_last_error(void);

/*
 * Reads (and with clear != 0 resets) the flag word of the current device.
 * Synchronises the device.  Returns PGQA_ERR_DEVICE_CHECK when any flag is set.
 */
PGQA_API pgqa_status pgqa_read_device_flags(uint32_t *flags_host, int clear);

/*
 * pgqa_kv_append -- paged KV append.
 *
 * Defined by the "flashlet" README, design bullets: the pool is laid out
 * [pages, page_size, kv_heads, head_dim] (FlashInfer's NHD) so that writing new
 * tokens is a single index copy of their rows into flat slots.
 *
 *   k_pool, v_pool  pools [num_pages, page_size, num_kv_heads, head_dim], dtype
 *   k, v            new rows [num_tokens, num_kv_heads, head_dim], dtype
 *   slot_mapping    [num_tokens] int64, device; row t goes to flat slot
 *                   slot_mapping[t] = page * page_size + offset.  A negative
 *                   slot skips the row (padding).  A slot >= num_pages*page_size
 *                   is skipped and raises PGQA_FLAG_SLOT_RANGE.  Two rows with
 *                   the same slot in one call race (undefined which one lands).
 * num_kv_heads is 1 .. 2^20 (PGQA_ERR_UNSUPPORTED above).  The copy is
 * bit-exact.  num_tokens == 0 enqueues nothing.
 */
PGQA_API pgqa_status pgqa_kv_append(void *k_pool, void *v_pool, int64_t num_pages, int page_size,
                           int num_kv_heads, int head_dim, pgqa_dtype dtype,
                           const void *k, const void *v, const int64_t *slot_mapping,
                           int64_t num_tokens, pgqa_stream_t stream);

/* ------------------------------------------------------------------------- */
/* plan / run                                                                */
/* ------------------------------------------------------------------------- */

/*
 * The plan()/run() split follows the "flashlet" README (backends/base.py:
 * AttentionBackend ABC with plan() / run(); design bullets: metadata in
 * persistent device buffers updated in place each step).  A plan owns device
 * buffers sized once at creation (work list, merge list, split partials), so
 * their addresses never change and run() can be captured in a CUDA graph.  A
 * captured run() also fixes its launch sizes and kernel variants (the counts of
 * slices, merges and prefill tiles, which pgqa_plan_get_info reports, and the
 * pipeline depth): replay it after a pgqa_plan_update only when the update
 * describes the same schedule, and capture again otherwise.
 */
typedef struct pgqa_plan pgqa_plan;

typedef struct pgqa_plan_config {
    int num_qo_heads;     /* Hq */
    int num_kv_heads;     /* Hkv; Hq % Hkv == 0 */
    int head_dim;         /* 64 or 128 */
    int page_size;        /* 16, 32, 64, 128 or 256 */
    pgqa_dtype dtype;     /* q/k/v element type: PGQA_BF16 or PGQA_FP16 */
    int max_batch;        /* most requests one plan_update may describe */
    int64_t max_q_rows;   /* most query rows one run may carry (decode + prefill rows) */
    int max_splits;       /* cap on slices per (request, kv head); 0 = no cap; 1 = never split */
    int split_tokens;     /* > 0 forces this slice length (rounded up to the kernel tile);
                             0 = choose it so that the slices fill the SMs */
    int ctas_per_sm;      /* CTA slots per SM assumed by the split heuristic; 0 = the decode
                             kernel's resident CTAs per SM, at most 2 */
    int decode_kernel;    /* PGQA_DECODE_AUTO (tensor cores), PGQA_DECODE_TENSOR_CORE or
                             PGQA_DECODE_CUDA_CORE (fp32 FMA; kept as a measured alternative) */
    int pipeline_stages;  /* tensor-core kernel: shared-memory stages per warp, 2 or 3, or 1 for
                             the wide form (ten warps of one tile each, for slices of at most
                             ten warp tiles and groups of up to 8 heads); 0 = chosen per
                             plan_update: 1 when every slice fits the wide form, 3 when a
                             whole slice fits in flight, or when a grid of long slices is
                             less than one wave at two CTAs per SM and no prefill segment
                             shares the call; else 2 */
    int prefill_splits;   /* key slices per prefill tile (1..8); 0 = as many as fit one wave */
    int rope_max_position; /* RoPE plans: positions 0 .. rope_max_position - 1 are valid */
    double rope_theta;    /* > 0: rotary position embedding with this base (see below);
                             0: none */
    int prefill_kernel;   /* requests with several query rows: PGQA_PREFILL_TCGEN05 (5th-
                             generation tensor cores, S and O in tensor memory) or
                             PGQA_PREFILL_MMA_SYNC; PGQA_PREFILL_AUTO takes tcgen05, the
                             faster one on GB300 at every shape measured */
    int test_stall_wait_us; /* 0 for normal use.  A test of the failure path, 1..1000000:
                             in every CTA of the tensor-core decode kernel one warp
                             withholds the copies of its first tile, waits that many
                             microseconds for them, gives up, raises
                             PGQA_FLAG_WAIT_TIMEOUT and ends with the CTA (whose output
                             is then meaningless), instead of hanging.  Only that
                             kernel's per-item schedule honours it. */
} pgqa_plan_config;

#define PGQA_PREFILL_AUTO 0
#define PGQA_PREFILL_TCGEN05 1
#define PGQA_PREFILL_MMA_SYNC 2

/*
 * Rotary position embedding (RoPE).  The "flashlet" README lists a RoPE fusion
 * kernel among its milestones and "Torchlet"'s Qwen2.5-style model includes
 * RoPE; neither writes it out.  It is taken in the rotate-half form of the
 * Qwen2.5 models: for i < head_dim/2, channels i and i + head_dim/2 turn by
 * phi = pos * rope_theta^(-2i/head_dim):
 *     x'[i]            = x[i] cos(phi) - x[i + head_dim/2] sin(phi)
 *     x'[i + head_dim/2] = x[i + head_dim/2] cos(phi) + x[i] sin(phi).
 * A plan with rope_theta > 0 builds a (cos, sin) table of rope_max_position
 * rows (fp64 angles rounded to fp32; head_dim * 4 bytes per row) once in
 * pgqa_plan_create, and then:
 *   - pgqa_run and pgqa_append_run take q BEFORE rotation: each query row is
 *     rotated at its position, the key position of its own token (a request
 *     with N keys and L query rows has them at N - L .. N - 1);
 *   - pgqa_append_run takes k_new before rotation and stores (and attends) it
 *     rotated at its key position; v_new is not rotated;
 *   - the pool holds rotated keys (pgqa_kv_append_rope writes them).
 * The rotation runs in fp32 and rounds once to the plan's dtype (nearest, ties
 * to even).  plan_update rejects a request whose query rows outnumber its keys
 * or whose keys reach past rope_max_position (PGQA_ERR_INVALID_ARG).  RoPE
 * plans need the tensor-core kernels (PGQA_ERR_UNSUPPORTED with
 * PGQA_DECODE_CUDA_CORE) and run one CTA per work item.
 */

#define PGQA_DECODE_AUTO 0
#define PGQA_DECODE_TENSOR_CORE 1
#define PGQA_DECODE_CUDA_CORE 2

/*
 * Creates a plan on the current device.  Allocates its device and pinned host
 * buffers (the only allocations the library makes) and, for a RoPE plan, builds
 * its rotary table (synchronously).  *plan is set to NULL on failure.  Its lists
 * are sized from max_q_rows, max_batch and num_kv_heads; a plan whose work list
 * or prefill-tile list would pass 2^26 entries is refused (PGQA_ERR_CAPACITY).
 */
PGQA_API pgqa_status pgqa_plan_create(pgqa_plan **plan, const pgqa_plan_config *cfg);

/*
 * pgqa_kv_append_rope -- paged KV append with the plan's rotary embedding on K.
 *
 * The append of pgqa_kv_append (the "flashlet" README, design bullets: one copy
 * of each new token's row into its flat slot) with each K row rotated at
 * positions[t] on the way (the RoPE fusion of the "flashlet" README's
 * milestones; the rotation is the one described above).  Shapes, dtype,
 * head_dim and num_kv_heads are the plan's.
 *
 *   k_pool, v_pool  pools [num_pages, page_size, num_kv_heads, head_dim]
 *   k, v            new rows [num_tokens, num_kv_heads, head_dim], k before rotation
 *   slot_mapping    [num_tokens] int64, device: as in pgqa_kv_append
 *   positions       [num_tokens] int32, device: the token's position; a
 *                   position outside [0, rope_max_position) skips the row (K
 *                   and V) and raises PGQA_FLAG_ROPE_POSITION
 * Enqueued on `stream`; ordered after the stream's previous kernel.
 * Errors: PGQA_ERR_INVALID_ARG for a plan without RoPE, NULL or misaligned
 * pointers, negative sizes.
 */
PGQA_API pgqa_status pgqa_kv_append_rope(const pgqa_plan *plan, void *k_pool, void *v_pool, int64_t num_pages,
                                         const void *k, const void *v, const int64_t *slot_mapping,
                                         const int32_t *positions, int64_t num_tokens, pgqa_stream_t stream);

/*
 * pgqa_plan_update -- plan().
 *
 * Split-KV as in "A library kernel for decode", section "What changed": each
 * request's cached keys are cut into slices, one partial per slice is computed
 * in parallel and the partials are merged, so one request's history spreads
 * over many SMs.  The slice length is chosen here, from the kv lengths, so
 * that the slices of all requests fill the GPU's SMs.
 *
 *   kv_indptr_host      [batch+1] int32, host; pages of request b are
 *                       kv_indices[kv_indptr[b] .. kv_indptr[b+1])
 *   last_page_len_host  [batch] int32, host; rows used in the request's last
 *                       page, in [1, page_size], or 0 for a request with no pages.
 *                       kv_len(b) = (npages - 1) * page_size + last_page_len[b].
 *   qo_indptr_host      [batch+1] int32, host, or NULL.  NULL: request b owns
 *                       exactly query row b (pure decode).  Otherwise request b
 *                       owns rows qo_indptr[b] .. qo_indptr[b+1] (the ragged
 *                       form of the "flashlet" README, design bullets:
 *                       qo_indptr lengths [512, 1, 1, ...] in one call).
 *   kv_indices          [kv_indptr[batch]] int32, DEVICE; its final contents must
 *                       be in place (in stream order) when plan_update is called,
 *                       and it must stay valid and unchanged until the last run()
 *                       that uses this plan (the kernels read it before waiting
 *                       on the preceding kernel).
 *   kv_indices_host     optional host mirror of kv_indices (NULL allowed).  When
 *                       given, every index is checked here against num_pages;
 *                       when not, the kernels skip out-of-range pages and raise
 *                       PGQA_FLAG_PAGE_INDEX.
 *   num_pages           pages in each pool
 *   causal              for rows of a request with L query rows over N keys, row
 *                       i may attend keys j <= N - L + i (bottom-right).  It has
 *                       no effect on single-row (decode) requests.
 * The host arrays are read before the call returns.  One asynchronous copy of
 * the work list into the plan's device buffer is enqueued on `stream`; a
 * run() on another stream must be ordered after it by the caller.
 * Errors: PGQA_ERR_BAD_PAGE_TABLE (non-monotone indptr or qo_indptr,
 * last_page_len out of range, index out of range when a host mirror is
 * given), PGQA_ERR_CAPACITY (batch, rows or work items beyond the configured
 * maxima).
 */
PGQA_API pgqa_status pgqa_plan_update(pgqa_plan *plan, const int32_t *kv_indptr_host,
                             const int32_t *last_page_len_host, const int32_t *qo_indptr_host,
                             int batch, const int32_t *kv_indices,
                             const int32_t *kv_indices_host, int64_t num_pages, int causal,
                             pgqa_stream_t stream);

/*
 * pgqa_run -- run(): attention for every query row of the last plan_update.
 *
 *   q          [total_q_rows, Hq, head_dim], the plan's dtype
 *   k_pool     [num_pages, page_size, Hkv, head_dim], the plan's dtype
 *   v_pool     same shape
 *   out        [total_q_rows, Hq, head_dim] of out_dtype (the plan's dtype or PGQA_FP32)
 *   lse        [total_q_rows, Hq] fp32 natural-log log-sum-exp of the scaled
 *              scores, or NULL.  A row with no key gets out = 0, lse = -inf.
 *   sm_scale   score scale; <= 0 selects 1/sqrt(head_dim)
 * Launches the split-KV partial kernel and, when some row was split, the
 * merge kernel.  Outputs are bit-for-bit repeatable for the same plan and inputs.
 */
PGQA_API pgqa_status pgqa_run(pgqa_plan *plan, const void *q, const void *k_pool, const void *v_pool,
                     void *out, pgqa_dtype out_dtype, float *lse, float sm_scale,
                     pgqa_stream_t stream);

/*
 * pgqa_append_run -- kv_append and run() of one decode (or prefill) step in one launch.
 *
 * The paged append of the "flashlet" README's design bullets (new tokens' rows
 * copied into their slots), folded into the attention call that reads them:
 * request b's last qo_len(b) key positions (qo_len = its query rows; 1 for pure
 * decode) take their K/V rows from k_new / v_new rows qo_indptr[b] ..
 * qo_indptr[b+1] (row b when the plan has no qo_indptr).  The kernel uses those
 * rows directly for the attention and also stores them into their pool slots,
 * which the page table must already cover (kv_len counts the new tokens).
 * Other arguments and the result are those of pgqa_run.
 *
 *   k_new, v_new  [total_q_rows, num_kv_heads, head_dim], the plan's dtype; both NULL
 *                 for a step without new rows (pgqa_run with `flags`)
 *   k_pool, v_pool  written (new rows only) and read
 *   flags         0, or PGQA_RUN_POOL_STABLE: no kernel still running when this
 *                 call's kernel starts writes any pool row this call reads
 *                 (other than the new rows).  The K/V loads then begin before
 *                 the kernel waits for its predecessor on the stream, hiding the
 *                 memory latency behind that kernel's tail.  A kernel that wrote
 *                 those rows and is the immediate predecessor voids the promise.
 * Errors: as pgqa_run; with new rows, PGQA_ERR_UNSUPPORTED for a plan created
 * with PGQA_DECODE_CUDA_CORE and PGQA_ERR_INVALID_ARG when a request has more
 * query rows than keys; PGQA_ERR_INVALID_ARG when only one of k_new, v_new is
 * NULL.
 */
#define PGQA_RUN_POOL_STABLE 1

PGQA_API pgqa_status pgqa_append_run(pgqa_plan *plan, const void *k_new, const void *v_new, const void *q,
                                     void *k_pool, void *v_pool, void *out, pgqa_dtype out_dtype, float *lse,
                                     float sm_scale, int flags, pgqa_stream_t stream);

/*
 * pgqa_decode_static_scratch -- split-KV decode that allocates nothing.
 *
 * None of the pages has a counterpart to this call.  It serves callers of this
 * library that cannot allocate device memory: processes whose device memory is
 * reserved up front and handed out by another allocator (a framework's caching
 * allocator, an arena sized at start-up), where an allocation outside that
 * reserve fails or fragments it; and embedded or real-time hosts that forbid
 * allocation after initialisation, since cudaMalloc and cudaFree may block or
 * synchronise the device at unpredictable times.  It needs no plan: the slices
 * are cut on the device from the device-side page table, and the work list,
 * merge list and split partials live in one 8 MiB array inside the library (a
 * static device array, held by every GPU that loads the library until the
 * process exits).  No cudaMalloc, cudaFree or allocating library routine is
 * called.
 *
 *   q            [batch, num_qo_heads, head_dim]: one decode row per request
 *   k_pool/v_pool  as for pgqa_run
 *   kv_indptr    [batch+1] int32, DEVICE
 *   kv_indices   [num_indices] int32, DEVICE; may be NULL when num_indices is 0
 *   num_indices  entries of kv_indices.  The table is checked on the device
 *                where it is first read: a request whose page range
 *                [kv_indptr[b], kv_indptr[b+1]) is negative, decreasing or
 *                reaches past num_indices, or that has no pages but a non-zero
 *                last_page_len, gets no keys (out = 0, lse = -inf) and raises
 *                PGQA_FLAG_PAGE_INDEX; kv_indices is never read outside
 *                [0, num_indices).  Page indices >= num_pages are skipped and
 *                raise the same flag.
 *   last_page_len [batch] int32, DEVICE (values outside [1, page_size] for a
 *                request with pages are clamped and raise PGQA_FLAG_PAGE_INDEX)
 *   splits       slices per (request, kv head), 1..256 (1 = no merge)
 *   out, out_dtype, lse, sm_scale  as for pgqa_run
 * batch * num_kv_heads * splits must fit the array (about 8 MiB of work items
 * and fp32 partials); otherwise PGQA_ERR_CAPACITY and nothing is launched.
 * The first call on a device looks up the array's device address (once, with
 * that device current); make that first call before any stream capture.  All
 * calls share the array, which keeps what the last call left in it: calls whose
 * kernels may overlap on the GPU (different streams without ordering) race.
 * Nothing in the array needs to start zeroed: each call writes its work list
 * and partials before reading them.
 */
PGQA_API pgqa_status pgqa_decode_static_scratch(const void *q, const void *k_pool, const void *v_pool,
                                                const int32_t *kv_indptr, const int32_t *kv_indices,
                                                int64_t num_indices, const int32_t *last_page_len, int batch,
                                                int64_t num_pages, int page_size, int num_qo_heads,
                                                int num_kv_heads, int head_dim, pgqa_dtype dtype, int splits,
                                                void *out, pgqa_dtype out_dtype, float *lse, float sm_scale,
                                                pgqa_stream_t stream);

/* Frees the plan's buffers (synchronising with its last enqueued copy).  NULL is a no-op. */
PGQA_API pgqa_status pgqa_plan_destroy(pgqa_plan *plan);

/* What the last plan_update decided (host-side, no synchronisation). */
typedef struct pgqa_plan_info {
    int num_items;          /* CTAs of the partial kernel */
    int num_merge_tasks;    /* (query row, kv head) pairs whose slices are merged */
    int split_tokens;       /* slice length used */
    int max_splits_used;    /* most slices any (request, kv head) got */
    int total_q_rows;
    int num_sms;            /* SMs of the plan's device */
    int64_t kv_tokens;      /* sum of kv_len over requests */
    int num_prefill_tiles;  /* CTAs of the prefill-segment kernel (requests with > 1 query row) */
} pgqa_plan_info;

PGQA_API pgqa_status pgqa_plan_get_info(const pgqa_plan *plan, pgqa_plan_info *info);

/*
 * pgqa_plan_schedule -- the schedule pgqa_plan_update would build, computed on
 * the host alone.
 *
 * Runs the checks and the split heuristic of pgqa_plan_update (split-KV as in
 * "A library kernel for decode", section "What changed"; the ragged form of
 * the "flashlet" README, design bullets) for a GPU with num_sms SMs, and
 * returns the work lists instead of uploading them.  It touches no device and
 * allocates nothing on one, so it runs on a machine without a GPU: to see how
 * a batch will be cut, or to size a plan, before any launch.
 *
 *   cfg                 plan options, checked as pgqa_plan_create checks them.
 *                       The heuristic assumes cfg->ctas_per_sm CTA slots per
 *                       SM, or 2 when it is 0 (what every decode kernel
 *                       variant has on GB300, so the schedule equals the one
 *                       a plan on a GB300 with the same num_sms builds).
 *   num_sms             SMs of the target GPU (152 on GB300), >= 1
 *   kv_indptr_host, last_page_len_host, qo_indptr_host, batch, num_pages,
 *   causal              as for pgqa_plan_update
 *   kv_indices_host     [kv_indptr[batch]] int32, HOST: checked against
 *                       [0, num_pages) like pgqa_plan_update's host mirror
 *   slices, max_slices  caller-owned host array, or NULL (then only counted):
 *                       one entry per decode CTA, in launch order
 *   merges, max_merges  as above, one entry per merged (query row, kv head)
 *   tiles, max_tiles    as above, one entry per prefill-segment CTA
 *   info                out: the counts and decisions (always written when
 *                       the table passes its checks)
 *
 * Errors: every status pgqa_plan_create and pgqa_plan_update return for the
 * same options and table (no PGQA_ERR_CUDA); PGQA_ERR_CAPACITY also when a
 * non-NULL array holds fewer entries than the schedule has (info still says
 * how many).
 */
typedef struct pgqa_slice {
    int32_t q_row;         /* query row */
    int32_t kv_head;
    int32_t key_begin;     /* keys [key_begin, key_end) of the row's request; key_begin is */
    int32_t key_end;       /*   a multiple of the kernel's warp tile (32 keys at head_dim 64, else 16) */
    int32_t partial_slot;  /* -1: the CTA writes the (row, kv head) output; else the split partial it fills */
    int32_t append_pos;    /* pgqa_append_run: key position whose new K/V row this CTA stores, or -1 */
} pgqa_slice;

typedef struct pgqa_merge {
    int32_t q_row;
    int32_t kv_head;
    int32_t slot_base;     /* partials slot_base .. slot_base + num_splits - 1 are merged */
    int32_t num_splits;
} pgqa_merge;

typedef struct pgqa_prefill_tile {
    int32_t q_row0;        /* first query row of the request */
    int32_t rows;          /* L, the request's query rows */
    int32_t n_keys;        /* N, the request's keys */
    int32_t kv_head;
    int32_t pair0;         /* first (row, head) pair of the tile; pair m = i * G + h for row */
    int32_t pairs;         /*   q_row0 + i and head h of the group; the tile holds up to `pairs` */
    int32_t key_begin;     /* key slice [key_begin, key_end) of this CTA */
    int32_t key_end;
    int32_t partial_base;  /* -1: final rows; else partial of (row i, split s) is partial_base + i * num_splits + s */
    int32_t split;         /* s */
    int32_t num_splits;
} pgqa_prefill_tile;

typedef struct pgqa_schedule_info {
    int num_items;          /* decode CTAs (slices) */
    int num_merge_tasks;
    int num_prefill_tiles;
    int split_tokens;       /* slice length chosen for the decode rows */
    int max_splits_used;    /* most slices any (row, kv head) got */
    int pipeline_stages;    /* the tensor-core decode kernel's depth, 2 or 3; 1 = its wide form */
    int total_q_rows;
    int64_t kv_tokens;      /* sum of kv_len over requests */
} pgqa_schedule_info;

PGQA_API pgqa_status pgqa_plan_schedule(const pgqa_plan_config *cfg, int num_sms, const int32_t *kv_indptr_host,
                                        const int32_t *last_page_len_host, const int32_t *qo_indptr_host, int batch,
                                        const int32_t *kv_indices_host, int64_t num_pages, int causal,
                                        pgqa_slice *slices, int max_slices, pgqa_merge *merges, int max_merges,
                                        pgqa_prefill_tile *tiles, int max_tiles, pgqa_schedule_info *info);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDGQA_H */
