// Chunked-prefill segment of a ragged call: causal attention of a request's L
// query rows (a prompt chunk) over its N cached + new keys, on tensor cores.
//
// "flashlet" README, design bullets: one ragged plan()/run() serves chunked
// prefills and decode rows together (qo_indptr lengths [512, 1, 1, ...]) with a
// causal mask over both.  Rows of the chunk follow the bottom-right alignment:
// row i of an L-row chunk over N keys attends keys j <= N - L + i.
//
// Work: one CTA per (request, kv head, 64 consecutive (row, head) pairs), the
// pairs of a kv head's G query heads packed as m = i * G + h, so that every K/V
// tile staged in shared memory serves the whole GQA group.  Four warps take 16
// pairs each.  Per 64-key tile (mma.sync m16n8k16, fp32 accumulate):
//   S[16 pairs x 64 keys]  = Q[16 x d] . K^T         (K rows through ldmatrix)
//   O[16 pairs x d]       += P[16 x 64] . V           (V through ldmatrix.trans)
// P leaves the score accumulator directly as the A fragment of the second
// product (register reuse, no shuffles), carried as hi + lo 16-bit terms.  K/V
// tiles arrive through 3-D TMA boxes with 128-byte swizzle into a three-stage
// CTA-wide ring; a fused call patches the chunk's new rows in from k_new/v_new
// and stores them into their pool slots.
#pragma once

#include <climits>

#include "decode_tc.cuh"

namespace pgqa {

template <int D>
struct PrefillCfg {
    static constexpr int KT = 64;                      // keys per tile
    static constexpr int NW = 4;                       // warps; 16 pairs each
    static constexpr int MP = NW * 16;                 // pairs per CTA
    static constexpr int ST = 3;                       // CTA-wide stages
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = KT * 128;
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int PIPE_BYTES = ST * STAGE_BYTES;
    static constexpr int SMEM_BYTES = PIPE_BYTES + ST * 8 + kSlicePageCap * 4;
    static constexpr int KS = D / 16;                  // k-steps of Q.K^T
    static constexpr int NT = KT / 8;                  // key n-tiles of S
    static constexpr int DT = D / 8;                   // d n-tiles of O
};

template <int D>
__device__ __forceinline__ uint32_t ptile_off(int r, int c) {
    return (c >> 3) * (PrefillCfg<D>::HALF_BYTES) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <int D, bool ROPE, typename T>
__global__ void __launch_bounds__(128, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const PrefillParams p, int G) {
    using C = PrefillCfg<D>;
    using M = MmaType<T>;
    constexpr int CH = D / 8;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int lm = lane >> 3, lr = lane & 7;
    uint8_t *pipe = smem;
    const uint32_t bar0 = smem_addr(smem + C::PIPE_BYTES);
    int32_t *page_buf = reinterpret_cast<int32_t *>(smem + C::PIPE_BYTES + C::ST * 8);

    if (smem_addr(smem) & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.flags, PGQA_FLAG_SMEM_ALIGN);
        pdl_wait();
        return;
    }
    const PrefillItem it = p.items[blockIdx.x];  // written by plan_update's copy only
    const int key_begin = it.key_begin, key_end = it.key_end;
    const int ntiles = key_end > key_begin ? (key_end - key_begin + C::KT - 1) / C::KT : 0;
    const bool fused = p.k_new != nullptr;
    const int new_begin = it.n_keys - it.rows;   // the chunk's own keys (a fused call supplies them)
    // Chunk ch of the new K (rotated at its key position when the plan uses RoPE) or V
    // row of key position pos >= new_begin.
    auto new_chunk = [&](bool isv, int pos, int ch) -> uint4 {
        const T *row = static_cast<const T *>(isv ? p.v_new : p.k_new) +
                       (static_cast<size_t>(it.q_row0 + pos - new_begin) * p.num_kv_heads + it.kv_head) * D;
        if (ROPE && !isv)
            return rope_chunk<T, D>(row, ch, p.rope_cs + static_cast<size_t>(pos) * (D / 2));
        return __ldg(reinterpret_cast<const uint4 *>(row + ch * 8));
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::ST; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_barrier_init();
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    const SlicePages pages =
        stage_slice_pages(page_buf, p.kv_indices, it.page_base, key_begin, key_end, p.page_size);
    __syncthreads();
    const uint64_t policy = l2_evict_first_policy();

    auto issue = [&](int kt) {
        const int s = kt % C::ST;
        const uint32_t kdst = smem_addr(pipe + s * C::STAGE_BYTES);
        const uint32_t vdst = kdst + C::TILE_BYTES;
        const uint32_t bar = bar0 + 8 * s;
        const int t0 = key_begin + kt * C::KT;
        int nvalid = 0;
        for (int r = 0; r < C::KT && t0 + r < key_end; r += p.box_rows) {
            const int64_t page = pages(t0 + r, p.page_size);
            if (page >= 0 && page < p.num_pages) ++nvalid;
        }
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid * p.box_rows * D * 2 * 2));
        for (int r = 0; r < C::KT; r += p.box_rows) {
            const int tt = t0 + r;
            if (tt >= key_end) break;
            const int64_t page = pages(tt, p.page_size);
            if (page < 0 || page >= p.num_pages) {  // skipped (stale rows) and reported
                atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
                continue;
            }
            const int row = static_cast<int>(page * p.page_size + tt % p.page_size);
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) {
                const uint32_t off = hf * C::HALF_BYTES + r * 128;
                tma_load_3d_hint(kdst + off, &tm_k, hf * 64, it.kv_head, row, bar, policy);
                tma_load_3d_hint(vdst + off, &tm_v, hf * 64, it.kv_head, row, bar, policy);
            }
        }
    };

    const int pre = ntiles < C::ST ? ntiles : C::ST;
    if (p.prefetch_pool && threadIdx.x == 0)
        for (int kt = 0; kt < pre; ++kt) issue(kt);
    pdl_wait();
    pdl_launch_dependents();
    if (!p.prefetch_pool && threadIdx.x == 0)
        for (int kt = 0; kt < pre; ++kt) issue(kt);

    // This lane's two pair rows: r = 0 -> pair m0 + 16 warp + g8, r = 1 -> + 8.
    int limit[2];       // last admissible key of the row (< 0: none)
    bool valid_row[2];  // the pair is a real (row, head) of the request
    int qi[2];          // the pair's row within the request
    uint32_t qa[C::KS][4];
    {
        const T *qb[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int m = it.pair0 + warp * 16 + g8 + 8 * r;
            const int i = m / G, h = m - (m / G) * G;
            const bool valid = i < it.rows;
            qi[r] = i;
            valid_row[r] = valid;
            limit[r] = !valid ? -1 : (p.causal ? it.n_keys - it.rows + i : it.n_keys - 1);
            limit[r] = min(limit[r], key_end - 1);  // keys of this CTA's slice only
            qb[r] = static_cast<const T *>(p.q) +
                    (static_cast<size_t>(it.q_row0 + (valid ? i : 0)) * p.num_qo_heads + it.kv_head * G + h) * D;
            if (!valid) qb[r] = nullptr;
        }
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
            const int d0 = ks * 16 + 2 * c4;
            qa[ks][0] = qb[0] ? __ldg(reinterpret_cast<const uint32_t *>(qb[0] + d0)) : 0u;
            qa[ks][1] = qb[1] ? __ldg(reinterpret_cast<const uint32_t *>(qb[1] + d0)) : 0u;
            qa[ks][2] = qb[0] ? __ldg(reinterpret_cast<const uint32_t *>(qb[0] + d0 + 8)) : 0u;
            qa[ks][3] = qb[1] ? __ldg(reinterpret_cast<const uint32_t *>(qb[1] + d0 + 8)) : 0u;
        }
    }
    if (ROPE) {
        // Rotary embedding of each real row at its position new_begin + i: channels
        // 16 ks + 2 c4 (+1, +8, +9) pair with the same channels of k-step ks + KS/2.
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (!valid_row[r]) continue;
            const float2 *cs = p.rope_cs + static_cast<size_t>(new_begin + qi[r]) * (D / 2);
#pragma unroll
            for (int ks = 0; ks < C::KS / 2; ++ks) {
                const float4 c0 = __ldg(reinterpret_cast<const float4 *>(cs + ks * 16 + 2 * c4));
                const float4 c1 = __ldg(reinterpret_cast<const float4 *>(cs + ks * 16 + 2 * c4 + 8));
                rope_rotate2<T>(qa[ks][r], qa[ks + C::KS / 2][r], c0);
                rope_rotate2<T>(qa[ks][2 + r], qa[ks + C::KS / 2][2 + r], c1);
            }
        }
    }
    // Largest / smallest admissible key over the warp's real rows (rows grow with m).
    int warp_limit = max(limit[0], limit[1]);
    int warp_min = min(valid_row[0] ? limit[0] : INT_MAX, valid_row[1] ? limit[1] : INT_MAX);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        warp_limit = max(warp_limit, __shfl_xor_sync(0xffffffffu, warp_limit, m));
        warp_min = min(warp_min, __shfl_xor_sync(0xffffffffu, warp_min, m));
    }

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[C::DT][4];
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;

    bool ok = true;
    int waited = 0;
    for (int kt = 0; kt < ntiles; ++kt) {
        const int s = kt % C::ST;
        if (!__syncthreads_and(mbar_wait_bounded(bar0 + 8 * s, (kt / C::ST) & 1))) {
            if (threadIdx.x == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            ok = false;
            break;
        }
        waited = kt + 1;
        uint8_t *kp = pipe + s * C::STAGE_BYTES;
        const uint32_t kb = smem_addr(kp);
        const uint32_t vb = kb + C::TILE_BYTES;
        const int t0 = key_begin + kt * C::KT;
        const int nvalid = min(C::KT, key_end - t0);

        // ---- fused append: the chunk's own rows come from k_new / v_new
        bool patched = false;
        if (fused && max(new_begin, t0) < t0 + nvalid) {
            for (int idx = threadIdx.x; idx < nvalid * 2 * CH; idx += 128) {
                const int r = idx / (2 * CH);
                const int rem = idx - r * 2 * CH;
                const bool isv = rem >= CH;
                const int ch = rem - (isv ? CH : 0);
                const int pos = t0 + r;
                if (pos < new_begin) continue;
                *reinterpret_cast<uint4 *>(kp + (isv ? C::TILE_BYTES : 0) + ptile_off<D>(r, ch)) =
                    new_chunk(isv, pos, ch);
            }
            patched = true;
            __syncthreads();
        }

        if (t0 <= warp_limit) {
            // ---- S = Q K^T
            float sc[C::NT][4];
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
                for (int nt = 0; nt < C::NT; nt += 2) {
                    // matrices: (keys nt, chunk 2ks), (nt, 2ks+1), (nt+1, 2ks), (nt+1, 2ks+1)
                    uint32_t b[4];
                    ldsm_x4(b, kb + ptile_off<D>((nt + (lm >> 1)) * 8 + lr, 2 * ks + (lm & 1)));
                    M::mma(sc[nt], qa[ks], b[0], b[1]);
                    M::mma(sc[nt + 1], qa[ks], b[2], b[3]);
                }
            }
            // ---- mask (only a tile reaching past some row's bound, or past the slice end),
            // row max of the raw scores (the scale is positive and folded into exp2 below)
            if (t0 + C::KT - 1 > warp_min || nvalid < C::KT) {
#pragma unroll
                for (int nt = 0; nt < C::NT; ++nt) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int key = t0 + nt * 8 + 2 * c4 + (j & 1);
                        if (key > limit[j >> 1]) sc[nt][j] = -INFINITY;
                    }
                }
            }
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) {
                mx[0] = fmaxf(mx[0], fmaxf(sc[nt][0], sc[nt][1]));
                mx[1] = fmaxf(mx[1], fmaxf(sc[nt][2], sc[nt][3]));
            }
            float neg_m[2];  // -(running max) in scaled log2 units; 0 while a row has seen no key
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mn = fmaxf(m_run[r], mx[r] * p.scale_log2);
                const float alpha = (mn == m_run[r]) ? 1.f : ex2_approx(m_run[r] - mn);
                m_run[r] = mn;
                l_run[r] *= alpha;
#pragma unroll
                for (int dt = 0; dt < C::DT; ++dt) {
                    o[dt][2 * r] *= alpha;
                    o[dt][2 * r + 1] *= alpha;
                }
                neg_m[r] = (mn == -INFINITY) ? 0.f : -mn;
            }
            // ---- P (A fragments, hi + lo) and O += P V
            const bool tail = nvalid < C::KT;
#pragma unroll
            for (int kk = 0; kk < C::KT / 16; ++kk) {
                uint32_t ahi[4], alo[4];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int nt = 2 * kk + half;
                    float pr[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // exp2(s * scale_log2 - m): a masked score (-inf) gives 0
                        pr[j] = ex2_approx(fmaf(sc[nt][j], p.scale_log2, neg_m[j >> 1]));
                        l_run[j >> 1] += pr[j];
                    }
                    const uint32_t h01 = M::pack(pr[0], pr[1]), h23 = M::pack(pr[2], pr[3]);
                    const float2 f01 = unpack2<T>(h01), f23 = unpack2<T>(h23);
                    ahi[2 * half] = h01;
                    ahi[2 * half + 1] = h23;
                    alo[2 * half] = M::pack(pr[0] - f01.x, pr[1] - f01.y);
                    alo[2 * half + 1] = M::pack(pr[2] - f23.x, pr[3] - f23.y);
                }
                // A register order: (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15)
                const uint32_t a_hi[4] = {ahi[0], ahi[1], ahi[2], ahi[3]};
                const uint32_t a_lo[4] = {alo[0], alo[1], alo[2], alo[3]};
                uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
                if (tail) {  // V rows past the slice end may hold anything: zero them
                    const int k0 = kk * 16 + 2 * c4;
                    keep0 = (k0 < nvalid ? 0x0000ffffu : 0u) | (k0 + 1 < nvalid ? 0xffff0000u : 0u);
                    keep1 = (k0 + 8 < nvalid ? 0x0000ffffu : 0u) | (k0 + 9 < nvalid ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int dt = 0; dt < C::DT; dt += 2) {
                    // matrices: (keys 16kk+0-7, chunk dt), (16kk+8-15, dt), (16kk+0-7, dt+1), (16kk+8-15, dt+1)
                    uint32_t b[4];
                    ldsm_x4_t(b, vb + ptile_off<D>(kk * 16 + (lm & 1) * 8 + lr, dt + (lm >> 1)));
                    if (tail) {
                        b[0] &= keep0;
                        b[1] &= keep1;
                        b[2] &= keep0;
                        b[3] &= keep1;
                    }
                    M::mma(o[dt], a_hi, b[0], b[1]);
                    M::mma(o[dt], a_lo, b[0], b[1]);
                    M::mma(o[dt + 1], a_hi, b[2], b[3]);
                    M::mma(o[dt + 1], a_lo, b[2], b[3]);
                }
            }
        }
        if (patched) fence_proxy_async_smem();
        __syncthreads();  // every warp is done with stage s
        if (threadIdx.x == 0 && kt + C::ST < ntiles) issue(kt + C::ST);
    }
    if (!ok && threadIdx.x == 0) {
        const int issued = ntiles < waited + C::ST ? ntiles : waited + C::ST;
        for (int kt = waited; kt < issued; ++kt) mbar_wait_bounded(bar0 + 8 * (kt % C::ST), (kt / C::ST) & 1);
    }

    // ---- fused append: the split-0 CTA holding pair (i, head 0) stores row i's new K/V
    if (fused && it.split == 0) {
        for (int idx = threadIdx.x; idx < C::MP * 2 * CH; idx += 128) {
            const int mloc = idx / (2 * CH);
            const int m = it.pair0 + mloc;
            if (m % G != 0) continue;
            const int i = m / G;
            if (i >= it.rows) continue;
            const int rem = idx - mloc * 2 * CH;
            const bool isv = rem >= CH;
            const int ch = rem - (isv ? CH : 0);
            const int pos = new_begin + i;
            const int64_t page = p.kv_indices[it.page_base + pos / p.page_size];
            if (page < 0 || page >= p.num_pages) {
                atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
                continue;
            }
            T *dst = static_cast<T *>(isv ? p.v_pool : p.k_pool) +
                     ((page * p.page_size + pos % p.page_size) * p.num_kv_heads + it.kv_head) * D + ch * 8;
            *reinterpret_cast<uint4 *>(dst) = new_chunk(isv, pos, ch);
        }
    }

    // ---- normalise and store: row r of this lane, channels 8 dt + 2 c4, +1
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        if (!valid_row[r]) continue;
        const int m = it.pair0 + warp * 16 + g8 + 8 * r;
        const int i = m / G, h = m - (m / G) * G;
        const size_t row = static_cast<size_t>(it.q_row0 + i) * p.num_qo_heads + it.kv_head * G + h;
        const float L = l_run[r];
        // L == 0 only for a row with no admissible key; NaN (a poisoned row) propagates.
        const float inv = (L == 0.f) ? 0.f : rcp_approx(L);
        const float lse2 = (L == 0.f) ? -INFINITY : m_run[r] + lg2_approx(L);
        if (it.part_base >= 0) {  // split keys: normalised partial + its log2-sum-exp
            const size_t slot = static_cast<size_t>(it.part_base + i * it.num_splits + it.split) * G + h;
#pragma unroll
            for (int dt = 0; dt < C::DT; ++dt)
                *reinterpret_cast<float2 *>(p.partial_o + slot * D + dt * 8 + 2 * c4) =
                    make_float2(o[dt][2 * r] * inv, o[dt][2 * r + 1] * inv);
            if (c4 == 0) p.partial_lse[slot] = lse2;
            continue;
        }
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) {
            const float v0 = o[dt][2 * r] * inv, v1 = o[dt][2 * r + 1] * inv;
            const size_t oi = row * D + dt * 8 + 2 * c4;
            if (p.out_dtype == PGQA_FP32)
                *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + oi) = make_float2(v0, v1);
            else
                *reinterpret_cast<uint32_t *>(static_cast<T *>(p.out) + oi) = M::pack(v0, v1);
        }
        if (c4 == 0 && p.lse != nullptr) p.lse[row] = lse2 * 0.6931471805599453f;
    }
}

template <int D, bool ROPE, typename T>
cudaError_t launch_prefill_tc_r(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const PrefillParams &p,
                                int num_items, bool pdl, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    auto kern = prefill_tc_kernel<D, ROPE, T>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_items);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, p, group);
}

// Plans without RoPE run an instantiation with no trace of it.
template <int D, typename T>
cudaError_t launch_prefill_tc(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const PrefillParams &p,
                              int num_items, bool pdl, cudaStream_t stream) {
    return p.rope_cs != nullptr ? launch_prefill_tc_r<D, true, T>(group, tm_k, tm_v, p, num_items, pdl, stream)
                                : launch_prefill_tc_r<D, false, T>(group, tm_k, tm_v, p, num_items, pdl, stream);
}

}  // namespace pgqa
