// Split-KV paged GQA decode, tensor-core partial kernel, persistent form.
//
// The arithmetic is the one of decode_tc.cuh (swap-AB mma.sync tiles, hi + lo P,
// log2-domain online softmax); what changes is the schedule.  One CTA per SM walks
// the work list (items blockIdx.x, blockIdx.x + gridDim.x, ...; the list is
// sorted longest first), and every warp's TMA ring runs on across item
// boundaries: while a warp finishes one item, the K/V tiles of its next item are
// already in flight.  Per item, warps 1..3 leave (m, l, O) in one of two
// shared-memory slots and move on; warp 0 combines them (named barriers 1-2
// "deposited", 3-4 "slot free again").
//
// With one CTA per SM per call, an SM always has room for the CTA of the next
// call on the stream (programmatic dependent launch): that CTA issues its first
// K/V loads while this call drains, so HBM stays busy across back-to-back calls.
#pragma once

#include "decode_tc.cuh"

namespace pgqa {

template <int D, int STAGES>
struct TcpCfg {
    static constexpr int TW = decode_warp_tile(D);
    static constexpr int MT = TW / 16;
    static constexpr int HALVES = D / 64;
    static constexpr int NW = kDecodeWarps;
    static constexpr int ST = STAGES;
    static constexpr int HALF_BYTES = TW * 128;
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int PIPE_BYTES = NW * ST * STAGE_BYTES;
    static constexpr int BAR_BYTES = (NW * ST * 8 + 15) / 16 * 16;  // mbarriers, padded to 16 bytes
    static constexpr int DT = D / 16;
    static constexpr int KS = D / 16;
    static constexpr int OS = D + 4;
    static constexpr int SLOT_FLOATS = 16 + 8 * OS;                 // m[8], l[8], O[8][OS]
    static constexpr int COMBINE_BYTES = 2 * (NW - 1) * SLOT_FLOATS * 4;
    static constexpr int FIN_BYTES = 8 * OS * 4;
    static constexpr int SMEM_BYTES = PIPE_BYTES + BAR_BYTES + COMBINE_BYTES + FIN_BYTES;
    static_assert(HALF_BYTES % 1024 == 0, "128B-swizzled blocks start on 1024-byte boundaries");
    static_assert((PIPE_BYTES + BAR_BYTES) % 16 == 0, "combine slots are 16-byte aligned");
};

template <int D, int STAGES, typename T>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2)
    decode_tcp_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const DecodeParams p, int G, int n_items) {
    using C = TcpCfg<D, STAGES>;
    using M = MmaType<T>;
    constexpr int CH = D / 8;
    constexpr int OS = C::OS;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int lm = lane >> 3, lr = lane & 7;

    uint8_t *pipe = smem;
    const uint32_t bar0 = smem_addr(smem + C::PIPE_BYTES) + warp * C::ST * 8;
    float *cslots = reinterpret_cast<float *>(smem + C::PIPE_BYTES + C::BAR_BYTES);  // [2][NW-1][SLOT]
    float *fin = cslots + 2 * (C::NW - 1) * C::SLOT_FLOATS;                          // [8][OS]

    if (smem_addr(smem) & 1023u) {  // the stage layout assumes this alignment of the window
        if (threadIdx.x == 0) atomicOr(p.flags, PGQA_FLAG_SMEM_ALIGN);
        pdl_wait();
        return;
    }
    const int nj = (n_items - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                   static_cast<int>(gridDim.x);
    const bool fused = p.k_new != nullptr;
    auto item_at = [&](int j) -> WorkItem { return p.items[blockIdx.x + j * gridDim.x]; };
    auto tiles_of = [&](const WorkItem &w) { return (w.tok_end - w.tok_begin + C::TW - 1) / C::TW; };

    if (lane == 0) {
        for (int s = 0; s < C::ST; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_barrier_init();
        if (warp == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
    }
    __syncwarp();
    const uint64_t policy = l2_evict_first_policy();

    // ---- producer (lane 0): this warp's tiles over the CTA's items, in order.
    // The work list and kv_indices are final once plan_update is enqueued, so they
    // may be read before the grid-dependency wait.
    int pj = 0, pt = warp, pnt = 0, issued = 0;
    WorkItem pit{};
    bool producing = true;
    if (lane == 0) {
        pit = item_at(0);
        pnt = tiles_of(pit);
        while (pj < nj && pt >= pnt) {
            ++pj;
            pt = warp;
            if (pj < nj) {
                pit = item_at(pj);
                pnt = tiles_of(pit);
            }
        }
    }
    auto issue_next = [&]() {
        if (pj >= nj || !producing) return;
        const int s = issued % C::ST;
        const uint32_t kdst = smem_addr(pipe + (warp * C::ST + s) * C::STAGE_BYTES);
        const uint32_t vdst = kdst + C::TILE_BYTES;
        const uint32_t bar = bar0 + 8 * s;
        const int t0 = pit.tok_begin + pt * C::TW;
        constexpr int MAXC = C::TW / 16;
        int rows[MAXC];
        int nvalid = 0;
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
            rows[c] = -1;
            const int tt = t0 + c * p.box_rows;
            if (c * p.box_rows < C::TW && tt < pit.tok_end) {
                const int64_t page = __ldg(p.kv_indices + pit.page_base + tt / p.page_size);
                if (page < 0 || page >= p.num_pages) {
                    atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
                } else {
                    rows[c] = static_cast<int>(page * p.page_size + tt % p.page_size);
                    ++nvalid;
                }
            }
        }
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid * p.box_rows * D * 2 * 2));
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
            if (rows[c] >= 0) {
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf) {
                    const uint32_t off = hf * C::HALF_BYTES + c * p.box_rows * 128;
                    tma_load_3d_hint(kdst + off, &tm_k, hf * 64, pit.kv_head, rows[c], bar, policy);
                    tma_load_3d_hint(vdst + off, &tm_v, hf * 64, pit.kv_head, rows[c], bar, policy);
                }
            }
        }
        ++issued;
        pt += C::NW;
        while (pj < nj && pt >= pnt) {
            ++pj;
            pt = warp;
            if (pj < nj) {
                pit = item_at(pj);
                pnt = tiles_of(pit);
            }
        }
    };

    if (p.defer_wait) {
        if (lane == 0)
            for (int k = 0; k < C::ST; ++k) issue_next();
    } else {
        if (p.prefetch_pool && lane == 0)
            for (int k = 0; k < C::ST; ++k) issue_next();
        pdl_wait();
        pdl_launch_dependents();  // older kernels are complete: a grid started early overlaps only us
        if (!p.prefetch_pool && lane == 0)
            for (int k = 0; k < C::ST; ++k) issue_next();
    }

    const bool row_lane = lane < 2 * CH;
    const int rch = lane % CH;
    const bool rv = lane >= CH;
    int consumed = 0;
    bool ok = true;

    for (int j = 0; j < nj; ++j) {
        const WorkItem it = item_at(j);
        const int ntiles = tiles_of(it);
        const int my_tiles = ntiles > warp ? (ntiles - warp + C::NW - 1) / C::NW : 0;

        uint32_t qf[C::KS][2];
        {
            const bool real = g8 < G;
            const T *qp = static_cast<const T *>(p.q) +
                          (static_cast<size_t>(it.q_row) * p.num_qo_heads + it.kv_head * G + (real ? g8 : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                const uint32_t *w = reinterpret_cast<const uint32_t *>(qp + ks * 16 + 2 * c4);
                qf[ks][0] = real ? __ldg(w) : 0u;
                qf[ks][1] = real ? __ldg(w + 4) : 0u;
            }
        }
        auto new_row_chunk = [&](int pos) -> uint4 {
            const T *src = static_cast<const T *>(rv ? p.v_new : p.k_new) +
                           (static_cast<size_t>(pos + it.new_row_base) * p.num_kv_heads + it.kv_head) * D + rch * 8;
            return __ldg(reinterpret_cast<const uint4 *>(src));
        };
        int pf_pos = -1;
        uint4 pf = make_uint4(0u, 0u, 0u, 0u);
        if (fused) {
            const int nb = max(it.new_begin, it.tok_begin);
            if (nb < it.tok_end && ((nb - it.tok_begin) / C::TW) % C::NW == warp) {
                pf_pos = nb;
                if (row_lane) pf = new_row_chunk(nb);
            }
        }

        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        float o[C::DT][4];
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;

        for (int k = 0; k < my_tiles; ++k) {
            const int s = consumed % C::ST;
            if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * s, (consumed / C::ST) & 1))) {
                if (lane == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
                ok = false;  // keep walking the items (barrier protocol intact), compute nothing
                if (lane == 0) producing = false;
            }
            ++consumed;
            if (!ok) continue;
            const int tile = warp + k * C::NW;
            const int tb = it.tok_begin + tile * C::TW;
            const int nvalid = min(C::TW, it.tok_end - tb);
            uint8_t *kp = pipe + (warp * C::ST + s) * C::STAGE_BYTES;
            const uint32_t kb = smem_addr(kp);
            const uint32_t vb = kb + C::TILE_BYTES;

            bool patched = false;
            if (fused) {
                const int nb = max(it.new_begin, tb);
                if (nb < tb + nvalid) {
                    for (int pos = nb; pos < tb + nvalid; ++pos) {
                        const uint4 val = (pos == pf_pos) ? pf : (row_lane ? new_row_chunk(pos) : pf);
                        if (row_lane)
                            *reinterpret_cast<uint4 *>(kp + (rv ? C::TILE_BYTES : 0) + tile_off<D>(pos - tb, rch)) = val;
                    }
                    patched = true;
                    __syncwarp();
                }
            }

            float sc[C::MT][4];
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    uint32_t a[4];
                    ldsm_x4(a, kb + tile_off<D>(mt * 16 + (lm & 1) * 8 + lr, 2 * ks + (lm >> 1)));
                    M::mma(sc[mt], a, qf[ks][0], qf[ks][1]);
                }
            }
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int tok = mt * 16 + g8 + (jj >> 1) * 8;
                    const float x = tok < nvalid ? sc[mt][jj] * p.scale_log2 : -INFINITY;
                    sc[mt][jj] = x;
                    mx[jj & 1] = fmaxf(mx[jj & 1], x);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
            }
            float alpha[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float mn = fmaxf(m_run[h], mx[h]);
                alpha[h] = (mn == m_run[h]) ? 1.f : ex2_approx(m_run[h] - mn);
                m_run[h] = mn;
                l_run[h] *= alpha[h];
            }
            if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
                for (int dt = 0; dt < C::DT; ++dt) {
                    o[dt][0] *= alpha[0];
                    o[dt][1] *= alpha[1];
                    o[dt][2] *= alpha[0];
                    o[dt][3] *= alpha[1];
                }
            }
            uint32_t pb_hi[C::MT][2], pb_lo[C::MT][2];
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                float pr[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float x = sc[mt][jj];
                    pr[jj] = (x == -INFINITY) ? 0.f : ex2_approx(x - m_run[jj & 1]);
                    l_run[jj & 1] += pr[jj];
                }
                const uint32_t h01 = M::pack(pr[0], pr[1]);
                const uint32_t h23 = M::pack(pr[2], pr[3]);
                const float2 f01 = unpack2<T>(h01), f23 = unpack2<T>(h23);
                const uint32_t l01 = M::pack(pr[0] - f01.x, pr[1] - f01.y);
                const uint32_t l23 = M::pack(pr[2] - f23.x, pr[3] - f23.y);
                pb_hi[mt][0] = movm_t(h01);
                pb_hi[mt][1] = movm_t(h23);
                pb_lo[mt][0] = movm_t(l01);
                pb_lo[mt][1] = movm_t(l23);
            }
            const bool partial = nvalid < C::TW;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                uint32_t keep01 = 0xffffffffu, keep89 = 0xffffffffu;
                if (partial) {
                    const int t = mt * 16 + 2 * c4;
                    keep01 = (t < nvalid ? 0x0000ffffu : 0u) | (t + 1 < nvalid ? 0xffff0000u : 0u);
                    keep89 = (t + 8 < nvalid ? 0x0000ffffu : 0u) | (t + 9 < nvalid ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int dt = 0; dt < C::DT; ++dt) {
                    uint32_t a[4];
                    ldsm_x4_t(a, vb + tile_off<D>(mt * 16 + (lm >> 1) * 8 + lr, 2 * dt + (lm & 1)));
                    if (partial) {
                        a[0] &= keep01;
                        a[1] &= keep01;
                        a[2] &= keep89;
                        a[3] &= keep89;
                    }
                    M::mma(o[dt], a, pb_hi[mt][0], pb_hi[mt][1]);
                    M::mma(o[dt], a, pb_lo[mt][0], pb_lo[mt][1]);
                }
            }
            if (patched) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) issue_next();
        }

        // ---- fused append: the item owning a query row stores that row's new K/V
        if (fused && it.write_pos >= 0 && ok) {
            const int pos = it.write_pos;
            const int nb = max(it.new_begin, it.tok_begin);
            const bool held = nb < it.tok_end && nb == pos;
            const int writer = held ? ((nb - it.tok_begin) / C::TW) % C::NW : 0;
            if (warp == writer && row_lane) {
                const int64_t page = __ldg(p.kv_indices + it.page_base + pos / p.page_size);
                if (page < 0 || page >= p.num_pages) {
                    if (rch == 0) atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
                } else {
                    const uint4 val = held ? pf : new_row_chunk(pos);
                    T *dst = static_cast<T *>(rv ? p.v_pool : p.k_pool) +
                             ((page * p.page_size + pos % p.page_size) * p.num_kv_heads + it.kv_head) * D + rch * 8;
                    *reinterpret_cast<uint4 *>(dst) = val;
                }
            }
        }

        // ---- combine the warps of item j
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 4);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 8);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 16);
        }
        const int par = j & 1;
        auto slot = [&](int w) { return cslots + (par * (C::NW - 1) + (w - 1)) * C::SLOT_FLOATS; };
        if (warp != 0) {
            if (j >= 2) named_bar_sync_id(3 + par, C::NW * 32);  // warp 0 is done with this slot
            float *st = slot(warp);
            if (g8 == 0) {
                st[2 * c4] = m_run[0];
                st[2 * c4 + 1] = m_run[1];
                st[8 + 2 * c4] = l_run[0];
                st[8 + 2 * c4 + 1] = l_run[1];
            }
#pragma unroll
            for (int dt = 0; dt < C::DT; ++dt) {
                float *ow = st + 16 + (2 * c4) * OS + dt * 16 + g8;
                ow[0] = o[dt][0];
                ow[OS] = o[dt][1];
                ow[8] = o[dt][2];
                ow[OS + 8] = o[dt][3];
            }
            named_bar_arrive_id(1 + par, C::NW * 32);
            continue;
        }
        named_bar_sync_id(1 + par, C::NW * 32);
        float f[C::NW][2], lse2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int hh = 2 * c4 + h;
            float Mx = m_run[h];
#pragma unroll
            for (int w = 1; w < C::NW; ++w) Mx = fmaxf(Mx, slot(w)[hh]);
            float L = (m_run[h] == -INFINITY) ? 0.f : l_run[h] * ex2_approx(m_run[h] - Mx);
#pragma unroll
            for (int w = 1; w < C::NW; ++w) {
                const float mw = slot(w)[hh];
                if (mw != -INFINITY) L += slot(w)[8 + hh] * ex2_approx(mw - Mx);
            }
            // L == 0 only when no key was admissible; a NaN (poisoned row) propagates.
            const float inv = (L == 0.f) ? 0.f : rcp_approx(L);
            f[0][h] = (m_run[h] == -INFINITY) ? 0.f : ex2_approx(m_run[h] - Mx) * inv;
#pragma unroll
            for (int w = 1; w < C::NW; ++w) {
                const float mw = slot(w)[hh];
                f[w][h] = (mw == -INFINITY) ? 0.f : ex2_approx(mw - Mx) * inv;
            }
            lse2[h] = (L == 0.f) ? -INFINITY : Mx + lg2_approx(L);
        }
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int h = jj & 1;
                const int off = (2 * c4 + h) * OS + dt * 16 + g8 + (jj >> 1) * 8;
                float acc = o[dt][jj] * f[0][h];
#pragma unroll
                for (int w = 1; w < C::NW; ++w) acc += slot(w)[16 + off] * f[w][h];
                fin[off] = acc;
            }
        }
        __syncwarp();
        if (j + 2 < nj) named_bar_arrive_id(3 + par, C::NW * 32);  // slot par may be refilled
        for (int idx = lane; idx < G * CH; idx += 32) {
            const int h = idx / CH;
            const int c8 = (idx - h * CH) * 8;
            const float4 a = *reinterpret_cast<const float4 *>(fin + h * OS + c8);
            const float4 b = *reinterpret_cast<const float4 *>(fin + h * OS + c8 + 4);
            const int head = it.kv_head * G + h;
            if (it.out_slot < 0) {
                const size_t oi = (static_cast<size_t>(it.q_row) * p.num_qo_heads + head) * D + c8;
                if (p.out_dtype == PGQA_FP32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + oi);
                    dst[0] = a;
                    dst[1] = b;
                } else {
                    uint4 v;
                    v.x = M::pack(a.x, a.y);
                    v.y = M::pack(a.z, a.w);
                    v.z = M::pack(b.x, b.y);
                    v.w = M::pack(b.z, b.w);
                    *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + oi) = v;
                }
            } else {
                float4 *dst =
                    reinterpret_cast<float4 *>(p.partial_o + (static_cast<size_t>(it.out_slot) * G + h) * D + c8);
                dst[0] = a;
                dst[1] = b;
            }
        }
        if (g8 == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int hh = 2 * c4 + h;
                if (hh < G) {
                    const int head = it.kv_head * G + hh;
                    if (it.out_slot < 0) {
                        if (p.lse != nullptr)
                            p.lse[static_cast<size_t>(it.q_row) * p.num_qo_heads + head] =
                                lse2[h] * 0.6931471805599453f;
                    } else {
                        p.partial_lse[static_cast<size_t>(it.out_slot) * G + hh] = lse2[h];
                    }
                }
            }
        }
        __syncwarp();  // fin is rewritten by the next item
    }

    if (!ok && lane == 0) {  // let copies already in flight land before shared memory goes away
        for (int k = consumed; k < issued; ++k) mbar_wait_bounded(bar0 + 8 * (k % C::ST), (k / C::ST) & 1);
    }
    if (p.defer_wait && warp == 0) {
        pdl_wait();  // completion order: finish only after the prefill grid before us
        pdl_launch_dependents();
    }
}

template <int D, int STAGES, typename T>
cudaError_t launch_decode_tcp_st(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                 const DecodeParams &p, int num_items, int grid, bool pdl, cudaStream_t stream) {
    using C = TcpCfg<D, STAGES>;
    auto kern = decode_tcp_kernel<D, STAGES, T>;
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
    cfg.gridDim = dim3(grid < num_items ? grid : num_items);
    cfg.blockDim = dim3(C::NW * 32);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, p, group, num_items);
}

// Persistent launch: d 64 keeps three stages per warp (112 KB, two CTAs per SM), d 128 two.
template <int D, typename T>
cudaError_t launch_decode_tcp(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeParams &p,
                              int num_items, int grid, bool pdl, cudaStream_t stream) {
    if (group < 1 || group > 8) return cudaErrorInvalidValue;  // one 8-head n tile
    if (p.rope_cs != nullptr) return cudaErrorInvalidValue;    // rotary plans run one CTA per item
    return launch_decode_tcp_st<D, D == 64 ? 3 : 2, T>(group, tm_k, tm_v, p, num_items, grid, pdl, stream);
}

}  // namespace pgqa
