// pa_prefix_m256.cuh -- chunked-prefix attention for head sizes up to 128 with 256 query rows
// per CTA.  "paged_attn.py", forward_prefix / _forward_prefix_pytorch: the same result as
// pa_prefix_kernel (pa_prefix.cuh), which documents the method; only the work split differs.
//
// The CTA's rows are two groups of 128 (rows j * G + g of the kv head's group, as there), and
// both groups use every key/value tile the loaders bring in.  Tensor memory holds, per group,
// two S buffers of 64 columns and O (head size <= 128 columns): 2 x 256 = all 512 columns.  The
// softmax writes P (bf16: hi and lo) back into the S buffer it has just read, and the score MMA
// of tile t + 2 reuses that buffer only after the value MMA of tile t has completed.  Q of both
// groups sits in shared memory.  Fourteen warps:
//   warp 0         allocates tensor memory; lane 0 issues group 0's score MMAs
//   warp 1         lane 0 issues group 0's value MMAs
//   warp 2 / 3     fill the key / the value ring (the loader of pa_prefix.cuh, one warp each)
//   warps 4-7      softmax of group 0 (warp 4 + w: rows 32 w .. 32 w + 31 of the group)
//   warps 8-11     softmax of group 1
//   warps 12 / 13  lane 0 issues group 1's score / value MMAs (a lane per group and product:
//                  a lane waiting on one group does not hold up the other group's MMAs)
// so each sub-partition runs two softmax warps, and while one group turns its scores into
// probabilities the tensor core works on the other group's products.
#pragma once

#include "pa_prefix.cuh"

namespace pa {

constexpr int kP2Threads = 14 * 32;
constexpr int kP2Rows = 256;
constexpr int kP2MmaWarp = 0, kP2PvWarp = 1, kP2KeyWarp = 2, kP2ValWarp = 3, kP2SoftmaxWarp0 = 4;
constexpr int kP2MmaWarp1 = 12, kP2PvWarp1 = 13;  // group 1's score / value lanes

template <bool BF16, int D>
struct Pfx2Cfg {
    static constexpr int DP = (D + 15) / 16 * 16;
    static constexpr int DPR = (DP + 31) / 32 * 32;
    static constexpr int NCR = D / 8;
    static constexpr int NCP = DP / 8;
    static constexpr int BN = 64;
    static constexpr int NP = BF16 ? 2 : 1;
    static constexpr int K_BYTES = BN * DP * 2;
    static constexpr int V_BYTES = BN * DP * 2;
    static constexpr int QG_BYTES = kPfxBM * DP * 2;  // one group's Q: [chunk][128 rows][16 bytes]
    static constexpr int CTL_BYTES = 1024;
    static constexpr int SLOTS = (227 * 1024 - 2 * QG_BYTES - CTL_BYTES) / K_BYTES;
    // About 30% of the slots hold keys: a key slot is released as soon as both groups' score
    // MMAs are done, a value slot only after the value MMAs, which trail by a softmax
    // (measured at d 128: 3 + 7 slots 797 TFLOP/s, 2 + 8 741, 5 + 5 787).
    static constexpr int NK0 = SLOTS * 3 / 10;
    static constexpr int NK = NK0 > 8 ? 8 : (NK0 < 2 ? 2 : NK0);
    static constexpr int NV = SLOTS - NK > 16 ? 16 : SLOTS - NK;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = NK * K_BYTES;
    static constexpr int OFF_Q = OFF_V + NV * V_BYTES;
    static constexpr int OFF_CTL = OFF_Q + 2 * QG_BYTES;
    static constexpr int SMEM = OFF_CTL + CTL_BYTES;
    // tensor memory of group g at g * 256: S buffers [0, 64) and [64, 128), O [128, 128 + DPR)
    static constexpr uint32_t TMEM_COLS = 512, COL_O = 128;
    static constexpr uint32_t IDESC_S = umma_idesc_f16(BF16, kPfxBM, BN);
    static constexpr uint32_t IDESC_O = umma_idesc_f16(BF16, kPfxBM, DP);
    static_assert(DPR <= 128, "two groups' S buffers and O fill the 512 columns only up to head size 128");
    static_assert(NK >= 2 && NV >= 2 && SMEM <= 227 * 1024, "shared memory");
};

template <bool BF16, int D>
__global__ void __launch_bounds__(kP2Threads, 1) pa_prefix_m256_kernel(const __grid_constant__ PrefixParams p) {
    using C = Pfx2Cfg<BF16, D>;
    constexpr int BN = C::BN, NK = C::NK, NV = C::NV;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = pfx_seq_order(p, blockIdx.z, reinterpret_cast<uint32_t*>(smem + C::OFF_CTL)), kvh = blockIdx.y;
    const int split = blockIdx.x / p.mt;
    const int row0 = (p.mt - 1 - blockIdx.x % p.mt) * kP2Rows;  // row tiles with more keys first
    const int G = p.G;
    int ctx = p.ctx_lens[s];
    const int q0 = p.qsl[s];
    const int q_len = p.qsl[s + 1] - q0;
    if (q_len < 0 || q_len > p.max_query_len || ctx < 0) {
        if (tid == 0 && split == 0) prefix_flag(128u);
        return;
    }
    const int rows_total = q_len * G;
    if (row0 >= rows_total) return;
    if (ctx > p.mbps * p.bs) {
        if (tid == 0) prefix_flag(64u);
        ctx = p.mbps * p.bs;
    }
    const int2 plan = pfx_split_plan((ctx + BN - 1) / BN, p.nsplit, p.split_tiles);
    if (split >= plan.x) return;
    const int tb = split * plan.y;
    const int n_ctx = min(plan.y, (ctx + BN - 1) / BN - tb);
    const bool last_split = split == plan.x - 1;
    const int ng = row0 + kPfxBM < rows_total ? 2 : 1;  // row groups with rows in the chunk
    const int row_last = min(row0 + kP2Rows, rows_total) - 1;
    const int n_tiles = n_ctx + (last_split ? (row_last / G) / BN + 1 : 0);

    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {
        if (tid == 0) prefix_flag(4u);
        return;
    }
    uint8_t* ctl = smem + C::OFF_CTL;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ctl);
    uint64_t* k_full = bars;              // [NK] keys (and the tile's page mask) in place
    uint64_t* k_empty = k_full + NK;      // [NK] both groups' score MMAs done, masks read
    uint64_t* v_full = k_empty + NK;      // [NV]
    uint64_t* v_empty = v_full + NV;      // [NV] both groups' value MMAs done
    uint64_t* s_full = v_empty + NV;      // [2 groups][2 buffers] S of the buffer's tile written
    uint64_t* p_full = s_full + 4;        // [2][2] P of the buffer's tile written (4 warps)
    uint64_t* o_done = p_full + 4;        // [2][2] value MMAs of the buffer's tile done
    uint64_t* q_full = o_done + 4;        // both groups' Q in shared memory
    uint64_t* fin = q_full + 1;           // [4] every MMA an issuing lane issued has completed
    constexpr int NBARS = 2 * NK + 2 * NV + 17;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 8 * NBARS + 4);
    uint32_t* bad_mask = reinterpret_cast<uint32_t*>(ctl + 8 * NBARS + 8);
    static_assert(8 * NBARS + 8 + 4 * NK <= C::CTL_BYTES, "control block");
    static_assert(4 * (kPfxOrderSeqs + 1) <= C::CTL_BYTES, "sequence-order scratch");

    // Barrier phases: S buffer b of group g holds tiles b, b + 2, ...; the score MMA of tile t
    // waits for the value MMA of tile t - 2 (o_done), the softmax of tile t for its scores
    // (s_full), the value MMA of tile t for P (p_full).  Each wait is for a phase its waiter
    // is the only one to pass, and no barrier can complete a second phase before that.
    if (tid == 0) {
        for (int i = 0; i < NK; ++i) {
            mbar_init(&k_full[i], 2);           // the copy arrive (+ bytes) and the key warp
            mbar_init(&k_empty[i], 5 * ng);  // each group's score-MMA commit and its softmax warps
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&v_full[i], 2);
            mbar_init(&v_empty[i], ng);  // each group's value-MMA commit
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(q_full, 4 * ng);
        for (int i = 0; i < 4; ++i) mbar_init(&fin[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    pfx_zero_padding<C, D>(smem, p, tid, kP2Threads);
    fence_proxy_async_smem();
    if (warp == kP2MmaWarp) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;
    const int32_t* table = p.block_tables + (int64_t)s * p.mbps;
    const PfxRange rng{tb, n_ctx, ctx, n_tiles, q0, q_len, kvh, table};

    if (warp == kP2KeyWarp || warp == kP2ValWarp) {
        // ------------------------------------------------------------------ loaders
        pfx_load_tiles<C, D, 32>(p, rng, warp == kP2KeyWarp, lane, lane, sbase, k_full, k_empty, v_full, v_empty,
                                 bad_mask, abort_flag);
    } else if (warp == kP2MmaWarp || warp == kP2MmaWarp1) {
        // ------------------------------------------------------------------ score MMAs
        const int g = warp == kP2MmaWarp1 ? 1 : 0;
        if (lane == 0 && g < ng) {
            const uint64_t kd0 = umma_desc(sbase + C::OFF_K, 128, C::DP * 16);
            const uint32_t kd_lo = (uint32_t)kd0, kd_hi = (uint32_t)(kd0 >> 32);
            // Q of group g: [chunk][128 rows][16 bytes] at OFF_Q + g * QG_BYTES; a K step (16 head
            // elements) is two chunks, 4 KiB apart
            const uint64_t qd0 = umma_desc(sbase + C::OFF_Q, kPfxBM * 16, 128);
            const uint32_t qd_lo = (uint32_t)qd0, qd_hi = (uint32_t)(qd0 >> 32);
            bool ok = pfx_wait(q_full, 0, abort_flag);
            for (int t = 0; ok && t < n_tiles; ++t) {
                ok = pfx_wait(&k_full[t % NK], (t / NK) & 1, abort_flag);
                const uint32_t k_lo = kd_lo + (uint32_t)((t % NK) * (C::K_BYTES >> 4));
                // this tile's S buffer held P of tile t - 2: its value MMA must be done
                if (ok && t >= 2) ok = pfx_wait(&o_done[g * 2 + (t & 1)], ((t - 2) >> 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_s = tm + g * 256 + (t & 1) * BN;
                const uint32_t q_lo = qd_lo + (uint32_t)(g * (C::QG_BYTES >> 4));
#pragma unroll
                for (int ks = 0; ks < C::DP / 16; ++ks)
                    umma_f16_ss(d_s, q_lo + ks * (2 * kPfxBM), qd_hi, k_lo + ks * 16, kd_hi, C::IDESC_S,
                                ks > 0 ? 1u : 0u);
                umma_commit(&s_full[g * 2 + (t & 1)]);
                umma_commit(&k_empty[t % NK]);
            }
            umma_commit(&fin[2 * g]);
            if (!mbar_wait_bounded(&fin[2 * g], 0, kWaitLimitNs)) prefix_flag(4u);
        }
        __syncwarp();
    } else if (warp == kP2PvWarp || warp == kP2PvWarp1) {
        // ------------------------------------------------------------------ value MMAs
        const int g = warp == kP2PvWarp1 ? 1 : 0;
        if (lane == 0 && g < ng) {
            const uint64_t vd0 = p.bs_log2 == 3   ? umma_desc(sbase + C::OFF_V, C::DP * 16, 128)
                                 : p.bs_log2 == 4 ? umma_desc_sw(sbase + C::OFF_V, 256, 6)
                                                  : umma_desc_sw(sbase + C::OFF_V, 512, 4);
            const uint32_t vd_lo = (uint32_t)vd0, vd_hi = (uint32_t)(vd0 >> 32);
            uint32_t voff[BN / 16];
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                voff[kk] = (uint32_t)(p.bs_log2 == 3   ? kk * 2 * (C::DP * 16)
                                      : p.bs_log2 == 4 ? kk * (C::DP * 32)
                                                       : (kk >> 1) * (C::DP * 64) + (kk & 1) * 32) >> 4;
            bool ok = true;
            for (int t = 0; ok && t < n_tiles; ++t) {
                ok = pfx_wait(&v_full[t % NV], (t / NV) & 1, abort_flag);
                const uint32_t v_lo = vd_lo + (uint32_t)((t % NV) * (C::V_BYTES >> 4));
                const uint32_t acc0 = t > 0 ? 1u : 0u;
                if (ok) ok = pfx_wait(&p_full[g * 2 + (t & 1)], (t >> 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                // P of this tile: its S buffer, bf16 hi in the first 32 columns, lo in the next 32
                const uint32_t a_p = tm + g * 256 + (t & 1) * BN;
#pragma unroll
                for (int h = 0; h < C::NP; ++h)
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        umma_f16_ts(tm + g * 256 + C::COL_O, a_p + h * (BN / 2) + kk * 8, v_lo + voff[kk], vd_hi,
                                    C::IDESC_O, (kk > 0 || h > 0) ? 1u : acc0);
                umma_commit(&o_done[g * 2 + (t & 1)]);
                umma_commit(&v_empty[t % NV]);
            }
            umma_commit(&fin[2 * g + 1]);
            if (!mbar_wait_bounded(&fin[2 * g + 1], 0, kWaitLimitNs)) prefix_flag(4u);
        }
        __syncwarp();
    } else if (warp >= kP2SoftmaxWarp0 && warp < kP2SoftmaxWarp0 + 8 && (warp - kP2SoftmaxWarp0) / 4 < ng) {
        // ------------------------------------------------------------------ softmax
        const int g = (warp - kP2SoftmaxWarp0) / 4;
        const int sw = warp & 3;  // tensor-memory lane quarter
        const int r = sw * 32 + lane;
        const int row = row0 + g * kPfxBM + r;
        const int lim = row / G;
        const uint32_t tl = tm + g * 256 + ((uint32_t)(sw * 32) << 16);
        {
            const uint8_t* qrow = nullptr;
            if (row < rows_total) {
                const int j = row / G, gg = row - j * G;
                qrow = p.q + ((int64_t)(q0 + j) * p.q_stride + (int64_t)(kvh * G + gg) * D) * 2;
            }
            const uint32_t sQ = sbase + C::OFF_Q + g * C::QG_BYTES + r * 16;
            for (int c = 0; c < C::NCP; ++c) {
                uint4 a = make_uint4(0u, 0u, 0u, 0u);
                if (qrow != nullptr && c < C::NCR) a = ld_nc_v4(qrow + c * 16);
                sts_v4(sQ + c * (kPfxBM * 16), a.x, a.y, a.z, a.w);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < n_tiles; ++t) {
            const int ks = t % NK;
            const int b = g * 2 + (t & 1);
            ok = pfx_warp_wait(&k_full[ks], (t / NK) & 1, abort_flag, lane) &&
                 pfx_warp_wait(&s_full[b], (t >> 1) & 1, abort_flag, lane);
            if (!ok) break;
            tc_fence_after();
            const uint32_t ts = tl + (t & 1) * BN;
            float sv[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(ts + c * 32, *reinterpret_cast<float(*)[32]>(&sv[c * 32]));
            const uint32_t bad = t < n_ctx ? bad_mask[ks] : 0u;
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&k_empty[ks]);

            if (t < n_ctx) {
                const int valid = min(BN, ctx - (tb + t) * BN);
                if (valid < BN || bad) {
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (i >= valid || ((bad >> (i >> p.bs_log2)) & 1u)) sv[i] = -INFINITY;
                }
            } else {
                const int lim_t = lim - (t - n_ctx) * BN;
                if (lim_t < BN - 1) {
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (i > lim_t) sv[i] = -INFINITY;
                }
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < BN / 2; ++e) mx[e & 3] = fmax3(mx[e & 3], sv[2 * e], sv[2 * e + 1]);
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.sl2;
            const bool need = mt > m_ref + 8.f;
            float corr = 1.f;
            if (need) {
                corr = ex2(m_ref - mt);
                m_ref = mt;
                l *= corr;
            }
            const float mu = m_ref == -INFINITY ? 0.f : m_ref;
            const float2 sl2v = make_float2(p.sl2, p.sl2), nmu = make_float2(-mu, -mu);
            float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t ph[BN / 2], pl[BN / 2];
#pragma unroll
            for (int e = 0; e < BN / 2; ++e) {
                const float2 x = ffma2(make_float2(sv[2 * e], sv[2 * e + 1]), sl2v, nmu);
                const float a = ex2(x.x), bb = ex2(x.y);
                sum2[e & 1] = fadd2(sum2[e & 1], make_float2(a, bb));
                const uint32_t h2 = pack2<BF16>(a, bb);
                ph[e] = h2;
                if constexpr (BF16) {
                    const float2 d = fsub2(make_float2(a, bb),
                                           make_float2(__uint_as_float(h2 << 16), __uint_as_float(h2 & 0xffff0000u)));
                    pl[e] = pack2<BF16>(d.x, d.y);
                }
            }
            l += (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
            // O holds every earlier tile before it is rescaled
            if (t > 0 && __any_sync(0xffffffffu, need)) {
                if (!(ok = pfx_warp_wait(&o_done[g * 2 + ((t - 1) & 1)], ((t - 1) >> 1) & 1, abort_flag, lane))) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < C::DPR / 32; ++c) {
                    float o[32];
                    tmem_ld32(tl + C::COL_O + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= corr;
                    tmem_st32(tl + C::COL_O + c * 32, o);
                }
                tmem_wait_st();
            }
            // P into the S buffer just read (bf16: hi, then lo)
            tmem_st32(ts, *reinterpret_cast<const float(*)[32]>(&ph[0]));
            if constexpr (BF16) tmem_st32(ts + BN / 2, *reinterpret_cast<const float(*)[32]>(&pl[0]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[b]);
        }
        if (ok && n_tiles > 0)
            ok = pfx_warp_wait(&o_done[g * 2 + ((n_tiles - 1) & 1)], ((n_tiles - 1) >> 1) & 1, abort_flag, lane);
        if (ok && plan.x > 1) {
            tc_fence_after();
            const int64_t item = (((int64_t)s * p.Hk + kvh) * p.mt_ws + row / kPfxBM) * p.nsplit + split;
            float* wrow = row < rows_total ? p.ws_o + (item * kPfxBM + r) * D : nullptr;
#pragma unroll 1
            for (int c = 0; c < C::DPR / 32; ++c) {
                float o[32];
                tmem_ld32(tl + C::COL_O + c * 32, o);
                tmem_wait_ld();
                if (wrow != nullptr) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (c * 32 + q * 4 < D)
                            *reinterpret_cast<float4*>(wrow + c * 32 + q * 4) =
                                make_float4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]);
                }
            }
            if (wrow != nullptr) p.ws_ml[item * kPfxBM + r] = make_float2(m_ref, l);
        } else if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            uint8_t* orow = nullptr;
            if (row < rows_total) {
                const int j = row / G, gg = row - j * G;
                orow = static_cast<uint8_t*>(p.out) + ((int64_t)(q0 + j) * p.H + kvh * G + gg) * (D * 2);
            }
#pragma unroll 1
            for (int c = 0; c < C::DPR / 32; ++c) {
                float o[32];
                tmem_ld32(tl + C::COL_O + c * 32, o);
                tmem_wait_ld();
                if (orow != nullptr) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int col = c * 32 + q * 8;
                        if (col < D) {
                            uint4 w;
                            w.x = pack2<BF16>(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv);
                            w.y = pack2<BF16>(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv);
                            w.z = pack2<BF16>(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv);
                            w.w = pack2<BF16>(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv);
                            *reinterpret_cast<uint4*>(orow + col * 2) = w;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kP2MmaWarp) tmem_dealloc(tm, C::TMEM_COLS);
}

template <bool BF16, int D>
cudaError_t launch_prefix_m256(const PrefixParams& p, dim3 grid, cudaStream_t stream) {
    using C = Pfx2Cfg<BF16, D>;
    cudaError_t e =
        cudaFuncSetAttribute(pa_prefix_m256_kernel<BF16, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    pa_prefix_m256_kernel<BF16, D><<<grid, kP2Threads, C::SMEM, stream>>>(p);
    return cudaGetLastError();
}

#ifndef PA_PFX_M256
#define PA_PFX_M256 1
#endif

// Kernel for (query dtype, head size): 256 rows per CTA up to head size 128 (PA_PFX_M256),
// else 128 rows per CTA; nullptr for an unsupported head size.
template <bool BF16>
PrefixFn prefix_select(int d) {
    switch (d) {
        case 64: return PA_PFX_M256 ? launch_prefix_m256<BF16, 64> : launch_prefix_kernel<BF16, 64>;
        case 80: return PA_PFX_M256 ? launch_prefix_m256<BF16, 80> : launch_prefix_kernel<BF16, 80>;
        case 96: return PA_PFX_M256 ? launch_prefix_m256<BF16, 96> : launch_prefix_kernel<BF16, 96>;
        case 112: return PA_PFX_M256 ? launch_prefix_m256<BF16, 112> : launch_prefix_kernel<BF16, 112>;
        case 120: return PA_PFX_M256 ? launch_prefix_m256<BF16, 120> : launch_prefix_kernel<BF16, 120>;
        case 128: return PA_PFX_M256 ? launch_prefix_m256<BF16, 128> : launch_prefix_kernel<BF16, 128>;
        case 192: return launch_prefix_kernel<BF16, 192>;
        case 256: return launch_prefix_kernel<BF16, 256>;
        default: return nullptr;
    }
}

template <bool BF16>
int prefix_tile_rows(int d) {
    return PA_PFX_M256 && d <= 128 ? kP2Rows : kPfxBM;
}

}  // namespace pa
