// pa_prefix.cuh -- chunked-prefix (prefill) attention over the paged cache for sm_103a.
// "paged_attn.py", forward_prefix / _forward_prefix_pytorch.
//
// Sequence s has ctx = context_lens[s] tokens in the paged cache and q_len new tokens whose
// query/key/value rows are dense (rows query_start_loc[s] .. query_start_loc[s+1]-1).  New
// token j of query head h sees every context token (no mask) and new tokens 0..j (causal),
// through kv head h / G:  out = softmax(scale * q K^T) V.
//
// One CTA owns (sequence, kv head, 128 query rows), a row being a (new token j, head g of
// the kv head's group) pair numbered j * G + g, so every key/value tile is read once per
// kv head and shared by the whole GQA group.  Eight warps hold 16 rows each; the scores of
// a 64-key tile are an m16n8k16 product with the query rows in shared memory and the keys
// straight from the copied pages (a key page [d/8][block_size][8] already has the 16-byte
// rows ldmatrix wants); the probabilities stay in registers as the A operand of the value
// product (fp32 accumulators, online softmax with exp2).  Tiles move global -> shared with
// 16-byte cp.async in a two-stage pipeline: context tiles page by page from the cache,
// chunk tiles from the dense rows.  Value tiles are [d][64 tokens] for context pages (rows
// of a value page) and [64 tokens][d] for dense rows (read with ldmatrix.trans).  Row
// strides carry 16 bytes of padding so the eight rows of every ldmatrix fall in distinct
// bank groups.  Masked keys never reach the value product as NaN: value chunks past the
// context or of an invalid page are zero-filled by the copy itself.
#pragma once

#include "pa_kernels.cuh"
#include "pa_ptx.cuh"

namespace pa {

template <int D>
struct PfxGeom {
    static constexpr int DP = (D + 15) / 16 * 16;  // head size padded to the MMA k step
    static constexpr int NCR = D / 8;              // 16-byte chunks of a row that exist
    static constexpr int NCP = DP / 8;             // chunks after padding
    static constexpr int RS = DP * 2 + 16;         // query / dense-value row stride, bytes
    static constexpr int VRS = kPfxBN * 2 + 16;    // paged-value row stride (one d row), bytes
    static constexpr int Q_BYTES = kPfxBM * RS;
    static constexpr int K_BYTES = NCP * kPfxBN * 16;
    static constexpr int V_BYTES = (DP * VRS > kPfxBN * RS) ? DP * VRS : kPfxBN * RS;
    static constexpr int STAGE = K_BYTES + V_BYTES;
    static constexpr int SMEM = Q_BYTES + kPfxStages * STAGE + 16 * kPfxStages;
    static constexpr int MIN_CTAS = DP <= 128 ? 2 : 1;
};

static __device__ unsigned int g_prefix_errors = 0;

__device__ __forceinline__ void prefix_flag(unsigned int bit) { atomicOr(&g_prefix_errors, bit); }

template <bool BF16, int D>
__global__ void __launch_bounds__(kPfxThreads, PfxGeom<D>::MIN_CTAS) pa_prefix_kernel(const PrefixParams p) {
    using Gm = PfxGeom<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.z, kvh = blockIdx.y;
    const int row0 = (gridDim.x - 1 - blockIdx.x) * kPfxBM;  // row tiles with more keys first
    const int G = p.G;
    const int q0 = p.qsl[s];
    const int q_len = p.qsl[s + 1] - q0;
    int ctx = p.ctx_lens[s];
    if (q_len < 0 || q_len > p.max_query_len || ctx < 0) {
        if (tid == 0) prefix_flag(128u);
        return;
    }
    const int rows_total = q_len * G;
    if (row0 >= rows_total) return;
    if (ctx > p.mbps * p.bs) {  // the table cannot hold the context: cap it (and report)
        if (tid == 0) prefix_flag(64u);
        ctx = p.mbps * p.bs;
    }

    const uint32_t sQ = smem_addr(smem);
    const uint32_t sStage0 = sQ + Gm::Q_BYTES;
    uint32_t* sflags = reinterpret_cast<uint32_t*>(smem + Gm::Q_BYTES + kPfxStages * Gm::STAGE);

    // Padding chunks of the key tiles are never copied: zero them once so that the zero
    // query padding meets zeros, not stale bits.
    if constexpr (Gm::NCP > Gm::NCR) {
        constexpr int per = (Gm::NCP - Gm::NCR) * kPfxBN;
        for (int idx = tid; idx < kPfxStages * per; idx += kPfxThreads) {
            const int st = idx / per, rem = idx % per;
            const int c = Gm::NCR + rem / kPfxBN, o = rem % kPfxBN;
            *reinterpret_cast<uint4*>(smem + Gm::Q_BYTES + st * Gm::STAGE + c * (kPfxBN * 16) + o * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }

    // Query rows of this tile (rows past the chunk and padding chunks read as zero).
    for (int idx = tid; idx < kPfxBM * Gm::NCP; idx += kPfxThreads) {
        const int r = idx / Gm::NCP, c = idx % Gm::NCP;
        const int row = row0 + r;
        const uint8_t* src = p.q;
        uint32_t nb = 0;
        if (row < rows_total && c < Gm::NCR) {
            const int j = row / G, g = row - (row / G) * G;
            src = p.q + ((int64_t)(q0 + j) * p.q_stride + (int64_t)(kvh * G + g) * D + c * 8) * 2;
            nb = 16;
        }
        cp_async16(sQ + r * Gm::RS + c * 16, src, nb);
    }

    const int n_ctx = (ctx + kPfxBN - 1) / kPfxBN;
    const int row_last = min(row0 + kPfxBM, rows_total) - 1;
    const int jmin = row0 / G;
    const int n_chunk = (row_last / G) / kPfxBN + 1;
    const int n_tiles = n_ctx + n_chunk;
    const int32_t* table = p.block_tables + (int64_t)s * p.mbps;
    const int64_t page_bytes = (int64_t)D * p.bs * 2;

    auto load_tile = [&](int t, int st) {
        const uint32_t sK = sStage0 + st * Gm::STAGE, sV = sK + Gm::K_BYTES;
        if (t < n_ctx) {
            const int t0 = t * kPfxBN;
            // keys: this thread's token o = tid % 64 is the same for all of its chunks
            {
                const int o = tid % kPfxBN;
                const bool live = t0 + o < ctx;
                const int b = live ? table[(t0 + o) >> p.bs_log2] : -1;
                const bool ok = live && (unsigned)b < (unsigned)p.num_blocks;
                const uint8_t* kp = ok ? p.kcache + ((int64_t)b * p.Hk + kvh) * page_bytes : p.kcache;
                const int slot = (o & (p.bs - 1)) * 16;
#pragma unroll
                for (int c = tid / kPfxBN; c < Gm::NCR; c += kPfxThreads / kPfxBN)
                    cp_async16(sK + c * (kPfxBN * 16) + o * 16, kp + (int64_t)c * p.bs * 16 + slot, ok ? 16u : 0u);
            }
            // values: this thread's 8-token chunk kc = tid % 8 (inside one page)
            {
                const int kc = tid % 8, o = kc * 8;
                const int nv = min(max(ctx - t0 - o, 0), 8);
                const int b = nv > 0 ? table[(t0 + o) >> p.bs_log2] : -1;
                const bool ok = nv > 0 && (unsigned)b < (unsigned)p.num_blocks;
                const uint8_t* vp = ok ? p.vcache + ((int64_t)b * p.Hk + kvh) * page_bytes : p.vcache;
                const int slot = (o & (p.bs - 1)) * 2;
                for (int dd = tid / 8; dd < D; dd += kPfxThreads / 8)
                    cp_async16(sV + dd * Gm::VRS + kc * 16, vp + (int64_t)dd * p.bs * 2 + slot,
                               ok ? (uint32_t)nv * 2u : 0u);
            }
            // pages of this tile whose id is outside the cache: masked, and reported
            if (warp == 0) {
                const int npg = kPfxBN >> p.bs_log2;
                bool bad = false;
                if (lane < npg) {
                    const int first = t0 + (lane << p.bs_log2);
                    if (first < ctx) {
                        const int b = table[first >> p.bs_log2];
                        bad = (unsigned)b >= (unsigned)p.num_blocks;
                    }
                }
                const uint32_t m = __ballot_sync(0xffffffffu, bad);
                if (lane == 0) {
                    sflags[st * 4] = m;
                    if (m) prefix_flag(32u);
                }
            }
        } else {
            const int kc0 = (t - n_ctx) * kPfxBN;
            {
                const int o = tid % kPfxBN;
                const int j = kc0 + o;
                const bool ok = j < q_len;
                const uint8_t* kr = ok ? p.k + ((int64_t)(q0 + j) * p.kv_stride + (int64_t)kvh * D) * 2 : p.k;
#pragma unroll
                for (int c = tid / kPfxBN; c < Gm::NCR; c += kPfxThreads / kPfxBN)
                    cp_async16(sK + c * (kPfxBN * 16) + o * 16, kr + c * 16, ok ? 16u : 0u);
            }
            for (int idx = tid; idx < kPfxBN * Gm::NCR; idx += kPfxThreads) {
                const int o = idx / Gm::NCR, c = idx % Gm::NCR;
                const int j = kc0 + o;
                const bool ok = j < q_len;
                const uint8_t* vr = ok ? p.v + ((int64_t)(q0 + j) * p.kv_stride + (int64_t)kvh * D) * 2 + c * 16 : p.v;
                cp_async16(sV + o * Gm::RS + c * 16, vr, ok ? 16u : 0u);
            }
        }
    };

    // Per-thread rows: r_a and r_a + 8 of the CTA's 128; their causal limits in the chunk.
    const int r_a = warp * 16 + (lane >> 2);
    int lim[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) lim[i] = (row0 + r_a + 8 * i) / G;

    float acc[Gm::DP / 8][4];
#pragma unroll
    for (int n = 0; n < Gm::DP / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

    load_tile(0, 0);
    cp_async_commit();

    for (int t = 0; t < n_tiles; ++t) {
        const int st = t & 1;
        if (t + 1 < n_tiles) load_tile(t + 1, st ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const uint32_t sK = sStage0 + st * Gm::STAGE, sV = sK + Gm::K_BYTES;
        const bool is_ctx = t < n_ctx;

        // S = Q K^T for this warp's 16 rows and the tile's 64 keys
        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < Gm::DP / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sQ + (warp * 16 + (lane & 15)) * Gm::RS + (2 * ks + (lane >> 4)) * 16, a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                const int tok = np * 16 + ((lane >> 4) << 3) + (lane & 7);
                const int ch = 2 * ks + ((lane >> 3) & 1);
                ldsm_x4(sK + ch * (kPfxBN * 16) + tok * 16, b0, b1, b2, b3);
                mma16816<BF16>(sc[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816<BF16>(sc[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }

        // scale into the exp2 domain, then mask
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[n][e] *= p.sl2;
        if (is_ctx) {
            const int valid = min(kPfxBN, ctx - t * kPfxBN);
            const uint32_t bad = sflags[st * 4];
            if (valid < kPfxBN || bad) {
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = n * 8 + (lane & 3) * 2 + (e & 1);
                        if (col >= valid || ((bad >> (col >> p.bs_log2)) & 1u)) sc[n][e] = -INFINITY;
                    }
            }
        } else {
            const int kc0 = (t - n_ctx) * kPfxBN;
            if (kc0 + kPfxBN - 1 > jmin) {
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = kc0 + n * 8 + (lane & 3) * 2 + (e & 1);
                        if (key > lim[e >> 1]) sc[n][e] = -INFINITY;
                    }
            }
        }

        // online softmax (row max over the quad that shares a row)
        float corr[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(sc[n][2 * i], sc[n][2 * i + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m_r[i], mx);
            const float mu = mn == -INFINITY ? 0.f : mn;
            corr[i] = ex2(m_r[i] - mu);
            m_r[i] = mn;
            float sum = 0.f;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                sc[n][2 * i] = ex2(sc[n][2 * i] - mu);
                sc[n][2 * i + 1] = ex2(sc[n][2 * i + 1] - mu);
                sum += sc[n][2 * i] + sc[n][2 * i + 1];
            }
            l_r[i] = l_r[i] * corr[i] + sum;
        }
#pragma unroll
        for (int n = 0; n < Gm::DP / 8; ++n) {
            acc[n][0] *= corr[0];
            acc[n][1] *= corr[0];
            acc[n][2] *= corr[1];
            acc[n][3] *= corr[1];
        }

        // O += P V; bf16 probabilities go in as hi + lo so they carry f16-like precision
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t pa[4], pl[4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float x0 = sc[2 * kk + h][2 * i], x1 = sc[2 * kk + h][2 * i + 1];
                    pa[2 * h + i] = pack2<BF16>(x0, x1);
                    if constexpr (BF16) {
                        const float h0 = __uint_as_float(pa[2 * h + i] << 16);
                        const float h1 = __uint_as_float(pa[2 * h + i] & 0xffff0000u);
                        pl[2 * h + i] = pack2<BF16>(x0 - h0, x1 - h1);
                    }
                }
            if (is_ctx) {
#pragma unroll
                for (int np = 0; np < Gm::DP / 16; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int dd = np * 16 + ((lane >> 4) << 3) + (lane & 7);
                    const int ch = 2 * kk + ((lane >> 3) & 1);
                    ldsm_x4(sV + dd * Gm::VRS + ch * 16, b0, b1, b2, b3);
                    mma16816<BF16>(acc[2 * np], pa[0], pa[1], pa[2], pa[3], b0, b1);
                    mma16816<BF16>(acc[2 * np + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
                    if constexpr (BF16) {
                        mma16816<BF16>(acc[2 * np], pl[0], pl[1], pl[2], pl[3], b0, b1);
                        mma16816<BF16>(acc[2 * np + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
                    }
                }
            } else {
#pragma unroll
                for (int np = 0; np < Gm::DP / 16; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int tok = kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
                    const int ch = 2 * np + (lane >> 4);
                    ldsm_x4_trans(sV + tok * Gm::RS + ch * 16, b0, b1, b2, b3);
                    mma16816<BF16>(acc[2 * np], pa[0], pa[1], pa[2], pa[3], b0, b1);
                    mma16816<BF16>(acc[2 * np + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
                    if constexpr (BF16) {
                        mma16816<BF16>(acc[2 * np], pl[0], pl[1], pl[2], pl[3], b0, b1);
                        mma16816<BF16>(acc[2 * np + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // normalise and store the rows that exist
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float l = l_r[i];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const float inv = 1.f / l;
        const int row = row0 + r_a + 8 * i;
        if (row < rows_total) {
            const int j = row / G, g = row - (row / G) * G;
            uint8_t* orow = static_cast<uint8_t*>(p.out) + ((int64_t)(q0 + j) * p.H + kvh * G + g) * (D * 2);
#pragma unroll
            for (int n = 0; n < Gm::DP / 8; ++n) {
                const int col = n * 8 + (lane & 3) * 2;
                if (col < D)
                    *reinterpret_cast<uint32_t*>(orow + col * 2) =
                        pack2<BF16>(acc[n][2 * i] * inv, acc[n][2 * i + 1] * inv);
            }
        }
    }
}

template <bool BF16, int D>
cudaError_t launch_prefix_kernel(const PrefixParams& p, dim3 grid, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(pa_prefix_kernel<BF16, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PfxGeom<D>::SMEM);
    if (e != cudaSuccess) return e;
    pa_prefix_kernel<BF16, D><<<grid, kPfxThreads, PfxGeom<D>::SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <bool BF16>
PrefixFn prefix_select(int d) {
    switch (d) {
        case 64: return launch_prefix_kernel<BF16, 64>;
        case 80: return launch_prefix_kernel<BF16, 80>;
        case 96: return launch_prefix_kernel<BF16, 96>;
        case 112: return launch_prefix_kernel<BF16, 112>;
        case 120: return launch_prefix_kernel<BF16, 120>;
        case 128: return launch_prefix_kernel<BF16, 128>;
        case 192: return launch_prefix_kernel<BF16, 192>;
        case 256: return launch_prefix_kernel<BF16, 256>;
        default: return nullptr;
    }
}

template <bool BF16>
cudaError_t prefix_read_errors(unsigned int* v, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_prefix_errors, sizeof(*v));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_prefix_errors, &z, sizeof(z));
}

}  // namespace pa
