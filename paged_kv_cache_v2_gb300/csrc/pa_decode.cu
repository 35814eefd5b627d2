// pa_decode.cu -- PagedAttention V2 single-query decode for sm_103a (GB300).
//
// What is computed ("paged_attention_v2_pytorch.py", paged_attention_v2_pytorch, and
// "paged_attention_v2_triton.py", _paged_attn_v2_reduce_kernel): for every sequence s,
// query head h and 512-token partition p, the scores s_t = scale * <q, k_t> * k_scale
// (+ slope_h * t), the partition max m_p, exp-sum l_p and normalised weighted V; then the
// log-sum-exp combine of the partitions into the output.
//
// How (GB300-first; the pages' PyTorch/Triton code is prior art, not the blueprint):
//  * Phase 1, one CTA per (partition, kv head, <= 8 query heads of that kv head, sequence):
//    every K and V byte of a partition is read from HBM once and serves all query heads
//    of its GQA group.  Four warps each own a ring of shared-memory slots; a slot holds
//    the K page and the V page of one (or two, for block size 8) cache block(s).  Each
//    page is one contiguous span (head_size * block_size elements), so it moves with ONE
//    1-D bulk copy (TMA engine, L2 evict-first) that completes on the slot's mbarrier; the
//    warp refills a slot as soon as it has consumed it, keeping several pages in flight.
//  * Scores and P.V run on the tensor cores with warp-level m16n8k16 MMA (fp32
//    accumulate): 16 tokens x 8 query heads per MMA, K rows fed straight from the x-packed
//    page with ldmatrix, V^T rows straight from the token-contiguous page, P moved from
//    the score fragment into the P.V operand with movmatrix.  fp8 e4m3 pages are widened
//    to f16 in registers (exact) for both products (a bf16 query is scaled per head by a
//    power of two into f16, also exact); k_scale and the softmax scale fold into one fp32
//    multiplier on the scores, v_scale into the final normalisation.
//  * The online softmax runs per warp in the base-2 domain; the warps' (m, l, acc) merge
//    through shared memory at the end of the partition.  A one-partition sequence writes
//    its normalised output directly (single pass); longer ones write tmp_output and the
//    statistics for phase 2.
//  * Phase 2, one CTA per (query head, sequence) with more than one partition: global max,
//    weights exp(m_p - g) l_p, and the weighted sum of the tmp_output rows (float4 loads,
//    eight warps over the partitions).  It is launched with programmatic dependent launch
//    so its launch overlaps the tail of phase 1.
//  * No spin-wait is unbounded: every mbarrier wait gives up after 2 s, records a device
//    error flag and drains its own copies (again bounded) before the block exits.  Bad
//    table entries are masked and flagged instead of being dereferenced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "pa_v2.h"
#include "pa_internal.h"
#include "pa_kernels.cuh"
#include "pa_prefix.h"
#include "pa_ptx.cuh"

namespace pa {

// ---------------------------------------------------------------------------------------
// Phase 2: log-sum-exp combine across partitions
// ---------------------------------------------------------------------------------------
// One CTA per (query head, sequence) with more than one partition; W warps (chosen from
// max_num_partitions on the host).  Warp w folds partitions w, w + W, ... into a running
// (m, l, acc) with the online rescaling, so its loads of max_logits, exp_sums and tmp rows
// do not wait on one another; the W partial states merge through shared memory.
// The combine is the pages' formula: g = max_p m_p, w_p = exp(m_p - g) l_p,
// out = sum_p w_p tmp_p / sum_p w_p.
constexpr int kP2MaxWarps = 16;
constexpr int kP2MaxCols = 2;  // float4 columns per lane: head_size <= 256
constexpr int kP2Pre = 8;      // partitions per warp and chunk whose tmp rows load up front

// four consecutive tmp_output elements of one partition row as fp32
template <bool BF16, bool TMP16>
__device__ __forceinline__ float4 load_tmp4(const void* base, int64_t idx4) {
    if constexpr (TMP16) {
        const uint2 w = reinterpret_cast<const uint2*>(base)[idx4];
        float4 r;
        if constexpr (BF16) {
            r.x = __uint_as_float(w.x << 16);
            r.y = __uint_as_float(w.x & 0xffff0000u);
            r.z = __uint_as_float(w.y << 16);
            r.w = __uint_as_float(w.y & 0xffff0000u);
        } else {
            r.x = f16_lo_to_f32(w.x);
            r.y = f16_hi_to_f32(w.x);
            r.z = f16_lo_to_f32(w.y);
            r.w = f16_hi_to_f32(w.y);
        }
        return r;
    } else {
        return reinterpret_cast<const float4*>(base)[idx4];
    }
}

template <bool BF16, bool TMP16>
__global__ void __launch_bounds__(kP2MaxWarps * 32)
pa_v2_phase2_kernel(const Phase2Params p) {
    extern __shared__ float sm2[];  // [W][D] partial sums
    __shared__ float wm[kP2MaxWarps], wl[kP2MaxWarps];
    const int h = blockIdx.x, s = blockIdx.y;
    // seq_lens is an input of the decode call: phase 1, which this kernel follows, read it
    // after its own dependency wait, so it can be read before this kernel's wait
    const int L = p.seq_lens[s];
    griddep_wait();
    const int P = min(L > 0 ? (L + kPartition - 1) / kPartition : 0, p.Pmax);
    if (P <= 1) return;  // written by phase 1 (single pass or empty)
    const int D = p.D, nq = D / 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
    const int64_t row = (int64_t)s * p.H + h;
    const float* ml = p.max_logits + row * p.Pmax;
    const float* es = p.exp_sums + row * p.Pmax;
    const int64_t tmp4 = row * p.Pmax * nq;  // first float4 group of this (sequence, head)

    // Warp w owns partitions w, w + W, ...  Their statistics load one per lane (32 at a
    // time) and reduce with shuffles; the tmp rows then stream with independent loads.
    float m = -INFINITY, l = 0.f;
    float4 acc[kP2MaxCols];
#pragma unroll
    for (int k = 0; k < kP2MaxCols; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int mine = P > warp ? (P - warp + W - 1) / W : 0;  // partitions of this warp
    for (int j0 = 0; j0 < mine; j0 += 32) {
        const int nc = min(32, mine - j0);
        // the tmp rows of this chunk's first kP2Pre partitions, loaded together with the
        // statistics that weight them rather than after them (one memory round trip fewer)
        float4 pre[kP2Pre][kP2MaxCols];
#pragma unroll
        for (int jj = 0; jj < kP2Pre; ++jj)
#pragma unroll
            for (int k = 0; k < kP2MaxCols; ++k) {
                const int c = lane + 32 * k;
                pre[jj][k] = jj < nc && c < nq
                                 ? load_tmp4<BF16, TMP16>(p.tmp_out, tmp4 + (warp + (int64_t)(j0 + jj) * W) * nq + c)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        float mj = -INFINITY, lj = 0.f;
        if (lane < nc) {
            const int i = warp + (j0 + lane) * W;
            mj = ml[i] * kLog2e;
            lj = es[i];
            if (!(lj > 0.f)) mj = -INFINITY;  // an all-masked partition adds nothing
        }
        float mc = mj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
        if (mc == -INFINITY) continue;
        const float wj = mj == -INFINITY ? 0.f : ex2(mj - mc) * lj;  // weight relative to mc
        float lc = wj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lc += __shfl_xor_sync(0xffffffffu, lc, o);
        float4 ac[kP2MaxCols];
#pragma unroll
        for (int k = 0; k < kP2MaxCols; ++k) ac[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int jj = 0; jj < kP2Pre; ++jj) {
            if (jj >= nc) break;  // nc is the same on every lane
            const float w = __shfl_sync(0xffffffffu, wj, jj);
#pragma unroll
            for (int k = 0; k < kP2MaxCols; ++k) {
                ac[k].x += w * pre[jj][k].x;
                ac[k].y += w * pre[jj][k].y;
                ac[k].z += w * pre[jj][k].z;
                ac[k].w += w * pre[jj][k].w;
            }
        }
#pragma unroll 4
        for (int jj = kP2Pre; jj < nc; ++jj) {
            const float w = __shfl_sync(0xffffffffu, wj, jj);
            const int64_t i = warp + (int64_t)(j0 + jj) * W;
#pragma unroll
            for (int k = 0; k < kP2MaxCols; ++k) {
                const int c = lane + 32 * k;
                if (c < nq) {
                    const float4 x = load_tmp4<BF16, TMP16>(p.tmp_out, tmp4 + i * nq + c);
                    ac[k].x += w * x.x;
                    ac[k].y += w * x.y;
                    ac[k].z += w * x.z;
                    ac[k].w += w * x.w;
                }
            }
        }
        // fold this chunk into the warp's running (m, l, acc)
        const float mn = fmaxf(m, mc);
        const float a = ex2(m - mn), b = ex2(mc - mn);  // m = -inf -> a = 0
        l = l * a + lc * b;
#pragma unroll
        for (int k = 0; k < kP2MaxCols; ++k) {
            acc[k].x = acc[k].x * a + ac[k].x * b;
            acc[k].y = acc[k].y * a + ac[k].y * b;
            acc[k].z = acc[k].z * a + ac[k].z * b;
            acc[k].w = acc[k].w * a + ac[k].w * b;
        }
        m = mn;
    }
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w]);
    float Lt = 0.f;
    for (int w = 0; w < W; ++w)
        if (wm[w] != -INFINITY) Lt += wl[w] * ex2(wm[w] - M);
    const float f = (m == -INFINITY) ? 0.f : ex2(m - M);
#pragma unroll
    for (int k = 0; k < kP2MaxCols; ++k) {
        const int c = lane + 32 * k;
        if (c < nq) {
            float* dst = sm2 + warp * D + 4 * c;
            dst[0] = acc[k].x * f;
            dst[1] = acc[k].y * f;
            dst[2] = acc[k].z * f;
            dst[3] = acc[k].w * f;
        }
    }
    __syncthreads();
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        float v = 0.f;
        for (int w = 0; w < W; ++w) v += sm2[w * D + i];
        store_out<BF16>(p.out, row * D + i, v * inv);
    }
}

// Phase 2, one warp per (sequence, query head) row and eight rows per CTA: the form for
// steps of at most 64 partitions and head size <= 128 (lane c holds output columns 4c..4c+3).
// A batch of many rows then needs few CTAs, and each row costs about one memory round trip:
// the statistics (two per lane) and the tmp rows of its first kP2RowChunk partitions load
// together, before any of them is used.
// ---------------------------------------------------------------------------------------
// Grid order: the sequences by decreasing partition count (most work first)
// ---------------------------------------------------------------------------------------
// One CTA: a counting sort on min(ceil(L / 512), kOrderBuckets - 1), largest first.  Within a
// bucket the order is whatever the shared-memory atomics give: it only schedules, and every
// sequence's results are the same in any order.
constexpr int kOrderThreads = 1024;
constexpr int kOrderMinSeqs = 16;  // below this the grid has few sequences to reorder
constexpr int kOrderedWaves = 8;     // an ordered grid's stride: about this many waves of CTAs
constexpr int kOrderedMaxParts = 16; // and at most this many partitions a CTA
constexpr int kOrderBuckets = 1024;

__global__ void __launch_bounds__(kOrderThreads) pa_v2_order_kernel(const int32_t* seq_lens, int S, int32_t* order) {
    __shared__ int cnt[kOrderBuckets];
    __shared__ int wsum[kOrderThreads / 32];
    // the lengths may come from the previous kernel in the stream
    griddep_wait();
    for (int b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) cnt[b] = 0;
    __syncthreads();
    // bucket 0 holds the most partitions
    auto bucket = [&](int L) {
        const int P = L > 0 ? (int)(((int64_t)L + kPartition - 1) / kPartition) : 0;
        return kOrderBuckets - 1 - min(P, kOrderBuckets - 1);
    };
    for (int i = threadIdx.x; i < S; i += blockDim.x) atomicAdd(&cnt[bucket(seq_lens[i])], 1);
    __syncthreads();
    // exclusive scan of the bucket counts (one bucket per thread: kOrderBuckets == blockDim.x)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int v = cnt[threadIdx.x];
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;  // inclusive sums of the warps
    }
    __syncthreads();
    cnt[threadIdx.x] = x - v + (warp > 0 ? wsum[warp - 1] : 0);
    __syncthreads();
    for (int i = threadIdx.x; i < S; i += blockDim.x) order[atomicAdd(&cnt[bucket(seq_lens[i])], 1)] = i;
    griddep_launch_dependents();
}

pa_status launch_order(const int32_t* seq_lens, int S, int32_t* order, cudaStream_t stream) {
    static_assert(kOrderBuckets == kOrderThreads, "one bucket per thread in the scan");
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kOrderThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, pa_v2_order_kernel, seq_lens, S, order) != cudaSuccess) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

constexpr int kP2RowsPerCta = 8;
constexpr int kP2RowChunk = 16;

template <bool BF16, bool TMP16>
__global__ void __launch_bounds__(kP2RowsPerCta * 32)
pa_v2_phase2_rows_kernel(const Phase2Params p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = (int64_t)blockIdx.x * kP2RowsPerCta + warp;  // s * H + h
    const bool live = row < (int64_t)p.S * p.H;
    // seq_lens is an input that phase 1 only read: safe to read before the wait
    const int L = live ? p.seq_lens[row / p.H] : 0;
    griddep_wait();
    const int P = min(L > 0 ? (L + kPartition - 1) / kPartition : 0, p.Pmax);
    if (!live || P <= 1) return;  // written by phase 1 (single pass or empty)
    const int nq = p.D / 4;
    const bool col = lane < nq;
    const float* ml = p.max_logits + row * p.Pmax;
    const float* es = p.exp_sums + row * p.Pmax;
    const int64_t tmp4 = row * p.Pmax * nq + lane;
    // issue every load of the first chunk before any arithmetic
    const float m0 = lane < P ? ml[lane] : -INFINITY, l0 = lane < P ? es[lane] : 0.f;
    const float m1 = lane + 32 < P ? ml[lane + 32] : -INFINITY, l1 = lane + 32 < P ? es[lane + 32] : 0.f;
    float4 x[kP2RowChunk];
#pragma unroll
    for (int j = 0; j < kP2RowChunk; ++j)
        x[j] = (j < P && col) ? load_tmp4<BF16, TMP16>(p.tmp_out, tmp4 + (int64_t)j * nq) : make_float4(0.f, 0.f, 0.f, 0.f);
    // weights exp(m_q - g) l_q, lane q holding partitions q and q + 32
    const float a0 = l0 > 0.f ? m0 * kLog2e : -INFINITY, a1 = l1 > 0.f ? m1 * kLog2e : -INFINITY;
    float gm = fmaxf(a0, a1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
    const float w0 = a0 == -INFINITY ? 0.f : l0 * ex2(a0 - gm), w1 = a1 == -INFINITY ? 0.f : l1 * ex2(a1 - gm);
    float tot = w0 + w1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < P; q0 += kP2RowChunk) {
        if (q0 > 0) {
#pragma unroll
            for (int j = 0; j < kP2RowChunk; ++j)
                x[j] = (q0 + j < P && col) ? load_tmp4<BF16, TMP16>(p.tmp_out, tmp4 + (int64_t)(q0 + j) * nq)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kP2RowChunk; ++j) {
            const int q = q0 + j;  // the same on every lane
            const float w = __shfl_sync(0xffffffffu, q < 32 ? w0 : w1, q & 31);
            acc.x = fmaf(w, x[j].x, acc.x);
            acc.y = fmaf(w, x[j].y, acc.y);
            acc.z = fmaf(w, x[j].z, acc.z);
            acc.w = fmaf(w, x[j].w, acc.w);
        }
    }
    if (col) {
        const float inv = tot > 0.f ? 1.f / tot : 0.f;
        store_out4<BF16>(p.out, row * p.D + 4 * lane, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
}

// Phase 2 over merged rows: phase-1 CTA px folded partitions px, px + R, ... into fp32 row
// px, so row r's weight is the sum of its partitions' exp(m_p - g) l_p.  One CTA per
// (query head, sequence), 256 threads: the statistics of every partition load together, then
// four groups of threads each take every fourth row over all columns (float4), and the
// groups' sums add in shared memory.
constexpr int kP2mThreads = 256;

template <bool BF16>
__global__ void __launch_bounds__(kP2mThreads)
pa_v2_phase2_merged_kernel(const Phase2Params p) {
    // [Pmax] log2 max, [Pmax] exp-sum, [R] row weights, then (16-byte aligned) [4][D] sums
    extern __shared__ __align__(16) float smm[];
    __shared__ float red[kP2mThreads / 32];
    const int h = blockIdx.x, s = blockIdx.y;
    const int L = p.seq_lens[s];  // an input phase 1 only read
    griddep_wait();
    const int P = min(L > 0 ? (L + kPartition - 1) / kPartition : 0, p.Pmax);
    if (P <= 1) return;
    const int R = min(p.rstride, P);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = (int64_t)s * p.H + h;
    float* pa2 = smm;
    float* pl = pa2 + p.Pmax;
    float* wr = pl + p.Pmax;
    float* part = smm + ((2 * p.Pmax + p.rstride + 3) & ~3);  // float4 stores: 16-byte aligned
    float gm = -INFINITY;
    for (int q = tid; q < P; q += kP2mThreads) {
        const float l = p.exp_sums[row * p.Pmax + q], m = p.max_logits[row * p.Pmax + q];
        const float a = l > 0.f ? m * kLog2e : -INFINITY;
        pa2[q] = a;
        pl[q] = l;
        gm = fmaxf(gm, a);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
    if (lane == 0) red[warp] = gm;
    __syncthreads();
    gm = red[0];
#pragma unroll
    for (int w = 1; w < kP2mThreads / 32; ++w) gm = fmaxf(gm, red[w]);
    float wsum = 0.f;
    for (int r = tid; r < R; r += kP2mThreads) {
        float w = 0.f;
        for (int q = r; q < P; q += p.rstride)
            if (pa2[q] != -INFINITY) w += pl[q] * ex2(pa2[q] - gm);
        wr[r] = w;
        wsum += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    __syncthreads();  // every warp is done with red[] as the maximum
    if (lane == 0) red[warp] = wsum;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kP2mThreads / 32; ++w) tot += red[w];
    // group gq takes rows gq, gq + 4, ...; its threads cover the row's float4 columns
    const int nq = p.D / 4, per = kP2mThreads / 4, gq = tid / per, c = tid - gq * per;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nq) {
        const float4* rows = reinterpret_cast<const float4*>(p.tmp_out) + row * p.Pmax * nq + c;
#pragma unroll 4
        for (int r = gq; r < R; r += 4) {
            const float4 x = rows[(int64_t)r * nq];
            const float w = wr[r];
            acc.x = fmaf(w, x.x, acc.x);
            acc.y = fmaf(w, x.y, acc.y);
            acc.z = fmaf(w, x.z, acc.z);
            acc.w = fmaf(w, x.w, acc.w);
        }
        reinterpret_cast<float4*>(part + gq * p.D)[c] = acc;
    }
    __syncthreads();
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    for (int i4 = tid; i4 < p.D / 4; i4 += kP2mThreads) {
        float4 v = reinterpret_cast<const float4*>(part)[i4];
#pragma unroll
        for (int g2 = 1; g2 < 4; ++g2) {
            const float4 u = reinterpret_cast<const float4*>(part + g2 * p.D)[i4];
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
        }
        store_out4<BF16>(p.out, row * p.D + 4 * i4, make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv));
    }
}

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------
static cudaEvent_t g_t_begin = nullptr, g_t_end = nullptr;

static bool supported_head_size(int d) {
    switch (d) {
        case 64: case 80: case 96: case 112: case 120: case 128: case 192: case 256: return true;
        default: return false;
    }
}

template <int BS, int KVB>
static Phase1Fn phase1_form(bool bf16, int d, int form) {
    switch (form) {
        case 1: return phase1_select<BS, KVB, 1>(bf16, d);
        case 2: return phase1_select<BS, KVB, 2>(bf16, d);
        case 3: return phase1_select<BS, KVB, 3>(bf16, d);
        default: return phase1_select<BS, KVB, 0>(bf16, d);
    }
}

// form: 0 per-tensor scales, 1 per-kv-head scales, 2 per-tensor scales with an ordered grid,
// 3 per-tensor scales with the cross-warp value reduction in pairs of warps
static Phase1Fn phase1_for(bool bf16, bool fp8, int d, int bs, int form) {
    switch (bs) {
        case 8: return fp8 ? phase1_form<8, 1>(bf16, d, form) : phase1_form<8, 2>(bf16, d, form);
        case 16: return fp8 ? phase1_form<16, 1>(bf16, d, form) : phase1_form<16, 2>(bf16, d, form);
        case 32: return fp8 ? phase1_form<32, 1>(bf16, d, form) : phase1_form<32, 2>(bf16, d, form);
        default: return nullptr;
    }
}

// Opt a kernel into `bytes` of dynamic shared memory once per (kernel, device).
static std::mutex g_host_cache_mu;  // guards the two per-process caches below

static cudaError_t ensure_smem(const void* fn, size_t bytes) {
    struct Entry { const void* fn; int dev; size_t bytes; };
    static Entry cache[256];
    static int n = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_host_cache_mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].fn == fn && cache[i].dev == dev && cache[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (n < 256) cache[n++] = Entry{fn, dev, bytes};
    return cudaSuccess;
}

// SM count of the current device and resident CTAs per SM of `fn` at (threads, smem): queried
// once per (kernel, device, size) -- the occupancy query costs microseconds of host time per
// call, a visible share of a ~90 us decode step launched from an idle queue.
static cudaError_t occupancy(const void* fn, int threads, size_t smem, int* sms, int* per_sm) {
    struct Entry { const void* fn; int dev, threads; size_t smem; int sms, per_sm; };
    static Entry cache[256];
    static int n = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_host_cache_mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].fn == fn && cache[i].dev == dev && cache[i].threads == threads && cache[i].smem == smem) {
            *sms = cache[i].sms;
            *per_sm = cache[i].per_sm;
            return cudaSuccess;
        }
    if ((e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, fn, threads, smem)) != cudaSuccess) return e;
    if (n < 256) cache[n++] = Entry{fn, dev, threads, smem, *sms, *per_sm};
    return cudaSuccess;
}

static bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Optional host-side check of the table contents (PA_CHECK=1); synchronises the stream.
static pa_status host_check_tables(const int32_t* block_tables, int mbps, int num_blocks,
                                   const int32_t* seq_lens, int num_seqs, int block_size,
                                   int max_seq_len, cudaStream_t stream) {
    const char* env = getenv("PA_CHECK");
    if (env == nullptr || env[0] != '1') return PA_OK;
    if (num_seqs == 0) return PA_OK;
    int32_t* lens = (int32_t*)malloc(sizeof(int32_t) * num_seqs);
    int32_t* tab = (int32_t*)malloc(sizeof(int32_t) * (size_t)num_seqs * mbps);
    if (!lens || !tab) { free(lens); free(tab); return PA_ERR_CUDA; }
    pa_status st = PA_OK;
    if (cudaMemcpyAsync(lens, seq_lens, sizeof(int32_t) * num_seqs, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyAsync(tab, block_tables, sizeof(int32_t) * (size_t)num_seqs * mbps, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        st = PA_ERR_CUDA;
    } else {
        for (int s = 0; s < num_seqs && st == PA_OK; ++s) {
            const int L = lens[s];
            if (L < 0 || L > max_seq_len) { st = PA_ERR_INVALID_ARG; break; }
            const int nb = (L + block_size - 1) / block_size;
            if (nb > mbps) { st = PA_ERR_INVALID_ARG; break; }
            for (int b = 0; b < nb; ++b) {
                const int id = tab[(size_t)s * mbps + b];
                if (id < 0 || id >= num_blocks) { st = PA_ERR_INVALID_ARG; break; }
            }
        }
    }
    free(lens);
    free(tab);
    return st;
}

}  // namespace pa

using namespace pa;

extern "C" int pa_v2_partition_size(void) { return kPartition; }

extern "C" const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported combination";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_SCRATCH_TOO_SMALL: return "step needs more than the fixed no-allocation scratch";
    }
    return "unknown status";
}

cudaError_t pa::read_decode_errors(unsigned int* v, bool reset) {
    cudaError_t (*readers[])(unsigned int*, bool) = {
        phase1_read_errors<8, 2, 0>, phase1_read_errors<16, 2, 0>, phase1_read_errors<32, 2, 0>,
        phase1_read_errors<8, 1, 0>, phase1_read_errors<16, 1, 0>, phase1_read_errors<32, 1, 0>,
        phase1_read_errors<8, 2, 1>, phase1_read_errors<16, 2, 1>, phase1_read_errors<32, 2, 1>,
        phase1_read_errors<8, 1, 1>, phase1_read_errors<16, 1, 1>, phase1_read_errors<32, 1, 1>,
        phase1_read_errors<8, 2, 2>, phase1_read_errors<16, 2, 2>, phase1_read_errors<32, 2, 2>,
        phase1_read_errors<8, 1, 2>, phase1_read_errors<16, 1, 2>, phase1_read_errors<32, 1, 2>,
        phase1_read_errors<8, 2, 3>, phase1_read_errors<16, 2, 3>, phase1_read_errors<32, 2, 3>,
        phase1_read_errors<8, 1, 3>, phase1_read_errors<16, 1, 3>, phase1_read_errors<32, 1, 3>};
    unsigned int all = 0;
    for (auto rd : readers) {
        unsigned int w = 0;
        const cudaError_t e = rd(&w, reset);
        if (e != cudaSuccess) return e;
        all |= w;
    }
    *v = all;
    return cudaSuccess;
}

extern "C" pa_status pa_get_device_errors(uint32_t* flags, int reset) {
    if (flags == nullptr) return PA_ERR_INVALID_ARG;
    unsigned int a = 0, b = 0, c = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
    if (read_decode_errors(&a, reset != 0) != cudaSuccess) return PA_ERR_CUDA;
    if (read_cache_errors(&b, reset != 0) != cudaSuccess) return PA_ERR_CUDA;
    if (read_block_errors(&c, reset != 0) != cudaSuccess) return PA_ERR_CUDA;
    unsigned int d = 0, e = 0;
    if (prefix_read_errors<false>(&d, reset != 0) != cudaSuccess) return PA_ERR_CUDA;
    if (prefix_read_errors<true>(&e, reset != 0) != cudaSuccess) return PA_ERR_CUDA;
    *flags = a | b | c | d | e;
    return PA_OK;
}

void pa::timing_events(cudaEvent_t* begin, cudaEvent_t* end) {
    *begin = g_t_begin;
    *end = g_t_end;
}

extern "C" pa_status pa_v2_set_timing_events(cudaEvent_t begin, cudaEvent_t end) {
    if ((begin == nullptr) != (end == nullptr)) return PA_ERR_INVALID_ARG;
    g_t_begin = begin;
    g_t_end = end;
    return PA_OK;
}

pa_status pa::validate_decode(const DecodeArgs& a) {
    if (a.num_seqs < 0 || a.num_heads <= 0 || a.num_kv_heads <= 0) return PA_ERR_INVALID_ARG;
    if (a.num_heads % a.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (a.q_dtype != PA_DT_F16 && a.q_dtype != PA_DT_BF16) return PA_ERR_UNSUPPORTED;
    if (a.kv_cache_dtype != PA_KV_AUTO && a.kv_cache_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
    if (a.tmp_dtype != PA_DT_F32 && a.tmp_dtype != a.q_dtype) return PA_ERR_UNSUPPORTED;
    if (!supported_head_size(a.head_size)) return PA_ERR_UNSUPPORTED;
    const int x = a.kv_cache_dtype == PA_KV_FP8_E4M3 ? 16 : 8;
    if (a.head_size % x != 0) return PA_ERR_INVALID_ARG;
    if (a.block_size <= 0 || kPartition % a.block_size != 0) return PA_ERR_INVALID_ARG;
    if (a.block_size != 8 && a.block_size != 16 && a.block_size != 32) return PA_ERR_UNSUPPORTED;
    if (!(a.scale == a.scale) || !isfinite(a.scale)) return PA_ERR_INVALID_ARG;
    if ((a.k_scales == nullptr) != (a.v_scales == nullptr) || !aligned(a.k_scales, 4) || !aligned(a.v_scales, 4))
        return PA_ERR_INVALID_ARG;
    if (!(a.k_scale > 0.f) || !isfinite(a.k_scale) || !(a.v_scale > 0.f) || !isfinite(a.v_scale))
        return PA_ERR_INVALID_ARG;
    if (a.max_seq_len < 0 || a.max_num_partitions < 1) return PA_ERR_INVALID_ARG;
    if ((int64_t)a.max_num_partitions * kPartition < (int64_t)a.max_seq_len) return PA_ERR_INVALID_ARG;
    if (a.max_blocks_per_seq < 0 ||
        (int64_t)a.max_blocks_per_seq * a.block_size < (int64_t)a.max_seq_len)
        return PA_ERR_INVALID_ARG;
    if (a.num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (a.num_seqs > 65535) return PA_ERR_UNSUPPORTED;
    if ((int64_t)a.num_kv_heads * ((a.num_heads / a.num_kv_heads + kMaxHeadsPerCta - 1) / kMaxHeadsPerCta) > 65535)
        return PA_ERR_UNSUPPORTED;
    if (a.num_seqs == 0) return PA_OK;
    if (!a.output || !a.exp_sums || !a.max_logits || !a.tmp_output || !a.query || !a.key_cache ||
        !a.value_cache || !a.block_tables || !a.seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned(a.key_cache, 16) || !aligned(a.value_cache, 16) || !aligned(a.query, 16) ||
        !aligned(a.output, 4) || !aligned(a.tmp_output, 16) || !aligned(a.exp_sums, 4) ||
        !aligned(a.max_logits, 4) || !aligned(a.block_tables, 4) || !aligned(a.seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int64_t pa::decode_num_counters(int num_seqs, int num_heads, int num_kv_heads) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return 0;
    const int G = num_heads / num_kv_heads;
    return (int64_t)num_seqs * num_kv_heads * ((G + kMaxHeadsPerCta - 1) / kMaxHeadsPerCta);
}

// Overrides for tuning runs and tests, read once: the partition stride (PA_DECODE_PX=n), the
// page ring per CTA in KiB (PA_DECODE_RING_KIB=n) and the CTAs per partition
// (PA_DECODE_SPLIT=k); 0 or unset: the heuristics.
static int env_int(const char* name) {
    const char* e = getenv(name);
    return e ? atoi(e) : 0;
}
static int px_override() {
    static const int v = env_int("PA_DECODE_PX");
    return v;
}
static int ring_override_kib() {
    static const int v = env_int("PA_DECODE_RING_KIB");
    return v;
}
// The paired cross-warp reduction where it raises the CTAs an SM (PA_DECODE_PAIR = 0 turns it off)
static bool pair_enabled() {
    static const bool v = [] {
        const char* e = getenv("PA_DECODE_PAIR");
        return e == nullptr || atoi(e) != 0;
    }();
    return v;
}
// CTAs per partition (PA_DECODE_SPLIT = 1, 2 or 4), when the grid has one partition per CTA
static int split_override() {
    static const int v = [] {
        const int k = env_int("PA_DECODE_SPLIT");
        return (k == 1 || k == 2 || k == 4) ? k : 0;
    }();
    return v;
}

// SM count and opt-in shared memory per block of a device, queried once per device.
static cudaError_t sm_count(int dev, int* sms, int* optin) {
    constexpr int kMaxDev = 64;
    static int cache_sms[kMaxDev] = {}, cache_optin[kMaxDev] = {};
    static std::mutex mu;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache_sms[dev] == 0) {
        cudaError_t e = cudaDeviceGetAttribute(&cache_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&cache_optin[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) {
            cache_sms[dev] = 0;
            return e;
        }
    }
    *sms = cache_sms[dev];
    *optin = cache_optin[dev];
    return cudaSuccess;
}

pa_status pa::launch_decode(const DecodeArgs& a, float* exp_sums, float* max_logits, void* tmp_out,
                            uint32_t* counters) {
    const bool bf16 = a.q_dtype == PA_DT_BF16;
    const bool fp8 = a.kv_cache_dtype == PA_KV_FP8_E4M3;
    const int D = a.head_size, bs = a.block_size;
    const int G = a.num_heads / a.num_kv_heads;
    const int ngroups = (G + kMaxHeadsPerCta - 1) / kMaxHeadsPerCta;
    const int kvb = fp8 ? 1 : 2;
    const int pps = fp8 ? 32 / bs : (bs >= 16 ? 1 : 16 / bs);  // pages per ring slot, as in the kernel
    const uint32_t page_bytes = (uint32_t)D * bs * kvb;
    const uint32_t slot_bytes = 2u * pps * page_bytes;
    int dev = 0, optin = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || sm_count(dev, &nsm, &optin) != cudaSuccess) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    optin -= kPhase1StaticSmem;  // the kernel's static shared memory comes out of the same budget
    // Ring depth: about kRingTarget bytes of pages per CTA, at least one slot per warp.  (A
    // deeper ring for small grids measured slower: 96 / 128 / 192 KiB gave 22.4 / 26.9 /
    // 27.3 us against 22.0 us on a two-sequence batch, as fewer CTAs then fit an SM.)
    const uint32_t target = ring_override_kib() > 0 ? (uint32_t)ring_override_kib() * 1024u : kRingTarget;
    (void)nsm;
    int nstage = (int)(target / (kWarps * slot_bytes));
    nstage = nstage < 1 ? 1 : (nstage > 8 ? 8 : nstage);
    if (nstage < PA_MIN_STAGES && (uint32_t)PA_MIN_STAGES * kWarps * slot_bytes <= 160u * 1024u) nstage = PA_MIN_STAGES;
    const int red_heads = G < kMaxHeadsPerCta ? G : kMaxHeadsPerCta;
    // red_rows: rows of the cross-warp value reduction, one a warp (kWarps) or, in form 3, one
    // a pair of warps
    auto smem_for = [&](int ns, int red_rows) {
        return (size_t)kWarps * ns * slot_bytes + kWarps * ns * sizeof(uint64_t) +
               (2 * kWarps + 4) * kMaxHeadsPerCta * sizeof(float) +
               (size_t)red_rows * red_heads * (D + 4) * sizeof(float);
    };
    // staged rows of the fused append: 2 x D 16-bit values after the rest
    const size_t app_bytes = a.new_key != nullptr ? (size_t)4 * D : 0;
    while (nstage > 1 && smem_for(nstage, kWarps) + app_bytes > (size_t)optin) --nstage;  // a deep ring that does not fit
    const uint32_t ring = (uint32_t)kWarps * nstage * slot_bytes;
    size_t nrow_off = (smem_for(nstage, kWarps) + 15) & ~(size_t)15;
    size_t smem1 = nrow_off + app_bytes;

    Phase1Fn fn = phase1_for(bf16, fp8, D, bs, a.k_scales != nullptr ? 1 : 0);
    if (fn == nullptr) return PA_ERR_UNSUPPORTED;
    if (smem1 > (size_t)optin) return PA_ERR_UNSUPPORTED;
    if (ensure_smem((const void*)fn, smem1) != cudaSuccess) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    // Form 3 (per-tensor scales): the cross-warp value reduction in half the rows (pairs of
    // warps add into one), where the shared memory it saves lets one more CTA share an SM --
    // 8 query heads a CTA at head size 128: 81 against 73 KiB, three CTAs an SM instead of two
    // (16:1 GQA batch, phase 1 67.9 against 84.2 us).  Elsewhere the extra barrier and the
    // read-modify-write cost 0.3-2% (Llama, ragged MHA, fp8, long-context batches), so the
    // form is taken only where it raises the CTAs an SM.
    bool paired = false;
    if (a.k_scales == nullptr && pair_enabled()) {
        const size_t off2 = (smem_for(nstage, kWarps / 2) + 15) & ~(size_t)15;
        Phase1Fn f3 = phase1_for(bf16, fp8, D, bs, 3);
        int sms0 = 0, per0 = 0, sms3 = 0, per3 = 0;
        if (f3 != nullptr && occupancy((const void*)fn, kWarps * 32, smem1, &sms0, &per0) == cudaSuccess &&
            ensure_smem((const void*)f3, off2 + app_bytes) == cudaSuccess &&
            occupancy((const void*)f3, kWarps * 32, off2 + app_bytes, &sms3, &per3) == cudaSuccess && per3 > per0) {
            fn = f3;
            nrow_off = off2;
            smem1 = off2 + app_bytes;
            paired = true;
        }
        (void)cudaGetLastError();
    }

    Phase1Params p1;
    p1.out = a.output;
    p1.exp_sums = exp_sums;
    p1.max_logits = max_logits;
    p1.tmp_out = tmp_out;
    p1.query = a.query;
    p1.kcache = (const uint8_t*)a.key_cache;
    p1.vcache = (const uint8_t*)a.value_cache;
    p1.block_tables = a.block_tables;
    p1.seq_lens = a.seq_lens;
    p1.alibi = a.alibi_slopes;
    p1.H = a.num_heads;
    p1.Hk = a.num_kv_heads;
    p1.G = G;
    p1.ngroups = ngroups;
    p1.bs = bs;
    p1.mbps = a.max_blocks_per_seq;
    p1.num_blocks = a.num_blocks;
    p1.Pmax = a.max_num_partitions;
    p1.nstage = nstage;
    p1.ring_bytes = ring;
    p1.qk_scale_log2 = a.scale * a.k_scale * kLog2e;
    p1.v_scale = a.v_scale;
    p1.k_scales = a.k_scales;
    p1.v_scales = a.v_scales;
    p1.scale = a.scale;
    p1.tmp16 = a.tmp_dtype != PA_DT_F32;
    p1.counters = nullptr;
    p1.merge = 0;
    p1.csplit = 1;
    p1.mrg_off = (uint32_t)smem1;  // used only when a merge row is added below
    p1.new_k = (const uint16_t*)a.new_key;
    p1.new_v = (const uint16_t*)a.new_value;
    p1.nk_stride = a.new_key_stride;
    p1.nv_stride = a.new_value_stride;
    p1.k_enc = a.k_scale;
    p1.v_enc = a.v_scale;
    p1.order = nullptr;
    p1.nrow_off = (uint32_t)nrow_off;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    // Partition stride PX: each CTA takes partitions px, px + PX, ...  One partition per CTA
    // (PX = max_num_partitions) schedules finest, but a ragged batch whose longest sequence
    // is far above the typical one would then launch mostly empty CTAs, each holding a
    // shared-memory slot while it starts.  So PX is capped to keep the grid within about
    // PA_GRID_WAVES full waves, and each CTA takes at most 8 partitions.  A batch of few rows
    // (sequences x kv heads x head groups, fewer than the GPU has CTA slots) of long sequences
    // instead gets exactly one wave: PX = slots / rows, each CTA streaming its partitions
    // back to back (measured on 4 x 100K tokens: 251 us against 264 us for one partition per
    // CTA and 317 us for 1.3 waves).
    const int64_t Pmax = a.max_num_partitions;
    const int64_t rows = (int64_t)a.num_kv_heads * ngroups * a.num_seqs;
    int64_t slots = 0, PX = 1;
    bool few_rows = false;  // one wave of CTAs, each streaming many partitions
    // CTA slots of the GPU at this shared-memory size, and the partition stride for them
    auto plan = [&](size_t smem) -> bool {
        int sms = 0, per_sm = 0;
        if (occupancy((const void*)fn, kWarps * 32, smem, &sms, &per_sm) != cudaSuccess) return false;
        slots = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
        few_rows = rows < slots && rows * Pmax > slots;
        if (few_rows) {
            // as many partitions a CTA as the slots allow, then the fewest CTAs that still
            // need no more rounds: with every CTA busy to the end, none runs its last
            // partitions alone at a single CTA's rate (4 x 100K tokens, 2 CTAs an SM:
            // 18 CTAs a row of 11 rounds each 254.3 us, against 259.1 us for 19 CTAs of
            // which 13 finish a round early)
            PX = slots / rows;
            if (PX >= 1) PX = (Pmax + (Pmax + PX - 1) / PX - 1) / ((Pmax + PX - 1) / PX);
        } else {
            PX = (int64_t)PA_GRID_WAVES * slots / rows;
            const int64_t px_min = (Pmax + 7) / 8;
            if (PX < px_min) PX = px_min;
        }
        if (px_override() > 0) PX = px_override();
        if (PX > Pmax) PX = Pmax;
        if (PX < 1) PX = 1;
        return true;
    };
    if (!plan(smem1)) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    // An ordered grid (order scratch, per-tensor scales, a wide batch) takes fewer, longer
    // CTAs: about 8 waves of them, up to 16 partitions each, since the longest start first
    // and the tail no longer waits on them.  Measured (phase 1, ordered): fp8 batch PX 2 / 3 /
    // 4 172.4 / 172.1 / 172.6 us against 175.3 us at PX 7 (16 waves, index order); ragged MHA
    // batch PX 4 / 5 / 6 432.9 / 434.1 / 436.1 us against 438.3 us at PX 7.  Where that still
    // leaves CTAs of fewer than 4 partitions (the Llama batch: PX 7 of 8) the grid keeps its
    // index order and the 16-wave stride.
    bool ordered = false;
    if (a.order != nullptr && a.k_scales == nullptr && !paired && !few_rows && a.num_seqs >= kOrderMinSeqs &&
        px_override() <= 0) {
        int64_t px_ord = (int64_t)kOrderedWaves * slots / rows;
        const int64_t px_min = (Pmax + kOrderedMaxParts - 1) / kOrderedMaxParts;
        if (px_ord < px_min) px_ord = px_min;
        if (px_ord > Pmax) px_ord = Pmax;
        if (px_ord >= 1 && (Pmax + px_ord - 1) / px_ord >= 4) {
            PX = px_ord;
            ordered = true;
        }
    } else if (a.order != nullptr && a.k_scales == nullptr && !paired && !few_rows && a.num_seqs >= kOrderMinSeqs) {
        ordered = (Pmax + PX - 1) / PX >= 4;  // a stride set for a tuning run
    }

    // Fused combine (V1/V2 dispatch, "paged_attn.py" forward_decode, re-decided for this GPU):
    // with arrival counters the last CTA of each (sequence, head group) merges the partitions,
    // so no second kernel waits for the whole grid.  Arriving costs every CTA a fence and an
    // atomic round trip at its end (about 2 us of its slot), which a grid of many waves pays
    // many times over; a grid of at most two waves pays it once and saves the second
    // kernel's launch and wait.  So the combine is fused only there.  With an fp32 tmp_output
    // every CTA folds its own partitions into one row (the last CTA merges PX rows); a 16-bit
    // one keeps a row per partition.  Either way the rows the last CTA merges are bounded by
    // kFusedRowBytes.
    bool fused = counters != nullptr && Pmax > 1 && rows * PX <= 2 * slots;
    // A CTA folds its partitions into one row only where it streams many of them (few long
    // rows): in a wide batch striding under the wave budget the extra shared-memory row would
    // cost CTAs per SM (fp8 batch: 280.6 against 213.8 us per step).
    const bool merge = (fused || (a.tmp_scratch && few_rows)) && a.tmp_dtype == PA_DT_F32 && PX < Pmax;
    if (merge) {
        // CTAs that stream several partitions keep their running row in shared memory
        const size_t with_row = smem1 + (size_t)red_heads * D * sizeof(float);
        if (with_row > (size_t)optin || ensure_smem((const void*)fn, with_row) != cudaSuccess || !plan(with_row)) {
            (void)cudaGetLastError();
            return PA_ERR_CUDA;
        }
        smem1 = with_row;
        fused = fused && rows * PX <= 2 * slots;
    }
    p1.merge = merge ? 1 : 0;
    if (fused) {
        const int64_t R = merge ? PX : Pmax;
        const int64_t row_bytes = (int64_t)red_heads * D * (a.tmp_dtype == PA_DT_F32 ? 4 : 2);
        // the row weights and partition statistics live in the idle page ring during the combine
        if ((kMaxHeadsPerCta + (int64_t)red_heads * (R + 2 * Pmax)) * (int64_t)sizeof(float) > (int64_t)ring ||
            R * row_bytes > kFusedRowBytes)
            fused = false;
        if (fused) p1.counters = counters;
    }

    // Cluster split of one-partition CTAs: K CTAs share each partition's pages, so a small
    // grid runs more warps per SM; the partners' partials travel to the cluster's first CTA,
    // into its idle page ring.
    // Off unless asked for (PA_DECODE_SPLIT): on a two-sequence batch (16 rows x 15
    // partitions) two CTAs per partition measured 18.4 us against 16.3 us for one, the two
    // cluster barriers and the partner hand-off costing more than the finer spread of pages.
    int K = 1;
    if (PX == Pmax && !p1.merge) {
        if (split_override() > 0) K = split_override();
        while (K > 1 && (int64_t)(K - 1) * (2 * kMaxHeadsPerCta + red_heads * D) * (int64_t)sizeof(float) > (int64_t)ring)
            K /= 2;
    }
    p1.csplit = K;
    // Grid order: where CTAs stride over several partitions their work differs several-fold,
    // and a long sequence scheduled last leaves a tail; serving the sequences with the most
    // partitions first removes it (the order kernel runs first; every CTA then loads its
    // sequence from the order).  Measured at the 16-wave stride: ragged MHA step 448.8 against
    // 458.3 us; fp8 batch (CTAs of up to 3 partitions) 198.8 against 197.9 us, the order
    // kernel costing more than it saved there -- hence grids are ordered only with CTAs of 4
    // or more partitions.  (With per-kv-head scales the grid keeps its index order: the
    // ordered form exists for per-tensor scales only.)
    if (ordered && K == 1) {
        fn = phase1_for(bf16, fp8, D, bs, 2);
        if (fn == nullptr || ensure_smem((const void*)fn, smem1) != cudaSuccess) {
            (void)cudaGetLastError();
            return PA_ERR_CUDA;
        }
        const pa_status so = launch_order(a.seq_lens, a.num_seqs, a.order, a.stream);
        if (so != PA_OK) return so;
        p1.order = a.order;
    }
    cudaLaunchAttribute attrs1[2];
    attrs1[0] = attr[0];
    attrs1[1].id = cudaLaunchAttributeClusterDimension;
    attrs1[1].val.clusterDim.x = (unsigned)K;
    attrs1[1].val.clusterDim.y = 1;
    attrs1[1].val.clusterDim.z = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(PX * ngroups * K), (unsigned)a.num_kv_heads, (unsigned)a.num_seqs);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem1;
    cfg.stream = a.stream;
    cfg.attrs = attrs1;
    cfg.numAttrs = K > 1 ? 2 : 1;
    if (g_t_begin != nullptr) cudaEventRecord(g_t_begin, a.stream);
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p1);
    if (g_t_end != nullptr) cudaEventRecord(g_t_end, a.stream);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // leave no launch error behind for the caller's next call
        return PA_ERR_CUDA;
    }

    if (a.max_num_partitions > 1 && !fused) {
        Phase2Params p2;
        p2.out = a.output;
        p2.exp_sums = exp_sums;
        p2.max_logits = max_logits;
        p2.tmp_out = tmp_out;
        p2.seq_lens = a.seq_lens;
        p2.S = a.num_seqs;
        p2.H = a.num_heads;
        p2.D = D;
        p2.Pmax = a.max_num_partitions;
        p2.rstride = (int)PX;
        const bool t16 = a.tmp_dtype != PA_DT_F32;
        const size_t smem_m = (size_t)(((2 * a.max_num_partitions + PX + 3) & ~(int64_t)3) + 4 * D) * sizeof(float);
        if (p1.merge && smem_m <= 48 * 1024) {
            // rows merged by the phase-1 CTAs (PX of them per sequence and head)
            void (*fm)(const Phase2Params) = bf16 ? pa_v2_phase2_merged_kernel<true> : pa_v2_phase2_merged_kernel<false>;
            cudaLaunchConfig_t cm = {};
            cm.gridDim = dim3((unsigned)a.num_heads, (unsigned)a.num_seqs, 1);
            cm.blockDim = dim3(kP2mThreads, 1, 1);
            cm.dynamicSmemBytes = smem_m;
            cm.stream = a.stream;
            cm.attrs = attr;
            cm.numAttrs = 1;
            if (cudaLaunchKernelEx(&cm, fm, p2) != cudaSuccess) {
                (void)cudaGetLastError();
                return PA_ERR_CUDA;
            }
            return PA_OK;
        }
        if (a.max_num_partitions <= 64 && D <= 128) {
            // one warp per row (a wide batch of short and medium sequences)
            void (*fr)(const Phase2Params) =
                bf16 ? (t16 ? pa_v2_phase2_rows_kernel<true, true> : pa_v2_phase2_rows_kernel<true, false>)
                     : (t16 ? pa_v2_phase2_rows_kernel<false, true> : pa_v2_phase2_rows_kernel<false, false>);
            const int64_t nrows = (int64_t)a.num_seqs * a.num_heads;
            cudaLaunchConfig_t cr = {};
            cr.gridDim = dim3((unsigned)((nrows + kP2RowsPerCta - 1) / kP2RowsPerCta), 1, 1);
            cr.blockDim = dim3(kP2RowsPerCta * 32, 1, 1);
            cr.dynamicSmemBytes = 0;
            cr.stream = a.stream;
            cr.attrs = attr;
            cr.numAttrs = 1;
            if (cudaLaunchKernelEx(&cr, fr, p2) != cudaSuccess) {
                (void)cudaGetLastError();
                return PA_ERR_CUDA;
            }
            return PA_OK;
        }
        // Warps per combine: about 8 partitions per warp, 1 .. 16 warps.
        int w2 = (a.max_num_partitions + 7) / 8;
        w2 = w2 < 1 ? 1 : (w2 > kP2MaxWarps ? kP2MaxWarps : w2);
        const size_t smem2 = (size_t)w2 * D * sizeof(float);
        void (*fn2)(const Phase2Params) =
            bf16 ? (t16 ? pa_v2_phase2_kernel<true, true> : pa_v2_phase2_kernel<true, false>)
                 : (t16 ? pa_v2_phase2_kernel<false, true> : pa_v2_phase2_kernel<false, false>);
        if (ensure_smem((const void*)fn2, smem2) != cudaSuccess) {
            (void)cudaGetLastError();
            return PA_ERR_CUDA;
        }
        cudaLaunchConfig_t cfg2 = {};
        cfg2.gridDim = dim3((unsigned)a.num_heads, (unsigned)a.num_seqs, 1);
        cfg2.blockDim = dim3((unsigned)(32 * w2), 1, 1);
        cfg2.dynamicSmemBytes = smem2;
        cfg2.stream = a.stream;
        cfg2.attrs = attr;
        cfg2.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg2, fn2, p2);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return PA_ERR_CUDA;
        }
    }
    return PA_OK;
}

static pa_status decode_impl(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                             const void* query, const void* key_cache, const void* value_cache, int num_seqs,
                             int num_heads, int num_kv_heads, int head_size, float scale,
                             const int32_t* block_tables, int max_blocks_per_seq, int num_blocks,
                             const int32_t* seq_lens, int block_size, int max_seq_len, int max_num_partitions,
                             const float* alibi_slopes, pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype,
                             pa_dtype tmp_dtype, float k_scale, float v_scale, const float* k_scales,
                             const float* v_scales, cudaStream_t stream) {
    DecodeArgs a;
    a.output = output;
    a.exp_sums = exp_sums;
    a.max_logits = max_logits;
    a.tmp_output = tmp_output;
    a.query = query;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_size = head_size;
    a.scale = scale;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.seq_lens = seq_lens;
    a.block_size = block_size;
    a.max_seq_len = max_seq_len;
    a.max_num_partitions = max_num_partitions;
    a.alibi_slopes = alibi_slopes;
    a.q_dtype = q_dtype;
    a.kv_cache_dtype = kv_cache_dtype;
    a.tmp_dtype = tmp_dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.stream = stream;
    pa_status st = validate_decode(a);
    if (st != PA_OK || num_seqs == 0) return st;
    st = host_check_tables(block_tables, max_blocks_per_seq, num_blocks, seq_lens, num_seqs, block_size,
                           max_seq_len, stream);
    if (st != PA_OK) return st;
    return launch_decode(a, exp_sums, max_logits, tmp_output);
}

extern "C" pa_status pa_v2_decode(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                                  const void* query, const void* key_cache, const void* value_cache,
                                  int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                  float scale, const int32_t* block_tables, int max_blocks_per_seq,
                                  int num_blocks, const int32_t* seq_lens, int block_size,
                                  int max_seq_len, int max_num_partitions, const float* alibi_slopes,
                                  pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype, pa_dtype tmp_dtype,
                                  float k_scale, float v_scale, cudaStream_t stream) {
    return decode_impl(output, exp_sums, max_logits, tmp_output, query, key_cache, value_cache, num_seqs,
                       num_heads, num_kv_heads, head_size, scale, block_tables, max_blocks_per_seq, num_blocks,
                       seq_lens, block_size, max_seq_len, max_num_partitions, alibi_slopes, q_dtype,
                       kv_cache_dtype, tmp_dtype, k_scale, v_scale, nullptr, nullptr, stream);
}

extern "C" pa_status pa_v2_decode_head_scales(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                                              const void* query, const void* key_cache, const void* value_cache,
                                              int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                              float scale, const int32_t* block_tables, int max_blocks_per_seq,
                                              int num_blocks, const int32_t* seq_lens, int block_size,
                                              int max_seq_len, int max_num_partitions, const float* alibi_slopes,
                                              pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype,
                                              pa_dtype tmp_dtype, const float* k_scales, const float* v_scales,
                                              cudaStream_t stream) {
    if (k_scales == nullptr || v_scales == nullptr) return PA_ERR_INVALID_ARG;
    return decode_impl(output, exp_sums, max_logits, tmp_output, query, key_cache, value_cache, num_seqs,
                       num_heads, num_kv_heads, head_size, scale, block_tables, max_blocks_per_seq, num_blocks,
                       seq_lens, block_size, max_seq_len, max_num_partitions, alibi_slopes, q_dtype,
                       kv_cache_dtype, tmp_dtype, 1.f, 1.f, k_scales, v_scales, stream);
}

extern "C" int64_t pa_v2_decode_num_counters(int num_seqs, int num_heads, int num_kv_heads) {
    return decode_num_counters(num_seqs, num_heads, num_kv_heads);
}

extern "C" pa_status pa_v2_decode_fused(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                                        const void* query, const void* key_cache, const void* value_cache,
                                        int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                        float scale, const int32_t* block_tables, int max_blocks_per_seq,
                                        int num_blocks, const int32_t* seq_lens, int block_size,
                                        int max_seq_len, int max_num_partitions, const float* alibi_slopes,
                                        pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype, pa_dtype tmp_dtype,
                                        float k_scale, float v_scale, uint32_t* counters, int64_t num_counters,
                                        cudaStream_t stream) {
    DecodeArgs a;
    a.output = output;
    a.exp_sums = exp_sums;
    a.max_logits = max_logits;
    a.tmp_output = tmp_output;
    a.query = query;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_size = head_size;
    a.scale = scale;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.seq_lens = seq_lens;
    a.block_size = block_size;
    a.max_seq_len = max_seq_len;
    a.max_num_partitions = max_num_partitions;
    a.alibi_slopes = alibi_slopes;
    a.q_dtype = q_dtype;
    a.kv_cache_dtype = kv_cache_dtype;
    a.tmp_dtype = tmp_dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.stream = stream;
    pa_status st = validate_decode(a);
    if (st != PA_OK || num_seqs == 0) return st;
    if (counters != nullptr &&
        (!aligned(counters, 4) || num_counters < decode_num_counters(num_seqs, num_heads, num_kv_heads)))
        return PA_ERR_INVALID_ARG;
    a.tmp_scratch = counters != nullptr;
    st = host_check_tables(block_tables, max_blocks_per_seq, num_blocks, seq_lens, num_seqs, block_size,
                           max_seq_len, stream);
    if (st != PA_OK) return st;
    return launch_decode(a, exp_sums, max_logits, tmp_output, counters);
}

static pa_status append_impl(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                             const void* query, const void* key, const void* value, int64_t key_stride_s,
                             int64_t value_stride_s, void* key_cache, void* value_cache, int num_seqs,
                             int num_heads, int num_kv_heads, int head_size, float scale,
                             const int32_t* block_tables, int max_blocks_per_seq, int num_blocks,
                             const int32_t* seq_lens, int block_size, int max_seq_len, int max_num_partitions,
                             const float* alibi_slopes, pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype,
                             pa_dtype tmp_dtype, float k_scale, float v_scale, const float* k_scales,
                             const float* v_scales, int32_t* order, cudaStream_t stream) {
    DecodeArgs a;
    a.output = output;
    a.exp_sums = exp_sums;
    a.max_logits = max_logits;
    a.tmp_output = tmp_output;
    a.query = query;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_size = head_size;
    a.scale = scale;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.seq_lens = seq_lens;
    a.block_size = block_size;
    a.max_seq_len = max_seq_len;
    a.max_num_partitions = max_num_partitions;
    a.alibi_slopes = alibi_slopes;
    a.q_dtype = q_dtype;
    a.kv_cache_dtype = kv_cache_dtype;
    a.tmp_dtype = tmp_dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.stream = stream;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.order = order;
    a.new_key = key;
    a.new_value = value;
    a.new_key_stride = key_stride_s;
    a.new_value_stride = value_stride_s;
    a.tmp_scratch = true;
    pa_status st = validate_decode(a);
    if (st != PA_OK || num_seqs == 0) return st;
    const int64_t row = (int64_t)num_kv_heads * head_size;
    if (key == nullptr || value == nullptr || key_stride_s < row || value_stride_s < row || key_stride_s % 8 != 0 ||
        value_stride_s % 8 != 0 || !aligned(key, 16) || !aligned(value, 16) || !aligned(order, 4))
        return PA_ERR_INVALID_ARG;
    st = host_check_tables(block_tables, max_blocks_per_seq, num_blocks, seq_lens, num_seqs, block_size,
                           max_seq_len, stream);
    if (st != PA_OK) return st;
    return launch_decode(a, exp_sums, max_logits, tmp_output);
}

extern "C" pa_status pa_v2_decode_append(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                                         const void* query, const void* key, const void* value,
                                         int64_t key_stride_s, int64_t value_stride_s, void* key_cache,
                                         void* value_cache, int num_seqs, int num_heads, int num_kv_heads,
                                         int head_size, float scale, const int32_t* block_tables,
                                         int max_blocks_per_seq, int num_blocks, const int32_t* seq_lens,
                                         int block_size, int max_seq_len, int max_num_partitions,
                                         const float* alibi_slopes, pa_dtype q_dtype,
                                         pa_kv_cache_dtype kv_cache_dtype, pa_dtype tmp_dtype, float k_scale,
                                         float v_scale, int32_t* order, cudaStream_t stream) {
    return append_impl(output, exp_sums, max_logits, tmp_output, query, key, value, key_stride_s, value_stride_s,
                       key_cache, value_cache, num_seqs, num_heads, num_kv_heads, head_size, scale, block_tables,
                       max_blocks_per_seq, num_blocks, seq_lens, block_size, max_seq_len, max_num_partitions,
                       alibi_slopes, q_dtype, kv_cache_dtype, tmp_dtype, k_scale, v_scale, nullptr, nullptr, order,
                       stream);
}

extern "C" pa_status pa_v2_decode_append_head_scales(
    void* output, float* exp_sums, float* max_logits, void* tmp_output, const void* query, const void* key,
    const void* value, int64_t key_stride_s, int64_t value_stride_s, void* key_cache, void* value_cache,
    int num_seqs, int num_heads, int num_kv_heads, int head_size, float scale, const int32_t* block_tables,
    int max_blocks_per_seq, int num_blocks, const int32_t* seq_lens, int block_size, int max_seq_len,
    int max_num_partitions, const float* alibi_slopes, pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype,
    pa_dtype tmp_dtype, const float* k_scales, const float* v_scales, int32_t* order, cudaStream_t stream) {
    if (k_scales == nullptr || v_scales == nullptr) return PA_ERR_INVALID_ARG;
    return append_impl(output, exp_sums, max_logits, tmp_output, query, key, value, key_stride_s, value_stride_s,
                       key_cache, value_cache, num_seqs, num_heads, num_kv_heads, head_size, scale, block_tables,
                       max_blocks_per_seq, num_blocks, seq_lens, block_size, max_seq_len, max_num_partitions,
                       alibi_slopes, q_dtype, kv_cache_dtype, tmp_dtype, 1.f, 1.f, k_scales, v_scales, order, stream);
}

extern "C" pa_status pa_v2_decode_order(const int32_t* seq_lens, int num_seqs, int32_t* order, cudaStream_t stream) {
    if (num_seqs < 0 || num_seqs > 65535) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (seq_lens == nullptr || order == nullptr || !aligned(seq_lens, 4) || !aligned(order, 4))
        return PA_ERR_INVALID_ARG;
    return launch_order(seq_lens, num_seqs, order, stream);
}

// ---------------------------------------------------------------------------------------
// No-allocation entry point: the V2 workspace in a fixed file-scope device array
// ---------------------------------------------------------------------------------------
namespace pa {

// Device scratch for pa_v2_decode_noalloc: exp_sums, max_logits and tmp_output of one call.
// In host code this name is only a stand-in for the symbol; the device address comes from
// cudaGetSymbolAddress (looked up once per device, with that device current).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

static pa_status noalloc_scratch(unsigned char** out) {
    static std::mutex mu;
    static unsigned char* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            return PA_ERR_CUDA;
        }
        addr[dev] = static_cast<unsigned char*>(ptr);
    }
    *out = addr[dev];
    return PA_OK;
}

}  // namespace pa

extern "C" pa_status pa_v2_decode_noalloc(void* output, const void* query, const void* key_cache,
                                          const void* value_cache, int num_seqs, int num_heads,
                                          int num_kv_heads, int head_size, float scale,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          int num_blocks, const int32_t* seq_lens, int block_size,
                                          int max_seq_len, const float* alibi_slopes,
                                          pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype,
                                          float k_scale, float v_scale, cudaStream_t stream) {
    if (num_seqs < 0 || num_heads <= 0 || head_size <= 0 || max_seq_len < 0) return PA_ERR_INVALID_ARG;
    const int P = max_seq_len > 0 ? (max_seq_len + kPartition - 1) / kPartition : 1;
    const size_t rows = (size_t)num_seqs * (size_t)num_heads * (size_t)P;
    const size_t stat_bytes = (rows * sizeof(float) + 255u) & ~(size_t)255u;
    const size_t need = 2 * stat_bytes + rows * (size_t)head_size * sizeof(float);
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_SCRATCH_TOO_SMALL;

    DecodeArgs a;
    a.output = output;
    a.query = query;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_size = head_size;
    a.scale = scale;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.seq_lens = seq_lens;
    a.block_size = block_size;
    a.max_seq_len = max_seq_len;
    a.max_num_partitions = P;
    a.alibi_slopes = alibi_slopes;
    a.q_dtype = q_dtype;
    a.kv_cache_dtype = kv_cache_dtype;
    a.tmp_dtype = PA_DT_F32;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.stream = stream;
    // placeholders so the shared argument check sees a workspace; replaced below
    a.exp_sums = a.max_logits = reinterpret_cast<float*>(256);
    a.tmp_output = reinterpret_cast<void*>(256);
    pa_status st = validate_decode(a);
    if (st != PA_OK || num_seqs == 0) return st;

    unsigned char* base = nullptr;
    st = noalloc_scratch(&base);
    if (st != PA_OK) return st;
    float* es = reinterpret_cast<float*>(base);
    float* ml = reinterpret_cast<float*>(base + stat_bytes);
    float* tmp = reinterpret_cast<float*>(base + 2 * stat_bytes);
    a.exp_sums = es;
    a.max_logits = ml;
    a.tmp_output = tmp;
    return launch_decode(a, es, ml, tmp);
}
