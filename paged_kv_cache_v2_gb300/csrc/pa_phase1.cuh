// pa_phase1.cuh -- the phase-1 kernel of PagedAttention V2 decode (see pa_decode.cu for the
// design), templated on the block size; pa_phase1_bs{8,16,32}.cu instantiate it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_kernels.cuh"
#include "pa_ptx.cuh"

namespace pa {

// One error word per translation unit (each block size has its own).
static __device__ unsigned int g_phase1_errors = 0;

__device__ __forceinline__ void flag_error(unsigned int bit) { atomicOr(&g_phase1_errors, bit); }

// Token order of the 16 MMA rows for fp8 pages.  An fp8 V row hands each thread four
// consecutive tokens, while the P operand (via movmatrix) hands thread t logical rows
// {2t, 2t+1, 8+2t, 9+2t}; this order makes both agree (with the two halves swapped for
// t >= 2) and keeps the K-row ldmatrix free of bank conflicts.
static __device__ __constant__ int8_t c_fp8_row_token[16] = {0, 1, 4, 5, 10, 11, 14, 15,
                                                      2, 3, 6, 7, 8, 9, 12, 13};

// One step of a running log-sum-exp merge of normalised rows: the row so far has max A and
// exp-sum Lc (log2 units), the new part max a and exp-sum l.  Returns the factors that the
// merged normalised row takes from the old row (fo) and from the new part (fn), and updates
// (A, Lc).  An empty side (max -inf) gets factor 0, so its contents are never read.
__device__ __forceinline__ void merge_factors(float& A, float& Lc, float a, float l, float& fo, float& fn) {
    const float An = fmaxf(A, a);
    if (An == -INFINITY) {
        fo = fn = 0.f;
        return;
    }
    const float x = Lc * ex2(A - An), y = l * ex2(a - An);  // a side at -inf contributes 0
    const float Ln = x + y;
    fo = Ln > 0.f ? x / Ln : 0.f;
    fn = Ln > 0.f ? y / Ln : 0.f;
    A = An;
    Lc = Ln;
}

// The combine of phase 2 ("paged_attention_v2_triton.py", _paged_attn_v2_reduce_kernel), run
// by the last CTA of a (sequence, head group) to finish: g = max_p m_p and weights
// exp(m_p - g) l_p from the partition statistics, and the weighted mean of the rows.  Row r
// of tmp_output holds the normalised merge of partitions r, r + rstride, ... (one partition
// per row when rstride >= Pl), so its weight is the sum of theirs.  Reads go to L2 (ld.cg):
// the rows were written by other CTAs.  Two memory round trips: every partition's statistics
// together, then the rows (sixteen in flight per thread).  `wsm` is shared memory for
// 8 + nh * (rows + 2 * Pl) floats.
template <bool BF16, int D>
__device__ __forceinline__ void fused_combine(const Phase1Params& p, int s, int h0, int nh, int Pl, int rstride,
                                              float* wsm) {
    const int R = min(rstride, Pl);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* tot = wsm;
    float* wts = tot + kMaxHeadsPerCta;  // [nh][R] row weights
    float* pa2 = wts + nh * R;           // [nh][Pl] partition max, log2 units (-inf: empty)
    float* pl = pa2 + nh * Pl;           // [nh][Pl] partition exp-sum
    for (int hh = warp; hh < nh; hh += kWarps) {
        const int64_t srow = ((int64_t)s * p.H + h0 + hh) * p.Pmax;
        float gm = -INFINITY;
#pragma unroll 4
        for (int q = lane; q < Pl; q += 32) {
            const float l = __ldcg(p.exp_sums + srow + q), m = __ldcg(p.max_logits + srow + q);
            const float a = l > 0.f ? m * kLog2e : -INFINITY;
            pa2[hh * Pl + q] = a;
            pl[hh * Pl + q] = l;
            gm = fmaxf(gm, a);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
        __syncwarp();
        float sum = 0.f;
        for (int r = lane; r < R; r += 32) {
            float w = 0.f;
            for (int q = r; q < Pl; q += rstride) {
                const float a = pa2[hh * Pl + q];
                if (a != -INFINITY) w += pl[hh * Pl + q] * ex2(a - gm);
            }
            wts[hh * R + r] = w;
            sum += w;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) tot[hh] = sum;
    }
    __syncthreads();
    constexpr int D4 = D / 4;  // four output elements per thread and step
    for (int e = threadIdx.x; e < nh * D4; e += blockDim.x) {
        const int hh = e / D4, c = e - hh * D4;
        const int64_t row = (int64_t)s * p.H + h0 + hh;
        const float* w = wts + hh * R;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 16
        for (int r = 0; r < R; ++r) {
            const int64_t i4 = (row * p.Pmax + r) * D4 + c;
            float4 x;
            if (p.tmp16) {
                const uint2 u = __ldcg(reinterpret_cast<const uint2*>(p.tmp_out) + i4);
                if constexpr (BF16) {
                    x = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                    __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
                } else {
                    x = make_float4(f16_lo_to_f32(u.x), f16_hi_to_f32(u.x), f16_lo_to_f32(u.y), f16_hi_to_f32(u.y));
                }
            } else {
                x = __ldcg(reinterpret_cast<const float4*>(p.tmp_out) + i4);
            }
            const float wr = w[r];
            acc.x = fmaf(wr, x.x, acc.x);
            acc.y = fmaf(wr, x.y, acc.y);
            acc.z = fmaf(wr, x.z, acc.z);
            acc.w = fmaf(wr, x.w, acc.w);
        }
        const float t = tot[hh];
        const float inv = t > 0.f ? 1.f / t : 0.f;
        const int64_t o = row * D + 4 * c;
        store_out<BF16>(p.out, o, acc.x * inv);
        store_out<BF16>(p.out, o + 1, acc.y * inv);
        store_out<BF16>(p.out, o + 2, acc.z * inv);
        store_out<BF16>(p.out, o + 3, acc.w * inv);
    }
}

// Encode of the cache writer ("paged_attn.py", write_to_paged_cache): a bitwise copy for a
// 16-bit cache, e4m3fn (round to nearest even, saturating) of x / scale for an fp8 cache,
// the division in IEEE fp32.
template <bool BF16>
__device__ __forceinline__ float row_f32(uint16_t v) {
    if constexpr (BF16)
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
    else
        return __half2float(__ushort_as_half(v));
}

// Write the staged key/value rows of one token (slot o of a page) into the shared-memory copy
// of its K and V pages and, when page >= 0 (the page's (block, kv head) index), into the
// caches.  The rows are staged as the cache stores them (the bits of a 16-bit cache, the e4m3
// codes of an fp8 one): the key row (D elements), then the value row.  Lane c moves K chunk c
// (16 bytes of the x-packed page) and V elements lane, lane + 32, ...
template <int KVB, int D, int BS>
__device__ __forceinline__ void append_token(const Phase1Params& p, const uint8_t* nrow, uint8_t* kpage,
                                             uint8_t* vpage, int o, int64_t page, int lane) {
    constexpr int X = 16 / KVB;  // elements per 16-byte chunk
    constexpr uint32_t page_bytes = (uint32_t)D * BS * KVB;
    uint8_t* kc = page >= 0 ? const_cast<uint8_t*>(p.kcache) + page * page_bytes : nullptr;
    uint8_t* vc = page >= 0 ? const_cast<uint8_t*>(p.vcache) + page * page_bytes : nullptr;
    for (int c = lane; c < D / X; c += 32) {
        const uint4 chunk = reinterpret_cast<const uint4*>(nrow)[c];
        const uint32_t off = (uint32_t)(c * BS + o) * 16u;
        *reinterpret_cast<uint4*>(kpage + off) = chunk;
        if (kc) *reinterpret_cast<uint4*>(kc + off) = chunk;
    }
    for (int i = lane; i < D; i += 32) {
        const uint32_t off = (uint32_t)(i * BS + o) * KVB;
        if constexpr (KVB == 2) {
            const uint16_t v = reinterpret_cast<const uint16_t*>(nrow)[D + i];
            *reinterpret_cast<uint16_t*>(vpage + off) = v;
            if (vc) *reinterpret_cast<uint16_t*>(vc + off) = v;
        } else {
            const uint8_t v = nrow[D + i];
            vpage[off] = v;
            if (vc) vc[off] = v;
        }
    }
}

// ---------------------------------------------------------------------------------------
// Phase 1
// ---------------------------------------------------------------------------------------
// Several CTAs per SM hide each other's partition boundaries; registers are capped so that
// twelve warps (sixteen for head sizes <= 96, whose rings are smaller) fit on an SM.
#ifndef PA_FP8_MIN_CTAS
#define PA_FP8_MIN_CTAS 3
#endif
// FORM 0: per-tensor scales, sequences in grid order; 1: per-kv-head scales (p.k_scales);
// 2: per-tensor scales, sequence order[blockIdx.z] (p.order); 3: per-tensor scales, the
// cross-warp value reduction in pairs of warps (half its shared memory).  Form 0 keeps the scale
// factors in the constant bank and the sequence index as blockIdx.z, so its page loop holds
// no register for them: the kernels run at their register caps, and each of those registers
// measured 1-3% (fp8 batch, long context) when the forms were one kernel.
template <bool BF16, int KVB, int D, int BS, int FORM>
__global__ void __launch_bounds__(kWarps * 32, KVB == 2 ? (D <= 96 ? 16 : 12) / kWarps
                                                        : ((BF16 && D >= 192) ? 8 : 4 * PA_FP8_MIN_CTAS) / kWarps)
pa_v2_phase1_kernel(const Phase1Params p) {
    constexpr bool HS = FORM == 1, ORD = FORM == 2;
    // rows of the cross-warp reduction of the value accumulators: one a warp, or (form 3) one
    // a pair of warps, half the shared memory, where that lets one more CTA share an SM
    constexpr int RED = FORM == 3 ? kWarps / 2 : kWarps;
    constexpr bool FP8 = (KVB == 1);
    constexpr int NK = (D + 15) / 16;          // 16-wide steps over the head dimension
    constexpr bool HALF_STEP = (D % 16) != 0;  // head_size 120: last step has 8 elements
    static_assert(!(FP8 && HALF_STEP), "fp8 pages need head_size % 16 == 0");
    extern __shared__ __align__(128) uint8_t smem[];

    // This CTA handles partitions px, px + PX, ... of one sequence for one group of <= 8
    // query heads sharing a kv head.
    // blockIdx.x = px * ngroups + grp: the head groups of one kv head (more than 8 query
    // heads per kv head) are neighbours in the grid, so they start together and stream the
    // same pages at about the same time -- the later ones find them in L2.
    // With csplit > 1, blockIdx.x = (px * ngroups + grp) * csplit + kc and the csplit CTAs of
    // one partition form a cluster (kc = rank in it).
    const int ng = p.ngroups, K = p.csplit;
    const int kc = K == 1 ? 0 : (int)(blockIdx.x % (unsigned)K);
    const int bx = K == 1 ? (int)blockIdx.x : (int)(blockIdx.x / (unsigned)K);
    const int gx = K == 1 ? (int)gridDim.x : (int)(gridDim.x / (unsigned)K);
    const int px = ng == 1 ? bx : bx / ng;
    const int PX = ng == 1 ? gx : gx / ng;
    const int grp = bx - px * ng;
    const int kvh = blockIdx.y;
    int s = blockIdx.z;  // the sequence: blockIdx.z, or order[blockIdx.z] (read after the wait)
    // Per warp: the value scale and the two encode divisors (per-kv-head scales), in shared
    // memory so that the page loop does not hold them.
    __shared__ float wscale[kWarps][3];
    static_assert(sizeof(wscale) == kPhase1StaticSmem, "the host sizes shared memory with this");
    const int h0 = kvh * p.G + grp * kMaxHeadsPerCta;
    const int nh = min(kMaxHeadsPerCta, p.G - grp * kMaxHeadsPerCta);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the partition's slots are dealt to the cluster's K * kWarps warps: this warp is gw
    const int gw = kc * kWarps + warp, KW = K * kWarps;
    const int g = lane >> 2, t = lane & 3;
    const int H = p.H;
    constexpr int bs = BS;
    static_assert(BS == 8 || BS == 16 || BS == 32, "block size 8, 16 or 32");
    constexpr int bs_log2 = bs == 8 ? 3 : (bs == 16 ? 4 : 5);
    // A slot holds the K and V pages of 16 tokens (32 for fp8 caches: one k32 MMA step).
    constexpr int pps = FP8 ? 32 / bs : (bs >= 16 ? 1 : 16 / bs);  // pages per slot
    constexpr int pps_log2 = pps == 1 ? 0 : (pps == 2 ? 1 : 2);
    constexpr int slot_tokens = pps * bs;
    constexpr int tiles_per_slot = slot_tokens / 16;
    constexpr int ppart = kPartition / bs;  // pages in a full partition
    constexpr uint32_t page_bytes = (uint32_t)D * bs * KVB;
    constexpr uint32_t slot_bytes = 2u * pps * page_bytes;
    const int nstage = p.nstage;

    // Raw table entries of partition q: lane i holds pages i and 32 + i.
    auto load_ids = [&](int q, int& r0, int& r1) {
        const int32_t* trow = p.block_tables + (int64_t)s * p.mbps;
        r0 = r1 = -1;
        if (q < p.Pmax) {
            const int lb = q * ppart;
            if (lb + lane < p.mbps) r0 = trow[lb + lane];
            if (ppart > 32 && lb + 32 + lane < p.mbps) r1 = trow[lb + 32 + lane];
        }
    };
    // Every input is read only after the wait on the previous kernel in the stream: that
    // kernel may have written the tables, the lengths or the query (a serving loop prepares
    // them on the device each step), and only the wait makes its writes visible.  The ids of
    // the first two partitions and the length then load in parallel.
    griddep_wait();
    if (ORD && p.order != nullptr) {
        s = p.order[blockIdx.z];
        if (s < 0 || s >= (int)gridDim.z) {
            // not a permutation of the sequences: nothing to serve (flagged)
            if (threadIdx.x == 0) flag_error(512u);
            griddep_launch_dependents();
            return;
        }
    }
    int c0, c1, n0, n1;
    load_ids(px, c0, c1);
    load_ids(px + PX, n0, n1);
    const int L = p.seq_lens[s];

    const int P = L > 0 ? (L + kPartition - 1) / kPartition : 0;
    if (threadIdx.x == 0 && px == 0 && kc == 0 && (L < 0 || P > p.Pmax)) flag_error(2u);
    const int Pl = min(P, p.Pmax);  // partitions with tokens that the grid covers
    // This CTA's partitions past the end: max_logits = -inf, exp_sums = 0.
    for (int q = px; q < p.Pmax && kc == 0; q += PX) {
        if (q >= Pl && threadIdx.x < nh) {
            const int64_t sidx = ((int64_t)s * H + h0 + threadIdx.x) * p.Pmax + q;
            p.max_logits[sidx] = -INFINITY;
            p.exp_sums[sidx] = 0.f;
        }
    }
    if (px == 0 && L <= 0 && kc == 0) {
        for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
            store_out<BF16>(p.out, ((int64_t)s * H + h0) * D + i, 0.f);
    }
    if (px >= Pl) {
        griddep_launch_dependents();
        return;
    }

    auto npages_of = [&](int q) { return ((min(L, (q + 1) * kPartition) - 1) >> bs_log2) - q * ppart + 1; };
    auto my_slots_of = [&](int np) {
        const int ns = (np + pps - 1) >> pps_log2;
        return ns > gw ? (ns - gw + KW - 1) / KW : 0;
    };
    // Check the raw table entries of partition q once: entries of pages that do not exist or
    // lie outside [0, num_blocks) become -1 (the latter flagged), and bit i of the returned
    // mask says page i of the partition can be read.
    auto validate = [&](int q, int& r0, int& r1) -> uint64_t {
        const int np = npages_of(q), lb = q * ppart;
        const bool e0 = lane < np, e1 = 32 + lane < np;
        const bool ok0 = e0 && r0 >= 0 && r0 < p.num_blocks && lb + lane < p.mbps;
        const bool ok1 = e1 && r1 >= 0 && r1 < p.num_blocks && lb + 32 + lane < p.mbps;
        if ((e0 && !ok0) || (e1 && !ok1)) flag_error(1u);
        r0 = ok0 ? r0 : -1;
        r1 = ok1 ? r1 : -1;
        return (uint64_t)__ballot_sync(0xffffffffu, ok0) | ((uint64_t)__ballot_sync(0xffffffffu, ok1) << 32);
    };
    auto page_id = [&](int r0, int r1, int pg) -> int {
        return __shfl_sync(0xffffffffu, pg < 32 ? r0 : r1, pg & 31);
    };

    uint8_t* ring = smem + (size_t)warp * nstage * slot_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.ring_bytes) + warp * nstage;
    float* red_m = reinterpret_cast<float*>(smem + p.ring_bytes + kWarps * nstage * sizeof(uint64_t));
    float* red_l = red_m + kWarps * kMaxHeadsPerCta;
    float* fin_m = red_l + kWarps * kMaxHeadsPerCta;  // [8] merged max (log2 units)
    float* fin_l = fin_m + kMaxHeadsPerCta;           // [8] merged exp-sum
    float* fac_o = fin_l + kMaxHeadsPerCta;           // [8] CTA merge: factor on the row so far
    float* fac_n = fac_o + kMaxHeadsPerCta;           // [8] CTA merge: factor on this partition
    float* red_o = fac_n + kMaxHeadsPerCta;           // [RED][nh][D + 4] scaled accumulators
    constexpr int RS = D + 4;
    // CTA merge over several partitions: the running row [nh][D] (only when PX < Pmax)
    float* mrg = reinterpret_cast<float*>(smem + p.mrg_off);

    if (lane == 0) {
        for (int k = 0; k < nstage; ++k) mbar_init(&bars[k], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // Pages are read once: evict-first, except by head groups other than the last of their
    // kv head, whose pages a neighbouring CTA reads right after them.
    const uint64_t policy = grp == ng - 1 ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint8_t* kc_head = p.kcache + (size_t)kvh * page_bytes;
    const uint8_t* vc_head = p.vcache + (size_t)kvh * page_bytes;
    const size_t block_stride = (size_t)p.Hk * page_bytes;

    // The warp's pages form one stream across its partitions: the issue cursor (iq, ii)
    // runs up to nstage slots ahead of consumption and at most one partition ahead.
    int cq = px;            // partition being consumed
    int iq = px, ii = 0;    // issue cursor: partition, index among this warp's slots in it
    int i_my = my_slots_of(npages_of(iq));
    uint64_t cmask = validate(px, c0, c1);                           // readable pages of cq
    uint64_t nmask = px + PX < Pl ? validate(px + PX, n0, n1) : 0u;  // and of cq + PX
    uint32_t nis = 0, ncons = 0;  // slots issued / consumed by this warp
    // ring positions of the next slot to issue / consume, and the consumer's phase parity
    // (kept incrementally: a runtime modulo per slot costs more than the rest of the bookkeeping)
    int ipos = 0, cpos = 0;
    uint32_t cphase = 0;
    bool aborted = false;
    auto issue_more = [&]() {
        while (!aborted && (int)(nis - ncons) < nstage) {
            if (ii >= i_my) {
                // move on (also past partitions where this warp has no slots), but never
                // more than one partition ahead of the consumer
                if (iq >= cq + PX || iq + PX >= Pl) break;
                iq += PX;
                ii = 0;
                i_my = my_slots_of(npages_of(iq));
                continue;
            }
            const bool cur = iq == cq;
            const int r0 = cur ? c0 : n0, r1 = cur ? c1 : n1;
            const int j = gw + ii * KW;
            const uint32_t ok = (uint32_t)((cur ? cmask : nmask) >> (j * pps)) & ((1u << pps) - 1u);
            int b[4];
#pragma unroll
            for (int pg = 0; pg < 4; ++pg) b[pg] = pg < pps ? page_id(r0, r1, j * pps + pg) : -1;
            uint64_t* bar = &bars[ipos];
            uint8_t* kdst = ring + (size_t)ipos * slot_bytes;
            uint8_t* vdst = kdst + (size_t)pps * page_bytes;
            if constexpr (pps == 1) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar, (uint32_t)__popc(ok) * 2u * page_bytes);
                    if (ok & 1u) {
                        bulk_g2s(kdst, kc_head + (size_t)b[0] * block_stride, page_bytes, bar, policy);
                        bulk_g2s(vdst, vc_head + (size_t)b[0] * block_stride, page_bytes, bar, policy);
                    }
                }
            } else {
                // Several pages a slot: lanes 2 pg and 2 pg + 1 copy page pg's keys and values,
                // so one copy instruction serves the slot (each copy instruction holds the
                // issuing warp ~0.1 us; fp8 batch 188.3 against 190.6 us).  With one page a slot
                // lane 0 alone issues both (the extra warp barrier cost more than it saved).
                if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(ok) * 2u * page_bytes);
                __syncwarp();
                const int pg = lane >> 1;
                if (lane < 2 * pps && ((ok >> pg) & 1u)) {
                    int bsel = b[0];
#pragma unroll
                    for (int q = 1; q < 4; ++q)
                        if (q < pps && pg == q) bsel = b[q];
                    const bool isv = lane & 1;
                    bulk_g2s((isv ? vdst : kdst) + pg * page_bytes,
                             (isv ? vc_head : kc_head) + (size_t)bsel * block_stride, page_bytes, bar, policy);
                }
            }
            ++nis;
            ++ii;
            if (++ipos == nstage) ipos = 0;
        }
    };

    // ---- query fragments (MMA B operand: k = head dim, n = query head g) -------------------
    // 16-bit caches: the query row as f16/bf16 pairs.  fp8 cache with an f16 query: f16 pairs
    // in the order the widened fp8 K rows deliver the head dimension (4t..4t+3 of each 16).
    // fp8 cache with a bf16 query: the row scaled by a power of two per head, so that it is
    // exact in f16 (below); the scale is undone on the scores.
    constexpr int NS = (D + 31) / 32;  // k32 steps over the head dimension (fp8)
    uint32_t qf[NK][2];
    float qs0 = 1.f, qs1 = 1.f;  // per-column score factor undoing the query's scale (fp8, bf16 query)
    {
        const bool live = g < nh;
        const uint16_t* qrow = reinterpret_cast<const uint16_t*>(p.query) + ((int64_t)s * H + h0 + g) * D;
        if constexpr (!FP8) {
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t b0 = 0, b1 = 0;
                if (live) {
                    b0 = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * t);
                    if (!(HALF_STEP && kk == NK - 1))
                        b1 = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * t);
                }
                qf[kk][0] = b0;
                qf[kk][1] = b1;
            }
        } else if constexpr (!BF16) {
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint2 v = make_uint2(0u, 0u);
                if (live) v = *reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * t);
                qf[kk][0] = v.x;
                qf[kk][1] = v.y;
            }
        } else {
            // A bf16 query meets the widened fp8 keys in f16: each head's row is scaled by a
            // power of two so its largest element lands in [8192, 16384), which makes every
            // element exact in f16 (8 significant bits of 11, down to 2^-14 of the largest);
            // the scale is undone on the scores.  The thread holds elements 16 kk + 4t + i.
            uint2 w[NK];
            float amax = 0.f;
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                w[kk] = live ? *reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * t) : make_uint2(0u, 0u);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(__uint_as_float(w[kk].x << 16)), fabsf(__uint_as_float(w[kk].x & 0xffff0000u))),
                                         fmaxf(fabsf(__uint_as_float(w[kk].y << 16)), fabsf(__uint_as_float(w[kk].y & 0xffff0000u)))));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            int e = 0;
            if (amax > 0.f && amax < INFINITY) e = (int)floorf(__log2f(16384.f / amax));
            e = max(-120, min(120, e));
            const float alpha = exp2f((float)e);  // exact power of two
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                qf[kk][0] = pack2<false>(__uint_as_float(w[kk].x << 16) * alpha, __uint_as_float(w[kk].x & 0xffff0000u) * alpha);
                qf[kk][1] = pack2<false>(__uint_as_float(w[kk].y << 16) * alpha, __uint_as_float(w[kk].y & 0xffff0000u) * alpha);
            }
            // columns 2t, 2t+1 of the score fragment belong to heads 2t, 2t+1
            qs0 = 1.f / __shfl_sync(0xffffffffu, alpha, (2 * t) * 4);
            qs1 = 1.f / __shfl_sync(0xffffffffu, alpha, (2 * t + 1) * 4);
        }
    }
    issue_more();

    // Fused append: the warp that will consume the slot holding the sequence's newest token
    // (position L - 1) stages that token's key and value rows in shared memory now, while the
    // first pages are in flight.
    const bool app = p.new_k != nullptr && L > 0 && P <= p.Pmax && (Pl - 1 - px) % PX == 0;
    const int pg_last = app ? ((L - 1) >> bs_log2) - (Pl - 1) * ppart : 0;  // page in the last partition
    const int j_last = pg_last >> pps_log2;                                   // its slot
    const bool app_warp = app && (j_last % KW) == gw;
    uint8_t* nrow = smem + p.nrow_off;  // the key row, then the value row, as the cache stores them

    // ALiBi slopes of this thread's two head columns (2t, 2t+1), base-2 units.
    float sl0 = 0.f, sl1 = 0.f;
    if (p.alibi != nullptr) {
        if (2 * t < nh) sl0 = p.alibi[h0 + 2 * t] * kLog2e;
        if (2 * t + 1 < nh) sl1 = p.alibi[h0 + 2 * t + 1] * kLog2e;
    }
    // k_scale / v_scale: per tensor, or this kv head's (read after the dependency wait, like
    // every input); a per-head scale that is not finite and positive is flagged (bit 8) and
    // used as given.  The value-side factor and the encode divisors wait in shared memory
    // (one copy per warp) for the epilogue and the append, so the page loop holds only the
    // score multiplier in a register.
    float qk_mul = p.qk_scale_log2;
    if constexpr (HS) {
        if (p.k_scales != nullptr) {
            const float ks = p.k_scales[kvh], vs = p.v_scales[kvh];
            if (threadIdx.x == 0 && bx == 0 && s == 0 && !(ks > 0.f && ks < INFINITY && vs > 0.f && vs < INFINITY))
                flag_error(256u);
            qk_mul = __fmul_rn(__fmul_rn(p.scale, ks), kLog2e);
            if (lane == 0) {
                wscale[warp][0] = vs;
                wscale[warp][1] = ks;
                wscale[warp][2] = vs;
            }
        } else if (lane == 0) {
            wscale[warp][0] = p.v_scale;
            wscale[warp][1] = p.k_enc;
            wscale[warp][2] = p.v_enc;
        }
        __syncwarp();
    }
    // the value scale (read in the epilogue, after CTA barriers) and the encode divisors
    auto v_mul = [&]() -> float {
        if constexpr (HS) return wscale[0][0];
        else return p.v_scale;
    };
    auto enc_k = [&]() -> float {
        if constexpr (HS) return wscale[warp][1];
        else return p.k_enc;
    };
    auto enc_v = [&]() -> float {
        if constexpr (HS) return wscale[warp][2];
        else return p.v_enc;
    };
    if (app_warp) {
        const uint16_t* ks = p.new_k + (int64_t)s * p.nk_stride + (int64_t)kvh * D;
        const uint16_t* vs = p.new_v + (int64_t)s * p.nv_stride + (int64_t)kvh * D;
        if constexpr (KVB == 2) {
            for (int c = lane; c < D / 8; c += 32) {
                reinterpret_cast<uint4*>(nrow)[c] = reinterpret_cast<const uint4*>(ks)[c];
                reinterpret_cast<uint4*>(nrow + 2 * D)[c] = reinterpret_cast<const uint4*>(vs)[c];
            }
        } else {
            // encoded here, while the first pages are in flight, exactly as the cache writer
            // encodes (e4m3fn, saturating, of x / scale with an IEEE fp32 divide), so that the
            // slot holding the token only copies bytes
            const float ke = enc_k(), ve = enc_v();
            for (int c = lane; c < D / 8; c += 32) {  // 8 elements of each row a lane
                const uint4 kr = reinterpret_cast<const uint4*>(ks)[c];
                const uint4 vr = reinterpret_cast<const uint4*>(vs)[c];
                const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, vw[4] = {vr.x, vr.y, vr.z, vr.w};
                uint32_t kq[2], vq[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint16_t k01 = f32x2_to_e4m3x2(__fdiv_rn(row_f32<BF16>(lo16(kw[2 * h])), ke),
                                                         __fdiv_rn(row_f32<BF16>(hi16(kw[2 * h])), ke));
                    const uint16_t k23 = f32x2_to_e4m3x2(__fdiv_rn(row_f32<BF16>(lo16(kw[2 * h + 1])), ke),
                                                         __fdiv_rn(row_f32<BF16>(hi16(kw[2 * h + 1])), ke));
                    const uint16_t v01 = f32x2_to_e4m3x2(__fdiv_rn(row_f32<BF16>(lo16(vw[2 * h])), ve),
                                                         __fdiv_rn(row_f32<BF16>(hi16(vw[2 * h])), ve));
                    const uint16_t v23 = f32x2_to_e4m3x2(__fdiv_rn(row_f32<BF16>(lo16(vw[2 * h + 1])), ve),
                                                         __fdiv_rn(row_f32<BF16>(hi16(vw[2 * h + 1])), ve));
                    kq[h] = (uint32_t)k01 | ((uint32_t)k23 << 16);
                    vq[h] = (uint32_t)v01 | ((uint32_t)v23 << 16);
                }
                reinterpret_cast<uint2*>(nrow)[c] = make_uint2(kq[0], kq[1]);
                reinterpret_cast<uint2*>(nrow + D)[c] = make_uint2(vq[0], vq[1]);
            }
        }
        __syncwarp();
    }
    const float qk_mul0 = qk_mul * qs0, qk_mul1 = qk_mul * qs1;  // fp8 with a bf16 query: per-column scale

    // Per-lane ldmatrix row of the K page: token within the 16-token tile, chunk offset.
    const int k_tok = FP8 ? c_fp8_row_token[(lane & 7) + 8 * ((lane >> 3) & 1)] : (lane & 7) + 8 * ((lane >> 3) & 1);
    const int k_chunk = lane >> 4;
    // Physical tokens of this thread's two MMA rows (g, g + 8).
    const int tokA = FP8 ? c_fp8_row_token[g] : g;
    const int tokB = FP8 ? c_fp8_row_token[g + 8] : g + 8;
    // Where a partition's result goes.  A one-partition sequence writes the output directly
    // (single pass).  Otherwise each partition writes its own tmp_output row -- or, when the
    // CTA merges its partitions (p.merge: tmp_output is the caller's scratch), the CTA folds
    // them into fp32 row px, and a CTA that covers every partition of the sequence (PX == 1)
    // writes the output directly.
    const int nwork = min(PX, Pl);  // CTAs of this (sequence, head group) that have partitions
    const bool fused = p.counters != nullptr;
    const bool merge = p.merge != 0;
    const bool direct = (Pl == 1) || (merge && nwork == 1);
    // The CTA's running merge (lane t < 4 of warp 0 holds heads 2t and 2t + 1): max in log2
    // units relative to the sequence's last token, and the exp-sum at that max.
    float cA0 = -INFINITY, cA1 = -INFINITY, cL0 = 0.f, cL1 = 0.f;
    uint32_t drain_from = 0;

    for (; cq < Pl; cq += PX) {
        // ids of the partition after the next one (the issue cursor may need them soon)
        int nn0 = -1, nn1 = -1;
        if (cq + 2 * PX < Pl) load_ids(cq + 2 * PX, nn0, nn1);
        const int t0 = cq * kPartition;
        const int t1 = min(L, t0 + kPartition);
        const int tref = t1 - 1;  // ALiBi positions relative to the partition's last token
        const int c_np = npages_of(cq);
        const int my = my_slots_of(c_np);
        issue_more();  // in case the cursor is still behind this partition

        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        float acc[NK][4];
#pragma unroll
        for (int i = 0; i < NK; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

        for (int k = 0; k < my && !aborted; ++k) {
            const int pos = cpos;
            if (!mbar_wait_bounded(&bars[pos], cphase, kWaitLimitNs)) {
                if (lane == 0) flag_error(4u);
                aborted = true;
                drain_from = ncons;
                break;
            }
            const int j = gw + k * KW;
            const uint8_t* kslot = ring + (size_t)pos * slot_bytes;
            const uint8_t* vslot = kslot + (size_t)pps * page_bytes;
            const uint32_t kbase = smem_addr(kslot), vbase = smem_addr(vslot);
            const uint32_t okmask = (uint32_t)(cmask >> (j * pps)) & ((1u << pps) - 1u);
            const int stok0 = t0 + j * slot_tokens;
            if (app_warp && cq == Pl - 1 && j == j_last) {
                // the newest token: encode its staged rows into this page's copy in shared
                // memory and (one CTA per kv head) into the caches
                const int pg = pg_last & (pps - 1);
                if ((okmask >> pg) & 1u) {
                    const int b = page_id(c0, c1, pg_last);
                    const bool to_cache = grp == 0;
                    append_token<KVB, D, BS>(p, nrow, const_cast<uint8_t*>(kslot) + (size_t)pg * page_bytes,
                                             const_cast<uint8_t*>(vslot) + (size_t)pg * page_bytes, (L - 1) & (bs - 1),
                                             to_cache ? (int64_t)b * p.Hk + kvh : -1, lane);
                }
                __syncwarp();
            }

            if constexpr (FP8) {
                // ---- one 32-token slot: two 16-token score tiles, one k32 P.V step ----------
                const int lim = t1 - stok0;  // tokens [0, lim) of the slot are in range
                const bool full = lim >= 32 && okmask == (1u << pps) - 1u;
                auto tok_ok = [&](int tok) -> bool {
                    return tok < lim && ((okmask >> (tok >> bs_log2)) & 1u);
                };
                float sv[2][4];
                {
                    // S^T = K . Q^T with K widened to f16, both 16-token tiles at once (rows are
                    // tokens in c_fp8_row_token order): four independent MMA chains, two per
                    // tile, whose latencies overlap (fp8 batch 185.0 against 187.6 us with the
                    // tiles one after the other, and no register spills at head size 128)
                    uint32_t krow[2];
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        const int tt = tile * 16 + k_tok;
                        krow[tile] = kbase + (uint32_t)(tt >> bs_log2) * page_bytes +
                                     (uint32_t)(k_chunk * bs + (tt & (bs - 1))) * 16u;
                    }
                    float sc[2][4] = {}, sd[2][4] = {};
#pragma unroll
                    for (int st = 0; st < NS; ++st) {
                        uint32_t a[2][4];
#pragma unroll
                        for (int tile = 0; tile < 2; ++tile) {
                            if (2 * st + 1 < NK) {
                                ldsm_x4(krow[tile] + (uint32_t)st * 32u * bs, a[tile][0], a[tile][1], a[tile][2], a[tile][3]);
                            } else {
                                ldsm_x2(krow[tile] + (uint32_t)st * 32u * bs, a[tile][0], a[tile][1]);
                                a[tile][2] = a[tile][3] = 0u;
                            }
                        }
#pragma unroll
                        for (int tile = 0; tile < 2; ++tile) {
                            uint32_t w0l, w0h, w1l, w1h;
                            e4m3x4_to_f16x2x2(a[tile][0], w0l, w0h);
                            e4m3x4_to_f16x2x2(a[tile][1], w1l, w1h);
                            mma16816<false>(sc[tile], w0l, w1l, w0h, w1h, qf[2 * st][0], qf[2 * st][1]);
                        }
                        if (2 * st + 1 < NK) {
#pragma unroll
                            for (int tile = 0; tile < 2; ++tile) {
                                uint32_t w2l, w2h, w3l, w3h;
                                e4m3x4_to_f16x2x2(a[tile][2], w2l, w2h);
                                e4m3x4_to_f16x2x2(a[tile][3], w3l, w3h);
                                mma16816<false>(sd[tile], w2l, w3l, w2h, w3h, qf[2 * st + 1][0], qf[2 * st + 1][1]);
                            }
                        }
                    }
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        const int ttok0 = stok0 + tile * 16;
                        float s0 = (sc[tile][0] + sd[tile][0]) * qk_mul0, s1 = (sc[tile][1] + sd[tile][1]) * qk_mul1;
                        float s2 = (sc[tile][2] + sd[tile][2]) * qk_mul0, s3 = (sc[tile][3] + sd[tile][3]) * qk_mul1;
                        if (p.alibi != nullptr) {
                            const float ra = (float)(ttok0 + tokA - tref), rb = (float)(ttok0 + tokB - tref);
                            s0 = fmaf(sl0, ra, s0);
                            s1 = fmaf(sl1, ra, s1);
                            s2 = fmaf(sl0, rb, s2);
                            s3 = fmaf(sl1, rb, s3);
                        }
                        if (!full) {
                            if (!tok_ok(tile * 16 + tokA)) s0 = s1 = -INFINITY;
                            if (!tok_ok(tile * 16 + tokB)) s2 = s3 = -INFINITY;
                        }
                        sv[tile][0] = s0;
                        sv[tile][1] = s1;
                        sv[tile][2] = s2;
                        sv[tile][3] = s3;
                    }
                }
                // online softmax over the slot's 32 tokens
                float mx0 = fmaxf(fmaxf(sv[0][0], sv[0][2]), fmaxf(sv[1][0], sv[1][2]));
                float mx1 = fmaxf(fmaxf(sv[0][1], sv[0][3]), fmaxf(sv[1][1], sv[1][3]));
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float base0 = mn0 == -INFINITY ? 0.f : mn0;
                const float base1 = mn1 == -INFINITY ? 0.f : mn1;
                const float al0 = ex2(m0 - base0), al1 = ex2(m1 - base1);
                float pv[2][4];
#pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
                    pv[tile][0] = ex2(sv[tile][0] - base0);
                    pv[tile][1] = ex2(sv[tile][1] - base1);
                    pv[tile][2] = ex2(sv[tile][2] - base0);
                    pv[tile][3] = ex2(sv[tile][3] - base1);
                }
                l0 = fmaf(l0, al0, (pv[0][0] + pv[0][2]) + (pv[1][0] + pv[1][2]));
                l1 = fmaf(l1, al1, (pv[0][1] + pv[0][3]) + (pv[1][1] + pv[1][3]));
                if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
#pragma unroll
                    for (int i = 0; i < NK; ++i) {
                        acc[i][0] *= al0;
                        acc[i][1] *= al1;
                        acc[i][2] *= al0;
                        acc[i][3] *= al1;
                    }
                }
                m0 = mn0;
                m1 = mn1;
                // P^T operand in f16, transposed with movmatrix.  After the transpose thread t
                // holds P of tokens {4t..4t+3} of head g (rows 2t, 2t+1 and 8+2t, 9+2t in the
                // token order above; the two halves swap for t >= 2).
                uint32_t pb[2][2];
#pragma unroll
                for (int tile = 0; tile < 2; ++tile) {
                    const uint32_t x0 = movm_trans(pack2<false>(pv[tile][0], pv[tile][1]));
                    const uint32_t x1 = movm_trans(pack2<false>(pv[tile][2], pv[tile][3]));
                    pb[tile][0] = t < 2 ? x0 : x1;  // tokens 4t, 4t + 1
                    pb[tile][1] = t < 2 ? x1 : x0;  // tokens 4t + 2, 4t + 3
                }
                // O^T += V^T . P^T in f16: the V codes of a row (four consecutive tokens per
                // register, straight from the page) widened to f16 in registers (exact); for
                // the m16n8k16 step of tile u, k = 2t, 2t + 1, 2t + 8, 2t + 9 stand for tokens
                // 4t .. 4t + 3 of the tile, on both operands.  (The e4m3 tensor path, with P
                // split into two e4m3 terms, measured slower on this GPU.)
                uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;  // bytes of masked tokens -> 0
                if (!full) {
                    mlo = 0u;
                    mhi = 0u;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (tok_ok(4 * t + i)) mlo |= 0xffu << (8 * i);
                        if (tok_ok(16 + 4 * t + i)) mhi |= 0xffu << (8 * i);
                    }
                }
                auto pv_step = [&](float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
                    uint32_t x0l, x0h, x1l, x1h, x2l, x2h, x3l, x3h;
                    e4m3x4_to_f16x2x2(a0, x0l, x0h);
                    e4m3x4_to_f16x2x2(a1, x1l, x1h);
                    e4m3x4_to_f16x2x2(a2, x2l, x2h);
                    e4m3x4_to_f16x2x2(a3, x3l, x3h);
                    mma16816<false>(c, x0l, x1l, x0h, x1h, pb[0][0], pb[0][1]);
                    mma16816<false>(c, x2l, x3l, x2h, x3h, pb[1][0], pb[1][1]);
                };
                if (bs >= 16) {
                    const int vr = (lane & 7) + 8 * ((lane >> 3) & 1);
                    const int tk = 16 * (lane >> 4);  // token half of this lane's matrix row
                    const uint32_t vrow = vbase + (uint32_t)(tk >> bs_log2) * page_bytes + (uint32_t)(vr * bs + (tk & (bs - 1)));
#pragma unroll
                    for (int mt = 0; mt < NK; ++mt) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(vrow + (uint32_t)mt * 16u * bs, a0, a1, a2, a3);
                        if (!full) {
                            a0 &= mlo;
                            a1 &= mlo;
                            a2 &= mhi;
                            a3 &= mhi;
                        }
                        pv_step(acc[mt], a0, a1, a2, a3);
                    }
                } else {
                    // block size 8: a V row holds 8 tokens, so read each thread's 4 tokens
                    const uint32_t va = vbase + (uint32_t)(t >> 1) * page_bytes + (uint32_t)((4 * t) & 7);
                    const uint32_t vb = va + 2u * page_bytes;
#pragma unroll
                    for (int mt = 0; mt < NK; ++mt) {
                        const uint32_t r0 = (uint32_t)(mt * 16 + g) * bs, r1 = r0 + 8u * bs;
                        pv_step(acc[mt], lds_u32(va + r0) & mlo, lds_u32(va + r1) & mlo, lds_u32(vb + r0) & mhi,
                                lds_u32(vb + r1) & mhi);
                    }
                }
            } else {
                for (int tile = 0; tile < tiles_per_slot; ++tile) {
                    const int ttok0 = stok0 + tile * 16;
                    const int lim = t1 - ttok0;  // tokens [0, lim) of the tile are in range
                    if (lim <= 0) break;
                    const bool full = lim >= 16 && okmask == (pps == 1 ? 1u : 3u);
                    auto tok_ok = [&](int tok) -> bool {
                        const int pg = pps == 1 ? 0 : (tok >> 3);
                        return tok < lim && ((okmask >> pg) & 1u);
                    };

                    // ---- S^T = K . Q^T for 16 tokens x 8 heads ------------------------------------
                    uint32_t krow;
                    if (pps == 1)
                        krow = kbase + (uint32_t)(k_chunk * bs + tile * 16 + k_tok) * 16u;
                    else
                        krow = kbase + (uint32_t)(k_tok >> 3) * page_bytes + (uint32_t)(k_chunk * bs + (k_tok & 7)) * 16u;
                    // two accumulators (even and odd steps): two MMA dependency chains of half
                    // the length, which matters when few warps share a scheduler (small batches)
                    float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < NK; ++kk) {
                        uint32_t a0, a1, a2, a3;
                        if (HALF_STEP && kk == NK - 1) {
                            ldsm_x2(krow + (uint32_t)kk * 32u * bs, a0, a1);
                            a2 = a3 = 0u;
                        } else {
                            ldsm_x4(krow + (uint32_t)kk * 32u * bs, a0, a1, a2, a3);
                        }
                        mma16816<BF16>(kk & 1 ? sd : sc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) sc[i] += sd[i];

                    // ---- scores in base-2 units, masking, online softmax ---------------------------
                    float s0 = sc[0] * qk_mul, s1 = sc[1] * qk_mul;
                    float s2 = sc[2] * qk_mul, s3 = sc[3] * qk_mul;
                    if (p.alibi != nullptr) {
                        const float ra = (float)(ttok0 + tokA - tref), rb = (float)(ttok0 + tokB - tref);
                        s0 = fmaf(sl0, ra, s0);
                        s1 = fmaf(sl1, ra, s1);
                        s2 = fmaf(sl0, rb, s2);
                        s3 = fmaf(sl1, rb, s3);
                    }
                    if (!full) {
                        if (!tok_ok(tokA)) s0 = s1 = -INFINITY;
                        if (!tok_ok(tokB)) s2 = s3 = -INFINITY;
                    }
                    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
    #pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                    }
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
                    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
                    const float al0 = ex2(m0 - base0), al1 = ex2(m1 - base1);  // m = -inf -> 0
                    const float p0 = ex2(s0 - base0), p1 = ex2(s1 - base1);
                    const float p2 = ex2(s2 - base0), p3 = ex2(s3 - base1);
                    l0 = fmaf(l0, al0, p0 + p2);
                    l1 = fmaf(l1, al1, p1 + p3);
                    // Rescale the accumulators only when some head's running max moved (after the
                    // first tiles of a partition it rarely does); otherwise the factors are 1.
                    if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
    #pragma unroll
                        for (int i = 0; i < NK; ++i) {
                            acc[i][0] *= al0;
                            acc[i][1] *= al1;
                            acc[i][2] *= al0;
                            acc[i][3] *= al1;
                        }
                    }
                    m0 = mn0;
                    m1 = mn1;

                    // ---- P into the B operand of O^T += V^T . P^T ----------------------------------
                    const uint32_t pb0 = movm_trans(pack2<BF16>(p0, p1));
                    const uint32_t pb1 = movm_trans(pack2<BF16>(p2, p3));
                    uint32_t pl0 = 0, pl1 = 0;
                    if constexpr (BF16) {
                        // bf16 keeps 8 significant bits; add the rounding residual as a second term
                        // so P enters the product with ~16 bits, as with fp16.
                        const float q0 = p0 - __bfloat162float(__float2bfloat16_rn(p0));
                        const float q1 = p1 - __bfloat162float(__float2bfloat16_rn(p1));
                        const float q2 = p2 - __bfloat162float(__float2bfloat16_rn(p2));
                        const float q3 = p3 - __bfloat162float(__float2bfloat16_rn(p3));
                        pl0 = movm_trans(pack2<true>(q0, q1));
                        pl1 = movm_trans(pack2<true>(q2, q3));
                    }

                    // ---- O^T += V^T . P^T over the head dimension ---------------------------------
                        // lane -> (V row within the 16-row tile, token half)
                        const int vr = (lane & 7) + 8 * ((lane >> 3) & 1);
                        const int half = lane >> 4;
                        uint32_t vpage, vtok;
                        if (pps == 1) {
                            vpage = vbase;
                            vtok = (uint32_t)(tile * 16 + 8 * half);
                        } else {
                            vpage = vbase + (uint32_t)half * page_bytes;
                            vtok = 0;
                        }
                        if (full) {
    #pragma unroll
                            for (int mt = 0; mt < NK; ++mt) {
                                int row = mt * 16 + vr;
                                if (HALF_STEP && mt == NK - 1) row = min(row, D - 1);
                                uint32_t a0, a1, a2, a3;
                                ldsm_x4(vpage + ((uint32_t)row * bs + vtok) * 2u, a0, a1, a2, a3);
                                mma16816<BF16>(acc[mt], a0, a1, a2, a3, pb0, pb1);
                                if constexpr (BF16) mma16816<BF16>(acc[mt], a0, a1, a2, a3, pl0, pl1);
                            }
                        } else {
                            // zero the V columns of masked tokens (0 * NaN would poison every head):
                            // a0/a1 hold tokens (2t, 2t+1), a2/a3 tokens (8+2t, 9+2t)
                            const uint32_t mlo = (tok_ok(2 * t) ? 0x0000ffffu : 0u) | (tok_ok(2 * t + 1) ? 0xffff0000u : 0u);
                            const uint32_t mhi = (tok_ok(8 + 2 * t) ? 0x0000ffffu : 0u) | (tok_ok(9 + 2 * t) ? 0xffff0000u : 0u);
    #pragma unroll
                            for (int mt = 0; mt < NK; ++mt) {
                                int row = mt * 16 + vr;
                                if (HALF_STEP && mt == NK - 1) row = min(row, D - 1);
                                uint32_t a0, a1, a2, a3;
                                ldsm_x4(vpage + ((uint32_t)row * bs + vtok) * 2u, a0, a1, a2, a3);
                                a0 &= mlo;
                                a1 &= mlo;
                                a2 &= mhi;
                                a3 &= mhi;
                                mma16816<BF16>(acc[mt], a0, a1, a2, a3, pb0, pb1);
                                if constexpr (BF16) mma16816<BF16>(acc[mt], a0, a1, a2, a3, pl0, pl1);
                            }
                        }
                }
            }

            // Order this slot's generic-proxy reads before the async copy that refills it.
            ++ncons;
            if (++cpos == nstage) {
                cpos = 0;
                cphase ^= 1u;
            }
            fence_proxy_async_smem();
            __syncwarp();
            issue_more();
        }

        // ---- merge the warps' (m, l, acc) of this partition --------------------------------
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        }
        if (g == 0) {
            red_m[warp * kMaxHeadsPerCta + 2 * t] = m0;
            red_m[warp * kMaxHeadsPerCta + 2 * t + 1] = m1;
            red_l[warp * kMaxHeadsPerCta + 2 * t] = l0;
            red_l[warp * kMaxHeadsPerCta + 2 * t + 1] = l1;
        }
        __syncthreads();
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            M0 = fmaxf(M0, red_m[w * kMaxHeadsPerCta + 2 * t]);
            M1 = fmaxf(M1, red_m[w * kMaxHeadsPerCta + 2 * t + 1]);
        }
        const float f0 = m0 == -INFINITY ? 0.f : ex2(m0 - M0);
        const float f1 = m1 == -INFINITY ? 0.f : ex2(m1 - M1);
        if (warp == 0 && g == 0) {
            float L0 = 0.f, L1 = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float ma = red_m[w * kMaxHeadsPerCta + 2 * t], mb = red_m[w * kMaxHeadsPerCta + 2 * t + 1];
                if (ma != -INFINITY) L0 += red_l[w * kMaxHeadsPerCta + 2 * t] * ex2(ma - M0);
                if (mb != -INFINITY) L1 += red_l[w * kMaxHeadsPerCta + 2 * t + 1] * ex2(mb - M1);
            }
            fin_m[2 * t] = M0;
            fin_m[2 * t + 1] = M1;
            fin_l[2 * t] = L0;
            fin_l[2 * t + 1] = L1;
            if (merge) {
                // fold this partition into the CTA's row, in log2 units relative to the last
                // token (the ALiBi bias of the scores is relative to this partition's last)
                const float rel = (float)(tref - (L - 1));
                merge_factors(cA0, cL0, L0 > 0.f ? fmaf(sl0, rel, M0) : -INFINITY, L0, fac_o[2 * t], fac_n[2 * t]);
                merge_factors(cA1, cL1, L1 > 0.f ? fmaf(sl1, rel, M1) : -INFINITY, L1, fac_o[2 * t + 1],
                              fac_n[2 * t + 1]);
            }
        }
        // Each warp's scaled accumulators go to row `warp` of red_o.  Form 3: warps RED ..
        // kWarps - 1 write theirs to rows 0 .. RED - 1, then warps 0 .. RED - 1 add theirs.
        if constexpr (RED == kWarps) {
#pragma unroll
            for (int mt = 0; mt < NK; ++mt) {
                const int r0 = mt * 16 + g, r1 = r0 + 8;
                if (2 * t < nh) {
                    float* base = red_o + (warp * nh + 2 * t) * RS;
                    if (r0 < D) base[r0] = acc[mt][0] * f0;
                    if (r1 < D) base[r1] = acc[mt][2] * f0;
                }
                if (2 * t + 1 < nh) {
                    float* base = red_o + (warp * nh + 2 * t + 1) * RS;
                    if (r0 < D) base[r0] = acc[mt][1] * f1;
                    if (r1 < D) base[r1] = acc[mt][3] * f1;
                }
            }
        } else {
            auto put_rows = [&](int row, bool add) {
#pragma unroll
                for (int mt = 0; mt < NK; ++mt) {
                    const int r0 = mt * 16 + g, r1 = r0 + 8;
                    if (2 * t < nh) {
                        float* base = red_o + (row * nh + 2 * t) * RS;
                        if (r0 < D) base[r0] = add ? fmaf(acc[mt][0], f0, base[r0]) : acc[mt][0] * f0;
                        if (r1 < D) base[r1] = add ? fmaf(acc[mt][2], f0, base[r1]) : acc[mt][2] * f0;
                    }
                    if (2 * t + 1 < nh) {
                        float* base = red_o + (row * nh + 2 * t + 1) * RS;
                        if (r0 < D) base[r0] = add ? fmaf(acc[mt][1], f1, base[r0]) : acc[mt][1] * f1;
                        if (r1 < D) base[r1] = add ? fmaf(acc[mt][3], f1, base[r1]) : acc[mt][3] * f1;
                    }
                }
            };
            if (warp >= RED) put_rows(warp - RED, false);
            __syncthreads();
            if (warp < RED) put_rows(warp, true);
        }
        __syncthreads();

        // Cluster split: each CTA but the first hands its partial (max, exp-sum and normalised
        // rows) to the first one, whose page ring is idle now (one partition per CTA); the
        // first CTA merges them into the partition's result and alone writes it.
        bool skip_out = false;
        const float vmul = v_mul();  // read once: the loops below also write shared memory
        float* pbuf = reinterpret_cast<float*>(smem);
        const int pstride = 2 * kMaxHeadsPerCta + nh * D;
        if (K > 1) {
            // every CTA of the cluster is past its page loop: the first CTA's ring is idle
            // (all its copies have landed and been read) before any partner writes into it
            cluster_sync_all();
            if (kc != 0) {
                const uint32_t dst = mapa_cluster(smem_addr(pbuf + (kc - 1) * pstride), 0);
                if (threadIdx.x < nh) {
                    st_cluster_f32(dst + 4u * threadIdx.x, fin_m[threadIdx.x]);
                    st_cluster_f32(dst + 4u * (kMaxHeadsPerCta + threadIdx.x), fin_l[threadIdx.x]);
                }
                for (int e = threadIdx.x; e < nh * D; e += blockDim.x) {
                    const int hh = e / D, i = e - hh * D;
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < RED; ++w) v += red_o[(w * nh + hh) * RS + i];
                    const float lt = fin_l[hh];
                    st_cluster_f32(dst + 4u * (2 * kMaxHeadsPerCta + e), lt > 0.f ? v * (vmul / lt) : 0.f);
                }
            }
            cluster_sync_all();
            skip_out = kc != 0;
            if (!skip_out) {
                if (threadIdx.x < nh) {
                    // merged max and exp-sum; factor on this CTA's unnormalised sums (fac_o)
                    // and on each partner's normalised rows (over the partner's max slot)
                    const int hh = threadIdx.x;
                    const float ml = fin_m[hh], ll = fin_l[hh];
                    float M = ll > 0.f ? ml : -INFINITY;
                    for (int k = 0; k < K - 1; ++k)
                        if (pbuf[k * pstride + kMaxHeadsPerCta + hh] > 0.f) M = fmaxf(M, pbuf[k * pstride + hh]);
                    float Ls = ll > 0.f ? ll * ex2(ml - M) : 0.f;
                    for (int k = 0; k < K - 1; ++k) {
                        const float lk = pbuf[k * pstride + kMaxHeadsPerCta + hh];
                        if (lk > 0.f) Ls += lk * ex2(pbuf[k * pstride + hh] - M);
                    }
                    fac_o[hh] = (ll > 0.f && Ls > 0.f) ? ex2(ml - M) / Ls : 0.f;
                    for (int k = 0; k < K - 1; ++k) {
                        const float lk = pbuf[k * pstride + kMaxHeadsPerCta + hh];
                        pbuf[k * pstride + hh] = (lk > 0.f && Ls > 0.f) ? lk * ex2(pbuf[k * pstride + hh] - M) / Ls : 0.f;
                    }
                    fin_m[hh] = M;
                    fin_l[hh] = Ls;
                }
                __syncthreads();
            }
        }

        if (merge) {
            // the CTA's row so far (in shared memory) and this partition, each with its share
            // of the merged exp-sum; the last partition writes the row out (or the output)
            const bool first = cq == px, last_part = cq + PX >= Pl;
            for (int e = threadIdx.x; e < nh * D; e += blockDim.x) {
                const int hh = e / D, i = e - hh * D;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < RED; ++w) v += red_o[(w * nh + hh) * RS + i];
                const float lt = fin_l[hh];
                v = lt > 0.f ? v * (vmul / lt) : 0.f;
                const float fo = fac_o[hh];
                float r = v * fac_n[hh];
                if (fo != 0.f && !first) r = fmaf(mrg[e], fo, r);
                const int64_t row = (int64_t)s * H + h0 + hh;
                if (!last_part)
                    mrg[e] = r;
                else if (direct)
                    store_out<BF16>(p.out, row * D + i, r);
                else
                    static_cast<float*>(p.tmp_out)[(row * p.Pmax + px) * D + i] = r;
            }
        }
        if (K == 1) {
            // four consecutive elements a thread: float4 rows in shared memory (D and the row
            // stride D + 4 are multiples of 4), one 8- or 16-byte store
            for (int e4 = threadIdx.x; e4 < nh * D / 4 && !merge && !skip_out; e4 += blockDim.x) {
                const int e = 4 * e4, hh = e / D, i = e - hh * D;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int w = 0; w < RED; ++w) {
                    const float4 r = *reinterpret_cast<const float4*>(red_o + (w * nh + hh) * RS + i);
                    v.x += r.x;
                    v.y += r.y;
                    v.z += r.z;
                    v.w += r.w;
                }
                const float lt = fin_l[hh];
                const float f = lt > 0.f ? vmul / lt : 0.f;
                v.x *= f;
                v.y *= f;
                v.z *= f;
                v.w *= f;
                const int64_t row = (int64_t)s * H + h0 + hh;
                if (direct)
                    store_out4<BF16>(p.out, row * D + i, v);
                else if (p.tmp16)
                    store_out4<BF16>(p.tmp_out, (row * p.Pmax + cq) * D + i, v);
                else
                    reinterpret_cast<float4*>(p.tmp_out)[((row * p.Pmax + cq) * D + i) >> 2] = v;
            }
        } else {
            for (int e = threadIdx.x; e < nh * D && !merge && !skip_out; e += blockDim.x) {
                const int hh = e / D, i = e - hh * D;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < RED; ++w) v += red_o[(w * nh + hh) * RS + i];
                v *= vmul * fac_o[hh];
                for (int k = 0; k < K - 1; ++k) v = fmaf(pbuf[k * pstride + 2 * kMaxHeadsPerCta + e], pbuf[k * pstride + hh], v);
                const int64_t row = (int64_t)s * H + h0 + hh;
                if (direct)
                    store_out<BF16>(p.out, row * D + i, v);
                else if (p.tmp16)
                    store_out<BF16>(p.tmp_out, (row * p.Pmax + cq) * D + i, v);
                else
                    static_cast<float*>(p.tmp_out)[(row * p.Pmax + cq) * D + i] = v;
            }
        }
        if (threadIdx.x < nh && !skip_out) {
            const int hh = threadIdx.x;
            const int64_t sidx = ((int64_t)s * H + h0 + hh) * p.Pmax + cq;
            const float lt = fin_l[hh];
            float mlog = -INFINITY;
            if (lt > 0.f) {
                mlog = fin_m[hh] * kLn2;
                if (p.alibi != nullptr) mlog = fmaf(p.alibi[h0 + hh], (float)tref, mlog);
            }
            p.max_logits[sidx] = mlog;
            p.exp_sums[sidx] = lt;
        }
        __syncthreads();  // the merge buffers are reused by the next partition

        // move the id buffers one partition on (the next ones were checked already; the ones
        // after them were loaded at the start of this partition)
        c0 = n0;
        c1 = n1;
        cmask = nmask;
        n0 = nn0;
        n1 = nn1;
        nmask = cq + 2 * PX < Pl ? validate(cq + 2 * PX, n0, n1) : 0u;
    }

    if (aborted) {
        // Let every copy this warp started land before the block can exit.
        for (uint32_t n = drain_from; n < nis; ++n)
            (void)mbar_wait_bounded(&bars[n % nstage], (n / nstage) & 1u, kWaitLimitNs);
    }

    // Fused combine: count this CTA in; the last of the (sequence, head group) to arrive
    // merges the rows of all of them.  Nothing waits: every CTA but the last just exits.
    if (fused && Pl > 1 && !direct && kc == 0) {
        // the CTA's rows and statistics are written; one thread publishes them GPU-wide (the
        // fence after the barrier covers the writes of every thread of the CTA) and arrives
        __syncthreads();
        int* last = reinterpret_cast<int*>(red_m);
        if (threadIdx.x == 0) {
            __threadfence();
            uint32_t* ctr = p.counters + ((int64_t)s * gridDim.y + kvh) * ng + grp;
            const uint32_t before = atomicAdd(ctr, 1u);
            const bool is_last = before == (uint32_t)(nwork - 1);
            if (is_last) atomicExch(ctr, 0u);  // left at zero for the next call
            __threadfence();
            *last = is_last ? 1 : 0;
        }
        __syncthreads();
        if (*last) {
            // the page ring is idle now (every copy has landed): it holds the row weights
            fused_combine<BF16, D>(p, s, h0, nh, Pl, merge ? PX : Pl, reinterpret_cast<float*>(smem));
        }
    }
    griddep_launch_dependents();
}


template <bool BF16, int KVB, int BS, int FORM>
static Phase1Fn pick_phase1(int d) {
    switch (d) {
        case 64: return pa_v2_phase1_kernel<BF16, KVB, 64, BS, FORM>;
        case 80: return pa_v2_phase1_kernel<BF16, KVB, 80, BS, FORM>;
        case 96: return pa_v2_phase1_kernel<BF16, KVB, 96, BS, FORM>;
        case 112: return pa_v2_phase1_kernel<BF16, KVB, 112, BS, FORM>;
        case 128: return pa_v2_phase1_kernel<BF16, KVB, 128, BS, FORM>;
        case 192: return pa_v2_phase1_kernel<BF16, KVB, 192, BS, FORM>;
        case 256: return pa_v2_phase1_kernel<BF16, KVB, 256, BS, FORM>;
        case 120:
            if constexpr (KVB == 2) return pa_v2_phase1_kernel<BF16, KVB, 120, BS, FORM>;
            else return nullptr;
        default: return nullptr;
    }
}

template <int BS, int KVB, int FORM>
Phase1Fn phase1_select(bool bf16, int d) {
    return bf16 ? pick_phase1<true, KVB, BS, FORM>(d) : pick_phase1<false, KVB, BS, FORM>(d);
}

template <int BS, int KVB, int FORM>
cudaError_t phase1_read_errors(unsigned int* v, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_phase1_errors, sizeof(*v));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_phase1_errors, &z, sizeof(z));
}

}  // namespace pa
