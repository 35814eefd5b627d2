// pa_kernels.cuh -- definitions shared by the paged-attention kernels and their launchers:
// tuning constants, kernel parameter blocks, the output store.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

#ifndef PA_PHASE1_WARPS
#define PA_PHASE1_WARPS 4
#endif
#ifndef PA_RING_KIB
#define PA_RING_KIB 64
#endif
#ifndef PA_MIN_STAGES
#define PA_MIN_STAGES 1
#endif
#ifndef PA_GRID_WAVES
#define PA_GRID_WAVES 16
#endif

constexpr int kPartition = 512;
constexpr int kWarps = PA_PHASE1_WARPS;  // phase-1 warps per CTA
static_assert(kWarps % 2 == 0, "warps pair up in the cross-warp reduction of phase-1 form 3");
// phase 1's static shared memory: per warp, the value scale and the two encode divisors
constexpr int kPhase1StaticSmem = kWarps * 3 * (int)sizeof(float);
constexpr uint32_t kRingTarget = PA_RING_KIB * 1024u;  // shared-memory page ring per CTA
constexpr int kMaxHeadsPerCta = 8;     // the MMA N dimension
// Fused combine: most bytes of rows the last CTA of a (sequence, head group) merges.
#ifndef PA_FUSED_ROW_KIB
#define PA_FUSED_ROW_KIB 128
#endif
constexpr int64_t kFusedRowBytes = PA_FUSED_ROW_KIB * 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Phase1Params {
    void* out;
    float* exp_sums;
    float* max_logits;
    void* tmp_out;  // fp32, or the output dtype when tmp16
    const void* query;
    const uint8_t* kcache;
    const uint8_t* vcache;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const float* alibi;
    int H, Hk, G, ngroups, bs, mbps, num_blocks, Pmax, nstage;
    uint32_t ring_bytes;  // kWarps * nstage * slot bytes
    float qk_scale_log2;  // scale * k_scale * log2(e)
    float v_scale;
    // One k_scale / v_scale per kv head ([Hk] floats, device), or nullptr: then qk_scale_log2,
    // v_scale, k_enc and v_enc come from k_scales[kvh] / v_scales[kvh] (scale * k * log2(e)
    // rounded in that order, as the host rounds the per-tensor product).
    const float* k_scales;
    const float* v_scales;
    float scale;
    int tmp16;  // tmp_output holds the output dtype instead of fp32
    // Combine fused into phase 1 (counters != nullptr): the last CTA of a (sequence, head
    // group) to finish merges the partitions; counters[s * gridDim.y + blockIdx.y] counts the
    // CTAs that have finished and is reset to 0 by the last one.
    uint32_t* counters;
    // Each CTA merges its own partitions px, px + PX, ... into fp32 row px of tmp_output
    // (instead of one row per partition; tmp_output is then the caller's scratch), so the
    // combine -- the last CTA's or phase 2's -- merges at most PX rows.
    int merge;
    // CTAs per partition (1, 2 or 4; more than 1 only with one partition per CTA): a cluster
    // of csplit CTAs shares each partition's pages, and the others hand their partial
    // (max, exp-sum, rows) to the cluster's first CTA through distributed shared memory.
    int csplit;
    uint32_t mrg_off;  // shared-memory byte offset of the CTA merge row (merge with PX < Pmax)
    // Fused cache append (new_k != nullptr): the key/value rows of each sequence's newest
    // token, position seq_lens[s] - 1 ([S][Hk][D] in the query dtype, rows nk_stride /
    // nv_stride elements apart).  The CTA that streams that token's page writes them into
    // the caches (encoded as the cache writer does) and into its shared-memory copy of the
    // page, so the step needs no separate writer kernel.
    const uint16_t* new_k;
    const uint16_t* new_v;
    int64_t nk_stride, nv_stride;
    float k_enc, v_enc;   // k_scale, v_scale (the fp8 encode divides by them)
    // Grid order (or nullptr): blockIdx.z = z serves sequence order[z], a permutation of the
    // sequences that puts those with the most partitions first, so the CTAs that stream
    // many partitions start early instead of forming the grid's tail.
    const int32_t* order;
    uint32_t nrow_off;    // shared-memory byte offset of the staged new rows (2 x D x 2 bytes)
};

struct Phase2Params {
    void* out;
    const float* exp_sums;
    const float* max_logits;
    const void* tmp_out;  // fp32, or the output dtype (template parameter TMP16)
    const int32_t* seq_lens;
    int S, H, D, Pmax;
    int rstride;  // merged rows: row r holds partitions r, r + rstride, ... (phase-1 CTA merge)
};

template <bool BF16>
__device__ __forceinline__ void store_out(void* out, int64_t idx, float v) {
    if constexpr (BF16)
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
}

// Four consecutive output elements (idx a multiple of 4): one 8-byte store where the buffer
// allows it (the ABI asks only 4-byte alignment of the output), else four element stores.
template <bool BF16>
__device__ __forceinline__ void store_out4(void* out, int64_t idx, float4 v) {
    if (reinterpret_cast<uintptr_t>(out) & 7u) {
        store_out<BF16>(out, idx, v.x);
        store_out<BF16>(out, idx + 1, v.y);
        store_out<BF16>(out, idx + 2, v.z);
        store_out<BF16>(out, idx + 3, v.w);
        return;
    }
    uint2 w;
    if constexpr (BF16) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        w.x = *reinterpret_cast<const uint32_t*>(&a);
        w.y = *reinterpret_cast<const uint32_t*>(&b);
    } else {
        const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        w.x = *reinterpret_cast<const uint32_t*>(&a);
        w.y = *reinterpret_cast<const uint32_t*>(&b);
    }
    reinterpret_cast<uint2*>(out)[idx >> 2] = w;
}

using Phase1Fn = void (*)(const Phase1Params);

// Phase-1 kernel for (query dtype, head size) at block size BS, cache element bytes KVB (2:
// fp16/bf16, 1: fp8) and FORM (0: per-tensor scales; 1: per-kv-head scales; 2: per-tensor
// scales and an ordered grid), or nullptr; defined in pa_phase1_bs<BS>[_fp8][_hs|_ord].cu,
// one translation unit each so they build in parallel.
template <int BS, int KVB, int FORM>
Phase1Fn phase1_select(bool bf16, int d);
// Read (and optionally clear) the device error word of those kernels (one per unit).
template <int BS, int KVB, int FORM>
cudaError_t phase1_read_errors(unsigned int* v, bool reset);

}  // namespace pa
