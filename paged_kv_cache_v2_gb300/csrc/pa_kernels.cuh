// pa_kernels.cuh -- definitions shared by the paged-attention kernels and their launchers:
// tuning constants, kernel parameter blocks, the output store.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
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
constexpr uint32_t kRingTarget = PA_RING_KIB * 1024u;  // shared-memory page ring per CTA
constexpr int kMaxHeadsPerCta = 8;     // the MMA N dimension
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
    int tmp16;  // tmp_output holds the output dtype instead of fp32
};

struct Phase2Params {
    void* out;
    const float* exp_sums;
    const float* max_logits;
    const void* tmp_out;  // fp32, or the output dtype (template parameter TMP16)
    const int32_t* seq_lens;
    int H, D, Pmax;
};

template <bool BF16>
__device__ __forceinline__ void store_out(void* out, int64_t idx, float v) {
    if constexpr (BF16)
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
}

using Phase1Fn = void (*)(const Phase1Params);

// Phase-1 kernel for (query dtype, fp8 cache?, head size) at block size BS, or nullptr;
// defined in pa_phase1_bs<BS>.cu.
template <int BS>
Phase1Fn phase1_select(bool bf16, bool fp8, int d);
// Read (and optionally clear) the device error word of the block-size-BS phase-1 kernels.
template <int BS>
cudaError_t phase1_read_errors(unsigned int* v, bool reset);

// ---- chunked-prefix attention ----------------------------------------------------------
// Warp roles of the prefix kernel: warps 0-3 run the softmax (warp w owns tensor-memory lanes
// 32w..32w+31, i.e. query rows 32w..32w+31), warp 4 allocates tensor memory and one of its
// lanes issues the MMAs, warps 5-8 copy query, key and value tiles into shared memory.
constexpr int kPfxMmaWarp = 4;
constexpr int kPfxLoaderWarp0 = 5;
constexpr int kPfxLoaderThreads = 4 * 32;
constexpr int kPfxThreads = 9 * 32;
constexpr int kPfxBM = 128;    // query rows per CTA (the MMA M)
constexpr int kPfxStages = 2;  // key/value tile stages

struct PrefixParams {
    CUtensorMap kmap;  // key cache as {64 elems = 8 tokens x 8, block_size/8, d/8, blocks * kv heads}
    CUtensorMap vmap;  // value cache as {block_size keys, d, blocks * kv heads}, 32/64-byte swizzle
    void* out;
    const uint8_t* q;  // [T][q_stride] rows, head h at h * d
    const uint8_t* k;  // [T][kv_stride] rows, kv head at kvh * d
    const uint8_t* v;
    const uint8_t* kcache;
    const uint8_t* vcache;
    const int32_t* block_tables;
    const int32_t* qsl;
    const int32_t* ctx_lens;
    int H, Hk, G, bs, bs_log2, mbps, num_blocks, max_query_len;
    int64_t q_stride, kv_stride;  // elements between consecutive tokens
    float sl2;                    // scale * log2(e)
};

using PrefixFn = cudaError_t (*)(const PrefixParams&, dim3 grid, cudaStream_t);

// Prefix kernel launcher for (query dtype, head size), or nullptr; defined in pa_prefix_<dtype>.cu.
template <bool BF16>
PrefixFn prefix_select(int d);
template <bool BF16>
cudaError_t prefix_read_errors(unsigned int* v, bool reset);

}  // namespace pa
