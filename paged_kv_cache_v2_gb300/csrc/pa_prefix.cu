// pa_prefix.cu -- host entry point of chunked-prefix attention ("paged_attn.py",
// forward_prefix): argument checks, grid sizing, kernel selection, the split-context
// workspace.  The kernels live in pa_prefix.cuh (128 query rows per CTA: head sizes 192 and
// 256; the loader, the split plan and the combine) and pa_prefix_m256.cuh (256 rows per CTA:
// head sizes up to 128; prefix_select), instantiated per dtype in pa_prefix_f16.cu /
// pa_prefix_bf16.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "pa_internal.h"
#include "pa_kernels.cuh"
#include "pa_prefix.h"
#include "pa_v2.h"

using namespace pa;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Tensor maps of the paged caches for the prefix kernel's tile copies:
//   keys   {64 elements = 8 tokens x 8, block_size/8 token groups, d/8 chunks, blocks * kv
//          heads}, box {64, 1, d/8, 1}: 8 tokens of one page land as [d/8][8 tokens][16 bytes]
//          with 128-byte rows read from global memory;
//   values {block_size keys, d rows, blocks * kv heads}, box {block_size, d, 1} with the
//          32-byte (block size 16) or 64-byte (block size 32) swizzle: a whole page lands in the
//          swizzled K-major layout the value MMA reads.  Block size 8 pages are plain 16-byte
//          rows and move by 1-d bulk copies (the map is still encoded, unswizzled).
static bool encode_cache_maps(PrefixParams& p, const void* key_cache, const void* value_cache, int num_blocks,
                              int num_kv_heads, int head_size, int block_size) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t pages = (cuuint64_t)num_blocks * num_kv_heads;
    const cuuint64_t d = head_size, bs = block_size;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const cuuint64_t kdim[4] = {64, bs / 8, d / 8, pages};
    const cuuint64_t kstride[3] = {128, bs * 16, d * bs * 2};
    const cuuint32_t kbox[4] = {64, 1, (cuuint32_t)(d / 8), 1};
    if (enc(&p.kmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(key_cache), kdim, kstride, kbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const cuuint64_t vdim[3] = {bs, d, pages};
    const cuuint64_t vstride[2] = {bs * 2, d * bs * 2};
    const cuuint32_t vbox[3] = {(cuuint32_t)bs, (cuuint32_t)d, 1};
    const CUtensorMapSwizzle sw = block_size == 16   ? CU_TENSOR_MAP_SWIZZLE_32B
                                  : block_size == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                     : CU_TENSOR_MAP_SWIZZLE_NONE;
    return enc(&p.vmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(value_cache), vdim, vstride, vbox, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Default minimum context per split: 16384 keys (256 tiles of 64).
static constexpr int kDefaultSplitKeys = 16384;
static constexpr int kMaxSplits = 32;

static int64_t prefix_row_tiles(int max_query_len, int G) { return ((int64_t)max_query_len * G + kPfxBM - 1) / kPfxBM; }

extern "C" size_t pa_prefix_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                           int max_query_len, int max_splits) {
    if (max_splits <= 1 || num_seqs <= 0 || max_query_len <= 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_size <= 0 || num_heads % num_kv_heads || max_splits > kMaxSplits)
        return 0;
    const int64_t items =
        (int64_t)num_seqs * num_kv_heads * prefix_row_tiles(max_query_len, num_heads / num_kv_heads) * max_splits;
    return (size_t)(items * kPfxBM * ((int64_t)head_size * 4 + 8));
}

// Parts each context is cut into (1: none), for a call with these sizes and a workspace
// (has_ws): contexts over split_keys tokens (min_split_keys, 0: 16384) into up to max_splits
// parts, no more than the longest context the tables can hold would use; with min_split_keys
// = 0 only where one sequence's CTAs (cta_tiles row tiles of each kv head, one attention CTA
// an SM) would occupy fewer than half the SMs: a grid that already spreads every sequence over
// the GPU ran faster unsplit (4 sequences x 1024 new tokens over contexts up to 96K, head size
// 256: 2.82 against 3.04 ms cut into up to 7 parts).
static pa_status prefix_parts(int64_t cta_tiles, int num_kv_heads, int max_blocks_per_seq, int block_size,
                              int max_splits, int min_split_keys, bool has_ws, int* parts) {
    *parts = 1;
    if (!has_ws || max_splits <= 1) return PA_OK;
    const int64_t split_tiles = (min_split_keys > 0 ? min_split_keys : kDefaultSplitKeys) / 64;
    const int64_t max_ctx_tiles = ((int64_t)max_blocks_per_seq * block_size + 63) / 64;
    if (max_ctx_tiles <= split_tiles) return PA_OK;
    const int n = (int)std::min<int64_t>(max_splits, (max_ctx_tiles + split_tiles - 1) / split_tiles);
    if (min_split_keys == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return PA_ERR_CUDA;
        }
        if (2 * cta_tiles * num_kv_heads >= sms) return PA_OK;
    }
    *parts = n;
    return PA_OK;
}

extern "C" pa_status pa_prefix_num_parts(int num_heads, int num_kv_heads, int head_size, pa_dtype dtype,
                                         int max_query_len, int max_blocks_per_seq, int block_size, int max_splits,
                                         int min_split_keys, int has_workspace, int* parts) {
    if (parts == nullptr || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || max_query_len < 0 ||
        max_blocks_per_seq <= 0 || (block_size != 8 && block_size != 16 && block_size != 32) || max_splits < 1 ||
        max_splits > kMaxSplits || min_split_keys < 0 || min_split_keys % 64)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_DT_F16 && dtype != PA_DT_BF16) return PA_ERR_UNSUPPORTED;
    const bool bf16 = dtype == PA_DT_BF16;
    if ((bf16 ? prefix_select<true>(head_size) : prefix_select<false>(head_size)) == nullptr) return PA_ERR_UNSUPPORTED;
    const int G = num_heads / num_kv_heads;
    const int cta_rows = bf16 ? prefix_tile_rows<true>(head_size) : prefix_tile_rows<false>(head_size);
    const int64_t cta_tiles = ((int64_t)max_query_len * G + cta_rows - 1) / cta_rows;
    return prefix_parts(cta_tiles, num_kv_heads, max_blocks_per_seq, block_size, max_splits, min_split_keys,
                        has_workspace != 0, parts);
}

extern "C" pa_status pa_prefix(void* output, const void* query, const void* key, const void* value,
                               const void* key_cache, const void* value_cache, int num_seqs, int num_heads,
                               int num_kv_heads, int head_size, float scale, const int32_t* block_tables,
                               int max_blocks_per_seq, int num_blocks, const int32_t* query_start_loc,
                               const int32_t* context_lens, int max_query_len, int block_size,
                               int64_t q_row_stride, int64_t kv_row_stride, pa_dtype dtype, void* workspace,
                               size_t workspace_bytes, int max_splits, int min_split_keys, cudaStream_t stream) {
    if (num_seqs < 0 || num_seqs > 65535 || max_query_len < 0) return PA_ERR_INVALID_ARG;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || num_kv_heads > 65535)
        return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (dtype != PA_DT_F16 && dtype != PA_DT_BF16) return PA_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    const bool bf16 = dtype == PA_DT_BF16;
    PrefixFn fn = bf16 ? prefix_select<true>(head_size) : prefix_select<false>(head_size);
    if (fn == nullptr) return PA_ERR_UNSUPPORTED;
    const int G = num_heads / num_kv_heads;
    if ((int64_t)max_query_len * G > (1ll << 30) || (int64_t)max_blocks_per_seq * block_size > (1ll << 30))
        return PA_ERR_INVALID_ARG;
    // tensor-copy coordinates are signed 32-bit: a page is addressed as block * kv heads + kv head
    if ((int64_t)num_blocks * num_kv_heads >= (1ll << 31)) return PA_ERR_INVALID_ARG;
    if (q_row_stride < (int64_t)num_heads * head_size || kv_row_stride < (int64_t)num_kv_heads * head_size ||
        q_row_stride % 8 || kv_row_stride % 8)
        return PA_ERR_INVALID_ARG;
    const bool split = max_splits > 1 && workspace != nullptr;
    if (split) {
        if (max_splits > kMaxSplits || min_split_keys < 0 || min_split_keys % 64 || !aligned16(workspace))
            return PA_ERR_INVALID_ARG;
        if (num_seqs > 0 && max_query_len > 0 &&
            workspace_bytes <
                pa_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_query_len, max_splits))
            return PA_ERR_INVALID_ARG;
    }
    if (num_seqs == 0 || max_query_len == 0) return PA_OK;
    if (!output || !query || !key || !value || !key_cache || !value_cache || !block_tables || !query_start_loc ||
        !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(output) || !aligned16(query) || !aligned16(key) || !aligned16(value) || !aligned16(key_cache) ||
        !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;

    PrefixParams p;
    if (!encode_cache_maps(p, key_cache, value_cache, num_blocks, num_kv_heads, head_size, block_size))
        return PA_ERR_CUDA;
    p.out = output;
    p.q = static_cast<const uint8_t*>(query);
    p.k = static_cast<const uint8_t*>(key);
    p.v = static_cast<const uint8_t*>(value);
    p.kcache = static_cast<const uint8_t*>(key_cache);
    p.vcache = static_cast<const uint8_t*>(value_cache);
    p.block_tables = block_tables;
    p.qsl = query_start_loc;
    p.ctx_lens = context_lens;
    p.H = num_heads;
    p.Hk = num_kv_heads;
    p.G = G;
    p.bs = block_size;
    p.bs_log2 = block_size == 8 ? 3 : (block_size == 16 ? 4 : 5);
    p.mbps = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.max_query_len = max_query_len;
    p.q_stride = q_row_stride;
    p.kv_stride = kv_row_stride;
    p.sl2 = scale * kLog2e;
    const int64_t row_tiles = prefix_row_tiles(max_query_len, G);  // of 128 rows: the workspace's unit
    const int cta_rows = bf16 ? prefix_tile_rows<true>(head_size) : prefix_tile_rows<false>(head_size);
    const int64_t cta_tiles = ((int64_t)max_query_len * G + cta_rows - 1) / cta_rows;
    p.mt = (int)cta_tiles;
    p.mt_ws = (int)row_tiles;
    p.split_tiles = (min_split_keys > 0 ? min_split_keys : kDefaultSplitKeys) / 64;
    const pa_status plan = prefix_parts(cta_tiles, num_kv_heads, max_blocks_per_seq, block_size, max_splits,
                                        min_split_keys, split, &p.nsplit);
    if (plan != PA_OK) return plan;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = nullptr;
    if (p.nsplit > 1) {
        const int64_t rows = (int64_t)num_seqs * num_kv_heads * row_tiles * p.nsplit * kPfxBM;
        p.ws_ml = reinterpret_cast<float2*>(static_cast<float*>(workspace) + rows * head_size);
    }
    if (row_tiles * p.nsplit > INT32_MAX || ((int64_t)max_query_len * num_heads + 7) / 8 > INT32_MAX)
        return PA_ERR_INVALID_ARG;
    const dim3 grid((unsigned)(cta_tiles * p.nsplit), (unsigned)num_kv_heads, (unsigned)num_seqs);
    cudaEvent_t t_begin, t_end;
    timing_events(&t_begin, &t_end);
    if (t_begin != nullptr) cudaEventRecord(t_begin, stream);
    cudaError_t e = fn(p, grid, stream);
    if (t_end != nullptr) cudaEventRecord(t_end, stream);
    if (e == cudaSuccess && p.nsplit > 1) {
        const dim3 cgrid((unsigned)(((int64_t)max_query_len * num_heads + 7) / 8), (unsigned)num_seqs);
        e = bf16 ? launch_prefix_combine<true>(p, head_size, cgrid, stream)
                 : launch_prefix_combine<false>(p, head_size, cgrid, stream);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}
