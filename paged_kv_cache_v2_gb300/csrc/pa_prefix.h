// pa_prefix.h -- declarations shared by the prefix kernel (pa_prefix.cuh) and its host entry
// point (pa_prefix.cu): warp roles, launch parameters, the per-dtype launcher tables.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// ---- chunked-prefix attention ----------------------------------------------------------
// Warp roles of the prefix kernel: warp 0 allocates tensor memory and one of its lanes issues
// the score MMAs, one lane of warp 1 issues the value MMAs (an MMA issue blocks the issuing
// thread until the tensor core takes it, so the two products get a thread each), warps 2-3
// fill the key ring and warps 8-9 the value ring in shared memory, and warps 4-7 run the
// softmax (warp 4 + w owns tensor-memory lanes 32w..32w+31, i.e. query rows 32w..32w+31).
// Each sub-partition runs one softmax warp next to an MMA lane or a loader; the MMA lanes
// take the lowest warp numbers (measured about 1% faster than the softmax warps first).
constexpr int kPfxMmaWarp = 0, kPfxPvWarp = 1, kPfxKeyWarp0 = 2, kPfxSoftmaxWarp0 = 4, kPfxValWarp0 = 8;
static_assert(kPfxSoftmaxWarp0 % 4 == 0, "softmax warp w must own tensor-memory lane quarter w");
constexpr int kPfxThreads = 10 * 32;
constexpr int kPfxBM = 128;    // query rows per CTA (the MMA M)

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
    // Split contexts: the grid's x is mt row tiles (of the kernel's rows per CTA) x nsplit
    // splits.  A sequence with more than split_tiles 64-key context tiles is cut into at most
    // nsplit parts whose partial results (O rows of d fp32 values, and a (reference max, sum)
    // pair per row) go to ws_o / ws_ml at [((s * Hk + kvh) * mt_ws + r / 128) * nsplit +
    // split][r % 128] for row r = j * G + g of the kv head's group.
    int mt, mt_ws, nsplit, split_tiles;
    float* ws_o;
    float2* ws_ml;
};

using PrefixFn = cudaError_t (*)(const PrefixParams&, dim3 grid, cudaStream_t);

// Prefix kernel launcher for (query dtype, head size), or nullptr; defined in pa_prefix_<dtype>.cu.
template <bool BF16>
PrefixFn prefix_select(int d);
template <bool BF16>
cudaError_t prefix_read_errors(unsigned int* v, bool reset);
// Query rows per CTA of the kernel prefix_select picks (128, or 256 where two row groups share
// each key/value tile).
template <bool BF16>
int prefix_tile_rows(int d);
// The combine of split partial results (grid: ceil(max_query_len * H / 8) x num_seqs).
template <bool BF16>
cudaError_t launch_prefix_combine(const PrefixParams& p, int d, dim3 grid, cudaStream_t stream);

}  // namespace pa
