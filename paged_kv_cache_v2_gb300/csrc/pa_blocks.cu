// pa_blocks.cu -- whole-block moves between and inside paged caches for sm_103a:
// copy_blocks (copy-on-write inside every layer's K and V cache) and swap_blocks (moves
// between two caches, typically GPU and pinned host memory).  "paged_attn.py",
// copy_blocks / swap_blocks.
//
// copy_blocks: one CTA per (pair, layer); its 256 threads stream the K block and then the V
// block with 16-byte loads and stores, eight in flight per thread.  Block ids are checked on
// the device (out-of-range pairs are skipped and flagged) because the mapping lives there.
// swap_blocks: the mapping is on the host.  Where both caches are addressable from the
// device (device memory, pinned host memory) a kernel moves the blocks with the pairs in its
// launch parameters; otherwise each pair becomes one cudaMemcpyAsync of one contiguous block
// (no batched-copy API is used).
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_v2.h"

namespace pa {

static __device__ unsigned int g_block_errors = 0;

constexpr int kMaxLayersPerLaunch = 64;
constexpr int kCopyThreads = 256;

struct CopyParams {
    void* kc[kMaxLayersPerLaunch];
    void* vc[kMaxLayersPerLaunch];
    const int64_t* mapping;
    int64_t block_bytes;
    int num_blocks;
};

__global__ void __launch_bounds__(kCopyThreads) pa_copy_blocks_kernel(const CopyParams p) {
    const int pair = blockIdx.x, layer = blockIdx.y;
    const int64_t src = p.mapping[2 * (int64_t)pair], dst = p.mapping[2 * (int64_t)pair + 1];
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (threadIdx.x == 0 && layer == 0) atomicOr(&g_block_errors, 16u);
        return;
    }
    const int64_t n16 = p.block_bytes / 16;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
        uint4* base = reinterpret_cast<uint4*>(kv == 0 ? p.kc[layer] : p.vc[layer]);
        const uint4* s = base + src * n16;
        uint4* d = base + dst * n16;
        int64_t i = threadIdx.x;
        for (; i + 7 * kCopyThreads < n16; i += 8 * kCopyThreads) {
            uint4 r[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) r[u] = s[i + u * kCopyThreads];
#pragma unroll
            for (int u = 0; u < 8; ++u) d[i + u * kCopyThreads] = r[u];
        }
        for (; i < n16; i += kCopyThreads) d[i] = s[i];
    }
}

// swap_blocks by a kernel: one CTA per pair streams the block with 16-byte loads and stores,
// eight in flight per thread, reading and writing pinned host memory through its device
// mapping.  The pairs travel in the launch's parameters (the mapping is on the host).
constexpr int kSwapPairsPerLaunch = 480;  // 3840 bytes of pairs: within the 4 KiB of parameters

struct SwapParams {
    const uint8_t* src;
    uint8_t* dst;
    int64_t block_bytes;
    int2 pairs[kSwapPairsPerLaunch];
};

__global__ void __launch_bounds__(kCopyThreads) pa_swap_blocks_kernel(const SwapParams p) {
    const int2 pr = p.pairs[blockIdx.x];
    const int64_t n16 = p.block_bytes / 16;
    const uint4* s = reinterpret_cast<const uint4*>(p.src) + pr.x * n16;
    uint4* d = reinterpret_cast<uint4*>(p.dst) + pr.y * n16;
    int64_t i = threadIdx.x;
    for (; i + 7 * kCopyThreads < n16; i += 8 * kCopyThreads) {
        uint4 r[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) r[u] = s[i + u * kCopyThreads];
#pragma unroll
        for (int u = 0; u < 8; ++u) d[i + u * kCopyThreads] = r[u];
    }
    for (; i < n16; i += kCopyThreads) d[i] = s[i];
}

// The address under which the current device reaches `ptr`: device memory of the current
// device (or managed memory) as is, host memory pinned or registered while the current
// device was active through its device mapping; null for anything else (pageable host
// memory, another device's memory, host memory pinned for another device's context).
static const void* device_view(const void* ptr) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (at.type == cudaMemoryTypeManaged) return ptr;
    if (at.type == cudaMemoryTypeDevice) return at.device == dev ? ptr : nullptr;
    if (at.type == cudaMemoryTypeHost) return at.device == dev ? at.devicePointer : nullptr;
    return nullptr;
}

}  // namespace pa

using namespace pa;

cudaError_t pa::read_block_errors(unsigned int* v, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_block_errors, sizeof(*v));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_block_errors, &z, sizeof(z));
}

extern "C" pa_status pa_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                                    const int64_t* block_mapping, int num_pairs, int64_t block_bytes,
                                    int num_blocks, cudaStream_t stream) {
    if (num_layers < 0 || num_pairs < 0 || num_blocks <= 0 || block_bytes <= 0 || block_bytes % 16)
        return PA_ERR_INVALID_ARG;
    if (num_layers == 0 || num_pairs == 0) return PA_OK;
    if (num_pairs > 2147483647 / 2 || key_caches == nullptr || value_caches == nullptr || block_mapping == nullptr)
        return PA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(block_mapping) & 7) return PA_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l) {
        if (key_caches[l] == nullptr || value_caches[l] == nullptr) return PA_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(key_caches[l]) | reinterpret_cast<uintptr_t>(value_caches[l])) & 15)
            return PA_ERR_INVALID_ARG;
    }
    for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
        const int nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0 : kMaxLayersPerLaunch;
        CopyParams p = {};
        for (int l = 0; l < nl; ++l) {
            p.kc[l] = key_caches[l0 + l];
            p.vc[l] = value_caches[l0 + l];
        }
        p.mapping = block_mapping;
        p.block_bytes = block_bytes;
        p.num_blocks = num_blocks;
        pa_copy_blocks_kernel<<<dim3((unsigned)num_pairs, (unsigned)nl), kCopyThreads, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

extern "C" pa_status pa_swap_blocks(const void* src_cache, void* dst_cache, const int64_t* block_mapping,
                                    int num_pairs, int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                                    cudaStream_t stream) {
    if (num_pairs < 0 || block_bytes <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (src_cache == nullptr || dst_cache == nullptr || block_mapping == nullptr) return PA_ERR_INVALID_ARG;
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t s = block_mapping[2 * (int64_t)i], d = block_mapping[2 * (int64_t)i + 1];
        if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) return PA_ERR_INVALID_ARG;
    }
    // Both caches addressable from this device and blocks of whole 16-byte chunks: a kernel
    // moves every block of a launch (one launch per 480 pairs); else one copy per pair, which
    // costs a couple of microseconds of host time each (512 blocks out and 512 in of 32 KiB:
    // 16.3 GB/s against 186 GB/s for the same bytes as one copy each way).
    const void* src_dev = device_view(src_cache);
    const void* dst_dev = device_view(dst_cache);
    if (src_dev != nullptr && dst_dev != nullptr && block_bytes % 16 == 0 &&
        ((reinterpret_cast<uintptr_t>(src_dev) | reinterpret_cast<uintptr_t>(dst_dev)) & 15) == 0 &&
        src_num_blocks <= 2147483647 && dst_num_blocks <= 2147483647) {
        SwapParams p;
        p.src = static_cast<const uint8_t*>(src_dev);
        p.dst = static_cast<uint8_t*>(const_cast<void*>(dst_dev));
        p.block_bytes = block_bytes;
        for (int i0 = 0; i0 < num_pairs; i0 += kSwapPairsPerLaunch) {
            const int n = num_pairs - i0 < kSwapPairsPerLaunch ? num_pairs - i0 : kSwapPairsPerLaunch;
            for (int i = 0; i < n; ++i)
                p.pairs[i] = make_int2((int)block_mapping[2 * (int64_t)(i0 + i)],
                                       (int)block_mapping[2 * (int64_t)(i0 + i) + 1]);
            pa_swap_blocks_kernel<<<(unsigned)n, kCopyThreads, 0, stream>>>(p);
            if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
        }
        return PA_OK;
    }
    const char* src = static_cast<const char*>(src_cache);
    char* dst = static_cast<char*>(dst_cache);
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t s = block_mapping[2 * (int64_t)i], d = block_mapping[2 * (int64_t)i + 1];
        if (cudaMemcpyAsync(dst + d * block_bytes, src + s * block_bytes, (size_t)block_bytes, cudaMemcpyDefault,
                            stream) != cudaSuccess) {
            (void)cudaGetLastError();
            return PA_ERR_CUDA;
        }
    }
    return PA_OK;
}
