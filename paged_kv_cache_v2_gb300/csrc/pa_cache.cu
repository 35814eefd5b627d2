// pa_cache.cu -- slot-mapping cache writer ("paged_attn.py", write_to_paged_cache ->
// reshape_and_cache; cache views from split_kv_cache) for sm_103a.
//
// One CTA per new token, one thread per x-element chunk of one kv head: the K
// chunk is contiguous in both the source row and the cache (x elements = 16 bytes), so it
// is one 16-byte store; the V elements of a chunk land block_size elements apart
// (value_cache[b][h][i][o]).  fp16/bf16 caches get a bitwise copy; an fp8 cache gets
// e4m3fn(RNE, saturating) of x / k_scale with the division in IEEE fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_v2.h"
#include "pa_ptx.cuh"

namespace pa {

static __device__ unsigned int g_cache_errors = 0;

struct CacheParams {
    const uint16_t* key;
    const uint16_t* value;
    int64_t kstride, vstride;  // elements between consecutive tokens
    uint8_t* kcache;
    uint8_t* vcache;
    const int64_t* slots;
    int Hk, D, bs, num_blocks;
    float k_scale, v_scale;
    const float* k_scales;  // [Hk] per-kv-head scales replacing k_scale / v_scale, or nullptr
    const float* v_scales;
    int vec;  // 1 when 16-byte source loads are aligned
};

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t v) {
    if constexpr (BF16)
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
    else
        return __half2float(__ushort_as_half(v));
}

template <bool FP8, bool BF16>
__global__ void __launch_bounds__(512) pa_cache_write_kernel(const CacheParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int tok = blockIdx.x;
    constexpr int X = FP8 ? 16 : 8;
    const int nchunk = p.D / X;
    const int kvb = FP8 ? 1 : 2;
    union Chunk { uint4 v[X / 8]; uint16_t h[X]; };
    // key / value chunk c = (kv head, X-element group) of this token's rows
    auto load_chunk = [&](int c, Chunk& kc, Chunk& vc) {
        const int h = c / nchunk, ch = c - h * nchunk;
        const uint16_t* ks = p.key + tok * p.kstride + (int64_t)h * p.D + ch * X;
        const uint16_t* vs = p.value + tok * p.vstride + (int64_t)h * p.D + ch * X;
        if (p.vec) {
#pragma unroll
            for (int i = 0; i < X / 8; ++i) {
                kc.v[i] = reinterpret_cast<const uint4*>(ks)[i];
                vc.v[i] = reinterpret_cast<const uint4*>(vs)[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < X; ++i) {
                kc.h[i] = ks[i];
                vc.h[i] = vs[i];
            }
        }
    };
    // this thread's first chunk is read together with the slot (neither depends on the other)
    Chunk k0, v0;
    if (threadIdx.x < p.Hk * nchunk) load_chunk(threadIdx.x, k0, v0);
    const int64_t slot = p.slots[tok];
    if (slot < 0) return;
    if (slot >= (int64_t)p.num_blocks * p.bs) {
        if (threadIdx.x == 0) atomicOr(&g_cache_errors, 8u);
        return;
    }
    const int64_t b = slot / p.bs;
    const int o = (int)(slot - b * p.bs);
    for (int c = threadIdx.x; c < p.Hk * nchunk; c += blockDim.x) {
        const int h = c / nchunk, ch = c - h * nchunk;
        Chunk kc, vc;
        if (c == (int)threadIdx.x) {
            kc = k0;
            vc = v0;
        } else {
            load_chunk(c, kc, vc);
        }
        uint16_t* kv = kc.h;
        uint16_t* vv = vc.h;
        const int64_t head = b * p.Hk + h;
        uint8_t* kdst = p.kcache + (((head * nchunk + ch) * p.bs + o) * X) * kvb;
        if constexpr (FP8) {
            float ksc = p.k_scale, vsc = p.v_scale;
            if (p.k_scales != nullptr) {
                // this kv head's scales; one that is not finite and positive is flagged (bit 8)
                ksc = p.k_scales[h];
                vsc = p.v_scales[h];
                if (ch == 0 && tok == 0 && !(ksc > 0.f && ksc < INFINITY && vsc > 0.f && vsc < INFINITY))
                    atomicOr(&g_cache_errors, 256u);
            }
            union { uint4 v; uint16_t h[8]; } kq;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                kq.h[i] = f32x2_to_e4m3x2(__fdiv_rn(to_f32<BF16>(kv[2 * i]), ksc),
                                          __fdiv_rn(to_f32<BF16>(kv[2 * i + 1]), ksc));
            *reinterpret_cast<uint4*>(kdst) = kq.v;
#pragma unroll
            for (int i = 0; i < X; i += 2) {
                const uint16_t q = f32x2_to_e4m3x2(__fdiv_rn(to_f32<BF16>(vv[i]), vsc),
                                                   __fdiv_rn(to_f32<BF16>(vv[i + 1]), vsc));
                const int64_t r = (head * p.D + ch * X + i) * p.bs + o;
                p.vcache[r] = (uint8_t)(q & 0xff);
                p.vcache[r + p.bs] = (uint8_t)(q >> 8);
            }
        } else {
            *reinterpret_cast<uint4*>(kdst) = kc.v[0];
            uint16_t* vdst = reinterpret_cast<uint16_t*>(p.vcache);
#pragma unroll
            for (int i = 0; i < X; ++i) vdst[(head * p.D + ch * X + i) * p.bs + o] = vv[i];
        }
    }
}

}  // namespace pa

using namespace pa;

cudaError_t pa::read_cache_errors(unsigned int* v, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_cache_errors, sizeof(*v));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_cache_errors, &z, sizeof(z));
}

static pa_status cache_impl(const void* key, const void* value, int64_t key_stride_t, int64_t value_stride_t,
                            void* key_cache, void* value_cache, const int64_t* slot_mapping, int num_tokens,
                            int num_kv_heads, int head_size, int block_size, int num_blocks, pa_dtype src_dtype,
                            pa_kv_cache_dtype kv_cache_dtype, float k_scale, float v_scale, const float* k_scales,
                            const float* v_scales, cudaStream_t stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (src_dtype != PA_DT_F16 && src_dtype != PA_DT_BF16) return PA_ERR_UNSUPPORTED;
    if (kv_cache_dtype != PA_KV_AUTO && kv_cache_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
    switch (head_size) {
        case 64: case 80: case 96: case 112: case 120: case 128: case 192: case 256: break;
        default: return PA_ERR_UNSUPPORTED;
    }
    const bool fp8 = kv_cache_dtype == PA_KV_FP8_E4M3;
    const int x = fp8 ? 16 : 8;
    if (head_size % x) return PA_ERR_INVALID_ARG;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale)) return PA_ERR_INVALID_ARG;
    if ((k_scales == nullptr) != (v_scales == nullptr) || (reinterpret_cast<uintptr_t>(k_scales) & 3) ||
        (reinterpret_cast<uintptr_t>(v_scales) & 3))
        return PA_ERR_INVALID_ARG;
    if (key_stride_t < (int64_t)num_kv_heads * head_size || value_stride_t < (int64_t)num_kv_heads * head_size)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(key_cache) & 15) || (reinterpret_cast<uintptr_t>(value_cache) & 15) ||
        (reinterpret_cast<uintptr_t>(key) & 1) || (reinterpret_cast<uintptr_t>(value) & 1) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7))
        return PA_ERR_INVALID_ARG;
    CacheParams p;
    p.key = (const uint16_t*)key;
    p.value = (const uint16_t*)value;
    p.kstride = key_stride_t;
    p.vstride = value_stride_t;
    p.kcache = (uint8_t*)key_cache;
    p.vcache = (uint8_t*)value_cache;
    p.slots = slot_mapping;
    p.Hk = num_kv_heads;
    p.D = head_size;
    p.bs = block_size;
    p.num_blocks = num_blocks;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_scales = k_scales;
    p.v_scales = v_scales;
    p.vec = ((reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value)) & 15) == 0 &&
            (key_stride_t % 8) == 0 && (value_stride_t % 8) == 0;
    const bool bf16 = src_dtype == PA_DT_BF16;
    void (*fn)(const CacheParams) = fp8 ? (bf16 ? pa_cache_write_kernel<true, true> : pa_cache_write_kernel<true, false>)
                                        : (bf16 ? pa_cache_write_kernel<false, true> : pa_cache_write_kernel<false, false>);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_tokens, 1, 1);
    // one thread per (kv head, x-element chunk) of a token, so one pass covers the token
    // (every load of the CTA in one round trip); at most 512 threads
    int threads = ((num_kv_heads * (head_size / x) + 31) / 32) * 32;
    threads = threads > 512 ? 512 : threads;
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fn, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

extern "C" pa_status pa_reshape_and_cache(const void* key, const void* value, int64_t key_stride_t,
                                          int64_t value_stride_t, void* key_cache, void* value_cache,
                                          const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                          int head_size, int block_size, int num_blocks,
                                          pa_dtype src_dtype, pa_kv_cache_dtype kv_cache_dtype,
                                          float k_scale, float v_scale, cudaStream_t stream) {
    return cache_impl(key, value, key_stride_t, value_stride_t, key_cache, value_cache, slot_mapping, num_tokens,
                      num_kv_heads, head_size, block_size, num_blocks, src_dtype, kv_cache_dtype, k_scale, v_scale,
                      nullptr, nullptr, stream);
}

extern "C" pa_status pa_reshape_and_cache_head_scales(const void* key, const void* value, int64_t key_stride_t,
                                                      int64_t value_stride_t, void* key_cache, void* value_cache,
                                                      const int64_t* slot_mapping, int num_tokens,
                                                      int num_kv_heads, int head_size, int block_size,
                                                      int num_blocks, pa_dtype src_dtype,
                                                      pa_kv_cache_dtype kv_cache_dtype, const float* k_scales,
                                                      const float* v_scales, cudaStream_t stream) {
    if (k_scales == nullptr || v_scales == nullptr) return PA_ERR_INVALID_ARG;
    return cache_impl(key, value, key_stride_t, value_stride_t, key_cache, value_cache, slot_mapping, num_tokens,
                      num_kv_heads, head_size, block_size, num_blocks, src_dtype, kv_cache_dtype, 1.f, 1.f,
                      k_scales, v_scales, stream);
}
