// pa_prefix_bf16.cu -- chunked-prefix attention kernels for bf16 queries and caches, one per
// supported head size (a translation unit per dtype so the two compile in parallel).
#include "pa_prefix_m256.cuh"

namespace pa {
template PrefixFn prefix_select<true>(int d);
template cudaError_t prefix_read_errors<true>(unsigned int* v, bool reset);
template cudaError_t launch_prefix_combine<true>(const PrefixParams& p, int d, dim3 grid, cudaStream_t stream);
template int prefix_tile_rows<true>(int d);
}  // namespace pa
