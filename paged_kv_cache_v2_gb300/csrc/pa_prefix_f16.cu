// pa_prefix_f16.cu -- chunked-prefix attention kernels for f16 queries and caches, one per
// supported head size (a translation unit per dtype so the two compile in parallel).
#include "pa_prefix_m256.cuh"

namespace pa {
template PrefixFn prefix_select<false>(int d);
template cudaError_t prefix_read_errors<false>(unsigned int* v, bool reset);
template cudaError_t launch_prefix_combine<false>(const PrefixParams& p, int d, dim3 grid, cudaStream_t stream);
template int prefix_tile_rows<false>(int d);
}  // namespace pa
