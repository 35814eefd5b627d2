// pa_phase1_bs16_fp8_pair.cu -- phase-1 decode kernels for block size 16, fp8 caches, per-tensor scales,
// the cross-warp value reduction in pairs of warps (one translation unit per block size, cache type and
// form keeps the build parallel).
#include "pa_phase1.cuh"

namespace pa {
template Phase1Fn phase1_select<16, 1, 3>(bool bf16, int d);
template cudaError_t phase1_read_errors<16, 1, 3>(unsigned int* v, bool reset);
}  // namespace pa
