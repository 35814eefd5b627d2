// pa_phase1_bs32_fp8.cu -- phase-1 decode kernels for block size 32 and fp8 e4m3 caches (one
// translation unit per block size and cache type keeps the build parallel).
#include "pa_phase1.cuh"

namespace pa {
template Phase1Fn phase1_select<32, 1>(bool bf16, int d, bool head_scales);
template cudaError_t phase1_read_errors<32, 1>(unsigned int* v, bool reset);
}  // namespace pa
