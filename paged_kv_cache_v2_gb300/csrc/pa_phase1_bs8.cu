// pa_phase1_bs8.cu -- phase-1 decode kernels for block size 8 and fp16/bf16 caches (one
// translation unit per block size and cache type keeps the build parallel).
#include "pa_phase1.cuh"

namespace pa {
template Phase1Fn phase1_select<8, 2>(bool bf16, int d, bool head_scales);
template cudaError_t phase1_read_errors<8, 2>(unsigned int* v, bool reset);
}  // namespace pa
