// pa_phase1_bs8.cu -- phase-1 decode kernels for block size 8 (one translation unit per
// block size keeps the build parallel).
#include "pa_phase1.cuh"

namespace pa {
template Phase1Fn phase1_select<8>(bool bf16, bool fp8, int d);
template cudaError_t phase1_read_errors<8>(unsigned int* v, bool reset);
}  // namespace pa
