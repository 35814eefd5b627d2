// pa_phase1_bs32_ord.cu -- phase-1 decode kernels for block size 32, fp16/bf16 caches, per-tensor scales, ordered grid (one
// translation unit per block size, cache type and form keeps the build parallel).
#include "pa_phase1.cuh"

namespace pa {
template Phase1Fn phase1_select<32, 2, 2>(bool bf16, int d);
template cudaError_t phase1_read_errors<32, 2, 2>(unsigned int* v, bool reset);
}  // namespace pa
