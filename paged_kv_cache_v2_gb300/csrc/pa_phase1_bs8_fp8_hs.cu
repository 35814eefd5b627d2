// pa_phase1_bs8_fp8_hs.cu -- phase-1 decode kernels for block size 8, fp8 e4m3 caches, per-kv-head scales (one
// translation unit per block size, cache type and form keeps the build parallel).
#include "pa_phase1.cuh"

namespace pa {
template Phase1Fn phase1_select<8, 1, 1>(bool bf16, int d);
template cudaError_t phase1_read_errors<8, 1, 1>(unsigned int* v, bool reset);
}  // namespace pa
