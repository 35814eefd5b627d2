// pa_internal.h -- host-side plumbing shared by the library's translation units.
#pragma once

#include <stdint.h>

#include "pa_v2.h"

namespace pa {

struct DecodeArgs {
    void* output;
    float* exp_sums;
    float* max_logits;
    void* tmp_output;
    const void* query;
    const void* key_cache;
    const void* value_cache;
    int num_seqs, num_heads, num_kv_heads, head_size;
    float scale;
    const int32_t* block_tables;
    int max_blocks_per_seq, num_blocks;
    const int32_t* seq_lens;
    int block_size, max_seq_len, max_num_partitions;
    const float* alibi_slopes;
    pa_dtype q_dtype;
    pa_kv_cache_dtype kv_cache_dtype;
    pa_dtype tmp_dtype;
    float k_scale, v_scale;
    // one scale per kv head (device, [num_kv_heads]) in place of k_scale / v_scale, or null
    const float* k_scales = nullptr;
    const float* v_scales = nullptr;
    cudaStream_t stream;
    // fused cache append (pa_v2_decode_append): the newest token's key/value rows, or null
    const void* new_key = nullptr;
    const void* new_value = nullptr;
    int64_t new_key_stride = 0, new_value_stride = 0;  // elements between sequences' rows
    // tmp_output is the caller's scratch (its contents after the call are unspecified), so
    // CTAs that stream several partitions may fold them into one row
    bool tmp_scratch = false;
    // caller scratch of num_seqs ints for a grid order (most partitions first), or null; used
    // where CTAs stride over several partitions each
    int32_t* order = nullptr;
};

// Argument checks shared by the decode entry points (no device access).
pa_status validate_decode(const DecodeArgs& a);
// Enqueue phase 1 (+ phase 2) with the given workspace.  With `counters` (zeroed arrival
// counters, one per (sequence, kv head, head group)) the combine runs inside phase 1 when
// the step's shape allows it, and phase 2 is not launched.
pa_status launch_decode(const DecodeArgs& a, float* exp_sums, float* max_logits, void* tmp_out,
                        uint32_t* counters = nullptr);
// Enqueue the grid-order kernel: order[0..S) = the sequences by decreasing partition count.
pa_status launch_order(const int32_t* seq_lens, int S, int32_t* order, cudaStream_t stream);
// Arrival counters the fused combine needs for a step of this shape.
int64_t decode_num_counters(int num_seqs, int num_heads, int num_kv_heads);
// Read (and optionally clear) each translation unit's device error word on the current device.
cudaError_t read_decode_errors(unsigned int* v, bool reset);
cudaError_t read_cache_errors(unsigned int* v, bool reset);
cudaError_t read_block_errors(unsigned int* v, bool reset);
// The events pa_v2_set_timing_events installed (both null when none).
void timing_events(cudaEvent_t* begin, cudaEvent_t* end);

}  // namespace pa
