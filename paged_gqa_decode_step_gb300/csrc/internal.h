// Kernel argument blocks and launchers shared between the .cu files.
#pragma once

#include "common.cuh"

namespace pdattn {

struct PrepArgs {
    int rows, heads, kv_heads, head_dim, pages_per_row, num_pages, window, rope_len;
    const void* q;
    const void* k_new;
    const void* v_new;
    const int* positions;
    const int* table;
    const void* rope_cos;   // nullptr: copy without rotation
    const void* rope_sin;
    void* q_out;
    void* k_pool;
    void* v_pool;
    int rope_blocks;        // rows to rotate and write (0: none)
    int do_plan;            // 1: the last block builds the split plan
    int grid_attend;        // persistent CTAs of the attention launch
    int chunk_pages;        // 0: planner's choice
    char* ws;
    WsLayout L;
};

struct AttendArgs {
    int rows, heads, kv_heads, group, head_dim, pages_per_row, num_pages;
    float scale_log2;       // score scale times log2(e)
    const void* q;          // rotated queries [rows, heads, D]
    const int* table;
    const void* sinks;      // nullptr, or [heads] of T
    void* out;
    char* ws;
    WsLayout L;
};

cudaError_t launch_rope_tables(float theta, int D, int S, int dtype, void* cos_out, void* sin_out,
                               cudaStream_t stream);
cudaError_t launch_prep(const PrepArgs& a, int dtype, cudaStream_t stream);
// Sets the kernel's shared-memory limit (once per device) and launches.
cudaError_t launch_attend(const AttendArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                          int dtype, int grid, bool programmatic, cudaStream_t stream);
size_t attend_smem_bytes(int dtype, int head_dim);

}  // namespace pdattn
