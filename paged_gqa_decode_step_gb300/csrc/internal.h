// Kernel argument blocks and launchers shared between the .cu files.
#pragma once

#include "common.cuh"

namespace pdattn {

// Layers one multi-layer decode launch serves (its per-layer pointers and
// tensor maps travel as kernel parameters).
constexpr int kMaxLayers = 32;

// Parameter block of the single-layer launches: nothing per layer.
struct NoLayers {};

// Per-layer inputs of a multi-layer prep launch.  Row v of the launch is row
// v % layer_rows of layer v / layer_rows.
struct PrepLayers {
    const void* q[kMaxLayers];
    const void* k_new[kMaxLayers];
    const void* v_new[kMaxLayers];
    void* k_pool[kMaxLayers];
    void* v_pool[kMaxLayers];
    int window[kMaxLayers];
};

// Per-layer pools (as TMA maps), outputs and sinks of a multi-layer
// attention launch.
struct AttendLayers {
    CUtensorMap k[kMaxLayers];
    CUtensorMap v[kMaxLayers];
    void* out[kMaxLayers];
    const void* sinks[kMaxLayers];
    int window[kMaxLayers];
};

struct PrepArgs {
    int rows, heads, kv_heads, head_dim, pages_per_row, num_pages, window, rope_len;
    int layer_rows;         // multi-layer launches: rows per layer (rows = layers x layer_rows)
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
    int do_plan;            // 1: a planner launch builds the split plan first
    int grid_attend;        // persistent CTAs of the attention launch
    int chunk_pages;        // 0: planner's choice
    char* ws;
    WsLayout L;
};

struct AttendArgs {
    int rows, heads, kv_heads, group, head_dim, pages_per_row, num_pages;
    int layer_rows, n_layers;   // multi-layer launches: rows per layer, layers
    int window, chunk_pages;    // as given to the planner (first-wave items are derived from them)
    float scale_log2;       // score scale times log2(e)
    const void* q;          // rotated queries [rows, heads, D]
    const int* positions;   // [rows] (per layer in a multi-layer launch)
    const int* table;
    const void* sinks;      // nullptr, or [heads] of T
    void* out;
    char* ws;
    WsLayout L;
};

struct PrefillPrepArgs {
    int n_tokens, rows, heads, kv_heads, head_dim, pages_per_row, num_pages, window, rope_len;
    int tile_tokens;        // tokens per tile: two halves of 128 / (heads / kv_heads)
    const void* q;          // [n_tokens, heads, D]
    const void* k_new;      // [n_tokens, kv_heads, D]
    const void* v_new;
    const int* positions;   // [n_tokens]
    const int* row_of;      // [n_tokens] table row of each token (packed: segment id)
    const int* slots;       // [n_tokens] page * 64 + offset (packed: unused)
    const void* rope_cos;   // nullptr: copy without rotation
    const void* rope_sin;
    void* k_pool;
    void* v_pool;
    char* ws;
    PfLayout L;
};

struct PrefillArgs {
    int n_tokens, heads, kv_heads, group, tile_tokens, head_dim, pages_per_row, num_pages, window;
    int packed;             // 1: packed sequences (keys are the pack's 64-token blocks)
    float scale_log2;
    const int* positions;
    const int* table;
    const void* sinks;      // nullptr, or [heads] of bf16
    void* out;              // [n_tokens, heads, D]
    char* ws;
    PfLayout L;
};

cudaError_t launch_rope_tables(float theta, int D, int S, int dtype, void* cos_out, void* sin_out,
                               cudaStream_t stream);
// The split planner (one block, if a.do_plan), then the rope + cache write of
// a.rope_blocks rows (a programmatic dependent of the planner); *launches
// gets the number of launches made.
cudaError_t launch_prep(const PrepArgs& a, int dtype, cudaStream_t stream, int* launches);
// Multi-layer prep: rope + write of every layer's rows, one plan over all.
cudaError_t launch_prep_layers(const PrepArgs& a, const PrepLayers& lay, int dtype, cudaStream_t stream,
                               int* launches);
// Sets the kernel's shared-memory limit (once per device) and launches.
cudaError_t launch_attend(const AttendArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                          int dtype, int grid, bool programmatic, cudaStream_t stream);
// Multi-layer attention: one persistent launch over every layer's items.
cudaError_t launch_attend_layers(const AttendArgs& a, const AttendLayers& lay, int dtype, int grid,
                                 cudaStream_t stream);
size_t attend_smem_bytes(int dtype, int head_dim);
// The tile list (one block), then the rope + write of every token at its
// slot (programmatic launch that ends after the tile list): two launches.
cudaError_t launch_prefill_prep(const PrefillPrepArgs& a, int dtype, cudaStream_t stream);
// Tensor-core attention of the tiles (bf16, head dim 64 or 128).
cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, int grid, cudaStream_t stream);
size_t prefill_smem_bytes(int head_dim);
// Packed sequences: tile list and block summaries (one block), then rope of
// q and k into the workspace (programmatic launch ending after the plan).
cudaError_t launch_packed_prep(const PrefillPrepArgs& a, int dtype, cudaStream_t stream);
// Tensor-core attention of the packed tiles: k_map over the rotated keys and
// v_map over v, both [n, kv_heads, D] as 3-D tensors.
cudaError_t launch_packed(const PrefillArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                          const CUtensorMap& v_map, int grid, cudaStream_t stream);

}  // namespace pdattn
