/*
 * pdattn — one decode step of grouped-query attention over a paged KV cache,
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation is the `decode` body of GroupedQueryAttention on the Llama
 * example page ("src/attention.linnet": rope on q and k at pos, write_at of k
 * and v, attention over positions <= pos with scale rsqrt(f32(head dim)),
 * each kv head shared by Heads / KvHeads query heads), addressed through a
 * page table as the paged entries on the llama-3.1-8b-instruct architecture
 * page state it (`decode_paged(…, positions: Tensor[Rows; i32],
 * table: Tensor[Rows, Pages; i32])`, `PageSize: Dim = 64`), with the optional
 * sliding window of the gpt-oss-20b architecture page (`window: i32`).
 *
 * Layouts (all row-major, contiguous, DEVICE pointers unless stated):
 *   q, q_out, out     [rows, heads, head_dim]        element type T
 *   k_new, v_new      [rows, kv_heads, head_dim]     T
 *   positions         [rows]                         int32, pos of each row's new token
 *   table             [rows, pages_per_row]          int32 page ids into the pools
 *   k_pool, v_pool    [num_pages, kv_heads, 64, head_dim]  T
 *   rope cos / sin    [rope_len, head_dim]           T (from pdattn_rope_tables)
 * Row r's position t lives in pool page table[r, t / 64] at offset t % 64.
 * T is bf16 or f32 (pdattn_dtype).  head_dim is 64 or 128, page_size 64,
 * heads / kv_heads <= 8.  Pointers to T data must be 16-byte aligned.
 *
 * Pages: a step writes each row's new k and v into that row's last visible
 * page (table[r, pos / 64]); the attention may read a row's earlier pages
 * while those writes are still in flight.  So a page that some row writes
 * in a call must not also be an earlier page of another row in that call:
 * rows may share only pages that no row of the call writes (full prefix
 * pages), as a paged cache lays them out.
 *
 * Ownership: the caller allocates and owns every buffer, including the
 * workspace; the library allocates no device memory, keeps no per-call state
 * and frees nothing.  It caches only per-device properties.
 *
 * Errors: every call validates its arguments on the host and returns
 * PDATTN_EINVAL / PDATTN_EUNSUPPORTED before launching anything; launch
 * failures return PDATTN_ECUDA.  Calls are asynchronous on `stream`.  Bad
 * data found on the device (a position outside the table or the rope table,
 * a page id outside the pool, a wait that ran past its time limit) is
 * recorded in the workspace's status word; the affected rows are skipped and
 * their outputs are left unspecified.  pdattn_check_status() reports and
 * clears it.  pdattn_last_error() gives a message for the calling thread's
 * last failure.
 */
#ifndef PDATTN_H
#define PDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* pdattn_stream;

typedef enum {
    PDATTN_OK = 0,
    PDATTN_EINVAL = 1,        /* bad argument (host check) */
    PDATTN_EUNSUPPORTED = 2,  /* shape or type this build does not handle */
    PDATTN_ECUDA = 3,         /* a CUDA call failed */
    PDATTN_EBADPAGE = 4,      /* device: page id outside [0, num_pages) */
    PDATTN_ETIMEOUT = 5,      /* device: a bounded wait ran out */
    PDATTN_EBADPOS = 6        /* device: position outside the table or the rope table */
} pdattn_status;

typedef enum { PDATTN_BF16 = 0, PDATTN_F32 = 1 } pdattn_dtype;

typedef struct {
    int32_t rows;           /* Rows; 0 makes every call a no-op */
    int32_t heads;          /* Heads (query heads) */
    int32_t kv_heads;       /* KvHeads; heads % kv_heads == 0 */
    int32_t head_dim;       /* D = H / Heads: 64 or 128 */
    int32_t page_size;      /* PageSize: must be 64 */
    int32_t pages_per_row;  /* Pages: row stride of the table */
    int32_t num_pages;      /* pages in each pool */
    int32_t dtype;          /* pdattn_dtype of q, k, v, pools, tables and out */
    int32_t window;         /* <= 0: attend [0, pos]; W > 0: attend (pos - W, pos] */
    float scale;            /* score scale; 0 selects rsqrt(f32(head_dim)) */
    const void* rope_cos;   /* NULL: no rotation (positions were added upstream) */
    const void* rope_sin;   /* both NULL or both set */
    int32_t rope_len;       /* rows of the rope tables; positions must be below it */
    int32_t chunk_pages;    /* 0: the planner picks pages per split; else fixed */
    const void* sinks;      /* NULL, or [heads] of T: one attention-sink logit per query head
                               (gpt-oss-20b page, SinkAttention `param sinks`), read as an
                               extra softmax logit that carries no value */
} pdattn_params;

/*
 * Bytes of workspace the calls below need for these parameters on the
 * current device.  The workspace must be zero-filled once before first use;
 * the calls leave it reusable.  Calls that share a workspace must be
 * ordered (same stream or synchronised).
 */
size_t pdattn_workspace_size(const pdattn_params* p);

/*
 * Rotary tables (Llama example page, "src/rope.linnet", `tables`):
 * inv_freq[i] = exp(-(f32(i) * 2 / f32(D)) * log(theta)) in f32,
 * angle[s, i] = f32(s) * inv_freq[i], full = concat(angle, angle),
 * cos_out = cast<T>(cos(full)), sin_out = cast<T>(sin(full)), each
 * [length, head_dim].  cos, sin, exp and log are the correctly rounded f32
 * values (computed in double and rounded).  Build once per model.
 */
pdattn_status pdattn_rope_tables(float theta, int32_t head_dim, int32_t length, int32_t dtype,
                                 void* cos_out, void* sin_out, pdattn_stream stream);

/*
 * RoPE and cache write (Llama example page, "src/attention.linnet",
 * `decode`: rope on q and k, `write_at(cache, k, pos)`), paged: for each
 * row, q_out[r] = rope(q[r]) and the pool slot (table[r, pos / 64],
 * pos % 64) of every kv head receives rope(k_new[r]) and v_new[r].
 * rope(x) = x * cos[pos] + rotate_half(x) * sin[pos] with rotate_half(x) =
 * concat(-x[D/2:], x[:D/2]): f32 products, one f32 add, one rounding to T.
 * Without rope tables q_out is a copy of q and k_new is written as is.
 * q_out may alias q.  Writes are bit-exact copies of these values.
 */
pdattn_status pdattn_rope_write_kv(const pdattn_params* p, const void* q, const void* k_new,
                                   const void* v_new, const int32_t* positions,
                                   const int32_t* table, void* q_out, void* k_pool, void* v_pool,
                                   void* workspace, size_t workspace_bytes, pdattn_stream stream);

/*
 * Split plan for these positions: divides every row's visible pages into
 * chunks (pages per chunk from the total work and the SM count, or
 * p->chunk_pages) and orders the (row, kv head, chunk) work items
 * largest first, in the workspace.  pdattn_attend uses it.
 */
pdattn_status pdattn_plan(const pdattn_params* p, const int32_t* positions, void* workspace,
                          size_t workspace_bytes, pdattn_stream stream);

/*
 * Attention of already-rotated queries over the pools, which must already
 * hold position pos of every row (Llama example page, `decode`: mask
 * seen[s] = s <= pos, `grouped_attention(q, cache_k, cache_v,
 * rsqrt(f32(D)), seen)`), following the plan last made in this workspace
 * for the same positions: out[r, h] = sum_t softmax_t(scale * q[r, h] .
 * K[t, h / g]) V[t, h / g] over t in [lo, pos], fp32 online softmax,
 * split chunks merged on the device, result rounded to T.  With sinks,
 * the softmax denominator also holds exp(sinks[h]) (the sink is not scaled).
 */
pdattn_status pdattn_attend(const pdattn_params* p, const void* q_rot, const int32_t* positions,
                            const int32_t* table, const void* k_pool, const void* v_pool,
                            void* out, void* workspace, size_t workspace_bytes,
                            pdattn_stream stream);

/* pdattn_plan followed by pdattn_attend. */
pdattn_status pdattn_decode(const pdattn_params* p, const void* q_rot, const int32_t* positions,
                            const int32_t* table, const void* k_pool, const void* v_pool,
                            void* out, void* workspace, size_t workspace_bytes,
                            pdattn_stream stream);

/*
 * The whole step: the split plan, RoPE and cache write (rotated q kept in
 * the workspace), then attention; three launches, each a programmatic
 * dependent of the one before, with no host synchronisation.  Equivalent to
 * pdattn_rope_write_kv + pdattn_decode.
 */
pdattn_status pdattn_decode_fused(const pdattn_params* p, const void* q, const void* k_new,
                                  const void* v_new, const int32_t* positions,
                                  const int32_t* table, void* k_pool, void* v_pool, void* out,
                                  void* workspace, size_t workspace_bytes, pdattn_stream stream);

/*
 * One layer of a multi-layer decode call: that layer's inputs, cache and
 * output (device pointers, layouts as in pdattn_decode_fused), its window
 * (<= 0: attend [0, pos]) and its attention sinks (NULL or [heads] of T).
 */
typedef struct {
    const void* q;          /* [rows, heads, head_dim] */
    const void* k_new;      /* [rows, kv_heads, head_dim] */
    const void* v_new;      /* [rows, kv_heads, head_dim] */
    void* k_pool;           /* [num_pages, kv_heads, 64, head_dim] of this layer */
    void* v_pool;
    void* out;              /* [rows, heads, head_dim] */
    int32_t window;
    int32_t reserved;       /* must be 0 */
    const void* sinks;
} pdattn_layer;

/* Layers that one group of launches of pdattn_decode_layers serves. */
#define PDATTN_LAYERS_PER_LAUNCH 32

/*
 * Bytes of workspace pdattn_decode_layers needs for n_layers layers of these
 * parameters (0 if they are invalid); it covers
 * min(n_layers, PDATTN_LAYERS_PER_LAUNCH) layers' rows.
 */
size_t pdattn_layers_workspace_size(const pdattn_params* p, int32_t n_layers);

/*
 * The decode step of several layers at once.  The blocks of the model pages
 * repeat one decoder layer `Layers` times (llama-3.1-8b-instruct page; the
 * gpt-oss-20b page alternates a sliding-window and a full layer in each
 * `LayerPair`), every layer with its own cache under the same page table and
 * positions.  For each layer l the result is that of pdattn_decode_fused
 * with p and layers[l] (its pointers, window and sinks; p->window and
 * p->sinks are not read): rope and cache write at positions[r] through
 * table[r], then attention over that layer's pool.  Up to
 * PDATTN_LAYERS_PER_LAUNCH layers share three launches: one planner lists
 * every layer's work items together, one launch rotates and writes every
 * layer's rows, and one persistent attention launch runs every layer's
 * items, largest first, so short (sliding-window) layers fill in beside long
 * ones.  More layers run as successive groups of launches on the same
 * workspace.  `layers` is a HOST
 * array of n_layers descriptors, read during the call only.  The layers'
 * pools must not overlap one another.  A layer's q, k_new, v_new or out may
 * not alias another layer's.  n_layers == 0 or p->rows == 0 is a no-op.
 * Device errors are reported by pdattn_check_status(workspace).  This is a
 * batching of independent layers: each layer's q must be known when the call
 * is made, so it serves callers that hold several layers' queries at once
 * (several models or requests sharing a step, or layers whose inputs do not
 * depend on one another), not the layer-after-layer dependency of one
 * forward pass.
 */
pdattn_status pdattn_decode_layers(const pdattn_params* p, int32_t n_layers, const pdattn_layer* layers,
                                   const int32_t* positions, const int32_t* table, void* workspace,
                                   size_t workspace_bytes, pdattn_stream stream);

/*
 * pdattn_decode_fused without a workspace, for callers that cannot allocate
 * device memory (an allocator that is frozen once serving starts, a plugin
 * inside a program that owns all device memory, a C caller with no CUDA
 * allocator).  The paper has no counterpart: this is a packaging of the same
 * step.  Its scratch is one fixed 16 MiB array compiled into the library,
 * which every GPU that loads the library keeps until the process exits.
 * Parameters whose workspace (pdattn_workspace_size) exceeds 16 MiB are
 * rejected with PDATTN_EINVAL before any launch; the Llama-3.1-8B shape at
 * 256 rows needs about 10.6 MiB.  The first call on each device (with that
 * device current) looks up the array's device address, which issues no work
 * on any stream; make that first call before capturing any stream.  All calls
 * on a device share the one array: calls whose work overlaps on the GPU
 * (other streams, other threads) race and must be serialised by the caller.
 * No device-side error is reported: bad positions or page ids (those rows
 * are skipped), a device wait that ran past its limit and a rejected plan
 * all leave the call's return value PDATTN_OK, with the outputs of the
 * affected rows (after a timeout or a rejected plan, possibly of any row)
 * unwritten.  Check the inputs beforehand, or use pdattn_decode_fused and
 * pdattn_check_status where such reports matter.
 */
pdattn_status pdattn_decode_fused_noalloc(const pdattn_params* p, const void* q, const void* k_new,
                                          const void* v_new, const int32_t* positions,
                                          const int32_t* table, void* k_pool, void* v_pool,
                                          void* out, pdattn_stream stream);

/*
 * Bytes of workspace pdattn_prefill_paged needs for n_tokens packed tokens
 * (256-byte aligned; 0 if the parameters are invalid).
 */
size_t pdattn_prefill_workspace_size(const pdattn_params* p, int32_t n_tokens);

/*
 * Paged prefill of packed prompt tokens: `prefill_paged(…, positions, rows,
 * slots, table)` of the llama-3.1-8b-instruct architecture page, the prefill
 * half of its `step_paged`.  For each of the n_tokens tokens i:
 *   q_rot[i] = rope(q[i], positions[i]); the rotated k_new[i] and v_new[i]
 *   are written at pool slot slots[i] (page slots[i] / 64, offset
 *   slots[i] % 64).  Every token is written before any is read; then
 *   out[i, h] = sum_t softmax_t(scale * q_rot[i, h] . K[t, h / g]) V[t, h / g]
 *   over the positions t in [lo_i, positions[i]] of table row rows[i]
 *   (lo_i = 0, or positions[i] - window + 1 with a window), read through
 *   table[rows[i], t / 64], with the sinks of p as in pdattn_attend.
 * Layouts: q, out [n_tokens, heads, head_dim]; k_new, v_new [n_tokens,
 * kv_heads, head_dim]; positions, rows, slots [n_tokens] int32; table
 * [p->rows, pages_per_row].  p->rows is the number of table rows.  Tokens
 * of one row should be contiguous (consecutive positions give the best
 * tiles) but need not be.  The attention runs on the tensor cores and needs
 * dtype bf16 (PDATTN_EUNSUPPORTED otherwise).  The workspace
 * (pdattn_prefill_workspace_size) holds the rotated queries and the tile
 * list; a row index outside [0, rows) or a bad position is recorded as
 * PDATTN_EBADPOS and the call writes no output; a slot outside the pools
 * is recorded as PDATTN_EBADPAGE and that token's k / v are not written.
 * Cache slots outside a tile's key range never reach an output, whatever
 * they hold (non-finite values included).
 */
pdattn_status pdattn_prefill_paged(const pdattn_params* p, int32_t n_tokens, const void* q,
                                   const void* k_new, const void* v_new, const int32_t* positions,
                                   const int32_t* rows, const int32_t* slots, const int32_t* table,
                                   void* k_pool, void* v_pool, void* out, void* workspace,
                                   size_t workspace_bytes, pdattn_stream stream);

/*
 * The attention half of pdattn_prefill_paged alone: re-runs it over the
 * rotated queries and the tile list that the last pdattn_prefill_paged call
 * on this workspace left there, with the same parameters, n_tokens,
 * positions and table, against the pools as they are now.  For callers that
 * write the cache once and attend again (and for timing the attention).
 */
pdattn_status pdattn_prefill_attend(const pdattn_params* p, int32_t n_tokens, const int32_t* positions,
                                    const int32_t* table, const void* k_pool, const void* v_pool,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    pdattn_stream stream);

/*
 * Bytes of workspace pdattn_packed needs for n_tokens packed tokens (0 if the
 * parameters are invalid).
 */
size_t pdattn_packed_workspace_size(const pdattn_params* p, int32_t n_tokens);

/*
 * Packed sequences, no cache: `packed(x, positions, segments)` of the Llama
 * example page ("src/attention.linnet").  Several sequences lie in one row
 * of n_tokens tokens; token i sits at positions[i] of sequence segments[i].
 * q_rot[i] = rope(q[i], positions[i]) and k_rot[i] = rope(k[i],
 * positions[i]) (kept in the workspace); then
 *   out[i, h] = sum_j softmax_j(scale * q_rot[i, h] . k_rot[j, h / g]) v[j, h / g]
 * over the tokens j with segments[j] == segments[i] and positions[j] <=
 * positions[i] (the pages' mask `own`), and with a window W > 0 also
 * positions[j] > positions[i] - W; sinks as in pdattn_attend.
 * Layouts: q, out [n_tokens, heads, head_dim]; k, v [n_tokens, kv_heads,
 * head_dim]; positions, segments [n_tokens] int32.  Of p only heads,
 * kv_heads, head_dim, dtype (bf16), window, scale, the rope tables and
 * sinks are read.  Fast when every sequence is one run of consecutive
 * tokens with strictly increasing positions (as packing lays them out);
 * any other layout is handled exactly but visits the whole pack per tile.
 * A negative position or one past the rope table is recorded as
 * PDATTN_EBADPOS and no output is written.  The keys and values of one
 * sequence never reach another sequence's outputs, non-finite ones
 * included.
 */
pdattn_status pdattn_packed(const pdattn_params* p, int32_t n_tokens, const void* q, const void* k,
                            const void* v, const int32_t* positions, const int32_t* segments,
                            void* out, void* workspace, size_t workspace_bytes, pdattn_stream stream);

/*
 * The attention half of pdattn_packed alone: re-runs it over the rotated q
 * and k and the tile list that the last pdattn_packed call on this
 * workspace left there, with the same parameters, n_tokens, v and
 * positions (for timing the attention, or attending again).
 */
pdattn_status pdattn_packed_attend(const pdattn_params* p, int32_t n_tokens, const void* v,
                                   const int32_t* positions, void* out, void* workspace,
                                   size_t workspace_bytes, pdattn_stream stream);

/*
 * Synchronises `stream`, reads the workspace's device status word, clears
 * it and returns the first error it recorded (PDATTN_OK if none).  After
 * PDATTN_ETIMEOUT from decode attention the workspace's plan is withdrawn:
 * pdattn_attend on it is refused (PDATTN_EINVAL) until pdattn_plan,
 * pdattn_decode or pdattn_decode_fused plans again.
 */
pdattn_status pdattn_check_status(void* workspace, pdattn_stream stream);

/* Message for the calling thread's last failed call ("" if none). */
const char* pdattn_last_error(void);

/* Number of kernel launches the last successful call on this thread made. */
int32_t pdattn_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PDATTN_H */
