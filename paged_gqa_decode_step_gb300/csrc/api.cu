// extern "C" entry points of libpdattn: host-side validation, TMA
// descriptors and launches.  See include/pdattn.h for the contract.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/pdattn.h"
#include "internal.h"

using namespace pdattn;

namespace {

thread_local std::string g_error;
thread_local int g_launches = 0;

pdattn_status fail(pdattn_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_error = buf;
    return s;
}

pdattn_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PDATTN_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// SM count per device, read once.
int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Pool [num_pages, kv_heads, 64, D] viewed as a 2-D tensor of
// num_pages * kv_heads * 64 rows by D columns; boxes of 64 rows x 128 bytes,
// 128-byte swizzled.
pdattn_status make_pool_map(CUtensorMap* map, const void* pool, const pdattn_params* p) {
    auto fn = encode_fn();
    if (!fn) return fail(PDATTN_ECUDA, "cuTensorMapEncodeTiled is not available");
    const int elem = p->dtype == PDATTN_BF16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)p->head_dim, (cuuint64_t)p->num_pages * p->kv_heads * kPageSize};
    cuuint64_t strides[1] = {(cuuint64_t)p->head_dim * elem};
    cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)kPageSize};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, p->dtype == PDATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    2, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PDATTN_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PDATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

pdattn_status check_params(const pdattn_params* p) {
    if (!p) return fail(PDATTN_EINVAL, "params is NULL");
    if (p->rows < 0) return fail(PDATTN_EINVAL, "rows < 0");
    if (p->heads <= 0 || p->kv_heads <= 0 || p->heads % p->kv_heads != 0)
        return fail(PDATTN_EINVAL, "heads (%d) must be a positive multiple of kv_heads (%d)", p->heads, p->kv_heads);
    if (p->head_dim <= 0 || p->head_dim % 2 != 0) return fail(PDATTN_EINVAL, "head_dim must be even and positive");
    if (p->dtype != PDATTN_BF16 && p->dtype != PDATTN_F32) return fail(PDATTN_EINVAL, "unknown dtype %d", p->dtype);
    if (p->pages_per_row <= 0 || p->num_pages <= 0) return fail(PDATTN_EINVAL, "pages_per_row and num_pages must be > 0");
    if ((p->rope_cos == nullptr) != (p->rope_sin == nullptr))
        return fail(PDATTN_EINVAL, "rope_cos and rope_sin must be both set or both NULL");
    if (p->rope_cos && p->rope_len <= 0) return fail(PDATTN_EINVAL, "rope_len must be > 0 with rope tables");
    if (p->rope_cos && (!aligned16(p->rope_cos) || !aligned16(p->rope_sin)))
        return fail(PDATTN_EINVAL, "rope tables must be 16-byte aligned");
    if (p->chunk_pages < 0 || p->chunk_pages > kChunkMax)
        return fail(PDATTN_EINVAL, "chunk_pages must be in [0, %d]", kChunkMax);
    if (!(p->scale >= 0.f)) return fail(PDATTN_EINVAL, "scale must be >= 0 (0 selects rsqrt(head_dim))");
    if (p->page_size != kPageSize) return fail(PDATTN_EUNSUPPORTED, "page_size must be 64");
    if (p->head_dim != 64 && p->head_dim != 128) return fail(PDATTN_EUNSUPPORTED, "head_dim must be 64 or 128");
    if (p->heads / p->kv_heads > kMaxGroup) return fail(PDATTN_EUNSUPPORTED, "heads / kv_heads must be <= 8");
    if (p->kv_heads > 32767) return fail(PDATTN_EUNSUPPORTED, "kv_heads must be < 32768");
    if ((long long)p->num_pages * p->kv_heads * kPageSize >= (1ll << 31))
        return fail(PDATTN_EUNSUPPORTED, "pool too large for 32-bit TMA row coordinates");
    if ((long long)p->pages_per_row * kPageSize >= (1ll << 30)) return fail(PDATTN_EUNSUPPORTED, "pages_per_row too large");
    return PDATTN_OK;
}

int elem_bytes(const pdattn_params* p) { return p->dtype == PDATTN_BF16 ? 2 : 4; }

WsLayout layout_for(const pdattn_params* p, int grid) {
    return ws_layout(p->rows, p->heads, p->kv_heads, p->head_dim, p->pages_per_row, elem_bytes(p),
                     p->chunk_pages, grid);
}

pdattn_status check_ws(const pdattn_params* p, void* ws, size_t bytes, int grid, WsLayout* L) {
    if (!ws) return fail(PDATTN_EINVAL, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return fail(PDATTN_EINVAL, "workspace must be 256-byte aligned");
    *L = layout_for(p, grid);
    if (bytes < L->total)
        return fail(PDATTN_EINVAL, "workspace too small: %zu bytes given, %zu needed", bytes, L->total);
    return PDATTN_OK;
}

PrepArgs prep_args(const pdattn_params* p, const int32_t* positions, const int32_t* table, char* ws,
                   const WsLayout& L, int grid) {
    PrepArgs a = {};
    a.rows = p->rows;
    a.heads = p->heads;
    a.kv_heads = p->kv_heads;
    a.head_dim = p->head_dim;
    a.pages_per_row = p->pages_per_row;
    a.num_pages = p->num_pages;
    a.window = p->window;
    a.rope_len = p->rope_len;
    a.positions = positions;
    a.table = table;
    a.rope_cos = p->rope_cos;
    a.rope_sin = p->rope_sin;
    a.grid_attend = grid;
    a.chunk_pages = p->chunk_pages;
    a.ws = ws;
    a.L = L;
    return a;
}

float scale_log2(const pdattn_params* p) {
    const double s = p->scale > 0.f ? (double)p->scale : (double)(float)(1.0 / std::sqrt((double)p->head_dim));
    return (float)(s * 1.4426950408889634);
}

pdattn_status attend_impl(const pdattn_params* p, const void* q_rot, const int32_t* positions, const int32_t* table,
                          const void* k_pool, const void* v_pool, void* out, char* ws,
                          const WsLayout& L, int grid, bool programmatic, cudaStream_t stream) {
    CUtensorMap km, vm;
    pdattn_status s = make_pool_map(&km, k_pool, p);
    if (s != PDATTN_OK) return s;
    s = make_pool_map(&vm, v_pool, p);
    if (s != PDATTN_OK) return s;
    AttendArgs a = {};
    a.rows = p->rows;
    a.heads = p->heads;
    a.kv_heads = p->kv_heads;
    a.group = p->heads / p->kv_heads;
    a.head_dim = p->head_dim;
    a.pages_per_row = p->pages_per_row;
    a.num_pages = p->num_pages;
    a.window = p->window;
    a.chunk_pages = p->chunk_pages;
    a.scale_log2 = scale_log2(p);
    a.q = q_rot;
    a.positions = positions;
    a.table = table;
    a.sinks = p->sinks;
    a.out = out;
    a.ws = ws;
    a.L = L;
    cudaError_t e = launch_attend(a, km, vm, p->dtype, grid, programmatic, stream);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    ++g_launches;
    return PDATTN_OK;
}

}  // namespace

extern "C" {

size_t pdattn_workspace_size(const pdattn_params* p) {
    if (check_params(p) != PDATTN_OK) return 0;
    const int grid = sm_count();
    if (grid <= 0) return 0;
    return layout_for(p, grid).total;
}

pdattn_status pdattn_rope_tables(float theta, int32_t head_dim, int32_t length, int32_t dtype, void* cos_out,
                                 void* sin_out, pdattn_stream stream) {
    g_launches = 0;
    if (!(theta > 0.f)) return fail(PDATTN_EINVAL, "theta must be > 0");
    if (head_dim <= 0 || head_dim % 2 != 0) return fail(PDATTN_EINVAL, "head_dim must be even and positive");
    if (length < 0) return fail(PDATTN_EINVAL, "length must be >= 0");
    if (dtype != PDATTN_BF16 && dtype != PDATTN_F32) return fail(PDATTN_EINVAL, "unknown dtype");
    if (length > 0 && (!cos_out || !sin_out)) return fail(PDATTN_EINVAL, "NULL table pointer");
    cudaError_t e = launch_rope_tables(theta, head_dim, length, dtype, cos_out, sin_out, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
    g_launches = length > 0 ? 1 : 0;
    return PDATTN_OK;
}

pdattn_status pdattn_rope_write_kv(const pdattn_params* p, const void* q, const void* k_new, const void* v_new,
                                   const int32_t* positions, const int32_t* table, void* q_out, void* k_pool,
                                   void* v_pool, void* workspace, size_t workspace_bytes, pdattn_stream stream) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (p->rows == 0) return PDATTN_OK;
    if (!q || !k_new || !v_new || !positions || !table || !q_out || !k_pool || !v_pool)
        return fail(PDATTN_EINVAL, "NULL data pointer");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_out) || !aligned16(k_pool) ||
        !aligned16(v_pool))
        return fail(PDATTN_EINVAL, "q, k_new, v_new, q_out and the pools must be 16-byte aligned");
    const int grid = sm_count();
    if (grid <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    WsLayout L;
    s = check_ws(p, workspace, workspace_bytes, grid, &L);
    if (s != PDATTN_OK) return s;
    PrepArgs a = prep_args(p, positions, table, static_cast<char*>(workspace), L, grid);
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.q_out = q_out;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.rope_blocks = p->rows;
    a.do_plan = 0;
    int n = 0;
    cudaError_t e = launch_prep(a, p->dtype, (cudaStream_t)stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "rope/write launch");
    g_launches = n;
    return PDATTN_OK;
}

pdattn_status pdattn_plan(const pdattn_params* p, const int32_t* positions, void* workspace,
                          size_t workspace_bytes, pdattn_stream stream) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (p->rows == 0) return PDATTN_OK;
    if (!positions) return fail(PDATTN_EINVAL, "NULL positions");
    const int grid = sm_count();
    if (grid <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    WsLayout L;
    s = check_ws(p, workspace, workspace_bytes, grid, &L);
    if (s != PDATTN_OK) return s;
    PrepArgs a = prep_args(p, positions, nullptr, static_cast<char*>(workspace), L, grid);
    a.rope_blocks = 0;
    a.do_plan = 1;
    int n = 0;
    cudaError_t e = launch_prep(a, p->dtype, (cudaStream_t)stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "plan launch");
    g_launches = n;
    return PDATTN_OK;
}

static pdattn_status check_attend_ptrs(const void* q, const int32_t* positions, const int32_t* table,
                                       const void* k_pool, const void* v_pool, const void* out) {
    if (!q || !positions || !table || !k_pool || !v_pool || !out) return fail(PDATTN_EINVAL, "NULL data pointer");
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PDATTN_EINVAL, "q, the pools and out must be 16-byte aligned");
    return PDATTN_OK;
}

pdattn_status pdattn_attend(const pdattn_params* p, const void* q_rot, const int32_t* positions, const int32_t* table,
                            const void* k_pool, const void* v_pool, void* out, void* workspace,
                            size_t workspace_bytes, pdattn_stream stream) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (p->rows == 0) return PDATTN_OK;
    s = check_attend_ptrs(q_rot, positions, table, k_pool, v_pool, out);
    if (s != PDATTN_OK) return s;
    const int grid = sm_count();
    if (grid <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    WsLayout L;
    s = check_ws(p, workspace, workspace_bytes, grid, &L);
    if (s != PDATTN_OK) return s;
    return attend_impl(p, q_rot, positions, table, k_pool, v_pool, out, static_cast<char*>(workspace), L, grid, false,
                       (cudaStream_t)stream);
}

pdattn_status pdattn_decode(const pdattn_params* p, const void* q_rot, const int32_t* positions, const int32_t* table,
                            const void* k_pool, const void* v_pool, void* out, void* workspace,
                            size_t workspace_bytes, pdattn_stream stream) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (p->rows == 0) return PDATTN_OK;
    s = check_attend_ptrs(q_rot, positions, table, k_pool, v_pool, out);
    if (s != PDATTN_OK) return s;
    const int grid = sm_count();
    if (grid <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    WsLayout L;
    s = check_ws(p, workspace, workspace_bytes, grid, &L);
    if (s != PDATTN_OK) return s;
    PrepArgs a = prep_args(p, positions, table, static_cast<char*>(workspace), L, grid);
    a.rope_blocks = 0;
    a.do_plan = 1;
    int n = 0;
    cudaError_t e = launch_prep(a, p->dtype, (cudaStream_t)stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "plan launch");
    s = attend_impl(p, q_rot, positions, table, k_pool, v_pool, out, static_cast<char*>(workspace), L, grid, true,
                    (cudaStream_t)stream);
    if (s == PDATTN_OK) g_launches = n + 1;
    return s;
}

pdattn_status pdattn_decode_fused(const pdattn_params* p, const void* q, const void* k_new, const void* v_new,
                                  const int32_t* positions, const int32_t* table, void* k_pool, void* v_pool,
                                  void* out, void* workspace, size_t workspace_bytes, pdattn_stream stream) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (p->rows == 0) return PDATTN_OK;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return fail(PDATTN_EINVAL, "k_new and v_new must be non-NULL and 16-byte aligned");
    s = check_attend_ptrs(q, positions, table, k_pool, v_pool, out);
    if (s != PDATTN_OK) return s;
    const int grid = sm_count();
    if (grid <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    WsLayout L;
    s = check_ws(p, workspace, workspace_bytes, grid, &L);
    if (s != PDATTN_OK) return s;
    char* ws = static_cast<char*>(workspace);
    void* q_rot = ws + L.q_rot;
    PrepArgs a = prep_args(p, positions, table, ws, L, grid);
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.q_out = q_rot;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.rope_blocks = p->rows;
    a.do_plan = 1;
    int n = 0;
    cudaError_t e = launch_prep(a, p->dtype, (cudaStream_t)stream, &n);
    if (e != cudaSuccess) return cuda_fail(e, "plan + rope/write launches");
    s = attend_impl(p, q_rot, positions, table, k_pool, v_pool, out, ws, L, grid, true, (cudaStream_t)stream);
    if (s == PDATTN_OK) g_launches = n + 1;
    return s;
}

// Rows of one multi-layer launch: layers x rows, within the plan's int ranges.
static pdattn_status layers_rows(const pdattn_params* p, int32_t n_layers, int* v_rows) {
    const int lg = n_layers < kMaxLayers ? n_layers : kMaxLayers;
    const long long v = (long long)lg * p->rows;
    if (v * p->kv_heads * (long long)p->pages_per_row >= (1ll << 31) || v * p->heads >= (1ll << 31))
        return fail(PDATTN_EUNSUPPORTED, "layers x rows too large for one launch");
    *v_rows = (int)v;
    return PDATTN_OK;
}

static pdattn_params with_rows(const pdattn_params* p, int rows) {
    pdattn_params q = *p;
    q.rows = rows;
    return q;
}

size_t pdattn_layers_workspace_size(const pdattn_params* p, int32_t n_layers) {
    if (check_params(p) != PDATTN_OK || n_layers < 0) return 0;
    int v = 0;
    if (layers_rows(p, n_layers > 0 ? n_layers : 1, &v) != PDATTN_OK) return 0;
    const int grid = sm_count();
    if (grid <= 0) return 0;
    const pdattn_params pv = with_rows(p, v);
    return layout_for(&pv, grid).total;
}

pdattn_status pdattn_decode_layers(const pdattn_params* p, int32_t n_layers, const pdattn_layer* layers,
                                   const int32_t* positions, const int32_t* table, void* workspace,
                                   size_t workspace_bytes, pdattn_stream stream) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (n_layers < 0) return fail(PDATTN_EINVAL, "n_layers < 0");
    if (n_layers == 0 || p->rows == 0) return PDATTN_OK;
    if (!layers) return fail(PDATTN_EINVAL, "layers is NULL");
    if (!positions || !table) return fail(PDATTN_EINVAL, "NULL positions or table");
    for (int l = 0; l < n_layers; ++l) {
        const pdattn_layer& y = layers[l];
        if (!y.q || !y.k_new || !y.v_new || !y.k_pool || !y.v_pool || !y.out)
            return fail(PDATTN_EINVAL, "layer %d: NULL data pointer", l);
        if (!aligned16(y.q) || !aligned16(y.k_new) || !aligned16(y.v_new) || !aligned16(y.k_pool) ||
            !aligned16(y.v_pool) || !aligned16(y.out))
            return fail(PDATTN_EINVAL, "layer %d: q, k_new, v_new, the pools and out must be 16-byte aligned", l);
        if (y.reserved != 0) return fail(PDATTN_EINVAL, "layer %d: reserved field must be 0", l);
    }
    int v_max = 0;
    s = layers_rows(p, n_layers, &v_max);
    if (s != PDATTN_OK) return s;
    const int grid = sm_count();
    if (grid <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    const pdattn_params pmax = with_rows(p, v_max);
    WsLayout Lmax;
    s = check_ws(&pmax, workspace, workspace_bytes, grid, &Lmax);
    if (s != PDATTN_OK) return s;
    char* ws = static_cast<char*>(workspace);
    int launches = 0;
    for (int l0 = 0; l0 < n_layers; l0 += kMaxLayers) {
        const int lg = n_layers - l0 < kMaxLayers ? n_layers - l0 : kMaxLayers;
        const pdattn_params pv = with_rows(p, lg * p->rows);
        const WsLayout L = layout_for(&pv, grid);
        PrepArgs a = prep_args(&pv, positions, table, ws, L, grid);
        a.layer_rows = p->rows;
        a.q_out = ws + L.q_rot;
        a.rope_blocks = pv.rows;
        a.do_plan = 1;
        PrepLayers pl = {};
        AttendLayers al = {};
        for (int j = 0; j < lg; ++j) {
            const pdattn_layer& y = layers[l0 + j];
            pl.q[j] = y.q;
            pl.k_new[j] = y.k_new;
            pl.v_new[j] = y.v_new;
            pl.k_pool[j] = y.k_pool;
            pl.v_pool[j] = y.v_pool;
            pl.window[j] = y.window;
            if ((s = make_pool_map(&al.k[j], y.k_pool, p)) != PDATTN_OK) return s;
            if ((s = make_pool_map(&al.v[j], y.v_pool, p)) != PDATTN_OK) return s;
            al.out[j] = y.out;
            al.sinks[j] = y.sinks;
            al.window[j] = y.window;
        }
        int n = 0;
        cudaError_t e = launch_prep_layers(a, pl, p->dtype, (cudaStream_t)stream, &n);
        if (e != cudaSuccess) return cuda_fail(e, "multi-layer plan + rope/write launches");
        launches += n;
        AttendArgs aa = {};
        aa.rows = pv.rows;
        aa.heads = p->heads;
        aa.kv_heads = p->kv_heads;
        aa.group = p->heads / p->kv_heads;
        aa.head_dim = p->head_dim;
        aa.pages_per_row = p->pages_per_row;
        aa.num_pages = p->num_pages;
        aa.layer_rows = p->rows;
        aa.n_layers = lg;
        aa.chunk_pages = p->chunk_pages;
        aa.scale_log2 = scale_log2(p);
        aa.q = ws + L.q_rot;
        aa.positions = positions;
        aa.table = table;
        aa.ws = ws;
        aa.L = L;
        e = launch_attend_layers(aa, al, p->dtype, grid, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "multi-layer attention launch");
        launches += 1;
    }
    g_launches = launches;
    return PDATTN_OK;
}

size_t pdattn_prefill_workspace_size(const pdattn_params* p, int32_t n_tokens) {
    if (check_params(p) != PDATTN_OK || n_tokens < 0) return 0;
    return pf_layout(n_tokens, p->heads, p->head_dim, elem_bytes(p)).total;
}

// Shared body of the two prefill entry points; with_prep false re-runs the
// attention only, over the tile list and rotated queries in the workspace.
static pdattn_status prefill_impl(const pdattn_params* p, int32_t n_tokens, const void* q, const void* k_new,
                                  const void* v_new, const int32_t* positions, const int32_t* rows,
                                  const int32_t* slots, const int32_t* table, void* k_pool, void* v_pool,
                                  void* out, void* workspace, size_t workspace_bytes, pdattn_stream stream,
                                  bool with_prep) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (n_tokens < 0) return fail(PDATTN_EINVAL, "n_tokens < 0");
    if (p->dtype != PDATTN_BF16) return fail(PDATTN_EUNSUPPORTED, "prefill runs on the tensor cores: dtype must be bf16");
    if (p->rows <= 0) return fail(PDATTN_EINVAL, "prefill needs at least one table row");
    if (n_tokens == 0) return PDATTN_OK;
    if (!positions || !table || !k_pool || !v_pool || !out ||
        (with_prep && (!q || !k_new || !v_new || !rows || !slots)))
        return fail(PDATTN_EINVAL, "NULL data pointer");
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
        (with_prep && (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new))))
        return fail(PDATTN_EINVAL, "q, k_new, v_new, the pools and out must be 16-byte aligned");
    if (!workspace) return fail(PDATTN_EINVAL, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return fail(PDATTN_EINVAL, "workspace must be 256-byte aligned");
    const PfLayout L = pf_layout(n_tokens, p->heads, p->head_dim, 2);
    if (workspace_bytes < L.total)
        return fail(PDATTN_EINVAL, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, L.total);
    const int sms = sm_count();
    if (sms <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    char* ws = static_cast<char*>(workspace);
    const int g = p->heads / p->kv_heads;
    const int tile_tokens = 2 * (kPfRows / g);   // two halves of 128 / g tokens

    // Rotated queries [n_tokens, heads, D] as a 3-D tensor (D, heads, tokens):
    // one box = the g heads of a kv head for one half tile (128 / g tokens),
    // 64 columns wide.
    auto fn = encode_fn();
    if (!fn) return fail(PDATTN_ECUDA, "cuTensorMapEncodeTiled is not available");
    CUtensorMap qm, km, vm;
    {
        cuuint64_t dims[3] = {(cuuint64_t)p->head_dim, (cuuint64_t)p->heads, (cuuint64_t)n_tokens};
        cuuint64_t strides[2] = {(cuuint64_t)p->head_dim * 2, (cuuint64_t)p->heads * p->head_dim * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(tile_tokens / 2)};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws + L.q_rot, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PDATTN_ECUDA, "cuTensorMapEncodeTiled (queries) failed (%d)", (int)r);
    }
    s = make_pool_map(&km, k_pool, p);
    if (s != PDATTN_OK) return s;
    s = make_pool_map(&vm, v_pool, p);
    if (s != PDATTN_OK) return s;

    int launches = 0;
    if (with_prep) {
        PrefillPrepArgs pa = {};
        pa.n_tokens = n_tokens;
        pa.rows = p->rows;
        pa.heads = p->heads;
        pa.kv_heads = p->kv_heads;
        pa.head_dim = p->head_dim;
        pa.pages_per_row = p->pages_per_row;
        pa.num_pages = p->num_pages;
        pa.window = p->window;
        pa.rope_len = p->rope_len;
        pa.tile_tokens = tile_tokens;
        pa.q = q;
        pa.k_new = k_new;
        pa.v_new = v_new;
        pa.positions = positions;
        pa.row_of = rows;
        pa.slots = slots;
        pa.rope_cos = p->rope_cos;
        pa.rope_sin = p->rope_sin;
        pa.k_pool = k_pool;
        pa.v_pool = v_pool;
        pa.ws = ws;
        pa.L = L;
        cudaError_t e = launch_prefill_prep(pa, p->dtype, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "prefill tile/rope/write launch");
        launches += 2;
    }

    PrefillArgs aa = {};
    aa.n_tokens = n_tokens;
    aa.heads = p->heads;
    aa.kv_heads = p->kv_heads;
    aa.group = g;
    aa.tile_tokens = tile_tokens;
    aa.head_dim = p->head_dim;
    aa.pages_per_row = p->pages_per_row;
    aa.num_pages = p->num_pages;
    aa.window = p->window;
    aa.scale_log2 = scale_log2(p);
    aa.positions = positions;
    aa.table = table;
    aa.sinks = p->sinks;
    aa.out = out;
    aa.ws = ws;
    aa.L = L;
    const long long units = (long long)n_tokens * p->kv_heads;   // bound on tiles x kv heads
    const int grid = (int)(units < sms ? units : sms);
    cudaError_t e = launch_prefill(aa, qm, km, vm, grid, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
    g_launches = launches + 1;
    return PDATTN_OK;
}

pdattn_status pdattn_prefill_paged(const pdattn_params* p, int32_t n_tokens, const void* q, const void* k_new,
                                   const void* v_new, const int32_t* positions, const int32_t* rows,
                                   const int32_t* slots, const int32_t* table, void* k_pool, void* v_pool,
                                   void* out, void* workspace, size_t workspace_bytes, pdattn_stream stream) {
    return prefill_impl(p, n_tokens, q, k_new, v_new, positions, rows, slots, table, k_pool, v_pool, out,
                        workspace, workspace_bytes, stream, true);
}

pdattn_status pdattn_prefill_attend(const pdattn_params* p, int32_t n_tokens, const int32_t* positions,
                                    const int32_t* table, const void* k_pool, const void* v_pool, void* out,
                                    void* workspace, size_t workspace_bytes, pdattn_stream stream) {
    return prefill_impl(p, n_tokens, nullptr, nullptr, nullptr, positions, nullptr, nullptr, table,
                        const_cast<void*>(k_pool), const_cast<void*>(v_pool), out, workspace, workspace_bytes,
                        stream, false);
}

static pdattn_status check_packed_params(const pdattn_params* p) {
    if (!p) return fail(PDATTN_EINVAL, "params is NULL");
    if (p->heads <= 0 || p->kv_heads <= 0 || p->heads % p->kv_heads != 0)
        return fail(PDATTN_EINVAL, "heads (%d) must be a positive multiple of kv_heads (%d)", p->heads, p->kv_heads);
    if (p->head_dim <= 0 || p->head_dim % 2 != 0) return fail(PDATTN_EINVAL, "head_dim must be even and positive");
    if (p->dtype != PDATTN_BF16 && p->dtype != PDATTN_F32) return fail(PDATTN_EINVAL, "unknown dtype %d", p->dtype);
    if ((p->rope_cos == nullptr) != (p->rope_sin == nullptr))
        return fail(PDATTN_EINVAL, "rope_cos and rope_sin must be both set or both NULL");
    if (p->rope_cos && p->rope_len <= 0) return fail(PDATTN_EINVAL, "rope_len must be > 0 with rope tables");
    if (p->rope_cos && (!aligned16(p->rope_cos) || !aligned16(p->rope_sin)))
        return fail(PDATTN_EINVAL, "rope tables must be 16-byte aligned");
    if (!(p->scale >= 0.f)) return fail(PDATTN_EINVAL, "scale must be >= 0 (0 selects rsqrt(head_dim))");
    if (p->dtype != PDATTN_BF16) return fail(PDATTN_EUNSUPPORTED, "packed attention runs on the tensor cores: dtype must be bf16");
    if (p->head_dim != 64 && p->head_dim != 128) return fail(PDATTN_EUNSUPPORTED, "head_dim must be 64 or 128");
    if (p->heads / p->kv_heads > kMaxGroup) return fail(PDATTN_EUNSUPPORTED, "heads / kv_heads must be <= 8");
    return PDATTN_OK;
}

size_t pdattn_packed_workspace_size(const pdattn_params* p, int32_t n_tokens) {
    if (check_packed_params(p) != PDATTN_OK || n_tokens < 0) return 0;
    return pk_layout(n_tokens, p->heads, p->kv_heads, p->head_dim, 2).total;
}

// Shared body of the packed entry points; with_prep false re-runs the
// attention only, over the tile list and rotated q and k in the workspace.
static pdattn_status packed_impl(const pdattn_params* p, int32_t n_tokens, const void* q, const void* k,
                                 const void* v, const int32_t* positions, const int32_t* segments, void* out,
                                 void* workspace, size_t workspace_bytes, pdattn_stream stream, bool with_prep) {
    g_launches = 0;
    pdattn_status s = check_packed_params(p);
    if (s != PDATTN_OK) return s;
    if (n_tokens < 0) return fail(PDATTN_EINVAL, "n_tokens < 0");
    if (n_tokens == 0) return PDATTN_OK;
    if (!v || !positions || !out || (with_prep && (!q || !k || !segments)))
        return fail(PDATTN_EINVAL, "NULL data pointer");
    if (!aligned16(v) || !aligned16(out) || (with_prep && (!aligned16(q) || !aligned16(k))))
        return fail(PDATTN_EINVAL, "q, k, v and out must be 16-byte aligned");
    if (!workspace) return fail(PDATTN_EINVAL, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return fail(PDATTN_EINVAL, "workspace must be 256-byte aligned");
    const PfLayout L = pk_layout(n_tokens, p->heads, p->kv_heads, p->head_dim, 2);
    if (workspace_bytes < L.total)
        return fail(PDATTN_EINVAL, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, L.total);
    const int sms = sm_count();
    if (sms <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    char* ws = static_cast<char*>(workspace);
    const int g = p->heads / p->kv_heads, tile_tokens = 2 * (kPfRows / g), D = p->head_dim;

    auto fn = encode_fn();
    if (!fn) return fail(PDATTN_ECUDA, "cuTensorMapEncodeTiled is not available");
    // queries (D, heads, tokens), boxes of g heads x half a tile; keys and
    // values (D, kv_heads, tokens), boxes of one kv head x 64 tokens
    auto map3 = [&](CUtensorMap* m, const void* base, int heads, int box_h, int box_t) -> pdattn_status {
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)n_tokens};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)box_h, (cuuint32_t)box_t};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(PDATTN_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
        return PDATTN_OK;
    };
    CUtensorMap qm, km, vm;
    if ((s = map3(&qm, ws + L.q_rot, p->heads, g, tile_tokens / 2)) != PDATTN_OK) return s;
    if ((s = map3(&km, ws + L.k_rot, p->kv_heads, 1, kPageSize)) != PDATTN_OK) return s;
    if ((s = map3(&vm, v, p->kv_heads, 1, kPageSize)) != PDATTN_OK) return s;

    PrefillPrepArgs pa = {};
    pa.n_tokens = n_tokens;
    pa.rows = 0;
    pa.heads = p->heads;
    pa.kv_heads = p->kv_heads;
    pa.head_dim = D;
    pa.window = p->window;
    pa.rope_len = p->rope_len;
    pa.tile_tokens = tile_tokens;
    pa.q = q;
    pa.k_new = k;
    pa.v_new = v;
    pa.positions = positions;
    pa.row_of = segments;
    pa.rope_cos = p->rope_cos;
    pa.rope_sin = p->rope_sin;
    pa.ws = ws;
    pa.L = L;
    cudaError_t e = cudaSuccess;
    if (with_prep) {
        e = launch_packed_prep(pa, p->dtype, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "packed plan/rope launch");
    }

    PrefillArgs aa = {};
    aa.n_tokens = n_tokens;
    aa.heads = p->heads;
    aa.kv_heads = p->kv_heads;
    aa.group = g;
    aa.tile_tokens = tile_tokens;
    aa.head_dim = D;
    aa.window = p->window;
    aa.packed = 1;
    aa.scale_log2 = scale_log2(p);
    aa.positions = positions;
    aa.sinks = p->sinks;
    aa.out = out;
    aa.ws = ws;
    aa.L = L;
    const long long units = (long long)n_tokens * p->kv_heads;
    e = launch_packed(aa, qm, km, vm, (int)(units < sms ? units : sms), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "packed attention launch");
    g_launches = with_prep ? 3 : 1;
    return PDATTN_OK;
}

pdattn_status pdattn_packed(const pdattn_params* p, int32_t n_tokens, const void* q, const void* k, const void* v,
                            const int32_t* positions, const int32_t* segments, void* out, void* workspace,
                            size_t workspace_bytes, pdattn_stream stream) {
    return packed_impl(p, n_tokens, q, k, v, positions, segments, out, workspace, workspace_bytes, stream, true);
}

pdattn_status pdattn_packed_attend(const pdattn_params* p, int32_t n_tokens, const void* v, const int32_t* positions,
                                   void* out, void* workspace, size_t workspace_bytes, pdattn_stream stream) {
    return packed_impl(p, n_tokens, nullptr, nullptr, v, positions, nullptr, out, workspace, workspace_bytes, stream,
                       false);
}

pdattn_status pdattn_check_status(void* workspace, pdattn_stream stream) {
    if (!workspace) return fail(PDATTN_EINVAL, "workspace is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int status = 0;
    e = cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (status != 0) {
        const int zero = 0;
        e = cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "status clear");
    }
    if (status & kErrTimeout) return fail(PDATTN_ETIMEOUT, "a device wait ran past its limit (status 0x%x)", status);
    if (status & kErrBadPage) return fail(PDATTN_EBADPAGE, "a page id outside the pool (status 0x%x)", status);
    if (status & kErrBadPos) return fail(PDATTN_EBADPOS, "a position outside the table or rope table (status 0x%x)", status);
    if (status & kErrBadPlan) return fail(PDATTN_EINVAL, "attention ran without a matching plan (status 0x%x)", status);
    return PDATTN_OK;
}

const char* pdattn_last_error(void) { return g_error.c_str(); }

int32_t pdattn_last_launch_count(void) { return g_launches; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running
// under an allocator that forbids new device allocations once serving has
// started, plugins loaded into a host program that owns all device memory,
// or C callers without a CUDA allocator of their own.  For them the whole
// fused step runs with its scratch (split plan, partial results, counters
// and rotated queries) in one fixed array compiled into this library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kStaticScratchBytes of device memory until the process exits.
// Host code cannot use the variable's name as a device address; the first
// call on each device (with that device current) looks the address up with
// cudaGetSymbolAddress and keeps it.  Make that first call before capturing
// any stream.  The set-up issues no work on any stream: the array starts out
// zero-filled, and the planner that opens every call rewrites each control
// field the attention kernel reads, so nothing needs clearing.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mutex;
void* g_static_ptr[64] = {};

// Device address of the array on the current device; set up once per device.
pdattn_status static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PDATTN_EUNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || ptr == nullptr) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return PDATTN_OK;
}

}  // namespace

extern "C" pdattn_status pdattn_decode_fused_noalloc(const pdattn_params* p, const void* q, const void* k_new,
                                                     const void* v_new, const int32_t* positions,
                                                     const int32_t* table, void* k_pool, void* v_pool, void* out,
                                                     pdattn_stream stream) {
    g_launches = 0;
    pdattn_status s = check_params(p);
    if (s != PDATTN_OK) return s;
    if (p->rows == 0) return PDATTN_OK;
    const int grid = sm_count();
    if (grid <= 0) return fail(PDATTN_ECUDA, "no CUDA device");
    const size_t need = layout_for(p, grid).total;
    if (need > kStaticScratchBytes)
        return fail(PDATTN_EINVAL,
                    "these parameters need %zu bytes of scratch, more than the %zu-byte static array of "
                    "pdattn_decode_fused_noalloc; use pdattn_decode_fused with a workspace",
                    need, kStaticScratchBytes);
    void* scratch = nullptr;
    s = static_scratch(&scratch);
    if (s != PDATTN_OK) return s;
    // The planner that runs first in this call resets every counter the
    // attention kernel relies on, so nothing else in the array needs clearing.
    return pdattn_decode_fused(p, q, k_new, v_new, positions, table, k_pool, v_pool, out, scratch,
                               kStaticScratchBytes, stream);
}
