// RoPE tables, RoPE + paged cache write, and the split planner.
//
// Follows the Llama example page: "src/rope.linnet" (`tables`) for the
// tables and "src/attention.linnet" (`decode`: rope on q and k at pos, then
// `write_at` of k and v) for the write, with the paged slot of the
// llama-3.1-8b-instruct architecture page (`decode_paged`, PageSize = 64).
#include <climits>
#include <type_traits>

#include "internal.h"

namespace pdattn {

// ---------------------------------------------------------------------------
// Tables: inv_freq[i] = exp(-(f32(i) * 2 / f32(D)) * log(theta)) in f32,
// angle = f32(s) * inv_freq[i], full = concat(angle, angle), cast<T>(cos),
// cast<T>(sin).  Every f32 step is one correctly rounded operation; cos, sin,
// exp and log are evaluated in double and rounded to f32.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }

template <typename T>
__global__ void rope_tables_kernel(float theta, int D, int S, T* __restrict__ cos_out,
                                   T* __restrict__ sin_out) {
    const int half = D / 2;
    const float log_theta = static_cast<float>(log(static_cast<double>(theta)));
    const long long n = static_cast<long long>(S) * half;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
         idx += (long long)gridDim.x * blockDim.x) {
        const int s = static_cast<int>(idx / half);
        const int i = static_cast<int>(idx % half);
        const float two_i = __fmul_rn(static_cast<float>(i), 2.0f);
        const float ratio = __fdiv_rn(two_i, static_cast<float>(D));
        const float arg = __fmul_rn(-ratio, log_theta);
        const float inv_freq = static_cast<float>(exp(static_cast<double>(arg)));
        const float angle = __fmul_rn(static_cast<float>(s), inv_freq);
        const float c = static_cast<float>(cos(static_cast<double>(angle)));
        const float sn = static_cast<float>(sin(static_cast<double>(angle)));
        const size_t o = static_cast<size_t>(s) * D + i;
        cos_out[o] = from_f32<T>(c);
        cos_out[o + half] = from_f32<T>(c);
        sin_out[o] = from_f32<T>(sn);
        sin_out[o + half] = from_f32<T>(sn);
    }
}

// ---------------------------------------------------------------------------
// 16-byte vectors of T and the rotation of one pair of them.
// ---------------------------------------------------------------------------
template <typename T>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void to_f32(const uint4& v, float (&f)[8]) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
        #pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 t = __bfloat1622float2(h[k]);
            f[2 * k] = t.x;
            f[2 * k + 1] = t.y;
        }
    }
    __device__ static uint4 from_f32(const float (&f)[8]) {
        uint4 v;
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
        #pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = pack_bf16x2(f[2 * k], f[2 * k + 1]);
        return v;
    }
};
template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ static void to_f32(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 from_f32(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

// y_lo = x_lo * c_lo - x_hi * s_lo, y_hi = x_hi * c_hi + x_lo * s_hi: the
// pages' x * cos + rotate_half(x) * sin with rotate_half(x) = [-x_hi, x_lo].
// Separate f32 products and one f32 add (no fused multiply-add), then one
// rounding to T.
template <typename T>
__device__ __forceinline__ void rope_pair(const T* x, T* y, const T* cos_row, const T* sin_row,
                                          int half, int e0) {
    using V = Vec16<T>;
    constexpr int N = V::N;
    float xl[N], xh[N], cl[N], ch[N], sl[N], sh[N], yl[N], yh[N];
    V::to_f32(*reinterpret_cast<const uint4*>(x + e0), xl);
    V::to_f32(*reinterpret_cast<const uint4*>(x + half + e0), xh);
    V::to_f32(__ldg(reinterpret_cast<const uint4*>(cos_row + e0)), cl);
    V::to_f32(__ldg(reinterpret_cast<const uint4*>(cos_row + half + e0)), ch);
    V::to_f32(__ldg(reinterpret_cast<const uint4*>(sin_row + e0)), sl);
    V::to_f32(__ldg(reinterpret_cast<const uint4*>(sin_row + half + e0)), sh);
    #pragma unroll
    for (int k = 0; k < N; ++k) {
        yl[k] = __fsub_rn(__fmul_rn(xl[k], cl[k]), __fmul_rn(xh[k], sl[k]));
        yh[k] = __fadd_rn(__fmul_rn(xh[k], ch[k]), __fmul_rn(xl[k], sh[k]));
    }
    *reinterpret_cast<uint4*>(y + e0) = V::from_f32(yl);
    *reinterpret_cast<uint4*>(y + half + e0) = V::from_f32(yh);
}

// ---------------------------------------------------------------------------
// Prep kernel: blocks [0, rope_blocks) rotate and write one row each; the
// last block (if plan) builds the split plan.
// ---------------------------------------------------------------------------
// Rotates the Hq query vectors q into q_out and the Hk key vectors kn into
// k_dst (head h at k_dst + h * head_stride), and copies the value vectors vn
// to v_dst the same way; with write_kv false only the queries, and with
// v_dst == nullptr no values.  cos_row == nullptr: plain copies.
template <typename T>
__device__ __forceinline__ void rope_write_vectors(const T* q, T* q_out, const T* kn, const T* vn, T* k_dst, T* v_dst,
                                                   size_t head_stride, const T* cos_row, const T* sin_row, int Hq,
                                                   int Hk, int D, bool write_kv) {
    constexpr int N = Vec16<T>::N;
    const bool rope = cos_row != nullptr;
    const int half = D / 2;
    const int per_head = rope ? half / N : D / N;  // work units per head vector
    const int uq = Hq * per_head, uk = Hk * per_head, uv = v_dst ? Hk * (D / N) : 0;
    for (int u = threadIdx.x; u < uq + uk + uv; u += blockDim.x) {
        if (u < uq) {
            const int h = u / per_head, e0 = (u % per_head) * N;
            if (rope) {
                rope_pair<T>(q + (size_t)h * D, q_out + (size_t)h * D, cos_row, sin_row, half, e0);
            } else {
                *reinterpret_cast<uint4*>(q_out + (size_t)h * D + e0) =
                    *reinterpret_cast<const uint4*>(q + (size_t)h * D + e0);
            }
        } else if (!write_kv) {
            break;
        } else if (u < uq + uk) {
            const int v = u - uq, h = v / per_head, e0 = (v % per_head) * N;
            T* slot = k_dst + h * head_stride;
            if (rope) {
                rope_pair<T>(kn + (size_t)h * D, slot, cos_row, sin_row, half, e0);
            } else {
                *reinterpret_cast<uint4*>(slot + e0) =
                    __ldg(reinterpret_cast<const uint4*>(kn + (size_t)h * D + e0));
            }
        } else {
            const int v = u - uq - uk, h = v / (D / N), e0 = (v % (D / N)) * N;
            T* slot = v_dst + h * head_stride;
            *reinterpret_cast<uint4*>(slot + e0) =
                __ldg(reinterpret_cast<const uint4*>(vn + (size_t)h * D + e0));
        }
    }
}

// Pool slot (page, off) of kv head 0; kv head h is kPageSize * D further.
template <typename T>
__device__ __forceinline__ T* pool_slot(void* pool, int page, int Hk, int off, int D) {
    return static_cast<T*>(pool) + (((size_t)page * Hk) * kPageSize + off) * D;
}

// Launch row v: row v of the call, or in a multi-layer launch row
// v % layer_rows of layer v / layer_rows (the table and the positions are
// shared by every layer).
template <typename Lay>
__device__ __forceinline__ int table_row(const PrepArgs& a, int v) {
    if constexpr (std::is_same<Lay, PrepLayers>::value) return v % a.layer_rows;
    else return v;
}

template <typename Lay>
__device__ __forceinline__ int row_window(const PrepArgs& a, const Lay& lay, int v) {
    if constexpr (std::is_same<Lay, PrepLayers>::value) return lay.window[v / a.layer_rows];
    else return a.window;
}

template <typename T, typename Lay>
__device__ void rope_write_row(const PrepArgs& a, const Lay& lay, int row) {
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    const int D = a.head_dim, Hq = a.heads, Hk = a.kv_heads;
    const void *q = a.q, *k_new = a.k_new, *v_new = a.v_new;
    void *k_pool = a.k_pool, *v_pool = a.v_pool;
    int r = row;
    if constexpr (std::is_same<Lay, PrepLayers>::value) {
        const int l = row / a.layer_rows;
        r = row - l * a.layer_rows;
        q = lay.q[l];
        k_new = lay.k_new[l];
        v_new = lay.v_new[l];
        k_pool = lay.k_pool[l];
        v_pool = lay.v_pool[l];
    }
    const int pos = __ldg(a.positions + r);
    const bool rope = a.rope_cos != nullptr;
    if (pos < 0 || pos >= a.pages_per_row * kPageSize || (rope && pos >= a.rope_len)) {
        if (threadIdx.x == 0) set_error(ctrl, kErrBadPos);
        return;
    }
    const int page = __ldg(a.table + (size_t)r * a.pages_per_row + pos / kPageSize);
    const bool page_ok = page >= 0 && page < a.num_pages;
    if (!page_ok && threadIdx.x == 0) set_error(ctrl, kErrBadPage);
    const int off = pos % kPageSize, pg = page_ok ? page : 0;
    rope_write_vectors<T>(static_cast<const T*>(q) + (size_t)r * Hq * D,
                          static_cast<T*>(a.q_out) + (size_t)row * Hq * D,
                          static_cast<const T*>(k_new) + (size_t)r * Hk * D,
                          static_cast<const T*>(v_new) + (size_t)r * Hk * D, pool_slot<T>(k_pool, pg, Hk, off, D),
                          pool_slot<T>(v_pool, pg, Hk, off, D), (size_t)kPageSize * D,
                          rope ? static_cast<const T*>(a.rope_cos) + (size_t)pos * D : nullptr,
                          rope ? static_cast<const T*>(a.rope_sin) + (size_t)pos * D : nullptr, Hq, Hk, D, page_ok);
}


// One block.  Splits every row's visible pages [lo / 64, pos / 64] into
// chunks of C pages and lists the (row, kv head, chunk) items sorted by size,
// largest first (a counting sort over the C sizes), so that the persistent
// attention kernel hands out long items before short ones.  Each row reserves
// its items' places with one atomic per size it uses.
constexpr int kPlanRowsCap = 2048;   // rows whose item places fit the planner's shared array

__device__ __forceinline__ void write_item(ItemDesc* items, int at, int r, int h, int c, int nch, int base,
                                           int first_page, int npg, int pos, int lo) {
    int4* dst = reinterpret_cast<int4*>(items + at);
    dst[0] = make_int4(r, (h << 16) | c, nch, base + h * nch + c);
    dst[1] = make_int4(first_page, npg, pos, lo);
}

// Exclusive block scan (sum, or max with kMax) of one int per thread, with
// `identity` before the first thread; blockDim.x a multiple of 32.  *total
// gets the block's sum or max.
template <bool kMax>
__device__ int block_scan_excl(int v, int identity, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
    #pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x = kMax ? max(x, o) : x + o;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < nw ? s_warp[lane] : identity;
        #pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, t, d);
            if (lane >= d) t = kMax ? max(t, o) : t + o;
        }
        if (lane < nw) s_warp[lane] = t;
    }
    __syncthreads();
    int up = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) up = identity;
    const int pre = w > 0 ? s_warp[w - 1] : identity;
    const int ex = kMax ? max(pre, up) : pre + up;
    *total = s_warp[nw - 1];
    __syncthreads();
    return ex;
}

// One row per thread (rows <= kFirstWaveRows <= block size): every value
// stays in registers or shared memory after the positions are read once, so
// the plan costs one global round trip plus its stores.  The first wave
// (first_wave) takes items [0, nf); merge slots start at the exclusive prefix
// sum of nch * kv_heads; the other items follow, largest first.
template <typename Lay>
__device__ bool build_plan_small(const PrepArgs& a, const Lay& lay) {
    __shared__ int4 s_row[kFirstWaveRows];
    __shared__ int2 s_at2[kFirstWaveRows];
    __shared__ int s_cnt[kChunkMax + 2];
    __shared__ int s_cur[kChunkMax + 2];
    __shared__ int s_warp[16];
    __shared__ int s_warp_max[16];
    __shared__ int s_scan[32];
    __shared__ int s_chunk;
    const int tid = threadIdx.x, R = a.rows, Hk = a.kv_heads, max_pos = a.pages_per_row * kPageSize;
    if (R > (int)blockDim.x || R > kFirstWaveRows) return false;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    int4* row_info = reinterpret_cast<int4*>(a.ws + a.L.row_info);
    ItemDesc* items = reinterpret_cast<ItemDesc*>(a.ws + a.L.items);
    int* merge_cnt = reinterpret_cast<int*>(a.ws + a.L.merge_cnt);
    const int nf = first_wave(R, Hk, a.grid_attend);

    const bool mine = tid < R;
    const int pos = mine ? __ldg(a.positions + table_row<Lay>(a, tid)) : -1;
    const bool ok = mine && pos >= 0 && pos < max_pos;
    if (mine && !ok) set_error(ctrl, kErrBadPos);
    const int lo = ok ? row_lo(pos, row_window(a, lay, tid)) : 0;
    const int first = lo / kPageSize;
    const int n = ok ? pos / kPageSize - first + 1 : 0;
    for (int i = tid; i < kChunkMax + 2; i += blockDim.x) s_cnt[i] = 0;
    const int wsum = __reduce_add_sync(0xffffffffu, (unsigned)n);
    const int wmax = __reduce_max_sync(0xffffffffu, (unsigned)n);
    if ((tid & 31) == 0) {
        s_warp[tid >> 5] = wsum;
        s_warp_max[tid >> 5] = wmax;
    }
    __syncthreads();
    if (tid == 0) {
        long long total = 0;
        int longest = 0;
        for (int w = 0; w < (int)(blockDim.x + 31) / 32; ++w) {
            total += s_warp[w];
            longest = max(longest, s_warp_max[w]);
        }
        const int c = a.chunk_pages;
        s_chunk = c > 0 ? c : choose_chunk((unsigned long long)total, longest, R, Hk, a.grid_attend);
    }
    __syncthreads();
    const int C = s_chunk;
    const Chunking ch(n, C);
    const int nch = ch.nch;
    int total_slots = 0;
    const int base = block_scan_excl<false>(nch * Hk, 0, s_scan, &total_slots);
    // kv heads of this row whose chunk 0 is in the first wave
    const int ex = min(max(nf - tid * Hk, 0), Hk);
    if (ok) {
        const int cnt_big = ch.big * Hk - (ch.big > 0 ? ex : 0);
        const int cnt_small = (nch - ch.big) * Hk - (ch.big > 0 ? 0 : ex);
        if (cnt_big) atomicAdd(&s_cnt[ch.q + 1], cnt_big);
        if (cnt_small) atomicAdd(&s_cnt[ch.q], cnt_small);
    }
    if (mine) row_info[tid] = make_int4(ok ? pos : -1, lo, nch, base);
    __syncthreads();
    if (tid == 0) {
        int off = nf;
        for (int q = C; q >= 1; --q) { s_cur[q] = off; off += s_cnt[q]; }
        s_cnt[0] = off;
    }
    __syncthreads();
    const int n_items = s_cnt[0];
    const bool fits = n_items <= a.L.max_items;
    if (mine) {
        int at_big = 0, at_small = 0;
        if (ok && fits) {
            const int cnt_big = ch.big * Hk - (ch.big > 0 ? ex : 0);
            const int cnt_small = (nch - ch.big) * Hk - (ch.big > 0 ? 0 : ex);
            at_big = cnt_big ? atomicAdd(&s_cur[ch.q + 1], cnt_big) : 0;
            at_small = cnt_small ? atomicAdd(&s_cur[ch.q], cnt_small) : 0;
        }
        s_row[tid] = make_int4(ok ? pos : -1, lo, nch, base);
        s_at2[tid] = make_int2(at_big, at_small);
    }
    __syncthreads();
    for (int pr = tid; pr < R * Hk; pr += blockDim.x) {
        const int r = pr / Hk, h = pr % Hk;
        merge_cnt[pr] = 0;
        const int4 ri = s_row[r];
        if (!fits) continue;
        if (ri.x < 0) {
            // an invalid row keeps its first-wave places, as empty items
            if (pr < nf) write_item(items, pr, r, h, 0, 0, 0, 0, 0, -1, 0);
            continue;
        }
        const int2 at = s_at2[r];
        const int rf = ri.y / kPageSize;
        const Chunking rc(ri.x / kPageSize - rf + 1, C);
        const int rex = min(max(nf - r * Hk, 0), Hk);
        for (int c = 0; c < ri.z; ++c) {
            int idx;
            if (c == 0 && pr < nf) idx = pr;
            else if (c < rc.big) idx = at.x + c * Hk + h - rex;
            else idx = at.y + (c - rc.big) * Hk + h - (rc.big > 0 ? 0 : rex);
            write_item(items, idx, r, h, c, ri.z, ri.w, rf + rc.start(c), rc.size(c), ri.x, ri.y);
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (!fits) set_error(ctrl, kErrBadPlan);
        ctrl->n_items = fits ? n_items : 0;
        ctrl->chunk_pages = C;
        ctrl->grid = a.grid_attend;
        ctrl->next_item = a.grid_attend;   // CTA b takes item b first without an atomic
        ctrl->done_ctas = 0;
        ctrl->rows = R;
        ctrl->kv_heads = Hk;
        ctrl->pages_per_row = a.pages_per_row;
        ctrl->max_items = a.L.max_items;
        ctrl->group = a.heads / Hk;
        ctrl->head_dim = a.head_dim;
        ctrl->magic = kPlanMagic;
    }
    return true;
}

template <typename Lay>
__device__ void build_plan(const PrepArgs& a, const Lay& lay) {
    if (build_plan_small(a, lay)) return;
    __shared__ int2 s_at[kPlanRowsCap];
    __shared__ int s_cnt[kChunkMax + 1];
    __shared__ int s_cur[kChunkMax + 1];
    __shared__ unsigned long long s_work;
    __shared__ int s_longest;
    __shared__ int s_slots;
    __shared__ int s_chunk;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    int4* row_info = reinterpret_cast<int4*>(a.ws + a.L.row_info);
    ItemDesc* items = reinterpret_cast<ItemDesc*>(a.ws + a.L.items);
    int* merge_cnt = reinterpret_cast<int*>(a.ws + a.L.merge_cnt);
    const int tid = threadIdx.x, R = a.rows, Hk = a.kv_heads, max_pos = a.pages_per_row * kPageSize;

    if (tid == 0) { s_work = 0; s_slots = 0; s_longest = 0; }
    for (int i = tid; i <= kChunkMax; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();

    unsigned long long w = 0;
    int longest = 0;
    for (int r = tid; r < R; r += blockDim.x) {
        const int pos = __ldg(a.positions + table_row<Lay>(a, r));
        if (pos >= 0 && pos < max_pos) {
            const int n = pos / kPageSize - row_lo(pos, row_window(a, lay, r)) / kPageSize + 1;
            w += n;
            longest = max(longest, n);
        }
    }
    w = __reduce_add_sync(0xffffffffu, (unsigned)w);
    longest = __reduce_max_sync(0xffffffffu, (unsigned)longest);
    if ((tid & 31) == 0) {
        if (w) atomicAdd(&s_work, w);
        atomicMax(&s_longest, longest);
    }
    __syncthreads();
    if (tid == 0) {
        const int c = a.chunk_pages;
        s_chunk = c > 0 ? c : choose_chunk(s_work, s_longest, R, Hk, a.grid_attend);
    }
    __syncthreads();
    const int C = s_chunk;

    for (int r = tid; r < R; r += blockDim.x) {
        const int pos = __ldg(a.positions + table_row<Lay>(a, r));
        const bool ok = pos >= 0 && pos < max_pos;
        if (!ok) set_error(ctrl, kErrBadPos);
        const int lo = ok ? row_lo(pos, row_window(a, lay, r)) : 0;
        const int n = ok ? pos / kPageSize - lo / kPageSize + 1 : 0;
        const Chunking ch(n, C);
        if (ch.big) atomicAdd(&s_cnt[ch.q + 1], ch.big * Hk);
        if (n) atomicAdd(&s_cnt[ch.q], (ch.nch - ch.big) * Hk);
        const int base = ch.nch ? atomicAdd(&s_slots, ch.nch * Hk) : 0;
        row_info[r] = make_int4(ok ? pos : -1, lo, ch.nch, base);
    }
    __syncthreads();
    if (tid == 0) {
        int off = 0;
        for (int s = C; s >= 1; --s) { s_cur[s] = off; off += s_cnt[s]; }
        s_cnt[0] = off;  // total items
    }
    __syncthreads();
    const int n_items = s_cnt[0];
    const bool fits = n_items <= a.L.max_items;
    // Each row reserves its places (one atomic per size it uses); then the
    // (row, kv head) pairs write their items in parallel.  Rows past the
    // shared array's capacity write their own items.
    if (fits) {
        for (int r = tid; r < R; r += blockDim.x) {
            const int4 ri = row_info[r];
            const int pos = ri.x, lo = ri.y, nch = ri.z, base = ri.w;
            int at_big = 0, at_small = 0;
            if (pos >= 0) {
                const int first = lo / kPageSize;
                const Chunking ch(pos / kPageSize - first + 1, C);
                at_big = ch.big ? atomicAdd(&s_cur[ch.q + 1], ch.big * Hk) : 0;
                at_small = atomicAdd(&s_cur[ch.q], (nch - ch.big) * Hk);
                if (r >= kPlanRowsCap) {
                    for (int c = 0; c < nch; ++c)
                        for (int h = 0; h < Hk; ++h)
                            write_item(items, c < ch.big ? at_big + c * Hk + h : at_small + (c - ch.big) * Hk + h, r,
                                       h, c, nch, base, first + ch.start(c), ch.size(c), pos, lo);
                }
            }
            if (r < kPlanRowsCap) s_at[r] = make_int2(at_big, at_small);
        }
        __syncthreads();
        const int Rc = R < kPlanRowsCap ? R : kPlanRowsCap;
        for (long long pr = tid; pr < (long long)R * Hk; pr += blockDim.x) {
            const int r = (int)(pr / Hk), h = (int)(pr % Hk);
            merge_cnt[pr] = 0;
            if (r >= Rc) continue;
            const int4 ri = row_info[r];
            const int pos = ri.x, lo = ri.y, nch = ri.z, base = ri.w;
            if (pos < 0) continue;
            const int first = lo / kPageSize;
            const Chunking ch(pos / kPageSize - first + 1, C);
            const int2 at = s_at[r];
            for (int c = 0; c < nch; ++c)
                write_item(items, c < ch.big ? at.x + c * Hk + h : at.y + (c - ch.big) * Hk + h, r, h, c, nch, base,
                           first + ch.start(c), ch.size(c), pos, lo);
        }
    } else {
        for (long long pr = tid; pr < (long long)R * Hk; pr += blockDim.x) merge_cnt[pr] = 0;
    }
    __syncthreads();
    if (tid == 0) {
        if (!fits) set_error(ctrl, kErrBadPlan);
        ctrl->n_items = fits ? n_items : 0;
        ctrl->chunk_pages = C;
        ctrl->grid = a.grid_attend;
        ctrl->next_item = a.grid_attend;   // CTA b takes item b first without an atomic
        ctrl->done_ctas = 0;
        ctrl->rows = R;
        ctrl->kv_heads = Hk;
        ctrl->pages_per_row = a.pages_per_row;
        ctrl->max_items = a.L.max_items;
        ctrl->group = a.heads / Hk;
        ctrl->head_dim = a.head_dim;
        ctrl->magic = kPlanMagic;
    }
}

// The split planner: one block.  It lets the launch that follows start at
// once (the rope and cache-write blocks do not read the plan).
template <typename Lay>
__global__ void __launch_bounds__(512) plan_kernel(const __grid_constant__ PrepArgs a,
                                                  const __grid_constant__ Lay lay) {
    griddep_launch_dependents();
    build_plan(a, lay);
}

// RoPE and cache write: one block per row, no shared memory, so that the
// attention launch that follows (programmatic, one CTA per SM with most of
// the SM's shared memory) can start its prologue beside these blocks.  When
// a planner launch precedes this one (do_plan), the last block exits only
// after the planner has finished: the attention launch waits for this grid
// alone, and that wait then covers the plan as well.
constexpr int kRopeRowThreads = 256;

template <typename T, typename Lay>
__global__ void __launch_bounds__(kRopeRowThreads) rope_write_kernel(const __grid_constant__ PrepArgs a,
                                                                     const __grid_constant__ Lay lay) {
    griddep_launch_dependents();
    rope_write_row<T>(a, lay, blockIdx.x);
    if (a.do_plan && blockIdx.x == gridDim.x - 1) griddep_wait();
}

// ---------------------------------------------------------------------------
// Paged prefill (llama-3.1-8b-instruct page, `prefill_paged`): every packed
// token's q and k are rotated at its own position, k and v written at its
// slot (page * 64 + offset), and the tokens are cut into tiles for the
// tensor-core attention: runs of consecutive tokens of one row, at most
// tile_tokens long, listed by visible pages, largest first.
// ---------------------------------------------------------------------------
constexpr int kPfBuckets = 1024;     // sort buckets of tile sizes (pages, capped)


// The planners run as one block of kPrepThreads threads over chunks of
// kChunk tokens.  A chunk's row (or segment) ids and positions are staged in
// shared memory with coalesced loads, padded by one word every 32 so that
// each thread then reads its kPerThread consecutive tokens without bank
// conflicts.
constexpr int kPrepThreads = 512;
constexpr int kPerThread = 8;
constexpr int kChunk = kPrepThreads * kPerThread;
constexpr int kChunkPad = kChunk + kChunk / 32;

__device__ __forceinline__ int pad_idx(int i) { return i + (i >> 5); }

// Stages ids[base .. base + kChunk) and pos[...] (fill values past n).
__device__ __forceinline__ void stage_chunk(const int* __restrict__ ids, const int* __restrict__ pos, int base, int n,
                                            int id_fill, int pos_fill, int* s_id, int* s_pos) {
    for (int idx = threadIdx.x; idx < kChunk; idx += blockDim.x) {
        const int i = base + idx;
        s_id[pad_idx(idx)] = i < n ? __ldg(ids + i) : id_fill;
        s_pos[pad_idx(idx)] = i < n ? __ldg(pos + i) : pos_fill;
    }
}

// Counting sort of the tile descriptors by pages, largest first (bucket
// kPfBuckets - 1 first); s_off holds the histogram on entry.
__device__ void sort_tiles(const PfTile* raw, PfTile* tiles, int n_tiles, int* s_off, int* s_warp) {
    const int tid = threadIdx.x;
    constexpr int per = kPfBuckets / kPrepThreads;   // buckets per thread
    int h[per];
    int sum = 0;
    #pragma unroll
    for (int k = 0; k < per; ++k) {
        h[k] = s_off[kPfBuckets - 1 - (tid * per + k)];
        sum += h[k];
    }
    int total;
    int off = block_scan_excl<false>(sum, 0, s_warp, &total);
    #pragma unroll
    for (int k = 0; k < per; ++k) {
        s_off[kPfBuckets - 1 - (tid * per + k)] = off;
        off += h[k];
    }
    __syncthreads();
    for (int b = tid; b < n_tiles; b += blockDim.x) {
        const int4* src = reinterpret_cast<const int4*>(raw + b);
        const int4 d0 = src[0], d1 = src[1];
        const int at = atomicAdd(&s_off[d1.x < kPfBuckets ? d1.x : kPfBuckets - 1], 1);
        int4* dst = reinterpret_cast<int4*>(tiles + at);
        dst[0] = d0;
        dst[1] = d1;
    }
    __syncthreads();
}

__device__ void build_prefill_plan(const PrefillPrepArgs& a) {
    __shared__ int s_warp[32];
    __shared__ int s_off[kPfBuckets];
    __shared__ int s_bad;
    __shared__ int s_id[kChunkPad], s_pos[kChunkPad];
    const int tid = threadIdx.x, n = a.n_tokens, Tq = a.tile_tokens;
    const int max_pos = a.pages_per_row * kPageSize;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    PfTile* raw = reinterpret_cast<PfTile*>(a.ws + a.L.tiles_raw);
    PfTile* tiles = reinterpret_cast<PfTile*>(a.ws + a.L.tiles);
    for (int b = tid; b < kPfBuckets; b += blockDim.x) s_off[b] = 0;
    if (tid == 0) s_bad = 0;

    // 1. tile starts: a token starts a tile when it starts a run of its row
    //    or lies a multiple of Tq tokens after its run's start; each tile's
    //    visible positions [lo_min, pos_max] by atomics on its descriptor.
    int carry_run = 0, n_tiles = 0, id_before = -1;
    bool bad = false;
    for (int base = 0; base < n; base += kChunk) {
        stage_chunk(a.row_of, a.positions, base, n, -1, 0, s_id, s_pos);
        __syncthreads();
        const int i0 = base + tid * kPerThread;
        int r[kPerThread], ps[kPerThread];
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            r[k] = s_id[pad_idx(tid * kPerThread + k)];
            ps[k] = s_pos[pad_idx(tid * kPerThread + k)];
        }
        const int r_before = tid > 0 ? s_id[pad_idx(tid * kPerThread - 1)] : id_before;
        unsigned run_starts = 0;
        int last_start = -1;
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int i = i0 + k;
            if (i >= n) continue;
            if (r[k] < 0 || r[k] >= a.rows || ps[k] < 0 || ps[k] >= max_pos || (a.rope_cos && ps[k] >= a.rope_len))
                bad = true;
            if (i == 0 || r[k] != (k ? r[k - 1] : r_before)) {
                run_starts |= 1u << k;
                last_start = i;
            }
        }
        int block_last;
        int rs = block_scan_excl<true>(last_start, -1, s_warp, &block_last);
        rs = max(rs, carry_run);
        unsigned tile_starts = 0;
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int i = i0 + k;
            if (i >= n) continue;
            if (run_starts >> k & 1) rs = i;
            if ((i - rs) % Tq == 0) tile_starts |= 1u << k;
        }
        int chunk_tiles;
        const int first_id = n_tiles + block_scan_excl<false>(__popc(tile_starts), 0, s_warp, &chunk_tiles);
        int id = first_id;
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            if (tile_starts >> k & 1) {
                int4* dst = reinterpret_cast<int4*>(raw + id);
                dst[0] = make_int4(i0 + k, 0, r[k], 0);
                dst[1] = make_int4(0, INT_MAX, -1, 0);
                ++id;
            }
        }
        id_before = s_id[pad_idx(kChunk - 1)];
        __syncthreads();   // descriptors initialised before the atomics below; staging free
        int cur = first_id - 1, lmin = INT_MAX, pmax = -1;
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int i = i0 + k;
            if (i >= n) continue;
            if (tile_starts >> k & 1) {
                if (cur >= 0 && pmax >= 0) {
                    atomicMin(&raw[cur].lo_min, lmin);
                    atomicMax(&raw[cur].pos_max, pmax);
                }
                ++cur;
                lmin = INT_MAX;
                pmax = -1;
            }
            const int pos = ps[k] < 0 ? 0 : (ps[k] >= max_pos ? max_pos - 1 : ps[k]);
            lmin = min(lmin, row_lo(pos, a.window));
            pmax = max(pmax, pos);
        }
        if (cur >= 0 && pmax >= 0) {
            atomicMin(&raw[cur].lo_min, lmin);
            atomicMax(&raw[cur].pos_max, pmax);
        }
        carry_run = max(carry_run, block_last);
        n_tiles += chunk_tiles;
    }
    if (bad) atomicOr(&s_bad, 1);
    __syncthreads();   // every descriptor complete and visible to the block

    // 2. each tile's token count and pages; histogram of sizes
    for (int b = tid; b < n_tiles; b += blockDim.x) {
        const int t0 = raw[b].t0, t1 = b + 1 < n_tiles ? raw[b + 1].t0 : n;
        const int first = raw[b].lo_min / kPageSize, npg = raw[b].pos_max / kPageSize - first + 1;
        raw[b].ntok = t1 - t0;
        raw[b].first_page = first;
        raw[b].npg = npg;
        atomicAdd(&s_off[npg < kPfBuckets ? npg : kPfBuckets - 1], 1);
    }
    __syncthreads();
    sort_tiles(raw, tiles, n_tiles, s_off, s_warp);
    if (tid == 0) {
        if (s_bad) set_error(ctrl, kErrBadPos);
        ctrl->n_items = s_bad ? 0 : n_tiles;
        ctrl->next_item = 0;               // unit cursor: CTA b takes unit b first, later ones from here
        ctrl->done_ctas = 0;
        ctrl->kv_heads = a.kv_heads;
        ctrl->group = a.heads / a.kv_heads;
        ctrl->head_dim = a.head_dim;
        ctrl->magic = kPlanMagic;
    }
}

template <typename T>
__device__ void rope_write_token(const PrefillPrepArgs& a, int i) {
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    const int D = a.head_dim, Hq = a.heads, Hk = a.kv_heads;
    const int pos = __ldg(a.positions + i);
    const bool rope = a.rope_cos != nullptr;
    if (pos < 0 || pos >= a.pages_per_row * kPageSize || (rope && pos >= a.rope_len)) {
        if (threadIdx.x == 0) set_error(ctrl, kErrBadPos);
        return;
    }
    const int slot = __ldg(a.slots + i);
    const int page = slot >= 0 ? slot / kPageSize : -1;
    const bool page_ok = page >= 0 && page < a.num_pages;
    if (!page_ok && threadIdx.x == 0) set_error(ctrl, kErrBadPage);
    const int off = slot >= 0 ? slot % kPageSize : 0, pg = page_ok ? page : 0;
    rope_write_vectors<T>(static_cast<const T*>(a.q) + (size_t)i * Hq * D,
                          reinterpret_cast<T*>(a.ws + a.L.q_rot) + (size_t)i * Hq * D,
                          static_cast<const T*>(a.k_new) + (size_t)i * Hk * D,
                          static_cast<const T*>(a.v_new) + (size_t)i * Hk * D, pool_slot<T>(a.k_pool, pg, Hk, off, D),
                          pool_slot<T>(a.v_pool, pg, Hk, off, D), (size_t)kPageSize * D,
                          rope ? static_cast<const T*>(a.rope_cos) + (size_t)pos * D : nullptr,
                          rope ? static_cast<const T*>(a.rope_sin) + (size_t)pos * D : nullptr, Hq, Hk, D, page_ok);
}

// ---------------------------------------------------------------------------
// Packed sequences (Llama example page, `packed`): the pack is read as a
// contiguous cache of 64-token key blocks.  Tiles are runs of one segment id
// cut into tile_tokens.  When the pack is canonical (every segment id forms a
// single run, positions strictly increase along it) a tile visits the blocks
// from its run's start (or its window) to its own last token; otherwise every
// tile visits the whole pack, and the per-key mask alone decides.
// ---------------------------------------------------------------------------
constexpr int kPkHash = 1024;        // segment ids of runs, open addressing
constexpr int kPkRunsCap = kPkHash / 2;

__device__ __forceinline__ void pk_hash_insert(unsigned long long* tab, int id, int* noncanon) {
    const unsigned long long key = (1ull << 32) | (unsigned)id;
    unsigned h = ((unsigned)id * 2654435761u) & (kPkHash - 1);
    for (int probe = 0; probe < kPkHash; ++probe) {
        const unsigned long long prev = atomicCAS(&tab[h], 0ull, key);
        if (prev == 0ull) return;
        if (prev == key) {          // a second run of the same sequence
            *noncanon = 1;
            return;
        }
        h = (h + 1) & (kPkHash - 1);
    }
    *noncanon = 1;
}

__device__ void build_packed_plan(const PrefillPrepArgs& a) {
    __shared__ int s_warp[32];
    __shared__ int s_off[kPfBuckets];
    __shared__ int s_bad, s_noncanon, s_runs;
    __shared__ unsigned long long s_ids[kPkHash];
    __shared__ int s_id[kChunkPad], s_pos[kChunkPad];
    const int tid = threadIdx.x, n = a.n_tokens, Tq = a.tile_tokens, W = a.window;
    const int n64 = (n + kPageSize - 1) / kPageSize * kPageSize;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    PfTile* raw = reinterpret_cast<PfTile*>(a.ws + a.L.tiles_raw);
    PfTile* tiles = reinterpret_cast<PfTile*>(a.ws + a.L.tiles);
    int* seg_pad = reinterpret_cast<int*>(a.ws + a.L.seg_pad);
    int* pos_pad = reinterpret_cast<int*>(a.ws + a.L.pos_pad);
    int4* blk = reinterpret_cast<int4*>(a.ws + a.L.blk);
    for (int b = tid; b < kPfBuckets; b += blockDim.x) s_off[b] = 0;
    for (int b = tid; b < kPkHash; b += blockDim.x) s_ids[b] = 0ull;
    if (tid == 0) { s_bad = 0; s_noncanon = 0; s_runs = 0; }

    int carry_run = 0, n_tiles = 0, id_before = 0, pos_before = 0;
    bool bad = false, noncanon = false;
    static_assert(kPageSize % kPerThread == 0 && kPageSize / kPerThread <= 32, "a block's summary is one warp's");
    constexpr int kLanesPerBlock = kPageSize / kPerThread;
    for (int base = 0; base < n64; base += kChunk) {
        stage_chunk(a.row_of, a.positions, base, n, 0, INT_MAX, s_id, s_pos);
        __syncthreads();
        // the padded copies read by the attention kernel, coalesced
        for (int idx = tid; idx < kChunk && base + idx < n64; idx += blockDim.x) {
            seg_pad[base + idx] = s_id[pad_idx(idx)];
            pos_pad[base + idx] = s_pos[pad_idx(idx)];
        }
        const int i0 = base + tid * kPerThread;
        int r[kPerThread], ps[kPerThread];
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            r[k] = s_id[pad_idx(tid * kPerThread + k)];
            ps[k] = s_pos[pad_idx(tid * kPerThread + k)];
        }
        const int r_before = tid > 0 ? s_id[pad_idx(tid * kPerThread - 1)] : id_before;
        const int p_before = tid > 0 ? s_pos[pad_idx(tid * kPerThread - 1)] : pos_before;
        unsigned run_starts = 0;
        int last_start = -1;
        bool uniform = i0 + kPerThread <= n;
        int pmin = INT_MAX, pmax = INT_MIN;
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int i = i0 + k;
            if (i >= n) continue;
            if (ps[k] < 0 || (a.rope_cos && ps[k] >= a.rope_len)) bad = true;
            const bool start = i == 0 || r[k] != (k ? r[k - 1] : r_before);
            if (start) {
                run_starts |= 1u << k;
                last_start = i;
                if (atomicAdd(&s_runs, 1) >= kPkRunsCap) noncanon = true;
                else pk_hash_insert(s_ids, r[k], &s_noncanon);
            } else if (ps[k] <= (k ? ps[k - 1] : p_before)) {
                noncanon = true;
            }
            if (r[k] != r[0]) uniform = false;
            pmin = min(pmin, ps[k]);
            pmax = max(pmax, ps[k]);
        }
        // summary of each 64-token block from its kLanesPerBlock threads
        {
            int seg0 = r[0], uni_all = uniform ? 1 : 0, mn = pmin, mx = pmax;
            const int lead = __shfl_sync(0xffffffffu, seg0, (tid & 31) & ~(kLanesPerBlock - 1));
            uni_all = uni_all && seg0 == lead;
            #pragma unroll
            for (int d = 1; d < kLanesPerBlock; d <<= 1) {
                uni_all &= __shfl_xor_sync(0xffffffffu, uni_all, d);
                mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, d));
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
            }
            if ((tid & (kLanesPerBlock - 1)) == 0 && i0 < n) blk[i0 / kPageSize] = make_int4(uni_all, seg0, mn, mx);
        }
        int block_last;
        int rs = block_scan_excl<true>(last_start, -1, s_warp, &block_last);
        rs = max(rs, carry_run);
        unsigned tile_starts = 0;
        int starts_rs[kPerThread];
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int i = i0 + k;
            if (i < n && (run_starts >> k & 1)) rs = i;
            starts_rs[k] = rs;
            if (i < n && (i - rs) % Tq == 0) tile_starts |= 1u << k;
        }
        int chunk_tiles;
        int id = n_tiles + block_scan_excl<false>(__popc(tile_starts), 0, s_warp, &chunk_tiles);
        #pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            if (tile_starts >> k & 1) {
                int4* dst = reinterpret_cast<int4*>(raw + id);
                dst[0] = make_int4(i0 + k, 0, r[k], 0);
                dst[1] = make_int4(0, 0, 0, starts_rs[k]);   // .pad = start of the tile's run
                ++id;
            }
        }
        id_before = s_id[pad_idx(kChunk - 1)];
        pos_before = s_pos[pad_idx(kChunk - 1)];
        carry_run = max(carry_run, block_last);
        n_tiles += chunk_tiles;
        __syncthreads();   // staging free for the next chunk
    }
    if (bad) atomicOr(&s_bad, 1);
    if (noncanon) atomicOr(&s_noncanon, 1);
    __syncthreads();
    const bool canonical = s_noncanon == 0;

    // key blocks of each tile; histogram of sizes
    for (int b = tid; b < n_tiles; b += blockDim.x) {
        const int t0 = raw[b].t0, t1 = b + 1 < n_tiles ? raw[b + 1].t0 : n, run0 = raw[b].pad;
        int kf = 0, kl = n - 1;
        if (canonical) {
            kl = t1 - 1;
            kf = W > 0 ? max(run0, t0 - W + 1) : run0;
        }
        const int first = kf / kPageSize, npg = kl / kPageSize - first + 1;
        raw[b].ntok = t1 - t0;
        raw[b].first_page = first;
        raw[b].npg = npg;
        raw[b].lo_min = kf;
        raw[b].pos_max = kl;
        atomicAdd(&s_off[npg < kPfBuckets ? npg : kPfBuckets - 1], 1);
    }
    __syncthreads();
    sort_tiles(raw, tiles, n_tiles, s_off, s_warp);
    if (tid == 0) {
        if (s_bad) set_error(ctrl, kErrBadPos);
        ctrl->n_items = s_bad ? 0 : n_tiles;
        ctrl->next_item = 0;               // unit cursor: CTA b takes unit b first, later ones from here
        ctrl->done_ctas = 0;
        ctrl->kv_heads = a.kv_heads;
        ctrl->group = a.heads / a.kv_heads;
        ctrl->head_dim = a.head_dim;
        ctrl->rows = canonical ? 1 : 0;    // read by the attention kernel: index-range masks
        ctrl->magic = kPlanMagic;
    }
}

__global__ void __launch_bounds__(kPrepThreads) packed_plan_kernel(const __grid_constant__ PrefillPrepArgs a) {
    griddep_launch_dependents();
    build_packed_plan(a);
}

// The per-token rope kernels wait on their loads: twelve resident 128-thread
// blocks (at most 40 registers a thread) keep more loads in flight than the
// eleven that 44 registers allow; sixteen (32 registers) spill and measured
// slower.
constexpr int kRopeBlocksPerSm = 12;

// Block i rotates q and k of packed token i into the workspace.
template <typename T>
__global__ void __launch_bounds__(128, kRopeBlocksPerSm) packed_rope_kernel(const __grid_constant__ PrefillPrepArgs a) {
    griddep_launch_dependents();
    const int i = blockIdx.x, D = a.head_dim, Hq = a.heads, Hk = a.kv_heads;
    const int pos = __ldg(a.positions + i);
    const bool rope = a.rope_cos != nullptr;
    if (pos < 0 || (rope && pos >= a.rope_len)) {
        if (threadIdx.x == 0) set_error(reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl), kErrBadPos);
    } else {
        rope_write_vectors<T>(static_cast<const T*>(a.q) + (size_t)i * Hq * D,
                              reinterpret_cast<T*>(a.ws + a.L.q_rot) + (size_t)i * Hq * D,
                              static_cast<const T*>(a.k_new) + (size_t)i * Hk * D, nullptr,
                              reinterpret_cast<T*>(a.ws + a.L.k_rot) + (size_t)i * Hk * D, nullptr, (size_t)D,
                              rope ? static_cast<const T*>(a.rope_cos) + (size_t)pos * D : nullptr,
                              rope ? static_cast<const T*>(a.rope_sin) + (size_t)pos * D : nullptr, Hq, Hk, D, true);
    }
    // The last block (the last to start) waits for the planner, so this
    // grid completes after it; the other blocks leave their SM slots at once.
    if (blockIdx.x == gridDim.x - 1) griddep_wait();
}

// The tile list: one block.  Lets the rope kernel launched after it start
// at once.
__global__ void __launch_bounds__(kPrepThreads) prefill_plan_kernel(const __grid_constant__ PrefillPrepArgs a) {
    griddep_launch_dependents();
    build_prefill_plan(a);
}

// Block i rotates and writes token i.  The last block waits for the planner
// before it exits, so that the completion of this grid (all the attention
// kernel waits for) also covers the tile list; the other blocks do not wait,
// or a wave of them would hold every SM until the planner is done.
constexpr int kRopeThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kRopeThreads, kRopeBlocksPerSm) prefill_rope_kernel(const __grid_constant__ PrefillPrepArgs a) {
    griddep_launch_dependents();
    rope_write_token<T>(a, blockIdx.x);
    if (blockIdx.x == gridDim.x - 1) griddep_wait();
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
cudaError_t launch_rope_tables(float theta, int D, int S, int dtype, void* cos_out, void* sin_out,
                               cudaStream_t stream) {
    const long long n = (long long)S * (D / 2);
    if (n == 0) return cudaSuccess;
    const int block = 256;
    const int grid = (int)((n + block - 1) / block < 4096 ? (n + block - 1) / block : 4096);
    if (dtype == 0)
        rope_tables_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(
            theta, D, S, static_cast<__nv_bfloat16*>(cos_out), static_cast<__nv_bfloat16*>(sin_out));
    else
        rope_tables_kernel<float><<<grid, block, 0, stream>>>(
            theta, D, S, static_cast<float*>(cos_out), static_cast<float*>(sin_out));
    return cudaGetLastError();
}

// The planner (if a.do_plan) as an ordinary launch, then the rope + write
// blocks (if any) as its programmatic dependent.
template <typename Lay>
static cudaError_t launch_prep_any(const PrepArgs& a, const Lay& lay, int dtype, cudaStream_t stream,
                                   int* launches) {
    *launches = 0;
    if (a.do_plan) {
        plan_kernel<Lay><<<1, 512, 0, stream>>>(a, lay);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    if (a.rope_blocks == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.rope_blocks);
    cfg.blockDim = dim3(kRopeRowThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.do_plan ? 1 : 0;
    cudaError_t e = dtype == 0 ? cudaLaunchKernelEx(&cfg, rope_write_kernel<__nv_bfloat16, Lay>, a, lay)
                               : cudaLaunchKernelEx(&cfg, rope_write_kernel<float, Lay>, a, lay);
    if (e == cudaSuccess) ++*launches;
    return e;
}

cudaError_t launch_prep(const PrepArgs& a, int dtype, cudaStream_t stream, int* launches) {
    return launch_prep_any(a, NoLayers{}, dtype, stream, launches);
}

cudaError_t launch_prep_layers(const PrepArgs& a, const PrepLayers& lay, int dtype, cudaStream_t stream,
                               int* launches) {
    return launch_prep_any(a, lay, dtype, stream, launches);
}

cudaError_t launch_prefill_prep(const PrefillPrepArgs& a, int dtype, cudaStream_t stream) {
    if (a.n_tokens <= 0) return cudaSuccess;
    prefill_plan_kernel<<<1, kPrepThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_tokens);
    cfg.blockDim = dim3(kRopeThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == 0) return cudaLaunchKernelEx(&cfg, prefill_rope_kernel<__nv_bfloat16>, a);
    return cudaLaunchKernelEx(&cfg, prefill_rope_kernel<float>, a);
}

cudaError_t launch_packed_prep(const PrefillPrepArgs& a, int dtype, cudaStream_t stream) {
    if (a.n_tokens <= 0 || dtype != 0) return a.n_tokens <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    packed_plan_kernel<<<1, kPrepThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_tokens);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, packed_rope_kernel<__nv_bfloat16>, a);
}

}  // namespace pdattn
