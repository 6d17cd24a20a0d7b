// Split-KV flash-decode attention over a paged KV cache.
//
// The operation is the `decode` body of GroupedQueryAttention on the Llama
// example page ("src/attention.linnet": `seen[s] = s <= pos`,
// `grouped_attention(q, cache_k, cache_v, rsqrt(f32(D)), seen)`), where each
// kv head serves Heads / KvHeads query heads ("Key ideas", grouped-query
// attention), with the cache addressed through the page table of the paged
// entries (llama-3.1-8b-instruct architecture page, `decode_paged`).
//
// Design (one persistent CTA per SM, 5 warps):
//   * warp 4 (producer) takes (row, kv head, chunk) items from the plan with
//     an atomic cursor, and for every page of the chunk issues TMA loads of
//     the page's K and V tiles (64 tokens x D, 128-byte swizzled) into a ring
//     of shared-memory stages, plus a bulk copy of the item's query group on
//     its first page.  Full / empty mbarriers hand stages over.
//   * warps 0-3 (consumers) each take 16 of the page's 64 tokens.  bf16:
//     S^T = K Q^T on m16n8k16 tensor-core tiles (tokens as M, the <= 8 query
//     heads of the group as N, so each K/V byte is read from shared memory
//     once for the whole group), fp32 online softmax in registers, P^T moved
//     into the B-operand layout with movmatrix, O^T += V^T P^T on the same
//     tiles.  f32: the same dataflow on FP32 FMAs (lane per token for scores,
//     lane per dimension for values).
//   * at an item's last page the four warps merge their (max, sum, out)
//     through shared memory; a single-chunk row writes its output, otherwise
//     the chunk writes an fp32 partial and the last chunk to finish merges
//     all partials of the (row, kv head) and writes the output.
// Every mbarrier wait is bounded; a wait that runs out records
// kErrTimeout in the status word and the kernel winds down.
#include "internal.h"

namespace pdattn {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kNegBig = -1.0e30f;     // running-max start: finite, so exp2(m - m) = 1

enum : int { kFirst = 1, kLast = 2, kValid = 4, kTerm = 8, kPartial = 16 };

struct Meta {
    int row, kvh, nch, slot, t_lo, t_hi, flags, chunk;
};

template <typename T, int D>
struct Cfg {
    static constexpr int kElem = sizeof(T);
    static constexpr int kBoxCols = 128 / kElem;                 // columns per 128-byte box row
    static constexpr int kBoxes = D / kBoxCols;                  // boxes per K (or V) page
    static constexpr int kBoxBytes = kPageSize * 128;            // 8 KiB
    static constexpr int kTileBytes = kBoxes * kBoxBytes;        // one page of K (or V)
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = (kStageBytes <= 16384) ? 10 : (kStageBytes <= 32768 ? 5 : 2);
    static constexpr int kQBytes = kMaxGroup * D * kElem;
    static constexpr int kORow = D + 4;                          // padded row of the merge buffer
    static constexpr int kMergeFloats = 2 * kConsumerWarps * kMaxGroup + kConsumerWarps * kMaxGroup * kORow;
    static constexpr int kOffQ = kStages * kStageBytes;
    static constexpr int kOffMerge = kOffQ + kStages * kQBytes;
    static constexpr int kWarpQBytes = (kElem == 4) ? kConsumerWarps * kQBytes : 0;  // f32: private copies
    static constexpr int kOffWarpQ = kOffMerge + kMergeFloats * 4;
    static constexpr int kOffMeta = kOffWarpQ + kWarpQBytes;
    static constexpr int kOffBar = kOffMeta + kStages * (int)sizeof(Meta);
    static constexpr int kOffMisc = kOffBar + 3 * kStages * 8 + 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;           // + alignment slack
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static_assert(kOffBar % 8 == 0, "mbarrier alignment");
};

// Reusable barrier among the 128 consumer threads, on an mbarrier so that its
// wait is bounded.
struct ConsumerSync {
    uint32_t bar;
    uint32_t phase;
    __device__ bool sync() {
        mbar_arrive(bar);
        bool ok = mbar_wait(bar, phase);
        phase ^= 1;
        return ok;
    }
};

template <typename T>
__device__ __forceinline__ void store8(T* dst, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[8]) {
    uint4 w;
    w.x = pack_bf16x2(v[0], v[1]);
    w.y = pack_bf16x2(v[2], v[3]);
    w.z = pack_bf16x2(v[4], v[5]);
    w.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = w;
}
template <>
__device__ __forceinline__ void store8<float>(float* dst, const float (&v)[8]) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// ---------------------------------------------------------------------------
// Consumer state and page processing
// ---------------------------------------------------------------------------
template <typename T, int D>
struct Consumer;

// bf16: tensor-core tiles.  Lane layout of the m16n8 accumulators:
// row = lane / 4 (+8), column pair = 2 * (lane % 4).
template <int D>
struct Consumer<__nv_bfloat16, D> {
    static constexpr int KS = D / 16;     // k-steps over D for QK, m-tiles over D for PV
    uint32_t qf[KS][2];
    float o[KS][4];
    float m0, m1, l0, l1;                 // heads 2*(lane%4) and +1

    __device__ void begin(uint32_t qbuf, int lane) {
        // Q^T as the B operand: row = head, 8 dims per 16-byte chunk.
        #pragma unroll
        for (int p = 0; p < KS / 2; ++p) {
            const int head = lane & 7, chunk = 4 * p + (lane >> 3);
            ldsm_x4(qbuf + head * D * 2 + chunk * 16, qf[2 * p][0], qf[2 * p][1], qf[2 * p + 1][0],
                    qf[2 * p + 1][1]);
        }
        #pragma unroll
        for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        m0 = m1 = kNegBig;
        l0 = l1 = 0.f;
    }

    __device__ void page(uint32_t kbase, uint32_t vbase, int warp, int lane, int t_lo, int t_hi,
                         bool partial, float sl2) {
        const int tok0 = warp * 16;
        const int mi = lane >> 3, ri = lane & 7;
        // ---- S^T = K Q^T: 16 tokens x 8 heads
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int tok = tok0 + ri + ((mi & 1) << 3);
            #pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int chunk = ks * 2 + (mi >> 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(swz128(kbase + (chunk >> 3) * 8192, tok, chunk & 7), a0, a1, a2, a3);
                mma_bf16_16816(c, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            }
        }
        // ---- online softmax (log2 domain)
        const int ta = tok0 + (lane >> 2), tb = ta + 8;
        const bool va = ta >= t_lo && ta < t_hi, vb = tb >= t_lo && tb < t_hi;
        const float s0 = va ? c[0] * sl2 : -INFINITY;
        const float s1 = va ? c[1] * sl2 : -INFINITY;
        const float s2 = vb ? c[2] * sl2 : -INFINITY;
        const float s3 = vb ? c[3] * sl2 : -INFINITY;
        float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
        #pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, sh));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, sh));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float al0 = exp2_approx(m0 - n0), al1 = exp2_approx(m1 - n1);
        m0 = n0;
        m1 = n1;
        const uint32_t pa = pack_bf16x2(exp2_approx(s0 - n0), exp2_approx(s1 - n1));
        const uint32_t pb = pack_bf16x2(exp2_approx(s2 - n0), exp2_approx(s3 - n1));
        // the denominator sums the same bf16 weights the PV product uses
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa));
        const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pb));
        l0 = l0 * al0 + (fa.x + fb.x);
        l1 = l1 * al1 + (fa.y + fb.y);
        #pragma unroll
        for (int i = 0; i < KS; ++i) {
            o[i][0] *= al0; o[i][1] *= al1; o[i][2] *= al0; o[i][3] *= al1;
        }
        // ---- P^T into B-operand layout: B[k = token][n = head]
        const uint32_t b0 = movmatrix_trans(pa), b1 = movmatrix_trans(pb);
        // ---- O^T += V^T P^T: V^T tiles from the V page with transposed ldmatrix
        const int tok = tok0 + ri + ((mi >> 1) << 3);
        uint32_t keep_a = 0xffffffffu, keep_b = 0xffffffffu;
        if (partial) {
            // zero V of invisible tokens: their slots may hold anything, NaN included
            const int t = tok0 + 2 * (lane & 3);
            keep_a = ((t >= t_lo && t < t_hi) ? 0x0000ffffu : 0u) |
                     ((t + 1 >= t_lo && t + 1 < t_hi) ? 0xffff0000u : 0u);
            keep_b = ((t + 8 >= t_lo && t + 8 < t_hi) ? 0x0000ffffu : 0u) |
                     ((t + 9 >= t_lo && t + 9 < t_hi) ? 0xffff0000u : 0u);
        }
        #pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int chunk = mt * 2 + (mi & 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(swz128(vbase + (chunk >> 3) * 8192, tok, chunk & 7), a0, a1, a2, a3);
            a0 &= keep_a; a1 &= keep_a; a2 &= keep_b; a3 &= keep_b;
            mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
        }
    }

    // Put this warp's (m, l, o) for heads 0..7 into the merge buffer.
    __device__ void stash(float* sm_m, float* sm_l, float* sm_o, int warp, int lane) {
        float s0 = l0, s1 = l1;
        #pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, sh);
            s1 += __shfl_xor_sync(0xffffffffu, s1, sh);
        }
        const int h0 = 2 * (lane & 3);
        if (lane < 4) {
            sm_m[warp * kMaxGroup + h0] = m0;
            sm_m[warp * kMaxGroup + h0 + 1] = m1;
            sm_l[warp * kMaxGroup + h0] = s0;
            sm_l[warp * kMaxGroup + h0 + 1] = s1;
        }
        float* ow = sm_o + warp * kMaxGroup * (D + 4);
        const int d = lane >> 2;
        #pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            ow[h0 * (D + 4) + mt * 16 + d] = o[mt][0];
            ow[(h0 + 1) * (D + 4) + mt * 16 + d] = o[mt][1];
            ow[h0 * (D + 4) + mt * 16 + d + 8] = o[mt][2];
            ow[(h0 + 1) * (D + 4) + mt * 16 + d + 8] = o[mt][3];
        }
    }
};

// f32: FP32 FMAs.  Scores: lane = (token lane % 16, half of D lane / 16).
// Values: lane = dimension (lane + 32 e).
template <int D>
struct Consumer<float, D> {
    static constexpr int E = D / 32;
    float o[kMaxGroup][E];
    float m[kMaxGroup], l[kMaxGroup];
    uint32_t qbuf_addr;
    int g;

    // The stage's query buffer can be refilled for a later item while this
    // item is still running, so each warp keeps its own copy.
    __device__ void begin(uint32_t qbuf, uint32_t warp_q, int lane, int group) {
        qbuf_addr = warp_q;
        g = group;
        for (int i = lane; i < group * D / 4; i += 32) {
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(qbuf + i * 16));
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                         :: "r"(warp_q + i * 16), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
        }
        __syncwarp();
        #pragma unroll
        for (int j = 0; j < kMaxGroup; ++j) {
            m[j] = kNegBig;
            l[j] = 0.f;
            #pragma unroll
            for (int e = 0; e < E; ++e) o[j][e] = 0.f;
        }
    }

    __device__ void page(uint32_t kbase, uint32_t vbase, int warp, int lane, int t_lo, int t_hi,
                         bool partial, float sl2) {
        const int tok0 = warp * 16;
        const int t = tok0 + (lane & 15), half = lane >> 4;
        constexpr int kChunks = D / 8;            // 16-byte chunks in half a row
        float acc[kMaxGroup];
        #pragma unroll
        for (int j = 0; j < kMaxGroup; ++j) acc[j] = 0.f;
        #pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            const int col = half * (D / 2) + c * 4;          // first dimension of the chunk
            const int box = col / 32, cin = (col % 32) / 4;
            float4 kv;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(kv.x), "=f"(kv.y), "=f"(kv.z), "=f"(kv.w)
                         : "r"(swz128(kbase + box * 8192, t, cin)));
            #pragma unroll
            for (int j = 0; j < kMaxGroup; ++j) {
                if (j < g) {
                    float4 qv;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(qv.x), "=f"(qv.y), "=f"(qv.z), "=f"(qv.w)
                                 : "r"(qbuf_addr + (j * D + col) * 4));
                    acc[j] = fmaf(kv.x, qv.x, acc[j]);
                    acc[j] = fmaf(kv.y, qv.y, acc[j]);
                    acc[j] = fmaf(kv.z, qv.z, acc[j]);
                    acc[j] = fmaf(kv.w, qv.w, acc[j]);
                }
            }
        }
        const bool valid = t >= t_lo && t < t_hi;
        float p[kMaxGroup];
        #pragma unroll
        for (int j = 0; j < kMaxGroup; ++j) {
            if (j < g) {
                float s = acc[j] + __shfl_xor_sync(0xffffffffu, acc[j], 16);
                s = valid ? s * sl2 : -INFINITY;
                float x = s;
                #pragma unroll
                for (int sh = 1; sh < 16; sh <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, sh));
                const float n = fmaxf(m[j], x);
                const float al = exp2_approx(m[j] - n);
                m[j] = n;
                p[j] = exp2_approx(s - n);
                float ps = p[j];
                #pragma unroll
                for (int sh = 1; sh < 16; sh <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, sh);
                l[j] = l[j] * al + ps;
                #pragma unroll
                for (int e = 0; e < E; ++e) o[j][e] *= al;
            }
        }
        const int tt_lo = max(t_lo - tok0, 0), tt_hi = min(t_hi - tok0, 16);
        #pragma unroll 1
        for (int tt = tt_lo; tt < tt_hi; ++tt) {
            float v[E];
            #pragma unroll
            for (int e = 0; e < E; ++e) {
                asm volatile("ld.shared.f32 %0, [%1];"
                             : "=f"(v[e])
                             : "r"(swz128(vbase + e * 8192, tok0 + tt, lane >> 2) + (lane & 3) * 4));
            }
            #pragma unroll
            for (int j = 0; j < kMaxGroup; ++j) {
                if (j < g) {
                    const float pj = __shfl_sync(0xffffffffu, p[j], tt);
                    #pragma unroll
                    for (int e = 0; e < E; ++e) o[j][e] = fmaf(pj, v[e], o[j][e]);
                }
            }
        }
        (void)partial;
    }

    __device__ void stash(float* sm_m, float* sm_l, float* sm_o, int warp, int lane) {
        #pragma unroll
        for (int j = 0; j < kMaxGroup; ++j) {
            if (j < g) {
                if (lane == 0) {
                    sm_m[warp * kMaxGroup + j] = m[j];
                    sm_l[warp * kMaxGroup + j] = l[j];
                }
                #pragma unroll
                for (int e = 0; e < E; ++e) sm_o[(warp * kMaxGroup + j) * (D + 4) + e * 32 + lane] = o[j][e];
            }
        }
    }
};

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
attend_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
              const __grid_constant__ AttendArgs a) {
    using C = Cfg<T, D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::kOffBar;             // S barriers
    const uint32_t bar_empty = bar_full + 8 * S;              // S barriers
    const uint32_t bar_sync = bar_empty + 8 * S;              // consumer barrier
    Meta* meta = reinterpret_cast<Meta*>(smem + C::kOffMeta);
    float* sm_m = reinterpret_cast<float*>(smem + C::kOffMerge);
    float* sm_l = sm_m + kConsumerWarps * kMaxGroup;
    float* sm_o = sm_l + kConsumerWarps * kMaxGroup;
    int* s_flag = reinterpret_cast<int*>(smem + C::kOffMisc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_sync, kConsumerWarps * 32);
        fence_barrier_init();
    }
    // Query-group buffers: rows past the group stay zero.
    for (int i = threadIdx.x; i < S * C::kQBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + C::kOffQ)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_shared();
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
    }
    __syncthreads();

    // Everything below reads what the preceding launch wrote.
    griddep_wait();

    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    const int4* row_info = reinterpret_cast<const int4*>(a.ws + a.L.row_info);
    const int2* items = reinterpret_cast<const int2*>(a.ws + a.L.items);
    int* merge_cnt = reinterpret_cast<int*>(a.ws + a.L.merge_cnt);
    float2* part_ml = reinterpret_cast<float2*>(a.ws + a.L.part_ml);
    float* part_o = reinterpret_cast<float*>(a.ws + a.L.part_o);
    const int g = a.group, Hk = a.kv_heads;

    const uint32_t magic = __ldcg(&ctrl->magic);
    const int n_items = __ldcg(&ctrl->n_items);
    const int chunk_pages = __ldcg(&ctrl->chunk_pages);
    if (magic != kPlanMagic || __ldcg(&ctrl->rows) != a.rows || __ldcg(&ctrl->kv_heads) != Hk ||
        __ldcg(&ctrl->pages_per_row) != a.pages_per_row || __ldcg(&ctrl->max_items) != a.L.max_items ||
        __ldcg(&ctrl->group) != g || __ldcg(&ctrl->head_dim) != D || chunk_pages < 1 ||
        chunk_pages > kChunkMax || n_items > a.L.max_items) {
        if (threadIdx.x == 0) set_error(ctrl, kErrBadPlan);
        return;
    }

    if (warp == kConsumerWarps) {
        // ================= producer =================
        int stage = 0;
        uint32_t phase = 0;
        uint32_t armed = 0;                 // bit s: stage s has an unfinished arm
        uint32_t armed_par = 0;             // parity armed on stage s
        bool ok = true;
        int it = 0;
        if (lane == 0) it = atomicAdd(&ctrl->next_item, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        while (ok && it < n_items) {
            int nxt = 0;
            if (lane == 0) nxt = atomicAdd(&ctrl->next_item, 1);
            const int2 item = __ldcg(items + it);
            const int row = item.x, kvh = item.y >> 16, chunk = item.y & 0xffff;
            bool good = row >= 0 && row < a.rows && kvh < Hk;
            int4 ri = make_int4(-1, 0, 0, 0);
            if (good) ri = __ldcg(row_info + row);
            const int pos = ri.x, lo = ri.y, nch = ri.z;
            const int slot = ri.w + kvh * nch + chunk;
            good = good && pos >= 0 && lo >= 0 && lo <= pos && chunk < nch &&
                   pos < a.pages_per_row * kPageSize && slot >= 0 && slot < n_items;
            if (!good) {
                if (lane == 0) set_error(ctrl, kErrBadPlan);
                it = __shfl_sync(0xffffffffu, nxt, 0);
                continue;
            }
            const int first_page = lo / kPageSize + chunk * chunk_pages;
            const int last_page = min(first_page + chunk_pages - 1, pos / kPageSize);
            const int npg = last_page - first_page + 1;
            const int* trow = a.table + (size_t)row * a.pages_per_row;
            const int pid0 = lane < npg ? __ldg(trow + first_page + lane) : -1;
            const int pid1 = lane + 32 < npg ? __ldg(trow + first_page + lane + 32) : -1;
            for (int j = 0; j < npg; ++j) {
                const int pid = __shfl_sync(0xffffffffu, j < 32 ? pid0 : pid1, j & 31);
                int waited = 1;
                if (lane == 0) waited = mbar_wait(bar_empty + 8 * stage, phase ^ 1) ? 1 : 0;
                waited = __shfl_sync(0xffffffffu, waited, 0);
                if (!waited) { ok = false; break; }
                if (lane == 0) {
                    const bool pvalid = pid >= 0 && pid < a.num_pages;
                    if (!pvalid) set_error(ctrl, kErrBadPage);
                    const int p = first_page + j, t0 = p * kPageSize;
                    Meta mt;
                    mt.row = row;
                    mt.kvh = kvh;
                    mt.nch = nch;
                    mt.slot = slot;
                    mt.t_lo = max(lo, t0) - t0;
                    mt.t_hi = min(pos, t0 + kPageSize - 1) - t0 + 1;
                    mt.flags = (j == 0 ? kFirst : 0) | (j == npg - 1 ? kLast : 0) | (pvalid ? kValid : 0) |
                               ((mt.t_lo > 0 || mt.t_hi < kPageSize) ? kPartial : 0);
                    mt.chunk = chunk;
                    meta[stage] = mt;
                    uint32_t bytes = (pvalid ? C::kStageBytes : 0) + (j == 0 ? g * D * C::kElem : 0);
                    const uint32_t fb = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(fb, bytes);
                    const uint32_t dst = sbase + stage * C::kStageBytes;
                    if (pvalid) {
                        const int y = (pid * Hk + kvh) * kPageSize;
                        #pragma unroll
                        for (int b = 0; b < C::kBoxes; ++b) {
                            tma_load_2d(dst + b * C::kBoxBytes, &k_map, b * C::kBoxCols, y, fb);
                            tma_load_2d(dst + C::kTileBytes + b * C::kBoxBytes, &v_map, b * C::kBoxCols, y, fb);
                        }
                    }
                    if (j == 0) {
                        const T* qsrc = static_cast<const T*>(a.q) + ((size_t)row * a.heads + kvh * g) * D;
                        bulk_load(sbase + C::kOffQ + stage * C::kQBytes, qsrc, g * D * C::kElem, fb);
                    }
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                }
                __syncwarp();
                if (++stage == S) { stage = 0; phase ^= 1; }
            }
            it = __shfl_sync(0xffffffffu, nxt, 0);
        }
        if (ok) {
            // Terminator: the next stage carries no data, only the end flag.
            int waited = 1;
            if (lane == 0) waited = mbar_wait(bar_empty + 8 * stage, phase ^ 1) ? 1 : 0;
            waited = __shfl_sync(0xffffffffu, waited, 0);
            if (waited && lane == 0) {
                meta[stage].flags = kTerm;
                mbar_arrive(bar_full + 8 * stage);
            }
            ok = waited != 0;
        }
        if (lane == 0) {
            if (ok) {
                // Last CTA to finish fetching rewinds the cursor for the next launch.
                __threadfence();
                if (atomicAdd(&ctrl->done_ctas, 1) == (int)gridDim.x - 1) {
                    ctrl->next_item = 0;
                    ctrl->done_ctas = 0;
                }
            } else {
                set_error(ctrl, kErrTimeout);
                // Let copies in flight land before the CTA's shared memory goes away.
                for (int s = 0; s < S; ++s)
                    if (armed & (1u << s)) mbar_wait(bar_full + 8 * s, (armed_par >> s) & 1u, 200000000ull);
            }
        }
        return;
    }

    // ================= consumers =================
    Consumer<T, D> cs;
    ConsumerSync csync{bar_sync, 0};
    int stage = 0;
    uint32_t phase = 0;
    const int tid = threadIdx.x;     // 0..127
    while (true) {
        if (!mbar_wait(bar_full + 8 * stage, phase)) {
            if (lane == 0) set_error(ctrl, kErrTimeout);
            break;
        }
        const Meta mt = meta[stage];
        if (mt.flags & kTerm) break;
        const uint32_t kbase = sbase + stage * C::kStageBytes;
        if (mt.flags & kFirst) {
            if constexpr (sizeof(T) == 2)
                cs.begin(sbase + C::kOffQ + stage * C::kQBytes, lane);
            else
                cs.begin(sbase + C::kOffQ + stage * C::kQBytes, sbase + C::kOffWarpQ + warp * C::kQBytes,
                         lane, g);
        }
        if (mt.flags & kValid)
            cs.page(kbase, kbase + C::kTileBytes, warp, lane, mt.t_lo, mt.t_hi, (mt.flags & kPartial) != 0,
                    a.scale_log2);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
        if (++stage == S) { stage = 0; phase ^= 1; }
        if (!(mt.flags & kLast)) continue;

        // ---- item done: merge the four warps
        cs.stash(sm_m, sm_l, sm_o, warp, lane);
        if (!csync.sync()) { if (lane == 0) set_error(ctrl, kErrTimeout); break; }
        const int row = mt.row, kvh = mt.kvh, nch = mt.nch, slot = mt.slot;
        const int units = D / 8;
        const int j = tid / units, d0 = (tid % units) * 8;
        if (j < g) {
            float M = kNegBig;
            #pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * kMaxGroup + j]);
            float L = 0.f, O[8];
            #pragma unroll
            for (int e = 0; e < 8; ++e) O[e] = 0.f;
            #pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = exp2_approx(sm_m[w * kMaxGroup + j] - M);
                L += f * sm_l[w * kMaxGroup + j];
                const float* src = sm_o + (w * kMaxGroup + j) * (D + 4) + d0;
                #pragma unroll
                for (int e = 0; e < 8; ++e) O[e] += f * src[e];
            }
            if (nch == 1) {
                const float inv = 1.f / L;
                #pragma unroll
                for (int e = 0; e < 8; ++e) O[e] *= inv;
                store8<T>(static_cast<T*>(a.out) + ((size_t)row * a.heads + kvh * g + j) * D + d0, O);
            } else {
                float* dst = part_o + ((size_t)slot * g + j) * D + d0;
                reinterpret_cast<float4*>(dst)[0] = make_float4(O[0], O[1], O[2], O[3]);
                reinterpret_cast<float4*>(dst)[1] = make_float4(O[4], O[5], O[6], O[7]);
                if (d0 == 0) part_ml[(size_t)slot * g + j] = make_float2(M, L);
            }
        }
        if (nch > 1) {
            __threadfence();
            if (!csync.sync()) { if (lane == 0) set_error(ctrl, kErrTimeout); break; }
            if (tid == 0) {
                const int done = atomicAdd(merge_cnt + (size_t)row * Hk + kvh, 1);
                *s_flag = (done == nch - 1);
                if (done == nch - 1) merge_cnt[(size_t)row * Hk + kvh] = 0;
            }
            if (!csync.sync()) { if (lane == 0) set_error(ctrl, kErrTimeout); break; }
            if (*s_flag && j < g) {
                // Last chunk of this (row, kv head) to finish: merge every
                // chunk's partial, out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c.
                __threadfence();
                const int slot0 = slot - mt.chunk;
                float M = kNegBig;
                for (int c = 0; c < nch; ++c) M = fmaxf(M, __ldcg(part_ml + (size_t)(slot0 + c) * g + j).x);
                float L = 0.f, O[8];
                #pragma unroll
                for (int e = 0; e < 8; ++e) O[e] = 0.f;
                for (int c = 0; c < nch; ++c) {
                    const float2 ml = __ldcg(part_ml + (size_t)(slot0 + c) * g + j);
                    const float f = exp2_approx(ml.x - M);
                    L += f * ml.y;
                    const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)(slot0 + c) * g + j) * D + d0);
                    const float4 u = __ldcg(src), v = __ldcg(src + 1);
                    O[0] += f * u.x; O[1] += f * u.y; O[2] += f * u.z; O[3] += f * u.w;
                    O[4] += f * v.x; O[5] += f * v.y; O[6] += f * v.z; O[7] += f * v.w;
                }
                const float inv = 1.f / L;
                #pragma unroll
                for (int e = 0; e < 8; ++e) O[e] *= inv;
                store8<T>(static_cast<T*>(a.out) + ((size_t)row * a.heads + kvh * g + j) * D + d0, O);
            }
        }
        if (!csync.sync()) { if (lane == 0) set_error(ctrl, kErrTimeout); break; }
    }
}

// ---------------------------------------------------------------------------
// Host launcher
// ---------------------------------------------------------------------------
template <typename T, int D>
static cudaError_t launch_one(const AttendArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                              int grid, bool programmatic, cudaStream_t stream) {
    using C = Cfg<T, D>;
    auto kern = attend_kernel<T, D>;
    // The shared-memory opt-in is per function and device; setting it again is cheap.
    static int configured_mask = 0;   // bit per device id < 31
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        if (dev < 31) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, k_map, v_map, a);
}

cudaError_t launch_attend(const AttendArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                          int dtype, int grid, bool programmatic, cudaStream_t stream) {
    if (dtype == 0 && a.head_dim == 128)
        return launch_one<__nv_bfloat16, 128>(a, k_map, v_map, grid, programmatic, stream);
    if (dtype == 0 && a.head_dim == 64)
        return launch_one<__nv_bfloat16, 64>(a, k_map, v_map, grid, programmatic, stream);
    if (dtype == 1 && a.head_dim == 128)
        return launch_one<float, 128>(a, k_map, v_map, grid, programmatic, stream);
    if (dtype == 1 && a.head_dim == 64)
        return launch_one<float, 64>(a, k_map, v_map, grid, programmatic, stream);
    return cudaErrorInvalidValue;
}

size_t attend_smem_bytes(int dtype, int head_dim) {
    if (dtype == 0) return head_dim == 128 ? Cfg<__nv_bfloat16, 128>::kSmem : Cfg<__nv_bfloat16, 64>::kSmem;
    return head_dim == 128 ? Cfg<float, 128>::kSmem : Cfg<float, 64>::kSmem;
}

}  // namespace pdattn
