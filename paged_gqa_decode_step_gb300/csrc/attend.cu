// Split-KV flash-decode attention over a paged KV cache.
//
// The operation is the `decode` body of GroupedQueryAttention on the Llama
// example page ("src/attention.linnet": `seen[s] = s <= pos`,
// `grouped_attention(q, cache_k, cache_v, rsqrt(f32(D)), seen)`), where each
// kv head serves Heads / KvHeads query heads ("Key ideas", grouped-query
// attention), with the cache addressed through the page table of the paged
// entries (llama-3.1-8b-instruct architecture page, `decode_paged`).
//
// Design (one persistent CTA per SM, 6 warps):
//   * warp 5 (scheduler) takes (row, kv head, chunk) items from the plan with
//     an atomic cursor, loads each item's descriptor and page ids, and queues
//     them in shared memory a few items ahead, so that no global-memory
//     latency sits between two TMA issues.
//   * warp 4 (producer) pops items and, for every page, issues TMA loads of
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
#include <type_traits>

#include "internal.h"

namespace pdattn {

// Consumer warps: four, each with 16 of a page's 64 tokens (the rows of the
// bf16 MMA tile; the f32 consumer uses the same split).
constexpr int kConsumerWarps = 4;
constexpr int kEpilogueWarps = 2;
constexpr int kItemSlots = 4;           // items the scheduler may hold ahead of the producer
constexpr int kBacklogBytes = 256 << 10;  // K/V bytes queued ahead of the TMA issue point
constexpr float kNegBig = -1.0e30f;     // running-max start: finite, so exp2(m - m) = 1
constexpr size_t kTablePrefetchMax = size_t(8) << 20;   // larger page tables are not prefetched

enum : int { kFirst = 1, kLast = 2, kTerm = 8 };

// Per-stage meta.  t_lo / t_hi: visible token range in stage coordinates
// (page p of the stage holds tokens [64 p, 64 p + 64)); flags: kFirst /
// kLast / kTerm, the number of pages in bits 8-11 and a valid bit per page
// from bit 16.
struct Meta {
    int row, kvh, nch, slot, t_lo, t_hi, flags, chunk;
};
constexpr int kPagesShift = 8;
constexpr int kValidShift = 16;

// Bytes from one query head to the next in a stage's query-group buffer:
// bf16 rows are padded by 16 bytes so that the eight row addresses of each
// ldmatrix fall in different banks; f32 rows stay packed.
template <typename T, int D>
__host__ __device__ constexpr int q_row_bytes() { return sizeof(T) == 2 ? D * 2 + 16 : D * (int)sizeof(T); }

template <typename T, int D, int G>
struct Cfg {
    // warp roles: consumers 0 .. kCW - 1, producer, scheduler, two epilogue warps
    static constexpr int kCW = kConsumerWarps;
    static constexpr int kProducer = kCW, kScheduler = kCW + 1, kEpilogue = kCW + 2;
    static constexpr int kThreads = (kCW + 2 + kEpilogueWarps) * 32;
    static constexpr int kElem = sizeof(T);
    static constexpr int kBoxCols = 128 / kElem;                 // columns per 128-byte box row
    static constexpr int kBoxes = D / kBoxCols;                  // boxes per K (or V) page
    static constexpr int kBoxBytes = kPageSize * 128;            // 8 KiB
    static constexpr int kTileBytes = kBoxes * kBoxBytes;        // one page of K (or V)
    // Small pages travel two to a stage, so the producer's per-stage work
    // (barrier, meta, arm) is spread over 32 KiB like the larger pages.
    static constexpr int kPagesPerStage = (kTileBytes == kBoxBytes && kElem == 2) ? 2 : 1;
    static constexpr int kStageBytes = 2 * kPagesPerStage * kTileBytes;   // K pages, then V pages
    static constexpr int kStages = (kStageBytes <= 16384) ? 10 : (kStageBytes <= 32768 ? 5 : 2);
    static constexpr int kQRow = q_row_bytes<T, D>();
    // bf16: eight head rows (the MMA's N; rows past the group stay zero); f32: G
    static constexpr int kQHeads = kElem == 2 ? kMaxGroup : G;
    static constexpr int kQBytes = kQHeads * kQRow;
    static constexpr int kORow = D + 4;                          // padded head row of a stashed output
    static constexpr int kOffQ = kStages * kStageBytes;
    static constexpr int kWarpQBytes = (kElem == 4 && G > 1) ? kCW * kQBytes : 0;  // f32: private copies
    static constexpr int kWarpPBytes = (kElem == 4) ? kCW * G * (64 / kCW) * 4 : 0;   // f32: p buffers
    static constexpr int kOffWarpQ = kOffQ + kStages * kQBytes;
    static constexpr int kOffWarpP = kOffWarpQ + kWarpQBytes;
    static constexpr int kOffItems = kOffWarpP + kWarpPBytes;    // kItemSlots x (ItemDesc + 64 page ids)
    static constexpr int kItemBytes = (int)sizeof(ItemDesc) + kChunkMax * 4;
    // Epilogue slots: Meta, then each consumer warp's (m, l) per head and
    // its O[head][kORow] (fp32, unnormalised); the epilogue warps merge the
    // four warps.  Two slots per epilogue warp at head dim 64, one at 128.
    static constexpr int kEpiSlots = D == 128 ? 2 : 4;
    static constexpr int kEpiHeads = kElem == 2 ? kMaxGroup : G;   // heads each warp stashes
    static constexpr int kEpiOffO = (int)sizeof(Meta) + kCW * kEpiHeads * 8;
    static constexpr int kEpiBytes = kEpiOffO + kCW * kEpiHeads * kORow * 4;
    static constexpr int kOffEpi = kOffItems + kItemSlots * kItemBytes;
    static constexpr int kOffMeta = kOffEpi + kEpiSlots * kEpiBytes;
    static constexpr int kOffBar = kOffMeta + kStages * (int)sizeof(Meta);
    static constexpr int kNumBars = 2 * kStages + 2 * kItemSlots + 2 * kEpiSlots;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;           // + alignment slack
    // pages the scheduler keeps queued beyond the producer's issue point
    static constexpr int kPageBytes = 2 * kTileBytes;                 // K and V of one page
    static constexpr int kBacklogPages = kBacklogBytes / kPageBytes > 2 ? kBacklogBytes / kPageBytes : 2;
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static_assert(kOffBar % 8 == 0, "mbarrier alignment");
    static_assert(kEpiOffO % 16 == 0 && kEpiBytes % 16 == 0 && kOffEpi % 16 == 0, "16-byte stash rows");
};


template <typename T>
__device__ __forceinline__ float load_f32(const void* base, int i);
template <>
__device__ __forceinline__ float load_f32<__nv_bfloat16>(const void* base, int i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}
template <>
__device__ __forceinline__ float load_f32<float>(const void* base, int i) {
    return static_cast<const float*>(base)[i];
}

// Final normalisation of one head's (M, L, O) (base-2 logits): with a sink
// logit s (natural units) the softmax denominator gains e^s, i.e. with
// M' = max(M, s log2 e): O e^(M - M') / (L e^(M - M') + e^(s log2 e - M')).
// Returns the factor to multiply O with.
__device__ __forceinline__ float out_scale(float M, float L, bool has_sink, float sink_log2) {
    if (!has_sink) return 1.f / L;
    const float Mp = fmaxf(M, sink_log2);
    const float f = exp2_approx(M - Mp);
    return f / (L * f + exp2_approx(sink_log2 - Mp));
}

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
template <typename T, int D, int G>
struct Consumer;

// bf16: tensor-core tiles (always 8 heads wide; G is unused).  Lane layout of the m16n8 accumulators:
// row = lane / 4 (+8), column pair = 2 * (lane % 4).
template <int D, int G>
struct Consumer<__nv_bfloat16, D, G> {
    static constexpr int KS = D / 16;     // k-steps over D for QK, m-tiles over D for PV
    uint32_t qf[KS][2];
    float o[KS][4];
    float m0, m1, l0, l1;                 // heads 2*(lane%4) and +1

    __device__ void begin(uint32_t qbuf, int lane) {
        // Q^T as the B operand: row = head, 8 dims per 16-byte chunk.
        #pragma unroll
        for (int p = 0; p < KS / 2; ++p) {
            const int head = lane & 7, chunk = 4 * p + (lane >> 3);
            ldsm_x4(qbuf + head * q_row_bytes<__nv_bfloat16, D>() + chunk * 16, qf[2 * p][0], qf[2 * p][1], qf[2 * p + 1][0],
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
            // Issue every K fragment load before the MMAs (the loads stay in
            // program order), then accumulate in two independent chains.
            uint32_t ka[KS][4];
            const int tok = tok0 + ri + ((mi & 1) << 3);
            #pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int chunk = ks * 2 + (mi >> 1);
                ldsm_x4(swz128(kbase + (chunk >> 3) * 8192, tok, chunk & 7), ka[ks][0], ka[ks][1], ka[ks][2],
                        ka[ks][3]);
            }
            float c2[4] = {0.f, 0.f, 0.f, 0.f};
            #pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (ks & 1) mma_bf16_16816(c2, ka[ks][0], ka[ks][1], ka[ks][2], ka[ks][3], qf[ks][0], qf[ks][1]);
                else mma_bf16_16816(c, ka[ks][0], ka[ks][1], ka[ks][2], ka[ks][3], qf[ks][0], qf[ks][1]);
            }
            #pragma unroll
            for (int i = 0; i < 4; ++i) c[i] += c2[i];
        }
        // ---- V^T fragments, loaded now so their latency overlaps the softmax
        uint32_t va_[KS][4];
        {
            const int tok = tok0 + ri + ((mi >> 1) << 3);
            #pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int chunk = mt * 2 + (mi & 1);
                ldsm_x4_trans(swz128(vbase + (chunk >> 3) * 8192, tok, chunk & 7), va_[mt][0], va_[mt][1],
                              va_[mt][2], va_[mt][3]);
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
        // ---- O^T += V^T P^T with the V^T tiles loaded above
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
        for (int mt = 0; mt < KS; ++mt)
            mma_bf16_16816(o[mt], va_[mt][0] & keep_a, va_[mt][1] & keep_a, va_[mt][2] & keep_b,
                           va_[mt][3] & keep_b, b0, b1);
    }

    // Put this warp's (m, l) per head (ml[8]) and o for heads 0..7
    // (ow[8][D + 4]) into an epilogue slot.
    __device__ void stash(float2* ml, float* ow, int lane) {
        float s0 = l0, s1 = l1;
        #pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, sh);
            s1 += __shfl_xor_sync(0xffffffffu, s1, sh);
        }
        const int h0 = 2 * (lane & 3);
        if (lane < 4) {
            ml[h0] = make_float2(m0, s0);
            ml[h0 + 1] = make_float2(m1, s1);
        }
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

// f32: FP32 FMAs.
//   scores: lane = (token tok0 + lane % 16, half of D lane / 16), the halves
//           summed with one shuffle;
//   values: lane = (token parity lane / 16, VD consecutive dimensions
//           (lane % 16) * VD), so each lane loads 16-byte pieces of V rows and
//           the two parities are summed once per item in stash().
// The probabilities go through a small per-warp buffer (read back as
// broadcast float4s).  G bounds the group at compile time; a one-head group
// keeps its query in registers.  The softmax is lazy: the running maximum is
// raised only when a score exceeds it by more than kLazyLog2 (one vote per
// page instead of a max reduction), so the weights stay below 2^kLazyLog2,
// and each lane keeps its own partial denominator, summed once per item.
constexpr float kLazyLog2 = 8.f;

template <int D, int G>
struct Consumer<float, D, G> {
    static constexpr int TPW = 64 / kConsumerWarps;   // tokens per warp
    static constexpr int NQ = 32 / TPW;       // lanes sharing one token's score (parts of D)
    static constexpr int DQ = D / NQ;         // dimensions per part
    static constexpr int VD = D / 16;          // value dimensions per lane
    static constexpr bool kQRegs = (G == 1);
    float o[G][VD];
    float m[G], l[G];
    float qr[kQRegs ? DQ : 1];
    const float* wq;       // this warp's copy of the query group [g][D] (G > 1)
    float* sp;             // this warp's probabilities [G][TPW]
    int g;

    __device__ void begin(const float* qbuf, float* warp_q, float* warp_p, int lane, int group) {
        g = group;
        sp = warp_p;
        if constexpr (kQRegs) {
            const int part = lane / TPW;
            #pragma unroll
            for (int i = 0; i < DQ / 4; ++i) {
                const float4 v = reinterpret_cast<const float4*>(qbuf + part * DQ)[i];
                qr[4 * i] = v.x; qr[4 * i + 1] = v.y; qr[4 * i + 2] = v.z; qr[4 * i + 3] = v.w;
            }
            wq = nullptr;
        } else {
            // The stage's query buffer can be refilled for a later item while
            // this item is still running, so each warp keeps its own copy.
            wq = warp_q;
            for (int i = lane; i < group * D / 4; i += 32)
                reinterpret_cast<float4*>(warp_q)[i] = reinterpret_cast<const float4*>(qbuf)[i];
            __syncwarp();
        }
        #pragma unroll
        for (int j = 0; j < G; ++j) {
            m[j] = kNegBig;
            l[j] = 0.f;
            #pragma unroll
            for (int e = 0; e < VD; ++e) o[j][e] = 0.f;
        }
    }

    __device__ void page(const uint8_t* kbase, const uint8_t* vbase, int warp, int lane, int t_lo, int t_hi,
                         bool partial, float sl2) {
        const int tok0 = warp * TPW;
        const int tl = lane % TPW, qp = lane / TPW, t = tok0 + tl;
        // Independent partial sums per head (NA of them) keep the dot
        // product's FMA chain short; they are added once at the end.
        constexpr int NA = G == 1 ? 4 : (G == 2 ? 2 : 1);
        float part[G][NA];
        #pragma unroll
        for (int j = 0; j < G; ++j)
            #pragma unroll
            for (int a = 0; a < NA; ++a) part[j][a] = 0.f;
        // full unroll when the query sits in registers (its index must be static)
        #pragma unroll (G >= 4 ? 2 : DQ / 4)
        for (int c = 0; c < DQ / 4; ++c) {
            const int col = qp * DQ + c * 4;                 // first dimension of the chunk
            const float4 kv = *reinterpret_cast<const float4*>(kbase + swz128((col / 32) * 8192, t, (col % 32) / 4));
            #pragma unroll
            for (int j = 0; j < G; ++j) {
                if (j < g) {
                    float4 qv;
                    if constexpr (kQRegs) qv = make_float4(qr[4 * c], qr[4 * c + 1], qr[4 * c + 2], qr[4 * c + 3]);
                    else qv = *reinterpret_cast<const float4*>(wq + j * D + col);
                    float& pa = part[j][c % NA];
                    pa = fmaf(kv.x, qv.x, pa);
                    pa = fmaf(kv.y, qv.y, pa);
                    pa = fmaf(kv.z, qv.z, pa);
                    pa = fmaf(kv.w, qv.w, pa);
                }
            }
        }
        float acc[G];
        #pragma unroll
        for (int j = 0; j < G; ++j) {
            acc[j] = part[j][0];
            #pragma unroll
            for (int a = 1; a < NA; ++a) acc[j] += part[j][a];
        }
        const bool valid = t >= t_lo && t < t_hi;
        #pragma unroll
        for (int j = 0; j < G; ++j) {
            if (j < g) {
                float sc = acc[j];
                #pragma unroll
                for (int sh = TPW; sh < 32; sh <<= 1) sc += __shfl_xor_sync(0xffffffffu, sc, sh);
                sc = valid ? sc * sl2 : -INFINITY;
                if (__any_sync(0xffffffffu, sc > m[j] + kLazyLog2)) {
                    float x = sc;
                    #pragma unroll
                    for (int sh = 1; sh < TPW; sh <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, sh));
                    const float n = fmaxf(m[j], x);
                    const float al = exp2_approx(m[j] - n);
                    m[j] = n;
                    l[j] *= al;
                    #pragma unroll
                    for (int e = 0; e < VD; ++e) o[j][e] *= al;
                }
                const float pj = exp2_approx(sc - m[j]);
                if (qp == 0) l[j] += pj;            // this lane's token; summed over lanes in stash()
                // token tl goes to slot parity * TPW / 2 + index within its parity
                if (qp == 0) sp[j * TPW + (tl & 1) * (TPW / 2) + (tl >> 1)] = pj;
            }
        }
        __syncwarp();
        const int par = lane >> 4, dg = (lane & 15) * VD;
        #pragma unroll
        for (int k = 0; k < TPW / 2; ++k) {
            const int row = tok0 + 2 * k + par;
            float v[VD];
            #pragma unroll
            for (int q4 = 0; q4 < VD / 4; ++q4) {
                const int col = dg + 4 * q4;
                const float4 w4 = *reinterpret_cast<const float4*>(vbase + swz128((col / 32) * 8192, row, (col % 32) / 4));
                v[4 * q4] = w4.x; v[4 * q4 + 1] = w4.y; v[4 * q4 + 2] = w4.z; v[4 * q4 + 3] = w4.w;
            }
            if (partial) {
                // invisible tokens have p = 0, but their slots may hold NaN
                const bool vis = row >= t_lo && row < t_hi;
                #pragma unroll
                for (int e = 0; e < VD; ++e) v[e] = vis ? v[e] : 0.f;
            }
            #pragma unroll
            for (int j = 0; j < G; ++j) {
                if (j < g) {
                    const float pk = sp[j * TPW + par * (TPW / 2) + k];
                    #pragma unroll
                    for (int e = 0; e < VD; ++e) o[j][e] = fmaf(pk, v[e], o[j][e]);
                }
            }
        }
        __syncwarp();   // sp is rewritten by the next page
    }

    __device__ void stash(float2* ml, float* ow, int lane) {
        #pragma unroll
        for (int j = 0; j < G; ++j) {
            if (j < g) {
                float lt = l[j];
                #pragma unroll
                for (int sh = 1; sh < 32; sh <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, sh);
                if (lane == 0) ml[j] = make_float2(m[j], lt);
                #pragma unroll
                for (int e = 0; e < VD; ++e) {
                    const float tot = o[j][e] + __shfl_xor_sync(0xffffffffu, o[j][e], 16);
                    if (lane < 16) ow[j * (D + 4) + lane * VD + e] = tot;
                }
            }
        }
    }
};

// ---------------------------------------------------------------------------
// The first-wave item of CTA b (chunk 0 of (row, kv head) pair b), derived
// from the call's inputs exactly as the planner derives it: the positions
// and windows give every row's visible pages, their total and maximum give
// the split size, and the merge slot starts at the prefix sum of nch *
// kv_heads over the rows before.  Whole warp.  Returns false for a row
// whose position is out of range (the planner leaves an empty item there).
// ---------------------------------------------------------------------------
template <typename Lay>
__device__ bool first_wave_item(const AttendArgs& a, const Lay& lay, int b, int lane, int grid, int4* d0, int4* d1) {
    constexpr bool kMulti = std::is_same<Lay, AttendLayers>::value;
    const int Hk = a.kv_heads, max_pos = a.pages_per_row * kPageSize;
    auto pages_of = [&](int v, int* pos_out, int* lo_out) -> int {
        const int pos = __ldg(a.positions + (kMulti ? v % a.layer_rows : v));
        if (pos < 0 || pos >= max_pos) return 0;
        int w = a.window;
        if constexpr (kMulti) w = lay.window[v / a.layer_rows];
        const int lo = row_lo(pos, w);
        *pos_out = pos;
        *lo_out = lo;
        return pos / kPageSize - lo / kPageSize + 1;
    };
    int pos = 0, lo = 0;
    unsigned long long tot = 0;
    int longest = 0;
    for (int v = lane; v < a.rows; v += 32) {
        const int n = pages_of(v, &pos, &lo);
        tot += (unsigned long long)n;
        longest = max(longest, n);
    }
    #pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, sh);
    longest = (int)__reduce_max_sync(0xffffffffu, (unsigned)longest);
    const int C = a.chunk_pages > 0 ? a.chunk_pages : choose_chunk(tot, longest, a.rows, Hk, grid);
    const int row = b / Hk, kvh = b % Hk;
    int part = 0;
    for (int v = lane; v < row; v += 32) part += Chunking(pages_of(v, &pos, &lo), C).nch;
    part = (int)__reduce_add_sync(0xffffffffu, (unsigned)part);
    const int n = pages_of(row, &pos, &lo);
    if (n == 0) return false;
    const Chunking ch(n, C);
    *d0 = make_int4(row, kvh << 16, ch.nch, part * Hk + kvh * ch.nch);
    *d1 = make_int4(lo / kPageSize, ch.size(0), pos, lo);
    return true;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <typename T, int D, int G, typename Lay>
__global__ void __launch_bounds__(Cfg<T, D, G>::kThreads, 1)
attend_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
              const __grid_constant__ AttendArgs a, const __grid_constant__ Lay lay) {
    using C = Cfg<T, D, G>;
    constexpr int kThreads = C::kThreads, kCW = C::kCW;
    constexpr int kProducerWarp = C::kProducer, kSchedulerWarp = C::kScheduler, kEpilogueWarp = C::kEpilogue;
    // Multi-layer launch: item row v is row v % layer_rows of layer
    // v / layer_rows, whose pools, output and sinks come from `lay`.
    constexpr bool kMulti = std::is_same<Lay, AttendLayers>::value;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::kOffBar;             // S barriers: stage holds data
    const uint32_t bar_empty = bar_full + 8 * S;              // S barriers: stage may be refilled
    const uint32_t bar_ifull = bar_empty + 8 * S;             // kItemSlots: item queued
    const uint32_t bar_iempty = bar_ifull + 8 * kItemSlots;   // kItemSlots: item slot free
    const uint32_t bar_efull = bar_iempty + 8 * kItemSlots;   // C::kEpiSlots: finished item queued
    const uint32_t bar_eempty = bar_efull + 8 * C::kEpiSlots; // C::kEpiSlots: epilogue slot free
    Meta* meta = reinterpret_cast<Meta*>(smem + C::kOffMeta);
    int* s_flag = reinterpret_cast<int*>(smem + C::kOffMisc);
    volatile int* s_issued = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);  // pages issued so far
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);   // 1: the plan was refused
    volatile int* s_early = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 12);  // 1: item 0 queued before the wait
    uint8_t* item_q = smem + C::kOffItems;
    uint8_t* epi_q = smem + C::kOffEpi;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kCW);
        }
        *s_issued = 0;
        *s_abort = 0;
        *s_early = 0;
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(bar_ifull + 8 * s, 1);
            mbar_init(bar_iempty + 8 * s, 1);
        }
        for (int s = 0; s < C::kEpiSlots; ++s) {
            mbar_init(bar_efull + 8 * s, kCW * 32);
            mbar_init(bar_eempty + 8 * s, 1);
        }
        fence_barrier_init();
    }
    // Query-group buffers: rows past the group stay zero.
    for (int i = threadIdx.x; i < S * C::kQBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + C::kOffQ)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_shared();
    if constexpr (kMulti) {
        if (warp == kProducerWarp && lane < a.n_layers) {
            prefetch_tensormap(&lay.k[lane]);
            prefetch_tensormap(&lay.v[lane]);
        }
    } else if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
    }
    if (warp == kSchedulerWarp) {
        // The page table is an input of the call (no launch of this call
        // writes it): pull it into L2 while the preceding launch finishes, so
        // that the page-id reads after the wait below hit L2.
        const size_t tbytes = (size_t)(kMulti ? a.layer_rows : a.rows) * a.pages_per_row * sizeof(int);
        if (tbytes <= kTablePrefetchMax) {
            const char* tb = reinterpret_cast<const char*>(a.table);
            for (size_t off = ((size_t)blockIdx.x * 32 + lane) * 128; off < tbytes; off += (size_t)gridDim.x * 32 * 128)
                prefetch_l2(tb + off);
        }
    }
    __syncthreads();

    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    const ItemDesc* items = reinterpret_cast<const ItemDesc*>(a.ws + a.L.items);
    int* merge_cnt = reinterpret_cast<int*>(a.ws + a.L.merge_cnt);
    float2* part_ml = reinterpret_cast<float2*>(a.ws + a.L.part_ml);
    float* part_o = reinterpret_cast<float*>(a.ws + a.L.part_o);
    const int g = a.group, Hk = a.kv_heads;
    const int nf = first_wave(a.rows, Hk, gridDim.x);

    // The plan header in one round trip: four independent 16-byte loads
    // (fields status .. test_hold; see Ctrl), checked in registers.  Only
    // after the wait for the preceding launch (the planner's).
    auto read_plan = [&](int* n_items, int* chunk_pages) -> bool {
        const int4 h0 = __ldcg(reinterpret_cast<const int4*>(ctrl));
        const int4 h1 = __ldcg(reinterpret_cast<const int4*>(ctrl) + 1);
        const int4 h2 = __ldcg(reinterpret_cast<const int4*>(ctrl) + 2);
        const int4 h3 = __ldcg(reinterpret_cast<const int4*>(ctrl) + 3);
        *n_items = h0.w;
        *chunk_pages = h1.x;
        return (uint32_t)h1.y == kPlanMagic && h1.z == a.rows && h1.w == Hk && h2.x == a.pages_per_row &&
               h2.y == a.L.max_items && h2.z == g && h2.w == D && h3.x == (int)gridDim.x && h1.x >= 1 &&
               h1.x <= kChunkMax && h0.w <= a.L.max_items;
    };

    if (warp == kSchedulerWarp) {
        // ================= scheduler =================
        // Item slot layout: ItemDesc (npg < 0 marks the end, 0 an empty
        // item), then 64 page ids.
        int islot = 0;
        uint32_t iphase = 0;
        bool ok = true;
        int queued = 0;                     // pages handed to the producer so far
        auto queue_item = [&](int4 d0, int4 d1, int pid0, int pid1) -> bool {
            int waited = 1;
            if (lane == 0) waited = mbar_wait(bar_iempty + 8 * islot, iphase ^ 1) ? 1 : 0;
            waited = __shfl_sync(0xffffffffu, waited, 0);
            if (!waited) return false;
            uint8_t* slotp = item_q + islot * C::kItemBytes;
            if (lane == 0) {
                reinterpret_cast<int4*>(slotp)[0] = d0;
                reinterpret_cast<int4*>(slotp)[1] = d1;
            }
            int* pids = reinterpret_cast<int*>(slotp + sizeof(ItemDesc));
            pids[lane] = pid0;
            pids[lane + 32] = pid1;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ifull + 8 * islot);
            if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
            return true;
        };
        auto load_pids = [&](int row, int first, int npg, int* pid0, int* pid1) {
            const int trow_i = kMulti ? row % a.layer_rows : row;
            const int* trow = a.table + (size_t)trow_i * a.pages_per_row + first;
            *pid0 = lane < npg ? __ldg(trow + lane) : -1;
            *pid1 = lane + 32 < npg ? __ldg(trow + lane + 32) : -1;
        };
        // The first-wave item comes from the call's inputs (positions, the
        // table), which no launch of this call writes: it is queued before
        // the wait, so that its pages load while the planner and the rope
        // launch finish.
        int4 sd0 = make_int4(0, 0, 0, 0), sd1 = make_int4(0, 0, 0, 0);
        bool static_item = false;
        if ((int)blockIdx.x < nf) {
            static_item = first_wave_item(a, lay, (int)blockIdx.x, lane, (int)gridDim.x, &sd0, &sd1);
            if (static_item) {
                int pid0, pid1;
                load_pids(sd0.x, sd1.x, sd1.y, &pid0, &pid1);
                if (lane == 0) *s_early = 1;   // published by the item barrier's arrival
                ok = queue_item(sd0, sd1, pid0, pid1);
                queued += sd1.y;
            }
        }

        // Everything below reads what the preceding launch wrote.
        griddep_wait();
        int4 first_d0 = make_int4(0, 0, 0, 0), first_d1 = make_int4(0, 0, 0, 0);
        if ((int)blockIdx.x < a.L.max_items) {
            first_d0 = __ldcg(reinterpret_cast<const int4*>(items + blockIdx.x));
            first_d1 = __ldcg(reinterpret_cast<const int4*>(items + blockIdx.x) + 1);
        }
        int n_items = 0, chunk_pages = 0;
        const bool plan_ok = read_plan(&n_items, &chunk_pages);
        if (!plan_ok || !ok) {
            if (lane == 0) {
                if (!plan_ok) set_error(ctrl, kErrBadPlan);
                else fail_timeout(ctrl);
                *s_abort = 1;
            }
            // let the producer leave its item wait at once
            queue_item(make_int4(0, 0, 0, 0), make_int4(0, -1, 0, 0), -1, -1);
            return;
        }
        if (static_item) {
            // the planner's item b must be the one derived above
            const bool same = first_d0.x == sd0.x && first_d0.y == sd0.y && first_d0.z == sd0.z &&
                              first_d0.w == sd0.w && first_d1.x == sd1.x && first_d1.y == sd1.y &&
                              first_d1.z == sd1.z && first_d1.w == sd1.w && (int)blockIdx.x < n_items;
            if (!same && lane == 0) set_error(ctrl, kErrBadPlan);
        }
        bool first = !static_item;
        while (true) {
            int it = (int)blockIdx.x;
            if (!first) {
                // Reserve the next item only when fewer than kBacklogPages
                // queued pages wait to be issued: short items pipeline, long
                // ones do not hold back work other CTAs could take.
                if (lane == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (queued - *s_issued >= C::kBacklogPages) {
                        __nanosleep(32);
                        if (globaltimer_ns() - t0 > 2000000000ull) { ok = false; break; }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (lane == 0) it = atomicAdd(&ctrl->next_item, 1);
                it = __shfl_sync(0xffffffffu, it, 0);
            }
            const bool term = it >= n_items;
            int4 d0 = make_int4(0, 0, 0, 0), d1 = make_int4(0, -1, 0, 0);
            int pid0 = -1, pid1 = -1;
            bool good = true;
            if (!term) {
                if (first) {
                    d0 = first_d0;
                    d1 = first_d1;
                } else {
                    d0 = __ldcg(reinterpret_cast<const int4*>(items + it));
                    d1 = __ldcg(reinterpret_cast<const int4*>(items + it) + 1);
                }
                if (d1.y == 0) { first = false; continue; }   // an empty first-wave item (a bad row)
                const int row = d0.x, kvh = d0.y >> 16, chunk = d0.y & 0xffff, nch = d0.z, slot = d0.w;
                const int first = d1.x, npg = d1.y, pos = d1.z, lo = d1.w;
                good = row >= 0 && row < a.rows && kvh < Hk && chunk < nch && slot >= 0 && slot < n_items &&
                       npg >= 1 && npg <= chunk_pages && first >= 0 && pos >= 0 && lo >= 0 && lo <= pos &&
                       pos < a.pages_per_row * kPageSize && first + npg - 1 <= pos / kPageSize &&
                       first >= lo / kPageSize;
                if (good) load_pids(row, first, npg, &pid0, &pid1);
                else if (lane == 0) set_error(ctrl, kErrBadPlan);
            }
            first = false;
            if (!good) continue;
            if (term) d1.y = -1;
            if (!queue_item(d0, d1, pid0, pid1)) { ok = false; break; }
            if (term) break;
            queued += d1.y;
        }
        if (lane == 0) {
            if (!ok) fail_timeout(ctrl);
            // The last CTA to finish fetching rewinds the cursor for the next
            // launch (after a timeout too: every scheduler has left its loop).
            __threadfence();
            if (atomicAdd(&ctrl->done_ctas, 1) == (int)gridDim.x - 1) {
                ctrl->next_item = (int)gridDim.x;
                ctrl->done_ctas = 0;
            }
        }
        return;
    }

    if (warp == kProducerWarp) {
        // ================= producer =================
        // One lane runs the page loop: per page it waits for a free stage,
        // writes the stage's meta, arms the full barrier and issues the TMA
        // copies.  No warp-wide collectives sit in the loop.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int islot = 0;
            uint32_t iphase = 0;
            uint32_t armed = 0;                 // bit s: stage s has an unfinished arm
            uint32_t armed_par = 0;             // parity armed on stage s
            int issued = 0;
            bool ok = true, aborted = false;
            // test hook, written (if at all) before the call
            bool hold = blockIdx.x == 0 && __ldcg(&ctrl->test_hold) != 0;
            // Until the wait for the preceding launch, only the first-wave
            // item's pages are loaded: not the row's last page (this call
            // writes a slot there) and not its rotated queries (the rope
            // launch writes them), and no more stages than the ring holds.
            bool dep = false;
            bool q_pending = false;
            uint32_t q_dst = 0, q_bar = 0;
            const T* q_src = nullptr;
            int pre_stages = 0;
            bool first_item = true;
            auto issue_q = [&](uint32_t qdst, const T* qsrc, uint32_t fb) {
                if constexpr (C::kQRow == D * C::kElem) {
                    bulk_load(qdst, qsrc, g * D * C::kElem, fb);
                } else {
                    for (int h = 0; h < g; ++h) bulk_load(qdst + h * C::kQRow, qsrc + h * D, D * C::kElem, fb);
                }
            };
            auto resolve = [&]() {
                if (dep) return;
                griddep_wait();
                dep = true;
                int n_items, chunk_pages;
                if (!read_plan(&n_items, &chunk_pages)) aborted = true;   // the scheduler reports it
                // Issued even for a refused plan (the source lies inside the
                // rotated queries either way), so that every armed stage
                // completes and can be waited for before the CTA exits.
                if (q_pending) issue_q(q_dst, q_src, q_bar);
                q_pending = false;
            };
            while (ok && !aborted) {
                if (!mbar_wait(bar_ifull + 8 * islot, iphase)) { ok = false; break; }
                const uint8_t* slotp = item_q + islot * C::kItemBytes;
                const int4 d0 = reinterpret_cast<const int4*>(slotp)[0];
                const int4 d1 = reinterpret_cast<const int4*>(slotp)[1];
                const int* pids = reinterpret_cast<const int*>(slotp + sizeof(ItemDesc));
                const int npg = d1.y;
                if (npg < 0) break;             // end of the work
                const int row = d0.x, kvh = d0.y >> 16, chunk = d0.y & 0xffff, nch = d0.z, slot = d0.w;
                const int first_page = d1.x, pos = d1.z, lo = d1.w;
                const int y_kv = kvh * kPageSize;
                const T* qsrc = static_cast<const T*>(a.q) + ((size_t)row * a.heads + kvh * g) * D;
                const CUtensorMap* km = &k_map;
                const CUtensorMap* vm = &v_map;
                if constexpr (kMulti) {
                    const int l = row / a.layer_rows;
                    km = &lay.k[l];
                    vm = &lay.v[l];
                }
                if (!(first_item && *s_early)) resolve();   // only the first-wave item starts early
                first_item = false;
                if (aborted) break;
                constexpr int P = C::kPagesPerStage;
                const int last_page = pos / kPageSize;   // holds this call's new slot
                for (int j = 0; j < npg; j += P) {
                    const int np = min(P, npg - j);
                    if (!dep && (pre_stages >= S || first_page + j + np - 1 >= last_page)) resolve();
                    if (aborted) break;
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1)) { ok = false; break; }
                    if (hold) {
                        // test hook: this stage is never armed nor filled
                        hold = false;
                        if (!dep) ++pre_stages;
                        if (++stage == S) { stage = 0; phase ^= 1; }
                        continue;
                    }
                    const int t0 = (first_page + j) * kPageSize;
                    const int t_lo = max(lo, t0) - t0;
                    const int t_hi = min(pos, t0 + np * kPageSize - 1) - t0 + 1;
                    int flags = (j == 0 ? kFirst : 0) | (j + np == npg ? kLast : 0) | (np << kPagesShift);
                    uint32_t bytes = (j == 0 ? g * D * C::kElem : 0);
                    const uint32_t fb = bar_full + 8 * stage;
                    const uint32_t dst = sbase + stage * C::kStageBytes;
                    int pidv[P];
                    #pragma unroll
                    for (int p = 0; p < P; ++p) {
                        pidv[p] = p < np ? pids[j + p] : -1;
                        if (p < np && pidv[p] >= 0 && pidv[p] < a.num_pages) {
                            flags |= 1 << (kValidShift + p);
                            bytes += 2 * C::kTileBytes;
                        } else if (p < np) {
                            set_error(ctrl, kErrBadPage);
                        }
                    }
                    int4* mp = reinterpret_cast<int4*>(meta + stage);
                    mp[0] = make_int4(row, kvh, nch, slot);
                    mp[1] = make_int4(t_lo, t_hi, flags, chunk);
                    mbar_arrive_expect_tx(fb, bytes);
                    #pragma unroll
                    for (int p = 0; p < P; ++p) {
                        if (flags & (1 << (kValidShift + p))) {
                            const int y = pidv[p] * Hk * kPageSize + y_kv;
                            #pragma unroll
                            for (int bx = 0; bx < C::kBoxes; ++bx) {
                                tma_load_2d(dst + p * C::kTileBytes + bx * C::kBoxBytes, km, bx * C::kBoxCols, y, fb);
                                tma_load_2d(dst + (P + p) * C::kTileBytes + bx * C::kBoxBytes, vm, bx * C::kBoxCols, y,
                                            fb);
                            }
                        }
                    }
                    if (j == 0) {
                        const uint32_t qdst = sbase + C::kOffQ + stage * C::kQBytes;
                        if (dep) {
                            issue_q(qdst, qsrc, fb);
                        } else {
                            q_pending = true;
                            q_dst = qdst;
                            q_src = qsrc;
                            q_bar = fb;
                        }
                    }
                    if (!dep) ++pre_stages;
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    issued += np;
                    *s_issued = issued;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
                if (!ok || aborted) break;
                resolve();   // later items come after the wait
                if (aborted) break;
                mbar_arrive(bar_iempty + 8 * islot);
                if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
            }
            if (ok && !aborted) {
                // Terminator: the next stage carries no data, only the end flag.
                if (mbar_wait(bar_empty + 8 * stage, phase ^ 1)) {
                    meta[stage].flags = kTerm;
                    mbar_arrive(bar_full + 8 * stage);
                } else {
                    ok = false;
                }
            }
            if (!ok || aborted) {
                if (!ok) fail_timeout(ctrl);
                resolve();   // issues a pending query copy, so that its stage completes
                // Let the copies in flight land before the CTA's shared memory
                // goes away (after a refused plan the consumers have left and
                // nothing reads them).
                for (int s2 = 0; s2 < S; ++s2)
                    if (armed & (1u << s2)) mbar_wait(bar_full + 8 * s2, (armed_par >> s2) & 1u, 200000000ull);
            }
        }
        __syncwarp();
        return;
    }

    // Consumers and epilogue: everything below reads what the preceding
    // launch wrote.
    griddep_wait();
    {
        int n_items, chunk_pages;
        if (!read_plan(&n_items, &chunk_pages)) return;   // the scheduler reports it
    }

    if (warp >= kEpilogueWarp) {
        // ================= epilogue =================
        // Writes finished items: the output when the (row, kv head) is one
        // chunk, else the chunk's fp32 partial; the last chunk of a (row, kv
        // head) to arrive merges every partial and writes the output.  Two
        // warps share the slots (warp e takes slots e, e + 2, ...), so one
        // item's atomic and merge reads overlap the next item's work.
        static_assert(C::kEpiSlots % kEpilogueWarps == 0, "epilogue slots split evenly over the warps");
        const int ew = warp - kEpilogueWarp;
        int eslot = ew;
        uint32_t ephase = 0;
        while (true) {
            int waited = 1;
            if (lane == 0) waited = mbar_wait(bar_efull + 8 * eslot, ephase) ? 1 : 0;
            waited = __shfl_sync(0xffffffffu, waited, 0);
            if (!waited) { if (lane == 0) fail_timeout(ctrl); break; }
            const uint8_t* ep = epi_q + eslot * C::kEpiBytes;
            const Meta mt = *reinterpret_cast<const Meta*>(ep);
            if (mt.flags & kTerm) break;
            const float2* eml = reinterpret_cast<const float2*>(ep + sizeof(Meta));   // [warp][head]
            const float* eo = reinterpret_cast<const float*>(ep + C::kEpiOffO);        // [warp][head][kORow]
            // The four consumer warps' (m, l, o) of head j, dims d0 .. d0 + 7,
            // merged: M = max m_w, L = sum e^(m_w - M) l_w, O = sum e^(m_w - M) o_w.
            auto merge4 = [&](int j, int d0, float& M, float& L, float (&O)[8]) {
                M = kNegBig;
                #pragma unroll
                for (int w = 0; w < kCW; ++w) M = fmaxf(M, eml[w * C::kEpiHeads + j].x);
                L = 0.f;
                #pragma unroll
                for (int e = 0; e < 8; ++e) O[e] = 0.f;
                #pragma unroll
                for (int w = 0; w < kCW; ++w) {
                    const float2 ml = eml[w * C::kEpiHeads + j];
                    const float f = exp2_approx(ml.x - M);
                    L += f * ml.y;
                    const float4* src = reinterpret_cast<const float4*>(eo + (w * C::kEpiHeads + j) * C::kORow + d0);
                    const float4 p0 = src[0], p1 = src[1];
                    O[0] += f * p0.x; O[1] += f * p0.y; O[2] += f * p0.z; O[3] += f * p0.w;
                    O[4] += f * p1.x; O[5] += f * p1.y; O[6] += f * p1.z; O[7] += f * p1.w;
                }
            };
            const int row = mt.row, kvh = mt.kvh, nch = mt.nch, slot = mt.slot;
            T* out_base = static_cast<T*>(a.out) + ((size_t)row * a.heads + kvh * g) * D;
            const void* sinks = a.sinks;
            if constexpr (kMulti) {
                const int l = row / a.layer_rows;
                out_base = static_cast<T*>(lay.out[l]) + ((size_t)(row - l * a.layer_rows) * a.heads + kvh * g) * D;
                sinks = lay.sinks[l];
            }
            const bool has_sink = sinks != nullptr;
            if (nch == 1) {
                for (int u = lane; u < g * D / 8; u += 32) {
                    const int j = u / (D / 8), d0 = (u % (D / 8)) * 8;
                    float M, L, O[8];
                    merge4(j, d0, M, L, O);
                    const float sk = has_sink ? load_f32<T>(sinks, kvh * g + j) * 1.4426950408889634f : 0.f;
                    const float inv = out_scale(M, L, has_sink, sk);
                    #pragma unroll
                    for (int e = 0; e < 8; ++e) O[e] *= inv;
                    store8<T>(out_base + j * D + d0, O);
                }
            } else {
                for (int u = lane; u < g * D / 8; u += 32) {
                    const int j = u / (D / 8), d0 = (u % (D / 8)) * 8;
                    float M, L, O[8];
                    merge4(j, d0, M, L, O);
                    float4* dst = reinterpret_cast<float4*>(part_o + ((size_t)slot * g + j) * D + d0);
                    dst[0] = make_float4(O[0], O[1], O[2], O[3]);
                    dst[1] = make_float4(O[4], O[5], O[6], O[7]);
                    if (d0 == 0) part_ml[(size_t)slot * g + j] = make_float2(M, L);
                }
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    // Release this chunk's partial and, for the last chunk to
                    // arrive, acquire every other chunk's (one acq_rel atomic).
                    const int done = atomic_add_acq_rel_gpu(merge_cnt + (size_t)row * Hk + kvh, 1);
                    last = done == nch - 1;
                    if (last) merge_cnt[(size_t)row * Hk + kvh] = 0;   // ready for the next launch
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                __syncwarp();
                if (last) {
                    // out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c over the chunks
                    const int slot0 = slot - mt.chunk;
                    for (int u = lane; u < g * D / 8; u += 32) {
                        const int j = u / (D / 8), d0 = (u % (D / 8)) * 8;
                        // one pass with a running maximum, so the loads of
                        // every chunk go out together
                        float M = kNegBig, L = 0.f, O[8];
                        #pragma unroll
                        for (int e = 0; e < 8; ++e) O[e] = 0.f;
                        #pragma unroll 4
                        for (int c = 0; c < nch; ++c) {
                            const float2 ml = __ldcg(part_ml + (size_t)(slot0 + c) * g + j);
                            const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)(slot0 + c) * g + j) * D + d0);
                            const float4 p0 = __ldcg(src), p1 = __ldcg(src + 1);
                            const float Mn = fmaxf(M, ml.x);
                            const float fa = exp2_approx(M - Mn), f = exp2_approx(ml.x - Mn);
                            M = Mn;
                            L = L * fa + f * ml.y;
                            O[0] = O[0] * fa + f * p0.x; O[1] = O[1] * fa + f * p0.y;
                            O[2] = O[2] * fa + f * p0.z; O[3] = O[3] * fa + f * p0.w;
                            O[4] = O[4] * fa + f * p1.x; O[5] = O[5] * fa + f * p1.y;
                            O[6] = O[6] * fa + f * p1.z; O[7] = O[7] * fa + f * p1.w;
                        }
                        const float sk = has_sink ? load_f32<T>(sinks, kvh * g + j) * 1.4426950408889634f : 0.f;
                        const float inv = out_scale(M, L, has_sink, sk);
                        #pragma unroll
                        for (int e = 0; e < 8; ++e) O[e] *= inv;
                        store8<T>(out_base + j * D + d0, O);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_eempty + 8 * eslot);
            eslot += kEpilogueWarps;
            if (eslot >= C::kEpiSlots) { eslot -= C::kEpiSlots; ephase ^= 1; }
        }
        return;
    }

    // ================= consumers =================
    Consumer<T, D, G> cs;
    int stage = 0;
    uint32_t phase = 0;
    int eslot = 0;
    uint32_t ephase = 0;
    const int tid = threadIdx.x;     // 0 .. kCW * 32 - 1
    bool ok = true;
    while (true) {
        if (!mbar_wait(bar_full + 8 * stage, phase)) {
            if (lane == 0) fail_timeout(ctrl);
            ok = false;
            break;
        }
        const Meta mt = meta[stage];
        if (mt.flags & kTerm) break;
        const uint32_t kbase = sbase + stage * C::kStageBytes;
        if (mt.flags & kFirst) {
            if constexpr (sizeof(T) == 2)
                cs.begin(sbase + C::kOffQ + stage * C::kQBytes, lane);
            else
                cs.begin(reinterpret_cast<const float*>(smem + C::kOffQ + stage * C::kQBytes),
                         reinterpret_cast<float*>(smem + C::kOffWarpQ + warp * C::kQBytes),
                         reinterpret_cast<float*>(smem + C::kOffWarpP + warp * G * (64 / kCW) * 4), lane, g);
        }
        {
            constexpr int P = C::kPagesPerStage;
            const int np = (mt.flags >> kPagesShift) & 15;
            #pragma unroll
            for (int p = 0; p < P; ++p) {
                if (p < np && (mt.flags & (1 << (kValidShift + p)))) {
                    const int lo_p = mt.t_lo - p * kPageSize, hi_p = mt.t_hi - p * kPageSize;
                    const bool partial = lo_p > 0 || hi_p < kPageSize;
                    if constexpr (sizeof(T) == 2)
                        cs.page(kbase + p * C::kTileBytes, kbase + (P + p) * C::kTileBytes, warp, lane, lo_p, hi_p,
                                partial, a.scale_log2);
                    else
                        cs.page(smem + stage * C::kStageBytes + p * C::kTileBytes,
                                smem + stage * C::kStageBytes + (P + p) * C::kTileBytes, warp, lane, lo_p, hi_p, partial,
                                a.scale_log2);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
        if (++stage == S) { stage = 0; phase ^= 1; }
        if (!(mt.flags & kLast)) continue;

        // ---- item done: this warp's (m, l, o) into the next epilogue slot,
        // with no wait on the other consumer warps (the epilogue warps merge
        // the four); the slot is handed over once all 128 threads arrived.
        if (!mbar_wait(bar_eempty + 8 * eslot, ephase ^ 1)) {
            if (lane == 0) fail_timeout(ctrl);
            ok = false;
            break;
        }
        uint8_t* ep = epi_q + eslot * C::kEpiBytes;
        cs.stash(reinterpret_cast<float2*>(ep + sizeof(Meta)) + warp * C::kEpiHeads,
                 reinterpret_cast<float*>(ep + C::kEpiOffO) + warp * C::kEpiHeads * C::kORow, lane);
        if (tid == 0) *reinterpret_cast<Meta*>(ep) = mt;
        mbar_arrive(bar_efull + 8 * eslot);
        if (++eslot == C::kEpiSlots) { eslot = 0; ephase ^= 1; }
    }
    // Tell each epilogue warp that no more items follow: the next slot of
    // each warp's share (the next kEpilogueWarps slots) carries the end flag.
    for (int e = 0; ok && e < kEpilogueWarps; ++e) {
        if (mbar_wait(bar_eempty + 8 * eslot, ephase ^ 1)) {
            if (tid == 0) reinterpret_cast<Meta*>(epi_q + eslot * C::kEpiBytes)->flags = kTerm;
            mbar_arrive(bar_efull + 8 * eslot);
        } else {
            if (lane == 0) fail_timeout(ctrl);
            ok = false;
        }
        if (++eslot == C::kEpiSlots) { eslot = 0; ephase ^= 1; }
    }
}

// ---------------------------------------------------------------------------
// Host launcher
// ---------------------------------------------------------------------------
template <typename T, int D, int G, typename Lay = NoLayers>
static cudaError_t launch_one(const AttendArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                              int grid, bool programmatic, cudaStream_t stream, const Lay& lay = Lay{}) {
    using C = Cfg<T, D, G>;
    auto kern = attend_kernel<T, D, G, Lay>;
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
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, k_map, v_map, a, lay);
}

template <int D>
static cudaError_t launch_f32(const AttendArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map, int grid,
                              bool programmatic, cudaStream_t stream) {
    if (a.group <= 1) return launch_one<float, D, 1>(a, k_map, v_map, grid, programmatic, stream);
    if (a.group <= 2) return launch_one<float, D, 2>(a, k_map, v_map, grid, programmatic, stream);
    if (a.group <= 4) return launch_one<float, D, 4>(a, k_map, v_map, grid, programmatic, stream);
    return launch_one<float, D, 8>(a, k_map, v_map, grid, programmatic, stream);
}

cudaError_t launch_attend(const AttendArgs& a, const CUtensorMap& k_map, const CUtensorMap& v_map,
                          int dtype, int grid, bool programmatic, cudaStream_t stream) {
    if (dtype == 0 && a.head_dim == 128)
        return launch_one<__nv_bfloat16, 128, kMaxGroup>(a, k_map, v_map, grid, programmatic, stream);
    if (dtype == 0 && a.head_dim == 64)
        return launch_one<__nv_bfloat16, 64, kMaxGroup>(a, k_map, v_map, grid, programmatic, stream);
    if (dtype == 1 && a.head_dim == 128) return launch_f32<128>(a, k_map, v_map, grid, programmatic, stream);
    if (dtype == 1 && a.head_dim == 64) return launch_f32<64>(a, k_map, v_map, grid, programmatic, stream);
    return cudaErrorInvalidValue;
}

// Multi-layer launches: bf16 at head dim 64 / 128 (groups up to 8 on one
// instance) and f32 with one-head groups (plain multi-head attention) or any
// group up to 8.  Always a programmatic dependent of the prep launch.
cudaError_t launch_attend_layers(const AttendArgs& a, const AttendLayers& lay, int dtype, int grid,
                                 cudaStream_t stream) {
    const CUtensorMap& k0 = lay.k[0];
    const CUtensorMap& v0 = lay.v[0];
    if (dtype == 0 && a.head_dim == 128)
        return launch_one<__nv_bfloat16, 128, kMaxGroup, AttendLayers>(a, k0, v0, grid, true, stream, lay);
    if (dtype == 0 && a.head_dim == 64)
        return launch_one<__nv_bfloat16, 64, kMaxGroup, AttendLayers>(a, k0, v0, grid, true, stream, lay);
    if (dtype == 1 && a.head_dim == 128)
        return a.group <= 1 ? launch_one<float, 128, 1, AttendLayers>(a, k0, v0, grid, true, stream, lay)
                            : launch_one<float, 128, 8, AttendLayers>(a, k0, v0, grid, true, stream, lay);
    if (dtype == 1 && a.head_dim == 64)
        return a.group <= 1 ? launch_one<float, 64, 1, AttendLayers>(a, k0, v0, grid, true, stream, lay)
                            : launch_one<float, 64, 8, AttendLayers>(a, k0, v0, grid, true, stream, lay);
    return cudaErrorInvalidValue;
}

size_t attend_smem_bytes(int dtype, int head_dim) {
    if (dtype == 0)
        return head_dim == 128 ? Cfg<__nv_bfloat16, 128, kMaxGroup>::kSmem : Cfg<__nv_bfloat16, 64, kMaxGroup>::kSmem;
    return head_dim == 128 ? Cfg<float, 128, kMaxGroup>::kSmem : Cfg<float, 64, kMaxGroup>::kSmem;
}

}  // namespace pdattn
