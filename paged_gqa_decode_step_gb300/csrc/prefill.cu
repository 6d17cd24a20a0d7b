// Paged prefill attention on the fifth-generation tensor cores (tcgen05).
//
// llama-3.1-8b-instruct architecture page, `prefill_paged` (the prefill half
// of `step_paged`): packed prompt tokens, each with its table row, position
// and cache slot.  After the prep kernel has rotated and written every token,
// each token attends over its row's cached positions [lo, pos] through the
// page table, lo = 0 or pos - window + 1 (gpt-oss-20b page, sliding window),
// with optional per-head sinks (gpt-oss-20b page, SinkAttention).
//
// Work unit = one tile of up to 256 / g consecutive tokens of one row times
// one kv head, in two halves of 128 / g tokens.  Each half's g query heads
// per token stack into the 128 rows of an MMA (row m = token m / g, head
// kvh * g + m % g), so one K/V read serves 256 query rows.  Keys come in
// blocks of 128 (two 64-token pages); per block and half:
//   S  = Q K^T      tcgen05.mma M=128 N=128 K=D, fp32 accumulator in TMEM
//   softmax         one thread per MMA row: mask, running max, exp2, sum
//   P               bf16, written back over the first 64 columns of S
//   O += P V        tcgen05.mma M=128 N=D K=128, P read from tensor memory,
//                   V read from shared memory MN-major
// The issuer runs PV_A(j-1) S_A(j) PV_B(j-1) S_B(j): each half's S follows
// its previous PV (P lives in S's columns), and each half's softmax runs
// while the tensor core works for the other half.  Blocks of successive
// units form one stream, so a unit's first S follows the previous unit's
// last PV of the same half.  The running max is raised lazily: O is
// rescaled in TMEM only when a row's max grows by more than 2^8 (S of a
// block done implies the PV before it is done).
//
// Units are taken in the planner's descending-cost order: CTA b starts with
// unit b, later ones come from a global cursor that the last CTA out rewinds.
// The producer passes each unit with its tile descriptor to the other roles
// through a small shared-memory ring.  K and V of a stage fill and drain on
// separate barriers.
//
// Packed sequences (Llama example page, `packed`) run the same kernel: the
// pack is a contiguous cache of 64-token pages, K and V come by 3-D TMA from
// the rotated keys and the values [n, kv_heads, D].  A canonical pack
// without a window masks by pack index like a cache row; otherwise the mask
// is per key (same segment id, position <= the query's, inside the window),
// from segment ids and positions copied into shared memory with each block.
//
// Warpgroups: 0 = warp 0 TMA producer, warp 1 TMEM owner and MMA issuer,
// warps 2 and 3 the V guard (before a block's PV they zero the V rows no
// query of the tile may see); 1 and 2 = softmax and epilogue of halves A and B
// (warp w reads TMEM lanes 32 * (w % 4) .. + 31).  The issuing warpgroup
// hands registers to the softmax warpgroups (setmaxnreg), which hold a
// whole 128-key row of S.  Every wait is bounded; on a timeout the kernel
// sets the error flag, drains its own copies and MMAs, frees TMEM and
// returns.
#include <climits>

#include "internal.h"

namespace pdattn {
namespace {

constexpr int kPfThreads = 384;
constexpr uint64_t kPfTimeoutNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.0f;    // lazy rescale threshold (log2 units)

template <int D, bool kPacked = false>
struct PfCfg {
    static constexpr int kBoxes = D / 64;                 // 64-element column boxes
    static constexpr int kQBytes = kBoxes * 16384;        // one half: 128 rows x 128 B per box
    static constexpr int kKBytes = kBoxes * 16384;        // K (or V) of a block: 128 keys x 128 B per box
    static constexpr int kPageBytes = 8192;               // one page's 64 rows of a box
    static constexpr int kStageBytes = 2 * kKBytes;       // K then V of one block
    static constexpr int kStages = D == 128 ? 2 : 5;
    static constexpr int kMaskStages = kPacked ? kStages : 1;
    static_assert(kStages <= 8, "V ready barriers per stage");
    static constexpr int kOffQ = 0;                       // halves A, B
    static constexpr int kOffStage = 2 * kQBytes;
    static constexpr int kSmem = kOffStage + kStages * kStageBytes + 1024;   // + alignment slack
    // TMEM: S of half h at column 128 h (128 columns; the first 64 then hold
    // P as bf16 pairs); O of half h at 256 + h D.
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 256;
    static_assert(kSmem + kMaskStages * 1024 <= 227 * 1024 - 1536, "shared memory budget");
};

// Registers per thread after the hand-over: the launch gives 384 threads 168
// each (64512); the issuing warpgroup keeps 72, the softmax warpgroups 216
// (128 x 72 + 256 x 216 = 64512).
constexpr uint32_t kRegsIssue = 72, kRegsSoftmax = 216;
static_assert(128 * kRegsIssue + 256 * kRegsSoftmax <= 384 * 168, "register hand-over exceeds the launch");

// --- tcgen05 / TMA wrappers ---------------------------------------------------

// Shared-memory matrix descriptor: 128-byte swizzle, start, leading and
// stride byte offsets (encoded >> 4), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// A / B K-major (0) or MN-major (1), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The issuing warps run their loops with all 32 lanes (warp-uniform control
// flow and operands); each of these instructions is issued once, by the lane
// elect.sync picks.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same with A in tensor memory (a_tmem: row m = lane m, two bf16 per column).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The barrier arrives once every MMA issued so far by this warp is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void elect_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}"
        ::"r"(bar), "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void elect_tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void elect_tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                             uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void elect_bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Warp-wide bounded wait: every lane polls, and the warp agrees on the result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, Ctrl* ctrl);

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed fp32 pairs (one instruction for two lanes of work): d = a * b + c
// with b, c shared, and d += b.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n mov.b64 rc, {%5, %5};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

__device__ __forceinline__ void fadd2(float& d0, float& d1, float b0, float b1) {
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%0, %1};\n mov.b64 rb, {%2, %3};\n"
        " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
        : "+f"(d0), "+f"(d1) : "f"(b0), "f"(b1));
}

// a0 += low bf16 of p, a1 += high bf16 of p (exact widening, f32 adds).
__device__ __forceinline__ void add_bf16x2_f32(float& a0, float& a1, uint32_t p) {
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n add.rn.f32.bf16 %0, lo, %0;\n"
        " add.rn.f32.bf16 %1, hi, %1;\n}"
        : "+f"(a0), "+f"(a1) : "r"(p));
}

// Max of 64 values as eight short independent chains.
__device__ __forceinline__ float max64(const uint32_t (&s)[64]) {
    float acc[8];
    #pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float* v = reinterpret_cast<const float*>(&s[8 * k]);
        float x = fmax3(v[0], v[1], v[2]);
        x = fmax3(x, v[3], v[4]);
        x = fmax3(x, v[5], v[6]);
        acc[k] = fmaxf(x, v[7]);
    }
    return fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

__device__ __forceinline__ float max128(const uint32_t (&s)[128]) {
    return fmaxf(max64(*reinterpret_cast<const uint32_t(*)[64]>(&s[0])),
                 max64(*reinterpret_cast<const uint32_t(*)[64]>(&s[64])));
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int* abort, Ctrl* ctrl) {
    if (mbar_test_wait(bar, parity)) return true;
    uint64_t t0 = 0;
    #pragma unroll 1
    for (int i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 15) {
            if (*abort) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kPfTimeoutNs) {
                *abort = 1;
                set_error(ctrl, kErrTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, Ctrl* ctrl) {
    return __all_sync(0xffffffffu, pf_wait(bar, parity, abort, ctrl));
}

// Broadcast of lane 0's value: the loops of the issuing warps stay uniform.
__device__ __forceinline__ int uni(int v) { return __shfl_sync(0xffffffffu, v, 0); }

// Units reach a CTA through a small ring: the producer takes the next unit
// of the descending-cost list (CTA b starts with unit b, later ones come
// from a global cursor), so a CTA that finishes early takes more work.
constexpr int kUnitSlots = 4;
constexpr int kUnitReaders = 11;     // the issuing warp, the two V guard warps and the eight softmax warps

struct PfBars {
    uint64_t q_full[2], q_empty[2];   // [half]: Q loaded / every S of the unit reading it done
    uint64_t mma_done;
    uint64_t unit_full[kUnitSlots], unit_empty[kUnitSlots];
    uint64_t s_full[2];      // [half]: S of the block done (its previous PV too)
    uint64_t v_ready[8];     // [stage]: V of the block landed and its rows outside the tile's range zeroed
    uint64_t p_full[2];      // [half]: P of the block written (one arrival per warp of the half)
    uint64_t o_done[2];      // [half]: the unit's last PV done
};

// A slot of the unit ring: the unit and its tile descriptor, so that no
// reader waits on a global load at a unit boundary.
struct __align__(32) UnitSlot {
    PfTile t;
    int u;
    int pad[7];
};

// The next unit from the producer's ring (whole warp) and its tile: -1 once
// there is no more work, -2 on abort.
__device__ __forceinline__ int take_unit(PfBars& bars, const UnitSlot* s_unit, uint32_t k, int lane,
                                         volatile int* abort, Ctrl* ctrl, PfTile& t) {
    const int slot = k % kUnitSlots;
    if (!warp_wait(smem_u32(&bars.unit_full[slot]), (k / kUnitSlots) & 1, abort, ctrl)) return -2;
    const volatile int4* src = reinterpret_cast<const volatile int4*>(&s_unit[slot]);
    const int4 t0 = make_int4(src[0].x, src[0].y, src[0].z, src[0].w);
    const int4 t1 = make_int4(src[1].x, src[1].y, src[1].z, src[1].w);
    const int u = src[2].x;
    t.t0 = t0.x; t.ntok = t0.y; t.row = t0.z; t.first_page = t0.w;
    t.npg = t1.x; t.lo_min = t1.y; t.pos_max = t1.z; t.pad = t1.w;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars.unit_empty[slot]));
    return u;
}

// Softmax and epilogue of one half (128 threads, one MMA row each).
template <int D, bool kPacked>
__device__ __forceinline__ void softmax_half(const PrefillArgs& a, int half, int quarter, int lane, uint32_t tmem,
                                             PfBars& bars, const int (*s_mask)[256], uint64_t* v_full,
                                             const UnitSlot* s_unit, volatile int* abort, Ctrl* ctrl) {
    using C = PfCfg<D, kPacked>;
    const int* seg_pad = reinterpret_cast<const int*>(a.ws + a.L.seg_pad);
    const int4* blk = reinterpret_cast<const int4*>(a.ws + a.L.blk);
    const int W = a.window;
    const bool canonical_no_window = kPacked && W <= 0 && ctrl->rows == 1;
    const int Hk = a.kv_heads, g = a.group, Tq = a.tile_tokens / 2;
    const int m = quarter * 32 + lane;                    // MMA row = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + 128u * half, o_addr = tmem + lane_base + C::kColO + half * D;
    const int tq = m / g, jh = m % g;
    const float sl2 = a.scale_log2;
    const __nv_bfloat16* sinks = static_cast<const __nv_bfloat16*>(a.sinks);
    const bool out_wide = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;   // rows are D * 2 bytes apart
    const uint32_t s_full = smem_u32(&bars.s_full[half]), p_full = smem_u32(&bars.p_full[half]);
    // A canonical pack (every sequence one run, positions rising) without a
    // window sees exactly the tokens [run start, own index] of the pack.
    const bool by_index = !kPacked || canonical_no_window;
    const int tok = half * Tq + tq;                       // token of this row within a tile
    uint32_t it = 0, ch = 0, uh = 0;     // blocks of every unit / of units with this half; units with it
    bool ok = true;
    // The row's position (and segment id) of a unit load while the previous
    // unit's epilogue runs: the next unit is taken before it.
    uint32_t k = 0;
    PfTile t;
    int u = take_unit(bars, s_unit, k++, lane, abort, ctrl, t);
    int pos_next = -1, seg_next = 0;
    auto row_inputs = [&](const PfTile& tt, int& p, int& sg) {
        p = -1;
        sg = 0;
        if (tq < Tq && tok < tt.ntok) {
            p = __ldg(a.positions + tt.t0 + tok);
            if (!by_index) sg = seg_pad[tt.t0 + tok];
        }
    };
    if (u >= 0) row_inputs(t, pos_next, seg_next);
    while (u >= 0) {
        const int kvh = u % Hk, nb = (t.npg + 1) / 2;
        const bool present = half == 0 || t.ntok > Tq;
        if (!present) {
            it += nb;
            u = take_unit(bars, s_unit, k++, lane, abort, ctrl, t);
            if (u >= 0) row_inputs(t, pos_next, seg_next);
            continue;
        }
        const bool active = tq < Tq && tok < t.ntok;
        int pos = -1, lo = 0;
        const int seg = seg_next;
        if (active) {
            pos = pos_next < 0 ? 0 : pos_next;
            lo = (W > 0 && pos - W + 1 > 0) ? pos - W + 1 : 0;
        }
        const int key_lo = kPacked ? t.pad : lo, key_hi = kPacked ? (active ? t.t0 + tok : -1) : pos;
        float m_run = -INFINITY, l = 0.f;
        for (int b = 0; b < nb; ++b) {
            const uint32_t j = ch + b;
            const int pg0 = t.first_page + 2 * b, npb = min(2, t.npg - 2 * b);   // pages in this block
            ok = pf_wait(s_full, j & 1, abort, ctrl);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t s[128];
            #pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_ld32(s_addr + 32 * q4, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q4]));
            tmem_wait_ld();
            const int key0 = pg0 * kPageSize;
            if (by_index) {
                // keys c of this block visible to the row: key_lo <= key0 + c <= key_hi;
                // 32-column chunks visible to every row of the warp skip the test
                const int c_lo = key_lo - key0, c_hi = min(key_hi - key0, npb * kPageSize - 1);
                if (!__all_sync(0xffffffffu, c_lo <= 0 && c_hi >= 2 * kPageSize - 1)) {
                    #pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int b0 = 32 * q4;
                        if (!__all_sync(0xffffffffu, c_lo <= b0 && c_hi >= b0 + 31)) {
                            #pragma unroll
                            for (int c = b0; c < b0 + 32; ++c)
                                if (c < c_lo || c > c_hi) s[c] = __float_as_uint(-INFINITY);
                        }
                    }
                }
            } else {
                // key c is visible when it belongs to the row's sequence at a
                // position <= pos (and inside the window); a page wholly of
                // that sequence and before pos skips the test
                bool full = active && npb == 2;
                #pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int4 bi = blk[min(pg0 + q, pg0 + npb - 1)];
                    full = full && bi.x && bi.y == seg && bi.w <= pos && (W <= 0 || bi.z > pos - W);
                }
                if (!__all_sync(0xffffffffu, full)) {
                    const int st = (it + b) % C::kStages;
                    // the stage's ids and positions came by bulk copy with V
                    mbar_wait(smem_u32(&v_full[st]), ((it + b) / C::kStages) & 1, kPfTimeoutNs);
                    const int4* sg = reinterpret_cast<const int4*>(s_mask[st]);
                    const int4* sp = reinterpret_cast<const int4*>(s_mask[st] + 128);
                    #pragma unroll
                    for (int c4 = 0; c4 < 32; ++c4) {
                        const int4 g4 = sg[c4], p4 = sp[c4];
                        const int gs[4] = {g4.x, g4.y, g4.z, g4.w}, pp[4] = {p4.x, p4.y, p4.z, p4.w};
                        #pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 4 * c4 + e;
                            const bool vis = active && c < npb * kPageSize && gs[e] == seg && pp[e] <= pos &&
                                             (W <= 0 || pp[e] > pos - W);
                            if (!vis) s[c] = __float_as_uint(-INFINITY);
                        }
                    }
                }
            }
            const float mx = max128(s) * sl2;              // scale > 0: the max commutes with it
            const bool need = mx > m_run + kRescaleLog2;
            float alpha = 1.f;
            if (need) {
                alpha = exp2_approx(m_run - mx);           // 0 while m_run is -inf
                m_run = mx;
                l *= alpha;
            }
            const float neg_mu = m_run == -INFINITY ? 0.f : -m_run;
            // O (complete up to the previous block: its PV preceded this S) is
            // rescaled only when some row's max grew past the threshold
            if (b > 0 && __any_sync(0xffffffffu, need && alpha != 1.f)) {
                #pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(o_addr + c0, o);
                    tmem_wait_ld();
                    #pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tmem_st32(o_addr + c0, o);
                }
            }
            // P as bf16 pairs over the first 64 columns of S.  The denominator
            // sums the same rounded weights, so the normalised weights are an
            // exact convex combination.  Packs sum them after the hand-over,
            // off the path to the next MMA; prefill sums them in line (there
            // the deferred sum competes for issue with the other half's
            // softmax and measured slower).
            uint32_t pk[64];
            float acc[8];
            // (in line: bf16 + f32 adds; deferred: the pair unpacked, one f32x2
            // add; each measured faster where it is used)
            auto add_pair = [&](int c, uint32_t p) {
                const int q = c & 3;                      // four pair accumulators
                if constexpr (!kPacked) {
                    if (c < 4) {
                        acc[2 * q] = 0.f;
                        acc[2 * q + 1] = 0.f;
                    }
                    add_bf16x2_f32(acc[2 * q], acc[2 * q + 1], p);
                } else {
                    const float lw = __uint_as_float(p << 16), hw = __uint_as_float(p & 0xffff0000u);
                    if (c < 4) {
                        acc[2 * q] = lw;
                        acc[2 * q + 1] = hw;
                    } else {
                        fadd2(acc[2 * q], acc[2 * q + 1], lw, hw);
                    }
                }
            };
            #pragma unroll
            for (int h64 = 0; h64 < 2; ++h64) {
                #pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const int cc = 64 * h64 + c;
                    float x0, x1;
                    ffma2(x0, x1, __uint_as_float(s[cc]), __uint_as_float(s[cc + 1]), sl2, neg_mu);
                    pk[cc >> 1] = pack_bf16x2(exp2_approx(x0), exp2_approx(x1));
                    if constexpr (!kPacked) add_pair(cc >> 1, pk[cc >> 1]);
                }
                tmem_st32(s_addr + 32 * h64, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32 * h64]));
            }
            // every lane's stores are complete and fenced before its warp's
            // one arrival (128 single arrivals on one word serialise)
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            if constexpr (kPacked) {
                #pragma unroll
                for (int c = 0; c < 64; ++c) add_pair(c, pk[c]);
            }
            l += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        }
        if (!ok) break;
        // The next unit, whose row inputs load under this epilogue.
        PfTile tn;
        const int un = take_unit(bars, s_unit, k++, lane, abort, ctrl, tn);
        if (un >= 0) row_inputs(tn, pos_next, seg_next);
        // Epilogue: O / l (with the sink's share of the denominator).
        ok = warp_wait(smem_u32(&bars.o_done[half]), uh & 1, abort, ctrl);
        if (!ok) break;
        tc_fence_after();
        const int h = kvh * g + jh;
        float inv = l > 0.f ? 1.f / l : 0.f;
        if (sinks != nullptr && active) {
            const float sk = __bfloat162float(sinks[h]) * 1.4426950408889634f;
            const float mu = m_run == -INFINITY ? sk : m_run;
            const float Mp = fmaxf(mu, sk);
            const float f = exp2_approx(mu - Mp);
            inv = f / (l * f + exp2_approx(sk - Mp));
        }
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(t.t0 + tok) * a.heads + h) * D;
        // 64 columns per round trip to TMEM; 32-byte stores (whole sectors)
        // when the output is 32-byte aligned, else 16-byte ones
        #pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t o[64];
            tmem_ld32(o_addr + c0, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            tmem_ld32(o_addr + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
            tmem_wait_ld();
            if (active) {
                #pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t w[8];
                    #pragma unroll
                    for (int e = 0; e < 8; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(o[16 * v + 2 * e]) * inv,
                                           __uint_as_float(o[16 * v + 2 * e + 1]) * inv);
                    __nv_bfloat16* dst = orow + c0 + 16 * v;
                    if (out_wide) {
                        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                                     ::"l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                                       "r"(w[6]), "r"(w[7])
                                     : "memory");
                    } else {
                        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
        }
        // The next unit's first PV overwrites O only after this read (its
        // p_full arrival follows in program order).
        tc_fence_before();
        ch += nb;
        it += nb;
        ++uh;
        u = un;
        t = tn;
    }
}

template <int D, bool kPacked>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map, const __grid_constant__ PrefillArgs a) {
    using C = PfCfg<D, kPacked>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // K and V of a stage fill and drain separately: K is free once the
    // block's S is done, V (with the packed mask) once its PV is
    __shared__ __align__(8) uint64_t k_full[C::kStages], k_empty[C::kStages];
    __shared__ __align__(8) uint64_t v_full[C::kStages], v_empty[C::kStages];
    __shared__ __align__(8) PfBars bars;
    __shared__ __align__(16) int s_mask[C::kMaskStages][256];   // packed: segment ids [0,128), positions [128,256)
    __shared__ UnitSlot s_unit[kUnitSlots];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t q_s = sb + C::kOffQ, st_s = sb + C::kOffStage;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    volatile int* abort = &s_abort;

    // Rows of the Q tiles that no token fills stay zero.
    for (int i = tid; i < 2 * C::kQBytes / 16; i += kPfThreads)
        reinterpret_cast<uint4*>(sm + C::kOffQ)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&k_full[s]), 1);
            mbar_init(smem_u32(&k_empty[s]), 1);
            mbar_init(smem_u32(&v_full[s]), 1);
            mbar_init(smem_u32(&v_empty[s]), 1);
            mbar_init(smem_u32(&bars.v_ready[s]), 2);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(smem_u32(&bars.q_full[h]), 1);
            mbar_init(smem_u32(&bars.q_empty[h]), 1);
        }
        mbar_init(smem_u32(&bars.mma_done), 1);
        for (int k = 0; k < kUnitSlots; ++k) {
            mbar_init(smem_u32(&bars.unit_full[k]), 1);
            mbar_init(smem_u32(&bars.unit_empty[k]), kUnitReaders);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(smem_u32(&bars.s_full[h]), 1);
            mbar_init(smem_u32(&bars.p_full[h]), 4);
            mbar_init(smem_u32(&bars.o_done[h]), 1);
        }
        s_abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&q_map);
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&v_map);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&s_tmem)), "r"(C::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_proxy_async_shared();     // zeroed Q rows, before any MMA reads them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // Everything below reads what the prep kernel wrote.
    griddep_wait();
    const int Hk = a.kv_heads, g = a.group, Tq = a.tile_tokens / 2;
    const int n_units = (ctrl->magic == kPlanMagic ? ctrl->n_items : 0) * Hk;
    const PfTile* tiles = reinterpret_cast<const PfTile*>(a.ws + a.L.tiles);

    // The issuing warpgroup hands registers to the softmax warpgroups.
    if (warp >= 4) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ---------------- softmax + epilogue: warps 4..7 half A, 8..11 half B ----------------
        softmax_half<D, kPacked>(a, (warp - 4) >> 2, warp & 3, lane, tmem, bars, s_mask, v_full, s_unit, abort,
                                 ctrl);
    } else {
      // one setmaxnreg site for the whole issuing warpgroup
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
      if (warp == 0) {
        // ---------------- TMA producer (whole warp, one lane issues) ----------------
        uint32_t kit = 0, vit = 0, uq[2] = {0, 0};   // K, V blocks loaded; units whose Q half h was loaded
        bool ok = true;
        int u = blockIdx.x;
        for (uint32_t k = 0; ok; ++k) {
            if (k > 0) {
                int v = 0;
                if (lane == 0) v = (int)gridDim.x + atomicAdd(&ctrl->next_item, 1);
                u = __shfl_sync(0xffffffffu, v, 0);
            }
            const int slot = k % kUnitSlots;
            PfTile t = {};
            if (u < n_units) t = tiles[u / Hk];
            ok = warp_wait(smem_u32(&bars.unit_empty[slot]), ((k / kUnitSlots) & 1) ^ 1, abort, ctrl);
            if (!ok) break;
            if (lane == 0) {
                int4* dst = reinterpret_cast<int4*>(&s_unit[slot]);
                dst[0] = make_int4(t.t0, t.ntok, t.row, t.first_page);
                dst[1] = make_int4(t.npg, t.lo_min, t.pos_max, t.pad);
                dst[2] = make_int4(u < n_units ? u : -1, 0, 0, 0);
                mbar_arrive(smem_u32(&bars.unit_full[slot]));
            }
            __syncwarp();
            if (u >= n_units) break;
            const int kvh = u % Hk, nh = uni(t.ntok > Tq ? 2 : 1), npg = uni(t.npg), t0 = uni(t.t0);
            const int first = uni(t.first_page), row = uni(t.row), nb = (npg + 1) / 2;
            const int* trow = kPacked ? nullptr : a.table + (size_t)row * a.pages_per_row + first;
            // The unit's page ids, 32 at a time: lane l holds page pid_base + l
            // (pid_cur) and the next window's (pid_nxt, read a window ahead),
            // so no load waits for the table but the unit's first.
            int pid_base = -32, pid_cur = 0, pid_nxt = 0;
            // Page q of block bk: the cache page (paged) or the pack's key
            // index (packed) of rows [64 q, 64 q + 64) of every box.
            auto page_of = [&](int bk, int q) -> int {
                if (kPacked) return (first + 2 * bk + q) * kPageSize;
                const int pi = 2 * bk + q;              // pages are visited in order
                if (pi - pid_base >= 32) {
                    if (pid_base < 0) pid_cur = lane < npg ? __ldg(trow + lane) : 0;
                    else pid_cur = pid_nxt;
                    pid_base += 32;
                    pid_nxt = pid_base + 32 + lane < npg ? __ldg(trow + pid_base + 32 + lane) : 0;
                }
                int page = __shfl_sync(0xffffffffu, pid_cur, pi & 31);
                if (page < 0 || page >= a.num_pages) {
                    if (lane == 0) set_error(ctrl, kErrBadPage);
                    page = 0;
                }
                return (page * Hk + kvh) * kPageSize;
            };
            auto load_k = [&](int bk) -> bool {
                const int s = kit % C::kStages, npb = min(2, npg - 2 * bk);
                if (!warp_wait(smem_u32(&k_empty[s]), ((kit / C::kStages) & 1) ^ 1, abort, ctrl)) return false;
                const uint32_t kb = st_s + s * C::kStageBytes, kf = smem_u32(&k_full[s]);
                elect_arrive_expect_tx(kf, npb * C::kBoxes * C::kPageBytes);
                for (int q = 0; q < npb; ++q) {
                    const int y = page_of(bk, q);
                    for (int b = 0; b < C::kBoxes; ++b) {
                        if (kPacked) elect_tma_3d(kb + b * 16384 + q * C::kPageBytes, &k_map, b * 64, kvh, y, kf);
                        else elect_tma_2d(kb + b * 16384 + q * C::kPageBytes, &k_map, b * 64, y, kf);
                    }
                }
                ++kit;
                return true;
            };
            auto load_v = [&](int bk) -> bool {
                const int s = vit % C::kStages, npb = min(2, npg - 2 * bk);
                if (!warp_wait(smem_u32(&v_empty[s]), ((vit / C::kStages) & 1) ^ 1, abort, ctrl)) return false;
                const uint32_t vb = st_s + s * C::kStageBytes + C::kKBytes, vf = smem_u32(&v_full[s]);
                elect_arrive_expect_tx(vf, npb * (C::kBoxes * C::kPageBytes + (kPacked ? 512 : 0)));
                for (int q = 0; q < npb; ++q) {
                    const int y = page_of(bk, q);
                    for (int b = 0; b < C::kBoxes; ++b) {
                        if (kPacked) elect_tma_3d(vb + b * 16384 + q * C::kPageBytes, &v_map, b * 64, kvh, y, vf);
                        else elect_tma_2d(vb + b * 16384 + q * C::kPageBytes, &v_map, b * 64, y, vf);
                    }
                    if (kPacked) {
                        // segment ids and positions of the block's keys, for the per-key mask
                        const uint32_t mb = smem_u32(&s_mask[kPacked ? s : 0][0]);
                        elect_bulk_load(mb + q * 256, reinterpret_cast<const int*>(a.ws + a.L.seg_pad) + y, 256, vf);
                        elect_bulk_load(mb + 512 + q * 256, reinterpret_cast<const int*>(a.ws + a.L.pos_pad) + y, 256,
                                        vf);
                    }
                }
                ++vit;
                return true;
            };
            // K of the first block goes first: its stage frees before the
            // previous unit's last S is done, which is what Q waits for.
            ok = load_k(0);
            #pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!ok || h >= nh) break;
                ok = warp_wait(smem_u32(&bars.q_empty[h]), (uq[h] & 1) ^ 1, abort, ctrl);
                if (!ok) break;
                const uint32_t qf = smem_u32(&bars.q_full[h]);
                elect_arrive_expect_tx(qf, C::kBoxes * 128 * g * Tq);
                for (int b = 0; b < C::kBoxes; ++b)
                    elect_tma_3d(q_s + h * C::kQBytes + b * 16384, &q_map, b * 64, kvh * g, t0 + h * Tq, qf);
                ++uq[h];
            }
            ok = ok && load_v(0);
            for (int bk = 1; bk < nb && ok; ++bk) ok = load_k(bk) && load_v(bk);
        }
        // Drain: every load issued has landed before exit.
        for (uint32_t k = 0; k < (uint32_t)C::kStages && k < kit; ++k) {
            const uint32_t j = kit - 1 - k;
            mbar_wait(smem_u32(&k_full[j % C::kStages]), (j / C::kStages) & 1, kPfTimeoutNs);
        }
        for (uint32_t k = 0; k < (uint32_t)C::kStages && k < vit; ++k) {
            const uint32_t j = vit - 1 - k;
            mbar_wait(smem_u32(&v_full[j % C::kStages]), (j / C::kStages) & 1, kPfTimeoutNs);
        }
        #pragma unroll
        for (int h = 0; h < 2; ++h)
            if (uq[h] > 0) mbar_wait(smem_u32(&bars.q_full[h]), (uq[h] - 1) & 1, kPfTimeoutNs);
    } else if (warp == 1) {
        // ---------------- MMA issuer (whole warp, one lane issues) ----------------
        constexpr uint32_t idesc_s = instr_desc(128, 128, 0, 0);
        constexpr uint32_t idesc_s64 = instr_desc(128, 64, 0, 0);    // a block of one page
        constexpr uint32_t idesc_o = instr_desc(128, D, 0, 1);
        bool issued = false;
        bool ok = true;
        // Descriptors are built once: the start-address field (bits 0..13,
        // address >> 4) is linear, so every operand below is a base
        // descriptor plus a constant.
        const uint64_t dq = smem_desc(q_s, 16, 1024), dk = smem_desc(st_s, 16, 1024);
        const uint64_t dv = smem_desc(st_s + C::kKBytes, 16384, 1024);
        // S_h = Q_h K^T of the block in stage s (N = 128 keys, or 64 when
        // the block holds one page: the softmax masks the other 64 columns)
        auto qk = [&](int h, int s, bool one_page) {
            const uint32_t idesc = one_page ? idesc_s64 : idesc_s;
            const uint64_t a0 = dq + (uint64_t)(h * (C::kQBytes >> 4));
            const uint64_t b0 = dk + (uint64_t)(s * (C::kStageBytes >> 4));
            #pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                umma_bf16(tmem + 128u * h, a0 + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2),
                          b0 + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2), idesc, ks > 0 ? 1u : 0u);
            umma_commit(smem_u32(&bars.s_full[h]));
        };
        // O_h += P_h V of the block in stage s; P of block j sits over S_h
        // (8 columns per 16 keys); the first block of a unit overwrites O_h.
        // A one-page block stops after 64 keys (the weights beyond are 0).
        auto pv = [&](int h, uint32_t j, int s, bool first, bool one_page) -> bool {
            if (!warp_wait(smem_u32(&bars.p_full[h]), j & 1, abort, ctrl)) return false;
            tc_fence_after();
            const uint64_t b0 = dv + (uint64_t)(s * (C::kStageBytes >> 4));
            #pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                if (ks < 4 || !one_page)
                    umma_bf16_ts(tmem + C::kColO + h * D, tmem + 128u * h + ks * 8, b0 + (uint64_t)(ks * 128),
                                 idesc_o, (first && ks == 0) ? 0u : 1u);
            return true;
        };
        // Blocks of successive units form one stream, one step per block (and
        // a last one for the end): for each half, the PV of the pending block
        // (possibly the previous unit's last), then the S of this one, so a
        // unit boundary leaves no gap in the tensor pipe beyond the Q load.
        // The pending block is always the previous one (index it - 1,
        // counters cs_h - 1).  The half loop stays rolled so that each MMA
        // sequence is issued from one place; per-half state is selected by
        // value.
        constexpr uint32_t kPend = 1, kPendFirst = 2, kPendLast = 4, kPendOne = 8, kPendB = 16, kEnd = 32;
        uint32_t it = 0, uq0 = 0, uq1 = 0, cs0 = 0, cs1 = 0, f = 0;   // blocks; units / S per half; flags
        int nh = 0, npg = 0, bk = 0;                                  // the current unit and block
        for (uint32_t k = 0; ok;) {
            if (2 * bk >= npg) {                                      // the unit is done: the next one
                if (npg > 0) {
                    ++uq0;
                    if (nh == 2) ++uq1;
                }
                PfTile t;
                const int u = take_unit(bars, s_unit, k++, lane, abort, ctrl, t);
                if (u == -2) {
                    ok = false;
                    break;
                }
                nh = 0;
                npg = 0;
                bk = 0;
                if (u < 0) {
                    f |= kEnd;
                } else {
                    nh = uni(t.ntok > Tq ? 2 : 1);
                    npg = uni(t.npg);
                }
            }
            const int s = it % C::kStages;
            const bool one = npg - 2 * bk == 1;
            #pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if ((f & kPend) && (h == 0 || (f & kPendB))) {
                    if (h == 0) {
                        ok = warp_wait(smem_u32(&bars.v_ready[(it - 1) % C::kStages]), ((it - 1) / C::kStages) & 1, abort,
                                       ctrl);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    ok = pv(h, (h ? cs1 : cs0) - 1, (it - 1) % C::kStages, f & kPendFirst, f & kPendOne);
                    if (!ok) break;
                    if (f & kPendLast) umma_commit(smem_u32(&bars.o_done[h]));
                }
                if (h < nh) {
                    if (h == 0) {
                        ok = warp_wait(smem_u32(&k_full[s]), (it / C::kStages) & 1, abort, ctrl);
                        if (!ok) break;
                    }
                    if (bk == 0) {
                        ok = warp_wait(smem_u32(&bars.q_full[h]), (h ? uq1 : uq0) & 1, abort, ctrl);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    issued = true;
                    qk(h, s, one);
                }
            }
            if (!ok) break;
            if (f & kPend) umma_commit(smem_u32(&v_empty[(it - 1) % C::kStages]));   // the pending block's PV issued
            if (f & kEnd) break;
            umma_commit(smem_u32(&k_empty[s]));                                       // this block's S issued
            const bool last = 2 * (bk + 1) >= npg;
            if (last) {
                umma_commit(smem_u32(&bars.q_empty[0]));
                if (nh == 2) umma_commit(smem_u32(&bars.q_empty[1]));
            }
            f = kPend | (bk == 0 ? kPendFirst : 0) | (last ? kPendLast : 0) | (one ? kPendOne : 0) |
                (nh == 2 ? kPendB : 0);
            ++cs0;
            if (nh == 2) ++cs1;
            ++it;
            ++bk;
        }
        // Drain: every MMA issued has finished before TMEM is freed.
        if (issued) {
            umma_commit(smem_u32(&bars.mma_done));
            mbar_wait(smem_u32(&bars.mma_done), 0, kPfTimeoutNs);
        }
      } else {
        // ---------------- V guard (warps 2 and 3) ----------------
        // V rows of a block outside the tile's key range [lo_min, pos_max]
        // hold no key of the tile (stale cache slots, another sequence of
        // the pack: possibly non-finite), and every row's weight there is 0:
        // they are zeroed so that 0 * V stays 0 in PV.  The issuer starts a
        // block's PV only once both warps have passed it.
        // Tiles of a cache row or of a canonical pack see a key range; in a
        // pack of any other layout a tile (one run, one segment id) sees the
        // keys of its segment at positions <= its last query's (and inside
        // the window of its first), row by row from the block's ids.
        constexpr int kPieces = C::kBoxes * 8;         // 16-byte pieces of a V row
        const int gw = warp - 2;
        const bool by_key = kPacked && ctrl->rows == 0;
        const int* seg_pad = reinterpret_cast<const int*>(a.ws + a.L.seg_pad);
        const int W = a.window;
        uint32_t it = 0;
        bool ok = true;
        for (uint32_t k = 0; ok; ++k) {
            PfTile t;
            const int u = take_unit(bars, s_unit, k, lane, abort, ctrl, t);
            if (u < 0) break;
            const int npg = t.npg, first = t.first_page, lo_min = t.lo_min, pos_max = t.pos_max;
            int tseg = 0, pmin = INT_MAX, pmax = -1;
            if (by_key) {
                const int t0 = t.t0, ntok = t.ntok;
                tseg = seg_pad[t0];
                for (int i = lane; i < ntok; i += 32) {
                    const int p = max(__ldg(a.positions + t0 + i), 0);
                    pmin = min(pmin, p);
                    pmax = max(pmax, p);
                }
                #pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, d));
                    pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, d));
                }
            }
            for (int bk = 0; 2 * bk < npg; ++bk, ++it) {
                const int st = it % C::kStages;
                ok = warp_wait(smem_u32(&v_full[st]), (it / C::kStages) & 1, abort, ctrl);
                if (!ok) break;
                const int key0 = (first + 2 * bk) * kPageSize, rows = min(2, npg - 2 * bk) * kPageSize;
                const uint32_t vb = st_s + st * C::kStageBytes + C::kKBytes;
                auto zero_row = [&](int r) {
                    #pragma unroll
                    for (int piece = 0; piece < kPieces; ++piece)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                                     ::"r"(vb + (piece >> 3) * 16384 + r * 128 + (piece & 7) * 16), "r"(0)
                                     : "memory");
                };
                if (by_key) {
                    // the block's segment ids and positions came with V
                    bool any = false;
                    for (int r = gw * 32 + lane; r < rows; r += 64) {
                        const int sg = s_mask[kPacked ? st : 0][r], pp = s_mask[kPacked ? st : 0][128 + r];
                        if (!(sg == tseg && pp <= pmax && (W <= 0 || pp > pmin - W))) {
                            zero_row(r);
                            any = true;
                        }
                    }
                    if (__any_sync(0xffffffffu, any)) fence_proxy_async_shared();
                } else {
                    const int v_lo = max(lo_min - key0, 0), v_hi = min(pos_max - key0, rows - 1);   // rows kept
                    const int n_lo = v_lo, n_hi = rows - 1 - v_hi;                                 // rows zeroed
                    if (n_lo > 0 || n_hi > 0) {
                        for (int zr = gw * 32 + lane; zr < n_lo + n_hi; zr += 64)
                            zero_row(zr < n_lo ? zr : v_hi + 1 + (zr - n_lo));
                        fence_proxy_async_shared();
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars.v_ready[st]));
            }
        }
      }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        // The last CTA out rewinds the unit cursor for the next launch.
        __threadfence();
        if (atomicAdd(&ctrl->done_ctas, 1) == (int)gridDim.x - 1) {
            ctrl->next_item = 0;
            ctrl->done_ctas = 0;
        }
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
}

template <int D, bool kPacked>
cudaError_t launch_d(const PrefillArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                     const CUtensorMap& v_map, int grid, cudaStream_t stream) {
    using C = PfCfg<D, kPacked>;
    auto kern = prefill_kernel<D, kPacked>;
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
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kern, q_map, k_map, v_map, a);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, int grid, cudaStream_t stream) {
    if (a.head_dim == 128) return launch_d<128, false>(a, q_map, k_map, v_map, grid, stream);
    if (a.head_dim == 64) return launch_d<64, false>(a, q_map, k_map, v_map, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_packed(const PrefillArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                          const CUtensorMap& v_map, int grid, cudaStream_t stream) {
    if (a.head_dim == 128) return launch_d<128, true>(a, q_map, k_map, v_map, grid, stream);
    if (a.head_dim == 64) return launch_d<64, true>(a, q_map, k_map, v_map, grid, stream);
    return cudaErrorInvalidValue;
}

size_t prefill_smem_bytes(int head_dim) {
    return head_dim == 128 ? PfCfg<128, false>::kSmem : PfCfg<64, false>::kSmem;
}

}  // namespace pdattn
