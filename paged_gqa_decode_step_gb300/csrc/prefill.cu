// Paged prefill attention on the fifth-generation tensor cores (tcgen05).
//
// llama-3.1-8b-instruct architecture page, `prefill_paged` (the prefill half
// of `step_paged`): packed prompt tokens, each with its table row, position
// and cache slot.  After the prep kernel has rotated and written every token,
// each token attends over its row's cached positions [lo, pos] through the
// page table, lo = 0 or pos - window + 1 (gpt-oss-20b page, sliding window),
// with optional per-head sinks (gpt-oss-20b page, SinkAttention).
//
// Work unit = one tile of up to 128 / g consecutive tokens of one row times
// one kv head.  The tile's g query heads per token stack into the 128 rows of
// the MMA (row m = token (m / g), head kvh * g + m % g), so one K/V page read
// serves every query of the tile.  Per page of 64 keys:
//   S  = Q K^T      tcgen05.mma M=128 N=64 K=D, fp32 accumulator in TMEM
//   softmax         one thread per MMA row: mask, running max, exp2, sum
//   P               bf16 in shared memory (128-byte swizzle, K-major)
//   O += P V        tcgen05.mma M=128 N=D K=64, V page read MN-major
// S is double-buffered in TMEM so that S of page j+1 runs under the softmax
// of page j.  The running max is raised lazily: O is rescaled in TMEM only
// when a row's max grows by more than 2^8, so that most pages need no
// round trip through the accumulator.
//
// Warps: 0 = TMA producer (Q box, K and V pages), 1 = TMEM owner and MMA
// issuer, 2..5 = softmax and epilogue (warp w reads TMEM lanes
// 32 * (w % 4) .. + 31).  Every wait is bounded; on a timeout the kernel sets
// the error flag, drains its own copies and MMAs, frees TMEM and returns.
#include <climits>

#include "internal.h"

namespace pdattn {
namespace {

constexpr int kPfThreads = 192;
constexpr uint64_t kPfTimeoutNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.0f;    // lazy rescale threshold (log2 units)

template <int D>
struct PfCfg {
    static constexpr int kBoxes = D / 64;                 // 64-element column boxes
    static constexpr int kQBytes = kBoxes * 16384;        // 128 rows x 128 B per box
    static constexpr int kKvBytes = kBoxes * 8192;        // one page of K (or V): 64 rows x 128 B per box
    static constexpr int kStageBytes = 2 * kKvBytes;
    static constexpr int kStages = D == 128 ? 4 : 8;
    static constexpr int kPBytes = 16384;                 // 128 rows x 64 bf16
    static constexpr int kOffQ = 0;
    static constexpr int kOffStage = kQBytes;
    static constexpr int kOffP = kOffStage + kStages * kStageBytes;
    static constexpr int kSmem = kOffP + 2 * kPBytes + 1024;   // + alignment slack
    static constexpr uint32_t kTmemCols = 256;            // S0 [0,64)  S1 [64,128)  O [128,128+D)
    static constexpr uint32_t kColO = 128;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

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

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The barrier arrives once every MMA issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
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

struct PfBars {
    uint64_t q_full, q_empty, s_full[2], p_full[2], pv_done[2], mma_done;
};

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map, const __grid_constant__ PrefillArgs a) {
    using C = PfCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t kv_full[C::kStages];
    __shared__ __align__(8) uint64_t kv_empty[C::kStages];
    __shared__ __align__(8) PfBars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t q_s = sb + C::kOffQ, st_s = sb + C::kOffStage, p_s = sb + C::kOffP;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(a.ws + a.L.ctrl);
    volatile int* abort = &s_abort;

    // Rows of the Q tile that no token fills stay zero.
    for (int i = tid; i < C::kQBytes / 16; i += kPfThreads)
        reinterpret_cast<uint4*>(sm + C::kOffQ)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&kv_full[s]), 1);
            mbar_init(smem_u32(&kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&bars.q_full), 1);
        mbar_init(smem_u32(&bars.q_empty), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars.s_full[b]), 1);
            mbar_init(smem_u32(&bars.p_full[b]), 128);
            mbar_init(smem_u32(&bars.pv_done[b]), 1);
        }
        mbar_init(smem_u32(&bars.mma_done), 1);
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
    const int Hk = a.kv_heads, g = a.group, Tq = a.tile_tokens;
    const int n_units = (ctrl->magic == kPlanMagic ? ctrl->n_items : 0) * Hk;
    const PfTile* tiles = reinterpret_cast<const PfTile*>(a.ws + a.L.tiles);

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t it = 0, ui = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++ui) {
                const PfTile t = tiles[u / Hk];
                const int kvh = u % Hk;
                ok = pf_wait(smem_u32(&bars.q_empty), (ui & 1) ^ 1, abort, ctrl);
                if (!ok) break;
                mbar_arrive_expect_tx(smem_u32(&bars.q_full), C::kBoxes * 128 * g * Tq);
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(q_s + b * 16384, &q_map, b * 64, kvh * g, t.t0, smem_u32(&bars.q_full));
                const int* trow = a.table + (size_t)t.row * a.pages_per_row;
                for (int k = 0; k < t.npg; ++k, ++it) {
                    const int s = it % C::kStages;
                    ok = pf_wait(smem_u32(&kv_empty[s]), ((it / C::kStages) & 1) ^ 1, abort, ctrl);
                    if (!ok) break;
                    int page = __ldg(trow + t.first_page + k);
                    if (page < 0 || page >= a.num_pages) {
                        set_error(ctrl, kErrBadPage);
                        page = 0;
                    }
                    const int y = (page * Hk + kvh) * kPageSize;
                    const uint32_t kb = st_s + s * C::kStageBytes, vb = kb + C::kKvBytes;
                    mbar_arrive_expect_tx(smem_u32(&kv_full[s]), C::kStageBytes);
                    for (int b = 0; b < C::kBoxes; ++b) {
                        tma_load_2d(kb + b * 8192, &k_map, b * 64, y, smem_u32(&kv_full[s]));
                        tma_load_2d(vb + b * 8192, &v_map, b * 64, y, smem_u32(&kv_full[s]));
                    }
                }
            }
            // Drain: the last load of each stage and of Q has landed before exit.
            for (uint32_t k = 0; k < (uint32_t)C::kStages && k < it; ++k) {
                const uint32_t j = it - 1 - k;
                mbar_wait(smem_u32(&kv_full[j % C::kStages]), (j / C::kStages) & 1, kPfTimeoutNs);
            }
            if (ui > 0) mbar_wait(smem_u32(&bars.q_full), (ui - 1) & 1, kPfTimeoutNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = instr_desc(128, 64, 0, 0);
            constexpr uint32_t idesc_o = instr_desc(128, D, 0, 1);
            uint32_t it = 0, ui = 0;
            bool ok = true;
            // O += P_j V_j; the first page of a unit overwrites O.
            auto pv = [&](uint32_t j, bool first) -> bool {
                if (!pf_wait(smem_u32(&bars.p_full[j & 1]), (j >> 1) & 1, abort, ctrl)) return false;
                tc_fence_after();
                const uint32_t vb = st_s + (j % C::kStages) * C::kStageBytes + C::kKvBytes;
                const uint32_t pb = p_s + (j & 1) * C::kPBytes;
                #pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16(tmem + C::kColO, smem_desc(pb + ks * 32, 16, 1024),
                              smem_desc(vb + ks * 2048, 8192, 1024), idesc_o, (first && ks == 0) ? 0u : 1u);
                umma_commit(smem_u32(&bars.pv_done[j & 1]));
                umma_commit(smem_u32(&kv_empty[j % C::kStages]));
                return true;
            };
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++ui) {
                const PfTile t = tiles[u / Hk];
                ok = pf_wait(smem_u32(&bars.q_full), ui & 1, abort, ctrl);
                if (!ok) break;
                tc_fence_after();
                for (int k = 0; k < t.npg && ok; ++k) {
                    const uint32_t j = it + k;
                    const int s = j % C::kStages;
                    ok = pf_wait(smem_u32(&kv_full[s]), (j / C::kStages) & 1, abort, ctrl);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kb = st_s + s * C::kStageBytes;
                    #pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma_bf16(tmem + (j & 1) * 64, smem_desc(q_s + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                  smem_desc(kb + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), idesc_s,
                                  ks > 0 ? 1u : 0u);
                    umma_commit(smem_u32(&bars.s_full[j & 1]));
                    if (k > 0) ok = pv(j - 1, k == 1);
                }
                if (!ok) break;
                umma_commit(smem_u32(&bars.q_empty));      // Q is free once every S of the unit is done
                ok = pv(it + t.npg - 1, t.npg == 1);
                it += t.npg;
            }
            // Drain: every MMA issued has finished before TMEM is freed.
            if (ui > 0) {
                umma_commit(smem_u32(&bars.mma_done));
                mbar_wait(smem_u32(&bars.mma_done), 0, kPfTimeoutNs);
            }
        }
    } else {
        // ---------------- softmax + epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;
        const int m = quarter * 32 + lane;           // MMA row = TMEM lane
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const int tq = m / g, jh = m % g;
        const float sl2 = a.scale_log2;
        const __nv_bfloat16* sinks = static_cast<const __nv_bfloat16*>(a.sinks);
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const PfTile t = tiles[u / Hk];
            const int kvh = u % Hk;
            const bool active = tq < Tq && tq < t.ntok;
            int pos = -1, lo = 0;
            if (active) {
                pos = __ldg(a.positions + t.t0 + tq);
                pos = pos < 0 ? 0 : pos;
                lo = (a.window > 0 && pos - a.window + 1 > 0) ? pos - a.window + 1 : 0;
            }
            float m_run = -INFINITY, l = 0.f;
            for (int k = 0; k < t.npg; ++k) {
                const uint32_t j = it + k;
                const int pg = t.first_page + k;
                ok = pf_wait(smem_u32(&bars.s_full[j & 1]), (j >> 1) & 1, abort, ctrl);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t s[64];
                tmem_ld32(tmem + lane_base + (j & 1) * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld32(tmem + lane_base + (j & 1) * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tmem_wait_ld();
                // keys c of this page visible to the row: lo <= pg*64 + c <= pos
                const int c_lo = lo - pg * kPageSize, c_hi = pos - pg * kPageSize;
                float x[64];
                float mx = -INFINITY;
                #pragma unroll
                for (int c = 0; c < 64; ++c) {
                    x[c] = (c >= c_lo && c <= c_hi) ? __uint_as_float(s[c]) * sl2 : -INFINITY;
                    mx = fmaxf(mx, x[c]);
                }
                const bool need = mx > m_run + kRescaleLog2;
                float alpha = 1.f;
                if (need) {
                    alpha = exp2_approx(m_run - mx);   // 0 while m_run is -inf
                    m_run = mx;
                    l *= alpha;
                }
                const float mu = m_run == -INFINITY ? 0.f : m_run;
                uint32_t pk[32];
                float sum = 0.f;
                // The denominator sums the bf16 weights the PV MMA multiplies,
                // so the normalised weights are an exact convex combination.
                #pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    pk[c >> 1] = pack_bf16x2(exp2_approx(x[c] - mu), exp2_approx(x[c + 1] - mu));
                    const float2 r = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[c >> 1]));
                    sum += r.x + r.y;
                }
                l += sum;
                // PV of the previous page is done: O may be rescaled, P buffer j&1 is free.
                if (j > 0) {
                    ok = pf_wait(smem_u32(&bars.pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, abort, ctrl);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                }
                if (k > 0 && __any_sync(0xffffffffu, need && alpha != 1.f)) {
                    #pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + C::kColO + c0, o);
                        tmem_wait_ld();
                        #pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(tmem + lane_base + C::kColO + c0, o);
                    }
                    tmem_wait_st();
                }
                const uint32_t pb = p_s + (j & 1) * C::kPBytes;
                #pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                 ::"r"(swz128(pb, m, ch)), "r"(pk[4 * ch]), "r"(pk[4 * ch + 1]),
                                   "r"(pk[4 * ch + 2]), "r"(pk[4 * ch + 3])
                                 : "memory");
                // V rows outside every row's range hold no cached value of this
                // tile (possibly stale or non-finite): zero them so 0 * V stays 0.
                const int v_lo = t.lo_min - pg * kPageSize, v_hi = t.pos_max - pg * kPageSize;
                if (v_lo > 0 || v_hi < kPageSize - 1) {
                    const uint32_t vb = st_s + (j % C::kStages) * C::kStageBytes + C::kKvBytes;
                    for (int i = m; i < kPageSize * C::kBoxes * 8; i += 128) {
                        const int r = i / (C::kBoxes * 8), rest = i % (C::kBoxes * 8);
                        if (r < v_lo || r > v_hi)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                                         ::"r"(vb + (rest >> 3) * 8192 + r * 128 + (rest & 7) * 16), "r"(0)
                                         : "memory");
                    }
                }
                fence_proxy_async_shared();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars.p_full[j & 1]));
            }
            if (!ok) break;
            // Epilogue: O / l (with the sink's share of the denominator).
            const uint32_t jl = it + t.npg - 1;
            ok = pf_wait(smem_u32(&bars.pv_done[jl & 1]), (jl >> 1) & 1, abort, ctrl);
            ok = __all_sync(0xffffffffu, ok);
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
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(t.t0 + tq) * a.heads + h) * D;
            #pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + C::kColO + c0, o);
                tmem_wait_ld();
                if (active) {
                    #pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c0 + 8 * v) = w;
                    }
                }
            }
            // The next unit's first PV overwrites O only after this read
            // (its p_full arrival follows in program order).
            tc_fence_before();
            it += t.npg;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
}

template <int D>
cudaError_t launch_d(const PrefillArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                     const CUtensorMap& v_map, int grid, cudaStream_t stream) {
    auto kern = prefill_kernel<D>;
    static int configured_mask = 0;   // bit per device id < 31
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<D>::kSmem);
        if (e != cudaSuccess) return e;
        if (dev < 31) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = PfCfg<D>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, q_map, k_map, v_map, a);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, int grid, cudaStream_t stream) {
    if (a.head_dim == 128) return launch_d<128>(a, q_map, k_map, v_map, grid, stream);
    if (a.head_dim == 64) return launch_d<64>(a, q_map, k_map, v_map, grid, stream);
    return cudaErrorInvalidValue;
}

size_t prefill_smem_bytes(int head_dim) {
    return head_dim == 128 ? PfCfg<128>::kSmem : PfCfg<64>::kSmem;
}

}  // namespace pdattn
