// Device helpers shared by the pdattn kernels: inline PTX for mbarriers,
// TMA / bulk copies, warp-level MMA, and the workspace layout.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pdattn {

constexpr int kPageSize = 64;
constexpr int kMaxGroup = 8;          // query heads per kv head (the MMA's N)
constexpr int kChunkMax = 64;         // largest pages-per-split the planner picks
constexpr int kItemsPerCta = 4;       // planner's target work items per persistent CTA
constexpr uint32_t kPlanMagic = 0x70646174u;

// Status bits in the workspace's status word.
constexpr int kErrBadPage = 1;
constexpr int kErrBadPos = 2;
constexpr int kErrTimeout = 4;
constexpr int kErrBadPlan = 8;

// Control block at the start of the workspace (256 bytes).
struct Ctrl {
    int status;        // OR of kErr* bits; cleared by pdattn_check_status
    int next_item;     // persistent-scheduler cursor (decode: starts at `grid`; prefill / packed: at 0)
    int done_ctas;     // CTAs that finished fetching work
    int n_items;       // work items in the plan
    int chunk_pages;   // pages per split chosen by the plan
    uint32_t magic;    // kPlanMagic once a plan is written
    int rows, kv_heads, pages_per_row, max_items, group, head_dim;
    int grid;          // persistent CTAs of the attention launch: CTA b starts with item b
    // Test hook, never set by a call: when nonzero, CTA 0 of the decode
    // attention kernel leaves the first stage of its first item unissued, so
    // that the consumers' bounded wait on it runs out (the timeout path).
    int test_hold;
    int pad[50];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");
static_assert(offsetof(Ctrl, test_hold) == 52, "test hook offset is part of the test contract");

// One work item of the plan: pages [first_page, first_page + npg) of one
// (row, kv head), chunk `chunk` of `nch`; `slot` indexes its fp32 partial.
// Self-contained so that the scheduler needs one load per item.
struct __align__(32) ItemDesc {
    int row, kvh_chunk, nch, slot;     // kvh_chunk = kv_head << 16 | chunk
    int first_page, npg, pos, lo;      // visible positions of the row: [lo, pos]
};
static_assert(sizeof(ItemDesc) == 32, "item descriptor is 32 bytes");

// Byte offsets of the workspace regions (all 256-byte aligned).
struct WsLayout {
    size_t ctrl, row_info, items, merge_cnt, part_ml, part_o, q_rot, total;
    int max_items;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// The split plan's arithmetic, shared by the planner and by the attention
// kernel, which derives its first item from the same inputs (positions,
// windows, split size) before the plan is ready.
// ---------------------------------------------------------------------------

// Visible positions of a row: [lo, pos] with lo = 0 or pos - window + 1.
__host__ __device__ __forceinline__ int row_lo(int pos, int window) {
    return (window > 0 && pos - window + 1 > 0) ? pos - window + 1 : 0;
}

// Pages per split.  A split costs its chunk a partial write and the row a
// merge, so rows stay whole (up to kChunkMax pages) unless the longest row
// exceeds twice the average work per CTA, or there are fewer than two
// (row, kv head) pairs per CTA; then chunks aim at kItemsPerCta (long rows)
// or 2 * kItemsPerCta (few pairs) items per CTA.  Sweeps on GB300: whole
// rows are 4-21% faster wherever the balance allows them (gpt-oss-20b, the
// serving batch); 32 Llama rows (256 pairs) run 3% faster in 16-page chunks.
__host__ __device__ __forceinline__ int choose_chunk(unsigned long long row_pages, int max_row_pages, int rows,
                                                     int Hk, int grid) {
    const unsigned long long work = row_pages * (unsigned long long)Hk;   // page items
    const bool few_pairs = (long long)rows * Hk < 2ll * grid;
    if (!few_pairs && (unsigned long long)max_row_pages * grid <= 2ull * work) return kChunkMax;
    const unsigned long long per = (unsigned long long)(few_pairs ? 2 * kItemsPerCta : kItemsPerCta) * grid;
    const unsigned long long cc = (work + per - 1) / per;
    return (int)(cc < 1 ? 1 : (cc > kChunkMax ? kChunkMax : cc));
}

// A row of n visible pages in nch = ceil(n / C) chunks of equal size, up to
// one page apart: the first `big` chunks hold q + 1 pages, the others q (so
// no row ends in a short tail chunk whose merge would come last).
struct Chunking {
    int nch, q, big;
    __host__ __device__ Chunking(int n, int C)
        : nch((n + C - 1) / C), q(n > 0 ? n / ((n + C - 1) / C) : 0), big(n > 0 ? n % ((n + C - 1) / C) : 0) {}
    __host__ __device__ int size(int c) const { return c < big ? q + 1 : q; }
    __host__ __device__ int start(int c) const { return c * q + (c < big ? c : big); }   // pages after the row's first
};

// The plan's first wave.  With at most kFirstWaveRows rows, items
// [0, first_wave) are chunk 0 of the (row, kv head) pairs 0, 1, ... in
// row-major order (an invalid row leaves an empty item, npg 0), and the
// chunks' merge slots start at an exclusive prefix sum of nch * kv_heads over
// the rows.  The attention kernel's CTA b can then derive item b from the
// call's inputs and start loading it before the planner has finished.  The
// other items follow, largest first.
constexpr int kFirstWaveRows = 512;
__host__ __device__ __forceinline__ int first_wave(int rows, int kv_heads, int grid) {
    const long long pairs = (long long)rows * kv_heads;
    return rows <= kFirstWaveRows ? (int)(pairs < grid ? pairs : grid) : 0;
}

// max work items: min over split choices of the planner, see the planner
// (plus one empty first-wave item per CTA at most).
__host__ __device__ inline int plan_max_items(int rows, int kv_heads, int pages_per_row,
                                              int chunk_pages, int grid) {
    long long rh = (long long)rows * kv_heads;
    long long n;
    if (chunk_pages > 0) {
        n = rh * ((pages_per_row + chunk_pages - 1) / chunk_pages);
    } else {
        long long a = 2ll * kItemsPerCta * grid + rh;   // the few-pairs target of choose_chunk
        long long b = rh * ((pages_per_row + kChunkMax - 1) / kChunkMax);
        n = a > b ? a : b;
    }
    return (int)(n + grid);
}

__host__ __device__ inline WsLayout ws_layout(int rows, int heads, int kv_heads, int head_dim,
                                              int pages_per_row, int elem_bytes, int chunk_pages,
                                              int grid) {
    WsLayout L;
    int g = heads / kv_heads;
    L.max_items = plan_max_items(rows, kv_heads, pages_per_row, chunk_pages, grid);
    size_t off = 0;
    L.ctrl = off; off += 256;
    L.row_info = off; off = align256(off + sizeof(int4) * (size_t)rows);
    L.items = off; off = align256(off + sizeof(ItemDesc) * (size_t)L.max_items);
    L.merge_cnt = off; off = align256(off + sizeof(int) * (size_t)rows * kv_heads);
    L.part_ml = off; off = align256(off + sizeof(float2) * (size_t)L.max_items * g);
    L.part_o = off; off = align256(off + sizeof(float) * (size_t)L.max_items * g * head_dim);
    L.q_rot = off; off = align256(off + (size_t)elem_bytes * rows * heads * head_dim);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------------------
// Paged prefill: tiles of consecutive tokens of one row and the workspace.
// ---------------------------------------------------------------------------
constexpr int kPfRows = 128;          // MMA rows of half a prefill tile: tokens x query heads of a group

// Tokens [t0, t0 + ntok) of table row `row`; they see pages
// [first_page, first_page + npg) of the row, positions [lo_min, pos_max].
struct __align__(32) PfTile {
    int t0, ntok, row, first_page;
    int npg, lo_min, pos_max, pad;
};
static_assert(sizeof(PfTile) == 32, "prefill tile descriptor is 32 bytes");

struct PfLayout {
    size_t ctrl, tiles_raw, tiles, q_rot, total;
    // packed attention only (0 otherwise): rotated keys [n, kv_heads, D],
    // segment ids and positions padded to whole 64-token blocks, and one
    // int4 summary per block {all one segment, segment, min pos, max pos}
    size_t k_rot, seg_pad, pos_pad, blk;
};

// Tiles never outnumber tokens.
__host__ __device__ inline PfLayout pf_layout(int n_tokens, int heads, int head_dim, int elem_bytes) {
    PfLayout L;
    size_t off = 0;
    L.ctrl = off; off += 256;
    L.tiles_raw = off; off = align256(off + sizeof(PfTile) * (size_t)n_tokens);
    L.tiles = off; off = align256(off + sizeof(PfTile) * (size_t)n_tokens);
    L.q_rot = off; off = align256(off + (size_t)elem_bytes * n_tokens * heads * head_dim);
    L.total = off;
    L.k_rot = L.seg_pad = L.pos_pad = L.blk = 0;
    return L;
}

__host__ __device__ inline PfLayout pk_layout(int n_tokens, int heads, int kv_heads, int head_dim, int elem_bytes) {
    PfLayout L = pf_layout(n_tokens, heads, head_dim, elem_bytes);
    const size_t blocks = ((size_t)n_tokens + kPageSize - 1) / kPageSize;
    size_t off = L.total;
    L.k_rot = off; off = align256(off + (size_t)elem_bytes * n_tokens * kv_heads * head_dim);
    L.seg_pad = off; off = align256(off + sizeof(int) * blocks * kPageSize);
    L.pos_pad = off; off = align256(off + sizeof(int) * blocks * kPageSize);
    L.blk = off; off = align256(off + sizeof(int4) * blocks);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking check of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; gives up after
// `timeout_ns` and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t timeout_ns = 2000000000ull) {
    if (mbar_test_wait(bar, parity)) return true;
    #pragma unroll 1
    for (int i = 0; i < 256; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    #pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// Fetch the 128-byte line holding `p` into L2 (a hint: no data returns).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Register-only instructions are not volatile so the compiler may schedule
// them around the (volatile, ordered) shared-memory loads.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x on the SFU.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Address of 16-byte chunk `chunk` (0..7) of row `row` in a 64-row x 128-byte
// box written by TMA with 128-byte swizzling (box base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t box, int row, int chunk) {
    return box + row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void set_error(Ctrl* ctrl, int bits) { atomicOr(&ctrl->status, bits); }

// atomicAdd with acquire-release semantics at GPU scope: the caller's earlier
// writes (and those ordered before them in its warp) are visible to whoever
// acquires the new value, and writes released before the value it reads are
// visible to the caller.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// A bounded wait ran out: record it and withdraw the plan, whose cursor and
// merge counters are now stale, so that a later attention-only call on this
// workspace is refused (kErrBadPlan) until a planner runs again.
__device__ __forceinline__ void fail_timeout(Ctrl* ctrl) {
    set_error(ctrl, kErrTimeout);
    atomicExch(&ctrl->magic, 0u);
}

}  // namespace pdattn
