// sm_103a fused restore + tensor-core product for prefill
// (afx_prefill_fused, afx_prefill_fused_batch).
//
// The operation: Y[t][r] = sum_c W[r][c] X[t][c] for the N token vectors of
// a prompt ("Memory requirements of language model inference on a consumer
// GPU", section "Loading one part of the model at a time": the prompt goes
// through each layer as a whole before the answer is produced token by
// token), with W restored from its exponent-coded container on the way ("Why
// Weight Offloading Slows Inference", section "Lossless compression: fewer
// bytes to read, more work to unpack": the released bits are restored before
// compute; the restore is that page's t_unpack of Eq. (1)).  No restored
// matrix is ever written out: restored weights pass through a small ring
// per CTA that stays in L2 on their way to the tensor cores.
//
// Weight order.  The container holds W in tile order: 128 x 64 tiles of W,
// row-major inside a tile, the tiles of one 128-row band (an "m-tile") in
// column order, the bands in row order (afx_tile_order writes it).  A
// band's weights are then one contiguous range of the stream, and each
// 8192-weight tile is the A operand of four MMAs (K = 16 each).
//
// Work decomposition.  A work item is one m-tile of one matrix for one pass
// of up to 512 tokens; the host assigns items to persistent CTAs (longest
// first, each to the least loaded CTA), one CTA per SM.
//   - 22 decoding warps restore the item's sub-tiles (32 chunks each,
//     interleaved across the warps) with the byte-step decoder of the
//     restore kernel.  A warp decodes into its stage first (that needs no
//     output position), then places the sub-tile by adding the code counts
//     the warps before it published in shared memory after their scans, and
//     stores the restored weights, joined with their sign|mantissa bytes,
//     into the CTA's ring of 16 tiles in global memory (256 KB, written and
//     read back within microseconds, so it stays in L2) with coalesced
//     16-byte stores.  Each store range is counted into the tile's barrier;
//     the 8192th weight completes it;
//   - a producer lane moves each complete tile from the ring into one of
//     two shared-memory A stages with TMA (128-byte rows and swizzle), and
//     a second producer lane loads the token vectors: 64 columns x up to
//     128 tokens per stage (128-byte swizzle), a 48 KB ring of stages;
//   - an MMA warp issues tcgen05.mma (M = 128, N = up to 128 tokens, K = 16)
//     into up to four float32 accumulators in tensor memory (512 tokens a
//     pass) and frees ring tiles and stages with tcgen05.commit;
//   - four epilogue warps read the accumulators with tcgen05.ld (each its
//     32-lane quarter) and store Y, row by row of W, coalesced across lanes.
// Every wait is bounded; a wait that runs out sets AFX_DEV_TIMEOUT and an
// abort flag that every role polls, copies in flight are waited for, and the
// CTA frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <queue>
#include <vector>

#include "afx_warp_decode.cuh"

namespace afx {

constexpr int kPfDecodeWarps = 22;
constexpr int kPfProducerWarp = kPfDecodeWarps;      // lane 0: A tiles, lane 16: token vectors
constexpr int kPfMmaWarp = kPfDecodeWarps + 1;
constexpr int kPfEpiWarp0 = kPfDecodeWarps + 2;
constexpr int kPfWarps = kPfDecodeWarps + 6;
constexpr int kPfThreads = kPfWarps * 32;
constexpr uint32_t kDecodeBarrier = 1;                // named barrier of the decoding warps
constexpr uint32_t kSliceK = 16;                      // K of one MMA
constexpr uint32_t kTileRows = 128, kTileCols = 64, kTileElems = kTileRows * kTileCols;  // an A tile
constexpr uint32_t kTileBytes = kTileElems * 2;
constexpr uint32_t kRingTiles = 16;                  // A tiles in the CTA's ring in global memory (256 KB)
constexpr uint32_t kAStages = 2;                      // A tiles in shared memory
constexpr uint32_t kBRingBytes = 49152;               // the activation ring: as many stages as fit, at most kBSlotsMax
constexpr uint32_t kBSlotsMax = 16;
constexpr uint32_t kTotRing = 128;                    // published sub-tile code counts
constexpr uint32_t kMaxHalfTokens = 128;              // N of one MMA
constexpr uint32_t kMaxHalves = 4;                    // accumulators of one pass
constexpr uint32_t kMaxPassTokens = kMaxHalves * kMaxHalfTokens;
constexpr int kPfMaxItems = 2048;
constexpr int kPfMaxCtas = 256;

static_assert(kPfThreads <= 1024, "one CTA of at most 1024 threads");
static_assert(kTileCols / kSliceK == 4, "four K = 16 MMAs per 64-column tile");
static_assert(kPfEpiWarp0 % 4 == 0, "the epilogue warps cover the four lane quarters of tensor memory in order");
static_assert(kPfDecodeWarps - 1 <= 32 && kTotRing >= 4 * kPfDecodeWarps, "look-back reads one count per lane");

struct PrefillMatrix {
    TensorArgs t;       // sections, geometry and code tables; t.y = Y [n_tokens][rows]
    uint32_t k_tiles;   // A tiles per m-tile: cols / 64
    uint32_t single;    // 1: one exponent for every weight (no coded stream)
    uint32_t fill;      // that exponent
};

// An item: matrix << 28 | pass << 19 | part << 17 | m-tile.  part 0 is the
// whole m-tile, 1 and 2 its first and second half of the tiles (an m-tile
// split in two along K for balance; each half's products are added into a
// zeroed Y, and two float32 partial sums added to zero give the same bits in
// either order).
struct ItemInfo {
    uint32_t mi, pass, part, mt;
};

__host__ __device__ inline ItemInfo item_info(uint32_t code) {
    return ItemInfo{code >> 28, (code >> 19) & 0x1FFu, (code >> 17) & 3u, code & 0x1FFFFu};
}

__host__ __device__ inline uint32_t item_code(uint32_t mi, uint32_t pass, uint32_t part, uint32_t mt) {
    return mi << 28 | pass << 19 | part << 17 | mt;
}

// The item's tiles [kb, ke) of its m-tile's k_tiles.
__host__ __device__ inline void item_tiles(uint32_t part, uint32_t k_tiles, uint32_t* kb, uint32_t* ke) {
    *kb = part == 2 ? k_tiles / 2 : 0;
    *ke = part == 1 ? k_tiles / 2 : k_tiles;
}

struct PrefillArgs {
    CUtensorMap tmap[kMaxTensors];  // X of each matrix: [n_tokens][cols] BF16, box 64 x n_mma, 128-byte swizzle
    CUtensorMap ring_map;           // the rings: [CTAs * 16 * 128][64] BF16, box 64 x 128, 128-byte swizzle
    PrefillMatrix m[kMaxTensors];
    uint16_t* ring;                 // CTA c's ring at ring + c * 16 * 8192
    uint32_t count, n_tokens, n_mma, halves, pass_tokens, tab_bytes, tmem_cols, wait_limit, max_chunk_bytes;
    int32_t* status;
    uint16_t cta_begin[kPfMaxCtas + 1];
    uint32_t items[kPfMaxItems];
};

// Control block in shared memory.
struct PfCtl {
    uint64_t ring_full[kRingTiles], ring_empty[kRingTiles];
    uint64_t a_full[kAStages], a_empty[kAStages];
    uint64_t b_full[kBSlotsMax], b_empty[kBSlotsMax];
    uint64_t acc_full, acc_empty, drain_a, drain_b, drain_mma;
    uint64_t totals[kTotRing];  // (ordinal + 1) << 32 | code count of a sub-tile, at ordinal % kTotRing
    uint32_t tmem_base;
    int32_t abort_flag;
};

// Shared-memory layout (offsets from a 1024-byte aligned base).
struct PfLayout {
    uint32_t a, b, b_stage, b_slots, ctl, shw, slots, streams, wstride, total;
};

__host__ __device__ inline uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline PfLayout pf_layout(uint32_t tab_bytes, uint32_t n_mma, uint32_t max_chunk_bytes) {
    PfLayout L;
    L.a = 0;
    // an activation stage holds 64 columns of the tokens of one
    // accumulator; small stages come many to the ring
    L.b_stage = round_up(n_mma * kTileCols * 2, 1024);
    L.b_slots = kBRingBytes / L.b_stage < kBSlotsMax ? kBRingBytes / L.b_stage : kBSlotsMax;
    L.b = L.a + kAStages * kTileBytes;
    L.ctl = L.b + L.b_slots * L.b_stage;
    L.shw = round_up(L.ctl + static_cast<uint32_t>(sizeof(PfCtl)), 16);
    L.slots = round_up(L.shw + static_cast<uint32_t>(sharedw_table_offset()) + tab_bytes, 16);
    L.streams = L.slots + kPfDecodeWarps * static_cast<uint32_t>(sizeof(WarpSlot));
    L.wstride = kWarpChunks * max_chunk_bytes + kStreamPad;
    L.total = L.streams + kPfDecodeWarps * 2 * L.wstride;
    return L;
}

// ---- tensor-core, TMA and barrier helpers ------------------------------------------

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// OR of p over the n threads of named barrier id (a barrier as well).
__device__ __forceinline__ bool named_red_or(uint32_t id, uint32_t n, bool p) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(p ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

struct DecodeSync {
    __device__ __forceinline__ void operator()() const { named_sync(kDecodeBarrier, kPfDecodeWarps * 32); }
};

__device__ __forceinline__ void mbar_init_count(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// The 16 x rows box at (x, y) of the tensor map into shared dst, completing on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint32_t x, uint32_t y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Shared-memory matrix descriptor, K-major, 128-byte rows with the
// 128-byte swizzle, 8-row groups 1024 bytes apart (both operands, as the
// TMA writes them).  The K = 16 steps inside a 64-column tile start 32
// bytes apart.  Fields: start address >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29, unused for swizzled K-major), stride byte offset >> 4
// (32-45), descriptor version 1 (46), layout 2 = 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (uint64_t{1} << 16) | (uint64_t{1024 >> 4} << 32) |
           (uint64_t{1} << 46) | (uint64_t{2} << 61);
}

// D[tmem] (+)= A * B^T: BF16 operands, float32 accumulator.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc ? 1u : 0u)
        : "memory");
}

// bar gets one arrival once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_count(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Orders this thread's earlier generic-proxy writes to global memory before
// later async-proxy reads of them (the TMA loads of the ring).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

// Waits for phase `parity` of bar, at most limit polls, giving up early
// once another role has raised the abort flag.  A wait that runs out raises
// the flag and AFX_DEV_TIMEOUT.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, uint32_t limit, PfCtl& ctl, int32_t* status) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 31u && *reinterpret_cast<volatile int32_t*>(&ctl.abort_flag)) return false;
    }
    *reinterpret_cast<volatile int32_t*>(&ctl.abort_flag) = 1;
    raise_status(status, AFX_DEV_TIMEOUT);
    return false;
}

// ---- the decoding warps: restored weights into the ring ---------------------------------

// Stores tile weights [i0, i1) at dst (the tile's first weight in the
// ring): the stage byte of tile weight i is stage[(i + d) mod 2^32] (d is
// the tile's first position minus the stage's, which may be negative, and
// need not be a multiple of 8) and its sign|mantissa byte sm[i] (sm points
// at the tile's first weight).  Groups of 8 whole weights go out as 16-byte
// stores, one group per lane at a time; the partial groups at either end
// (shared with neighbouring ranges) weight by weight.
__device__ __forceinline__ void tile_store(uint16_t* dst, const uint8_t* stage, uint32_t d, const uint8_t* sm,
                                            uint32_t i0, uint32_t i1, int lane) {
    const uint32_t f0 = (i0 + 7) & ~7u, f1 = i1 & ~7u;
    const uint32_t head_end = f0 < i1 ? f0 : i1;
    for (uint32_t i = i0 + lane; i < head_end; i += 32) {
        const uint32_t k = i + d;  // stage index, wrapped to 32 bits
        AFX_CHECK(k < static_cast<uint32_t>(kWarpStage) && i < kTileElems, kChkMergeStage);
        dst[i] = join1(stage[k], __ldg(sm + i));
    }
    const uint32_t tail0 = f1 > f0 ? f1 : f0;
    for (uint32_t i = tail0 + lane; i < i1; i += 32) {
        const uint32_t k = i + d;
        AFX_CHECK(k < static_cast<uint32_t>(kWarpStage) && i < kTileElems, kChkMergeStage);
        dst[i] = join1(stage[k], __ldg(sm + i));
    }
    // the stage bytes of a group start at any byte: three aligned words,
    // shifted into place (i is a multiple of 8, so k & 3 == d & 3).  A lane
    // takes four groups at a time and loads their sign|mantissa bytes first,
    // so the four loads are in flight together
    const uint32_t sh = (d & 3u) * 8u;
    const uint32_t gend = f1 >> 3;
    for (uint32_t g0 = (f0 >> 3) + lane; g0 < gend; g0 += 128) {
        uint2 raw[4];
#pragma unroll
        for (uint32_t u = 0; u < 4; ++u) {
            const uint32_t g = g0 + 32 * u;
            raw[u] = g < gend ? __ldg(reinterpret_cast<const uint2*>(sm + (g << 3))) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (uint32_t u = 0; u < 4; ++u) {
            const uint32_t g = g0 + 32 * u;
            if (g < gend) {
                const uint32_t i = g << 3, k = i + d;
                AFX_CHECK(k + 8 <= static_cast<uint32_t>(kWarpStage) && i + 8 <= kTileElems, kChkMergeStage);
                const uint32_t* w = reinterpret_cast<const uint32_t*>(stage + (k & ~3u));
                const uint32_t w0 = w[0], w1 = w[1], w2 = (k & 3u) ? w[2] : 0u;
                const uint2 r8 = make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
                *reinterpret_cast<uint4*>(dst + i) = join8(r8, raw[u]);
            }
        }
    }
}

// The range [o0, o1) of the tensor's weights (positions in the container's
// tile order), clipped to the item's [p_lo, p_hi), into the CTA's ring: for
// each tile met, wait until its ring slot is free, store, and count the
// weights into the slot's barrier (8192 complete it).  The item's tiles
// have sequence numbers q_base + 0, 1, ...  Returns false when a wait gave
// up.
__device__ __forceinline__ bool ring_store(uint16_t* ring, PfCtl& ctl, const uint8_t* stage, uint64_t stage_o,
                                           const uint8_t* sm, uint64_t o0, uint64_t o1, uint64_t p_lo, uint64_t p_hi,
                                           uint32_t q_base, uint32_t wait_limit, int32_t* status, int lane) {
    const uint64_t c0 = o0 > p_lo ? o0 : p_lo, c1 = o1 < p_hi ? o1 : p_hi;
    if (c0 >= c1) return true;
    const uint32_t g0 = static_cast<uint32_t>((c0 - p_lo) / kTileElems), g1 = static_cast<uint32_t>((c1 - 1 - p_lo) / kTileElems);
    for (uint32_t g = g0; g <= g1; ++g) {
        const uint32_t q = q_base + g, slot = q % kRingTiles;
        if (!__all_sync(0xFFFFFFFFu,
                        pf_wait(&ctl.ring_empty[slot], ((q / kRingTiles) & 1u) ^ 1u, wait_limit, ctl, status)))
            return false;
        const uint64_t t_lo = p_lo + static_cast<uint64_t>(g) * kTileElems;
        const uint64_t a = c0 > t_lo ? c0 : t_lo, b = c1 < t_lo + kTileElems ? c1 : t_lo + kTileElems;
        const uint32_t i0 = static_cast<uint32_t>(a - t_lo), i1 = static_cast<uint32_t>(b - t_lo);
        AFX_CHECK(i1 <= kTileElems && a - stage_o + (i1 - i0) <= static_cast<uint64_t>(kWarpStage), kChkMergeStage);
        tile_store(ring + static_cast<size_t>(slot) * kTileElems, stage, static_cast<uint32_t>(t_lo - stage_o),
                    sm + t_lo, i0, i1, lane);
        fence_proxy_async_global();  // the TMA reads the tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive_count(&ctl.ring_full[slot], i1 - i0);
    }
    return true;
}

// The sub-tile holding the code of output position p: the last block whose
// index entry is <= p (a 32-way search, one load per lane and step), then
// the last of its 16 sub-tiles whose first code is at or before p; *start
// gets that sub-tile's first output position.
__device__ __forceinline__ uint64_t find_sub_tile(const TensorArgs& t, uint64_t p, int lane, uint64_t* start) {
    uint64_t lo = 0, hi = t.n_blocks;  // the block is in [lo, hi)
    while (hi - lo > 1) {
        const uint64_t step = (hi - lo + 31) / 32;
        const uint64_t idx = lo + static_cast<uint64_t>(lane) * step;
        const bool le = idx < hi && __ldg(t.block_index + idx) <= p;
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, le);
        const int top = m ? 31 - __clz(static_cast<int>(m)) : 0;
        lo = lo + static_cast<uint64_t>(top) * step;
        hi = lo + step < hi ? lo + step : hi;
    }
    const uint64_t b = lo;
    // lane l sums the counts of chunks [b * 512 + 16 l, + 16)
    uint32_t sum = 0;
    const uint64_t cbase = b * kThreads + static_cast<uint64_t>(lane) * 16;
#pragma unroll 4
    for (uint32_t j = 0; j < 16; ++j)
        if (cbase + j < t.n_chunks) sum += __ldg(t.chunk_index + cbase + j) >> 5;
    uint32_t inc = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (lane >= d) inc += o;
    }
    // sub-tile k starts after lanes 0 .. 2k-1: lane 2k's exclusive prefix
    const uint64_t start_k = __ldg(t.block_index + b) + (inc - sum);
    const uint64_t n_sub = (t.n_chunks + kWarpChunks - 1) / kWarpChunks;
    const bool cand = (lane & 1) == 0 && start_k <= p && b * kSubtilesPerBlock + (lane >> 1) < n_sub;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, cand);
    const int top = m ? 31 - __clz(static_cast<int>(m)) : 0;
    *start = __shfl_sync(0xFFFFFFFFu, start_k, top);
    return b * kSubtilesPerBlock + static_cast<uint64_t>(top >> 1);
}

// base plus the code counts of the `count` (<= 32) sub-tiles with ordinals
// ord0 .. ord0 + count - 1, read from the published counts: lane k waits
// until the entry of ordinal ord0 + k carries that ordinal.  Returns false
// when a wait gave up (the abort flag or the limit).
__device__ __forceinline__ bool add_published(PfCtl& ctl, uint32_t ord0, uint32_t count, uint64_t& base,
                                              uint32_t wait_limit, int32_t* status, int lane) {
    uint32_t v = 0;
    bool ok = true;
    if (static_cast<uint32_t>(lane) < count) {
        const uint32_t ord = ord0 + lane;
        const volatile uint64_t* e = &ctl.totals[ord % kTotRing];
        uint32_t i = 0;
        for (;; ++i) {
            const uint64_t x = *e;
            if (static_cast<uint32_t>(x >> 32) == ord + 1) {
                v = static_cast<uint32_t>(x);
                break;
            }
            if (i == wait_limit) {
                ok = false;
                *reinterpret_cast<volatile int32_t*>(&ctl.abort_flag) = 1;
                raise_status(status, AFX_DEV_TIMEOUT);
                break;
            }
            if ((i & 31u) == 31u && *reinterpret_cast<volatile int32_t*>(&ctl.abort_flag)) {
                ok = false;
                break;
            }
        }
    }
    base += warp_sum(v);
    return __all_sync(0xFFFFFFFFu, ok);
}

// Restores the item's weights [p_lo, p_hi) of tensor t with decoding warp
// `warp`: sub-tiles s_lo + warp, s_lo + warp + 26, ... of the sub-tiles that
// hold them, staged one ahead by bulk copies as in the restore kernel.  The
// item's sub-tiles have ordinals ord_base + (s - s_lo); each warp publishes
// its sub-tile's code count right after the scan and places the sub-tile
// from the counts of the sub-tiles before it (back to its own previous one).
// Returns false when a wait gave up (the staging copies still in flight are
// waited for first).
__device__ bool pf_decode_item(const TabView& tv, WarpSlot& ws, uint8_t* wstream, uint32_t wstride,
                               const TensorArgs& t, uint64_t p_lo, uint64_t p_hi, uint32_t q_base, uint32_t& ord_base,
                               uint16_t* ring, PfCtl& ctl, int warp, int lane, int32_t* status, uint32_t wait_limit,
                               uint32_t& phases) {
    const uint32_t T = t.chunk_bytes;
    const uint32_t chunk_bits = 8u * T;
    const uint32_t sub_bytes = kWarpChunks * T, sub_bits = 8u * sub_bytes;
    const bool fsm = t.tab.fsm != 0;
    const uint32_t skip_row0 = t.tab.fsm_rows * kFsmRowBytes;
    const uint64_t n_sub = (t.n_chunks + kWarpChunks - 1) / kWarpChunks;
    const uint64_t n = t.n;
    uint64_t start, unused;
    const uint64_t s_lo = find_sub_tile(t, p_lo, lane, &start);
    const uint64_t s_hi = find_sub_tile(t, p_hi - 1, lane, &unused) + 1;
    const uint32_t ord0 = ord_base;
    ord_base += static_cast<uint32_t>(s_hi - s_lo);
    uint64_t s = s_lo + static_cast<uint64_t>(warp);
    if (s >= s_hi || s_hi > n_sub) return true;
    const uint8_t* exp_base = reinterpret_cast<const uint8_t*>(t.exp_words);
    if (lane == 0)
        warp_issue_bulk(ws, wstream, t, s, s < t.n_sub_full, exp_base + s * sub_bytes,
                        t.chunk_index + s * kWarpChunks, sub_bytes, 0, false);
    // the first sub-tile starts after the counts of the item's sub-tiles before it
    uint32_t from = ord0, count = static_cast<uint32_t>(warp);
    int buf = 0;
    for (; s < s_hi; s += kPfDecodeWarps) {
        const uint64_t s_next = s + kPfDecodeWarps;
        const bool more = s_next < s_hi;
        const uint32_t ord = ord0 + static_cast<uint32_t>(s - s_lo);
        if (more && lane == 0)
            warp_issue_bulk(ws, wstream + (buf ^ 1) * wstride, t, s_next, s_next < t.n_sub_full,
                            exp_base + s_next * sub_bytes, t.chunk_index + s_next * kWarpChunks, sub_bytes, buf ^ 1,
                            false);
        const uint32_t parity = (phases >> buf) & 1u;
        const bool arrived = mbar_wait(&ws.bar[buf], parity, wait_limit);
        phases ^= 1u << buf;
        if (!__all_sync(0xFFFFFFFFu, arrived)) {
            // flag it, let the copies in flight land (bounded), and stop
            if (lane == 0) {
                raise_status(status, AFX_DEV_TIMEOUT);
                *reinterpret_cast<volatile int32_t*>(&ctl.abort_flag) = 1;
            }
            bool drained = mbar_wait(&ws.bar[buf], parity, wait_limit);
            if (more) {
                drained = mbar_wait(&ws.bar[buf ^ 1], (phases >> (buf ^ 1)) & 1u, wait_limit) && drained;
                phases ^= 1u << (buf ^ 1);
            }
            if (!__all_sync(0xFFFFFFFFu, drained) && lane == 0) raise_status(status, AFX_DEV_UNDRAINED);
            return false;
        }
        const bool full = s < t.n_sub_full;
        const uint32_t nexist =
            full ? 64u : static_cast<uint32_t>(min(t.n_chunks - min(t.n_chunks, s * kWarpChunks), uint64_t{64}));
        const uint32_t entry = static_cast<uint32_t>(lane) < nexist ? ws.chunk[buf][lane] : 0u;
        const uint32_t gap = entry & 31u;
        uint32_t cnt = entry >> 5;
        bool bad = false;
        if (gap > 23u || cnt > chunk_bits - gap || cnt > static_cast<uint32_t>(kMaxChunkCodes)) {
            bad = true;
            cnt = 0;
        }
        uint32_t inc = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if (lane >= d) inc += o;
        }
        const uint32_t total = __shfl_sync(0xFFFFFFFFu, inc, 31);
        if (lane == 0)  // the next sub-tiles' warps place theirs from this count
            *reinterpret_cast<volatile uint64_t*>(&ctl.totals[ord % kTotRing]) =
                (static_cast<uint64_t>(ord + 1) << 32) | total;
        // decode first, into the stage from index 0: it needs no output
        // position, so the warps before this one have time to publish theirs
        const uint32_t next = static_cast<uint32_t>(lane) + 1 < nexist ? ws.chunk[buf][lane + 1] : 0u;
        const uint32_t* stream = reinterpret_cast<const uint32_t*>(wstream + static_cast<size_t>(buf) * wstride);
        const uint32_t chunk_end = (lane + 1) * chunk_bits;
        bool stepped = false;
        FsmLane fl;
        if (cnt) {
            const uint32_t s_run = inc - cnt;
            if (fsm) {
                uint32_t stream_end = sub_bits;
                if (!full) {
                    const uint64_t bit0 = s * static_cast<uint64_t>(sub_bits);
                    const uint64_t left = t.total_bits > bit0 ? t.total_bits - bit0 : 0;
                    stream_end = left < sub_bits ? static_cast<uint32_t>(left) : sub_bits;
                }
                AFX_CHECK((lane + 1) * (T >> 2) <= wstride >> 2, kChkStreamWords);
                if (chunk_end <= stream_end) {
                    fsm_chunk_steps(tv, stream + lane * (T >> 2), T >> 2, gap, skip_row0, ws.stage, s_run, fl);
                    stepped = true;
                } else {
                    AFX_CHECK(s_run + cnt <= static_cast<uint32_t>(kWarpStage), kChkStageRun);
                    bad = decode_run_fsm(tv, stream, lane * (T >> 2), gap, cnt, ws.stage, s_run, next, chunk_end,
                                         stream_end);
                }
            } else {
                AFX_CHECK(s_run + cnt <= static_cast<uint32_t>(kWarpStage), kChkStageRun);
                bad = decode_run(tv, stream, warp_stream_bytes(t, s) >> 2, lane * (T >> 2), gap, cnt, ws.stage, s_run,
                                 next, chunk_end);
            }
        }
        __syncwarp();
        if (stepped) {
            AFX_CHECK(reinterpret_cast<uint8_t*>(fl.wout) + 4 <= ws.stage + kWarpStage, kChkStagePending);
            bad = fsm_chunk_finish(tv, stream, fl, cnt, chunk_end, next);
        }
        if (bad) raise_status(status, AFX_DEV_BAD_CHUNK);
        // this sub-tile starts after the published counts since `from`
        if (!add_published(ctl, from, count, start, wait_limit, status, lane)) {
            if (more) {  // the next sub-tile's copies are in flight: let them land
                const bool drained = mbar_wait(&ws.bar[buf ^ 1], (phases >> (buf ^ 1)) & 1u, wait_limit);
                phases ^= 1u << (buf ^ 1);
                if (!__all_sync(0xFFFFFFFFu, drained) && lane == 0) raise_status(status, AFX_DEV_UNDRAINED);
            }
            return false;
        }
        const uint64_t o0 = start, o1 = start + total;
        const bool in_range = o0 <= n && o1 <= n;
        if (lane == 0) {
            if (!in_range) {
                raise_status(status, AFX_DEV_BAD_BLOCK);
            } else {
                // the block index must agree with the counts where a block ends
                const uint64_t blk = s / kSubtilesPerBlock;
                if (s + 1 == n_sub) {
                    if (o1 != n || __ldg(t.block_index + t.n_blocks) != n) raise_status(status, AFX_DEV_BAD_BLOCK);
                } else if ((s + 1) % kSubtilesPerBlock == 0 && __ldg(t.block_index + blk + 1) != o1) {
                    raise_status(status, AFX_DEV_BAD_BLOCK);
                }
                if (s == 0 && o0 != 0) raise_status(status, AFX_DEV_BAD_BLOCK);
                if (o0 < o1) {  // the raw bytes the merge reads next
                    const uint64_t a0 = o0 & ~uint64_t(15), a1 = (o1 + 15) & ~uint64_t(15);
                    prefetch_l2(t.sm + a0, static_cast<uint32_t>(a1 - a0));
                }
                if (more && total) {
                    // and, one sub-tile ahead, those of this warp's next
                    // sub-tile: it starts about 21 sub-tiles of this one's
                    // size further on (256 weights of slack either side)
                    const uint64_t est = o1 + static_cast<uint64_t>(kPfDecodeWarps - 1) * total;
                    const uint64_t a0 = (est > 256 ? est - 256 : 0) & ~uint64_t(15);
                    const uint64_t e1 = est + total + 256 < n ? est + total + 256 : n;
                    const uint64_t a1 = (e1 + 15) & ~uint64_t(15);
                    if (a1 > a0) prefetch_l2(t.sm + a0, static_cast<uint32_t>(a1 - a0));
                }
            }
        }
        __syncwarp();
        // the sub-tile's weights go into the ring even when its stream was
        // bad (the output is then unspecified), so that every tile completes
        const uint64_t w0 = in_range ? o0 : 0, w1 = in_range ? o1 : 0;
        if (!ring_store(ring, ctl, ws.stage, o0, t.sm, w0, w1, p_lo, p_hi, q_base, wait_limit, status, lane)) {
            if (more) {  // the next sub-tile's copies are in flight: let them land
                const bool drained = mbar_wait(&ws.bar[buf ^ 1], (phases >> (buf ^ 1)) & 1u, wait_limit);
                phases ^= 1u << (buf ^ 1);
                if (!__all_sync(0xFFFFFFFFu, drained) && lane == 0) raise_status(status, AFX_DEV_UNDRAINED);
            }
            return false;
        }
        // the next sub-tile (26 on) starts after this one and the 25 between
        start = o1;
        from = ord + 1;
        count = kPfDecodeWarps - 1;
        buf ^= 1;
        fence_proxy_async_smem();  // this buffer's reads come before the bulk copy that refills it
        __syncwarp();
    }
    return true;
}

// Items of a tensor with one exponent for every weight: pieces of 2048
// weights, interleaved across the decoding warps, joined with the constant
// exponent (the warp's stage holds it at every index).
__device__ bool pf_fill_item(const PrefillMatrix& pm, WarpSlot& ws, uint64_t p_lo, uint64_t p_hi, uint32_t q_base,
                             uint16_t* ring, PfCtl& ctl, int warp, int lane, int32_t* status, uint32_t wait_limit) {
    constexpr uint32_t kPiece = 2048;
    static_assert(kPiece + 8 <= static_cast<uint32_t>(kWarpStage), "a fill piece fits the stage");
    const uint32_t f4 = ror8(pm.fill) * 0x01010101u;
    for (uint32_t i = lane; i < (kPiece + 8) / 4; i += 32) reinterpret_cast<uint32_t*>(ws.stage)[i] = f4;
    if (lane == 0 && warp == 0 && p_lo == 0 && __ldg(pm.t.block_index) != pm.t.n) raise_status(status, AFX_DEV_BAD_BLOCK);
    __syncwarp();
    for (uint64_t o = p_lo + static_cast<uint64_t>(warp) * kPiece; o < p_hi; o += kPfDecodeWarps * kPiece) {
        const uint64_t e = o + kPiece < p_hi ? o + kPiece : p_hi;
        if (!ring_store(ring, ctl, ws.stage, o, pm.t.sm, o, e, p_lo, p_hi, q_base, wait_limit, status, lane))
            return false;
    }
    return true;
}

// ---- the kernel ----------------------------------------------------------------------

__global__ void __launch_bounds__(kPfThreads, 1) prefill_fused_kernel(const __grid_constant__ PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const PfLayout L = pf_layout(a.tab_bytes, a.n_mma, a.max_chunk_bytes);
    uint8_t* stage_a = smem + L.a;
    uint8_t* ring_b = smem + L.b;
    PfCtl& ctl = *reinterpret_cast<PfCtl*>(smem + L.ctl);
    SharedW& sh = *reinterpret_cast<SharedW*>(smem + L.shw);
    uint8_t* tabr = smem + L.shw + sharedw_table_offset();
    WarpSlot* slots = reinterpret_cast<WarpSlot*>(smem + L.slots);
    uint16_t* const ring = a.ring + static_cast<size_t>(blockIdx.x) * kRingTiles * kTileElems;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t it0 = a.cta_begin[blockIdx.x], it1 = a.cta_begin[blockIdx.x + 1];
    const uint32_t wait_limit = a.wait_limit ? a.wait_limit : kWaitLimit;
    int32_t* const status = a.status;

    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < kRingTiles; ++i) {
            mbar_init_count(&ctl.ring_full[i], kTileElems);  // counts weights
            mbar_init_count(&ctl.ring_empty[i], 1);
        }
        for (uint32_t i = 0; i < kAStages; ++i) {
            mbar_init_count(&ctl.a_full[i], 1);
            mbar_init_count(&ctl.a_empty[i], 1);
        }
        for (uint32_t i = 0; i < L.b_slots; ++i) {
            mbar_init_count(&ctl.b_full[i], 1);
            mbar_init_count(&ctl.b_empty[i], 1);
        }
        for (uint32_t i = 0; i < kTotRing; ++i) ctl.totals[i] = 0;
        mbar_init_count(&ctl.acc_full, 1);
        mbar_init_count(&ctl.acc_empty, 4);
        mbar_init_count(&ctl.drain_mma, 1);
        ctl.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp < kPfDecodeWarps && lane == 0) {
        mbar_init(&slots[warp].bar[0]);
        mbar_init(&slots[warp].bar[1]);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == kPfMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&ctl.tmem_base)),
                     "r"(a.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;

    if (warp < kPfDecodeWarps) {
        // ---- restore the items' weights into the ring
        WarpSlot& ws = slots[warp];
        uint8_t* wstream = smem + L.streams + static_cast<size_t>(warp) * 2 * L.wstride;
        TabView tv;
        tv.lut = reinterpret_cast<const uint32_t*>(tabr);
        tv.len0 = tabr + kLutSize * 4;
        tv.limit = sh.ct.limit;
        tv.base = sh.ct.base;
        tv.sorted = sh.ct.sorted;
        tv.first = sh.first;
        tv.fsm = reinterpret_cast<const char*>(tabr);
        tv.depth = sh.ct.state_depth;
        tv.fsm_bytes = a.tab_bytes;
        tv.esc_base = ~0u;  // the state tables here hold every node
        uint32_t phases = 0, q_base = 0, ord_base = 0;
        int built = -1;
        for (uint32_t it = it0; it < it1; ++it) {
            const ItemInfo ii = item_info(a.items[it]);
            const uint32_t mi = ii.mi;
            const PrefillMatrix& pm = a.m[mi];
            uint32_t kb, ke;
            item_tiles(ii.part, pm.k_tiles, &kb, &ke);
            if (!pm.single && static_cast<int>(mi) != built) {
                // every decoding warp is done with the previous tables; all
                // build, or all skip once a wait anywhere has given up
                if (!named_red_or(kDecodeBarrier, kPfDecodeWarps * 32,
                                  *reinterpret_cast<volatile int32_t*>(&ctl.abort_flag) != 0))
                    build_tables_w(sh, tabr, pm.t.tab, threadIdx.x, kPfDecodeWarps * 32, DecodeSync{});
                built = static_cast<int>(mi);
            }
            const uint64_t p_lo = (static_cast<uint64_t>(ii.mt) * pm.k_tiles + kb) * kTileElems;
            const uint64_t p_hi = p_lo + static_cast<uint64_t>(ke - kb) * kTileElems;
            if (!*reinterpret_cast<volatile int32_t*>(&ctl.abort_flag)) {
                if (pm.single)
                    pf_fill_item(pm, ws, p_lo, p_hi, q_base, ring, ctl, warp, lane, status, wait_limit);
                else
                    pf_decode_item(tv, ws, wstream, L.wstride, pm.t, p_lo, p_hi, q_base, ord_base, ring, ctl, warp,
                                   lane, status, wait_limit, phases);
            }
            q_base += ke - kb;
        }
    } else if (warp == kPfProducerWarp) {
        if (lane == 0) {
            // ---- complete ring tiles into the A stages, in sequence
            uint32_t q = 0;
            bool ok = true;
            for (uint32_t it = it0; it < it1 && ok; ++it) {
                const ItemInfo ii = item_info(a.items[it]);
                uint32_t kb, ke;
                item_tiles(ii.part, a.m[ii.mi].k_tiles, &kb, &ke);
                for (uint32_t g = kb; g < ke; ++g, ++q) {
                    const uint32_t slot = q % kRingTiles, st = q % kAStages;
                    if (!pf_wait(&ctl.ring_full[slot], (q / kRingTiles) & 1u, wait_limit, ctl, status) ||
                        !pf_wait(&ctl.a_empty[st], ((q / kAStages) & 1u) ^ 1u, wait_limit, ctl, status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&ctl.a_full[st], kTileBytes);
                    tma_load_2d(stage_a + st * kTileBytes, &a.ring_map, 0,
                                (blockIdx.x * kRingTiles + slot) * kTileRows, &ctl.a_full[st]);
                }
            }
            if (!ok) {  // the loads still in flight land before the CTA exits
                for (uint32_t j = q > kAStages ? q - kAStages : 0; j < q; ++j)
                    if (!mbar_wait(&ctl.a_full[j % kAStages], (j / kAStages) & 1u, wait_limit))
                        raise_status(status, AFX_DEV_UNDRAINED);
            }
        } else if (lane == 16) {
            // ---- token vectors into the B ring, in the order the MMAs take them
            uint32_t bseq = 0;
            bool ok = true;
            const uint32_t stage_bytes = a.n_mma * kTileCols * 2;
            for (uint32_t it = it0; it < it1 && ok; ++it) {
                const ItemInfo ii = item_info(a.items[it]);
                const uint32_t mi = ii.mi;
                uint32_t kb, ke;
                item_tiles(ii.part, a.m[mi].k_tiles, &kb, &ke);
                const uint32_t y0 = ii.pass * a.pass_tokens;
                for (uint32_t g = kb; g < ke && ok; ++g)
                    for (uint32_t h = 0; h < a.halves; ++h) {
                        const uint32_t b = bseq % L.b_slots;
                        if (!pf_wait(&ctl.b_empty[b], ((bseq / L.b_slots) & 1u) ^ 1u, wait_limit, ctl, status)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(&ctl.b_full[b], stage_bytes);
                        tma_load_2d(ring_b + b * L.b_stage, &a.tmap[mi], g * kTileCols, y0 + h * a.n_mma, &ctl.b_full[b]);
                        ++bseq;
                    }
            }
            if (!ok) {
                for (uint32_t j = bseq > L.b_slots ? bseq - L.b_slots : 0; j < bseq; ++j)
                    if (!mbar_wait(&ctl.b_full[j % L.b_slots], (j / L.b_slots) & 1u, wait_limit))
                        raise_status(status, AFX_DEV_UNDRAINED);
            }
        }
        __syncwarp();
    } else if (warp == kPfMmaWarp) {
        // ---- the products, into the accumulator in tensor memory
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((a.n_mma >> 3) << 17) | ((kTileRows >> 4) << 24);
            uint32_t q = 0, bseq = 0, n_item = 0;
            bool ok = true;
            for (uint32_t it = it0; it < it1 && ok; ++it) {
                const ItemInfo ii = item_info(a.items[it]);
                uint32_t kb, ke;
                item_tiles(ii.part, a.m[ii.mi].k_tiles, &kb, &ke);
                if (n_item > 0) {  // the epilogue has read the previous item's accumulator
                    ok = pf_wait(&ctl.acc_empty, (n_item - 1) & 1u, wait_limit, ctl, status);
                    tc_fence_after();
                }
                for (uint32_t g = 0; g < ke - kb && ok; ++g, ++q) {
                    const uint32_t st = q % kAStages;
                    if (!pf_wait(&ctl.a_full[st], (q / kAStages) & 1u, wait_limit, ctl, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive(&ctl.ring_empty[q % kRingTiles]);  // the TMA has read the tile: its slot is free
                    tc_fence_after();
                    const uint64_t a_desc = desc_sw128(smem_u32(stage_a + st * kTileBytes));
                    for (uint32_t h = 0; h < a.halves; ++h) {
                        const uint32_t b = bseq % L.b_slots;
                        if (!pf_wait(&ctl.b_full[b], (bseq / L.b_slots) & 1u, wait_limit, ctl, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t b_desc = desc_sw128(smem_u32(ring_b + b * L.b_stage));
                        const uint32_t d_tmem = tmem + h * a.n_mma;
                        // the K = 16 steps start 32 bytes apart: 2 in the
                        // descriptors' start-address field
                        tc_mma(d_tmem, a_desc, b_desc, idesc, g != 0);
                        tc_mma(d_tmem, a_desc + 2, b_desc + 2, idesc, true);
                        tc_mma(d_tmem, a_desc + 4, b_desc + 4, idesc, true);
                        tc_mma(d_tmem, a_desc + 6, b_desc + 6, idesc, true);
                        tc_commit(&ctl.b_empty[b]);
                        ++bseq;
                    }
                    if (ok) tc_commit(&ctl.a_empty[st]);
                }
                if (ok) {
                    tc_commit(&ctl.acc_full);
                    ++n_item;
                }
            }
            if (!ok) {  // the products in flight finish before the tensor memory is freed
                tc_commit(&ctl.drain_mma);
                if (!mbar_wait(&ctl.drain_mma, 0, wait_limit)) raise_status(status, AFX_DEV_UNDRAINED);
            }
        }
        __syncwarp();
    } else {
        // ---- accumulator -> Y
        const uint32_t quarter = static_cast<uint32_t>(warp) & 3u;
        uint32_t n_item = 0;
        for (uint32_t it = it0; it < it1; ++it) {
            const ItemInfo ii = item_info(a.items[it]);
            const PrefillMatrix& pm = a.m[ii.mi];
            if (!__all_sync(0xFFFFFFFFu, pf_wait(&ctl.acc_full, n_item & 1u, wait_limit, ctl, status))) break;
            tc_fence_after();
            const uint32_t y0 = ii.pass * a.pass_tokens;
            const uint32_t valid = min(a.pass_tokens, a.n_tokens - y0);
            const uint64_t rows = pm.t.rows;
            float* y = pm.t.y + static_cast<uint64_t>(y0) * rows + static_cast<uint64_t>(ii.mt) * kTileRows + quarter * 32 + lane;
            for (uint32_t c0 = 0; c0 < valid; c0 += 16) {
                uint32_t v[16];
                tc_ld16(tmem + ((quarter * 32u) << 16) + c0, v);
                if (ii.part == 0) {
#pragma unroll
                    for (uint32_t j = 0; j < 16; ++j)
                        if (c0 + j < valid) y[static_cast<uint64_t>(c0 + j) * rows] = __uint_as_float(v[j]);
                } else {  // one of two halves of the sum: added into the zeroed Y
#pragma unroll
                    for (uint32_t j = 0; j < 16; ++j)
                        if (c0 + j < valid) atomicAdd(y + static_cast<uint64_t>(c0 + j) * rows, __uint_as_float(v[j]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.acc_empty);
            ++n_item;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kPfMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
    }
}

}  // namespace afx


// ---- host side --------------------------------------------------------------------------

namespace afx {

// Defined with the restore kernels (afx_decode.cu).
void fill_tensor(const afx_desc& d, const void* container, TensorArgs& t);
afx_status prepare_kernel(const void* func, int threads, size_t smem, int* blocks_per_sm);
int sm_count();

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's cuTensorMapEncodeTiled, found through the runtime (the
// library does not link the driver library itself).
EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// A row-major BF16 matrix [rows][cols] in device memory, read as boxes of
// 64 columns x box_rows rows with the 128-byte swizzle the MMA descriptors
// name; rows past the end read as zeros.  X [n_tokens][cols] (box: the
// tokens of one accumulator) and the rings [CTAs * 16 * 128][64] (box: a
// tile).
afx_status make_map(CUtensorMap* map, const uint16_t* x, uint32_t cols, uint64_t rows, uint32_t box_rows) {
    const EncodeTiledFn enc = encode_tiled();
    if (!enc) return afx_fail(AFX_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver", 0);
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {kTileCols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[96];
        snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
        return afx_fail(AFX_E_CUDA, msg, 0);
    }
    return AFX_OK;
}

bool device_memory(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice;
}

uint32_t pow2_at_least(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

// Tokens per MMA and accumulators per pass for n_tokens: one pass of up to
// 512 tokens in up to four accumulators of at most 128 tokens each, N a
// multiple of 16; more tokens take passes of 512.
void token_split(uint32_t n_tokens, uint32_t* n_mma, uint32_t* halves) {
    if (n_tokens <= kMaxPassTokens) {
        *halves = (n_tokens + kMaxHalfTokens - 1) / kMaxHalfTokens;
        *n_mma = round_up((n_tokens + *halves - 1) / *halves, 16);
    } else {
        *halves = kMaxHalves;
        *n_mma = kMaxHalfTokens;
    }
}

// One launch over items[0 .. n) (codes matrix << 28 | pass << 18 | m-tile):
// each item to the least loaded CTA, largest first (an item costs its
// k-tiles); each CTA takes its items in code order, so that consecutive
// items share a matrix's decode tables.
afx_status launch_items(PrefillArgs& pa, const std::vector<uint32_t>& codes, size_t begin, size_t end, size_t smem,
                        uint32_t max_ctas, cudaStream_t s) {
    const size_t n = end - begin;
    const uint32_t G = static_cast<uint32_t>(std::min<size_t>(n, max_ctas));
    std::vector<uint32_t> order(n);
    for (size_t i = 0; i < n; ++i) order[i] = codes[begin + i];
    auto tiles_of = [&](uint32_t code) {
        const ItemInfo ii = item_info(code);
        uint32_t kb, ke;
        item_tiles(ii.part, pa.m[ii.mi].k_tiles, &kb, &ke);
        return ke - kb;
    };
    std::stable_sort(order.begin(), order.end(), [&](uint32_t x, uint32_t y) { return tiles_of(x) > tiles_of(y); });
    using Load = std::pair<uint64_t, uint32_t>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (uint32_t c = 0; c < G; ++c) heap.push({0, c});
    std::vector<std::vector<uint32_t>> per(G);
    for (uint32_t code : order) {
        Load l = heap.top();
        heap.pop();
        per[l.second].push_back(code);
        l.first += tiles_of(code);
        heap.push(l);
    }
    uint32_t k = 0;
    for (uint32_t c = 0; c < G; ++c) {
        std::sort(per[c].begin(), per[c].end());
        pa.cta_begin[c] = static_cast<uint16_t>(k);
        for (uint32_t code : per[c]) pa.items[k++] = code;
    }
    pa.cta_begin[G] = static_cast<uint16_t>(k);
    prefill_fused_kernel<<<G, kPfThreads, smem, s>>>(pa);
    AFX_CUDA_TRY(cudaGetLastError(), "prefill_fused_kernel launch");
    return AFX_OK;
}

}  // namespace

}  // namespace afx

using namespace afx;

extern "C" afx_status afx_tile_order(const uint16_t* w, uint32_t rows, uint32_t cols, uint16_t* out) {
    if (!w || !out) return afx_fail(AFX_E_ARG, "null pointer", 0);
    if (rows == 0 || cols == 0 || rows % kTileRows || cols % kTileCols)
        return afx_fail(AFX_E_ARG, "rows must be a multiple of 128 and cols a multiple of 64", 0);
    const uint64_t kt = cols / kTileCols;
    for (uint64_t m = 0; m < rows / kTileRows; ++m)
        for (uint64_t g = 0; g < kt; ++g) {
            uint16_t* dst = out + (m * kt + g) * kTileElems;
            const uint16_t* src = w + m * kTileRows * cols + g * kTileCols;
            for (uint64_t r = 0; r < kTileRows; ++r)
                std::memcpy(dst + r * kTileCols, src + r * cols, kTileCols * sizeof(uint16_t));
        }
    return AFX_OK;
}

extern "C" afx_status afx_prefill_fused_workspace(uint64_t* bytes) {
    if (!bytes) return afx_fail(AFX_E_ARG, "null pointer", 0);
    const int sms = sm_count();
    if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
    *bytes = static_cast<uint64_t>(std::min(sms, kPfMaxCtas)) * kRingTiles * kTileBytes;
    return AFX_OK;
}

extern "C" afx_status afx_prefill_fused_batch(const afx_desc* descs, const void* const* containers,
                                              const uint32_t* rows, const uint32_t* cols, const uint16_t* const* xs,
                                              uint32_t n_tokens, float* const* ys, uint32_t count,
                                              void* workspace, uint64_t workspace_bytes, afx_stream_t stream,
                                              int32_t* status) {
    if (count == 0) return AFX_OK;
    if (!descs || !containers || !rows || !cols || !xs || !ys) return afx_fail(AFX_E_ARG, "null array", 0);
    if (n_tokens == 0) return afx_fail(AFX_E_ARG, "n_tokens must be at least 1", 0);
    // the CTAs' rings: as many CTAs as the workspace holds rings, at most one per SM
    const int sms = sm_count();
    if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
    const uint64_t ring_bytes = static_cast<uint64_t>(kRingTiles) * kTileBytes;
    const uint32_t max_ctas = static_cast<uint32_t>(
        std::min<uint64_t>({workspace ? workspace_bytes / ring_bytes : 0, static_cast<uint64_t>(sms),
                            static_cast<uint64_t>(kPfMaxCtas)}));
    if (max_ctas == 0) return afx_fail(AFX_E_NOSPACE, "the workspace must hold at least one ring (256 KB)", 0);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return afx_fail(AFX_E_ARG, "the workspace must be 256-byte aligned", 0);
    if (!device_memory(workspace)) return afx_fail(AFX_E_ARG, "the workspace must be in device memory", 0);
    uint32_t n_mma = 0, halves = 0;
    token_split(n_tokens, &n_mma, &halves);
    const uint32_t pass_tokens = n_mma * halves;
    const uint32_t passes = (n_tokens + pass_tokens - 1) / pass_tokens;
    if (passes > 512) return afx_fail(AFX_E_ARG, "n_tokens must be at most 262144", 0);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = -1, optin = 0;
    AFX_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    AFX_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev), "cudaDeviceGetAttribute");
    std::unique_ptr<PrefillArgs> pa(new PrefillArgs);
    for (uint32_t i0 = 0; i0 < count; i0 += kMaxTensors) {
        const uint32_t cnt = std::min<uint32_t>(count - i0, kMaxTensors);
        std::memset(static_cast<void*>(pa.get()), 0, offsetof(PrefillArgs, cta_begin));
        pa->count = cnt;
        pa->n_tokens = n_tokens;
        pa->n_mma = n_mma;
        pa->halves = halves;
        pa->pass_tokens = pass_tokens;
        pa->tmem_cols = pow2_at_least(pass_tokens);
        pa->status = status;
        pa->ring = static_cast<uint16_t*>(workspace);
        const afx_status rst =
            make_map(&pa->ring_map, static_cast<const uint16_t*>(workspace), kTileCols,
                     static_cast<uint64_t>(max_ctas) * kRingTiles * kTileRows, kTileRows);
        if (rst != AFX_OK) return rst;
        uint32_t max_T = 4;
        std::vector<uint32_t> codes;
        for (uint32_t k = 0; k < cnt; ++k) {
            const uint32_t i = i0 + k;
            const afx_desc& d = descs[i];
            if (afx_check_desc(&d) != AFX_OK) return afx_fail(AFX_E_FORMAT, "invalid container description", 0);
            if (d.format != AFX_FMT_BF16) return afx_fail(AFX_E_ARG, "the fused prefill product takes BF16 containers", 0);
            if (rows[i] == 0 || cols[i] == 0 || rows[i] % kTileRows || cols[i] % kTileCols)
                return afx_fail(AFX_E_ARG, "rows must be a multiple of 128 and cols a multiple of 64", 0);
            if (static_cast<uint64_t>(rows[i]) * cols[i] != d.n) return afx_fail(AFX_E_ARG, "rows * cols != n", 0);
            if (rows[i] / kTileRows > (1u << 17)) return afx_fail(AFX_E_ARG, "too many rows", 0);
            if (d.nsym >= 2 && d.block_chunks != static_cast<uint32_t>(kThreads))
                return afx_fail(AFX_E_FORMAT, "the decoder needs 512 chunks per block", 0);
            if (!containers[i] || !ys[i] || !xs[i]) return afx_fail(AFX_E_ARG, "null pointer", 0);
            if (reinterpret_cast<uintptr_t>(containers[i]) & 255u || reinterpret_cast<uintptr_t>(xs[i]) & 15u)
                return afx_fail(AFX_E_ARG, "containers must be 256-byte and x 16-byte aligned", 0);
            if (!device_memory(containers[i]) || !device_memory(xs[i]) || !device_memory(ys[i]))
                return afx_fail(AFX_E_ARG, "containers, x and y must be in device memory", 0);
            PrefillMatrix& pm = pa->m[k];
            fill_tensor(d, containers[i], pm.t);
            pm.t.y = ys[i];
            pm.t.rows = rows[i];
            pm.t.cols = cols[i];
            pm.k_tiles = cols[i] / kTileCols;
            pm.single = d.nsym == 1 ? 1u : 0u;
            pm.fill = d.fill;
            max_T = std::max(max_T, d.chunk_bytes);
            const afx_status mst = make_map(&pa->tmap[k], xs[i], cols[i], n_tokens, n_mma);
            if (mst != AFX_OK) return mst;
        }
        // items: every m-tile for every pass; an m-tile larger than half a
        // CTA's share of all the tiles is split in two along K, and its
        // matrix's Y is zeroed first (the two halves are added into it)
        const int sms_now = sm_count();
        uint64_t all_tiles = 0;
        for (uint32_t k = 0; k < cnt; ++k)
            all_tiles += static_cast<uint64_t>(pa->m[k].t.rows / kTileRows) * pa->m[k].k_tiles * passes;
        const uint64_t share = all_tiles / std::max<uint64_t>(1, std::min<uint64_t>(max_ctas, sms_now > 0 ? sms_now : 1));
        for (uint32_t k = 0; k < cnt; ++k) {
            const PrefillMatrix& pm = pa->m[k];
            const bool split = pm.k_tiles >= 2 && 2ull * pm.k_tiles > share;
            if (split)
                AFX_CUDA_TRY(cudaMemsetAsync(pm.t.y, 0, static_cast<size_t>(n_tokens) * pm.t.rows * sizeof(float), s),
                             "cudaMemsetAsync");
            for (uint32_t p = 0; p < passes; ++p)
                for (uint32_t mt = 0; mt < pm.t.rows / kTileRows; ++mt) {
                    if (split) {
                        codes.push_back(item_code(k, p, 1, mt));
                        codes.push_back(item_code(k, p, 2, mt));
                    } else {
                        codes.push_back(item_code(k, p, 0, mt));
                    }
                }
        }
        pa->max_chunk_bytes = max_T;
        // decode tables: the state table where all of it fits beside the
        // rings and the warps' buffers, else the 12-bit table
        const PfLayout L0 = pf_layout(0, n_mma, max_T);
        const int64_t budget = static_cast<int64_t>(optin) - 1024 - static_cast<int64_t>(L0.total) - 16;
        if (budget < static_cast<int64_t>(kLutTabBytes)) return afx_fail(AFX_E_ARG, "launch needs too much shared memory", 0);
        uint32_t tab_bytes = kLutTabBytes;
        for (uint32_t k = 0; k < cnt; ++k) {
            CodeTables& tab = pa->m[k].t.tab;
            if (!tab.fsm) continue;
            const int64_t need = static_cast<int64_t>(tab.n_states + kSkipRows) * kFsmRowBytes;
            if (tab.n_states > static_cast<uint32_t>(kMaxStates) || need > budget) {
                tab.fsm = 0;
            } else {
                tab.fsm_rows = tab.n_states;
                tab_bytes = std::max<uint32_t>(tab_bytes, static_cast<uint32_t>(need));
            }
        }
        pa->tab_bytes = tab_bytes;
        const size_t smem = pf_layout(tab_bytes, n_mma, max_T).total + 1024;
        int per_sm = 0;
        const afx_status pst = prepare_kernel(reinterpret_cast<const void*>(prefill_fused_kernel), kPfThreads, smem, &per_sm);
        if (pst != AFX_OK) return pst;
        for (size_t b = 0; b < codes.size(); b += kPfMaxItems) {
            const afx_status lst = launch_items(*pa, codes, b, std::min(codes.size(), b + kPfMaxItems), smem, max_ctas, s);
            if (lst != AFX_OK) return lst;
        }
    }
    return AFX_OK;
}

extern "C" afx_status afx_prefill_fused(const afx_desc* desc, const void* container, uint32_t rows, uint32_t cols,
                                        const uint16_t* x, uint32_t n_tokens, float* y, void* workspace,
                                        uint64_t workspace_bytes, afx_stream_t stream, int32_t* status) {
    if (!desc) return afx_fail(AFX_E_ARG, "null description", 0);
    return afx_prefill_fused_batch(desc, &container, &rows, &cols, &x, n_tokens, &y, 1, workspace, workspace_bytes,
                                   stream, status);
}

// Bits of the bounds checks that fired in this module (bounds-checked
// builds), read and cleared; afx_debug_bounds_report adds them to its own.
extern "C" __attribute__((visibility("hidden"))) uint32_t afx_prefill_bounds_bits(void) {
    unsigned int bits = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&bits, g_bounds_report, sizeof bits) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaMemcpyToSymbol(g_bounds_report, &zero, sizeof zero);
    return bits;
}
