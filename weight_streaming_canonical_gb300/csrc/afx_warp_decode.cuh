// Device-side pieces of the afx restore shared by the kernels of
// afx_decode.cu (restore, fused GEMV) and afx_prefill_fused.cu (fused
// restore + tensor-core product): the launch structures, the decode tables,
// the staging copies and the warp decoder of one 32-chunk sub-tile.
//
// The operation: "Why Weight Offloading Slows Inference", section
// "Lossless compression: fewer bytes to read, more work to unpack" -- every
// weight's exponent was stored with a shorter code for common values, its
// sign and mantissa raw; the released bits are restored before compute.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "afx_internal.h"

namespace afx {

#define AFX_CUDA_TRY(call, what)                                            \
    do {                                                                    \
        const cudaError_t e_ = (call);                                      \
        if (e_ != cudaSuccess) return afx_fail(AFX_E_CUDA, (what), e_);     \
    } while (0)

constexpr int kThreads = AFX_DECODE_THREADS;
constexpr int kWarps = kThreads / 32;
constexpr int kLutBits = 12;
constexpr int kLutSize = 1 << kLutBits;
constexpr int kStageBytes = AFX_BLOCK_CAPACITY + 16;
constexpr int kMaxBatch = 4;       // GEMV activation rows
constexpr int kMaxTensors = 16;    // tensors per launch
constexpr int kStreamPad = 32;     // stream bytes staged past a tile's own chunks
constexpr int kChunkStage = kThreads + 8;  // chunk entries staged per tile (the next tile's first included)

// Canonical decode tables, built on the host from the 256 code lengths.
// In 24-bit left-aligned code space all codes of length <= L lie in
// [0, limit[L]); a 24-bit peek v has the length L = the smallest L with
// v < limit[L], and its symbol's stage byte is sorted[base[L] + (v >> (24 - L))].
// Stage bytes are what the merge of the tensor's element format wants: the
// exponent rotated right by one bit for BF16 (see ror8), and the exponent at
// its place in the element's high byte for FP16 (<< 2) and E4M3 (<< 3).
//
// The internal nodes of the code tree (the prefixes that are not codes yet)
// are numbered for the byte-step decoder: depth by depth, prefix value
// ascending, the root first.  A prefix of depth d is internal when it lies
// at or past limit[d] in d-bit space, so depth d holds the prefixes
// [limit[d] >> (24 - d), 2^d) and node (d, p) is number
// state_base[d] + p - (limit[d] >> (24 - d)).  A complete code of nsym
// symbols has nsym - 1 of them.
constexpr int kMaxStates = 56;
struct CodeTables {
    uint32_t limit[AFX_MAX_CODE_LEN + 1];
    int32_t base[AFX_MAX_CODE_LEN + 1];
    uint32_t state_base[AFX_MAX_CODE_LEN + 1];
    uint8_t sorted[256];
    uint8_t state_depth[kMaxStates];
    uint32_t n_states;  // internal nodes (nsym - 1)
    uint32_t fsm;       // 1: the restore path decodes this tensor a byte at a time
    uint32_t fsm_rows;  // nodes held as state-table rows: the first fsm_rows (all, or the shallowest)
};

// One tensor of a launch.
struct TensorArgs {
    const uint32_t* exp_words;
    const uint8_t* sm;
    const uint8_t* hi;         // FP16: the 3 leading fraction bits, a nibble per element (nullptr otherwise)
    const uint16_t* chunk_index;
    const uint64_t* block_index;
    uint64_t n, n_chunks, n_blocks, exp_bytes;
    uint64_t total_bits;       // coded bits in the stream
    uint64_t n_sub_full;       // leading sub-tiles whose chunks, next entry and stream pad all exist
    uint64_t tile_begin;       // first tile of this tensor in the launch's tile list
    uint64_t sub_begin;        // warp GEMV: first sub-tile of this tensor in the launch's sub-tile list
    uint32_t chunk_bytes;      // T
    uint32_t rows_per_warp;    // GEMV: capacity of the per-warp partial table
    uint32_t pair_codes;       // host: codes a 64-chunk sub-tile holds, 5 standard deviations above the mean
    void* out;                 // restore: n elements (uint16 BF16 / FP16, uint8 E4M3)
    const uint16_t* x;         // GEMV: [B][cols]
    float* y;                  // GEMV: [B][rows]
    float* ws;                 // GEMV: [n_blocks][2][B]
    uint32_t rows, cols;
    CodeTables tab;
};

struct LaunchArgs {
    uint32_t count;
    uint32_t max_chunk_bytes;
    uint32_t max_rows_per_warp;
    uint32_t tab_bytes;        // restore path: size of the shared decode-table region
    uint64_t total_tiles;
    uint64_t total_subs;       // warp GEMV: sub-tiles of all tensors
    uint32_t wait_limit;       // polls of a staging wait before it gives up (0: kWaitLimit)
    uint32_t stall;            // failure injection for tests: arm the staging barriers, issue no copies
    uint32_t host_src;         // restore: the containers are in pinned host memory (restore_store_host_kernel)
    uint32_t kind;             // restore: element kind, kKindBF16 / kKindFP16 / kKindE4M3
    uint32_t partial;          // BF16 tensors whose state tables keep only their shallowest nodes
    uint32_t pair_stage;       // restore: 0, or two chunks a lane with a stage of this many bytes a warp
    int32_t* status;
    TensorArgs t[kMaxTensors];
};

struct Shared {
    uint32_t lut[kLutSize];   // up to 3 codes per 12-bit peek: bits 0-3 total length, 4-5 count, 8-31 rotated exponents
    uint8_t len0[kLutSize];   // length of the first code of a 12-bit peek (0: longer than 12 bits)
    uint32_t limit[AFX_MAX_CODE_LEN + 1];
    int32_t base[AFX_MAX_CODE_LEN + 1];
    uint8_t sorted[256];
    alignas(16) uint16_t chunk[2][kChunkStage];  // cp.async destinations: 16-byte aligned rows
    alignas(16) uint64_t block_pair[2][2];
    uint32_t warp_total[kWarps];
    int32_t tile_ok;
    alignas(16) uint8_t stage[kStageBytes];  // rotated exponent of weight (o0 & ~7) + i at stage[i]
    // dynamic part: stream[2][kThreads * max_T + kStreamPad], then GEMV partials
};

constexpr size_t shared_fixed_bytes() { return (sizeof(Shared) + 15) & ~size_t(15); }
static_assert(offsetof(Shared, chunk) % 16 == 0 && (kChunkStage * 2) % 16 == 0, "cp.async rows must be 16-byte aligned");
static_assert(offsetof(Shared, stage) % 16 == 0, "stage must be 16-byte aligned");

// ---- small device helpers ------------------------------------------------------

__device__ __forceinline__ void raise_status(int32_t* status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// Bounds-checked builds.  Compute-sanitizer is not available, so a build
// with AFX_DEBUG_BOUNDS=1 checks, on the restore path, every range a kernel
// is about to read or write against its buffer (stage, stream buffer,
// decode tables, output); a failed check ORs its bit into g_bounds_report,
// which afx_debug_bounds_report reads.  In regular builds the checks
// compile to nothing.
#ifndef AFX_DEBUG_BOUNDS
#define AFX_DEBUG_BOUNDS 0
#endif
static __device__ unsigned int g_bounds_report;  // one per translation unit (module)
enum BoundsCheck : unsigned {
    kChkTableState = 0,   // a byte step's state offset inside the state table
    kChkStageSteps,       // the byte steps' stage words inside the warp's stage
    kChkStreamWords,      // a chunk's words inside the stream buffer
    kChkStagePending,     // pending bytes inside the stage
    kChkStageRun,         // a 12-bit-table or partial-chunk run inside the stage
    kChkMergeStage,       // the merged range inside the stage
    kChkMergeOutput,      // the merged range inside the output
    kChkStagingBytes,     // staged bytes inside the stream buffer and chunk rows
    kChkTableBuild,       // a built entry's next state inside the table
};
#define AFX_CHECK(cond, bit)                                                      \
    do {                                                                          \
        if (AFX_DEBUG_BOUNDS && !(cond)) atomicOr(&g_bounds_report, 1u << (bit)); \
    } while (0)

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// One request that pulls [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// mbarrier-tracked bulk copies (the TMA engine's non-tensor form): one
// thread arms the barrier with the bytes to expect and issues the copies;
// every waiting thread polls the barrier's phase.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// [src, src + bytes) to shared dst, completing on bar; both addresses and
// bytes multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of bar with the given parity to complete, giving up
// after kWaitLimit polls (a copy of a few hundred bytes takes microseconds;
// the limit is far beyond that).  Returns false on timeout.
constexpr uint32_t kWaitLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Orders this thread's earlier shared-memory reads before later writes of
// the async proxy (a bulk copy refilling the same buffer).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Exponents are kept rotated right by one bit, R = (e >> 1) | (e << 7), in
// the decode tables and the stage buffer.  A BF16 weight's high byte is
// sign | e >> 1 = (R & 0x7F) | (s & 0x80) and its low byte is
// e << 7 | mantissa = (R & 0x80) | (s & 0x7F), with s the sign|mantissa
// byte; so four weights take two bit selects and two byte interleaves.
__host__ __device__ __forceinline__ uint32_t ror8(uint32_t e) { return ((e >> 1) | (e << 7)) & 0xFFu; }

__device__ __forceinline__ uint2 join4(uint32_t r4, uint32_t s4) {
    const uint32_t hi = (r4 & 0x7F7F7F7Fu) | (s4 & 0x80808080u);
    const uint32_t lo = (s4 & 0x7F7F7F7Fu) | (r4 & 0x80808080u);
    return make_uint2(__byte_perm(lo, hi, 0x5140), __byte_perm(lo, hi, 0x7362));
}

__device__ __forceinline__ uint4 join8(uint2 r8, uint2 s8) {
    const uint2 a = join4(r8.x, s8.x), b = join4(r8.y, s8.y);
    return make_uint4(a.x, a.y, b.x, b.y);
}

// One weight from a rotated exponent r and its sign|mantissa byte s.
__device__ __forceinline__ uint16_t join1(uint32_t r, uint32_t s) {
    return static_cast<uint16_t>((((r & 0x7Fu) | (s & 0x80u)) << 8) | (s & 0x7Fu) | (r & 0x80u));
}

// E4M3 elements: byte = sign << 7 | e << 3 | mantissa, from the stage byte
// e << 3 and the raw nibble sign << 3 | mantissa.  Four at a time: s4 holds
// four stage bytes, n4 four nibbles (one per byte).
__device__ __forceinline__ uint32_t e4m3_join4(uint32_t s4, uint32_t n4) {
    return ((n4 & 0x08080808u) << 4) | s4 | (n4 & 0x07070707u);
}

// Sixteen E4M3 elements from their 16 stage bytes (two uint2) and their 8
// raw bytes (element 2k in the low nibble of byte k).
__device__ __forceinline__ uint4 e4m3_join16(uint2 ra, uint2 rb, uint2 raw) {
    const uint32_t lo0 = raw.x & 0x0F0F0F0Fu, hi0 = (raw.x >> 4) & 0x0F0F0F0Fu;
    const uint32_t lo1 = raw.y & 0x0F0F0F0Fu, hi1 = (raw.y >> 4) & 0x0F0F0F0Fu;
    return make_uint4(e4m3_join4(ra.x, __byte_perm(lo0, hi0, 0x5140)), e4m3_join4(ra.y, __byte_perm(lo0, hi0, 0x7362)),
                      e4m3_join4(rb.x, __byte_perm(lo1, hi1, 0x5140)), e4m3_join4(rb.y, __byte_perm(lo1, hi1, 0x7362)));
}

// FP16 elements: high byte = sign << 7 | e << 2 | h >> 1, low byte = (h & 1)
// << 7 | the 7 trailing fraction bits, from the stage byte e << 2, the raw
// byte (sign << 7 | trailing bits) and h, the 3 leading fraction bits.  Four
// at a time: s4, r4 and f4 hold one value per byte.
__device__ __forceinline__ uint2 fp16_join4(uint32_t s4, uint32_t r4, uint32_t f4) {
    const uint32_t hi = (r4 & 0x80808080u) | s4 | ((f4 >> 1) & 0x03030303u);
    const uint32_t lo = ((f4 << 7) & 0x80808080u) | (r4 & 0x7F7F7F7Fu);
    return make_uint2(__byte_perm(lo, hi, 0x5140), __byte_perm(lo, hi, 0x7362));
}

// Eight FP16 elements from their stage bytes, raw bytes and the hi-section
// word of their group (element j in nibble j, lowest first): the nibbles
// are spread one per byte with two byte permutes, as for E4M3's raw
// nibbles; fp16_join4 reads bits 0..2 of each (bit 3 is zero).
__device__ __forceinline__ uint4 fp16_join8(uint2 s8, uint2 r8, uint32_t h32) {
    const uint32_t even = h32 & 0x0F0F0F0Fu, odd = (h32 >> 4) & 0x0F0F0F0Fu;
    const uint2 a = fp16_join4(s8.x, r8.x, __byte_perm(even, odd, 0x5140));
    const uint2 b = fp16_join4(s8.y, r8.y, __byte_perm(even, odd, 0x7362));
    return make_uint4(a.x, a.y, b.x, b.y);
}

// The 3 leading fraction bits of FP16 element o: its hi-section nibble.
__device__ __forceinline__ uint32_t fp16_hi3(const uint8_t* hi, uint64_t o) {
    return (static_cast<uint32_t>(hi[o >> 1]) >> (4u * static_cast<uint32_t>(o & 1u))) & 0x7u;
}

__device__ __forceinline__ uint16_t fp16_join1(uint32_t s, uint32_t r, uint32_t h) {
    const uint2 v = fp16_join4(s & 0xFFu, r & 0xFFu, h & 0x7u);
    return static_cast<uint16_t>(v.x & 0xFFFFu);
}

__device__ __forceinline__ uint8_t e4m3_join1(uint32_t r, uint32_t nib) {
    return static_cast<uint8_t>(e4m3_join4(r & 0xFFu, nib & 0xFu) & 0xFFu);
}

// ---- decode tables ---------------------------------------------------------------
//
// Rebuilt whenever a CTA moves to another tensor.  Step 1 gives every 12-bit
// peek its first code (exponent, length) using the canonical limits; a
// thread's 16 consecutive peeks have non-decreasing lengths, so one search
// plus short advances suffices.  The (length << 8 | exponent) pairs go to a
// scratch table (free shared memory between tiles).  Step 2 chains up
// to three first codes per peek: after the first code of length L1, the
// remaining 12 - L1 peek bits start the second code, which counts only if
// it ends within the 12 bits, and likewise for the third.

template <class S>
__device__ __forceinline__ void build_tables(S& sh, uint16_t* first /* 8 KB scratch */, const CodeTables& tab) {
    const int tid = threadIdx.x;
    for (int i = tid; i <= AFX_MAX_CODE_LEN; i += kThreads) {
        sh.limit[i] = tab.limit[i];
        sh.base[i] = tab.base[i];
    }
    for (int i = tid; i < 256; i += kThreads) sh.sorted[i] = tab.sorted[i];
    constexpr int kPer = kLutSize / kThreads;
    {
        const int p0 = tid * kPer;
        int L = 1;
        while (L <= kLutBits && (static_cast<uint32_t>(p0) << (24 - kLutBits)) >= tab.limit[L]) ++L;
        for (int j = 0; j < kPer; ++j) {
            const uint32_t p = static_cast<uint32_t>(p0 + j);
            const uint32_t v = p << (24 - kLutBits);
            while (L <= kLutBits && v >= tab.limit[L]) ++L;
            uint16_t e = 0;
            if (L <= kLutBits)
                e = static_cast<uint16_t>((L << 8) | tab.sorted[tab.base[L] + static_cast<int32_t>(v >> (24 - L))]);
            first[p] = e;
            sh.len0[p] = static_cast<uint8_t>(e >> 8);
        }
    }
    __syncthreads();
    for (int j = 0; j < kPer; ++j) {
        const uint32_t p = static_cast<uint32_t>(tid * kPer + j);
        const uint32_t f1 = first[p];
        const uint32_t l1 = f1 >> 8;
        uint32_t entry = 0;
        if (l1) {
            uint32_t bits = l1, count = 1, syms = f1 & 0xFFu;
            const uint32_t f2 = first[(p << l1) & (kLutSize - 1)];
            const uint32_t l2 = f2 >> 8;
            if (l2 && bits + l2 <= kLutBits) {
                bits += l2;
                syms |= (f2 & 0xFFu) << 8;
                count = 2;
                const uint32_t f3 = first[(p << bits) & (kLutSize - 1)];
                const uint32_t l3 = f3 >> 8;
                if (l3 && bits + l3 <= kLutBits) {
                    bits += l3;
                    syms |= (f3 & 0xFFu) << 16;
                    count = 3;
                }
            }
            entry = bits | (count << 4) | (syms << 8);
        }
        sh.lut[p] = entry;
    }
    __syncthreads();
}

// One code from a 32-bit window: its stage byte, length in len (0 on a bad code).
template <class S>
__device__ __forceinline__ uint32_t decode_one(const S& sh, uint32_t win, uint32_t& len) {
    const uint32_t p = win >> (32 - kLutBits);
    uint32_t L = sh.len0[p];
    if (L) {
        len = L;
        return (sh.lut[p] >> 8) & 0xFFu;
    }
    const uint32_t v = win >> 8;
    L = kLutBits + 1;
    while (L <= AFX_MAX_CODE_LEN && v >= sh.limit[L]) ++L;
    if (L > AFX_MAX_CODE_LEN) {
        len = 0;
        return 0;
    }
    len = L;
    return sh.sorted[sh.base[L] + static_cast<int32_t>(v >> (24 - L))];
}

// ---- tile staging ----------------------------------------------------------------

__device__ __forceinline__ uint32_t stream_stage_bytes(const TensorArgs& t, uint64_t b) {
    const uint64_t byte0 = b * static_cast<uint64_t>(kThreads) * t.chunk_bytes;
    const uint64_t want = static_cast<uint64_t>(kThreads) * t.chunk_bytes + kStreamPad;
    const uint64_t avail = t.exp_bytes > byte0 ? t.exp_bytes - byte0 : 0;
    return static_cast<uint32_t>(want < avail ? want : avail);
}

// Issues the cp.async copies of tile b of tensor t into buffer slot `buf`
// and commits them as one group (every thread commits, possibly empty).
__device__ __forceinline__ void issue_tile(Shared& sh, uint8_t* stream_base, uint32_t stream_stride, const TensorArgs& t, uint64_t b,
                           int buf) {
    const int tid = threadIdx.x;
    uint8_t* dst = stream_base + static_cast<size_t>(buf) * stream_stride;
    const uint8_t* src =
        reinterpret_cast<const uint8_t*>(t.exp_words) + b * static_cast<uint64_t>(kThreads) * t.chunk_bytes;
    const uint32_t bytes = stream_stage_bytes(t, b);
    for (uint32_t i = tid * 16u; i < bytes; i += kThreads * 16u) cp_async16(dst + i, src + i);
    // chunk entries of this tile and the next tile's first eight, inside the
    // chunk section and its zero padding (rounded up to 16 bytes)
    const uint64_t cb0 = b * static_cast<uint64_t>(kThreads) * 2;
    const uint64_t csec = (t.n_chunks * 2 + 15) & ~uint64_t(15);
    const uint64_t cavail = csec > cb0 ? csec - cb0 : 0;
    const uint32_t cbytes = static_cast<uint32_t>(cavail < kChunkStage * 2 ? cavail : kChunkStage * 2);
    const uint8_t* csrc = reinterpret_cast<const uint8_t*>(t.chunk_index) + cb0;
    uint8_t* cdst = reinterpret_cast<uint8_t*>(sh.chunk[buf]);
    for (uint32_t i = tid * 16u; i < cbytes; i += kThreads * 16u) cp_async16(cdst + i, csrc + i);
    if (tid == 0) {
        cp_async8(&sh.block_pair[buf][0], t.block_index + b);
        cp_async8(&sh.block_pair[buf][1], t.block_index + b + 1);
    }
    cp_async_commit();
}

// Exclusive block-wide scan of one count per thread: warp-shuffle scans of
// the counts and then of the warp totals.
__device__ __forceinline__ uint32_t block_exclusive_scan(Shared& sh, uint32_t v, uint32_t* total) {
    static_assert(kWarps <= 32, "one warp scans the warp totals");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) sh.warp_total[warp] = inc;
    __syncthreads();
    uint32_t wt = lane < kWarps ? sh.warp_total[lane] : 0u;
#pragma unroll
    for (int d = 1; d < kWarps; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, wt, d);
        if (lane >= d) wt += o;
    }
    const uint32_t before = __shfl_sync(0xFFFFFFFFu, wt, (warp + 31) & 31);
    *total = __shfl_sync(0xFFFFFFFFu, wt, kWarps - 1);
    return (warp ? before : 0u) + inc - v;
}

// Appends n8 / 8 exponents (low bytes of `bytes`) to the word accumulator
// and stores every completed word.
__device__ __forceinline__ void append(uint32_t bytes, uint32_t n8, uint32_t& acc, uint32_t& fill_bits,
                                       uint32_t*& wout) {
    const uint32_t word = acc | (bytes << fill_bits);
    const uint32_t carry = __funnelshift_l(bytes, 0u, fill_bits);  // bytes >> (32 - fill), 0 when fill is 0
    fill_bits += n8;
    if (fill_bits >= 32) {
        *wout++ = word;
        acc = carry;
        fill_bits -= 32;
    } else {
        acc = word;
    }
}

// Decodes the cnt codes of one chunk into stage[s0 .. s0 + cnt): the chunk
// starts at stream word k0 and its first code at bit `gap` of that word;
// staged_words words are valid.  `next` is the following chunk's index
// entry (0 if none) and chunk_end the bit offset of this chunk's end in the
// staged stream.  Returns true when the stream is not valid.
template <class S>
__device__ __forceinline__ bool decode_run(const S& sh, const uint32_t* stream, uint32_t staged_words, uint32_t k0,
                                           uint32_t gap, uint32_t cnt, uint8_t* stage, uint32_t s0, uint32_t next,
                                           uint32_t chunk_end) {
    bool bad = false;
    {
        uint32_t k = k0;
        uint32_t w0 = stream[k], w1 = stream[k + 1];
        k += 2;
        uint32_t pos = gap;  // bit of w0 where the next code starts (0..31)
        uint32_t i = 0;
        // head: codes until the stage index is word aligned, from one lookup
        // when it holds them all (their exact length from the first-code
        // lengths), else one code at a time
        const uint32_t head = min(cnt, (0u - s0) & 3u);
        if (head) {
            const uint32_t win = __funnelshift_l(w1, w0, pos);
            const uint32_t e = sh.lut[win >> (32 - kLutBits)];
            if (((e >> 4) & 3u) >= head) {
                uint32_t bits = sh.len0[win >> (32 - kLutBits)];
                stage[s0] = static_cast<uint8_t>(e >> 8);
                if (head > 1) {
                    bits += sh.len0[(win << bits) >> (32 - kLutBits)];
                    stage[s0 + 1] = static_cast<uint8_t>(e >> 16);
                }
                if (head > 2) {
                    bits += sh.len0[(win << bits) >> (32 - kLutBits)];
                    stage[s0 + 2] = static_cast<uint8_t>(e >> 24);
                }
                pos += bits;
                i = head;
                if (pos >= 32) {
                    pos -= 32;
                    w0 = w1;
                    w1 = k < staged_words ? stream[k] : 0u;
                    ++k;
                }
            }
        }
        for (; i < head; ++i) {
            uint32_t len;
            const uint32_t sym = decode_one(sh, __funnelshift_l(w1, w0, pos), len);
            if (!len) {
                bad = true;
                break;
            }
            stage[s0 + i] = static_cast<uint8_t>(sym);
            pos += len;
            if (pos >= 32) {
                pos -= 32;
                w0 = w1;
                w1 = k < staged_words ? stream[k] : 0u;
                ++k;
            }
        }
        uint32_t* wout = reinterpret_cast<uint32_t*>(stage + s0 + i);
        uint32_t acc = 0, fill = 0;
        // body: up to three codes per table lookup, never past cnt
        while (!bad && i + 3 <= cnt) {
            const uint32_t win = __funnelshift_l(w1, w0, pos);
            const uint32_t e = sh.lut[win >> (32 - kLutBits)];
            uint32_t n = (e >> 4) & 3u;
            uint32_t bytes;
            if (n) {
                pos += e & 15u;
                bytes = e >> 8;
            } else {  // the first code is longer than 12 bits
                uint32_t len;
                bytes = decode_one(sh, win, len);
                if (!len) {
                    bad = true;
                    break;
                }
                pos += len;
                n = 1;
            }
            append(bytes, n * 8, acc, fill, wout);
            i += n;
            if (pos >= 32) {
                pos -= 32;
                w0 = w1;
                w1 = k < staged_words ? stream[k] : 0u;
                ++k;
            }
        }
        // tail: the last one or two codes, from one lookup when it holds them
        if (!bad && i < cnt) {
            const uint32_t r = cnt - i;  // 1 or 2
            const uint32_t win = __funnelshift_l(w1, w0, pos);
            const uint32_t e = sh.lut[win >> (32 - kLutBits)];
            if (((e >> 4) & 3u) >= r) {
                uint32_t bits = sh.len0[win >> (32 - kLutBits)];
                if (r > 1) bits += sh.len0[(win << bits) >> (32 - kLutBits)];
                append((e >> 8) & (r > 1 ? 0xFFFFu : 0xFFu), 8 * r, acc, fill, wout);
                i = cnt;
                pos += bits;
                if (pos >= 32) {
                    pos -= 32;
                    w0 = w1;
                    w1 = k < staged_words ? stream[k] : 0u;
                    ++k;
                }
            }
        }
        while (!bad && i < cnt) {
            uint32_t len;
            const uint32_t sym = decode_one(sh, __funnelshift_l(w1, w0, pos), len);
            if (!len) {
                bad = true;
                break;
            }
            append(sym, 8, acc, fill, wout);
            ++i;
            pos += len;
            if (pos >= 32) {
                pos -= 32;
                w0 = w1;
                w1 = k < staged_words ? stream[k] : 0u;
                ++k;
            }
        }
        // pending exponents (at most three) go out as bytes
        uint8_t* tail = reinterpret_cast<uint8_t*>(wout);
        for (uint32_t j = 0; j * 8 < fill; ++j) tail[j] = static_cast<uint8_t>(acc >> (8 * j));
        // the codes must end exactly where the next chunk's first code begins
        if (!bad) {
            const uint32_t end_bit = (k - 2) * 32u + pos;  // bit offset inside the staged stream
            if ((next >> 5) != 0)
                bad = end_bit != chunk_end + (next & 31u);
            else
                bad = end_bit > chunk_end + AFX_MAX_CODE_LEN;
        }
    }
    return bad;
}

// Decodes tile b of tensor t (staged in slot buf) into sh.stage.  Returns
// false, uniformly, when the tile must be skipped.
__device__ __forceinline__ bool decode_tile(Shared& sh, const uint32_t* stream, const TensorArgs& t, uint64_t b, int buf,
                            int32_t* status, uint64_t& o0, uint64_t& o1) {
    const int tid = threadIdx.x;
    const uint32_t T = t.chunk_bytes;
    const uint32_t chunk_bits = 8u * T;
    const uint64_t c0 = b * kThreads;
    o0 = sh.block_pair[buf][0];
    o1 = sh.block_pair[buf][1];
    if (tid == 0) {
        sh.tile_ok = 1;
        // the tile's sign|mantissa bytes are needed after the decode
        if (o0 < o1 && o1 <= t.n) {
            const uint64_t a0 = o0 & ~uint64_t(15), a1 = (o1 + 15) & ~uint64_t(15);
            prefetch_l2(t.sm + a0, static_cast<uint32_t>(a1 - a0));
        }
    }

    const uint32_t entry = (c0 + tid < t.n_chunks) ? sh.chunk[buf][tid] : 0u;
    const uint32_t gap = entry & 31u;
    uint32_t cnt = entry >> 5;
    bool bad = false;
    if (gap > 23u || cnt > chunk_bits - gap) {
        bad = true;
        cnt = 0;
    }
    uint32_t total = 0;
    const uint32_t off = block_exclusive_scan(sh, cnt, &total);  // contains a __syncthreads
    const bool last_ok = b + 1 != t.n_blocks || o1 == t.n;       // the block index ends at n
    if (o1 < o0 || o1 - o0 != total || total > AFX_BLOCK_CAPACITY || o1 > t.n || !last_ok) {
        if (tid == 0) raise_status(status, AFX_DEV_BAD_BLOCK);
        return false;
    }

    if (cnt) {
        const uint32_t next = (c0 + tid + 1 < t.n_chunks) ? sh.chunk[buf][tid + 1] : 0u;
        bad = decode_run(sh, stream, stream_stage_bytes(t, b) >> 2, tid * (T >> 2), gap, cnt, sh.stage,
                         static_cast<uint32_t>(o0 & 7u) + off, next, (tid + 1) * chunk_bits);
    }
    if (bad) {
        raise_status(status, AFX_DEV_BAD_CHUNK);
        sh.tile_ok = 0;
    }
    __syncthreads();
    return sh.tile_ok != 0;
}

// ---- warp-independent restore ------------------------------------------------------
//
// The restore (store) path splits every block further into sub-tiles of 32
// chunks, one warp each.  A CTA still owns a contiguous run of blocks and
// one copy of the decode tables, but its warps run on their own: each takes
// a contiguous run of sub-tiles of the current tensor, stages them with
// cp.async one sub-tile ahead, places its lanes' codes with a warp-shuffle
// scan, and carries the output index of the next sub-tile forward as a
// running sum.  The first sub-tile of a run starts at the block index entry
// of its block plus the counts of that block's earlier chunks.  The running
// sum is checked against the block index at every block boundary that a run
// crosses or ends on, so every entry of the block index is verified.  The
// only CTA barriers are those around a rebuild of the tables.
//
// Byte-step decoding.  When no code is 1 bit long, a lane decodes its chunk
// eight stream bits at a time through a state machine whose state is the
// internal node reached by the bits of the code in progress: entry (state,
// byte) holds the rotated
// exponents of the (at most four) codes that end within the byte, their
// count, and the next state.  Every lane steps through all T bytes of its
// chunk from the chunk's first word, so the lanes of a warp run the same
// loop with aligned word loads.  The gap (the tail of the previous chunk's
// last code) is dropped by starting in one of seven skip rows (the first
// 1..7 bits of the byte end an earlier code) and, for gaps of 8 or more, by
// not stepping through the first one or two bytes.  After the last byte the
// state's depth says where the code that crosses the chunk end began; that
// one code is decoded on its own.  The partial last chunk of a stream and
// tensors with 1-bit codes use the 12-bit multi-code table.
//
// A tree with more internal nodes than shared memory holds rows for keeps
// rows for its first fsm_rows nodes (the shallowest: numbered depth by
// depth, they carry the most probable prefixes).  A byte that leaves the
// code in progress at a node without a row yields an escape: the state value
// esc_base + d, d the bits of that code read so far.  The lane then decodes
// that one code from its first bit through the first-code table and resumes
// byte steps at the byte where it ends (in the skip row of the bits it takes
// there).  Only tensors with such a partial table run the loop that checks
// for escapes; a tree whose nodes all have rows runs the plain loop.

constexpr int kWarpChunks = 32;                                  // chunks per sub-tile
constexpr int kSubtilesPerBlock = kThreads / kWarpChunks;        // 16
constexpr int kMaxChunkCodes = AFX_BLOCK_CAPACITY / kThreads;    // codes one chunk may hold
constexpr int kWarpStage = kWarpChunks * kMaxChunkCodes + 16;    // exponents of one sub-tile
constexpr int kWarpChunkStage = 40;                              // 33 entries staged (80 bytes)
constexpr int kRestoreMaxWarps = 32;
constexpr uint32_t kLutTabBytes = kLutSize * 4 + kLutSize;       // 12-bit table + first-code lengths
constexpr uint32_t kFsmRowBytes = 256 * 8;                       // one state: 256 entries of 8 bytes
constexpr uint32_t kSkipRows = 7;                                // rows that first drop 1..7 bits of a byte
constexpr uint32_t kMinFsmRows = 16;                             // fewest node rows worth a partial table

struct WarpSlot {
    alignas(16) uint16_t chunk[2][kWarpChunkStage];
    alignas(16) uint8_t stage[kWarpStage];
    uint64_t bar[2];    // completion of the bulk copies into stream buffer / chunk row 0 and 1
};

// Fixed part of the restore kernel's shared memory.  It is followed by the
// decode-table region (LaunchArgs::tab_bytes: the 12-bit table and the
// first-code lengths, or the state table), one WarpSlot per warp and two
// stream buffers per warp.
struct SharedW {
    alignas(16) CodeTables ct;       // the tensor's code tables, copied from the launch parameters
    alignas(16) uint16_t first[kLutSize];  // first code of a 12-bit peek: length << 8 | stage byte
    alignas(16) uint8_t tab[16];     // start of the table region
};

static_assert(sizeof(WarpSlot) % 16 == 0 && offsetof(WarpSlot, stage) % 16 == 0, "warp slots stay 16-byte aligned");
static_assert(offsetof(SharedW, tab) % 16 == 0, "table region must be 16-byte aligned");

constexpr size_t sharedw_table_offset() { return offsetof(SharedW, tab); }

// The tables as the decoders see them (pointers into shared memory).
struct TabView {
    const uint32_t* lut;
    const uint8_t* len0;
    const uint32_t* limit;
    const int32_t* base;
    const uint8_t* sorted;
    const uint16_t* first;
    const char* fsm;
    const uint8_t* depth;
    uint32_t fsm_bytes;  // size of the state table (bounds-checked builds)
    uint32_t esc_base;   // state values from here are escapes (a table without every node), else ~0u
};

// One code from a 32-bit window through the first-code table (exact
// length in len), falling back to the canonical limits past 12 bits.  The
// code is complete (the host checks Kraft equality), so every window holds
// a code of at most 24 bits.
__device__ __forceinline__ uint32_t decode_first(const TabView& tv, uint32_t win, uint32_t& len) {
    const uint32_t f = tv.first[win >> (32 - kLutBits)];
    if (f >> 8) {
        len = f >> 8;
        return f & 0xFFu;
    }
    const uint32_t v = win >> 8;
    uint32_t L = kLutBits + 1;
    while (L < AFX_MAX_CODE_LEN && v >= tv.limit[L]) ++L;
    len = L;
    return tv.sorted[tv.base[L] + static_cast<int32_t>(v >> (24 - L))];
}

__device__ __forceinline__ uint32_t stream_window(const uint32_t* stream, uint32_t bit) {
    return __funnelshift_l(stream[(bit >> 5) + 1], stream[bit >> 5], bit & 31u);
}

// The barrier of a whole CTA, for build_tables_w.
struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Builds the tables of tensor tab with threads 0 .. nthreads-1 of the CTA;
// sync() is the barrier of exactly those threads (the whole CTA, or the
// decoding warps of a CTA whose other warps have other roles).
// First pass: the first code of every 12-bit peek (a thread's consecutive
// peeks have non-decreasing lengths, so one search plus short advances).
// Second pass, state-machine tensors: entry (s, b) decodes node s's prefix
// followed by byte b from the start of the code in progress, keeps every
// code that ends within those bits, and names the node of the bits left
// over.  Other tensors: up to three first codes chained per 12-bit peek.
template <class Sync>
__device__ void build_tables_w(SharedW& sh, uint8_t* tabr, const CodeTables& tab, int tid, int nthreads,
                               const Sync& sync) {
    {   // warp w copies words w, w + nwarps, ... of the launch parameters' tables;
        // the lanes of a warp read the same word, one access for the warp
        static_assert(sizeof(CodeTables) % 4 == 0, "CodeTables is copied as words");
        constexpr int kWords = sizeof(CodeTables) / 4;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&tab);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&sh.ct);
        const int nw = nthreads >> 5;
        for (int j = tid >> 5; j < kWords; j += nw) {
            const uint32_t v = src[j];
            if ((tid & 31) == 0) dst[j] = v;
        }
    }
    sync();
    const uint32_t* const limit = sh.ct.limit;
    const int32_t* const base = sh.ct.base;
    const uint32_t* const state_base = sh.ct.state_base;
    const uint8_t* const sorted = sh.ct.sorted;
    for (int p0 = tid * 4; p0 < kLutSize; p0 += nthreads * 4) {
        int L = 1;
        while (L <= kLutBits && (static_cast<uint32_t>(p0) << (24 - kLutBits)) >= limit[L]) ++L;
        for (int j = 0; j < 4; ++j) {
            const uint32_t p = static_cast<uint32_t>(p0 + j);
            const uint32_t v = p << (24 - kLutBits);
            while (L <= kLutBits && v >= limit[L]) ++L;
            uint16_t e = 0;
            if (L <= kLutBits)
                e = static_cast<uint16_t>((L << 8) | sorted[base[L] + static_cast<int32_t>(v >> (24 - L))]);
            sh.first[p] = e;
        }
    }
    sync();
    if (sh.ct.fsm) {
        TabView tv{};
        tv.limit = limit;
        tv.base = base;
        tv.sorted = sorted;
        tv.first = sh.first;
        uint2* fsm = reinterpret_cast<uint2*>(tabr);
        const uint32_t nodes = sh.ct.n_states;
        const uint32_t rows = sh.ct.fsm_rows;  // nodes with a row; a transition to another node escapes
        const uint32_t esc_base = (rows + kSkipRows) * kFsmRowBytes;
        // the root row and the skip rows, code by code
        for (uint32_t i = tid; i < (1 + kSkipRows) * 256u; i += nthreads) {
            const uint32_t h = i >> 8, b = i & 255u;  // h: bits of the byte that end an earlier code
            const uint32_t avail = 8 - h;
            const uint32_t V = b << (24 + h);
            uint32_t pos = 0, out = 0, cnt = 0;
            while (cnt < 4) {
                uint32_t len;
                const uint32_t sym = decode_first(tv, V << pos, len);
                if (len > avail - pos) break;
                out |= sym << (8 * cnt);
                ++cnt;
                pos += len;
            }
            const uint32_t r = avail - pos;
            const uint32_t q = r ? (V << pos) >> (32 - r) : 0u;
            const uint32_t lo_r = r ? limit[r] >> (24 - r) : 0u;
            const uint32_t next = state_base[r] + q - lo_r;
            AFX_CHECK(next < nodes, kChkTableBuild);
            const uint32_t go = next < rows ? next * kFsmRowBytes : esc_base + r;
            fsm[(h ? rows + h - 1 : 0u) * 256u + b] = make_uint2(out, go | ((cnt * 8u) << 26));
        }
        sync();
        // node rows: the code in progress ends h bits into the byte (or does
        // not end in it); the rest of the byte is skip row h
        for (uint32_t i = 256u + tid; i < rows * 256u; i += nthreads) {
            const uint32_t s = i >> 8, b = i & 255u;
            const uint32_t d = sh.ct.state_depth[s];
            const uint32_t lo_d = limit[d] >> (24 - d);
            const uint32_t p = lo_d + s - state_base[d];
            uint32_t len;
            const uint32_t sym = decode_first(tv, (p << (32 - d)) | (b << (24 - d)), len);
            const uint32_t h = len - d;
            uint2 e;
            if (h > 8) {  // still inside the code: the node of its first d + 8 bits
                const uint32_t d8 = d + 8;
                const uint32_t next = state_base[d8] + ((p << 8) | b) - (limit[d8] >> (24 - d8));
                AFX_CHECK(next < nodes, kChkTableBuild);
                e = make_uint2(0u, next < rows ? next * kFsmRowBytes : esc_base + d8);
            } else if (h == 8) {
                e = make_uint2(sym, 8u << 26);
            } else {
                const uint2 rest = fsm[(rows + h - 1) * 256u + b];
                e = make_uint2(sym | (rest.x << 8), rest.y + (8u << 26));
            }
            fsm[i] = e;
        }
    } else {
        uint32_t* lut = reinterpret_cast<uint32_t*>(tabr);
        uint8_t* len0 = tabr + kLutSize * 4;
        for (int p = tid; p < kLutSize; p += nthreads) {
            const uint32_t f1 = sh.first[p];
            const uint32_t l1 = f1 >> 8;
            uint32_t entry = 0;
            if (l1) {
                uint32_t bits = l1, count = 1, syms = f1 & 0xFFu;
                const uint32_t f2 = sh.first[(static_cast<uint32_t>(p) << l1) & (kLutSize - 1)];
                const uint32_t l2 = f2 >> 8;
                if (l2 && bits + l2 <= kLutBits) {
                    bits += l2;
                    syms |= (f2 & 0xFFu) << 8;
                    count = 2;
                    const uint32_t f3 = sh.first[(static_cast<uint32_t>(p) << bits) & (kLutSize - 1)];
                    const uint32_t l3 = f3 >> 8;
                    if (l3 && bits + l3 <= kLutBits) {
                        bits += l3;
                        syms |= (f3 & 0xFFu) << 16;
                        count = 3;
                    }
                }
                entry = bits | (count << 4) | (syms << 8);
            }
            lut[p] = entry;
            len0[p] = static_cast<uint8_t>(l1);
        }
    }
    sync();
}

// One step of the state machine: the byte b read in state st (the byte
// offset of its row).
__device__ __forceinline__ void fsm_step(const char* fsm, uint32_t& st, uint32_t b, uint32_t& acc, uint32_t& fill,
                                         uint32_t*& wout) {
    const uint2 e = *reinterpret_cast<const uint2*>(fsm + st + (b << 3));
    append(e.x, e.y >> 26, acc, fill, wout);
    st = e.y & 0x3FFFFFFu;
}

// The same step with the state offset checked in bounds-checked builds.
__device__ __forceinline__ void fsm_step_checked(const TabView& tv, uint32_t& st, uint32_t b, uint32_t& acc,
                                                 uint32_t& fill, uint32_t*& wout) {
    AFX_CHECK(st + (b << 3) + 8 <= tv.fsm_bytes, kChkTableState);
    fsm_step(tv.fsm, st, b, acc, fill, wout);
}

// Byte-step counterpart of decode_run (same contract).  stream_end is the
// bit offset in the staged stream where the coded bits end: the padding
// after it decodes as codes, so no step reads past it.
__device__ __forceinline__ bool decode_run_fsm(const TabView& tv, const uint32_t* stream, uint32_t k0, uint32_t gap,
                                               uint32_t cnt, uint8_t* stage, uint32_t s0, uint32_t next,
                                               uint32_t chunk_end, uint32_t stream_end) {
    uint32_t P = k0 * 32u + gap;  // bit of the next code in the staged stream
    uint32_t i = 0;
    // head: codes until the stage index is word aligned, one at a time
    const uint32_t head = min(cnt, (0u - s0) & 3u);
    for (; i < head; ++i) {
        uint32_t len;
        stage[s0 + i] = static_cast<uint8_t>(decode_first(tv, stream_window(stream, P), len));
        P += len;
    }
    uint32_t* wout = reinterpret_cast<uint32_t*>(stage + s0 + i);
    const uint32_t* const w_begin = wout;
    uint32_t acc = 0, fill = 0;
    bool bad = false;
    if (i < cnt) {
        // whole bytes of the chunk's bits from the code at P (none with a
        // partial table: its codes all go through the tail loop below)
        const uint32_t lim = min(chunk_end, stream_end);
        const uint32_t steps = lim > P && tv.esc_base == ~0u ? (lim - P) >> 3 : 0u;
        uint32_t k = P >> 5;
        const uint32_t sh = P & 31u;
        uint32_t w0 = stream[k], w1 = stream[k + 1];
        uint32_t st = 0;  // the root
        for (uint32_t q = steps >> 2; q; --q) {
            const uint32_t X = __funnelshift_l(w1, w0, sh);
            w0 = w1;
            w1 = stream[k + 2];
            ++k;
            fsm_step(tv.fsm, st, X >> 24, acc, fill, wout);
            fsm_step(tv.fsm, st, __byte_perm(X, 0u, 0x4442), acc, fill, wout);
            fsm_step(tv.fsm, st, __byte_perm(X, 0u, 0x4441), acc, fill, wout);
            fsm_step(tv.fsm, st, X & 0xFFu, acc, fill, wout);
        }
        const uint32_t rem = steps & 3u;
        if (rem) {
            const uint32_t X = __funnelshift_l(w1, w0, sh);
            fsm_step(tv.fsm, st, X >> 24, acc, fill, wout);
            if (rem > 1) fsm_step(tv.fsm, st, __byte_perm(X, 0u, 0x4442), acc, fill, wout);
            if (rem > 2) fsm_step(tv.fsm, st, __byte_perm(X, 0u, 0x4441), acc, fill, wout);
        }
        // the code in progress began depth(st) bits before the last step's end
        P += 8 * steps - tv.depth[st / kFsmRowBytes];
        i += 4 * static_cast<uint32_t>(wout - w_begin) + (fill >> 3);
        bad = i > cnt;
    }
    // tail: the codes that start in the last bits of the chunk
    while (!bad && i < cnt) {
        if (P >= chunk_end) {
            bad = true;
            break;
        }
        uint32_t len;
        const uint32_t sym = decode_first(tv, stream_window(stream, P), len);
        append(sym, 8, acc, fill, wout);
        P += len;
        ++i;
    }
    uint8_t* tail = reinterpret_cast<uint8_t*>(wout);
    for (uint32_t j = 0; j * 8 < fill; ++j) tail[j] = static_cast<uint8_t>(acc >> (8 * j));
    if (!bad) {
        if ((next >> 5) != 0)
            bad = P != chunk_end + (next & 31u);
        else
            bad = P > chunk_end + AFX_MAX_CODE_LEN;
    }
    return bad;
}

// What a lane's byte steps leave for after the warp barrier: the
// exponents not yet stored (acc, fill bits), the word they go to, the byte
// of that word where this lane's own bytes begin, the count of codes
// emitted and the final state.
struct FsmLane {
    uint32_t* wout;
    uint32_t acc, fill, first, emitted, st;
    uint32_t xend;  // partial tables: where a code that an escape decoded past the chunk end ends (0: none)
};

// All T bytes of a full chunk whose first word is words[0] (byte-step
// decoding).  Completed stage words are stored whole, including a first
// word shared with the previous lane: that lane stores its bytes of the
// word only after the warp barrier.
__device__ __forceinline__ void fsm_chunk_steps(const TabView& tv, const uint32_t* words, uint32_t nwords, uint32_t gap,
                                                uint32_t skip_row0, uint8_t* stage, uint32_t s_run, FsmLane& fl,
                                                uint32_t stage_cap = kWarpStage) {
    uint32_t* wout = reinterpret_cast<uint32_t*>(stage + (s_run & ~3u));
    const uint32_t* const w_begin = wout;
    uint32_t acc = 0, fill = 8 * (s_run & 3u);
    const uint32_t h = gap & 7u;
    uint32_t st = h ? skip_row0 + (h - 1) * kFsmRowBytes : 0u;
    const uint32_t X0 = words[0];
    if (gap < 8) fsm_step_checked(tv, st, X0 >> 24, acc, fill, wout);
    if (gap < 16) fsm_step_checked(tv, st, __byte_perm(X0, 0u, 0x4442), acc, fill, wout);
    fsm_step_checked(tv, st, __byte_perm(X0, 0u, 0x4441), acc, fill, wout);
    fsm_step_checked(tv, st, X0 & 0xFFu, acc, fill, wout);
    for (uint32_t w = 1; w < nwords; ++w) {
        const uint32_t X = words[w];
        fsm_step_checked(tv, st, X >> 24, acc, fill, wout);
        fsm_step_checked(tv, st, __byte_perm(X, 0u, 0x4442), acc, fill, wout);
        fsm_step_checked(tv, st, __byte_perm(X, 0u, 0x4441), acc, fill, wout);
        fsm_step_checked(tv, st, X & 0xFFu, acc, fill, wout);
    }
    AFX_CHECK(reinterpret_cast<uint8_t*>(wout) <= stage + stage_cap, kChkStageSteps);
    fl.wout = wout;
    fl.acc = acc;
    fl.fill = fill;
    fl.first = wout == w_begin ? (s_run & 3u) : 0u;
    fl.emitted = 4 * static_cast<uint32_t>(wout - w_begin) + (fill >> 3) - (s_run & 3u);
    fl.st = st;
}

// fsm_chunk_steps for a run of 4k words (a 16-byte chunk or larger, or a
// two-chunk span of 8-byte chunks or larger): the words come in as 16-byte
// loads.  The lanes' runs lie 16 or more bytes apart, so word loads put
// four lanes (16-byte chunks) or eight (32-byte spans) on each bank and
// the shared-memory pipe replays them; 16-byte loads of 16-byte chunks
// are conflict-free, and of 32-byte spans take twice the minimum passes.
__device__ __forceinline__ void fsm_span_steps(const TabView& tv, const uint32_t* words, uint32_t nwords, uint32_t gap,
                                               uint32_t skip_row0, uint8_t* stage, uint32_t s_run, FsmLane& fl,
                                               uint32_t stage_cap) {
    uint32_t* wout = reinterpret_cast<uint32_t*>(stage + (s_run & ~3u));
    const uint32_t* const w_begin = wout;
    uint32_t acc = 0, fill = 8 * (s_run & 3u);
    const uint32_t h = gap & 7u;
    uint32_t st = h ? skip_row0 + (h - 1) * kFsmRowBytes : 0u;
    auto word = [&](uint32_t X) {
        fsm_step_checked(tv, st, X >> 24, acc, fill, wout);
        fsm_step_checked(tv, st, __byte_perm(X, 0u, 0x4442), acc, fill, wout);
        fsm_step_checked(tv, st, __byte_perm(X, 0u, 0x4441), acc, fill, wout);
        fsm_step_checked(tv, st, X & 0xFFu, acc, fill, wout);
    };
    const uint4 X0 = *reinterpret_cast<const uint4*>(words);
    if (gap < 8) fsm_step_checked(tv, st, X0.x >> 24, acc, fill, wout);
    if (gap < 16) fsm_step_checked(tv, st, __byte_perm(X0.x, 0u, 0x4442), acc, fill, wout);
    fsm_step_checked(tv, st, __byte_perm(X0.x, 0u, 0x4441), acc, fill, wout);
    fsm_step_checked(tv, st, X0.x & 0xFFu, acc, fill, wout);
    word(X0.y);
    word(X0.z);
    word(X0.w);
    for (uint32_t w = 4; w < nwords; w += 4) {
        const uint4 X = *reinterpret_cast<const uint4*>(words + w);
        word(X.x);
        word(X.y);
        word(X.z);
        word(X.w);
    }
    AFX_CHECK(reinterpret_cast<uint8_t*>(wout) <= stage + stage_cap, kChkStageSteps);
    fl.wout = wout;
    fl.acc = acc;
    fl.fill = fill;
    fl.first = wout == w_begin ? (s_run & 3u) : 0u;
    fl.emitted = 4 * static_cast<uint32_t>(wout - w_begin) + (fill >> 3) - (s_run & 3u);
    fl.st = st;
}

// fsm_chunk_steps for a partial table: the same steps from stream word k0
// (the chunk's first), four to a word while no escape comes, with each
// escape handled where it comes.  The code an escape decodes may cross the
// chunk end; the lane then stops there and records where it ends (fl.xend,
// a bit of the staged stream).
__device__ __forceinline__ void fsm_chunk_steps_esc(const TabView& tv, const uint32_t* stream, uint32_t k0,
                                                    uint32_t nbytes, uint32_t gap, uint32_t skip_row0, uint8_t* stage,
                                                    uint32_t s_run, FsmLane& fl, uint32_t stage_cap = kWarpStage) {
    uint32_t* wout = reinterpret_cast<uint32_t*>(stage + (s_run & ~3u));
    const uint32_t* const w_begin = wout;
    uint32_t acc = 0, fill = 8 * (s_run & 3u);
    const uint32_t h0 = gap & 7u;
    uint32_t st = h0 ? skip_row0 + (h0 - 1) * kFsmRowBytes : 0u;
    uint32_t xend = 0;
    uint32_t j = gap >> 3;  // the next byte to step
    while (j < nbytes) {
        const uint32_t X = stream[k0 + (j >> 2)];
        uint32_t done;  // bytes of this word stepped; the last of them escaped if st >= esc_base
        if ((j & 3u) == 0) {
            fsm_step_checked(tv, st, X >> 24, acc, fill, wout);
            done = 1;
            if (st < tv.esc_base) {
                fsm_step_checked(tv, st, __byte_perm(X, 0u, 0x4442), acc, fill, wout);
                done = 2;
                if (st < tv.esc_base) {
                    fsm_step_checked(tv, st, __byte_perm(X, 0u, 0x4441), acc, fill, wout);
                    done = 3;
                    if (st < tv.esc_base) {
                        fsm_step_checked(tv, st, X & 0xFFu, acc, fill, wout);
                        done = 4;
                    }
                }
            }
        } else {  // after an escape: one byte at a time up to the word boundary
            fsm_step_checked(tv, st, (X >> (24u - 8u * (j & 3u))) & 0xFFu, acc, fill, wout);
            done = 1;
        }
        j += done;
        if (st >= tv.esc_base) {
            // the code in progress began st - esc_base bits before byte j's start
            const uint32_t P = 8u * j - (st - tv.esc_base);
            uint32_t len;
            const uint32_t sym = decode_first(tv, stream_window(stream, 32u * k0 + P), len);
            append(sym, 8, acc, fill, wout);
            const uint32_t e = P + len;
            st = 0u;
            if (e >= 8u * nbytes) {  // it ends at or past the chunk end
                if (e > 8u * nbytes) xend = 32u * k0 + e;
                break;
            }
            j = e >> 3;
            if (e & 7u) st = skip_row0 + ((e & 7u) - 1) * kFsmRowBytes;
        }
    }
    AFX_CHECK(reinterpret_cast<uint8_t*>(wout) <= stage + stage_cap, kChkStageSteps);
    fl.wout = wout;
    fl.acc = acc;
    fl.fill = fill;
    fl.first = wout == w_begin ? (s_run & 3u) : 0u;
    fl.emitted = 4 * static_cast<uint32_t>(wout - w_begin) + (fill >> 3) - (s_run & 3u);
    fl.st = st;
    fl.xend = xend;
}

// After the warp barrier: the code that crosses the chunk end (if the final
// state is not the root), the lane's pending bytes, and the checks of the
// count and of where the next chunk's first code begins.  Returns true when
// the stream is not valid.  kPartial: the lane ran fsm_chunk_steps_esc.
template <bool kPartial = false>
__device__ __forceinline__ bool fsm_chunk_finish(const TabView& tv, const uint32_t* stream, const FsmLane& fl,
                                                 uint32_t cnt, uint32_t chunk_end, uint32_t next) {
    const uint32_t d = tv.depth[fl.st / kFsmRowBytes];
    uint32_t end = chunk_end, emitted = fl.emitted, acc = fl.acc, fill = fl.fill;
    if constexpr (kPartial) {
        if (fl.xend) end = fl.xend;
    }
    if (d) {
        uint32_t len;
        const uint32_t sym = decode_first(tv, stream_window(stream, chunk_end - d), len);
        end = chunk_end - d + len;
        acc |= sym << fill;  // fill <= 24 here
        fill += 8;
        ++emitted;
    }
    uint8_t* p = reinterpret_cast<uint8_t*>(fl.wout);
    const uint32_t pending = fill >> 3;  // 0..4 bytes
#pragma unroll
    for (uint32_t j = 0; j < 4; ++j)
        if (j >= fl.first && j < pending) p[j] = static_cast<uint8_t>(acc >> (8 * j));
    bool bad = emitted != cnt;
    if ((next >> 5) != 0)
        bad = bad || end != chunk_end + (next & 31u);
    else
        bad = bad || end > chunk_end + AFX_MAX_CODE_LEN;
    return bad;
}

__device__ __forceinline__ uint32_t warp_stream_bytes(const TensorArgs& t, uint64_t s) {
    const uint64_t byte0 = s * kWarpChunks * t.chunk_bytes;
    const uint64_t want = static_cast<uint64_t>(kWarpChunks) * t.chunk_bytes + kStreamPad;
    const uint64_t avail = t.exp_bytes > byte0 ? t.exp_bytes - byte0 : 0;
    return static_cast<uint32_t>(want < avail ? want : avail);
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
    return v;
}

// Bytes staged for sub-tile s: the stream bytes of its 32 chunks plus the
// pad, and its 40 chunk entries (the next sub-tile's first included).  A
// full sub-tile (TensorArgs::n_sub_full) has all of them; the last ones take
// what the sections hold.  Both are multiples of 16.
__device__ __forceinline__ uint2 sub_tile_bytes(const TensorArgs& t, uint64_t s, bool full, uint32_t sub_bytes) {
    if (full) return make_uint2(sub_bytes + kStreamPad, kWarpChunkStage * 2);
    const uint64_t cb0 = s * kWarpChunks * 2;
    const uint64_t csec = (t.n_chunks * 2 + 15) & ~uint64_t(15);
    const uint64_t cavail = csec > cb0 ? csec - cb0 : 0;
    return make_uint2(warp_stream_bytes(t, s),
                      static_cast<uint32_t>(cavail < kWarpChunkStage * 2 ? cavail : kWarpChunkStage * 2));
}

// Stages sub-tile s in buffer b with two bulk copies on ws.bar[b], issued
// by lane 0 (device-resident containers).  Every size and address is a
// multiple of 16.
__device__ __forceinline__ void warp_issue_bulk(WarpSlot& ws, uint8_t* stream_dst, const TensorArgs& t, uint64_t s,
                                                bool full, const uint8_t* exp_src, const uint16_t* chunk_src,
                                                uint32_t sub_bytes, int b, bool stall) {
    const uint2 nb = sub_tile_bytes(t, s, full, sub_bytes);
    AFX_CHECK(nb.x <= sub_bytes + kStreamPad && nb.y <= kWarpChunkStage * 2, kChkStagingBytes);
    mbar_expect_tx(&ws.bar[b], nb.x + nb.y);
    if (stall) return;  // failure injection: the bytes never come
    if (nb.x) bulk_copy_g2s(stream_dst, exp_src, nb.x, &ws.bar[b]);
    if (nb.y) bulk_copy_g2s(ws.chunk[b], chunk_src, nb.y, &ws.bar[b]);
}

// The same staging from a container in pinned host memory, read over the
// host link with plain 16-byte loads by all lanes (no bulk copies).
__device__ __forceinline__ void warp_stage_host(WarpSlot& ws, uint8_t* stream_dst, const TensorArgs& t, uint64_t s,
                                                bool full, const uint8_t* exp_src, const uint16_t* chunk_src,
                                                uint32_t sub_bytes, int b, int lane) {
    const uint2 nb = sub_tile_bytes(t, s, full, sub_bytes);
    AFX_CHECK(nb.x <= sub_bytes + kStreamPad && nb.y <= kWarpChunkStage * 2, kChkStagingBytes);
    for (uint32_t i = lane * 16u; i < nb.x; i += 32 * 16u)
        *reinterpret_cast<uint4*>(stream_dst + i) = *reinterpret_cast<const uint4*>(exp_src + i);
    if (lane * 16u < nb.y)
        *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws.chunk[b]) + lane * 16) =
            *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(chunk_src) + lane * 16);
}

}  // namespace afx
