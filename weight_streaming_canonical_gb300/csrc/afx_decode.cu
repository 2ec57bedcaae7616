// sm_103a kernels of afx: restore BF16 weights from the exponent-coded
// container, alone (afx_decode) or fused into a batch-1..4 GEMV
// (afx_decode_gemv).
//
// The operation: "Why Weight Offloading Slows Inference", section
// "Lossless compression: fewer bytes to read, more work to unpack" -- every
// weight's exponent was stored with a shorter code for common values, its
// sign and mantissa raw; the released bits are restored before compute.
// This is the t_unpack term of that page's Eq. (1).
//
// Work decomposition (one CTA tile = one block of the container = 256
// chunks of 8*T stream bits, persistent CTAs loop over tiles):
//   1. stage the tile's stream words and chunk-index entries in shared
//      memory;
//   2. each thread takes one chunk: the index gives the bit offset of its
//      first codeword and how many codewords start in it; a warp-shuffle
//      plus block prefix scan of those counts places every thread's run of
//      outputs inside the tile;
//   3. each thread decodes its codewords through a two-level table in
//      shared memory (a 4096-entry table resolves every code of at most 12
//      bits from a 12-bit peek; longer codes, up to 24 bits, fall back to a
//      per-length canonical search) into a shared exponent buffer;
//   4. the whole CTA joins exponents with the sign|mantissa bytes in
//      aligned groups of 8 weights: 8-byte coalesced loads of
//      sign|mantissa and 16-byte coalesced BF16 stores (or, fused, 8
//      products per batch row with no store of the weights at all).
// Every index read from the container is checked before it is used to
// address shared or global memory; a bad value sets a status bit and the
// tile is skipped.  No kernel waits on anything but __syncthreads.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "afx_internal.h"

thread_local char g_last_error[256] = "no error";

extern "C" afx_status afx_fail(afx_status status, const char* what, int cuda_error) {
    if (cuda_error)
        snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", what,
                 cudaGetErrorName(static_cast<cudaError_t>(cuda_error)),
                 cudaGetErrorString(static_cast<cudaError_t>(cuda_error)));
    else
        snprintf(g_last_error, sizeof g_last_error, "%s", what);
    return status;
}

extern "C" const char* afx_last_error(void) { return g_last_error; }

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
constexpr int kMaxBatch = 4;

// Canonical decode tables, built on the host from the 256 code lengths.
// In 24-bit left-aligned code space, all codes of length <= L lie in
// [0, limit[L]); a 24-bit peek v therefore has the length L = the smallest L
// with v < limit[L], and its exponent is sorted[base[L] + (v >> (24 - L))].
struct CodeTables {
    uint32_t limit[AFX_MAX_CODE_LEN + 1];
    int32_t base[AFX_MAX_CODE_LEN + 1];
    uint8_t sorted[256];
};

struct TileShared {
    uint16_t lut[kLutSize];  // (length << 8) | exponent for codes <= 12 bits; 0 = longer code
    uint32_t limit[AFX_MAX_CODE_LEN + 1];
    int32_t base[AFX_MAX_CODE_LEN + 1];
    uint8_t sorted[256];
    uint16_t chunk[kThreads + 1];  // this tile's chunk entries plus the next tile's first
    uint32_t warp_total[kWarps];
    int32_t tile_ok;
    uint8_t stage[kStageBytes];  // exponents of the tile, at (o - o0 + (o0 & 7))
    // followed by the staged stream words (dynamic size)
};

struct DecodeArgs {
    const uint32_t* exp_words;   // exp section
    const uint8_t* sm;           // sign|mantissa section
    const uint16_t* chunk_index;
    const uint64_t* block_index;
    uint64_t n;
    uint64_t n_chunks;
    uint64_t n_blocks;
    uint64_t exp_bytes;
    uint32_t chunk_bytes;        // T
    int32_t* status;
};

__device__ __forceinline__ void raise_status(int32_t* status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// BF16 from exponent and sign|mantissa: sign to bit 15, exponent to bits
// 7..14, mantissa to bits 0..6.  Four weights per call: e4 and s4 hold four
// exponent and four sign|mantissa bytes; the result is two u32 of packed
// BF16 pairs.  byte_perm interleaves to (e << 8) | s per 16-bit lane; then
// s bits 0..6 stay, e moves down one bit to 7..14, s bit 7 moves to 15.
__device__ __forceinline__ uint32_t join_pair(uint32_t x) {
    return (x & 0x007F007Fu) | ((x >> 1) & 0x7F807F80u) | ((x << 8) & 0x80008000u);
}

__device__ __forceinline__ uint2 join4(uint32_t e4, uint32_t s4) {
    uint2 r;
    r.x = join_pair(__byte_perm(s4, e4, 0x5140));
    r.y = join_pair(__byte_perm(s4, e4, 0x7362));
    return r;
}

__device__ __forceinline__ uint16_t join1(uint32_t e, uint32_t s) {
    return static_cast<uint16_t>(((s & 0x80u) << 8) | (e << 7) | (s & 0x7Fu));
}

__device__ void build_tables(TileShared& sh, const CodeTables& tab) {
    const int tid = threadIdx.x;
    for (int i = tid; i <= AFX_MAX_CODE_LEN; i += kThreads) {
        sh.limit[i] = tab.limit[i];
        sh.base[i] = tab.base[i];
    }
    for (int i = tid; i < 256; i += kThreads) sh.sorted[i] = tab.sorted[i];
    for (int p = tid; p < kLutSize; p += kThreads) {
        const uint32_t v = static_cast<uint32_t>(p) << (24 - kLutBits);
        int len = 0;  // smallest L <= 12 with v < limit[L]; 0 = the code is longer
#pragma unroll
        for (int L = kLutBits; L >= 1; --L)
            if (v < tab.limit[L]) len = L;
        uint16_t entry = 0;
        if (len) {
            const uint32_t sym = tab.sorted[tab.base[len] + static_cast<int32_t>(v >> (24 - len))];
            entry = static_cast<uint16_t>((len << 8) | sym);
        }
        sh.lut[p] = entry;
    }
}

// Exclusive block-wide scan of one count per thread; returns this thread's
// offset and writes the total into *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(TileShared& sh, uint32_t v, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) sh.warp_total[warp] = inc;
    __syncthreads();
    uint32_t warp_off = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = sh.warp_total[w];
        if (w < warp) warp_off += t;
        all += t;
    }
    *total = all;
    return warp_off + inc - v;
}

// Stages tile b, scans, decodes the tile's exponents into sh.stage.
// Returns false (uniformly) when the tile must be skipped.
__device__ bool decode_tile(TileShared& sh, uint32_t* stream, const DecodeArgs& a, uint64_t b, uint64_t& o0,
                            uint64_t& o1) {
    const int tid = threadIdx.x;
    const uint32_t T = a.chunk_bytes;
    const uint32_t words_per_chunk = T >> 2;
    const uint64_t tile_byte0 = b * static_cast<uint64_t>(kThreads) * T;
    const uint64_t want = static_cast<uint64_t>(kThreads) * T + 16;
    const uint64_t avail_bytes = a.exp_bytes > tile_byte0 ? a.exp_bytes - tile_byte0 : 0;
    const uint32_t stage_bytes = static_cast<uint32_t>(want < avail_bytes ? want : avail_bytes);
    const uint32_t staged_words = stage_bytes >> 2;

    // 1. stage stream words (16-byte vectors) and chunk entries
    {
        const uint4* src = reinterpret_cast<const uint4*>(a.exp_words + (tile_byte0 >> 2));
        uint4* dst = reinterpret_cast<uint4*>(stream);
        for (uint32_t i = tid; i < (stage_bytes >> 4); i += kThreads) dst[i] = __ldg(src + i);
        const uint64_t c0 = b * kThreads;
        for (int i = tid; i <= kThreads; i += kThreads) {
            const uint64_t c = c0 + i;
            sh.chunk[i] = c < a.n_chunks ? __ldg(a.chunk_index + c) : uint16_t(0);
        }
        if (tid == 0) sh.tile_ok = 1;
    }
    o0 = __ldg(a.block_index + b);
    o1 = __ldg(a.block_index + b + 1);
    __syncthreads();

    // 2. counts and placement
    const uint32_t entry = sh.chunk[tid];
    const uint32_t gap = entry & 31u;
    uint32_t cnt = entry >> 5;
    const uint32_t chunk_bits = 8u * T;
    if (cnt > chunk_bits - gap || gap > 23u) {
        raise_status(a.status, AFX_DEV_BAD_CHUNK);
        sh.tile_ok = 0;
        cnt = 0;
    }
    uint32_t total = 0;
    const uint32_t off = block_exclusive_scan(sh, cnt, &total);
    const bool last_ok = b + 1 != a.n_blocks || o1 == a.n;  // the block index ends at n
    if (o1 < o0 || o1 - o0 != total || total > AFX_BLOCK_CAPACITY || o1 > a.n || !last_ok) {
        if (tid == 0) raise_status(a.status, AFX_DEV_BAD_BLOCK);
        return false;  // uniform: every thread sees the same o0, o1, total
    }

    // 3. decode this thread's codewords
    if (cnt) {
        uint32_t widx = tid * words_per_chunk;
        uint64_t buf = (static_cast<uint64_t>(stream[widx]) << 32) | stream[widx + 1];
        buf <<= gap;
        int avail = 64 - static_cast<int>(gap);
        widx += 2;
        uint8_t* out = sh.stage + (o0 & 7u) + off;
        bool bad = false;
        for (uint32_t i = 0; i < cnt; ++i) {
            if (avail < 32) {
                if (widx >= staged_words) {
                    bad = true;
                    break;
                }
                buf |= static_cast<uint64_t>(stream[widx++]) << (32 - avail);
                avail += 32;
            }
            const uint32_t e = sh.lut[static_cast<uint32_t>(buf >> (64 - kLutBits))];
            uint32_t len = e >> 8;
            uint32_t sym = e & 0xFFu;
            if (len == 0) {
                const uint32_t v = static_cast<uint32_t>(buf >> 40);
                len = kLutBits + 1;
                while (len <= AFX_MAX_CODE_LEN && v >= sh.limit[len]) ++len;
                if (len > AFX_MAX_CODE_LEN) {
                    bad = true;
                    break;
                }
                sym = sh.sorted[sh.base[len] + static_cast<int32_t>(v >> (24 - len))];
            }
            buf <<= len;
            avail -= static_cast<int>(len);
            out[i] = static_cast<uint8_t>(sym);
        }
        // the codewords must end exactly where the next chunk's first begins
        const uint32_t next = sh.chunk[tid + 1];
        const uint32_t end = widx * 32u - static_cast<uint32_t>(avail);
        const uint32_t chunk_end = (tid + 1) * chunk_bits;
        if (!bad) {
            if ((next >> 5) != 0)
                bad = end != chunk_end + (next & 31u);
            else
                bad = end > chunk_end + AFX_MAX_CODE_LEN;
        }
        if (bad) {
            raise_status(a.status, AFX_DEV_BAD_CHUNK);
            sh.tile_ok = 0;
        }
    }
    __syncthreads();
    return sh.tile_ok != 0;
}

struct StoreArgs {
    uint16_t* out;
};

__global__ void __launch_bounds__(kThreads) decode_store_kernel(const DecodeArgs a, const CodeTables tab,
                                                                 const StoreArgs st) {
    extern __shared__ __align__(16) uint8_t smem[];
    TileShared& sh = *reinterpret_cast<TileShared*>(smem);
    uint32_t* stream = reinterpret_cast<uint32_t*>(smem + ((sizeof(TileShared) + 15) & ~size_t(15)));
    build_tables(sh, tab);
    __syncthreads();
    for (uint64_t b = blockIdx.x; b < a.n_blocks; b += gridDim.x) {
        uint64_t o0, o1;
        if (decode_tile(sh, stream, a, b, o0, o1)) {
            const uint64_t ob0 = o0 & ~uint64_t(7);  // stage[i] holds weight ob0 + i
            const uint64_t g0 = o0 >> 3, g1 = (o1 + 7) >> 3;
            for (uint64_t g = g0 + threadIdx.x; g < g1; g += kThreads) {
                const uint64_t ob = g << 3;
                const uint32_t si = static_cast<uint32_t>(ob - ob0);  // multiple of 8
                if (ob >= o0 && ob + 8 <= o1) {
                    const uint2 e8 = *reinterpret_cast<const uint2*>(sh.stage + si);
                    const uint2 s8 = __ldg(reinterpret_cast<const uint2*>(a.sm + ob));
                    const uint2 lo = join4(e8.x, s8.x);
                    const uint2 hi = join4(e8.y, s8.y);
                    uint4 v;
                    v.x = lo.x;
                    v.y = lo.y;
                    v.z = hi.x;
                    v.w = hi.y;
                    __stcs(reinterpret_cast<uint4*>(st.out + ob), v);
                } else {
                    for (uint32_t k = 0; k < 8; ++k) {
                        const uint64_t o = ob + k;
                        if (o >= o0 && o < o1) st.out[o] = join1(sh.stage[si + k], a.sm[o]);
                    }
                }
            }
        }
        __syncthreads();
    }
}

// One exponent for every weight: out[i] = join(fill, sm[i]).  The block
// index holds the single entry n.
__global__ void fill_store_kernel(const uint8_t* __restrict__ sm, const uint64_t* __restrict__ block_index,
                                  uint32_t fill, uint64_t n, uint16_t* __restrict__ out, int32_t* status) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && block_index[0] != n) raise_status(status, AFX_DEV_BAD_BLOCK);
    const uint64_t groups = (n + 7) >> 3;
    const uint32_t f4 = fill * 0x01010101u;
    for (uint64_t g = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; g < groups;
         g += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const uint64_t ob = g << 3;
        if (ob + 8 <= n) {
            const uint2 s8 = __ldg(reinterpret_cast<const uint2*>(sm + ob));
            const uint2 lo = join4(f4, s8.x);
            const uint2 hi = join4(f4, s8.y);
            __stcs(reinterpret_cast<uint4*>(out + ob), make_uint4(lo.x, lo.y, hi.x, hi.y));
        } else {
            for (uint64_t o = ob; o < n; ++o) out[o] = join1(fill, sm[o]);
        }
    }
}

// ---- fused GEMV ------------------------------------------------------------
//
// y[b][r] = sum_c W[r][c] x[b][c].  Within a tile, warp w takes a contiguous
// slice of 8-weight groups, so it meets the rows of its slice in order.
// Each lane keeps float32 sums for the warp's current row; when the row
// changes the warp reduces them with a fixed butterfly and stores one
// partial per (warp, row) in shared memory.  Then every row of the tile is
// summed over warps in warp order: rows that lie wholly in the tile go to
// y, the tile's first and last (partial) rows go to the workspace, and
// gemv_fixup_kernel adds those across tiles in tile order.  Every sum has a
// fixed order, so y is reproducible bit for bit.

struct GemvArgs {
    const uint16_t* x;
    float* y;
    float* ws;          // [n_blocks][2][batch]
    uint32_t rows, cols;
    uint32_t batch;
    uint32_t rows_per_warp;  // capacity of the per-warp partial table
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

template <int B>
__device__ __forceinline__ void warp_flush(float (&acc)[kMaxBatch], float* part, uint32_t slot, int lane) {
#pragma unroll
    for (int b = 0; b < B; ++b) {
        float v = acc[b];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
        if (lane == 0) part[slot * B + b] = v;
        acc[b] = 0.f;
    }
}

template <int B>
__global__ void __launch_bounds__(kThreads) decode_gemv_kernel(const DecodeArgs a, const CodeTables tab,
                                                                const GemvArgs g) {
    extern __shared__ __align__(16) uint8_t smem[];
    TileShared& sh = *reinterpret_cast<TileShared*>(smem);
    uint8_t* after = smem + ((sizeof(TileShared) + 15) & ~size_t(15));
    uint32_t* stream = reinterpret_cast<uint32_t*>(after);
    const uint32_t stream_bytes = kThreads * a.chunk_bytes + 16;
    float* part = reinterpret_cast<float*>(after + stream_bytes);   // [kWarps][rows_per_warp][B]
    uint64_t* warp_row0 = reinterpret_cast<uint64_t*>(part + kWarps * g.rows_per_warp * B);  // [kWarps]
    uint32_t* warp_nrows = reinterpret_cast<uint32_t*>(warp_row0 + kWarps);                   // [kWarps]

    build_tables(sh, tab);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t cols = g.cols;
    const bool vec_x = (cols & 7u) == 0;

    for (uint64_t tb = blockIdx.x; tb < a.n_blocks; tb += gridDim.x) {
        uint64_t o0, o1;
        if (!decode_tile(sh, stream, a, tb, o0, o1) || o0 == o1) {
            __syncthreads();
            continue;
        }
        const uint64_t ob0 = o0 & ~uint64_t(7);  // stage[i] holds weight ob0 + i
        const uint64_t g0 = o0 >> 3, g1 = (o1 + 7) >> 3;
        const uint64_t ng = g1 - g0;
        const uint64_t s_begin = g0 + ng * warp / kWarps, s_end = g0 + ng * (warp + 1) / kWarps;

        uint64_t cur = ~uint64_t(0), row0 = 0;
        uint32_t nrows = 0;
        if (s_begin < s_end) {
            const uint64_t first_o = (s_begin << 3) > o0 ? (s_begin << 3) : o0;
            row0 = first_o / cols;
            cur = row0;
        }
        float acc[kMaxBatch] = {0.f, 0.f, 0.f, 0.f};
        for (uint64_t base = s_begin; base < s_end; base += 32) {
            const uint64_t gi = base + lane;
            const bool active = gi < s_end;
            // rows met by this step: from the first element of the step to its last
            const uint64_t step_first = (base << 3) > o0 ? (base << 3) : o0;
            const uint64_t last_g = (base + 32 < s_end ? base + 32 : s_end) - 1;
            const uint64_t step_last = ((last_g << 3) + 7) < o1 - 1 ? ((last_g << 3) + 7) : o1 - 1;
            const uint64_t r_lo = step_first / cols, r_hi = step_last / cols;

            // this lane's products, split by row (a group meets at most two rows as cols >= 64)
            float ca[kMaxBatch] = {0.f, 0.f, 0.f, 0.f}, cb[kMaxBatch] = {0.f, 0.f, 0.f, 0.f};
            uint64_t ra = ~uint64_t(0), rb = ~uint64_t(0);
            if (active) {
                const uint64_t ob = gi << 3;
                const uint32_t si = static_cast<uint32_t>(ob - ob0);
                const bool full = ob >= o0 && ob + 8 <= o1;
                ra = (ob >= o0 ? ob : o0) / cols;
                const uint64_t c0 = ob - ra * cols;
                if (full && vec_x && c0 + 8 <= cols) {
                    const uint2 e8 = *reinterpret_cast<const uint2*>(sh.stage + si);
                    const uint2 s8 = __ldg(reinterpret_cast<const uint2*>(a.sm + ob));
                    const uint2 lo = join4(e8.x, s8.x);
                    const uint2 hi = join4(e8.y, s8.y);
                    float wv[8];
                    wv[0] = bf16_lo(lo.x); wv[1] = bf16_hi(lo.x);
                    wv[2] = bf16_lo(lo.y); wv[3] = bf16_hi(lo.y);
                    wv[4] = bf16_lo(hi.x); wv[5] = bf16_hi(hi.x);
                    wv[6] = bf16_lo(hi.y); wv[7] = bf16_hi(hi.y);
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(g.x + b * cols + c0));
                        float s = wv[0] * bf16_lo(xv.x);
                        s = fmaf(wv[1], bf16_hi(xv.x), s);
                        s = fmaf(wv[2], bf16_lo(xv.y), s);
                        s = fmaf(wv[3], bf16_hi(xv.y), s);
                        s = fmaf(wv[4], bf16_lo(xv.z), s);
                        s = fmaf(wv[5], bf16_hi(xv.z), s);
                        s = fmaf(wv[6], bf16_lo(xv.w), s);
                        s = fmaf(wv[7], bf16_hi(xv.w), s);
                        ca[b] = s;
                    }
                } else {
                    for (uint32_t k = 0; k < 8; ++k) {
                        const uint64_t o = ob + k;
                        if (o < o0 || o >= o1) continue;
                        const uint64_t r = o / cols;
                        const uint64_t c = o - r * cols;
                        const float wf = __uint_as_float(static_cast<uint32_t>(join1(sh.stage[si + k], a.sm[o])) << 16);
#pragma unroll
                        for (int b = 0; b < B; ++b) {
                            const float xf = __uint_as_float(static_cast<uint32_t>(g.x[b * cols + c]) << 16);
                            if (r == ra)
                                ca[b] = fmaf(wf, xf, ca[b]);
                            else {
                                cb[b] = fmaf(wf, xf, cb[b]);
                            }
                        }
                        if (r != ra) rb = r;
                    }
                }
            }
            for (uint64_t rr = r_lo; rr <= r_hi; ++rr) {
                if (rr != cur) {
                    warp_flush<B>(acc, part + static_cast<size_t>(warp) * g.rows_per_warp * B,
                                  static_cast<uint32_t>(cur - row0), lane);
                    cur = rr;
                }
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (ra == rr) acc[b] += ca[b];
                    if (rb == rr) acc[b] += cb[b];
                }
            }
        }
        if (s_begin < s_end) {
            warp_flush<B>(acc, part + static_cast<size_t>(warp) * g.rows_per_warp * B,
                          static_cast<uint32_t>(cur - row0), lane);
            nrows = static_cast<uint32_t>(cur - row0 + 1);
        }
        if (lane == 0) {
            warp_row0[warp] = row0;
            warp_nrows[warp] = nrows;
        }
        __syncthreads();

        // combine warps in order; whole rows to y, partial rows to the workspace
        const uint64_t r_first = o0 / cols, r_last = (o1 - 1) / cols;
        const uint64_t nr = r_last - r_first + 1;
        for (uint64_t i = threadIdx.x; i < nr * B; i += kThreads) {
            const uint64_t r = r_first + i / B;
            const int b = static_cast<int>(i % B);
            float s = 0.f;
            for (int w = 0; w < kWarps; ++w) {
                if (warp_nrows[w] && r >= warp_row0[w] && r < warp_row0[w] + warp_nrows[w])
                    s += part[(static_cast<size_t>(w) * g.rows_per_warp + (r - warp_row0[w])) * B + b];
            }
            const bool whole = r * cols >= o0 && (r + 1) * cols <= o1;
            if (whole)
                g.y[static_cast<uint64_t>(b) * g.rows + r] = s;
            else {
                const int slot = (r == r_first) ? 0 : 1;
                g.ws[(tb * 2 + slot) * B + b] = s;
            }
        }
        __syncthreads();
    }
}

// Rows split across tiles: the tile in which a row starts adds its own tail
// partial and the head partials of the following tiles, in tile order.
template <int B>
__global__ void gemv_fixup_kernel(const uint64_t* __restrict__ block_index, uint64_t n_blocks, GemvArgs g) {
    const uint64_t t = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x;
    if (t >= n_blocks) return;
    const uint64_t cols = g.cols;
    const uint64_t n = static_cast<uint64_t>(g.rows) * cols;
    const uint64_t o0 = block_index[t], o1 = block_index[t + 1];
    if (o1 <= o0 || o1 > n) return;  // empty, or a corrupt index the main kernel already flagged
    const uint64_t r_first = o0 / cols, r_last = (o1 - 1) / cols;
    const uint64_t row_start = r_last * cols, row_end = row_start + cols;
    if (row_start < o0 || row_end <= o1) return;  // not started here, or wholly inside
    float s[kMaxBatch];
    const int slot = (r_last == r_first) ? 0 : 1;
#pragma unroll
    for (int b = 0; b < B; ++b) s[b] = g.ws[(t * 2 + slot) * B + b];
    for (uint64_t u = t + 1; u < n_blocks; ++u) {
        const uint64_t p0 = block_index[u], p1 = block_index[u + 1];
        if (p1 < p0 || p1 > n) break;
        if (p1 == p0) continue;
#pragma unroll
        for (int b = 0; b < B; ++b) s[b] += g.ws[(u * 2 + 0) * B + b];
        if (p1 >= row_end) break;
    }
#pragma unroll
    for (int b = 0; b < B; ++b) g.y[static_cast<uint64_t>(b) * g.rows + r_last] = s[b];
}

// All weights share one exponent: one warp per row, fixed-order reduction.
template <int B>
__global__ void fill_gemv_kernel(const uint8_t* __restrict__ sm, const uint64_t* __restrict__ block_index,
                                 uint32_t fill, GemvArgs g, int32_t* status) {
    const int lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0 && block_index[0] != static_cast<uint64_t>(g.rows) * g.cols)
        raise_status(status, AFX_DEV_BAD_BLOCK);
    const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
    for (uint64_t r = blockIdx.x * static_cast<uint64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < g.rows;
         r += warps) {
        float acc[kMaxBatch] = {0.f, 0.f, 0.f, 0.f};
        for (uint64_t c = lane; c < g.cols; c += 32) {
            const uint64_t o = r * g.cols + c;
            const float wf = __uint_as_float(static_cast<uint32_t>(join1(fill, sm[o])) << 16);
#pragma unroll
            for (int b = 0; b < B; ++b)
                acc[b] = fmaf(wf, __uint_as_float(static_cast<uint32_t>(g.x[b * g.cols + c]) << 16), acc[b]);
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = acc[b];
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
            if (lane == 0) g.y[static_cast<uint64_t>(b) * g.rows + r] = v;
        }
    }
}

// ---- host launch helpers -----------------------------------------------------

void make_tables(const afx_desc& d, CodeTables& t) {
    std::memset(&t, 0, sizeof t);
    unsigned count[AFX_MAX_CODE_LEN + 1] = {0};
    for (int s = 0; s < 256; ++s)
        if (d.len[s]) ++count[d.len[s]];
    unsigned pos = 0;
    uint32_t first = 0;
    for (int L = 1; L <= AFX_MAX_CODE_LEN; ++L) {
        if (L > 1) first = (first + count[L - 1]) << 1;
        // symbols of length L in value order
        const unsigned first_pos = pos;
        for (int s = 0; s < 256; ++s)
            if (d.len[s] == L) t.sorted[pos++] = static_cast<uint8_t>(s);
        t.limit[L] = (first + count[L]) << (AFX_MAX_CODE_LEN - L);
        t.base[L] = static_cast<int32_t>(first_pos) - static_cast<int32_t>(first);
    }
}

size_t stream_stage_bytes(uint32_t T) { return static_cast<size_t>(kThreads) * T + 16; }
size_t tile_shared_bytes() { return (sizeof(TileShared) + 15) & ~size_t(15); }

std::mutex g_mutex;

// Per device: SM count, the kernels whose dynamic shared-memory limit has
// been raised, and per (kernel, dynamic shared bytes) the number of resident
// CTAs per SM.  The limit is a property of the kernel, so it is raised once
// per device to the device's opt-in maximum and never lowered; occupancy is
// queried once per launch size.
constexpr int kMaxDevices = 64;
constexpr int kCacheSlots = 64;
constexpr int kFuncSlots = 16;
struct OccupancySlot {
    const void* func;
    size_t smem;
    int per_sm;
};
struct DeviceCache {
    int sms = 0;
    int n_funcs = 0;
    const void* funcs[kFuncSlots];
    int used = 0;
    OccupancySlot slot[kCacheSlots];
};
DeviceCache g_devices[kMaxDevices];

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

afx_status prepare_kernel(const void* func, size_t smem, int* blocks_per_sm) {
    const int dev = current_device();
    if (dev < 0) return afx_fail(AFX_E_CUDA, "no current CUDA device", 0);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceCache& dc = g_devices[dev];
    for (int i = 0; i < dc.used; ++i)
        if (dc.slot[i].func == func && dc.slot[i].smem == smem) {
            *blocks_per_sm = dc.slot[i].per_sm;
            return AFX_OK;
        }
    bool raised = false;
    for (int i = 0; i < dc.n_funcs; ++i) raised = raised || dc.funcs[i] == func;
    if (!raised) {
        int optin = 0;
        AFX_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
                     "cudaDeviceGetAttribute");
        AFX_CUDA_TRY(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, optin),
                     "cudaFuncSetAttribute");
        if (dc.n_funcs < kFuncSlots) dc.funcs[dc.n_funcs++] = func;
    }
    AFX_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, func, kThreads, smem),
                 "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (*blocks_per_sm < 1) return afx_fail(AFX_E_CUDA, "kernel does not fit on an SM", 0);
    if (dc.used < kCacheSlots) dc.slot[dc.used++] = {func, smem, *blocks_per_sm};
    return AFX_OK;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_devices[dev].sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_devices[dev].sms = sms;
    }
    return g_devices[dev].sms;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

afx_status make_decode_args(const afx_desc& d, const void* container, int32_t* status, DecodeArgs& a) {
    const uint8_t* base = static_cast<const uint8_t*>(container);
    a.exp_words = reinterpret_cast<const uint32_t*>(base + d.off_exp);
    a.sm = base + d.off_sm;
    a.chunk_index = reinterpret_cast<const uint16_t*>(base + d.off_chunk);
    a.block_index = reinterpret_cast<const uint64_t*>(base + d.off_block);
    a.n = d.n;
    a.n_chunks = d.n_chunks;
    a.n_blocks = d.n_blocks;
    a.exp_bytes = d.exp_bytes;
    a.chunk_bytes = d.chunk_bytes;
    a.status = status;
    return AFX_OK;
}

}  // namespace afx

using namespace afx;

extern "C" afx_status afx_decode(const afx_desc* desc, const void* container, uint16_t* out, afx_stream_t stream,
                                 int32_t* status) {
    if (!desc || (!container && desc->n) || (!out && desc->n)) return AFX_E_ARG;
    afx_status st = afx_check_desc(desc);
    if (st != AFX_OK) return st;
    if (desc->n == 0) return AFX_OK;
    if (!aligned(container, 16) || !aligned(out, 16)) return AFX_E_ARG;
    if (desc->nsym >= 2 && desc->block_chunks != static_cast<uint32_t>(kThreads)) return AFX_E_ARG;
    const int sms = sm_count();
    if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* base = static_cast<const uint8_t*>(container);

    if (desc->nsym == 1) {
        const uint64_t groups = (desc->n + 7) / 8;
        const uint64_t blocks = std::min<uint64_t>((groups + 255) / 256, static_cast<uint64_t>(sms) * 8);
        fill_store_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            base + desc->off_sm, reinterpret_cast<const uint64_t*>(base + desc->off_block), desc->fill, desc->n, out,
            status);
        AFX_CUDA_TRY(cudaGetLastError(), "fill_store_kernel launch");
        return AFX_OK;
    }
    DecodeArgs a;
    make_decode_args(*desc, container, status, a);
    CodeTables tab;
    make_tables(*desc, tab);
    const size_t smem = tile_shared_bytes() + stream_stage_bytes(desc->chunk_bytes);
    int per_sm = 0;
    st = prepare_kernel(reinterpret_cast<const void*>(decode_store_kernel), smem, &per_sm);
    if (st != AFX_OK) return st;
    const uint64_t grid = std::min<uint64_t>(desc->n_blocks, static_cast<uint64_t>(sms) * per_sm);
    StoreArgs sa{out};
    decode_store_kernel<<<static_cast<unsigned>(grid), kThreads, smem, s>>>(a, tab, sa);
    AFX_CUDA_TRY(cudaGetLastError(), "decode_store_kernel launch");
    return AFX_OK;
}

namespace {

template <int B>
afx_status launch_gemv(const afx_desc& d, const void* container, const GemvArgs& g, cudaStream_t s,
                       int32_t* status, int sms) {
    const uint8_t* base = static_cast<const uint8_t*>(container);
    if (d.nsym == 1) {
        const uint64_t blocks = std::min<uint64_t>((g.rows + 7) / 8, static_cast<uint64_t>(sms) * 8);
        fill_gemv_kernel<B><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            base + d.off_sm, reinterpret_cast<const uint64_t*>(base + d.off_block), d.fill, g, status);
        AFX_CUDA_TRY(cudaGetLastError(), "fill_gemv_kernel launch");
        return AFX_OK;
    }
    DecodeArgs a;
    make_decode_args(d, container, status, a);
    CodeTables tab;
    make_tables(d, tab);
    const size_t part_bytes = static_cast<size_t>(kWarps) * g.rows_per_warp * B * sizeof(float);
    const size_t smem = tile_shared_bytes() + stream_stage_bytes(d.chunk_bytes) + part_bytes +
                        kWarps * (sizeof(uint64_t) + sizeof(uint32_t));
    if (smem > 227 * 1024) return afx_fail(AFX_E_ARG, "GEMV shape needs too much shared memory", 0);
    int per_sm = 0;
    const afx_status st = prepare_kernel(reinterpret_cast<const void*>(decode_gemv_kernel<B>), smem, &per_sm);
    if (st != AFX_OK) return st;
    const uint64_t grid = std::min<uint64_t>(d.n_blocks, static_cast<uint64_t>(sms) * per_sm);
    decode_gemv_kernel<B><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(a, tab, g);
    AFX_CUDA_TRY(cudaGetLastError(), "decode_gemv_kernel launch");
    const unsigned fix_blocks = static_cast<unsigned>((d.n_blocks + 127) / 128);
    gemv_fixup_kernel<B><<<fix_blocks, 128, 0, s>>>(a.block_index, d.n_blocks, g);
    AFX_CUDA_TRY(cudaGetLastError(), "gemv_fixup_kernel launch");
    return AFX_OK;
}

}  // namespace

extern "C" afx_status afx_decode_gemv(const afx_desc* desc, const void* container, uint32_t rows, uint32_t cols,
                                      const uint16_t* x, uint32_t batch, float* y, void* workspace,
                                      uint64_t workspace_bytes, afx_stream_t stream, int32_t* status) {
    if (!desc || !container || !x || !y) return AFX_E_ARG;
    afx_status st = afx_check_desc(desc);
    if (st != AFX_OK) return st;
    if (batch < 1 || batch > static_cast<uint32_t>(kMaxBatch)) return AFX_E_ARG;
    if (rows == 0 || cols < 64 || static_cast<uint64_t>(rows) * cols != desc->n) return AFX_E_ARG;
    if (!aligned(container, 16) || !aligned(x, 16)) return AFX_E_ARG;
    if (desc->nsym >= 2 && desc->block_chunks != static_cast<uint32_t>(kThreads)) return AFX_E_ARG;
    if (desc->nsym >= 2) {
        if (!workspace || !aligned(workspace, 16)) return AFX_E_ARG;
        if (workspace_bytes < afx_gemv_workspace_bytes(desc->n_blocks, batch)) return AFX_E_NOSPACE;
    }
    const int sms = sm_count();
    if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
    GemvArgs g;
    g.x = x;
    g.y = y;
    g.ws = static_cast<float*>(workspace);
    g.rows = rows;
    g.cols = cols;
    g.batch = batch;
    // rows a warp slice can meet: slice <= (capacity + 16) / 8 / warps + 1 groups
    const uint64_t slice_elems = ((AFX_BLOCK_CAPACITY + 16) / 8 / kWarps + 2) * 8;
    g.rows_per_warp = static_cast<uint32_t>(slice_elems / cols + 2);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (batch) {
        case 1: return launch_gemv<1>(*desc, container, g, s, status, sms);
        case 2: return launch_gemv<2>(*desc, container, g, s, status, sms);
        case 3: return launch_gemv<3>(*desc, container, g, s, status, sms);
        default: return launch_gemv<4>(*desc, container, g, s, status, sms);
    }
}
