// sm_103a kernels of afx: restore BF16 weights from the exponent-coded
// container, alone (afx_decode, afx_decode_batch) or fused into a batch-1..4
// GEMV (afx_decode_gemv, afx_decode_gemv_batch).
//
// The operation: "Why Weight Offloading Slows Inference", section
// "Lossless compression: fewer bytes to read, more work to unpack" -- every
// weight's exponent was stored with a shorter code for common values, its
// sign and mantissa raw; the released bits are restored before compute.
// This is the t_unpack term of that page's Eq. (1).
//
// Work decomposition.  One launch restores a list of tensors.  A tile is
// one block of a container (512 chunks of 8*T stream bits); the tiles of
// all tensors form one list, and each persistent CTA takes a contiguous
// run of it, so it meets at most a few tensors.  For each tile:
//   1. the tile's stream words, chunk entries and block-index pair arrive in
//      shared memory by cp.async, issued one tile ahead (double buffer); the
//      tile's sign|mantissa bytes are prefetched into L2 in one bulk request;
//   2. each thread takes one chunk: the index gives the bit offset of its
//      first codeword and how many codewords start in it; a warp-shuffle
//      plus block prefix scan of those counts places every thread's run of
//      exponents inside the tile;
//   3. each thread decodes its run from a 64-bit window of stream words
//      through two tables rebuilt in shared memory whenever the tensor
//      changes: a 4096-entry table that, from a 12-bit peek, yields up to
//      three whole codes (their exponents and total length), and a
//      4096-entry table of the first code's length for single steps; codes
//      longer than 12 bits fall back to a per-length canonical search.
//      Exponents are packed four to a word and stored as aligned words;
//   4. the whole CTA joins exponents with sign|mantissa bytes in aligned
//      groups of 8 weights: 8-byte coalesced loads and 16-byte coalesced
//      BF16 stores (or, fused, 8 products per batch row, and the weights
//      never reach global memory).
// Every value read from the container is checked before it addresses
// memory; a bad one sets a status bit and the tile is skipped.  The kernels
// wait only on __syncthreads and cp.async groups.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "afx_internal.h"
#include "afx_warp_decode.cuh"

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

// ---- epilogues ---------------------------------------------------------------------

// c + a * b with BF16 multiplicands and a float32 accumulator, rounded once
// (the BF16 values convert to float32 exactly, so this equals fmaf on the
// converted values): the multiply-adds take the BF16 bit patterns as they
// are, with no conversion instructions.  fma_bf16: a and b in the low 16
// bits; fma_bf16x2: the two halves of a and b, low half first.
__device__ __forceinline__ float fma_bf16(uint32_t a, uint32_t b, float c) {
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, al, bl, %0;\n}\n"
        : "+f"(c)
        : "r"(a), "r"(b));
    return c;
}

__device__ __forceinline__ float fma_bf16x2(uint32_t a, uint32_t b, float c) {
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
        " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %0, ah, bh, %0;\n}\n"
        : "+f"(c)
        : "r"(a), "r"(b));
    return c;
}

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

// y[b][r] = sum_c W[r][c] x[b][c] for the rows this tile meets.  Warp w
// takes a contiguous slice of 8-weight groups, keeps float32 sums for its
// current row and, when the row changes, reduces them with a fixed
// butterfly into one partial per (warp, row).  Rows are then summed over
// warps in warp order: rows wholly inside the tile go to y, the first and
// last (partial) rows to the workspace, which gemv_fixup_kernel adds across
// tiles in tile order.  Every sum has a fixed order: y is reproducible.
template <int B>
__device__ __forceinline__ void gemv_tile(const Shared& sh, const TensorArgs& t, uint64_t tile, uint64_t o0, uint64_t o1,
                          float* part, uint64_t* warp_row0, uint32_t* warp_nrows) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t cols = t.cols;
    const bool vec_x = (cols & 7u) == 0;
    const uint64_t ob0 = o0 & ~uint64_t(7);
    const uint64_t g0 = o0 >> 3, g1 = (o1 + 7) >> 3;
    const uint64_t ng = g1 - g0;
    const uint64_t s_begin = g0 + ng * warp / kWarps, s_end = g0 + ng * (warp + 1) / kWarps;
    float* wpart = part + static_cast<size_t>(warp) * t.rows_per_warp * B;

    uint64_t cur = 0, row0 = 0;
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
                const uint2 s8 = __ldg(reinterpret_cast<const uint2*>(t.sm + ob));
                const uint4 wv4 = join8(e8, s8);
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(t.x + b * cols + c0));
                    float s = fma_bf16x2(wv4.x, xv.x, 0.f);
                    s = fma_bf16x2(wv4.y, xv.y, s);
                    s = fma_bf16x2(wv4.z, xv.z, s);
                    s = fma_bf16x2(wv4.w, xv.w, s);
                    ca[b] = s;
                }
            } else {
                for (uint32_t q = 0; q < 8; ++q) {
                    const uint64_t o = ob + q;
                    if (o < o0 || o >= o1) continue;
                    const uint64_t r = o / cols;
                    const uint64_t c = o - r * cols;
                    const uint32_t wb = join1(sh.stage[si + q], t.sm[o]);
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        const uint32_t xb = t.x[b * cols + c];
                        if (r == ra)
                            ca[b] = fma_bf16(wb, xb, ca[b]);
                        else
                            cb[b] = fma_bf16(wb, xb, cb[b]);
                    }
                    if (r != ra) rb = r;
                }
            }
        }
        for (uint64_t rr = r_lo; rr <= r_hi; ++rr) {
            if (rr != cur) {
                warp_flush<B>(acc, wpart, static_cast<uint32_t>(cur - row0), lane);
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
        warp_flush<B>(acc, wpart, static_cast<uint32_t>(cur - row0), lane);
        nrows = static_cast<uint32_t>(cur - row0 + 1);
    }
    if (lane == 0) {
        warp_row0[warp] = row0;
        warp_nrows[warp] = nrows;
    }
    __syncthreads();

    const uint64_t r_first = o0 / cols, r_last = (o1 - 1) / cols;
    const uint64_t nr = r_last - r_first + 1;
    for (uint64_t i = threadIdx.x; i < nr * B; i += kThreads) {
        const uint64_t r = r_first + i / B;
        const int b = static_cast<int>(i % B);
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            if (warp_nrows[w] && r >= warp_row0[w] && r < warp_row0[w] + warp_nrows[w])
                s += part[(static_cast<size_t>(w) * t.rows_per_warp + (r - warp_row0[w])) * B + b];
        }
        const bool whole = r * cols >= o0 && (r + 1) * cols <= o1;
        if (whole)
            t.y[static_cast<uint64_t>(b) * t.rows + r] = s;
        else
            t.ws[(tile * 2 + (r == r_first ? 0 : 1)) * B + b] = s;
    }
}

// ---- the fused GEMV kernel ---------------------------------------------------------
//
// B in 1..4 activation rows; whole blocks per CTA tile.
template <int B>
__global__ void __launch_bounds__(kThreads, 2) restore_kernel(const __grid_constant__ LaunchArgs a) {
    static_assert(B >= 1 && B <= kMaxBatch, "restore_kernel is the fused GEMV path");
    extern __shared__ __align__(16) uint8_t smem[];
    Shared& sh = *reinterpret_cast<Shared*>(smem);
    uint8_t* stream_base = smem + shared_fixed_bytes();
    const uint32_t stream_stride = kThreads * a.max_chunk_bytes + kStreamPad;
    float* part = reinterpret_cast<float*>(stream_base + 2 * static_cast<size_t>(stream_stride));
    uint64_t* warp_row0 = reinterpret_cast<uint64_t*>(part + (B ? kWarps * a.max_rows_per_warp * B : 0));
    uint32_t* warp_nrows = reinterpret_cast<uint32_t*>(warp_row0 + kWarps);

    const uint64_t g_begin = a.total_tiles * blockIdx.x / gridDim.x;
    const uint64_t g_end = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
    if (g_begin >= g_end) return;

    uint32_t k = 0;  // tensor of the current tile
    while (k + 1 < a.count && g_begin >= a.t[k + 1].tile_begin) ++k;
    uint32_t kn = k;  // tensor of the next tile to issue
    int built = -1;
    issue_tile(sh, stream_base, stream_stride, a.t[k], g_begin - a.t[k].tile_begin, 0);
    int buf = 0;
    for (uint64_t g = g_begin; g < g_end; ++g) {
        if (g + 1 < g_end) {
            while (kn + 1 < a.count && g + 1 >= a.t[kn + 1].tile_begin) ++kn;
            issue_tile(sh, stream_base, stream_stride, a.t[kn], g + 1 - a.t[kn].tile_begin, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        while (k + 1 < a.count && g >= a.t[k + 1].tile_begin) ++k;
        const TensorArgs& t = a.t[k];
        __syncthreads();  // the staged tile is visible; the previous tile is done
        if (built != static_cast<int>(k)) {
            build_tables(sh, reinterpret_cast<uint16_t*>(sh.stage), t.tab);
            built = static_cast<int>(k);
        }
        const uint64_t b = g - t.tile_begin;
        uint64_t o0, o1;
        const uint32_t* stream =
            reinterpret_cast<const uint32_t*>(stream_base + static_cast<size_t>(buf) * stream_stride);
        if (decode_tile(sh, stream, t, b, buf, a.status, o0, o1) && o0 < o1) {
            gemv_tile<B>(sh, t, b, o0, o1, part, warp_row0, warp_nrows);
        }
        buf ^= 1;
    }
}

// Joins and stores `count` weights from o0 with the 32 lanes of a warp; the
// rotated exponent of weight o is at stage[o - (o0 & ~7)].  The first and
// last group of 8 may be shared with neighbouring ranges and go out weight
// by weight (lanes 0-7 and 8-15); the full groups between go out as 16-byte
// stores, one group per lane at a time.
__device__ __forceinline__ void warp_store(const uint8_t* stage, const uint8_t* sm, uint16_t* out, uint64_t o0,
                                           uint32_t count, int lane) {
    const uint64_t ob0 = o0 & ~uint64_t(7);
    const uint8_t* smb = sm + ob0;
    uint16_t* outb = out + ob0;
    const uint32_t a = static_cast<uint32_t>(o0) & 7u, b = a + count;  // the range, relative to ob0
    const uint32_t f0 = (a + 7) & ~7u, f1 = b & ~7u;                  // full groups [f0, f1)
    if (lane < 16) {
        const uint32_t r = lane < 8 ? lane : f1 + (lane & 7);
        const bool same_group = lane >= 8 && f1 == 0;  // the last group is the first one
        if (r >= a && r < b && (r < f0 || r >= f1) && !same_group) outb[r] = join1(stage[r], smb[r]);
    }
    if (f1 > f0) {
        const uint32_t nfull = (f1 - f0) >> 3;
        const uint2* smp = reinterpret_cast<const uint2*>(smb + f0);
        const uint2* stp = reinterpret_cast<const uint2*>(stage + f0);
        uint4* outp = reinterpret_cast<uint4*>(outb + f0);
        for (uint32_t j = lane; j < nfull; j += 32) __stcs(outp + j, join8(stp[j], __ldg(smp + j)));
    }
}

// The 8 weights of group w times x[b][c .. c + 8) added into acc[b], for
// every b (x[b][c] at x + b * cols + c; B * cols < 2^31 on this path).
template <int B>
__device__ __forceinline__ void gemv_group(const uint4& w, const uint16_t* x, uint32_t cols, uint32_t c,
                                           float (&acc)[B]) {
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + (b * cols + c)));
        float d = fma_bf16x2(w.x, xv.x, acc[b]);
        d = fma_bf16x2(w.y, xv.y, d);
        d = fma_bf16x2(w.z, xv.z, d);
        acc[b] = fma_bf16x2(w.w, xv.w, d);
    }
}

// Sums the V values v[0 .. V) (V a power of two, at most 32) over the 32
// lanes with one transposed butterfly: in each of the first log2(V) steps a
// lane keeps one half of its values and adds the half its partner sends
// for them, so that afterwards lane L holds a partial of value
// L >> (5 - log2 V) only; the remaining steps complete that sum.  Returns
// it; every lane gets the sum of its value.
template <int V>
__device__ __forceinline__ float warp_sum_transposed(float (&v)[V], int lane) {
    int m = 16;
#pragma unroll
    for (int c = V; c > 1; c >>= 1, m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < c / 2; ++k) {
            const float send = upper ? v[k] : v[k + c / 2];
            const float keep = upper ? v[k + c / 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
        }
    }
    float r = v[0];
#pragma unroll
    for (; m >= 1; m >>= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, m);
    return r;
}

// y[b][r] += sum over the weights [o0, o0 + count) of row r of W[r][c] x[b][c],
// for a matrix whose rows are at least kWarpStage weights long and a
// multiple of 8: a sub-tile meets at most two rows (r_a and r_a + 1) and no
// group of 8 straddles two rows.  Each lane keeps float32 sums for the two
// rows (the full groups of row r_a first, then those of row r_a + 1); one
// transposed butterfly reduces all 2B of them, and the workspace gets the
// sub-tile's start and its two row partials (zeros when the sub-tile is not
// valid).  gemv_fixup_warp_kernel adds each row's partials in sub-tile
// order, so y does not depend on how the grid split the work.
template <int B>
__device__ __forceinline__ void warp_gemv(const uint8_t* stage, const TensorArgs& t, uint64_t s, uint64_t o0,
                                          uint32_t count, bool ok, int lane) {
    float acc_a[B], acc_b[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc_a[b] = acc_b[b] = 0.f;
    if (ok && count) {
        const uint64_t cols = t.cols;
        const uint64_t ra = o0 / cols;
        const uint64_t ob0 = o0 & ~uint64_t(7);
        const uint32_t a = static_cast<uint32_t>(o0) & 7u, e = a + count;  // the range, relative to ob0
        const uint64_t next_row = (ra + 1) * cols;
        const uint32_t split = next_row - ob0 < e ? static_cast<uint32_t>(next_row - ob0) : e;  // row r_a + 1 from here
        const uint32_t cbase = static_cast<uint32_t>(ob0 - ra * cols);  // column of relative index 0 in row r_a
        const uint8_t* smb = t.sm + ob0;
        const uint16_t* x = t.x;
        const uint32_t cols32 = static_cast<uint32_t>(cols);
        const uint32_t f0 = (a + 7) & ~7u, f1 = e & ~7u;  // full groups [f0, f1)
        if (lane < 16) {  // weights outside the full groups, one per lane
            const uint32_t r = lane < 8 ? lane : f1 + (lane & 7);
            const bool same_group = lane >= 8 && f1 == 0;
            if (r >= a && r < e && (r < f0 || r >= f1) && !same_group) {
                const uint32_t w = join1(stage[r], smb[r]);
                const bool in_b = r >= split;
                const uint32_t c = in_b ? r - split : cbase + r;
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const uint32_t xb = __ldg(x + (b * cols32 + c));
                    if (in_b)
                        acc_b[b] = fma_bf16(w, xb, acc_b[b]);
                    else
                        acc_a[b] = fma_bf16(w, xb, acc_a[b]);
                }
            }
        }
        // full groups of row r_a: [f0, mid); of row r_a + 1: [mid, f1)
        const uint32_t mid = split < f1 ? (split > f0 ? split : f0) : f1;
        for (uint32_t r = f0 + 8 * lane; r < mid; r += 8 * 32)
            gemv_group<B>(join8(*reinterpret_cast<const uint2*>(stage + r), __ldg(reinterpret_cast<const uint2*>(smb + r))),
                          x, cols32, cbase + r, acc_a);
        for (uint32_t r = mid + 8 * lane; r < f1; r += 8 * 32)
            gemv_group<B>(join8(*reinterpret_cast<const uint2*>(stage + r), __ldg(reinterpret_cast<const uint2*>(smb + r))),
                          x, cols32, r - split, acc_b);
    }
    constexpr int V = B == 1 ? 2 : B == 2 ? 4 : 8;  // 2B values, padded to a power of two
    float v[V];
#pragma unroll
    for (int j = 0; j < V; ++j) v[j] = j < B ? acc_a[j] : j < 2 * B ? acc_b[j - B] : 0.f;
    const float sum = warp_sum_transposed<V>(v, lane);
    // lane L holds value j = L / (32 / V): row r_a's batch j for j < B, row
    // r_a + 1's batch j - B for B <= j < 2B; part[s][2B] is laid out the same way
    constexpr int kLanesPerValue = 32 / V;
    const int j = lane / kLanesPerValue;
    uint64_t* ws_o0 = reinterpret_cast<uint64_t*>(t.ws);
    float* part = reinterpret_cast<float*>(ws_o0 + t.n_blocks * kSubtilesPerBlock);
    if (lane % kLanesPerValue == 0 && j < 2 * B) part[s * 2 * B + j] = sum;
    if (lane == 0) ws_o0[s] = o0;
}

// Joins and stores `count` E4M3 elements from o0 with the 32 lanes of a
// warp; the stage byte of element o is at stage[o - (o0 & ~7)] and its
// raw nibble in byte o / 2 of raw.  Groups of 16 elements (one 16-byte
// store, 8 raw bytes) start at multiples of 16; the first and last group may
// be shared with neighbouring ranges and go out byte by byte (lanes 0-15
// and 16-31), the full groups between one per lane at a time.
__device__ __forceinline__ void warp_store_e4m3(const uint8_t* stage, const uint8_t* raw, uint8_t* out, uint64_t o0,
                                                uint32_t count, int lane) {
    const uint64_t g0 = o0 & ~uint64_t(15);
    const uint32_t d = static_cast<uint32_t>((o0 & ~uint64_t(7)) - g0);  // stage index of g0 + i is i - d
    const uint8_t* rawg = raw + g0 / 2;
    uint8_t* outg = out + g0;
    const uint32_t a = static_cast<uint32_t>(o0 - g0), b = a + count;  // the range, relative to g0
    const uint32_t f0 = (a + 15) & ~15u, f1 = b & ~15u;              // full groups [f0, f1)
    const uint32_t r = lane < 16 ? static_cast<uint32_t>(lane) : f1 + static_cast<uint32_t>(lane - 16);
    const bool mine = lane < 16 ? (r >= a && r < b && r < f0) : (r >= f0 && r < b);
    if (mine) outg[r] = e4m3_join1(stage[r - d], rawg[r >> 1] >> ((r & 1u) * 4));
    for (uint32_t q = f0 + 16 * lane; q < f1; q += 16 * 32) {
        const uint2 ra = *reinterpret_cast<const uint2*>(stage + q - d);
        const uint2 rb = *reinterpret_cast<const uint2*>(stage + q - d + 8);
        __stcs(reinterpret_cast<uint4*>(outg + q), e4m3_join16(ra, rb, __ldg(reinterpret_cast<const uint2*>(rawg + q / 2))));
    }
}

// Joins and stores `count` FP16 elements from o0 with the 32 lanes of a
// warp, as warp_store does for BF16, with each group of 8 also taking its
// 8 hi-section nibbles (the aligned word at byte g / 2 for the group at
// element g).
__device__ __forceinline__ void warp_store_fp16(const uint8_t* stage, const uint8_t* sm, const uint8_t* hi,
                                                uint16_t* out, uint64_t o0, uint32_t count, int lane) {
    const uint64_t ob0 = o0 & ~uint64_t(7);
    const uint8_t* smb = sm + ob0;
    uint16_t* outb = out + ob0;
    const uint32_t a = static_cast<uint32_t>(o0) & 7u, b = a + count;  // the range, relative to ob0
    const uint32_t f0 = (a + 7) & ~7u, f1 = b & ~7u;                  // full groups [f0, f1)
    if (lane < 16) {
        const uint32_t r = lane < 8 ? lane : f1 + (lane & 7);
        const bool same_group = lane >= 8 && f1 == 0;  // the last group is the first one
        if (r >= a && r < b && (r < f0 || r >= f1) && !same_group)
            outb[r] = fp16_join1(stage[r], smb[r], fp16_hi3(hi, ob0 + r));
    }
    if (f1 > f0) {
        const uint32_t nfull = (f1 - f0) >> 3;
        const uint2* smp = reinterpret_cast<const uint2*>(smb + f0);
        const uint2* stp = reinterpret_cast<const uint2*>(stage + f0);
        uint4* outp = reinterpret_cast<uint4*>(outb + f0);
        const uint32_t* hg = reinterpret_cast<const uint32_t*>(hi) + ((ob0 + f0) >> 3);  // the first full group's nibbles
        for (uint32_t j = lane; j < nfull; j += 32) __stcs(outp + j, fp16_join8(stp[j], __ldg(smp + j), __ldg(hg + j)));
    }
}

// What warp_run does with a decoded sub-tile: store BF16, FP16 or E4M3
// elements, or the fused GEMV above.  kRaw: what the raw sections hold --
// a byte per element (BF16), a byte and 3 hi-section bits (FP16), or a
// nibble (E4M3).
constexpr int kRawBytes = 0, kRawBytesHi = 1, kRawNibbles = 2;
constexpr uint32_t kKindBF16 = 0, kKindFP16 = 1, kKindE4M3 = 2;

struct StoreEpilogue {
    static constexpr bool kSlots = false;  // the sub-tile index is not used
    static constexpr int kRaw = kRawBytes;
    __device__ __forceinline__ void operator()(const uint8_t* stage, const TensorArgs& t, uint64_t, uint64_t o0,
                                               uint32_t count, bool ok, int lane) const {
        if (ok && count) warp_store(stage, t.sm, static_cast<uint16_t*>(t.out), o0, count, lane);
    }
};

struct StoreFP16Epilogue {
    static constexpr bool kSlots = false;  // the sub-tile index is not used
    static constexpr int kRaw = kRawBytesHi;
    __device__ __forceinline__ void operator()(const uint8_t* stage, const TensorArgs& t, uint64_t, uint64_t o0,
                                               uint32_t count, bool ok, int lane) const {
        if (ok && count) warp_store_fp16(stage, t.sm, t.hi, static_cast<uint16_t*>(t.out), o0, count, lane);
    }
};

struct StoreE4M3Epilogue {
    static constexpr bool kSlots = false;  // the sub-tile index is not used
    static constexpr int kRaw = kRawNibbles;
    __device__ __forceinline__ void operator()(const uint8_t* stage, const TensorArgs& t, uint64_t, uint64_t o0,
                                               uint32_t count, bool ok, int lane) const {
        if (ok && count) warp_store_e4m3(stage, t.sm, static_cast<uint8_t*>(t.out), o0, count, lane);
    }
};

template <int B>
struct GemvEpilogue {
    static constexpr bool kSlots = true;  // one workspace slot per 32-chunk sub-tile index
    static constexpr int kRaw = kRawBytes;
    __device__ __forceinline__ void operator()(const uint8_t* stage, const TensorArgs& t, uint64_t s, uint64_t o0,
                                               uint32_t count, bool ok, int lane) const {
        warp_gemv<B>(stage, t, s, o0, count, ok, lane);
    }
    // Slot s holds no weights: its start o and zero partials.
    __device__ __forceinline__ void empty(const TensorArgs& t, uint64_t s, uint64_t o, int lane) const {
        uint64_t* ws_o0 = reinterpret_cast<uint64_t*>(t.ws);
        float* part = reinterpret_cast<float*>(ws_o0 + t.n_blocks * kSubtilesPerBlock);
        if (lane < 2 * B) part[s * 2 * B + lane] = 0.f;
        if (lane == 0) ws_o0[s] = o;
    }
};

// Restores sub-tiles [s0, s1) of tensor t with one warp.  phases holds the
// parity each of the warp's two copy barriers waits for next.  Returns false
// when a staging copy timed out (the run is abandoned and flagged).
// kPartial: the tensor's state table holds only its shallowest nodes.
template <bool host_src, bool kPartial, class Epi>
__device__ __forceinline__ bool warp_run(const TabView& tv, WarpSlot& ws, uint8_t* wstream, uint32_t wstride,
                                         const TensorArgs& t, uint64_t s0, uint64_t s1, int lane, int32_t* status,
                                         uint32_t wait_limit, bool stall, uint32_t& phases, const Epi& epi) {
    const uint32_t T = t.chunk_bytes;
    const uint32_t chunk_bits = 8u * T;
    const uint32_t sub_bytes = kWarpChunks * T, sub_bits = 8u * sub_bytes;
    const bool fsm = t.tab.fsm != 0;
    const uint32_t skip_row0 = t.tab.fsm_rows * kFsmRowBytes;
    const uint64_t n_sub = (t.n_chunks + kWarpChunks - 1) / kWarpChunks;
    const uint64_t n_full = t.n_sub_full;
    const uint8_t* const sm = t.sm;
    const uint64_t n = t.n;
    // the output index of sub-tile s0's first code
    const uint64_t blk = s0 / kSubtilesPerBlock;
    uint32_t pre = 0;
    for (uint64_t c = blk * kThreads + lane; c < s0 * kWarpChunks; c += 32) pre += __ldg(t.chunk_index + c) >> 5;
    pre = warp_sum(pre);
    uint64_t start = __ldg(t.block_index + blk) + pre;
    if (s0 == 0 && start != 0 && lane == 0) raise_status(status, AFX_DEV_BAD_BLOCK);
    // sources of the next sub-tile to stage
    const uint8_t* exp_src = reinterpret_cast<const uint8_t*>(t.exp_words) + s0 * sub_bytes;
    const uint16_t* chunk_src = t.chunk_index + s0 * kWarpChunks;
    if (!host_src && lane == 0) warp_issue_bulk(ws, wstream, t, s0, s0 < n_full, exp_src, chunk_src, sub_bytes, 0, stall);
    const uint32_t nrun = static_cast<uint32_t>(s1 - s0);
    uint32_t sub_in_block = static_cast<uint32_t>(s0 % kSubtilesPerBlock);
    int buf = 0;
    bool timed_out = false, next_issued = false;
    for (uint32_t r = 0; r < nrun; ++r) {
        const uint64_t s = s0 + r;
        if constexpr (host_src) {  // the link is the bound: stage this sub-tile now, synchronously
            warp_stage_host(ws, wstream + buf * wstride, t, s, s < n_full, exp_src, chunk_src, sub_bytes, buf, lane);
            exp_src += sub_bytes;
            chunk_src += kWarpChunks;
            __syncwarp();
        } else if (r + 1 < nrun) {
            exp_src += sub_bytes;
            chunk_src += kWarpChunks;
            if (lane == 0)
                warp_issue_bulk(ws, wstream + (buf ^ 1) * wstride, t, s + 1, s + 1 < n_full, exp_src, chunk_src,
                                sub_bytes, buf ^ 1, stall);
        }
        bool arrived = true;
        if constexpr (!host_src) {
            arrived = mbar_wait(&ws.bar[buf], (phases >> buf) & 1u, wait_limit);
            phases ^= 1u << buf;
        }
        if (!__all_sync(0xFFFFFFFFu, arrived)) {
            timed_out = true;  // handled after the loop
            next_issued = r + 1 < nrun;
            break;
        }
        if (r != 0 && sub_in_block == 0) {  // a block boundary inside the run
            const uint64_t bo = __ldg(t.block_index + s / kSubtilesPerBlock);
            if (bo != start) {
                if (lane == 0) raise_status(status, AFX_DEV_BAD_BLOCK);
                start = bo;
            }
        }
        // chunk entries that exist from this sub-tile's first (33 read at most)
        const bool full = s < n_full;
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
        // a corrupt block index can put start anywhere: o0 <= n keeps o1 from
        // wrapping past 2^64 back into [0, n]
        const uint64_t o0 = start, o1 = start + total;
        const bool in_range = o0 <= n && o1 <= n;
        if (lane == 0) {
            if (!in_range)
                raise_status(status, AFX_DEV_BAD_BLOCK);
            else if (o0 < o1 && !host_src) {  // the raw bytes are needed after the decode
                if constexpr (Epi::kRaw == kRawNibbles) {
                    const uint64_t a0 = (o0 >> 1) & ~uint64_t(15), a1 = (((o1 + 1) >> 1) + 15) & ~uint64_t(15);
                    prefetch_l2(sm + a0, static_cast<uint32_t>(a1 - a0));
                } else {
                    const uint64_t a0 = o0 & ~uint64_t(15), a1 = (o1 + 15) & ~uint64_t(15);
                    prefetch_l2(sm + a0, static_cast<uint32_t>(a1 - a0));
                    if constexpr (Epi::kRaw == kRawBytesHi) {  // and the hi section's nibbles of the range
                        const uint64_t h0 = (o0 >> 1) & ~uint64_t(15), h1 = (((o1 + 1) >> 1) + 15) & ~uint64_t(15);
                        prefetch_l2(t.hi + h0, static_cast<uint32_t>(h1 - h0));
                    }
                }
            }
        }
        const uint32_t next = static_cast<uint32_t>(lane) + 1 < nexist ? ws.chunk[buf][lane + 1] : 0u;
        const uint32_t* stream = reinterpret_cast<const uint32_t*>(wstream + static_cast<size_t>(buf) * wstride);
        const uint32_t chunk_end = (lane + 1) * chunk_bits;
        bool stepped = false;  // byte steps done, finish after the barrier
        FsmLane fl;
        if (cnt && in_range) {
            const uint32_t s_run = static_cast<uint32_t>(o0 & 7u) + (inc - cnt);
            if (fsm) {
                uint32_t stream_end = sub_bits;
                if (!full) {
                    const uint64_t bit0 = s * static_cast<uint64_t>(sub_bits);
                    const uint64_t left = t.total_bits > bit0 ? t.total_bits - bit0 : 0;
                    stream_end = left < sub_bits ? static_cast<uint32_t>(left) : sub_bits;
                }
                AFX_CHECK((lane + 1) * (T >> 2) <= wstride >> 2, kChkStreamWords);
                if (chunk_end <= stream_end) {
                    if constexpr (kPartial)
                        fsm_chunk_steps_esc(tv, stream, lane * (T >> 2), T, gap, skip_row0, ws.stage, s_run, fl);
                    else if (T % 16 == 0)  // 16-byte loads of the chunk's words
                        fsm_span_steps(tv, stream + lane * (T >> 2), T >> 2, gap, skip_row0, ws.stage, s_run, fl,
                                       kWarpStage);
                    else
                        fsm_chunk_steps(tv, stream + lane * (T >> 2), T >> 2, gap, skip_row0, ws.stage, s_run, fl);
                    stepped = true;
                } else {  // the stream's partial last chunk
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
            bad = fsm_chunk_finish<kPartial>(tv, stream, fl, cnt, chunk_end, next);
        }
        if (bad) raise_status(status, AFX_DEV_BAD_CHUNK);
        const bool any_bad = __any_sync(0xFFFFFFFFu, bad);
        __syncwarp();
        if (!any_bad && in_range) {
            AFX_CHECK((o0 & 7u) + total <= static_cast<uint64_t>(kWarpStage), kChkMergeStage);
            AFX_CHECK(o0 + total <= n, kChkMergeOutput);
        }
        epi(ws.stage, t, s, o0, total, !any_bad && in_range, lane);
        start = o1;
        buf ^= 1;
        sub_in_block = (sub_in_block + 1) & (kSubtilesPerBlock - 1);
        fence_proxy_async_smem();  // this buffer's reads come before the bulk copy that refills it
        __syncwarp();
    }
    if (timed_out) {
        // give up on this run and flag it; the copy already issued into the
        // other buffer is waited for (bounded).  The copy whose wait ran out
        // may still land: the caller reports that (AFX_DEV_UNDRAINED).  This
        // path stays this small on purpose: more code here changes how the
        // compiler assigns the warp loop's 64 registers, and the batch-4 GEMV
        // then runs 30 % slower.
        if (lane == 0) raise_status(status, AFX_DEV_TIMEOUT);
        if (next_issued) {
            mbar_wait(&ws.bar[buf ^ 1], (phases >> (buf ^ 1)) & 1u, wait_limit);
            phases ^= 1u << (buf ^ 1);
        }
        return false;
    }
    // a run that ends on a block boundary checks the block index there; the
    // last run checks that the codes and the block index both end at n
    if (lane == 0) {
        if (s1 < n_sub && s1 % kSubtilesPerBlock == 0) {
            if (__ldg(t.block_index + s1 / kSubtilesPerBlock) != start) raise_status(status, AFX_DEV_BAD_BLOCK);
        }
        if (s1 == n_sub && (start != n || __ldg(t.block_index + t.n_blocks) != n))
            raise_status(status, AFX_DEV_BAD_BLOCK);
    }
    return true;
}

// ---- two chunks a lane ------------------------------------------------------------
//
// The same restore with sub-tiles of 64 chunks: lane l steps chunks 2l and
// 2l + 1 as one span of 2T bytes, from the first chunk's gap to the code
// that crosses the second chunk's end.  The work done once a chunk (the gap
// skip, the code crossing the end) and once a sub-tile (staging, scan, the
// merge's ragged ends) is then spread over twice the weights; the
// container is the same.  A span needs the first entry's gap and the sum of
// the two counts: the second entry's gap is not read (a corrupt one cannot
// change the result) and its count is checked through the sum.  Each warp
// has one stream buffer: the next sub-tile's copy is issued as soon as the
// lanes have read this one, and lands while the warp merges.  The stage
// holds LaunchArgs::pair_stage bytes; a sub-tile whose codes do not fit in
// it with kPairStageSlack to spare is decoded and merged as two halves of
// 16 lanes.
constexpr int kPairChunks = 2 * kWarpChunks;                   // chunks per sub-tile
constexpr int kPairSubtilesPerBlock = kThreads / kPairChunks;  // 8
constexpr int kPairChunkStage = 72;                            // 65 entries staged (144 bytes)
// Stage bytes past a sub-tile's codes that its lanes may write: a lane's
// byte steps emit up to 2 * kMaxChunkCodes + 1 codes whatever its count
// says, and store whole words.
constexpr uint32_t kPairStageSlack = 2 * kMaxChunkCodes + 8;
// The smallest stage: a half's codes (16 spans) with the slack, the
// sub-tile's offset within its group of 8 and 16 spare bytes.
constexpr uint32_t kPairStageMin = (16 * 2 * kMaxChunkCodes + kPairStageSlack + 7 + 16 + 15) & ~15u;

struct PairSlot {
    alignas(16) uint16_t chunk[kPairChunkStage];
    uint64_t bar;  // completion of the copies into the stream buffer and chunk
    uint64_t unused;
};
static_assert(sizeof(PairSlot) % 16 == 0, "pair slots keep the stage 16-byte aligned");

// Shared memory of one warp: its slot, its stage, its stream buffer.
__host__ __device__ constexpr uint32_t pair_warp_bytes(uint32_t max_chunk_bytes, uint32_t stage) {
    return static_cast<uint32_t>(sizeof(PairSlot)) + stage + kPairChunks * max_chunk_bytes + kStreamPad;
}

// Bytes staged for sub-tile s: its stream bytes plus the pad, and its 72
// chunk entries, or what the sections hold of them.  Both are multiples of
// 16.  A full sub-tile has all of them: s < n_sub_full / 2, since sub-tile s
// is full exactly when the 32-chunk sub-tile 2s + 1 is.
__device__ __forceinline__ uint2 pair_tile_bytes(const TensorArgs& t, uint64_t s, bool full, uint32_t sub_bytes) {
    if (full) return make_uint2(sub_bytes + kStreamPad, kPairChunkStage * 2);
    const uint64_t byte0 = s * sub_bytes, want = sub_bytes + kStreamPad;
    const uint64_t avail = t.exp_bytes > byte0 ? t.exp_bytes - byte0 : 0;
    const uint64_t cb0 = s * kPairChunks * 2;
    const uint64_t csec = (t.n_chunks * 2 + 15) & ~uint64_t(15);
    const uint64_t cavail = csec > cb0 ? csec - cb0 : 0;
    return make_uint2(static_cast<uint32_t>(want < avail ? want : avail),
                      static_cast<uint32_t>(cavail < kPairChunkStage * 2 ? cavail : kPairChunkStage * 2));
}

__device__ __forceinline__ void pair_issue_bulk(PairSlot& ps, uint8_t* stream_dst, const TensorArgs& t, uint64_t s,
                                                bool full, uint32_t sub_bytes, bool stall) {
    const uint2 nb = pair_tile_bytes(t, s, full, sub_bytes);
    AFX_CHECK(nb.x <= sub_bytes + kStreamPad && nb.y <= kPairChunkStage * 2, kChkStagingBytes);
    mbar_expect_tx(&ps.bar, nb.x + nb.y);
    if (stall) return;  // failure injection: the bytes never come
    if (nb.x) bulk_copy_g2s(stream_dst, reinterpret_cast<const uint8_t*>(t.exp_words) + s * sub_bytes, nb.x, &ps.bar);
    if (nb.y) bulk_copy_g2s(ps.chunk, t.chunk_index + s * kPairChunks, nb.y, &ps.bar);
}

// Restores the 64-chunk sub-tiles [s0, s1) of tensor t with one warp
// (device-resident containers).  phase is the parity the warp's copy
// barrier waits for next.  Returns false when a staging copy timed out.
// The epilogue of sub-tile s gets index 2s for its first (or only) pass
// and 2s + 1 for its second: a GEMV keeps the workspace layout of 32-chunk
// sub-tiles, with an empty slot 2s + 1 (no weights, zero partials) when
// the sub-tile was merged whole.
template <class Epi>
__device__ __forceinline__ bool warp_run_pair(const TabView& tv, PairSlot& ps, uint8_t* stage, uint32_t stage_cap,
                                              uint8_t* wstream, const TensorArgs& t, uint64_t s0, uint64_t s1,
                                              int lane, int32_t* status, uint32_t wait_limit, bool stall,
                                              uint32_t& phase, const Epi& epi) {
    const uint32_t T = t.chunk_bytes;
    const uint32_t chunk_bits = 8u * T, span_words = T >> 1;
    const uint32_t sub_bytes = kPairChunks * T, sub_bits = 8u * sub_bytes;
    const bool fsm = t.tab.fsm != 0;
    const uint32_t skip_row0 = t.tab.fsm_rows * kFsmRowBytes;
    const uint64_t n_sub = (t.n_chunks + kPairChunks - 1) / kPairChunks;
    const uint64_t n_full = t.n_sub_full / 2;
    const uint8_t* const sm = t.sm;
    const uint64_t n = t.n;
    // the output index of sub-tile s0's first code
    const uint64_t blk = s0 / kPairSubtilesPerBlock;
    uint32_t pre = 0;
    for (uint64_t c = blk * kThreads + lane; c < s0 * kPairChunks; c += 32) pre += __ldg(t.chunk_index + c) >> 5;
    pre = warp_sum(pre);
    uint64_t start = __ldg(t.block_index + blk) + pre;
    if (s0 == 0 && start != 0 && lane == 0) raise_status(status, AFX_DEV_BAD_BLOCK);
    if (lane == 0) pair_issue_bulk(ps, wstream, t, s0, s0 < n_full, sub_bytes, stall);
    const uint32_t* stream = reinterpret_cast<const uint32_t*>(wstream);
    const uint32_t nrun = static_cast<uint32_t>(s1 - s0);
    uint32_t sub_in_block = static_cast<uint32_t>(s0 % kPairSubtilesPerBlock);
    for (uint32_t r = 0; r < nrun; ++r) {
        const uint64_t s = s0 + r;
        const bool arrived = mbar_wait(&ps.bar, phase, wait_limit);
        phase ^= 1u;
        if (!__all_sync(0xFFFFFFFFu, arrived)) {
            // the copy may still land: the caller reports that (AFX_DEV_UNDRAINED)
            if (lane == 0) raise_status(status, AFX_DEV_TIMEOUT);
            return false;
        }
        if (r != 0 && sub_in_block == 0) {  // a block boundary inside the run
            const uint64_t bo = __ldg(t.block_index + s / kPairSubtilesPerBlock);
            if (bo != start) {
                if (lane == 0) raise_status(status, AFX_DEV_BAD_BLOCK);
                start = bo;
            }
        }
        const bool full = s < n_full;
        const uint32_t nexist = full ? static_cast<uint32_t>(kPairChunkStage)
                                     : static_cast<uint32_t>(min(t.n_chunks - min(t.n_chunks, s * kPairChunks),
                                                                 uint64_t{kPairChunkStage}));
        const uint32_t ia = 2u * static_cast<uint32_t>(lane);
        const uint32_t ea = ia < nexist ? ps.chunk[ia] : 0u;
        const uint32_t eb = ia + 1 < nexist ? ps.chunk[ia + 1] : 0u;
        const uint32_t next = ia + 2 < nexist ? ps.chunk[ia + 2] : 0u;
        const uint32_t gap = ea & 31u;
        uint32_t cnt = (ea >> 5) + (eb >> 5);
        bool bad = false;
        if (gap > 23u || (ea >> 5) > chunk_bits - gap || (ea >> 5) > static_cast<uint32_t>(kMaxChunkCodes) ||
            (eb & 31u) > 23u || (eb >> 5) > chunk_bits - (eb & 31u) ||
            (eb >> 5) > static_cast<uint32_t>(kMaxChunkCodes)) {
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
        const uint32_t half = __shfl_sync(0xFFFFFFFFu, inc, 15);  // the codes of lanes 0..15
        // a corrupt block index can put start anywhere: start <= n keeps the
        // end from wrapping past 2^64 back into [0, n]
        const bool in_range = start <= n && start + total <= n;
        if (lane == 0) {
            const uint64_t o0 = start, o1 = start + total;
            if (!in_range)
                raise_status(status, AFX_DEV_BAD_BLOCK);
            else if (o0 < o1) {  // the raw bytes are needed after the decode
                if constexpr (Epi::kRaw == kRawNibbles) {
                    const uint64_t a0 = (o0 >> 1) & ~uint64_t(15), a1 = (((o1 + 1) >> 1) + 15) & ~uint64_t(15);
                    prefetch_l2(sm + a0, static_cast<uint32_t>(a1 - a0));
                } else {
                    const uint64_t a0 = o0 & ~uint64_t(15), a1 = (o1 + 15) & ~uint64_t(15);
                    prefetch_l2(sm + a0, static_cast<uint32_t>(a1 - a0));
                    if constexpr (Epi::kRaw == kRawBytesHi) {  // and the hi section's nibbles of the range
                        const uint64_t h0 = (o0 >> 1) & ~uint64_t(15), h1 = (((o1 + 1) >> 1) + 15) & ~uint64_t(15);
                        prefetch_l2(t.hi + h0, static_cast<uint32_t>(h1 - h0));
                    }
                }
            }
        }
        const bool split = (static_cast<uint32_t>(start) & 7u) + total + kPairStageSlack > stage_cap;
        for (uint32_t p = 0; p < 2u; ++p) {
            if (p && !split) break;
            const uint32_t before = p ? half : 0u;  // codes merged by the earlier pass
            bool lbad = bad, stepped = false;
            FsmLane fl;
            if ((!split || (static_cast<uint32_t>(lane) >> 4) == p) && cnt && in_range) {
                const uint32_t s_run = (static_cast<uint32_t>(start + before) & 7u) + (inc - cnt) - before;
                const uint32_t span_end = (static_cast<uint32_t>(lane) + 1u) * 2u * chunk_bits;
                AFX_CHECK(s_run + 2u * kMaxChunkCodes + 8u <= stage_cap, kChkStageRun);
                AFX_CHECK((lane + 1) * span_words <= (sub_bytes + kStreamPad) >> 2, kChkStreamWords);
                uint32_t stream_end = sub_bits;
                if (!full) {
                    const uint64_t bit0 = s * static_cast<uint64_t>(sub_bits);
                    const uint64_t left = t.total_bits > bit0 ? t.total_bits - bit0 : 0;
                    stream_end = left < sub_bits ? static_cast<uint32_t>(left) : sub_bits;
                }
                if (fsm) {
                    if (span_end <= stream_end) {
                        if (span_words % 4 == 0)
                            fsm_span_steps(tv, stream + lane * span_words, span_words, gap, skip_row0, stage, s_run,
                                           fl, stage_cap);
                        else  // 4-byte chunks: a span is two words
                            fsm_chunk_steps(tv, stream + lane * span_words, span_words, gap, skip_row0, stage, s_run,
                                            fl, stage_cap);
                        stepped = true;
                    } else {  // the stream's partial last chunk
                        lbad = decode_run_fsm(tv, stream, lane * span_words, gap, cnt, stage, s_run, next, span_end,
                                              stream_end);
                    }
                } else {
                    lbad = decode_run(tv, stream, pair_tile_bytes(t, s, full, sub_bytes).x >> 2, lane * span_words,
                                      gap, cnt, stage, s_run, next, span_end);
                }
            }
            __syncwarp();
            if (stepped) {
                AFX_CHECK(reinterpret_cast<uint8_t*>(fl.wout) + 4 <= stage + stage_cap, kChkStagePending);
                lbad = fsm_chunk_finish(tv, stream, fl, cnt, (static_cast<uint32_t>(lane) + 1u) * 2u * chunk_bits,
                                        next);
            }
            if (!split || p) {  // the last reads of this stream buffer: refill it
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && r + 1 < nrun) pair_issue_bulk(ps, wstream, t, s + 1, s + 1 < n_full, sub_bytes, stall);
            }
            if (lbad) raise_status(status, AFX_DEV_BAD_CHUNK);
            const bool ok = !__any_sync(0xFFFFFFFFu, lbad) && in_range;
            __syncwarp();
            const uint32_t ptotal = split ? (p ? total - half : half) : total;
            if (ok) {
                AFX_CHECK(((start + before) & 7u) + ptotal <= static_cast<uint64_t>(stage_cap), kChkMergeStage);
                AFX_CHECK(start + before + ptotal <= n, kChkMergeOutput);
            }
            // the pass's workspace slot (GEMV): 2s and 2s + 1, one per half;
            // a sub-tile merged whole leaves slot 2s + 1 empty at its end
            epi(stage, t, 2 * s + p, start + before, ptotal, ok, lane);
            if constexpr (Epi::kSlots) {
                if (!split) epi.empty(t, 2 * s + 1, start + total, lane);
            }
            __syncwarp();
        }
        start += total;
        sub_in_block = (sub_in_block + 1) & (kPairSubtilesPerBlock - 1);
    }
    // a run that ends on a block boundary checks the block index there; the
    // last run checks that the codes and the block index both end at n
    if (lane == 0) {
        if (s1 < n_sub && s1 % kPairSubtilesPerBlock == 0) {
            if (__ldg(t.block_index + s1 / kPairSubtilesPerBlock) != start) raise_status(status, AFX_DEV_BAD_BLOCK);
        }
        if (s1 == n_sub && (start != n || __ldg(t.block_index + t.n_blocks) != n))
            raise_status(status, AFX_DEV_BAD_BLOCK);
    }
    return true;
}

// One CTA per SM (up to 32 warps) sharing one copy of the decode tables.
// host_src: the containers are in pinned host memory.  kPartial: the
// launch holds the tensors whose state tables keep only their shallowest
// nodes (their own kernels, so that the escape checks and their registers
// stay out of every other launch).
template <bool host_src, bool kPartial, class Epi>
__device__ __forceinline__ void restore_warps(const LaunchArgs& a, const Epi& epi) {
    extern __shared__ __align__(16) uint8_t smem[];
    // a following restore launch of the same call may take each SM as soon
    // as this CTA leaves it (it touches other tensors; see launch_restore)
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    SharedW& sh = *reinterpret_cast<SharedW*>(smem);
    uint8_t* tabr = smem + sharedw_table_offset();
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    WarpSlot* slots = reinterpret_cast<WarpSlot*>(tabr + a.tab_bytes);
    uint8_t* stream_all = reinterpret_cast<uint8_t*>(slots + nwarps);
    const uint32_t wstride = kWarpChunks * a.max_chunk_bytes + kStreamPad;
    WarpSlot& ws = slots[warp];
    uint8_t* wstream = stream_all + static_cast<size_t>(warp) * 2 * wstride;
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
    tv.esc_base = ~0u;

    const uint64_t g_begin = a.total_tiles * blockIdx.x / gridDim.x;
    const uint64_t g_end = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
    if (g_begin >= g_end) return;
    if (lane == 0) {
        mbar_init(&ws.bar[0]);
        mbar_init(&ws.bar[1]);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    uint32_t phases = 0;  // parity each copy barrier of this warp waits for next
    const uint32_t wait_limit = a.wait_limit ? a.wait_limit : kWaitLimit;
    bool alive = true;    // false after a staging copy timed out
    for (uint32_t k = 0; k < a.count; ++k) {
        const TensorArgs& t = a.t[k];
        const uint64_t t0 = t.tile_begin, t1 = t.tile_begin + t.n_blocks;
        if (t1 <= g_begin) continue;
        if (t0 >= g_end) break;
        // this tensor's blocks in the CTA's run, as sub-tiles
        const uint64_t b0 = (g_begin > t0 ? g_begin : t0) - t0, b1 = (g_end < t1 ? g_end : t1) - t0;
        const uint64_t n_sub = (t.n_chunks + kWarpChunks - 1) / kWarpChunks;
        const uint64_t sb = b0 * kSubtilesPerBlock;
        const uint64_t se = b1 * kSubtilesPerBlock < n_sub ? b1 * kSubtilesPerBlock : n_sub;
        __syncthreads();  // every warp is done with the previous tensor's tables
        build_tables_w(sh, tabr, t.tab, threadIdx.x, nthreads, CtaSync{});  // ends with __syncthreads
        const uint64_t span = se - sb;
        const uint64_t s0 = sb + span * warp / nwarps, s1 = sb + span * (warp + 1) / nwarps;
        if (alive && s0 < s1) {
            if constexpr (kPartial) tv.esc_base = (t.tab.fsm_rows + kSkipRows) * kFsmRowBytes;
            alive = warp_run<host_src, kPartial>(tv, ws, wstream, wstride, t, s0, s1, lane, a.status, wait_limit,
                                                 a.stall != 0, phases, epi);
            // a staging wait ran out: its copy may still land in shared memory
            // after the CTA moves on (the failure injection issues no copies)
            if (!alive && !host_src && !a.stall && lane == 0) raise_status(a.status, AFX_DEV_UNDRAINED);
        }
    }
}

// restore_warps with two chunks a lane (device-resident containers).  The
// shared memory holds the tables, then per warp its PairSlot, its stage of
// LaunchArgs::pair_stage bytes and its stream buffer.
template <class Epi>
__device__ __forceinline__ void restore_warps_pair(const LaunchArgs& a, const Epi& epi) {
    extern __shared__ __align__(16) uint8_t smem[];
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    SharedW& sh = *reinterpret_cast<SharedW*>(smem);
    uint8_t* tabr = smem + sharedw_table_offset();
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* wbase = tabr + a.tab_bytes + static_cast<size_t>(warp) * pair_warp_bytes(a.max_chunk_bytes, a.pair_stage);
    PairSlot& ps = *reinterpret_cast<PairSlot*>(wbase);
    uint8_t* stage = wbase + sizeof(PairSlot);
    uint8_t* wstream = stage + a.pair_stage;
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
    tv.esc_base = ~0u;

    const uint64_t g_begin = a.total_tiles * blockIdx.x / gridDim.x;
    const uint64_t g_end = a.total_tiles * (blockIdx.x + 1) / gridDim.x;
    if (g_begin >= g_end) return;
    if (lane == 0) {
        mbar_init(&ps.bar);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    uint32_t phase = 0;
    const uint32_t wait_limit = a.wait_limit ? a.wait_limit : kWaitLimit;
    bool alive = true;
    for (uint32_t k = 0; k < a.count; ++k) {
        const TensorArgs& t = a.t[k];
        const uint64_t t0 = t.tile_begin, t1 = t.tile_begin + t.n_blocks;
        if (t1 <= g_begin) continue;
        if (t0 >= g_end) break;
        const uint64_t b0 = (g_begin > t0 ? g_begin : t0) - t0, b1 = (g_end < t1 ? g_end : t1) - t0;
        const uint64_t n_sub = (t.n_chunks + kPairChunks - 1) / kPairChunks;
        const uint64_t sb = b0 * kPairSubtilesPerBlock;
        const uint64_t se = b1 * kPairSubtilesPerBlock < n_sub ? b1 * kPairSubtilesPerBlock : n_sub;
        __syncthreads();  // every warp is done with the previous tensor's tables
        build_tables_w(sh, tabr, t.tab, threadIdx.x, nthreads, CtaSync{});  // ends with __syncthreads
        const uint64_t span = se - sb;
        const uint64_t s0 = sb + span * warp / nwarps, s1 = sb + span * (warp + 1) / nwarps;
        if (alive && s0 < s1) {
            alive = warp_run_pair(tv, ps, stage, a.pair_stage, wstream, t, s0, s1, lane, a.status, wait_limit,
                                  a.stall != 0, phase, epi);
            if (!alive && !a.stall && lane == 0) raise_status(a.status, AFX_DEV_UNDRAINED);
        }
    }
}

__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1) restore_store_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<false, false>(a, StoreEpilogue{});
}

// The restore from containers in pinned host memory, read over the host link.
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_host_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<true, false>(a, StoreEpilogue{});
}

// The restore of E4M3 containers (raw nibbles, one byte per element), from
// device memory and from pinned host memory.
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_e4m3_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<false, false>(a, StoreE4M3Epilogue{});
}

__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_e4m3_host_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<true, false>(a, StoreE4M3Epilogue{});
}

// The restores with two chunks a lane (device-resident containers).
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_pair_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps_pair(a, StoreEpilogue{});
}

__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_fp16_pair_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps_pair(a, StoreFP16Epilogue{});
}

__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_e4m3_pair_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps_pair(a, StoreE4M3Epilogue{});
}

// The restore of FP16 containers (raw bytes plus the hi section's nibble per
// element), from device memory and from pinned host memory.
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_fp16_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<false, false>(a, StoreFP16Epilogue{});
}

__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_fp16_host_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<true, false>(a, StoreFP16Epilogue{});
}

template <int B>
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1) restore_gemv_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<false, false>(a, GemvEpilogue<B>{});
}

// The fused GEMV with two chunks a lane (batch 1; matrices whose rows hold at
// least LaunchArgs::pair_stage weights, so that a pass still meets at most
// two rows).
template <int B>
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_gemv_pair_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps_pair(a, GemvEpilogue<B>{});
}

// The BF16 restore and GEMV of tensors whose state tables keep only their
// shallowest nodes (code trees with more internal nodes than shared memory
// holds rows for).
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_partial_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<false, true>(a, StoreEpilogue{});
}

__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_store_host_partial_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<true, true>(a, StoreEpilogue{});
}

template <int B>
__global__ void __launch_bounds__(kRestoreMaxWarps * 32, 1)
    restore_gemv_partial_kernel(const __grid_constant__ LaunchArgs a) {
    restore_warps<false, true>(a, GemvEpilogue<B>{});
}

// Rows of the warp GEMV: the sub-tile in which a row starts adds its own
// partial of the row and the first-row partials of the following sub-tiles
// that still lie in the row, in sub-tile order.  One thread per sub-tile;
// the following sub-tiles' starts and partials are loaded four at a time
// (the sums still go in sub-tile order).  Launched as a programmatic
// dependent of the GEMV kernel: it waits for that grid's completion before
// reading anything.
template <int B>
__global__ void gemv_fixup_warp_kernel(const __grid_constant__ LaunchArgs a) {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const uint64_t g = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x;
    if (g >= a.total_subs) return;
    uint32_t k = 0;
    while (k + 1 < a.count && g >= a.t[k + 1].sub_begin) ++k;
    const TensorArgs& t = a.t[k];
    const uint64_t s = g - t.sub_begin;
    const uint64_t n_sub = (t.n_chunks + kWarpChunks - 1) / kWarpChunks;
    if (s >= n_sub) return;
    const uint64_t* ws_o0 = reinterpret_cast<const uint64_t*>(t.ws);
    const float* part = reinterpret_cast<const float*>(ws_o0 + t.n_blocks * kSubtilesPerBlock);
    const uint64_t cols = t.cols, n = t.n;
    const uint64_t o0 = ws_o0[s], o1 = s + 1 < n_sub ? ws_o0[s + 1] : n;
    if (o1 <= o0 || o1 > n) return;  // empty, or a corrupt stream the main kernel already flagged
    const bool narrow = o1 <= (uint64_t{1} << 32);  // 32-bit divisions
    const uint64_t ra = narrow ? static_cast<uint32_t>(o0) / t.cols : o0 / cols;
    const uint64_t r = narrow ? static_cast<uint32_t>(o1 - 1) / t.cols : (o1 - 1) / cols;
    const uint64_t row_start = r * cols, row_end = row_start + cols;
    if (row_start < o0 || r >= t.rows) return;  // the row began in an earlier sub-tile
    const int slot = r == ra ? 0 : 1;
    float sum[kMaxBatch];
#pragma unroll
    for (int b = 0; b < B; ++b) sum[b] = part[(s * 2 + slot) * B + b];
    constexpr int kAhead = 4;
    bool more = true;
    for (uint64_t u0 = s + 1; more && u0 < n_sub; u0 += kAhead) {
        uint64_t start[kAhead];
        float p[kAhead][kMaxBatch];
#pragma unroll
        for (int j = 0; j < kAhead; ++j) {
            const uint64_t u = u0 + j;
            start[j] = u < n_sub ? ws_o0[u] : row_end;
#pragma unroll
            for (int b = 0; b < B; ++b) p[j][b] = u < n_sub ? part[(u * 2) * B + b] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kAhead; ++j) {
            if (!more || start[j] >= row_end) {
                more = false;
            } else {
#pragma unroll
                for (int b = 0; b < B; ++b) sum[b] += p[j][b];
            }
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) t.y[static_cast<uint64_t>(b) * t.rows + r] = sum[b];
}

// Rows split across tiles: the tile in which a row starts adds its own tail
// partial and the head partials of the following tiles, in tile order.
template <int B>
__global__ void gemv_fixup_kernel(const __grid_constant__ LaunchArgs a) {
    const uint64_t g = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x;
    if (g >= a.total_tiles) return;
    uint32_t k = 0;
    while (k + 1 < a.count && g >= a.t[k + 1].tile_begin) ++k;
    const TensorArgs& t = a.t[k];
    const uint64_t tile = g - t.tile_begin;
    const uint64_t cols = t.cols;
    const uint64_t n = static_cast<uint64_t>(t.rows) * cols;
    const uint64_t o0 = t.block_index[tile], o1 = t.block_index[tile + 1];
    if (o1 <= o0 || o1 > n) return;  // empty, or a corrupt index the main kernel already flagged
    const uint64_t r_first = o0 / cols, r_last = (o1 - 1) / cols;
    const uint64_t row_start = r_last * cols, row_end = row_start + cols;
    if (row_start < o0 || row_end <= o1) return;  // the row did not start here, or ends here
    float s[kMaxBatch];
    const int slot = (r_last == r_first) ? 0 : 1;
#pragma unroll
    for (int b = 0; b < B; ++b) s[b] = t.ws[(tile * 2 + slot) * B + b];
    for (uint64_t u = tile + 1; u < t.n_blocks; ++u) {
        const uint64_t p0 = t.block_index[u], p1 = t.block_index[u + 1];
        if (p1 < p0 || p1 > n) break;
        if (p1 == p0) continue;
#pragma unroll
        for (int b = 0; b < B; ++b) s[b] += t.ws[(u * 2) * B + b];
        if (p1 >= row_end) break;
    }
#pragma unroll
    for (int b = 0; b < B; ++b) t.y[static_cast<uint64_t>(b) * t.rows + r_last] = s[b];
}

// One exponent for every weight: out[i] = join(fill, sm[i]).  The block
// index holds the single entry n.
__global__ void fill_store_kernel(const uint8_t* __restrict__ sm, const uint64_t* __restrict__ block_index,
                                  uint32_t fill, uint64_t n, uint16_t* __restrict__ out, int32_t* status) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && block_index[0] != n) raise_status(status, AFX_DEV_BAD_BLOCK);
    const uint64_t groups = (n + 7) >> 3;
    const uint32_t f4 = ror8(fill) * 0x01010101u;
    for (uint64_t g = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; g < groups;
         g += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const uint64_t ob = g << 3;
        if (ob + 8 <= n) {
            const uint2 s8 = __ldg(reinterpret_cast<const uint2*>(sm + ob));
            __stcs(reinterpret_cast<uint4*>(out + ob), join8(make_uint2(f4, f4), s8));
        } else {
            for (uint64_t o = ob; o < n; ++o) out[o] = join1(ror8(fill), sm[o]);
        }
    }
}

// E4M3 with one exponent for every element: 16 elements (8 raw bytes) per
// group; the ragged last group goes out element by element.
// FP16 with one exponent for every element: 8 elements (8 raw bytes, 4 hi
// bytes) per group; the ragged last group goes out element by element.
__global__ void fill_store_fp16_kernel(const uint8_t* __restrict__ raw, const uint8_t* __restrict__ hi,
                                       const uint64_t* __restrict__ block_index, uint32_t fill, uint64_t n,
                                       uint16_t* __restrict__ out, int32_t* status) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && block_index[0] != n) raise_status(status, AFX_DEV_BAD_BLOCK);
    const uint64_t groups = (n + 7) >> 3;
    const uint32_t s1 = (fill << 2) & 0xFFu, s4 = s1 * 0x01010101u;
    for (uint64_t g = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; g < groups;
         g += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const uint64_t ob = g << 3;
        if (ob + 8 <= n) {
            const uint32_t h32 = __ldg(reinterpret_cast<const uint32_t*>(hi) + g);
            const uint2 r8 = __ldg(reinterpret_cast<const uint2*>(raw + ob));
            __stcs(reinterpret_cast<uint4*>(out + ob), fp16_join8(make_uint2(s4, s4), r8, h32));
        } else {
            for (uint64_t o = ob; o < n; ++o) out[o] = fp16_join1(s1, raw[o], fp16_hi3(hi, o));
        }
    }
}

__global__ void fill_store_e4m3_kernel(const uint8_t* __restrict__ raw, const uint64_t* __restrict__ block_index,
                                       uint32_t fill, uint64_t n, uint8_t* __restrict__ out, int32_t* status) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && block_index[0] != n) raise_status(status, AFX_DEV_BAD_BLOCK);
    const uint64_t groups = (n + 15) >> 4;
    const uint32_t f4 = ((fill << 3) & 0xFFu) * 0x01010101u;
    for (uint64_t g = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; g < groups;
         g += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const uint64_t ob = g << 4;
        if (ob + 16 <= n) {
            const uint2 r8 = __ldg(reinterpret_cast<const uint2*>(raw + (ob >> 1)));
            __stcs(reinterpret_cast<uint4*>(out + ob), e4m3_join16(make_uint2(f4, f4), make_uint2(f4, f4), r8));
        } else {
            for (uint64_t o = ob; o < n; ++o) out[o] = e4m3_join1((fill << 3) & 0xFFu, raw[o >> 1] >> ((o & 1u) * 4));
        }
    }
}

// All weights share one exponent: one warp per row, fixed-order reduction.
template <int B>
__global__ void fill_gemv_kernel(const uint8_t* __restrict__ sm, const uint64_t* __restrict__ block_index,
                                 uint32_t fill, const uint16_t* __restrict__ x, float* __restrict__ y, uint32_t rows,
                                 uint32_t cols, int32_t* status) {
    const int lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0 && block_index[0] != static_cast<uint64_t>(rows) * cols)
        raise_status(status, AFX_DEV_BAD_BLOCK);
    const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
    for (uint64_t r = blockIdx.x * static_cast<uint64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        float acc[kMaxBatch] = {0.f, 0.f, 0.f, 0.f};
        for (uint64_t c = lane; c < cols; c += 32) {
            const uint32_t wb = join1(ror8(fill), sm[r * cols + c]);
#pragma unroll
            for (int b = 0; b < B; ++b) acc[b] = fma_bf16(wb, x[b * cols + c], acc[b]);
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = acc[b];
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
            if (lane == 0) y[static_cast<uint64_t>(b) * rows + r] = v;
        }
    }
}

// ---- host side ------------------------------------------------------------------------

// The stage byte of symbol s for the merge of format fmt.
uint32_t stage_byte(uint32_t fmt, uint32_t s) {
    return fmt == AFX_FMT_E4M3 ? (s << 3) & 0xFFu : fmt == AFX_FMT_FP16 ? (s << 2) & 0xFFu : ror8(s);
}

void make_tables(const afx_desc& d, CodeTables& t) {
    std::memset(&t, 0, sizeof t);
    unsigned count[AFX_MAX_CODE_LEN + 1] = {0};
    for (int s = 0; s < 256; ++s)
        if (d.len[s]) ++count[d.len[s]];
    unsigned pos = 0;
    uint32_t first = 0;
    for (int L = 1; L <= AFX_MAX_CODE_LEN; ++L) {
        if (L > 1) first = (first + count[L - 1]) << 1;
        const unsigned first_pos = pos;
        for (int s = 0; s < 256; ++s)
            if (d.len[s] == L) t.sorted[pos++] = static_cast<uint8_t>(stage_byte(d.format, static_cast<uint32_t>(s)));
        t.limit[L] = (first + count[L]) << (AFX_MAX_CODE_LEN - L);
        t.base[L] = static_cast<int32_t>(first_pos) - static_cast<int32_t>(first);
    }
    // internal nodes of the code tree, depth by depth (the root is node 0)
    unsigned min_len = AFX_MAX_CODE_LEN;
    for (int s = 0; s < 256; ++s)
        if (d.len[s]) min_len = std::min<unsigned>(min_len, d.len[s]);
    uint64_t states = 0;
    for (uint32_t depth = 0; depth <= AFX_MAX_CODE_LEN; ++depth) {
        t.state_base[depth] = static_cast<uint32_t>(std::min<uint64_t>(states, 0xFFFFFFFFu));
        if (depth >= d.max_len) continue;
        const uint64_t lo = depth ? (t.limit[depth] >> (AFX_MAX_CODE_LEN - depth)) : 0;
        const uint64_t here = (uint64_t{1} << depth) - lo;
        for (uint64_t k = 0; k < here && states + k < static_cast<uint64_t>(kMaxStates); ++k)
            t.state_depth[states + k] = static_cast<uint8_t>(depth);
        states += here;
    }
    t.n_states = static_cast<uint32_t>(std::min<uint64_t>(states, 0xFFFFFFFFu));
    t.fsm = d.nsym >= 2 && min_len >= 2 ? 1u : 0u;
    t.fsm_rows = static_cast<uint32_t>(std::min<uint64_t>(states, kMaxStates));
}

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
    int threads;
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

afx_status prepare_kernel(const void* func, int threads, size_t smem, int* blocks_per_sm) {
    const int dev = current_device();
    if (dev < 0) return afx_fail(AFX_E_CUDA, "no current CUDA device", 0);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceCache& dc = g_devices[dev];
    for (int i = 0; i < dc.used; ++i)
        if (dc.slot[i].func == func && dc.slot[i].smem == smem && dc.slot[i].threads == threads) {
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
    AFX_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, func, threads, smem),
                 "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (*blocks_per_sm < 1) return afx_fail(AFX_E_CUDA, "kernel does not fit on an SM", 0);
    if (dc.used < kCacheSlots) dc.slot[dc.used++] = {func, threads, smem, *blocks_per_sm};
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

void fill_tensor(const afx_desc& d, const void* container, TensorArgs& t) {
    std::memset(&t, 0, sizeof t);
    const uint8_t* base = static_cast<const uint8_t*>(container);
    t.exp_words = reinterpret_cast<const uint32_t*>(base + d.off_exp);
    t.sm = base + d.off_sm;
    t.hi = d.format == AFX_FMT_FP16 ? base + d.off_hi : nullptr;
    t.chunk_index = reinterpret_cast<const uint16_t*>(base + d.off_chunk);
    t.block_index = reinterpret_cast<const uint64_t*>(base + d.off_block);
    t.n = d.n;
    t.n_chunks = d.n_chunks;
    t.n_blocks = d.n_blocks;
    t.exp_bytes = d.exp_bytes;
    t.total_bits = d.total_bits;
    t.chunk_bytes = d.chunk_bytes;
    {
        // sub-tile s is full when chunks s*32 .. s*32+39 exist (the staged
        // entries) and its stream bytes plus the pad lie inside the section
        const uint64_t sub_bytes = static_cast<uint64_t>(kWarpChunks) * d.chunk_bytes;
        const uint64_t by_chunks = d.n_chunks >= kWarpChunkStage ? (d.n_chunks - kWarpChunkStage) / kWarpChunks + 1 : 0;
        const uint64_t by_bytes = d.exp_bytes >= sub_bytes + kStreamPad ? (d.exp_bytes - kStreamPad) / sub_bytes : 0;
        t.n_sub_full = std::min(by_chunks, by_bytes);
    }
    // The codes in a 64-chunk sub-tile: its bits over the mean code length,
    // with the spread of a count of codes whose lengths add up to a fixed
    // number of bits (variance bits * var(len) / mean(len)^3); the lengths'
    // variance is taken with each code's share 2^-len (the code is
    // complete, so the shares add up to 1).
    t.pair_codes = 0;
    if (d.total_bits && d.n) {
        double mu = 0.0, m2 = 0.0;
        for (int sym = 0; sym < 256; ++sym)
            if (d.len[sym]) {
                const double p = std::ldexp(1.0, -static_cast<int>(d.len[sym]));
                mu += p * d.len[sym];
                m2 += p * d.len[sym] * d.len[sym];
            }
        const double var = std::max(0.0, m2 - mu * mu);
        const double bits = static_cast<double>(kPairChunks) * 8.0 * d.chunk_bytes;
        const double mean_len = static_cast<double>(d.total_bits) / static_cast<double>(d.n);
        const double codes = bits / mean_len, sd = std::sqrt(bits * var / (mean_len * mean_len * mean_len));
        t.pair_codes = static_cast<uint32_t>(std::min(std::ceil(codes + 5.0 * sd), 65536.0));
    }
    make_tables(d, t.tab);
}

// Rows a GEMV warp slice can meet: a slice is at most
// (capacity + 16) / 8 / warps + 2 groups of 8 weights.
uint32_t gemv_rows_per_warp(uint32_t cols) {
    const uint64_t slice = ((AFX_BLOCK_CAPACITY + 16) / 8 / kWarps + 2) * 8;
    return static_cast<uint32_t>(slice / cols + 2);
}

// The warp path's CTAs take equal shares of a launch's tiles in order, and
// each builds the decode tables of every tensor its share touches, so a
// share that crosses into a new tensor pays one more build.  The host puts
// this many empty tiles in front of every tensor: about the time a CTA
// spends on one build, counted in blocks decoded (measured on the GB300:
// the Qwen3-14B-shaped layer runs 3.5 % faster with 4 to 8 of them than
// with none, and the same at every value in that range).
constexpr uint64_t kTableBuildTiles = 5;

// Up to 32 warps per CTA, one CTA per SM: the warp slots and stream
// buffers are fixed by the warp count and the largest T, the rest of the
// opt-in shared memory holds the tables.  A tensor whose state table does
// not fit keeps rows for as many of its shallowest nodes as fit (and
// escapes at the others), or, with fewer than kMinFsmRows of them, takes
// the 12-bit table.
// The warp count of a launch whose largest T is max_chunk_bytes, the shared
// memory its warps need, and how many node rows of a state table fit beside
// them.  Returns 0 when not even one warp and the 12-bit table fit.
int warp_shape(uint32_t max_chunk_bytes, size_t* fixed_out, size_t* fit_rows) {
    int optin = 0;
    const int dev = current_device();
    if (dev < 0 || cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    int warps = kRestoreMaxWarps;
    size_t fixed = 0;
    for (; warps >= 1; warps /= 2) {
        fixed = sharedw_table_offset() + static_cast<size_t>(warps) * sizeof(WarpSlot) +
                static_cast<size_t>(warps) * 2 * (kWarpChunks * max_chunk_bytes + kStreamPad);
        if (fixed + kLutTabBytes <= static_cast<size_t>(optin)) break;
    }
    if (warps < 1) return 0;
    const size_t rows = (static_cast<size_t>(optin) - fixed) / kFsmRowBytes;
    *fixed_out = fixed;
    *fit_rows = rows > kSkipRows ? rows - kSkipRows : 0;
    return warps;
}

// Expected escapes per chunk of a state table with rows for the first
// `rows` internal nodes, from the code lengths alone: symbol s stands for a
// share 2^-len(s) of the codes; a code escapes when a byte boundary falls
// after a prefix whose node has no row, and byte boundaries fall at each
// depth of a code with chance 1/8, so a code escapes with chance (the
// distinct depths mod 8 of its row-less prefixes) / 8.  Nodes are numbered
// as make_tables numbers them: depth by depth, the prefixes at depth d
// that are not codes being [first[d] + count[d], 2^d) in canonical order.
double escapes_per_chunk(const afx_desc& d, size_t rows) {
    uint64_t count[AFX_MAX_CODE_LEN + 1] = {0}, first[AFX_MAX_CODE_LEN + 1] = {0}, next[AFX_MAX_CODE_LEN + 1] = {0};
    uint64_t lo[AFX_MAX_CODE_LEN + 1] = {0}, base[AFX_MAX_CODE_LEN + 1] = {0};
    for (int sym = 0; sym < 256; ++sym)
        if (d.len[sym]) ++count[d.len[sym]];
    uint64_t nodes = 1;  // the root
    for (uint32_t L = 1; L <= AFX_MAX_CODE_LEN; ++L) {
        first[L] = L > 1 ? (first[L - 1] + count[L - 1]) << 1 : 0;
        next[L] = first[L];
        lo[L] = first[L] + count[L];
        base[L] = nodes;
        if (L < d.max_len) nodes += (uint64_t{1} << L) - lo[L];
    }
    double esc = 0.0, bits = 0.0;
    for (int sym = 0; sym < 256; ++sym) {  // canonical order within a length: ascending symbol
        const uint32_t L = d.len[sym];
        if (!L) continue;
        const uint64_t code = next[L]++;
        uint32_t phases = 0;
        for (uint32_t depth = 1; depth < L; ++depth)
            if (base[depth] + (code >> (L - depth)) - lo[depth] >= rows) phases |= 1u << (depth & 7u);
        esc += std::ldexp(static_cast<double>(__builtin_popcount(phases)) / 8.0, -static_cast<int>(L));
        bits += std::ldexp(static_cast<double>(L), -static_cast<int>(L));
    }
    return bits > 0.0 ? esc * 8.0 * d.chunk_bytes / bits : 0.0;
}

// Above this many expected escapes per chunk the 12-bit table restores
// faster than a partial state table (measured on the GB300 with geometric
// exponent mixes: 0.07 per chunk still gains, 1.3 loses a third).
constexpr double kMaxEscapesPerChunk = 0.1;

// A tensor restored with a partial state table: byte steps apply (no 1-bit
// code, two or more symbols), its internal nodes outnumber the rows that
// fit beside 32 warps staging chunks of its T, at least kMinFsmRows rows
// fit, and escapes are rare enough.  Such tensors get launches of their
// own; the rest of the wide trees take the 12-bit table.
bool partial_table(const afx_desc& d) {
    if (d.format != AFX_FMT_BF16 || d.nsym < 2) return false;
    for (int sym = 0; sym < 256; ++sym)
        if (d.len[sym] == 1) return false;
    size_t fixed = 0, fit = 0;
    if (warp_shape(d.chunk_bytes, &fixed, &fit) == 0) return false;
    const size_t rows = std::min<size_t>(fit, kMaxStates);
    if (d.nsym - 1 <= rows || rows < kMinFsmRows) return false;
    return escapes_per_chunk(d, rows) <= kMaxEscapesPerChunk;
}

afx_status warp_launch_config(LaunchArgs& la, int* warps_out, size_t* smem_out) {
    if (current_device() < 0) return afx_fail(AFX_E_CUDA, "no current CUDA device", 0);
    size_t fixed = 0, fit = 0;
    const int warps = warp_shape(la.max_chunk_bytes, &fixed, &fit);
    if (warps < 1) return afx_fail(AFX_E_ARG, "launch needs too much shared memory", 0);
    uint32_t tab_bytes = kLutTabBytes;
    for (uint32_t i = 0; i < la.count; ++i) {
        CodeTables& tab = la.t[i].tab;
        if (!tab.fsm) continue;
        const size_t rows = std::min<size_t>({tab.n_states, static_cast<size_t>(kMaxStates), fit});
        // a partial table only in a launch of the partial kernels
        if (rows < tab.n_states && (rows < kMinFsmRows || !la.partial)) {
            tab.fsm = 0;
            continue;
        }
        tab.fsm_rows = static_cast<uint32_t>(rows);
        tab_bytes = std::max<uint32_t>(tab_bytes, static_cast<uint32_t>((rows + kSkipRows) * kFsmRowBytes));
    }
    la.tab_bytes = tab_bytes;
    *warps_out = warps;
    *smem_out = fixed + tab_bytes;
    return AFX_OK;
}

// The largest stage a warp needs with two chunks a lane: every code of a
// sub-tile, the slack, the offset within a group of 8 and 16 spare bytes.
constexpr uint32_t kPairStageMax = (kPairChunks * kMaxChunkCodes + kPairStageSlack + 7 + 16 + 15) & ~15u;

// The stage of a restore launch with two chunks a lane, or 0 when the
// launch keeps one chunk a lane.  Two chunks a lane pay off when
// - each CTA has at least kPairMinBlocks blocks: a warp's share then holds
//   several 64-chunk sub-tiles, so that the last one does not leave the
//   SM's other warps waiting (a 4096 x 4096 matrix is 4.4 blocks a CTA);
// - 32 warps with their stream buffers and the launch's tables leave each
//   warp a stage that holds a sub-tile's codes (TensorArgs::pair_codes: 5
//   standard deviations above the mean, about 3300 for N(0, 0.02) weights)
//   and the slack, for all but kPairMaxSplitShare of the launch's weights.
//   Sub-tiles that do not fit (a norm vector's 1-bit codes, say) are
//   decoded in two halves of 16 lanes (warp_run_pair).
// AFX_CHUNKS_A_LANE=1 in the environment keeps one chunk a lane; =2 takes
// two wherever the stage fits, whatever the two rules say (so that tests
// reach the two-chunk path with small and ragged tensors).
constexpr uint64_t kPairMinBlocks = 16;
constexpr double kPairMaxSplitShare = 0.02;

uint32_t pair_stage_bytes(const LaunchArgs& la, uint64_t grid) {
    if (la.host_src || la.partial || la.kind > kKindE4M3) return 0;
    const char* e = std::getenv("AFX_CHUNKS_A_LANE");
    const bool force = e && e[0] == '2' && e[1] == 0;
    if (e && e[0] == '1' && e[1] == 0) return 0;
    if (!force && (grid == 0 || la.total_tiles < kPairMinBlocks * grid)) return 0;
    int optin = 0;
    const int dev = current_device();
    if (dev < 0 || cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 0;
    const size_t fixed = sharedw_table_offset() + la.tab_bytes;
    const size_t other = pair_warp_bytes(la.max_chunk_bytes, 0);
    if (fixed + kRestoreMaxWarps * (other + kPairStageMin) > static_cast<size_t>(optin)) return 0;
    const size_t per_warp = (static_cast<size_t>(optin) - fixed) / kRestoreMaxWarps;
    const uint32_t stage = static_cast<uint32_t>(std::min<size_t>((per_warp - other) & ~size_t(15), kPairStageMax));
    double all = 0.0, split = 0.0;
    for (uint32_t i = 0; i < la.count; ++i) {
        const TensorArgs& t = la.t[i];
        if (t.total_bits == 0) continue;
        all += static_cast<double>(t.n);
        if (static_cast<uint64_t>(t.pair_codes) + kPairStageSlack + 7 + 16 > stage) split += static_cast<double>(t.n);
    }
    return force || split <= kPairMaxSplitShare * all ? stage : 0;
}

// The warp GEMV (matrices whose rows hold at least kWarpStage weights, a
// multiple of 8) and its row fix-up.
template <int B>
afx_status launch_gemv_warp(LaunchArgs& la, cudaStream_t s) {
    if (la.count == 0 || la.total_tiles == 0) return AFX_OK;
    const int sms = sm_count();
    if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
    int warps = 0;
    size_t smem = 0;
    const afx_status st = warp_launch_config(la, &warps, &smem);
    if (st != AFX_OK) return st;
    int per_sm = 0;
    void (*kernel)(LaunchArgs) = la.partial ? restore_gemv_partial_kernel<B> : restore_gemv_kernel<B>;
    // two chunks a lane at batch 1 (measured on the layer's matrices: 6 %
    // faster at batch 1; at batch 4 the kernel's sums and loads then spill
    // and it runs 4 % slower)
    la.pair_stage = 0;
    if constexpr (B == 1) {
        la.pair_stage = pair_stage_bytes(la, std::min<uint64_t>(la.total_tiles, static_cast<uint64_t>(sms)));
        for (uint32_t i = 0; i < la.count && la.pair_stage; ++i)
            if (la.t[i].cols < la.pair_stage) la.pair_stage = 0;  // a pass could meet three rows
        if (la.pair_stage) {
            kernel = restore_gemv_pair_kernel<1>;
            warps = kRestoreMaxWarps;
            smem = sharedw_table_offset() + la.tab_bytes +
                   static_cast<size_t>(kRestoreMaxWarps) * pair_warp_bytes(la.max_chunk_bytes, la.pair_stage);
        }
    }
    const afx_status pst = prepare_kernel(reinterpret_cast<const void*>(kernel), warps * 32, smem, &per_sm);
    if (pst != AFX_OK) return pst;
    const uint64_t grid = std::min<uint64_t>(la.total_tiles, static_cast<uint64_t>(sms) * per_sm);
    kernel<<<static_cast<unsigned>(grid), warps * 32, smem, s>>>(la);
    AFX_CUDA_TRY(cudaGetLastError(), "restore_gemv_kernel launch");
    const unsigned fix_blocks = static_cast<unsigned>((la.total_subs + 255) / 256);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(fix_blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    AFX_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemv_fixup_warp_kernel<B>, la), "gemv_fixup_warp_kernel launch");
    return AFX_OK;
}

// The chunks a lane (1 or 2) a restore launch of la takes: the choice
// launch_restore<0> makes, without launching.
uint32_t restore_chunks_a_lane(LaunchArgs la) {
    int warps = 0;
    size_t smem = 0;
    const int sms = sm_count();
    if (sms <= 0 || warp_launch_config(la, &warps, &smem) != AFX_OK) return 1;
    return pair_stage_bytes(la, std::min<uint64_t>(la.total_tiles, static_cast<uint64_t>(sms))) ? 2u : 1u;
}

// programmatic: the launch follows another restore launch of the same
// afx_decode_batch call on this stream and may start while that one's last
// CTAs still run.  The two touch disjoint tensors, and the first launch of
// a call is ordered after all earlier work on the stream as usual, so this
// one starts after that work too.
template <int B>
afx_status launch_restore(LaunchArgs& la, cudaStream_t s, bool programmatic = false) {
    if (la.count == 0 || la.total_tiles == 0) return AFX_OK;
    const int sms = sm_count();
    if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
    if constexpr (B == 0) {
        int warps = 0;
        size_t smem = 0;
        const afx_status st = warp_launch_config(la, &warps, &smem);
        if (st != AFX_OK) return st;
        int per_sm = 0;
        void (*const kernels[3][2])(LaunchArgs) = {{restore_store_kernel, restore_store_host_kernel},
                                                    {restore_store_fp16_kernel, restore_store_fp16_host_kernel},
                                                    {restore_store_e4m3_kernel, restore_store_e4m3_host_kernel}};
        void (*kernel)(LaunchArgs) = kernels[la.kind < 3 ? la.kind : 0][la.host_src ? 1 : 0];
        if (la.partial) kernel = la.host_src ? restore_store_host_partial_kernel : restore_store_partial_kernel;
        la.pair_stage = pair_stage_bytes(la, std::min<uint64_t>(la.total_tiles, static_cast<uint64_t>(sms)));
        if (la.pair_stage) {
            void (*const pair_kernels[3])(LaunchArgs) = {restore_store_pair_kernel, restore_store_fp16_pair_kernel,
                                                          restore_store_e4m3_pair_kernel};
            kernel = pair_kernels[la.kind];
            warps = kRestoreMaxWarps;
            smem = sharedw_table_offset() + la.tab_bytes +
                   static_cast<size_t>(kRestoreMaxWarps) * pair_warp_bytes(la.max_chunk_bytes, la.pair_stage);
        }
        const afx_status pst = prepare_kernel(reinterpret_cast<const void*>(kernel), warps * 32, smem, &per_sm);
        if (pst != AFX_OK) return pst;
        const uint64_t grid = std::min<uint64_t>(la.total_tiles, static_cast<uint64_t>(sms) * per_sm);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(static_cast<unsigned>(warps * 32));
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = programmatic ? 1 : 0;
        AFX_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, la), "restore_store_kernel launch");
        return AFX_OK;
    } else {
        size_t smem = shared_fixed_bytes() + 2 * (static_cast<size_t>(kThreads) * la.max_chunk_bytes + kStreamPad);
        smem += static_cast<size_t>(kWarps) * la.max_rows_per_warp * B * sizeof(float) +
                kWarps * (sizeof(uint64_t) + sizeof(uint32_t));
        if (smem > 227 * 1024) return afx_fail(AFX_E_ARG, "launch needs too much shared memory", 0);
        int per_sm = 0;
        const afx_status st = prepare_kernel(reinterpret_cast<const void*>(restore_kernel<B>), kThreads, smem, &per_sm);
        if (st != AFX_OK) return st;
        const uint64_t grid = std::min<uint64_t>(la.total_tiles, static_cast<uint64_t>(sms) * per_sm);
        restore_kernel<B><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(la);
        AFX_CUDA_TRY(cudaGetLastError(), "restore_kernel launch");
        const unsigned fix_blocks = static_cast<unsigned>((la.total_tiles + 127) / 128);
        gemv_fixup_kernel<B><<<fix_blocks, 128, 0, s>>>(la);
        AFX_CUDA_TRY(cudaGetLastError(), "gemv_fixup_kernel launch");
        return AFX_OK;
    }
}

// Where a buffer lives.  Device memory is staged with bulk copies; pinned
// (or managed) host memory is read with plain loads; pageable host memory
// that the GPU cannot address is refused.
enum class Where { device, host, unusable };

Where where(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return Where::unusable;
    }
    if (at.type == cudaMemoryTypeDevice) return Where::device;
    // host memory the kernel can address with the same pointer
    if ((at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged) && at.devicePointer == p)
        return Where::host;
    return Where::unusable;
}

void reset_launch(LaunchArgs& la) {
    la.count = 0;
    la.total_tiles = 0;
    la.total_subs = 0;
    la.max_chunk_bytes = 0;
    la.max_rows_per_warp = 0;
}

// Zeroes the fields in front of the tensor slots.  Slot k is written in full
// (fill_tensor) before count passes it and the kernels read no slot at or
// past count, so the 13 KB of slots need no clearing on every call.
void clear_launch(LaunchArgs& la) { std::memset(&la, 0, offsetof(LaunchArgs, t)); }

}  // namespace afx

using namespace afx;

namespace {

// afx_decode_batch; stall_polls != 0 is the failure injection of
// afx_test_restore_stalled.  plan != nullptr: launch nothing and write, for
// each tensor, the chunks a lane of the restore launch it would go to (0
// for an empty tensor or a single-exponent fill); outs may then be null.
afx_status decode_batch(const afx_desc* descs, const void* const* containers, void* const* outs, uint32_t count,
                        afx_stream_t stream, int32_t* status, uint32_t stall_polls, uint32_t* plan = nullptr) {
    if (count && (!descs || !containers || (!outs && !plan))) return afx_fail(AFX_E_ARG, "null array", 0);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (uint32_t i = 0; i < count; ++i) {
        const afx_desc& d = descs[i];
        const afx_status st = afx_check_desc(&d);
        if (st != AFX_OK) return afx_fail(st, "invalid container description", 0);
        if (d.n == 0) continue;
        if (plan) {
            plan[i] = 0;
            if (!containers[i] || !aligned(containers[i], 16))
                return afx_fail(AFX_E_ARG, "containers must be 16-byte aligned", 0);
        } else if (!containers[i] || !outs[i] || !aligned(containers[i], 16) || !aligned(outs[i], 16))
            return afx_fail(AFX_E_ARG, "container and output must be 16-byte aligned", 0);
        if (d.nsym >= 2 && d.block_chunks != static_cast<uint32_t>(kThreads))
            return afx_fail(AFX_E_ARG, "the decoder runs 512 chunks per block", 0);
    }
    // [BF16, FP16, E4M3, BF16 with partial state tables][device-resident
    // containers, host-resident containers]
    constexpr int kLists = 4, kPartialList = 3;
    LaunchArgs lists[kLists][2];
    for (int f = 0; f < kLists; ++f)
        for (int h = 0; h < 2; ++h) {
            LaunchArgs& la = lists[f][h];
            clear_launch(la);
            la.status = status;
            la.wait_limit = stall_polls;
            la.stall = stall_polls != 0;
            la.host_src = static_cast<uint32_t>(h);
            la.kind = static_cast<uint32_t>(f == kPartialList ? kKindBF16 : f);
            la.partial = f == kPartialList ? 1u : 0u;
        }
    uint32_t restores = 0;  // restore launches made so far by this call
    uint32_t members[kLists][2][kMaxTensors];  // plan: the tensors of each list's pending launch
    auto flush = [&](LaunchArgs& la, const uint32_t* mem) -> afx_status {
        if (plan) {
            const uint32_t c = restore_chunks_a_lane(la);
            for (uint32_t k = 0; k < la.count; ++k) plan[mem[k]] = c;
            return AFX_OK;
        }
        const afx_status st = launch_restore<0>(la, s, restores > 0);
        ++restores;
        return st;
    };
    for (uint32_t i = 0; i < count; ++i) {
        const afx_desc& d = descs[i];
        if (d.n == 0) continue;
        const uint8_t* base = static_cast<const uint8_t*>(containers[i]);
        const Where wc = where(containers[i]), wo = plan ? Where::device : where(outs[i]);
        if (wc == Where::unusable || wo == Where::unusable)
            return afx_fail(AFX_E_ARG, "container and output must be device memory or pinned host memory", 0);
        if (stall_polls && wc != Where::device)
            return afx_fail(AFX_E_ARG, "the stalled test restore needs a device-resident container", 0);
        const bool e4m3 = d.format == AFX_FMT_E4M3, fp16 = d.format == AFX_FMT_FP16;
        const int list = e4m3 ? kKindE4M3 : fp16 ? kKindFP16 : partial_table(d) ? kPartialList : kKindBF16;
        LaunchArgs& la = lists[list][wc == Where::host ? 1 : 0];
        uint32_t* mem = members[list][wc == Where::host ? 1 : 0];
        if (d.nsym == 1 && plan) continue;
        if (d.nsym == 1) {
            const int sms = sm_count();
            if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
            const uint64_t groups = e4m3 ? (d.n + 15) / 16 : (d.n + 7) / 8;
            const uint64_t blocks = std::min<uint64_t>((groups + 255) / 256, static_cast<uint64_t>(sms) * 8);
            if (e4m3)
                fill_store_e4m3_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
                    base + d.off_sm, reinterpret_cast<const uint64_t*>(base + d.off_block), d.fill, d.n,
                    static_cast<uint8_t*>(outs[i]), status);
            else if (fp16)
                fill_store_fp16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
                    base + d.off_sm, base + d.off_hi, reinterpret_cast<const uint64_t*>(base + d.off_block), d.fill,
                    d.n, static_cast<uint16_t*>(outs[i]), status);
            else
                fill_store_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
                    base + d.off_sm, reinterpret_cast<const uint64_t*>(base + d.off_block), d.fill, d.n,
                    static_cast<uint16_t*>(outs[i]), status);
            AFX_CUDA_TRY(cudaGetLastError(), "fill_store_kernel launch");
            continue;
        }
        if (la.count == static_cast<uint32_t>(kMaxTensors)) {
            const afx_status st = flush(la, mem);
            if (st != AFX_OK) return st;
            reset_launch(la);
        }
        mem[la.count] = i;
        TensorArgs& t = la.t[la.count++];
        fill_tensor(d, containers[i], t);
        t.out = plan ? nullptr : outs[i];
        la.total_tiles += kTableBuildTiles;
        t.tile_begin = la.total_tiles;
        la.total_tiles += d.n_blocks;
        la.max_chunk_bytes = std::max(la.max_chunk_bytes, d.chunk_bytes);
    }
    for (int f = 0; f < kLists; ++f)
        for (int h = 0; h < 2; ++h) {
            LaunchArgs& la = lists[f][h];
            if (la.count == 0 || la.total_tiles == 0) continue;
            const afx_status st = flush(la, members[f][h]);
            if (st != AFX_OK) return st;
        }
    return AFX_OK;
}

}  // namespace

extern "C" afx_status afx_decode_batch(const afx_desc* descs, const void* const* containers, void* const* outs,
                                       uint32_t count, afx_stream_t stream, int32_t* status) {
    return decode_batch(descs, containers, outs, count, stream, status, 0);
}

extern "C" afx_status afx_decode_chunks_a_lane(const afx_desc* descs, const void* const* containers, uint32_t count,
                                               uint32_t* chunks) {
    if (count && !chunks) return afx_fail(AFX_E_ARG, "null array", 0);
    return decode_batch(descs, containers, nullptr, count, nullptr, nullptr, 0, chunks);
}

extern "C" afx_status afx_test_restore_stalled(const afx_desc* desc, const void* container, void* out,
                                               uint32_t wait_polls, afx_stream_t stream, int32_t* status) {
    if (!desc) return afx_fail(AFX_E_ARG, "null description", 0);
    if (desc->nsym < 2 || desc->n == 0) return afx_fail(AFX_E_ARG, "needs a coded tensor (two or more exponents)", 0);
    if (!container || !out || !status) return afx_fail(AFX_E_ARG, "null pointer", 0);
    if (wait_polls == 0 || wait_polls > kWaitLimit) return afx_fail(AFX_E_ARG, "wait_polls must be 1..2^22", 0);
    return decode_batch(desc, &container, &out, 1, stream, status, wait_polls);
}

// The bounds-check bits of the fused prefill kernel's module (afx_prefill_fused.cu).
extern "C" __attribute__((visibility("hidden"))) uint32_t afx_prefill_bounds_bits(void);

extern "C" afx_status afx_debug_bounds_report(uint32_t* bits, uint32_t* checked) {
    if (!bits) return afx_fail(AFX_E_ARG, "null pointer", 0);
    unsigned int v = 0;
    AFX_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_bounds_report, sizeof v), "cudaMemcpyFromSymbol");
    const unsigned int zero = 0;
    AFX_CUDA_TRY(cudaMemcpyToSymbol(g_bounds_report, &zero, sizeof zero), "cudaMemcpyToSymbol");
    *bits = v | afx_prefill_bounds_bits();
    if (checked) *checked = AFX_DEBUG_BOUNDS ? 1u : 0u;
    return AFX_OK;
}

extern "C" afx_status afx_decode_table_kind(const afx_desc* desc, uint32_t* kind, uint32_t* rows) {
    if (!desc || !kind || !rows) return afx_fail(AFX_E_ARG, "null pointer", 0);
    const afx_status st = afx_check_desc(desc);
    if (st != AFX_OK) return afx_fail(st, "invalid container description", 0);
    *kind = AFX_TABLE_FILL;
    *rows = 0;
    if (desc->nsym < 2) return AFX_OK;
    CodeTables t;
    make_tables(*desc, t);
    *kind = AFX_TABLE_LUT12;
    if (!t.fsm) return AFX_OK;
    size_t fixed = 0, fit = 0;
    if (current_device() < 0 || warp_shape(desc->chunk_bytes, &fixed, &fit) == 0)
        return afx_fail(AFX_E_CUDA, "no current CUDA device", 0);
    const size_t k = std::min<size_t>({t.n_states, static_cast<size_t>(kMaxStates), fit});
    if (k == t.n_states) {
        *kind = AFX_TABLE_STATES;
        *rows = static_cast<uint32_t>(k);
    } else if (partial_table(*desc) && k >= kMinFsmRows) {
        *kind = AFX_TABLE_PARTIAL;
        *rows = static_cast<uint32_t>(k);
    }
    return AFX_OK;
}

extern "C" afx_status afx_decode(const afx_desc* desc, const void* container, void* out, afx_stream_t stream,
                                 int32_t* status) {
    if (!desc) return afx_fail(AFX_E_ARG, "null description", 0);
    if (desc->n && (!container || !out)) return afx_fail(AFX_E_ARG, "null pointer", 0);
    return afx_decode_batch(desc, &container, &out, 1, stream, status);
}

namespace {

// Rows long enough for the warp GEMV: a sub-tile (at most kWarpStage - 16
// weights) then meets at most two rows, and rows start on groups of 8.
// Rows of at least kWarpStage weights, a multiple of 8, and short enough
// that kMaxBatch * cols indexes x in 32 bits.
bool warp_gemv_shape(uint32_t cols) {
    return cols >= static_cast<uint32_t>(kWarpStage) && cols % 8 == 0 && cols <= (1u << 29);
}

template <int B>
afx_status gemv_batch(const afx_desc* descs, const void* const* containers, const uint32_t* rows,
                      const uint32_t* cols, const uint16_t* const* xs, float* const* ys, void* const* workspaces,
                      uint32_t count, cudaStream_t s, int32_t* status) {
    LaunchArgs la, lw, lp;  // CTA-tile GEMV, warp GEMV, warp GEMV with partial state tables
    clear_launch(la);
    clear_launch(lw);
    clear_launch(lp);
    la.status = status;
    lw.status = status;
    lp.status = status;
    lp.partial = 1;
    for (uint32_t i = 0; i < count; ++i) {
        const afx_desc& d = descs[i];
        const uint8_t* base = static_cast<const uint8_t*>(containers[i]);
        if (d.nsym == 1) {
            const int sms = sm_count();
            if (sms <= 0) return afx_fail(AFX_E_CUDA, "cannot query the SM count", 0);
            const uint64_t blocks = std::min<uint64_t>((rows[i] + 7) / 8, static_cast<uint64_t>(sms) * 8);
            fill_gemv_kernel<B><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
                base + d.off_sm, reinterpret_cast<const uint64_t*>(base + d.off_block), d.fill, xs[i], ys[i], rows[i],
                cols[i], status);
            AFX_CUDA_TRY(cudaGetLastError(), "fill_gemv_kernel launch");
            continue;
        }
        const bool warp = warp_gemv_shape(cols[i]);
        LaunchArgs& L = warp ? (partial_table(d) ? lp : lw) : la;
        if (L.count == static_cast<uint32_t>(kMaxTensors)) {
            const afx_status st = warp ? launch_gemv_warp<B>(L, s) : launch_restore<B>(L, s);
            if (st != AFX_OK) return st;
            reset_launch(L);
        }
        TensorArgs& t = L.t[L.count++];
        fill_tensor(d, containers[i], t);
        t.x = xs[i];
        t.y = ys[i];
        t.ws = static_cast<float*>(workspaces[i]);
        t.rows = rows[i];
        t.cols = cols[i];
        t.rows_per_warp = gemv_rows_per_warp(cols[i]);
        if (warp) L.total_tiles += kTableBuildTiles;
        t.tile_begin = L.total_tiles;
        t.sub_begin = L.total_subs;
        L.total_tiles += d.n_blocks;
        L.total_subs += (d.n_chunks + kWarpChunks - 1) / kWarpChunks;
        L.max_chunk_bytes = std::max(L.max_chunk_bytes, d.chunk_bytes);
        L.max_rows_per_warp = std::max(L.max_rows_per_warp, t.rows_per_warp);
    }
    afx_status st = launch_gemv_warp<B>(lw, s);
    if (st == AFX_OK) st = launch_gemv_warp<B>(lp, s);
    if (st != AFX_OK) return st;
    return launch_restore<B>(la, s);
}

}  // namespace

extern "C" afx_status afx_decode_gemv_batch(const afx_desc* descs, const void* const* containers,
                                            const uint32_t* rows, const uint32_t* cols, const uint16_t* const* xs,
                                            uint32_t batch, float* const* ys, void* const* workspaces,
                                            const uint64_t* workspace_bytes, uint32_t count, afx_stream_t stream,
                                            int32_t* status) {
    if (count && (!descs || !containers || !rows || !cols || !xs || !ys || !workspaces || !workspace_bytes))
        return afx_fail(AFX_E_ARG, "null array", 0);
    if (batch < 1 || batch > static_cast<uint32_t>(kMaxBatch)) return afx_fail(AFX_E_ARG, "batch must be 1..4", 0);
    for (uint32_t i = 0; i < count; ++i) {
        const afx_desc& d = descs[i];
        const afx_status st = afx_check_desc(&d);
        if (st != AFX_OK) return afx_fail(st, "invalid container description", 0);
        if (!containers[i] || !xs[i] || !ys[i]) return afx_fail(AFX_E_ARG, "null pointer", 0);
        if (d.format != AFX_FMT_BF16) return afx_fail(AFX_E_ARG, "the fused GEMV takes BF16 containers", 0);
        if (rows[i] == 0 || cols[i] < 64 || static_cast<uint64_t>(rows[i]) * cols[i] != d.n)
            return afx_fail(AFX_E_ARG, "rows * cols must equal n, with cols >= 64", 0);
        if (!aligned(containers[i], 16) || !aligned(xs[i], 16))
            return afx_fail(AFX_E_ARG, "container and x must be 16-byte aligned", 0);
        if (where(containers[i]) != Where::device)
            return afx_fail(AFX_E_ARG, "the fused GEMV needs a device-resident container", 0);
        if (where(xs[i]) == Where::unusable || where(ys[i]) == Where::unusable)
            return afx_fail(AFX_E_ARG, "x and y must be device memory or pinned host memory", 0);
        if (d.nsym >= 2) {
            if (d.block_chunks != static_cast<uint32_t>(kThreads))
                return afx_fail(AFX_E_ARG, "the decoder runs 512 chunks per block", 0);
            if (!workspaces[i] || !aligned(workspaces[i], 16)) return afx_fail(AFX_E_ARG, "bad workspace", 0);
            if (workspace_bytes[i] < afx_gemv_workspace_bytes(d.n_blocks, batch))
                return afx_fail(AFX_E_NOSPACE, "workspace too small", 0);
        }
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (batch) {
        case 1: return gemv_batch<1>(descs, containers, rows, cols, xs, ys, workspaces, count, s, status);
        case 2: return gemv_batch<2>(descs, containers, rows, cols, xs, ys, workspaces, count, s, status);
        case 3: return gemv_batch<3>(descs, containers, rows, cols, xs, ys, workspaces, count, s, status);
        default: return gemv_batch<4>(descs, containers, rows, cols, xs, ys, workspaces, count, s, status);
    }
}

extern "C" afx_status afx_decode_gemv(const afx_desc* desc, const void* container, uint32_t rows, uint32_t cols,
                                      const uint16_t* x, uint32_t batch, float* y, void* workspace,
                                      uint64_t workspace_bytes, afx_stream_t stream, int32_t* status) {
    if (!desc) return afx_fail(AFX_E_ARG, "null description", 0);
    return afx_decode_gemv_batch(desc, &container, &rows, &cols, &x, batch, &y, &workspace, &workspace_bytes, 1,
                                 stream, status);
}

// ---- fused restore + GEMV with a fixed, library-owned workspace -------------------
//
// For callers that must not allocate device memory themselves: the
// workspace of the fused GEMV lives in one file-scope device array of
// AFX_STATIC_WORKSPACE_BYTES that every GPU loading the library holds until
// the process exits.  The array's name in host code is only a stand-in, so
// its device address is looked up with cudaGetSymbolAddress, with the
// device current, on the first call made on that device.  The address
// belongs to the context the module was loaded into: it is kept with that
// context's ID and looked up again when the calling thread's current
// context is another one (after cudaDeviceReset, or with a context the
// caller created).

static __device__ __align__(256) float g_static_workspace[AFX_STATIC_WORKSPACE_BYTES / sizeof(float)];

namespace {

struct StaticSlot {
    void* ptr;
    unsigned long long ctx_id;
    bool has_id;
};

std::mutex g_static_mutex;
StaticSlot g_static_slot[afx::kMaxDevices] = {};

// The driver's cuCtxGetCurrent and cuCtxGetId, found through the runtime
// (the library does not link the driver library itself).
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_ctx_fns_once;

// The ID of the calling thread's current context; false when there is
// none yet or the driver does not provide the calls.
bool current_context_id(unsigned long long* id) {
    std::call_once(g_ctx_fns_once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return false;
    void* ctx = nullptr;
    if (g_ctx_get_current(&ctx) != 0 || !ctx) return false;
    return g_ctx_get_id(ctx, id) == 0;
}

afx_status static_workspace(void** ptr) {
    int dev = -1;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return afx_fail(AFX_E_CUDA, "cudaGetDevice", e);
    if (dev < 0 || dev >= afx::kMaxDevices) return afx_fail(AFX_E_CUDA, "device ordinal out of range", 0);
    unsigned long long id = 0;
    bool has_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_static_mutex);
    StaticSlot& slot = g_static_slot[dev];
    if (!slot.ptr || !has_id || !slot.has_id || slot.ctx_id != id) {
        void* p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_static_workspace);
        if (r != cudaSuccess) return afx_fail(AFX_E_CUDA, "cudaGetSymbolAddress", r);
        if (!has_id) has_id = current_context_id(&id);  // the lookup may have created the context
        slot = StaticSlot{p, id, has_id};
    }
    *ptr = slot.ptr;
    return AFX_OK;
}

}  // namespace

extern "C" afx_status afx_decode_gemv_static(const afx_desc* desc, const void* container, uint32_t rows,
                                             uint32_t cols, const uint16_t* x, uint32_t batch, float* y,
                                             afx_stream_t stream, int32_t* status) {
    if (!desc) return afx_fail(AFX_E_ARG, "null description", 0);
    if (batch < 1 || batch > static_cast<uint32_t>(afx::kMaxBatch)) return afx_fail(AFX_E_ARG, "batch must be 1..4", 0);
    const afx_status st = afx_check_desc(desc);
    if (st != AFX_OK) return afx_fail(st, "invalid container description", 0);
    const uint64_t need = afx_gemv_workspace_bytes(desc->n_blocks, batch);
    if (desc->nsym >= 2 && need > AFX_STATIC_WORKSPACE_BYTES) {
        char msg[160];
        snprintf(msg, sizeof msg,
                 "this container needs %llu bytes of GEMV workspace; the static workspace holds %u bytes",
                 static_cast<unsigned long long>(need), static_cast<unsigned>(AFX_STATIC_WORKSPACE_BYTES));
        return afx_fail(AFX_E_NOSPACE, msg, 0);
    }
    void* ws = nullptr;
    const afx_status ws_st = static_workspace(&ws);
    if (ws_st != AFX_OK) return ws_st;
    return afx_decode_gemv(desc, container, rows, cols, x, batch, y, ws, AFX_STATIC_WORKSPACE_BYTES, stream, status);
}
