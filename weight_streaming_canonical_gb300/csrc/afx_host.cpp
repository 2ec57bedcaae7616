// Host side of afx: symbol histogram, length-limited canonical code,
// container planning, bit packing and header validation.  BF16 is the
// pages' format; FP16 and E4M3 share the container (the element format
// fixes which bits are coded and which are stored raw; see afx.h).
//
// The operation: "Why Weight Offloading Slows Inference", section
// "Lossless compression: fewer bytes to read, more work to unpack" --
// shorter codes for common BF16 exponent values (Huffman's
// minimum-redundancy code, that page's reference [2]); sign and mantissa
// stay raw.  Code lengths are capped at AFX_MAX_CODE_LEN bits with
// package-merge (Larmore and Hirschberg 1990), which is optimal among
// codes obeying the cap.
#include <algorithm>
#include <cstring>
#include <thread>
#include <vector>

#include "afx_internal.h"

namespace {

uint64_t round_up(uint64_t v, uint64_t m) { return (v + m - 1) / m * m; }

void put_le(uint8_t* p, unsigned bytes, uint64_t v) {
    for (unsigned i = 0; i < bytes; ++i) p[i] = static_cast<uint8_t>(v >> (8 * i));
}

uint64_t get_le(const uint8_t* p, unsigned bytes) {
    uint64_t v = 0;
    for (unsigned i = 0; i < bytes; ++i) v |= static_cast<uint64_t>(p[i]) << (8 * i);
    return v;
}

unsigned worker_count(uint64_t n) {
    unsigned hw = std::thread::hardware_concurrency();
    if (hw == 0) hw = 1;
    uint64_t by_size = n / (1u << 20) + 1;  // at least 1M weights per worker
    return static_cast<unsigned>(std::min<uint64_t>({hw, 32, by_size}));
}

// Package-merge by level selection.  Lists are built bottom-up (the
// deepest level holds the leaves; every shallower level merges the leaves
// with packages of adjacent pairs from the level below).  Then 2(m-1)
// items are selected at the top level; a selected leaf adds one to its
// symbol's length, and p selected packages select the first 2p items one
// level down.
struct PmItem {
    uint64_t weight;
    int leaf;  // symbol of a leaf, -1 for a package
};

afx_status package_merge(const uint64_t count[256], uint32_t max_len, uint8_t len[256]) {
    std::vector<int> syms;
    for (int s = 0; s < 256; ++s)
        if (count[s]) syms.push_back(s);
    std::memset(len, 0, 256);
    const size_t m = syms.size();
    if (m <= 1) return AFX_OK;
    if (max_len < 1 || max_len > AFX_MAX_CODE_LEN) return AFX_E_ARG;
    if ((uint64_t{1} << max_len) < m) return AFX_E_ARG;
    std::stable_sort(syms.begin(), syms.end(), [&](int a, int b) {
        return count[a] != count[b] ? count[a] < count[b] : a < b;
    });
    std::vector<PmItem> leaves(m);
    for (size_t i = 0; i < m; ++i) leaves[i] = {count[syms[i]], syms[i]};

    // level[d] for d = 1..max_len; level[max_len] = leaves
    std::vector<std::vector<PmItem>> level(max_len + 1);
    level[max_len] = leaves;
    for (uint32_t d = max_len - 1; d >= 1; --d) {
        const std::vector<PmItem>& below = level[d + 1];
        std::vector<PmItem> packages(below.size() / 2);
        for (size_t i = 0; i < packages.size(); ++i)
            packages[i] = {below[2 * i].weight + below[2 * i + 1].weight, -1};
        std::vector<PmItem>& cur = level[d];
        cur.reserve(m + packages.size());
        size_t a = 0, b = 0;
        while (a < m || b < packages.size()) {
            bool take_leaf = b >= packages.size() || (a < m && leaves[a].weight <= packages[b].weight);
            cur.push_back(take_leaf ? leaves[a++] : packages[b++]);
        }
        if (d == 1) break;
    }
    size_t select = 2 * (m - 1);
    for (uint32_t d = 1; d <= max_len && select > 0; ++d) {
        size_t packs = 0;
        for (size_t i = 0; i < select; ++i) {
            const PmItem& it = level[d][i];
            if (it.leaf >= 0)
                ++len[it.leaf];
            else
                ++packs;
        }
        select = 2 * packs;
    }
    return AFX_OK;
}

// Canonical codes: walk the symbols in (length, value) order; the next
// code is the previous one plus one, shifted left by the length increase.
void canonical_codes(const uint8_t len[256], uint32_t code[256]) {
    std::vector<int> order;
    for (int s = 0; s < 256; ++s) {
        code[s] = 0;
        if (len[s]) order.push_back(s);
    }
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return len[a] < len[b]; });
    uint32_t c = 0;
    unsigned prev = 0;
    for (size_t i = 0; i < order.size(); ++i) {
        unsigned l = len[order[i]];
        if (i == 0)
            c = 0;
        else
            c = (c + 1) << (l - prev);
        code[order[i]] = c;
        prev = l;
    }
}

bool format_ok(uint32_t fmt) { return fmt == AFX_FMT_BF16 || fmt == AFX_FMT_FP16 || fmt == AFX_FMT_E4M3; }

// Symbols a format's elements can produce: 256 for BF16 (its 8-bit
// exponent), 32 for FP16, 16 for E4M3.
unsigned symbol_range(uint32_t fmt) { return fmt == AFX_FMT_E4M3 ? 16u : fmt == AFX_FMT_FP16 ? 32u : 256u; }

uint64_t raw_bytes(uint32_t fmt, uint64_t n) { return fmt == AFX_FMT_E4M3 ? (n + 1) / 2 : n; }

// FP16's hi section: one nibble per element (the 3 leading fraction bits,
// bit 3 zero), element i in the low nibble of byte i / 2 for even i.
uint64_t hi_bytes(uint32_t fmt, uint64_t n) { return fmt == AFX_FMT_FP16 ? (n + 1) / 2 : 0; }

// The coded symbol is the exponent: BF16 bits 14..7, FP16 bits 14..10,
// E4M3 bits 6..3.  The raw byte of the 16-bit formats is the sign and bits
// 6..0; FP16's bits 9..7 go to the hi section.  E4M3's raw nibble is the
// sign and bits 2..0.
inline unsigned symbol_of(uint32_t fmt, unsigned v) {
    return fmt == AFX_FMT_E4M3 ? (v >> 3) & 0xFu : fmt == AFX_FMT_FP16 ? (v >> 10) & 0x1Fu : (v >> 7) & 0xFFu;
}

inline unsigned raw_of(uint32_t fmt, unsigned v) {
    return fmt == AFX_FMT_E4M3 ? ((v >> 4) & 0x8u) | (v & 0x7u) : ((v >> 8) & 0x80u) | (v & 0x7Fu);
}

inline unsigned element(const void* elems, uint32_t fmt, uint64_t i) {
    return fmt == AFX_FMT_E4M3 ? static_cast<const uint8_t*>(elems)[i] : static_cast<const uint16_t*>(elems)[i];
}

bool geometry_ok(uint32_t T, uint32_t C) {
    bool t_ok = T == 4 || T == 8 || T == 16 || T == 32 || T == 64;
    return t_ok && C >= 32 && C <= 1024 && C % 32 == 0;
}

void layout(uint64_t n, uint32_t fmt, uint64_t total_bits, uint32_t T, uint32_t C, afx_desc* d) {
    d->n = n;
    d->total_bits = total_bits;
    d->chunk_bytes = T;
    d->block_chunks = C;
    const uint64_t chunk_bits = 8ull * T;
    d->n_chunks = (total_bits + chunk_bits - 1) / chunk_bits;
    d->n_blocks = (d->n_chunks + C - 1) / C;
    d->off_exp = AFX_HEADER_BYTES;
    d->exp_bytes = round_up(d->n_chunks * T, 16) + 16;
    d->off_sm = round_up(d->off_exp + d->exp_bytes, 256);
    if (fmt == AFX_FMT_FP16) {
        d->off_hi = round_up(d->off_sm + raw_bytes(fmt, n), 256);
        d->off_chunk = round_up(d->off_hi + hi_bytes(fmt, n), 256);
    } else {
        d->off_hi = 0;
        d->off_chunk = round_up(d->off_sm + raw_bytes(fmt, n), 256);
    }
    d->format = fmt;
    d->off_block = round_up(d->off_chunk + 2 * d->n_chunks, 256);
    d->container_bytes = round_up(d->off_block + 8 * (d->n_blocks + 1), 256);
}

}  // namespace

extern "C" {

const char* afx_status_string(afx_status s) {
    switch (s) {
        case AFX_OK: return "ok";
        case AFX_E_ARG: return "invalid argument";
        case AFX_E_FORMAT: return "invalid container format";
        case AFX_E_CORRUPT: return "corrupt stream";
        case AFX_E_CUDA: return "CUDA error";
        case AFX_E_NOSPACE: return "buffer too small";
        case AFX_E_TIMEOUT: return "timed out";
    }
    return "unknown status";
}

afx_status afx_build_code(const uint16_t* w, uint64_t n, uint32_t max_len, afx_code* out) {
    return afx_build_code_fmt(w, n, AFX_FMT_BF16, max_len, out);
}

afx_status afx_build_code_fmt(const void* w, uint64_t n, uint32_t fmt, uint32_t max_len, afx_code* out) {
    if (!out || (n && !w) || !format_ok(fmt)) return AFX_E_ARG;
    std::memset(out, 0, sizeof(*out));
    out->format = fmt;
    const unsigned workers = worker_count(n);
    std::vector<std::vector<uint64_t>> part(workers, std::vector<uint64_t>(256, 0));
    auto count_range = [&](unsigned k) {
        uint64_t lo = n * k / workers, hi = n * (k + 1) / workers;
        uint64_t* h = part[k].data();
        if (fmt == AFX_FMT_E4M3) {
            const uint8_t* e = static_cast<const uint8_t*>(w);
            for (uint64_t i = lo; i < hi; ++i) ++h[(e[i] >> 3) & 0xFu];
        } else {
            const uint16_t* e = static_cast<const uint16_t*>(w);
            const unsigned shift = fmt == AFX_FMT_FP16 ? 10u : 7u, mask = fmt == AFX_FMT_FP16 ? 0x1Fu : 0xFFu;
        for (uint64_t i = lo; i < hi; ++i) ++h[(e[i] >> shift) & mask];
        }
    };
    if (workers == 1) {
        count_range(0);
    } else {
        std::vector<std::thread> pool;
        for (unsigned k = 0; k < workers; ++k) pool.emplace_back(count_range, k);
        for (auto& t : pool) t.join();
    }
    for (unsigned k = 0; k < workers; ++k)
        for (int s = 0; s < 256; ++s) out->count[s] += part[k][s];
    for (int s = 0; s < 256; ++s)
        if (out->count[s]) {
            ++out->nsym;
            out->fill = static_cast<uint32_t>(s);
        }
    if (out->nsym != 1) out->fill = 0;
    afx_status st = package_merge(out->count, max_len, out->len);
    if (st != AFX_OK) return st;
    canonical_codes(out->len, out->code);
    for (int s = 0; s < 256; ++s) out->max_len = std::max<uint32_t>(out->max_len, out->len[s]);
    return AFX_OK;
}

afx_status afx_encode_bound(uint64_t n, const afx_code* code, uint32_t T, uint32_t C, afx_desc* out) {
    if (!code || !out || !format_ok(code->format)) return AFX_E_ARG;
    for (unsigned s = symbol_range(code->format); s < 256; ++s)
        if (code->len[s] || code->count[s]) return AFX_E_ARG;
    if (C == 0) C = AFX_DECODE_THREADS;
    uint64_t total_bits = 0, present = 0;
    unsigned min_len = 255;
    for (int s = 0; s < 256; ++s) {
        if (!code->count[s]) continue;
        ++present;
        total_bits += code->count[s] * code->len[s];
        min_len = std::min<unsigned>(min_len, code->len[s]);
    }
    uint64_t counted = 0;
    for (int s = 0; s < 256; ++s) counted += code->count[s];
    if (counted != n || present != code->nsym) return AFX_E_ARG;
    if (present >= 2 && min_len == 0) return AFX_E_ARG;
    if (present <= 1) min_len = 1;
    if (T == 0) {
        // Largest of 32, 16, 8, 4 whose worst case fits the block capacity.
        T = 32;
        while (T > 4 && 8ull * T * C > static_cast<uint64_t>(AFX_BLOCK_CAPACITY) * min_len) T /= 2;
    }
    if (!geometry_ok(T, C)) return AFX_E_ARG;
    if (8ull * T * C > static_cast<uint64_t>(AFX_BLOCK_CAPACITY) * min_len) return AFX_E_ARG;
    std::memset(out, 0, sizeof(*out));
    layout(n, code->format, total_bits, T, C, out);
    out->nsym = code->nsym;
    out->fill = code->nsym == 1 ? code->fill : 0;
    out->max_len = code->nsym >= 2 ? code->max_len : 0;
    std::memcpy(out->len, code->len, 256);
    return AFX_OK;
}

afx_status afx_encode(const void* w, uint64_t n, const afx_code* code, const afx_desc* d, uint8_t* dst,
                      uint64_t dst_bytes) {
    if (!code || !d || !dst || (n && !w)) return AFX_E_ARG;
    if (d->n != n || !geometry_ok(d->chunk_bytes, d->block_chunks)) return AFX_E_ARG;
    const uint32_t fmt = d->format;
    if (!format_ok(fmt) || code->format != fmt) return AFX_E_ARG;
    if (dst_bytes < d->container_bytes) return AFX_E_NOSPACE;
    afx_desc check;
    layout(n, fmt, d->total_bits, d->chunk_bytes, d->block_chunks, &check);
    if (check.container_bytes != d->container_bytes || check.off_block != d->off_block) return AFX_E_ARG;
    if (std::memcmp(d->len, code->len, 256) != 0) return AFX_E_ARG;
    std::memset(dst, 0, d->container_bytes);

    uint8_t* h = dst;
    put_le(h + 0, 4, AFX_MAGIC);
    put_le(h + 4, 2, 1);
    put_le(h + 6, 2, AFX_HEADER_BYTES);
    put_le(h + 8, 8, d->n);
    put_le(h + 16, 8, d->total_bits);
    put_le(h + 24, 4, d->chunk_bytes);
    put_le(h + 28, 4, d->block_chunks);
    put_le(h + 32, 8, d->n_chunks);
    put_le(h + 40, 8, d->n_blocks);
    put_le(h + 48, 8, d->off_exp);
    put_le(h + 56, 8, d->exp_bytes);
    put_le(h + 64, 8, d->off_sm);
    put_le(h + 72, 8, d->off_chunk);
    put_le(h + 80, 8, d->off_block);
    put_le(h + 88, 8, d->container_bytes);
    put_le(h + 96, 4, d->max_len);
    put_le(h + 100, 4, d->nsym);
    put_le(h + 104, 4, d->fill);
    put_le(h + 108, 4, fmt);
    put_le(h + 112, 8, d->off_hi);
    std::memcpy(h + 256, code->len, 256);

    // The work is split into segments of whole groups of 8 elements (so every
    // raw byte, nibble pair and hi-section byte has one writer), run on
    // worker threads.
    const unsigned workers = worker_count(n);
    std::vector<uint64_t> seg(workers + 1);
    for (unsigned k = 0; k <= workers; ++k) seg[k] = std::min<uint64_t>(n, (n * k / workers + 7) & ~uint64_t{7});
    seg[workers] = n;
    auto parallel = [&](auto&& fn) {
        if (workers == 1) {
            fn(0u);
            return;
        }
        std::vector<std::thread> pool;
        for (unsigned k = 0; k < workers; ++k) pool.emplace_back(fn, k);
        for (auto& t : pool) t.join();
    };

    uint8_t* sm = dst + d->off_sm;
    uint8_t* hs = fmt == AFX_FMT_FP16 ? dst + d->off_hi : nullptr;
    std::vector<char> off_fill(workers, 0);  // single-symbol tensors: an element with another symbol
    parallel([&](unsigned k) {
        for (uint64_t i = seg[k]; i < seg[k + 1]; ++i) {
            const unsigned v = element(w, fmt, i);
            if (d->nsym <= 1 && symbol_of(fmt, v) != d->fill) off_fill[k] = 1;
            if (fmt == AFX_FMT_E4M3) {
                sm[i / 2] |= static_cast<uint8_t>(raw_of(fmt, v) << (4 * (i & 1)));
            } else {
                sm[i] = static_cast<uint8_t>(raw_of(fmt, v));
            }
            if (fmt == AFX_FMT_FP16)  // the 3 leading fraction bits, a nibble per element
                hs[i / 2] |= static_cast<uint8_t>(((v >> 7) & 0x7u) << (4 * (i & 1)));
        }
    });

    if (d->nsym <= 1) {
        for (unsigned k = 0; k < workers; ++k)
            if (off_fill[k]) return AFX_E_ARG;
        if (d->total_bits != 0) return AFX_E_ARG;
        put_le(dst + d->off_block, 8, n);
        return AFX_OK;
    }

    // Pass 1: each segment's coded bits.  The stream is written only when
    // they add up to the plan's total, so elements that do not match the code
    // cannot write past the stream section.
    std::vector<uint64_t> seg_bits(workers, 0);
    std::vector<char> seg_bad(workers, 0);
    parallel([&](unsigned k) {
        uint64_t bits = 0;
        for (uint64_t i = seg[k]; i < seg[k + 1]; ++i) {
            const unsigned l = code->len[symbol_of(fmt, element(w, fmt, i))];
            if (l == 0) seg_bad[k] = 1;
            bits += l;
        }
        seg_bits[k] = bits;
    });
    std::vector<uint64_t> seg_start(workers + 1, 0);
    for (unsigned k = 0; k < workers; ++k) {
        if (seg_bad[k]) return AFX_E_ARG;
        seg_start[k + 1] = seg_start[k] + seg_bits[k];
    }
    if (seg_start[workers] != d->total_bits) return AFX_E_ARG;

    // Pass 2: bit packing into u32 words, most significant bit first, with
    // the chunk index updated as each codeword starts.  A segment's first
    // and last word, and its first and last chunk entry, may be shared with
    // its neighbours: those are kept aside and merged after the workers.
    uint8_t* words = dst + d->off_exp;
    uint8_t* chunk_index = dst + d->off_chunk;
    const unsigned chunk_shift = static_cast<unsigned>(__builtin_ctz(8u * d->chunk_bytes));
    struct Edge {
        uint64_t word_i = ~uint64_t{0};
        uint32_t word = 0;
        uint64_t chunk = ~uint64_t{0};
        uint32_t gap = 0, count = 0;
    };
    std::vector<Edge> head(workers), tail(workers);
    parallel([&](unsigned k) {
        if (seg[k] == seg[k + 1]) return;
        uint64_t pos = seg_start[k];
        uint64_t word_i = pos >> 5;
        unsigned acc_bits = static_cast<unsigned>(pos & 31);  // bits of the word before this segment's (zeros)
        uint64_t acc = 0;
        bool first_word = true, first_chunk = true;
        uint64_t cur_chunk = ~uint64_t{0};
        uint32_t cur_count = 0, cur_gap = 0;
        auto flush_chunk = [&]() {
            if (cur_chunk == ~uint64_t{0}) return;
            if (first_chunk) {
                head[k].chunk = cur_chunk;
                head[k].gap = cur_gap;
                head[k].count = cur_count;
                first_chunk = false;
            } else {
                put_le(chunk_index + 2 * cur_chunk, 2, cur_gap | (cur_count << 5));
            }
        };
        for (uint64_t i = seg[k]; i < seg[k + 1]; ++i) {
            const unsigned e = symbol_of(fmt, element(w, fmt, i));
            const unsigned l = code->len[e];
            const uint64_t chunk = pos >> chunk_shift;
            if (chunk != cur_chunk) {
                flush_chunk();
                cur_chunk = chunk;
                cur_count = 0;
                cur_gap = static_cast<uint32_t>(pos - (chunk << chunk_shift));
            }
            ++cur_count;
            acc = (acc << l) | code->code[e];
            acc_bits += l;
            pos += l;
            if (acc_bits >= 32) {
                acc_bits -= 32;
                const uint32_t out = static_cast<uint32_t>(acc >> acc_bits);
                if (first_word) {
                    head[k].word_i = word_i;
                    head[k].word = out;
                    first_word = false;
                } else {
                    put_le(words + 4 * word_i, 4, out);
                }
                ++word_i;
                acc &= (uint64_t{1} << acc_bits) - 1;
            }
        }
        // the last chunk entry and the partial last word go to the merge
        tail[k].chunk = cur_chunk;
        tail[k].gap = cur_gap;
        tail[k].count = cur_count;
        if (first_chunk) {  // the segment's codes all started in one chunk: that entry is its head
            head[k].chunk = ~uint64_t{0};
        }
        if (acc_bits) {
            tail[k].word_i = word_i;
            tail[k].word = static_cast<uint32_t>(acc << (32 - acc_bits));
        }
    });
    // merge the edges in segment order: words by OR (each side's bits of a
    // shared word are zero in the other's), chunk entries by adding counts
    // (the gap is that of the first code starting in the chunk)
    uint64_t open_chunk = ~uint64_t{0};
    uint32_t open_gap = 0, open_count = 0;
    auto emit = [&](uint64_t chunk, uint32_t gap, uint32_t count) {
        if (chunk == ~uint64_t{0}) return;
        if (chunk == open_chunk) {
            open_count += count;
            return;
        }
        if (open_chunk != ~uint64_t{0}) put_le(chunk_index + 2 * open_chunk, 2, open_gap | (open_count << 5));
        open_chunk = chunk;
        open_gap = gap;
        open_count = count;
    };
    for (unsigned k = 0; k < workers; ++k) {
        for (const Edge* e : {&head[k], &tail[k]})
            if (e->word_i != ~uint64_t{0}) {
                const uint32_t v = static_cast<uint32_t>(get_le(words + 4 * e->word_i, 4)) | e->word;
                put_le(words + 4 * e->word_i, 4, v);
            }
        if (seg[k] == seg[k + 1]) continue;
        emit(head[k].chunk, head[k].gap, head[k].count);
        // chunks the segment wrote itself lie between its head and tail: the
        // open entry (the head's) closes before them
        if (tail[k].chunk != head[k].chunk && head[k].chunk != ~uint64_t{0} && open_chunk == head[k].chunk) {
            put_le(chunk_index + 2 * open_chunk, 2, open_gap | (open_count << 5));
            open_chunk = ~uint64_t{0};
        }
        emit(tail[k].chunk, tail[k].gap, tail[k].count);
    }
    if (open_chunk != ~uint64_t{0}) put_le(chunk_index + 2 * open_chunk, 2, open_gap | (open_count << 5));

    // Block index: weights before each block's first chunk.
    uint8_t* block_index = dst + d->off_block;
    uint64_t before = 0;
    for (uint64_t b = 0; b < d->n_blocks; ++b) {
        put_le(block_index + 8 * b, 8, before);
        const uint64_t c_end = std::min<uint64_t>((b + 1) * d->block_chunks, d->n_chunks);
        for (uint64_t c = b * d->block_chunks; c < c_end; ++c) before += get_le(chunk_index + 2 * c, 2) >> 5;
    }
    put_le(block_index + 8 * d->n_blocks, 8, n);
    return before == n ? AFX_OK : AFX_E_ARG;
}

afx_status afx_parse_header(const uint8_t* h, uint64_t bytes, afx_desc* out) {
    if (!h || !out || bytes < AFX_HEADER_BYTES) return AFX_E_ARG;
    if (get_le(h, 4) != AFX_MAGIC || get_le(h + 4, 2) != 1 || get_le(h + 6, 2) != AFX_HEADER_BYTES)
        return AFX_E_FORMAT;
    afx_desc d;
    std::memset(&d, 0, sizeof d);
    const uint64_t n = get_le(h + 8, 8), total_bits = get_le(h + 16, 8);
    const uint32_t T = static_cast<uint32_t>(get_le(h + 24, 4)), C = static_cast<uint32_t>(get_le(h + 28, 4));
    if (!geometry_ok(T, C)) return AFX_E_FORMAT;
    if (n > (uint64_t{1} << 48) || total_bits > 24 * n) return AFX_E_FORMAT;
    const uint32_t fmt = static_cast<uint32_t>(get_le(h + 108, 4));
    if (!format_ok(fmt)) return AFX_E_FORMAT;
    layout(n, fmt, total_bits, T, C, &d);
    if (get_le(h + 32, 8) != d.n_chunks || get_le(h + 40, 8) != d.n_blocks || get_le(h + 48, 8) != d.off_exp ||
        get_le(h + 56, 8) != d.exp_bytes || get_le(h + 64, 8) != d.off_sm || get_le(h + 72, 8) != d.off_chunk ||
        get_le(h + 80, 8) != d.off_block || get_le(h + 88, 8) != d.container_bytes || get_le(h + 112, 8) != d.off_hi)
        return AFX_E_FORMAT;
    for (unsigned i = 120; i < 256; ++i)
        if (h[i]) return AFX_E_FORMAT;
    d.max_len = static_cast<uint32_t>(get_le(h + 96, 4));
    d.nsym = static_cast<uint32_t>(get_le(h + 100, 4));
    d.fill = static_cast<uint32_t>(get_le(h + 104, 4));
    std::memcpy(d.len, h + 256, 256);
    unsigned longest = 0, coded = 0;
    uint64_t kraft = 0;
    for (int s = 0; s < 256; ++s) {
        if (d.len[s] > AFX_MAX_CODE_LEN) return AFX_E_FORMAT;
        if (d.len[s] && static_cast<unsigned>(s) >= symbol_range(fmt)) return AFX_E_FORMAT;
        if (d.len[s]) {
            ++coded;
            kraft += uint64_t{1} << (AFX_MAX_CODE_LEN - d.len[s]);
        }
        longest = std::max<unsigned>(longest, d.len[s]);
    }
    if (d.max_len != longest) return AFX_E_FORMAT;
    if (d.nsym >= 2) {
        if (coded != d.nsym || kraft != (uint64_t{1} << AFX_MAX_CODE_LEN) || d.fill != 0) return AFX_E_FORMAT;
        if (total_bits < n || total_bits == 0) return AFX_E_FORMAT;
        unsigned min_len = 255;
        for (int s = 0; s < 256; ++s)
            if (d.len[s]) min_len = std::min<unsigned>(min_len, d.len[s]);
        if (8ull * T * C > static_cast<uint64_t>(AFX_BLOCK_CAPACITY) * min_len) return AFX_E_FORMAT;
    } else {
        if (coded != 0 || total_bits != 0 || d.fill >= symbol_range(fmt)) return AFX_E_FORMAT;
        if (d.nsym == 0 && (n != 0 || d.fill != 0)) return AFX_E_FORMAT;
        if (d.nsym == 1 && n == 0) return AFX_E_FORMAT;
    }
    *out = d;
    return AFX_OK;
}

afx_status afx_check_desc(const afx_desc* d) {
    if (!d) return AFX_E_ARG;
    if (!geometry_ok(d->chunk_bytes, d->block_chunks)) return AFX_E_FORMAT;
    if (d->n > (uint64_t{1} << 48) || d->total_bits > 24 * d->n) return AFX_E_FORMAT;
    if (!format_ok(d->format)) return AFX_E_FORMAT;
    afx_desc L;
    layout(d->n, d->format, d->total_bits, d->chunk_bytes, d->block_chunks, &L);
    if (L.n_chunks != d->n_chunks || L.n_blocks != d->n_blocks || L.off_exp != d->off_exp ||
        L.exp_bytes != d->exp_bytes || L.off_sm != d->off_sm || L.off_chunk != d->off_chunk ||
        L.off_block != d->off_block || L.container_bytes != d->container_bytes || L.off_hi != d->off_hi)
        return AFX_E_FORMAT;
    unsigned longest = 0, coded = 0, min_len = 255;
    uint64_t kraft = 0;
    for (int s = 0; s < 256; ++s) {
        if (d->len[s] > AFX_MAX_CODE_LEN) return AFX_E_FORMAT;
        if (d->len[s] && static_cast<unsigned>(s) >= symbol_range(d->format)) return AFX_E_FORMAT;
        if (d->len[s]) {
            ++coded;
            kraft += uint64_t{1} << (AFX_MAX_CODE_LEN - d->len[s]);
            min_len = std::min<unsigned>(min_len, d->len[s]);
        }
        longest = std::max<unsigned>(longest, d->len[s]);
    }
    if (d->max_len != longest) return AFX_E_FORMAT;
    if (d->nsym >= 2) {
        if (coded != d->nsym || kraft != (uint64_t{1} << AFX_MAX_CODE_LEN)) return AFX_E_FORMAT;
        if (d->total_bits < d->n) return AFX_E_FORMAT;
        if (8ull * d->chunk_bytes * d->block_chunks > static_cast<uint64_t>(AFX_BLOCK_CAPACITY) * min_len)
            return AFX_E_FORMAT;
    } else {
        if (coded != 0 || d->total_bits != 0 || d->fill >= symbol_range(d->format)) return AFX_E_FORMAT;
        if (d->nsym == 1 && d->n == 0) return AFX_E_FORMAT;
        if (d->nsym == 0 && d->n != 0) return AFX_E_FORMAT;
    }
    return AFX_OK;
}

afx_status afx_decode_gemv_workspace(const afx_desc* d, uint32_t batch, uint64_t* bytes) {
    if (!d || !bytes || batch < 1 || batch > 4) return AFX_E_ARG;
    *bytes = afx_gemv_workspace_bytes(d->n_blocks, batch);
    return AFX_OK;
}

}  // extern "C"
