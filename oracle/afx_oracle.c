/*
 * afx oracle: a plain, slow, obviously correct CPU implementation of the
 * lossless BF16 weight unpack and of the GEMV that consumes the unpacked
 * weights.
 *
 * THIS FILE IS TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.  The product library never includes,
 * links or calls it, and it shares no header, table or helper with the
 * product: it is written from the container specification alone.
 *
 * What it follows:
 *  - "Why Weight Offloading Slows Inference", section "Lossless compression:
 *    fewer bytes to read, more work to unpack": the weights are stored
 *    without loss by giving common BF16 exponent values shorter codes, and
 *    the released bits are restored before computation.  The cited method is
 *    Huffman's minimum-redundancy code (that page's reference [2]).
 *  - "Memory requirements of language model inference on a consumer GPU",
 *    section "Number formats for weights" (Table 1 and the paragraph after
 *    it): BF16 is the released format and the weights must stay exact.  The
 *    BF16 field layout (1 sign, 8 exponent, 7 mantissa bits) is the standard
 *    one that page cites (its reference [2], Kalamkar et al. 2019).
 *  - The container layout is this library's own format (the pages fix none):
 *    a canonical Huffman code over the 8-bit exponent, length-limited to 24
 *    bits, a raw sign|mantissa byte per weight, and per-chunk bit-offset and
 *    output-count indices.  Byte offsets are restated below.
 *
 * Every routine here is the textbook definition, executed one bit or one
 * element at a time, with no blocking, tables or reordering:
 *  - orc_code_lengths: package-merge (Larmore and Hirschberg, 1990), the
 *    optimal length-limited prefix code, in its "coin collector" form.
 *  - orc_canonical_codes: the canonical assignment (count codes per length,
 *    first code per length, then consecutive codes in symbol order).
 *  - orc_encode / orc_decode: bit-by-bit packing and bit-serial decoding.
 *  - orc_gemv: y[b][r] = sum_c W[r][c] * x[b][c] with float64 products and
 *    float64 sums (every bf16 x bf16 product is exact in float64), rounded
 *    to float32 once at the end; A[b][r] = sum_c |W[r][c] * x[b][c]|.
 *
 * Element formats.  The pages treat BF16 only; the same container also
 * holds two other formats (this library's extension, its own reading).
 * Each element splits into an 8-bit-or-smaller symbol, which is coded, and
 * raw bits, which are stored as they are:
 *   0 BF16 (16 bits: sign, 8 exponent, 7 mantissa): symbol = exponent;
 *     raw byte = sign << 7 | mantissa.
 *   1 FP16 (IEEE 754 binary16: sign, 5 exponent, 10 fraction): symbol =
 *     exponent; raw byte = sign << 7 | the 7 trailing fraction bits; the 3
 *     leading fraction bits go to a second raw section, the "hi" section,
 *     one nibble per element: element i in the low nibble of byte i / 2
 *     for even i, the high nibble for odd i, its bit 3 zero (so the 8
 *     nibbles of elements 8g .. 8g + 7 are the aligned word at byte 4g).
 *   2 E4M3 (OCP 8-bit floating point, E4M3: sign, 4 exponent, 3 mantissa):
 *     symbol = exponent; raw nibble = sign << 3 | mantissa, two per byte,
 *     element 2k in the low nibble of byte k.
 *
 * Container (all integers little-endian):
 *   header, 512 bytes:
 *     0  u32 magic 0x31584641      4  u16 version 1     6  u16 header bytes 512
 *     8  u64 n (weights)          16  u64 total code bits
 *    24  u32 chunk bytes T        28  u32 chunks per block C
 *    32  u64 number of chunks     40  u64 number of blocks
 *    48  u64 exp section offset   56  u64 exp section bytes
 *    64  u64 sm section offset    72  u64 chunk index offset
 *    80  u64 block index offset   88  u64 container bytes
 *    96  u32 longest code length 100  u32 number of present exponents
 *   104  u32 fill exponent (when exactly one exponent is present)
 *   108  u32 element format (0 BF16, 1 FP16, 2 E4M3)
 *   112  u64 hi section offset (FP16; 0 for the other formats)
 *   120..255 zero;   256..511 code length of each symbol value 0..255
 *   exp section: u32 words; stream bit i is bit (31 - i mod 32) of word
 *     floor(i / 32); size = (chunks * T rounded up to 16) + 16 zero bytes.
 *   sm section: the raw bits, one byte per element ((sign << 7) | mantissa
 *     for BF16), or one nibble per element for E4M3 (ceil(n / 2) bytes).
 *   hi section (FP16 only, after the sm section): ceil(n / 2) bytes.
 *   chunk index: one u16 per chunk of 8*T stream bits:
 *     bits 0..4  = offset of the first codeword that starts in the chunk,
 *     bits 5..15 = number of codewords that start in the chunk.
 *   block index: u64 per block plus one: entry b = number of codewords that
 *     start before chunk b*C; the last entry is n.
 *   Every section starts at a multiple of 256 bytes; the container size is
 *   a multiple of 256.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_E_FORMAT 1
#define ORC_E_CORRUPT 2
#define ORC_E_INDEX 3
#define ORC_E_ARG 4

#define ORC_HEADER_BYTES 512u
#define ORC_MAGIC 0x31584641u

/* ---- BF16 fields ---------------------------------------------------------- */

static unsigned orc_exponent_of(uint16_t w) { return (w >> 7) & 0xFFu; }

static unsigned orc_sign_mantissa_of(uint16_t w) {
    unsigned sign = (w >> 15) & 1u;
    unsigned mantissa = w & 0x7Fu;
    return (sign << 7) | mantissa;
}

static uint16_t orc_join(unsigned exponent, unsigned sign_mantissa) {
    unsigned sign = (sign_mantissa >> 7) & 1u;
    unsigned mantissa = sign_mantissa & 0x7Fu;
    return (uint16_t)((sign << 15) | (exponent << 7) | mantissa);
}

#define ORC_FMT_BF16 0u
#define ORC_FMT_FP16 1u
#define ORC_FMT_E4M3 2u

static int orc_valid_format(unsigned fmt) { return fmt <= ORC_FMT_E4M3; }

static unsigned orc_elem_bytes(unsigned fmt) { return fmt == ORC_FMT_E4M3 ? 1u : 2u; }

static uint64_t orc_raw_bytes(unsigned fmt, uint64_t n) { return fmt == ORC_FMT_E4M3 ? (n + 1) / 2 : n; }

static unsigned orc_symbols_of_format(unsigned fmt) {
    return fmt == ORC_FMT_E4M3 ? 16u : fmt == ORC_FMT_FP16 ? 32u : 256u;
}

static uint64_t orc_hi_bytes(unsigned fmt, uint64_t n) { return fmt == ORC_FMT_FP16 ? (n + 1) / 2 : 0; }

static unsigned orc_read_elem(const void* elems, unsigned fmt, uint64_t i) {
    if (orc_elem_bytes(fmt) == 1) return ((const uint8_t*)elems)[i];
    return ((const uint16_t*)elems)[i];
}

static void orc_write_elem(void* elems, unsigned fmt, uint64_t i, unsigned v) {
    if (orc_elem_bytes(fmt) == 1)
        ((uint8_t*)elems)[i] = (uint8_t)v;
    else
        ((uint16_t*)elems)[i] = (uint16_t)v;
}

static unsigned orc_symbol_of(unsigned fmt, unsigned v) {
    if (fmt == ORC_FMT_FP16) return (v >> 10) & 0x1Fu; /* the exponent */
    if (fmt == ORC_FMT_E4M3) return (v >> 3) & 0xFu;
    return orc_exponent_of((uint16_t)v);
}

static unsigned orc_raw_of(unsigned fmt, unsigned v) {
    if (fmt == ORC_FMT_FP16) {
        unsigned sign = (v >> 15) & 1u;
        unsigned fraction = v & 0x3FFu;
        return (sign << 7) | (fraction & 0x7Fu);
    }
    if (fmt == ORC_FMT_E4M3) {
        unsigned sign = (v >> 7) & 1u;
        unsigned mantissa = v & 0x7u;
        return (sign << 3) | mantissa;
    }
    return orc_sign_mantissa_of((uint16_t)v);
}

/* the 3 leading fraction bits of an FP16 element (0 for the other formats) */
static unsigned orc_hi_of(unsigned fmt, unsigned v) {
    if (fmt == ORC_FMT_FP16) return ((v & 0x3FFu) >> 7) & 0x7u;
    return 0;
}

static unsigned orc_join_of(unsigned fmt, unsigned symbol, unsigned raw, unsigned hi) {
    if (fmt == ORC_FMT_FP16) {
        unsigned sign = (raw >> 7) & 1u;
        unsigned exponent = symbol;
        unsigned fraction = (hi << 7) | (raw & 0x7Fu);
        return (sign << 15) | (exponent << 10) | fraction;
    }
    if (fmt == ORC_FMT_E4M3) {
        unsigned sign = (raw >> 3) & 1u;
        unsigned mantissa = raw & 0x7u;
        return (sign << 7) | (symbol << 3) | mantissa;
    }
    return orc_join(symbol, raw);
}

/* raw bits of element i in the sm section */
static unsigned orc_get_raw(const uint8_t* sm, unsigned fmt, uint64_t i) {
    if (fmt == ORC_FMT_E4M3) return (sm[i / 2] >> (4 * (i % 2))) & 0xFu;
    return sm[i];
}

/* the hi-section nibble of element i (all 4 bits; bit 3 must be zero) */
static unsigned orc_get_hi(const uint8_t* hi, uint64_t i) { return (hi[i / 2] >> (4 * (i % 2))) & 0xFu; }

static void orc_put_hi(uint8_t* hi, uint64_t i, unsigned v) {
    hi[i / 2] = (uint8_t)(hi[i / 2] | ((v & 0x7u) << (4 * (i % 2))));
}

/* the section starts zeroed; element i's raw bits are OR-ed in */
static void orc_put_raw(uint8_t* sm, unsigned fmt, uint64_t i, unsigned raw) {
    if (fmt == ORC_FMT_E4M3)
        sm[i / 2] = (uint8_t)(sm[i / 2] | (raw << (4 * (i % 2))));
    else
        sm[i] = (uint8_t)raw;
}

/* ---- little-endian field access ------------------------------------------- */

static uint64_t orc_get(const uint8_t* p, unsigned bytes) {
    uint64_t v = 0;
    for (unsigned i = 0; i < bytes; i++) v |= (uint64_t)p[i] << (8 * i);
    return v;
}

static void orc_put(uint8_t* p, unsigned bytes, uint64_t v) {
    for (unsigned i = 0; i < bytes; i++) p[i] = (uint8_t)(v >> (8 * i));
}

static uint64_t orc_round_up(uint64_t v, uint64_t m) { return (v + m - 1) / m * m; }

/* ---- histogram ------------------------------------------------------------ */

int orc_histogram_fmt(const void* elems, uint64_t n, unsigned fmt, uint64_t hist[256]) {
    if (!orc_valid_format(fmt)) return ORC_E_ARG;
    for (int s = 0; s < 256; s++) hist[s] = 0;
    for (uint64_t i = 0; i < n; i++) hist[orc_symbol_of(fmt, orc_read_elem(elems, fmt, i))]++;
    return ORC_OK;
}

int orc_histogram(const uint16_t* w, uint64_t n, uint64_t hist[256]) {
    return orc_histogram_fmt(w, n, ORC_FMT_BF16, hist);
}

/* ---- package-merge ---------------------------------------------------------
 * Each item is a weight plus the multiset of leaves it contains.  Level
 * max_len starts with the leaves sorted by (count, symbol).  Going up one
 * level, adjacent items are paired into packages (an odd last item is
 * dropped) and the packages are merged with a fresh copy of the leaves
 * (leaves first on equal weight).  The first 2(m-1) items of the level-1
 * list are selected; a symbol's code length is the number of times it
 * occurs in the selection.
 */
typedef struct {
    uint64_t weight;
    uint8_t mult[256];
} orc_item;

int orc_code_lengths(const uint64_t hist[256], unsigned max_len, uint8_t len[256]) {
    for (int s = 0; s < 256; s++) len[s] = 0;
    int syms[256];
    int m = 0;
    for (int s = 0; s < 256; s++)
        if (hist[s] > 0) syms[m++] = s;
    if (m <= 1) return ORC_OK; /* zero or one symbol: no bits are needed */
    if (max_len < 1 || max_len > 24) return ORC_E_ARG;
    if (((uint64_t)1 << max_len) < (uint64_t)m) return ORC_E_ARG;

    /* insertion sort by (count, symbol) */
    for (int i = 1; i < m; i++) {
        int v = syms[i];
        int j = i - 1;
        while (j >= 0 && (hist[syms[j]] > hist[v] || (hist[syms[j]] == hist[v] && syms[j] > v))) {
            syms[j + 1] = syms[j];
            j--;
        }
        syms[j + 1] = v;
    }

    orc_item* leaves = (orc_item*)calloc((size_t)m, sizeof(orc_item));
    orc_item* cur = (orc_item*)calloc((size_t)(2 * m), sizeof(orc_item));
    orc_item* next = (orc_item*)calloc((size_t)(2 * m), sizeof(orc_item));
    orc_item* packages = (orc_item*)calloc((size_t)m, sizeof(orc_item));
    if (!leaves || !cur || !next || !packages) {
        free(leaves); free(cur); free(next); free(packages);
        return ORC_E_ARG;
    }
    for (int i = 0; i < m; i++) {
        leaves[i].weight = hist[syms[i]];
        leaves[i].mult[syms[i]] = 1;
    }
    memcpy(cur, leaves, (size_t)m * sizeof(orc_item));
    int cur_n = m;

    for (unsigned level = max_len; level >= 2; level--) {
        int pk = cur_n / 2;
        for (int i = 0; i < pk; i++) {
            packages[i].weight = cur[2 * i].weight + cur[2 * i + 1].weight;
            for (int s = 0; s < 256; s++)
                packages[i].mult[s] = (uint8_t)(cur[2 * i].mult[s] + cur[2 * i + 1].mult[s]);
        }
        int a = 0, b = 0, k = 0;
        while (a < m || b < pk) {
            if (b >= pk || (a < m && leaves[a].weight <= packages[b].weight))
                next[k++] = leaves[a++];
            else
                next[k++] = packages[b++];
        }
        orc_item* t = cur; cur = next; next = t;
        cur_n = k;
    }

    for (int i = 0; i < 2 * (m - 1); i++)
        for (int s = 0; s < 256; s++) len[s] = (uint8_t)(len[s] + cur[i].mult[s]);

    free(leaves); free(cur); free(next); free(packages);
    return ORC_OK;
}

/* ---- canonical codes -------------------------------------------------------
 * Codes of equal length are consecutive integers in symbol order, and the
 * first code of length L is (first code of length L-1 + number of codes of
 * length L-1) shifted left by one.
 */
int orc_canonical_codes(const uint8_t len[256], uint32_t code[256]) {
    unsigned count[33];
    uint32_t next_code[33];
    for (int L = 0; L <= 32; L++) count[L] = 0;
    for (int s = 0; s < 256; s++) {
        if (len[s] > 24) return ORC_E_ARG;
        if (len[s] > 0) count[len[s]]++;
    }
    uint32_t c = 0;
    next_code[0] = 0;
    for (int L = 1; L <= 32; L++) {
        c = (c + (L >= 2 ? count[L - 1] : 0)) << 1;
        next_code[L] = c;
    }
    for (int s = 0; s < 256; s++) {
        if (len[s] > 0)
            code[s] = next_code[len[s]]++;
        else
            code[s] = 0;
    }
    return ORC_OK;
}

/* ---- layout ----------------------------------------------------------------- */

typedef struct {
    uint64_t n, total_bits, n_chunks, n_blocks;
    uint64_t off_exp, exp_bytes, off_sm, off_hi, off_chunk, off_block, container_bytes;
    uint32_t T, C;
} orc_layout;

static int orc_valid_geometry(uint32_t T, uint32_t C) {
    if (!(T == 4 || T == 8 || T == 16 || T == 32 || T == 64)) return 0;
    if (C < 32 || C > 1024 || C % 32 != 0) return 0;
    return 1;
}

static void orc_make_layout(uint64_t n, unsigned fmt, uint64_t total_bits, uint32_t T, uint32_t C,
                            orc_layout* L) {
    L->n = n;
    L->total_bits = total_bits;
    L->T = T;
    L->C = C;
    uint64_t chunk_bits = 8ull * T;
    L->n_chunks = (total_bits + chunk_bits - 1) / chunk_bits;
    L->n_blocks = (L->n_chunks + C - 1) / C;
    L->off_exp = ORC_HEADER_BYTES;
    L->exp_bytes = orc_round_up(L->n_chunks * T, 16) + 16;
    L->off_sm = orc_round_up(L->off_exp + L->exp_bytes, 256);
    if (fmt == ORC_FMT_FP16) {
        L->off_hi = orc_round_up(L->off_sm + orc_raw_bytes(fmt, n), 256);
        L->off_chunk = orc_round_up(L->off_hi + orc_hi_bytes(fmt, n), 256);
    } else {
        L->off_hi = 0;
        L->off_chunk = orc_round_up(L->off_sm + orc_raw_bytes(fmt, n), 256);
    }
    L->off_block = orc_round_up(L->off_chunk + 2 * L->n_chunks, 256);
    L->container_bytes = orc_round_up(L->off_block + 8 * (L->n_blocks + 1), 256);
}

/* Size of the container for n elements whose codes total total_bits bits. */
int orc_container_bytes_fmt(uint64_t n, unsigned fmt, uint64_t total_bits, uint32_t T, uint32_t C,
                            uint64_t* bytes) {
    if (!orc_valid_geometry(T, C) || !orc_valid_format(fmt)) return ORC_E_ARG;
    orc_layout L;
    orc_make_layout(n, fmt, total_bits, T, C, &L);
    *bytes = L.container_bytes;
    return ORC_OK;
}

int orc_container_bytes(uint64_t n, uint64_t total_bits, uint32_t T, uint32_t C, uint64_t* bytes) {
    return orc_container_bytes_fmt(n, ORC_FMT_BF16, total_bits, T, C, bytes);
}

/* ---- stream bits -------------------------------------------------------------- */

static void orc_set_bit(uint8_t* exp_section, uint64_t i) {
    uint64_t word = i / 32;
    unsigned bit_in_word = 31u - (unsigned)(i % 32);
    uint8_t* wp = exp_section + 4 * word;
    uint32_t v = (uint32_t)orc_get(wp, 4);
    v |= (uint32_t)1u << bit_in_word;
    orc_put(wp, 4, v);
}

static unsigned orc_get_bit(const uint8_t* exp_section, uint64_t i) {
    uint64_t word = i / 32;
    unsigned bit_in_word = 31u - (unsigned)(i % 32);
    uint32_t v = (uint32_t)orc_get(exp_section + 4 * word, 4);
    return (v >> bit_in_word) & 1u;
}

/* ---- encode ------------------------------------------------------------------
 * Writes the whole container for the elements elems[0..n) of format fmt
 * with the given code lengths.  The lengths must give every present symbol
 * a code (or, with exactly one present symbol, be all zero), and no length
 * to a value the format's symbols cannot take.  dst must hold
 * orc_container_bytes_fmt().
 */
int orc_encode_fmt(const void* elems, uint64_t n, unsigned fmt, const uint8_t len[256], uint32_t T, uint32_t C,
                   uint8_t* dst, uint64_t dst_bytes) {
    if (!orc_valid_geometry(T, C) || !orc_valid_format(fmt)) return ORC_E_ARG;
    for (unsigned s = orc_symbols_of_format(fmt); s < 256; s++)
        if (len[s] != 0) return ORC_E_ARG;
    uint64_t hist[256];
    orc_histogram_fmt(elems, n, fmt, hist);
    unsigned nsym = 0, fill = 0, longest = 0;
    for (int s = 0; s < 256; s++) {
        if (hist[s] > 0) { nsym++; fill = (unsigned)s; }
        if (len[s] > longest) longest = len[s];
    }
    if (longest > 24) return ORC_E_ARG;
    uint64_t total_bits = 0;
    for (int s = 0; s < 256; s++) {
        if (hist[s] == 0) continue;
        if (nsym >= 2 && len[s] == 0) return ORC_E_ARG;
        total_bits += hist[s] * len[s];
    }
    if (nsym <= 1) {
        for (int s = 0; s < 256; s++)
            if (len[s] != 0) return ORC_E_ARG;
        if (nsym == 0) fill = 0;
    }
    uint32_t code[256];
    if (orc_canonical_codes(len, code) != ORC_OK) return ORC_E_ARG;

    orc_layout L;
    orc_make_layout(n, fmt, total_bits, T, C, &L);
    if (dst_bytes < L.container_bytes) return ORC_E_ARG;
    memset(dst, 0, L.container_bytes);

    /* header */
    orc_put(dst + 0, 4, ORC_MAGIC);
    orc_put(dst + 4, 2, 1);
    orc_put(dst + 6, 2, ORC_HEADER_BYTES);
    orc_put(dst + 8, 8, n);
    orc_put(dst + 16, 8, total_bits);
    orc_put(dst + 24, 4, T);
    orc_put(dst + 28, 4, C);
    orc_put(dst + 32, 8, L.n_chunks);
    orc_put(dst + 40, 8, L.n_blocks);
    orc_put(dst + 48, 8, L.off_exp);
    orc_put(dst + 56, 8, L.exp_bytes);
    orc_put(dst + 64, 8, L.off_sm);
    orc_put(dst + 72, 8, L.off_chunk);
    orc_put(dst + 80, 8, L.off_block);
    orc_put(dst + 88, 8, L.container_bytes);
    orc_put(dst + 96, 4, nsym >= 2 ? longest : 0);
    orc_put(dst + 100, 4, nsym);
    orc_put(dst + 104, 4, nsym == 1 ? fill : 0);
    orc_put(dst + 108, 4, fmt);
    orc_put(dst + 112, 8, L.off_hi);
    for (int s = 0; s < 256; s++) dst[256 + s] = len[s];

    /* exponent codes, one bit at a time, most significant code bit first;
       chunk counts and first-start offsets as each codeword starts */
    uint8_t* exp_section = dst + L.off_exp;
    uint64_t chunk_bits = 8ull * T;
    uint64_t* starts = (uint64_t*)calloc(L.n_chunks ? L.n_chunks : 1, sizeof(uint64_t));
    int64_t* first = (int64_t*)malloc((L.n_chunks ? L.n_chunks : 1) * sizeof(int64_t));
    if (!starts || !first) { free(starts); free(first); return ORC_E_ARG; }
    for (uint64_t c = 0; c < L.n_chunks; c++) first[c] = -1;
    uint64_t pos = 0;
    if (nsym >= 2) {
        for (uint64_t i = 0; i < n; i++) {
            unsigned e = orc_symbol_of(fmt, orc_read_elem(elems, fmt, i));
            uint64_t chunk = pos / chunk_bits;
            if (first[chunk] < 0) first[chunk] = (int64_t)(pos - chunk * chunk_bits);
            starts[chunk]++;
            for (int b = (int)len[e] - 1; b >= 0; b--) {
                if ((code[e] >> b) & 1u) orc_set_bit(exp_section, pos);
                pos++;
            }
        }
    }

    /* raw bits (sign|mantissa bytes for BF16) */
    for (uint64_t i = 0; i < n; i++) orc_put_raw(dst + L.off_sm, fmt, i, orc_raw_of(fmt, orc_read_elem(elems, fmt, i)));
    if (fmt == ORC_FMT_FP16)
        for (uint64_t i = 0; i < n; i++) orc_put_hi(dst + L.off_hi, i, orc_hi_of(fmt, orc_read_elem(elems, fmt, i)));

    /* chunk index */
    for (uint64_t c = 0; c < L.n_chunks; c++) {
        uint64_t gap = first[c] < 0 ? 0 : (uint64_t)first[c];
        if (gap > 31 || starts[c] > 2047) { free(starts); free(first); return ORC_E_ARG; }
        orc_put(dst + L.off_chunk + 2 * c, 2, gap | (starts[c] << 5));
    }

    /* block index */
    uint64_t before = 0;
    for (uint64_t b = 0; b < L.n_blocks; b++) {
        orc_put(dst + L.off_block + 8 * b, 8, before);
        for (uint64_t c = b * C; c < (b + 1) * C && c < L.n_chunks; c++) before += starts[c];
    }
    orc_put(dst + L.off_block + 8 * L.n_blocks, 8, n);

    free(starts);
    free(first);
    return ORC_OK;
}

int orc_encode(const uint16_t* w, uint64_t n, const uint8_t len[256], uint32_t T, uint32_t C,
               uint8_t* dst, uint64_t dst_bytes) {
    return orc_encode_fmt(w, n, ORC_FMT_BF16, len, T, C, dst, dst_bytes);
}

/* ---- decode ------------------------------------------------------------------
 * Parses the header, rebuilds the canonical code from the 256 lengths alone,
 * reads the symbol stream one bit at a time, and joins each symbol with its
 * raw bits.  out receives out_n elements of the header's format (uint16 for
 * BF16 and FP16, uint8 for E4M3).  The chunk and block indices are not used
 * to decode; they are checked afterwards against the codeword start
 * positions seen while decoding (ORC_E_INDEX on any difference).
 */
int orc_decode(const uint8_t* src, uint64_t src_bytes, void* out, uint64_t out_n) {
    if (src_bytes < ORC_HEADER_BYTES) return ORC_E_FORMAT;
    if (orc_get(src + 0, 4) != ORC_MAGIC) return ORC_E_FORMAT;
    if (orc_get(src + 4, 2) != 1 || orc_get(src + 6, 2) != ORC_HEADER_BYTES) return ORC_E_FORMAT;
    uint64_t n = orc_get(src + 8, 8);
    uint64_t total_bits = orc_get(src + 16, 8);
    uint32_t T = (uint32_t)orc_get(src + 24, 4);
    uint32_t C = (uint32_t)orc_get(src + 28, 4);
    if (!orc_valid_geometry(T, C)) return ORC_E_FORMAT;
    unsigned fmt = (unsigned)orc_get(src + 108, 4);
    if (!orc_valid_format(fmt)) return ORC_E_FORMAT;
    orc_layout L;
    orc_make_layout(n, fmt, total_bits, T, C, &L);
    if (orc_get(src + 32, 8) != L.n_chunks || orc_get(src + 40, 8) != L.n_blocks ||
        orc_get(src + 48, 8) != L.off_exp || orc_get(src + 56, 8) != L.exp_bytes ||
        orc_get(src + 64, 8) != L.off_sm || orc_get(src + 72, 8) != L.off_chunk ||
        orc_get(src + 80, 8) != L.off_block || orc_get(src + 88, 8) != L.container_bytes)
        return ORC_E_FORMAT;
    if (src_bytes < L.container_bytes) return ORC_E_FORMAT;
    if (out_n != n) return ORC_E_ARG;
    if (orc_get(src + 112, 8) != L.off_hi) return ORC_E_FORMAT;
    for (unsigned i = 120; i < 256; i++)
        if (src[i] != 0) return ORC_E_FORMAT;

    const uint8_t* len = src + 256;
    unsigned longest = 0, coded = 0;
    for (int s = 0; s < 256; s++) {
        if (len[s] > 24) return ORC_E_FORMAT;
        if (len[s] > 0 && (unsigned)s >= orc_symbols_of_format(fmt)) return ORC_E_FORMAT;
        if (len[s] > longest) longest = len[s];
        if (len[s] > 0) coded++;
    }
    unsigned nsym = (unsigned)orc_get(src + 100, 4);
    unsigned fill = (unsigned)orc_get(src + 104, 4);
    if (orc_get(src + 96, 4) != longest) return ORC_E_FORMAT;

    /* code tables from the lengths: count, first code and first sorted
       position of each length; symbols sorted by (length, value) */
    unsigned count[25] = {0};
    uint32_t first_code[25] = {0};
    unsigned first_pos[25] = {0};
    unsigned sorted[256];
    unsigned m = 0;
    for (unsigned Lb = 1; Lb <= 24; Lb++) {
        first_pos[Lb] = m;
        for (int s = 0; s < 256; s++)
            if (len[s] == Lb) { sorted[m++] = (unsigned)s; count[Lb]++; }
    }
    uint32_t c = 0;
    for (unsigned Lb = 1; Lb <= 24; Lb++) {
        c = (c + (Lb >= 2 ? count[Lb - 1] : 0)) << 1;
        first_code[Lb] = c;
    }

    if (nsym >= 2) {
        if (coded != nsym) return ORC_E_FORMAT;
        /* Kraft equality: sum over codes of 2^(24 - length) == 2^24 */
        uint64_t kraft = 0;
        for (int s = 0; s < 256; s++)
            if (len[s] > 0) kraft += (uint64_t)1 << (24 - len[s]);
        if (kraft != ((uint64_t)1 << 24)) return ORC_E_FORMAT;
        if (fill != 0) return ORC_E_FORMAT;
    } else {
        if (coded != 0 || total_bits != 0) return ORC_E_FORMAT;
        if (nsym == 0 && (n != 0 || fill != 0)) return ORC_E_FORMAT;
        if (nsym == 1 && (n == 0 || fill >= orc_symbols_of_format(fmt))) return ORC_E_FORMAT;
    }

    const uint8_t* exp_section = src + L.off_exp;
    const uint8_t* sm = src + L.off_sm;
    uint64_t chunk_bits = 8ull * T;
    uint64_t* starts = (uint64_t*)calloc(L.n_chunks ? L.n_chunks : 1, sizeof(uint64_t));
    int64_t* first = (int64_t*)malloc((L.n_chunks ? L.n_chunks : 1) * sizeof(int64_t));
    if (!starts || !first) { free(starts); free(first); return ORC_E_ARG; }
    for (uint64_t k = 0; k < L.n_chunks; k++) first[k] = -1;

    uint64_t pos = 0;
    int status = ORC_OK;
    for (uint64_t i = 0; i < n; i++) {
        unsigned e;
        if (nsym == 1) {
            e = fill;
        } else {
            if (pos >= total_bits) { status = ORC_E_CORRUPT; break; }
            uint64_t chunk = pos / chunk_bits;
            if (first[chunk] < 0) first[chunk] = (int64_t)(pos - chunk * chunk_bits);
            starts[chunk]++;
            uint32_t v = 0;
            int found = -1;
            for (unsigned Lb = 1; Lb <= 24; Lb++) {
                if (pos >= total_bits) break;
                v = (v << 1) | orc_get_bit(exp_section, pos);
                pos++;
                if (count[Lb] > 0 && v >= first_code[Lb] && v - first_code[Lb] < count[Lb]) {
                    found = (int)sorted[first_pos[Lb] + (v - first_code[Lb])];
                    break;
                }
            }
            if (found < 0) { status = ORC_E_CORRUPT; break; }
            e = (unsigned)found;
        }
        unsigned hi = fmt == ORC_FMT_FP16 ? orc_get_hi(src + L.off_hi, i) : 0u;
        if (hi > 7u) { status = ORC_E_FORMAT; break; } /* a hi nibble's bit 3 is zero */
        orc_write_elem(out, fmt, i, orc_join_of(fmt, e, orc_get_raw(sm, fmt, i), hi));
    }
    if (status == ORC_OK && pos != total_bits) status = ORC_E_CORRUPT;

    if (status == ORC_OK && fmt == ORC_FMT_E4M3 && n % 2 == 1 && (sm[n / 2] >> 4) != 0)
        status = ORC_E_FORMAT; /* the unused nibble after an odd count is zero */
    if (status == ORC_OK && fmt == ORC_FMT_FP16) {
        /* the hi section's nibble past element n - 1 (an odd n) is zero */
        if (n % 2 == 1 && (src[L.off_hi + n / 2] >> 4) != 0) status = ORC_E_FORMAT;
    }
    if (status == ORC_OK) {
        /* the stream's padding bits are zero */
        for (uint64_t b = total_bits; b < 8 * L.exp_bytes; b++)
            if (orc_get_bit(exp_section, b)) { status = ORC_E_FORMAT; break; }
    }
    if (status == ORC_OK) {
        for (uint64_t k = 0; k < L.n_chunks; k++) {
            uint64_t e = orc_get(src + L.off_chunk + 2 * k, 2);
            uint64_t gap = first[k] < 0 ? 0 : (uint64_t)first[k];
            if ((e & 31u) != gap || (e >> 5) != starts[k]) { status = ORC_E_INDEX; break; }
        }
    }
    if (status == ORC_OK) {
        uint64_t before = 0;
        for (uint64_t b = 0; b < L.n_blocks && status == ORC_OK; b++) {
            if (orc_get(src + L.off_block + 8 * b, 8) != before) status = ORC_E_INDEX;
            for (uint64_t k = b * C; k < (b + 1) * C && k < L.n_chunks; k++) before += starts[k];
        }
        if (status == ORC_OK && orc_get(src + L.off_block + 8 * L.n_blocks, 8) != n) status = ORC_E_INDEX;
    }
    free(starts);
    free(first);
    return status;
}

/* ---- GEMV ------------------------------------------------------------------------
 * W is row-major [rows][cols] (a row is one output), x is [B][cols], y and A
 * are [B][rows].  Products and sums in float64; y is rounded to float32 once.
 */
static double orc_bf16_value(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int orc_gemv(const uint16_t* W, uint64_t rows, uint64_t cols, const uint16_t* x, unsigned B,
             float* y, double* A) {
    if (B < 1) return ORC_E_ARG;
    for (unsigned b = 0; b < B; b++) {
        for (uint64_t r = 0; r < rows; r++) {
            double s = 0.0, a = 0.0;
            for (uint64_t c = 0; c < cols; c++) {
                double p = orc_bf16_value(W[r * cols + c]) * orc_bf16_value(x[(uint64_t)b * cols + c]);
                s += p;
                a += fabs(p);
            }
            y[(uint64_t)b * rows + r] = (float)s;
            A[(uint64_t)b * rows + r] = a;
        }
    }
    return ORC_OK;
}
