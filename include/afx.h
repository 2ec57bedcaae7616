/*
 * afx -- lossless BF16 weight unpack for NVIDIA GB300 (sm_103a).
 *
 * The operation: "Why Weight Offloading Slows Inference", section "Lossless
 * compression: fewer bytes to read, more work to unpack" -- weights are
 * stored without loss by giving common BF16 exponent values shorter codes
 * (Huffman's minimum-redundancy code, that page's reference [2]), and every
 * released bit is restored before computation.  The time this restore takes
 * is the t_unpack term of that page's Eq. (1), and Eq. (2) says compression
 * only pays when the read time it saves, (S - S_disk) / b_disk, exceeds it.
 * "Memory requirements of language model inference on a consumer GPU",
 * section "Number formats for weights", fixes BF16 as the released format
 * and requires the weights to stay exact.
 *
 * The container format is this library's own (the pages fix none):
 *   - a canonical Huffman code over the 8-bit BF16 exponent, code lengths
 *     at most 24 bits (package-merge);
 *   - a raw byte per weight holding sign and mantissa, (sign << 7) | mantissa;
 *   - a chunk index: for every chunk of 8*T stream bits, the bit offset of
 *     the first codeword that starts in it and how many codewords start in
 *     it (the per-chunk bit-offset and output-count indices);
 *   - a block index: for every block of C chunks, the number of weights that
 *     come before it.
 * Byte layout (little-endian; every section 256-byte aligned):
 *   header 512 B: magic "AFX1" (0x31584641), version 1, n, total code bits,
 *     T, C, chunk and block counts, section offsets and sizes, longest code
 *     length, number of present exponents, fill exponent, then the 256 code
 *     lengths at byte 256;
 *   exp section: u32 words, stream bit i = bit (31 - i % 32) of word i / 32,
 *     (chunks * T rounded up to 16) + 16 zero bytes long;
 *   sm section: n bytes;  chunk index: u16 per chunk = offset | count << 5;
 *   block index: u64 per block plus a final entry equal to n.
 *
 * Memory ownership: the caller allocates and frees every buffer.  No entry
 * point allocates device memory.  Entry points that take a stream are
 * asynchronous on that stream; the return value reports argument, format
 * and launch errors found on the host.  Errors found by a kernel (a corrupt
 * stream or index) are OR-ed into *status_dev (an int32 in device memory
 * that the caller zeroes and reads after synchronising; may be NULL).  No
 * entry point traps, aborts or waits on the device without a bound.
 * Every entry point is thread-safe and keeps no state between calls.
 */
#ifndef AFX_H
#define AFX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* afx_stream_t;

typedef enum afx_status {
    AFX_OK = 0,
    AFX_E_ARG = -1,     /* bad argument: null pointer, size, alignment, geometry */
    AFX_E_FORMAT = -2,  /* container header or code lengths are not valid */
    AFX_E_CORRUPT = -3, /* host found a corrupt stream (encoder input check) */
    AFX_E_CUDA = -4,    /* a CUDA runtime call failed */
    AFX_E_NOSPACE = -5, /* destination or workspace smaller than required */
    AFX_E_TIMEOUT = -6  /* a bounded host wait ran out */
} afx_status;

/* Bits OR-ed into *status_dev by the kernels. */
#define AFX_DEV_BAD_BLOCK 0x1 /* a block's chunk counts disagree with the block index */
#define AFX_DEV_BAD_CHUNK 0x2 /* a chunk's codewords do not end where the next chunk begins */
#define AFX_DEV_BAD_CODE 0x4  /* a bit pattern that is no codeword */
#define AFX_DEV_BAD_SHAPE 0x8 /* GEMV rows x cols disagree with the block index */
#define AFX_DEV_TIMEOUT 0x10  /* a staging copy did not arrive within the kernel's wait limit; work skipped */
#define AFX_DEV_UNDRAINED 0x20 /* with AFX_DEV_TIMEOUT: a copy into shared memory had not arrived when the
                                  warp gave up on it, and may land after the kernel's work on it ended */

/* Element formats a container can hold (header field at byte 108; the hi
 * section's offset is the u64 at byte 112, 0 unless FP16).  The
 * pages treat BF16 only; FP16 and E4M3 are this library's extension under
 * the same container:
 *   AFX_FMT_BF16  16-bit elements; coded symbol = the 8-bit exponent, raw
 *                 byte = sign << 7 | 7-bit mantissa.
 *   AFX_FMT_FP16  IEEE 754 binary16; coded symbol = the 5-bit exponent, raw
 *                 byte = sign << 7 | the 7 trailing fraction bits, and the 3
 *                 leading fraction bits in a second raw section (the hi
 *                 section, afx_desc::off_hi): one nibble per element,
 *                 element i in the low nibble of byte i / 2 for even i and
 *                 the high nibble for odd i, bit 3 zero.
 *   AFX_FMT_E4M3  OCP 8-bit float E4M3 (bias 7, largest 448); coded symbol =
 *                 the 4-bit exponent, raw nibble = sign << 3 | 3-bit
 *                 mantissa, two per byte, element 2k in the low nibble of
 *                 byte k. */
#define AFX_FMT_BF16 0u
#define AFX_FMT_FP16 1u
#define AFX_FMT_E4M3 2u

#define AFX_MAX_CODE_LEN 24
/* At most this many codewords start in one block (the decoder's per-block
   staging capacity); the encoder picks T so that this always holds. */
#define AFX_BLOCK_CAPACITY 32768
#define AFX_HEADER_BYTES 512

/* A code over the 256 symbol values (the exponents, for BF16). */
typedef struct afx_code {
    uint64_t count[256]; /* how many elements have each symbol */
    uint32_t code[256];  /* canonical code, right-aligned in len bits */
    uint8_t len[256];    /* code length; 0 = symbol absent (or the only one) */
    uint32_t nsym;       /* number of symbols present */
    uint32_t max_len;    /* longest code length (0 when nsym <= 1) */
    uint32_t fill;       /* the symbol when nsym == 1, else 0 */
    uint32_t format;     /* AFX_FMT_*: the element format the code was built for */
} afx_code;

/* Host-side description of one container: its geometry and section
   offsets.  Filled by afx_encode_bound or afx_parse_header. */
typedef struct afx_desc {
    uint64_t n;               /* weights */
    uint64_t total_bits;      /* sum of all code lengths */
    uint32_t chunk_bytes;     /* T: stream bytes per chunk, 4..64, power of two */
    uint32_t block_chunks;    /* C: chunks per block (the GPU decoder runs C = 512) */
    uint64_t n_chunks;        /* ceil(total_bits / (8 T)) */
    uint64_t n_blocks;        /* ceil(n_chunks / C) */
    uint64_t off_exp, exp_bytes;
    uint64_t off_sm;
    uint64_t off_hi;          /* FP16: the hi section (a nibble per element); 0 for the other formats */
    uint64_t off_chunk;
    uint64_t off_block;
    uint64_t container_bytes; /* whole container, a multiple of 256 */
    uint32_t max_len, nsym, fill;
    uint32_t format;          /* AFX_FMT_*; elements are 2 bytes (BF16, FP16) or 1 byte (E4M3) */
    uint8_t len[256];
} afx_desc;

/* Histogram of the exponents of w_host[0..n) and an optimal prefix code of
 * at most max_len bits (1..24; 24 is the format's cap) with canonical codes.
 * w_host: n BF16 bit patterns in host memory.  Host only, multithreaded.
 * Cites: "Why Weight Offloading Slows Inference", section "Lossless
 * compression: fewer bytes to read, more work to unpack" (shorter codes for
 * common BF16 exponents; Huffman, reference [2]).
 * Errors: AFX_E_ARG on a null pointer or a max_len too small for the
 * number of present exponents. */
afx_status afx_build_code(const uint16_t* w_host, uint64_t n, uint32_t max_len, afx_code* out);

/* afx_build_code for elements of any format: elems_host holds n elements of
 * `format` (uint16 for AFX_FMT_BF16 and AFX_FMT_FP16, uint8 for
 * AFX_FMT_E4M3) and the histogram is over that format's coded symbol.
 * out->format records the format; afx_encode_bound and afx_encode take it
 * from there.  Errors: as afx_build_code, and AFX_E_ARG on an unknown
 * format. */
afx_status afx_build_code_fmt(const void* elems_host, uint64_t n, uint32_t format, uint32_t max_len, afx_code* out);

/* Plans the container for n elements coded with `code` (in code->format): fills *out with the
 * geometry, section offsets and total size.  block_chunks = 0 picks C =
 * 512, the geometry the GPU decoder runs; chunk_bytes = 0 picks the largest
 * T of 32, 16, 8, 4 for which a block can never hold more than
 * AFX_BLOCK_CAPACITY codewords (T = 16, or 8 when some code is 1 bit long).
 * Host only.  Errors: AFX_E_ARG on a bad geometry or a T that could
 * overflow the block capacity. */
afx_status afx_encode_bound(uint64_t n, const afx_code* code, uint32_t chunk_bytes,
                            uint32_t block_chunks, afx_desc* out);

/* Writes the container for elems_host[0..n) into dst_host (dst_bytes >=
 * desc->container_bytes), using the code and the plan from
 * afx_encode_bound.  elems_host holds elements of desc->format (uint16 BF16
 * or FP16 patterns, or uint8 E4M3 patterns).  Host only.  Errors: AFX_E_ARG
 * when an element has a symbol that the code does not cover, or n or the
 * format differs from the plan; AFX_E_NOSPACE when dst is too small. */
afx_status afx_encode(const void* elems_host, uint64_t n, const afx_code* code, const afx_desc* desc,
                      uint8_t* dst_host, uint64_t dst_bytes);

/* Validates the header of a container held in host memory (magic, version,
 * geometry, section offsets, code lengths with the Kraft equality) and fills
 * *out.  Only the first AFX_HEADER_BYTES are read; bytes is the size the
 * caller holds (at least the header).  Errors: AFX_E_FORMAT. */
afx_status afx_parse_header(const uint8_t* header_host, uint64_t bytes, afx_desc* out);

/* Restores all n elements of one container: out_dev[i] = the i-th
 * element, bit for bit.  container_dev: the whole container, 16-byte
 * aligned, in device memory or in pinned (or managed) host memory; a
 * host-resident container is read by the kernel over the host link with no
 * staging copy ("zero copy").  out_dev: n elements of the container's
 * format (uint16 for BF16 and FP16, uint8 for E4M3), 16-byte aligned, in
 * device memory or pinned host memory.  desc: host copy of the container's
 * description.  Runs asynchronously on `stream`; never reads outside the
 * container or writes outside out_dev[0..n).  A corrupt stream or index
 * sets AFX_DEV_* bits in *status_dev (the output is then unspecified).
 * Cites: "Why Weight Offloading Slows Inference", section "Lossless
 * compression: fewer bytes to read, more work to unpack" (restore the
 * released bits before computation; t_unpack of Eq. (1)); the zero-copy
 * read is that page's load path over the link without the staging copy.
 * Errors: AFX_E_ARG (null or misaligned pointers, pageable host memory),
 * AFX_E_FORMAT (desc), AFX_E_CUDA (launch). */
afx_status afx_decode(const afx_desc* desc, const void* container_dev, void* out_dev,
                      afx_stream_t stream, int32_t* status_dev);

/* Restores several containers in one launch: outs_dev[i] gets the weights
 * of containers_dev[i] described by descs[i], for i < count.  The tiles of
 * all containers are shared out over one persistent grid, so small tensors
 * do not leave the GPU idle and the per-launch cost is paid once.  Same
 * arguments, alignment, ownership and errors as afx_decode, per container.
 * Cites: as afx_decode; and "Memory requirements of language model
 * inference on a consumer GPU", section "Loading one part of the model at a
 * time" -- a layer's weights are needed together. */
afx_status afx_decode_batch(const afx_desc* descs, const void* const* containers_dev, void* const* outs_dev,
                            uint32_t count, afx_stream_t stream, int32_t* status_dev);

/* How the restore kernels on the current device decode this container when
 * it is launched alone (a batch with a larger chunk size T can only move a
 * tensor toward the 12-bit table):
 *   AFX_TABLE_FILL     one exponent: no code, a fill of the raw bytes;
 *   AFX_TABLE_LUT12    the 12-bit multi-code table (a 1-bit code, or too
 *                      few state-table rows fit);
 *   AFX_TABLE_STATES   the byte-step state table with a row for every
 *                      internal node of the code tree;
 *   AFX_TABLE_PARTIAL  the byte-step state table with rows for the *rows
 *                      shallowest internal nodes; a code whose prefix
 *                      reaches another node is decoded on its own (BF16
 *                      trees with more nodes than shared memory holds rows
 *                      for; such tensors run in launches of their own).
 * *rows: the node rows of the state table (0 for FILL and LUT12).  Cites:
 * "Why Weight Offloading Slows Inference", section "Lossless compression:
 * fewer bytes to read, more work to unpack" (the decoder that sets
 * t_unpack).  Errors: AFX_E_ARG (null pointer), AFX_E_FORMAT (desc),
 * AFX_E_CUDA (no current device). */
#define AFX_TABLE_FILL 0u
#define AFX_TABLE_LUT12 1u
#define AFX_TABLE_STATES 2u
#define AFX_TABLE_PARTIAL 3u
afx_status afx_decode_table_kind(const afx_desc* desc, uint32_t* kind, uint32_t* rows);

/* How afx_decode_batch(descs, containers, ..., count, ...) would split the
 * stream among the lanes of a warp on the current device, without
 * launching anything: chunks[i] = 1 when container i's restore launch gives
 * each lane one chunk (sub-tiles of 32 chunks), 2 when it gives each lane
 * two consecutive chunks stepped as one span (sub-tiles of 64 chunks), and
 * 0 for an empty tensor or a single-exponent fill.  Two chunks a lane are
 * taken for BF16, FP16 and E4M3 containers in device memory whose launch
 * gives each CTA at least 16 blocks and leaves each warp a stage that holds
 * a 64-chunk sub-tile's codes; the environment variable
 * AFX_CHUNKS_A_LANE=1 (or 2) forces one chunk a lane (or two wherever the
 * stage fits, whatever the launch's size).  The fused GEMV at batch 1
 * (afx_decode_gemv, afx_decode_gemv_batch) takes two chunks a lane by the
 * same rules when every matrix's rows are at least as long as the stage.
 * containers[i] is read only for
 * where it lives (device or pinned host memory), not dereferenced.
 * Cites: "Why Weight Offloading Slows Inference", section "Lossless
 * compression: fewer bytes to read, more work to unpack" (the decoder that
 * sets t_unpack).  Errors: as afx_decode_batch's host-side checks;
 * AFX_E_ARG for a null chunks array. */
afx_status afx_decode_chunks_a_lane(const afx_desc* descs, const void* const* containers, uint32_t count,
                                    uint32_t* chunks);

/* Device workspace (bytes) that afx_decode_gemv needs for this container
 * and batch: for every run of 32 chunks (16 per block) its first weight
 * index (8 bytes) and one float per batch row for each of the two output
 * rows the run can meet. */
afx_status afx_decode_gemv_workspace(const afx_desc* desc, uint32_t batch, uint64_t* bytes);

/* Fused restore + GEMV: y_dev[b][r] = sum_c W[r][c] * x_dev[b][c] for
 * b < batch (1..4), where W is the container's weights viewed row-major as
 * [rows][cols] (rows * cols == n; a row is one output, PyTorch nn.Linear
 * layout) and x_dev is BF16 [batch][cols].  The restored weights never go
 * to global memory.  Each BF16 product is added into a float32 sum with
 * one rounding (fma.rn.f32.bf16); y_dev is float32
 * [batch][rows], overwritten, and bitwise reproducible run to run.
 * workspace_dev: afx_decode_gemv_workspace bytes of device memory, 16-byte
 * aligned, contents ignored.  Requires a BF16 container in device memory,
 * cols >= 64 and x_dev 16-byte aligned.
 * Cites: same passage as afx_decode -- the restored weights feed the
 * computation directly.
 * Errors: AFX_E_ARG (shape, batch, alignment), AFX_E_NOSPACE (workspace),
 * AFX_E_FORMAT, AFX_E_CUDA. */
afx_status afx_decode_gemv(const afx_desc* desc, const void* container_dev, uint32_t rows, uint32_t cols,
                           const uint16_t* x_dev, uint32_t batch, float* y_dev, void* workspace_dev,
                           uint64_t workspace_bytes, afx_stream_t stream, int32_t* status_dev);

/* Several fused restore + GEMV products in one launch, all with the same
 * batch (1..4): for i < count, ys_dev[i] = W_i x_i with W_i the weights of
 * containers_dev[i] viewed as [rows[i]][cols[i]] and x_i = xs_dev[i]
 * ([batch][cols[i]]).  workspaces_dev[i] holds workspace_bytes[i] >=
 * afx_decode_gemv_workspace(descs[i], batch).  Same rules and errors as
 * afx_decode_gemv, per product. */
afx_status afx_decode_gemv_batch(const afx_desc* descs, const void* const* containers_dev, const uint32_t* rows,
                                 const uint32_t* cols, const uint16_t* const* xs_dev, uint32_t batch,
                                 float* const* ys_dev, void* const* workspaces_dev, const uint64_t* workspace_bytes,
                                 uint32_t count, afx_stream_t stream, int32_t* status_dev);

/* Size of the device workspace that afx_decode_gemv_static owns: 4 MiB,
 * enough for a batch-4 product over a container of up to 6,553 blocks
 * (about 165M weights of N(0, 0.02) BF16), or batch 1 over 16,384 blocks. */
#define AFX_STATIC_WORKSPACE_BYTES (4u << 20)

/* afx_decode_gemv without the workspace argument, for callers that cannot
 * allocate device memory: for example a plugin called from inside another
 * runtime's enqueue step, where that runtime owns every device allocation,
 * or code that must not pay for cudaMalloc synchronising the device.  The
 * workspace is a file-scope device array of AFX_STATIC_WORKSPACE_BYTES in
 * this library, held by every GPU that loads it until the process exits;
 * the call itself allocates nothing.  The first call on a device looks up
 * that array's device address (cudaGetSymbolAddress) with the device
 * current, so make that first call before any stream capture.  The address
 * is kept with the ID of the context it was found in and looked up again
 * when a call comes from another current context (for example after
 * cudaDeviceReset, whose next call then also counts as a first call).  Every call
 * shares the one array and it keeps the last call's contents (nothing in
 * it needs to start at zero: each value read is written earlier in the same
 * call), so calls that overlap on the GPU, on any streams, race; run them
 * one after another.  Arguments, results and errors as afx_decode_gemv;
 * AFX_E_NOSPACE (with a message in afx_last_error) when the container needs
 * more workspace than AFX_STATIC_WORKSPACE_BYTES.
 * No counterpart on the pages: this is a deployment convenience of the
 * library, not part of the method. */
afx_status afx_decode_gemv_static(const afx_desc* desc, const void* container_dev, uint32_t rows, uint32_t cols,
                                  const uint16_t* x_dev, uint32_t batch, float* y_dev, afx_stream_t stream,
                                  int32_t* status_dev);

/* One tensor of a streamed layer. */
typedef enum afx_op_kind { AFX_OP_DECODE = 0, AFX_OP_GEMV = 1 } afx_op_kind;

typedef struct afx_op {
    afx_desc desc;          /* the tensor's container description */
    uint64_t offset;        /* byte offset of its container inside the layer blob (multiple of 256) */
    uint32_t kind;          /* afx_op_kind (AFX_OP_GEMV needs a BF16 container) */
    uint32_t rows, cols;    /* AFX_OP_GEMV: weight shape */
    uint32_t batch;         /* AFX_OP_GEMV: 1..4 */
    const uint16_t* x_dev;  /* AFX_OP_GEMV: [batch][cols] BF16 */
    void* out_dev;          /* AFX_OP_DECODE: n elements of desc.format;  AFX_OP_GEMV: float[batch][rows] */
    void* workspace_dev;    /* AFX_OP_GEMV */
    uint64_t workspace_bytes;
    void* out_host;         /* AFX_OP_DECODE, optional: pinned host buffer of n elements that receives out_dev */
} afx_op;

typedef struct afx_layer {
    const void* host_blob;  /* the layer's containers, pinned host memory (cudaHostAlloc) */
    uint64_t blob_bytes;
    const afx_op* ops;
    uint32_t n_ops;
    uint32_t reserved;
} afx_layer;

/* Streams layers from pinned host memory and runs their ops on one GPU:
 * layer l is copied (cudaMemcpyAsync on copy_stream) into device buffer
 * l % n_bufs while the ops of layer l-1 run on compute_stream; a buffer is
 * reused only after the ops that read it have finished (CUDA events, no
 * host waits).  dev_bufs: n_bufs (>= 2) device buffers of buf_bytes
 * (>= every blob_bytes), 256-byte aligned; they may be passed again to a
 * later call, whose first copy waits for all work already queued on
 * compute_stream.  Enqueues everything and returns; synchronise
 * compute_stream and d2h_stream to wait for the results.  Consecutive ops
 * of one kind (and, for GEMV, one batch size) run as one batch launch.
 * A decode op with out_host set also copies its restored weights to that
 * pinned host buffer, on d2h_stream (copy_stream when NULL) after the op,
 * so that copy overlaps the next layer's load and ops; give layers one
 * tensor each to overlap tensor by tensor.  An op whose device output
 * overlaps one that an earlier layer of the call is still copying back
 * waits for that copy, and compute_stream waits for the call's last copy
 * back before any later work on it, so outputs may be reused within and
 * across calls.
 * Cites: "Why Weight Offloading Slows Inference", section "Loading during
 * computation" and Figure 2 (load layer l+1 while layer l computes; a load
 * is free only if it finishes before the GPU needs it), and "Memory
 * requirements of language model inference on a consumer GPU", section
 * "Loading one part of the model at a time" (load, use, release each
 * layer in turn).
 * Errors: AFX_E_ARG, AFX_E_NOSPACE (a blob larger than buf_bytes),
 * AFX_E_FORMAT, AFX_E_CUDA. */
afx_status afx_stream_run(const afx_layer* layers, uint32_t n_layers, void* const* dev_bufs, uint32_t n_bufs,
                          uint64_t buf_bytes, afx_stream_t compute_stream, afx_stream_t copy_stream,
                          afx_stream_t d2h_stream, int32_t* status_dev);

/* Waits on the host until all work queued so far on `stream` has finished,
 * for at most timeout_ms milliseconds (0: no limit), by recording an event
 * and polling it; the host thread never blocks inside a CUDA call.  Then,
 * when status_dev is not NULL (the status word passed to the calls, in
 * device or pinned host memory), it reads that word behind the queued work
 * and stores it in *status_out (when not NULL; 0 otherwise).
 * Returns AFX_OK; AFX_E_CORRUPT when the status word has any AFX_DEV_* bit
 * set (the outputs of the flagged calls are unspecified); AFX_E_TIMEOUT
 * when the limit passed first -- nothing is cancelled, the work keeps
 * running and a later afx_sync can wait for it; AFX_E_CUDA when a CUDA call
 * failed (afx_last_error names it).
 * No counterpart on the pages: this is the library's failure detection
 * (a stream that never finishes becomes an error, not a hung host). */
afx_status afx_sync(afx_stream_t stream, uint32_t timeout_ms, const int32_t* status_dev, int32_t* status_out);

/* Failure injection for tests of the staging timeout: restores a coded
 * tensor (two or more exponents) as afx_decode, except that every staging
 * barrier is armed with the bytes it expects and no copy is issued.  Each
 * warp's first wait therefore gives up after wait_polls polls (1..2^22);
 * the kernel ORs AFX_DEV_TIMEOUT into *status_dev (required) and returns
 * without touching out_dev.  No copy was issued, so nothing is left in
 * flight and the context stays usable.  The production entry points wait
 * up to 2^22 polls; when one of their waits runs out, the warp waits
 * (bounded) for the copy it issued into its other buffer and ORs
 * AFX_DEV_UNDRAINED as well: the copy whose wait ran out may still land.
 * No counterpart on the pages: this exists to test the library's own
 * bounded waits.
 * Errors: AFX_E_ARG, AFX_E_FORMAT, AFX_E_CUDA. */
afx_status afx_test_restore_stalled(const afx_desc* desc, const void* container_dev, void* out_dev,
                                    uint32_t wait_polls, afx_stream_t stream, int32_t* status_dev);

/* ---- prefill -------------------------------------------------------------
 *
 * The prompt of a request multiplies every weight matrix by many token
 * vectors at once ("Memory requirements of language model inference on a
 * consumer GPU", section "Loading one part of the model at a time": the
 * prefill stage processes the whole prompt, then decoding produces one
 * token at a time).  That product is a dense contraction
 * for the tensor cores, and the restore (not HBM) bounds the weights' side:
 * the matrix is restored into scratch memory by the restore kernel, then
 * multiplied by cuBLAS (16-bit inputs, float32 accumulation).  BF16 and
 * FP16 containers are accepted, with activations of the same format;
 * E4M3 containers are refused (AFX_E_ARG). */

/* cuBLAS workspace these calls hand to cuBLAS (caller-owned device memory). */
#define AFX_PREFILL_GEMM_WORKSPACE_BYTES (32u << 20)

/* y_dev[t][r] = sum_c W[r][c] * x_dev[t][c] for t < n_tokens: W the
 * container's weights as [rows][cols] (rows * cols == n, row-major, as
 * afx_decode_gemv), x_dev [n_tokens][cols] in the container's format (BF16
 * or FP16), y_dev float32 [n_tokens][rows] (overwritten).  w_scratch_dev:
 * rows * cols 16-bit elements of device memory that receives the restored
 * W (16-byte aligned).
 * gemm_workspace_dev: AFX_PREFILL_GEMM_WORKSPACE_BYTES of device memory.
 * Enqueues the restore and the product on `stream`.  The first call on a
 * host thread creates that thread's cuBLAS handle for the device (cuBLAS
 * allocates its own small state then); calls allocate nothing else.
 * Status bits of the restore land in *status_dev as for afx_decode.
 * Errors: AFX_E_ARG, AFX_E_FORMAT, AFX_E_CUDA (a failed cuBLAS call too). */
afx_status afx_prefill(const afx_desc* desc, const void* container_dev, uint32_t rows, uint32_t cols,
                       const uint16_t* x_dev, uint32_t n_tokens, float* y_dev, uint16_t* w_scratch_dev,
                       void* gemm_workspace_dev, afx_stream_t stream, int32_t* status_dev);

/* afx_prefill over count matrices, in one of two forms.
 * w_scratch_dev[1] != NULL: pipelined on two streams -- the restore of
 * matrix i (restore_stream, into w_scratch_dev[i % 2]) may overlap the
 * product of matrix i-1 (gemm_stream); each product waits for its restore
 * and each scratch buffer is refilled only after the product that read it
 * (CUDA events, no host waits); both buffers hold the largest rows * cols
 * BF16.  w_scratch_dev[1] == NULL: all matrices are restored in one launch
 * into w_scratch_dev[0], back to back, each starting at a 256-byte
 * boundary (sum of round_up(2 * rows * cols, 256) bytes), then multiplied
 * in order, all on gemm_stream.  On a GPU where both kernels fill every SM
 * they run one after the other either way, and the one-launch form saves
 * the restore launches' ramps.  Synchronise gemm_stream for the results.
 * Same rules and errors as afx_prefill, per matrix. */
afx_status afx_prefill_batch(const afx_desc* descs, const void* const* containers_dev, const uint32_t* rows,
                             const uint32_t* cols, const uint16_t* const* xs_dev, uint32_t n_tokens,
                             float* const* ys_dev, uint32_t count, uint16_t* const* w_scratch_dev,
                             void* gemm_workspace_dev, afx_stream_t restore_stream, afx_stream_t gemm_stream,
                             int32_t* status_dev);

/* ---- fused prefill product ------------------------------------------------
 *
 * The prompt's token vectors through a weight matrix with the restore fused
 * into the tensor-core product: the restored weights go from the decoder
 * through a small L2-resident ring to the tensor cores' shared-memory
 * operand tiles; the restored matrix is never written out.  Cites: "Memory requirements of
 * language model inference on a consumer GPU", section "Loading one part of
 * the model at a time" (the prompt goes through each layer as a whole), and
 * "Why Weight Offloading Slows Inference", section "Lossless compression:
 * fewer bytes to read, more work to unpack" (the released bits are restored
 * before computation; t_unpack of Eq. (1)).
 *
 * The product reads the weights in tile order: the [rows][cols] matrix cut
 * into 128 x 64 tiles, each tile row-major, the tiles of a 128-row band in
 * column order, the bands in row order; element (r, c) at position
 * ((r / 128) * (cols / 64) + c / 64) * 8192 + (r % 128) * 64 + c % 64.
 * afx_tile_order writes that order; encode its output with afx_encode as
 * usual (the container format is unchanged, only the element order). */

/* out_host[tile order] = w_host[rows][cols] (row-major BF16 patterns, host
 * memory, rows a multiple of 128 and cols a multiple of 64; out_host holds
 * rows * cols elements and must not overlap w_host).  Errors: AFX_E_ARG. */
afx_status afx_tile_order(const uint16_t* w_host, uint32_t rows, uint32_t cols, uint16_t* out_host);

/* Bytes of device workspace afx_prefill_fused needs on the current device:
 * one 256 KB ring of restored tiles per CTA, one CTA per SM (38.9 MB on a
 * 152-SM GB300).  A smaller workspace runs fewer CTAs (at least one ring).
 * Errors: AFX_E_ARG, AFX_E_CUDA. */
afx_status afx_prefill_fused_workspace(uint64_t* bytes);

/* y_dev[t][r] = sum_c W[r][c] * x_dev[t][c] for t < n_tokens, where the
 * container holds W ([rows][cols], BF16) in tile order.  x_dev: BF16
 * [n_tokens][cols], row-major, 16-byte aligned; y_dev: float32
 * [n_tokens][rows], overwritten.  Products of BF16 pairs are exact and are
 * summed in float32 by the tensor cores, in a fixed order (y_dev is
 * bitwise reproducible).  rows a multiple of 128, cols a multiple of 64,
 * 1 <= n_tokens <= 262144 (up to 512 per pass over the weights; more
 * tokens restore the weights once per 512).  For balance across the SMs a
 * 128-row band may be split in two along the columns, its two partial sums
 * added into y_dev after a memset on the stream (two float32 additions to
 * zero give the same bits in either order).  The restored weights go through the
 * workspace (a ring of 16 tiles of 16 KB per CTA, written and read back
 * within microseconds, so it stays in L2; no restored matrix is written
 * out): workspace_dev, 256-byte aligned, of workspace_bytes (see
 * afx_prefill_fused_workspace), contents ignored; calls that overlap on the
 * GPU need their own workspaces.  The container, x_dev, y_dev and the
 * workspace in device memory (container 256-byte aligned).  Asynchronous on
 * stream; device-detected corruption or a wait past its limit sets AFX_DEV_*
 * bits in *status_dev (nullable; the outputs are then unspecified).
 * Errors: AFX_E_ARG (shape, alignment, memory kind, format), AFX_E_NOSPACE
 * (workspace smaller than one ring), AFX_E_FORMAT, AFX_E_CUDA. */
afx_status afx_prefill_fused(const afx_desc* desc, const void* container_dev, uint32_t rows, uint32_t cols,
                             const uint16_t* x_dev, uint32_t n_tokens, float* y_dev, void* workspace_dev,
                             uint64_t workspace_bytes, afx_stream_t stream, int32_t* status_dev);

/* afx_prefill_fused over count matrices in one launch (per 16 matrices),
 * all with the same n_tokens: ys_dev[i] = W_i xs_dev[i] with W_i the
 * tile-ordered weights of containers_dev[i], [rows[i]][cols[i]].  One
 * workspace for the call.  Same rules and errors as afx_prefill_fused, per
 * matrix. */
afx_status afx_prefill_fused_batch(const afx_desc* descs, const void* const* containers_dev, const uint32_t* rows,
                                   const uint32_t* cols, const uint16_t* const* xs_dev, uint32_t n_tokens,
                                   float* const* ys_dev, uint32_t count, void* workspace_dev, uint64_t workspace_bytes,
                                   afx_stream_t stream, int32_t* status_dev);

/* ---- residency planning ------------------------------------------------
 *
 * Where each tensor of a model lives during inference on one GPU with a
 * device-memory budget.  "Why Weight Offloading Slows Inference", section
 * "Lossless compression: fewer bytes to read, more work to unpack", Eq. (1)
 * (a step costs the reads plus t_unpack) and Eq. (2) (streaming compressed
 * weights pays when (S - S_disk) / b > t_unpack); "Memory requirements of
 * language model inference on a consumer GPU", section "Loading one part of
 * the model at a time" (what does not fit is loaded as needed). */
typedef enum afx_placement {
    AFX_RESIDENT_DECODED = 0,    /* BF16 in device memory: S bytes, no per-step cost */
    AFX_RESIDENT_COMPRESSED = 1, /* container in device memory: C bytes, restored each step */
    AFX_STREAM_COMPRESSED = 2,   /* container copied over the link each step, then restored */
    AFX_STREAM_RAW = 3           /* BF16 copied over the link each step */
} afx_placement;

typedef struct afx_plan_tensor {
    uint64_t decoded_bytes;    /* S: 2 bytes per weight */
    uint64_t compressed_bytes; /* C: the container */
} afx_plan_tensor;

typedef struct afx_plan_rates {
    double link_gbs;      /* b: host-to-device copy rate, GB/s (1e9 bytes/s) */
    double restore_gbs;   /* restore rate in decoded BF16 GB/s: t_unpack = S / restore_gbs */
    uint32_t overlapped;  /* 1: a streamed tensor's copy overlaps the previous one's restore, costing
                             max(C/b, t_unpack); 0: the two add, C/b + t_unpack (Eq. (2) as written) */
    uint32_t reserved;
} afx_plan_rates;

/* Chooses a placement for each of n tensors that minimises the modelled
 * per-step time (the sum of the tensors' costs) with the resident bytes at
 * most device_budget_bytes.  Costs per step: resident decoded 0; resident
 * compressed t_unpack; streamed compressed C/b + t_unpack (or the max when
 * overlapped); streamed raw S/b.  Exact dynamic programming over memory in
 * units of device_budget_bytes / 65536, every size rounded up to whole
 * units (so the plan always fits; it may leave part of a unit unused).
 * placement_out: n afx_placement values.  step_ms_out, resident_bytes_out:
 * the plan's modelled time and exact resident bytes (either may be NULL).
 * Host only.  Errors: AFX_E_ARG (null arrays, n == 0, rates not positive,
 * n above 65536). */
afx_status afx_plan_residency(const afx_plan_tensor* tensors, uint32_t n, uint64_t device_budget_bytes,
                              const afx_plan_rates* rates, uint32_t* placement_out, double* step_ms_out,
                              uint64_t* resident_bytes_out);

/* Bounds report of the restore kernels since the last call (the report is
 * cleared).  In a library built with AFX_DEBUG_BOUNDS=1 (the build's
 * --debug-bounds variant, libafx_debug.so) every range the restore path is
 * about to read or write is checked against its buffer first -- the warp's
 * exponent stage, the stream buffer, the state table, the output -- and a
 * failed check sets one bit of *bits (see BoundsCheck in the kernel
 * source); *checked is 1 in such a build and 0 in a regular one, whose
 * report stays 0.  A stand-in for a memory checker; no counterpart on the
 * pages.  Synchronises the device.  Errors: AFX_E_ARG, AFX_E_CUDA. */
afx_status afx_debug_bounds_report(uint32_t* bits, uint32_t* checked);

/* Static text for a status code. */
const char* afx_status_string(afx_status status);

/* The message of the last error an entry point returned on this thread
 * (with the CUDA error name when a CUDA call failed).  Never NULL; valid
 * until the next call into afx on this thread. */
const char* afx_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* AFX_H */
