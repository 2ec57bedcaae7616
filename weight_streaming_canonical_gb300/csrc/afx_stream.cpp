// Layer streaming: compressed layers move from pinned host memory to the GPU
// on a copy stream while the previous layer's ops run on a compute stream.
//
// "Why Weight Offloading Slows Inference", section "Loading during
// computation" and Figure 2: while the GPU computes one layer the next is
// already loading, and a load costs nothing only if it finishes before the
// GPU needs the weights.  "Memory requirements of language model inference
// on a consumer GPU", section "Loading one part of the model at a time":
// load a layer, use it, release its memory, go on to the next.  Here the
// copy carries the compressed container, so the link moves fewer bytes and
// the unpack runs on the GPU after the copy.
//
// Ordering uses CUDA events only: buffer l % n_bufs is refilled after the
// ops that read it have finished, and a layer's ops start after its copy.
// Restored tensors that go back to host memory are copied on a third
// stream after their layer's ops, so that with a full-duplex link the copy
// back overlaps the next layer's load.  An op whose output overlaps a
// device output that an earlier layer of the call is still copying back
// waits for that copy, and the compute stream waits for the last copy back
// at the end of the call, so later work on it cannot overwrite an output
// that is still being read.  The host never waits.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdio>
#include <vector>

#include "afx_internal.h"

namespace {

struct EventSet {
    std::vector<cudaEvent_t> ev;
    ~EventSet() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
    }
    bool create(size_t n) {
        ev.assign(n, nullptr);
        for (auto& e : ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
        return true;
    }
};

#define AFX_STREAM_TRY(call, what)                                        \
    do {                                                                  \
        const cudaError_t e_ = (call);                                    \
        if (e_ != cudaSuccess) return afx_fail(AFX_E_CUDA, (what), e_);   \
    } while (0)

bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

afx_status check_layer(const afx_layer& L, uint64_t buf_bytes) {
    if ((!L.host_blob && L.blob_bytes) || (!L.ops && L.n_ops)) return AFX_E_ARG;
    if (L.blob_bytes > buf_bytes) return AFX_E_NOSPACE;
    for (uint32_t i = 0; i < L.n_ops; ++i) {
        const afx_op& op = L.ops[i];
        afx_status st = afx_check_desc(&op.desc);
        if (st != AFX_OK) return st;
        if (op.offset % 256 != 0 || op.offset > L.blob_bytes || op.desc.container_bytes > L.blob_bytes - op.offset)
            return AFX_E_ARG;
        if (op.kind == AFX_OP_DECODE) {
            if (op.desc.n && !op.out_dev) return AFX_E_ARG;
        } else if (op.kind == AFX_OP_GEMV) {
            if (!op.x_dev || !op.out_dev || op.batch < 1 || op.batch > 4) return AFX_E_ARG;
            if (op.desc.format != AFX_FMT_BF16) return AFX_E_ARG;
            if (static_cast<uint64_t>(op.rows) * op.cols != op.desc.n) return AFX_E_ARG;
        } else {
            return AFX_E_ARG;
        }
    }
    return AFX_OK;
}

// An NVTX range for as long as the object lives (a profiler's timeline shows
// where each layer's copy and ops were enqueued; without a tool attached the
// calls do nothing).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

// Runs ops[0..count), all of one kind (and one batch size), as one batch call.
afx_status run_group(const afx_op* ops, uint32_t count, uint8_t* buf, afx_stream_t stream, int32_t* status_dev) {
    std::vector<afx_desc> descs(count);
    std::vector<const void*> containers(count);
    for (uint32_t i = 0; i < count; ++i) {
        descs[i] = ops[i].desc;
        containers[i] = buf + ops[i].offset;
    }
    if (ops[0].kind == AFX_OP_DECODE) {
        std::vector<void*> outs(count);
        for (uint32_t i = 0; i < count; ++i) outs[i] = ops[i].out_dev;
        return afx_decode_batch(descs.data(), containers.data(), outs.data(), count, stream, status_dev);
    }
    std::vector<uint32_t> rows(count), cols(count);
    std::vector<const uint16_t*> xs(count);
    std::vector<float*> ys(count);
    std::vector<void*> ws(count);
    std::vector<uint64_t> ws_bytes(count);
    for (uint32_t i = 0; i < count; ++i) {
        rows[i] = ops[i].rows;
        cols[i] = ops[i].cols;
        xs[i] = ops[i].x_dev;
        ys[i] = static_cast<float*>(ops[i].out_dev);
        ws[i] = ops[i].workspace_dev;
        ws_bytes[i] = ops[i].workspace_bytes;
    }
    return afx_decode_gemv_batch(descs.data(), containers.data(), rows.data(), cols.data(), xs.data(), ops[0].batch,
                                 ys.data(), ws.data(), ws_bytes.data(), count, stream, status_dev);
}

}  // namespace

extern "C" afx_status afx_stream_run(const afx_layer* layers, uint32_t n_layers, void* const* dev_bufs,
                                     uint32_t n_bufs, uint64_t buf_bytes, afx_stream_t compute_stream,
                                     afx_stream_t copy_stream, afx_stream_t d2h_stream, int32_t* status_dev) {
    if ((!layers && n_layers) || !dev_bufs || n_bufs < 2) return AFX_E_ARG;
    for (uint32_t k = 0; k < n_bufs; ++k)
        if (!dev_bufs[k] || !aligned256(dev_bufs[k])) return AFX_E_ARG;
    for (uint32_t l = 0; l < n_layers; ++l) {
        afx_status st = check_layer(layers[l], buf_bytes);
        if (st != AFX_OK) return st;
    }
    cudaStream_t compute = reinterpret_cast<cudaStream_t>(compute_stream);
    cudaStream_t copy = reinterpret_cast<cudaStream_t>(copy_stream);
    cudaStream_t d2h = d2h_stream ? reinterpret_cast<cudaStream_t>(d2h_stream) : copy;
    EventSet copied, consumed, entry;
    if (!copied.create(n_bufs) || !consumed.create(n_bufs) || !entry.create(1))
        return afx_fail(AFX_E_CUDA, "cudaEventCreateWithFlags", static_cast<int>(cudaGetLastError()));
    // The buffers may still be read by work an earlier call queued on the
    // compute stream: the first copy of this call waits for all of it.
    AFX_STREAM_TRY(cudaEventRecord(entry.ev[0], compute), "cudaEventRecord");
    AFX_STREAM_TRY(cudaStreamWaitEvent(copy, entry.ev[0], 0), "cudaStreamWaitEvent");

    // device outputs being copied back to the host, with the event that
    // marks the end of their layer's copies
    struct Returning {
        const uint8_t* begin;
        const uint8_t* end;
        size_t event;
    };
    std::vector<Returning> returning;
    EventSet returned;
    size_t n_returned = 0;
    for (uint32_t l = 0; l < n_layers; ++l)
        for (uint32_t i = 0; i < layers[l].n_ops; ++i)
            if (layers[l].ops[i].kind == AFX_OP_DECODE && layers[l].ops[i].out_host) {
                ++n_returned;
                break;
            }
    if (n_returned && !returned.create(n_returned))
        return afx_fail(AFX_E_CUDA, "cudaEventCreateWithFlags", static_cast<int>(cudaGetLastError()));
    size_t next_returned = 0;

    NvtxRange run_range("afx_stream_run");
    for (uint32_t l = 0; l < n_layers; ++l) {
        const afx_layer& L = layers[l];
        const uint32_t k = l % n_bufs;
        char name[48];
        snprintf(name, sizeof name, "afx layer %u: copy and ops", l);
        NvtxRange layer_range(name);
        uint8_t* buf = static_cast<uint8_t*>(dev_bufs[k]);
        if (l >= n_bufs) AFX_STREAM_TRY(cudaStreamWaitEvent(copy, consumed.ev[k], 0), "cudaStreamWaitEvent");
        if (L.blob_bytes)
            AFX_STREAM_TRY(cudaMemcpyAsync(buf, L.host_blob, L.blob_bytes, cudaMemcpyHostToDevice, copy),
                           "cudaMemcpyAsync");
        AFX_STREAM_TRY(cudaEventRecord(copied.ev[k], copy), "cudaEventRecord");
        AFX_STREAM_TRY(cudaStreamWaitEvent(compute, copied.ev[k], 0), "cudaStreamWaitEvent");
        // an output still being copied back by an earlier layer is not overwritten before that copy
        for (uint32_t i = 0; i < L.n_ops && !returning.empty(); ++i) {
            const afx_op& op = L.ops[i];
            const uint64_t bytes = op.kind == AFX_OP_GEMV ? uint64_t{4} * op.batch * op.rows
                                   : op.desc.format == AFX_FMT_E4M3 ? op.desc.n : op.desc.n * sizeof(uint16_t);
            const uint8_t* b = static_cast<const uint8_t*>(op.out_dev);
            for (const Returning& r : returning)
                if (bytes && b < r.end && r.begin < b + bytes)
                    AFX_STREAM_TRY(cudaStreamWaitEvent(compute, returned.ev[r.event], 0), "cudaStreamWaitEvent");
        }
        // consecutive ops of one kind (and one GEMV batch size) share a launch
        for (uint32_t i = 0; i < L.n_ops;) {
            uint32_t j = i + 1;
            while (j < L.n_ops && L.ops[j].kind == L.ops[i].kind &&
                   (L.ops[i].kind == AFX_OP_DECODE || L.ops[j].batch == L.ops[i].batch))
                ++j;
            const afx_status st = run_group(L.ops + i, j - i, buf, compute_stream, status_dev);
            if (st != AFX_OK) return st;
            i = j;
        }
        AFX_STREAM_TRY(cudaEventRecord(consumed.ev[k], compute), "cudaEventRecord");
        bool to_host = false;
        for (uint32_t i = 0; i < L.n_ops; ++i) to_host = to_host || (L.ops[i].kind == AFX_OP_DECODE && L.ops[i].out_host);
        if (to_host) {
            AFX_STREAM_TRY(cudaStreamWaitEvent(d2h, consumed.ev[k], 0), "cudaStreamWaitEvent");
            for (uint32_t i = 0; i < L.n_ops; ++i) {
                const afx_op& op = L.ops[i];
                if (op.kind != AFX_OP_DECODE || !op.out_host || op.desc.n == 0) continue;
                const uint64_t bytes = op.desc.format == AFX_FMT_E4M3 ? op.desc.n : op.desc.n * sizeof(uint16_t);
                AFX_STREAM_TRY(cudaMemcpyAsync(op.out_host, op.out_dev, bytes,
                                               cudaMemcpyDeviceToHost, d2h),
                               "cudaMemcpyAsync");
                const uint8_t* b = static_cast<const uint8_t*>(op.out_dev);
                returning.push_back({b, b + bytes, next_returned});
            }
            AFX_STREAM_TRY(cudaEventRecord(returned.ev[next_returned], d2h), "cudaEventRecord");
            ++next_returned;
        }
    }
    // later work on the compute stream (another call's ops included) comes
    // after the copies back have read their device outputs
    if (next_returned)
        AFX_STREAM_TRY(cudaStreamWaitEvent(compute, returned.ev[next_returned - 1], 0), "cudaStreamWaitEvent");
    return AFX_OK;
}
