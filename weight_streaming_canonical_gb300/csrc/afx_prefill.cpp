// Prefill products: Y = X W^T for many token vectors at once.
//
// "Memory requirements of language model inference on a consumer GPU",
// section "Loading one part of the model at a time": the prefill stage
// processes the whole prompt before decoding produces tokens one by one.
// With hundreds of tokens the product is a dense contraction for the
// tensor cores, while the weights' side is bounded by the restore, which is
// limited by its instruction rate rather than by HBM.  So the matrix is
// restored into scratch memory by the restore kernel and multiplied by
// cuBLAS (BF16 or FP16 inputs, float32 accumulation).  A list of matrices is either
// pipelined (the restore of the next on its own stream while the current one
// is multiplied, ordered by CUDA events only) or restored in one launch and
// then multiplied: the restore kernel holds a whole SM per CTA, so where it
// fills every SM the two streams cannot share the GPU and the one-launch
// form, which saves the per-launch ramps of small matrices, is the faster.
#include <cublas_v2.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <vector>

#include "afx_internal.h"

namespace {

#define AFX_PF_CUDA(call, what)                                          \
    do {                                                                 \
        const cudaError_t e_ = (call);                                   \
        if (e_ != cudaSuccess) return afx_fail(AFX_E_CUDA, (what), e_);  \
    } while (0)

#define AFX_PF_CUBLAS(call, what)                                         \
    do {                                                                  \
        if ((call) != CUBLAS_STATUS_SUCCESS) return afx_fail(AFX_E_CUDA, (what), 0); \
    } while (0)

// One cuBLAS handle per host thread and device, created on first use and
// kept for the life of the process (handles are not destroyed at exit: the
// CUDA context may already be gone then).
constexpr int kMaxDevices = 64;
thread_local cublasHandle_t t_handles[kMaxDevices] = {};

afx_status handle_for_current_device(cublasHandle_t* out) {
    int dev = -1;
    AFX_PF_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return afx_fail(AFX_E_CUDA, "device ordinal out of range", 0);
    if (!t_handles[dev]) AFX_PF_CUBLAS(cublasCreate(&t_handles[dev]), "cublasCreate");
    *out = t_handles[dev];
    return AFX_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

afx_status check_product(const afx_desc& d, const void* container, uint32_t rows, uint32_t cols,
                         const uint16_t* x, uint32_t n_tokens, const float* y) {
    const afx_status st = afx_check_desc(&d);
    if (st != AFX_OK) return afx_fail(st, "invalid container description", 0);
    if (d.format != AFX_FMT_BF16 && d.format != AFX_FMT_FP16)
        return afx_fail(AFX_E_ARG, "prefill takes BF16 or FP16 containers", 0);
    if (!container || !x || !y) return afx_fail(AFX_E_ARG, "null pointer", 0);
    if (rows == 0 || cols == 0 || n_tokens == 0 || static_cast<uint64_t>(rows) * cols != d.n)
        return afx_fail(AFX_E_ARG, "rows * cols must equal n and n_tokens must be positive", 0);
    if (rows > INT_MAX || cols > INT_MAX || n_tokens > INT_MAX)
        return afx_fail(AFX_E_ARG, "dimensions must fit in int", 0);
    if (!aligned16(x) || !aligned16(y)) return afx_fail(AFX_E_ARG, "x and y must be 16-byte aligned", 0);
    return AFX_OK;
}

// y[t][r] = sum_c w[r][c] x[t][c]: in cuBLAS's column-major terms
// y^T (rows x n) = (w as cols x rows)^T * (x as cols x n).  w and x are
// both BF16 or both FP16 (the container's format).
afx_status product(cublasHandle_t h, const uint16_t* w, const uint16_t* x, float* y, uint32_t rows, uint32_t cols,
                   uint32_t n_tokens, uint32_t format, void* workspace, cudaStream_t s) {
    const cudaDataType_t type = format == AFX_FMT_FP16 ? CUDA_R_16F : CUDA_R_16BF;
    AFX_PF_CUBLAS(cublasSetStream(h, s), "cublasSetStream");
    AFX_PF_CUBLAS(cublasSetWorkspace(h, workspace, AFX_PREFILL_GEMM_WORKSPACE_BYTES), "cublasSetWorkspace");
    const float alpha = 1.0f, beta = 0.0f;
    AFX_PF_CUBLAS(cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, static_cast<int>(rows), static_cast<int>(n_tokens),
                               static_cast<int>(cols), &alpha, w, type, static_cast<int>(cols), x, type,
                               static_cast<int>(cols), &beta, y, CUDA_R_32F, static_cast<int>(rows),
                               CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT),
                  "cublasGemmEx");
    return AFX_OK;
}

struct Events {
    std::vector<cudaEvent_t> ev;
    ~Events() {
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

}  // namespace

extern "C" afx_status afx_prefill(const afx_desc* desc, const void* container_dev, uint32_t rows, uint32_t cols,
                                  const uint16_t* x_dev, uint32_t n_tokens, float* y_dev, uint16_t* w_scratch_dev,
                                  void* gemm_workspace_dev, afx_stream_t stream, int32_t* status_dev) {
    if (!desc) return afx_fail(AFX_E_ARG, "null description", 0);
    afx_status st = check_product(*desc, container_dev, rows, cols, x_dev, n_tokens, y_dev);
    if (st != AFX_OK) return st;
    if (!w_scratch_dev || !gemm_workspace_dev || !aligned16(w_scratch_dev))
        return afx_fail(AFX_E_ARG, "scratch and workspace must be 16-byte aligned device memory", 0);
    cublasHandle_t h;
    st = handle_for_current_device(&h);
    if (st != AFX_OK) return st;
    st = afx_decode(desc, container_dev, w_scratch_dev, stream, status_dev);
    if (st != AFX_OK) return st;
    return product(h, w_scratch_dev, x_dev, y_dev, rows, cols, n_tokens, desc->format, gemm_workspace_dev,
                   reinterpret_cast<cudaStream_t>(stream));
}

extern "C" afx_status afx_prefill_batch(const afx_desc* descs, const void* const* containers_dev, const uint32_t* rows,
                                        const uint32_t* cols, const uint16_t* const* xs_dev, uint32_t n_tokens,
                                        float* const* ys_dev, uint32_t count, uint16_t* const* w_scratch_dev,
                                        void* gemm_workspace_dev, afx_stream_t restore_stream,
                                        afx_stream_t gemm_stream, int32_t* status_dev) {
    if (count && (!descs || !containers_dev || !rows || !cols || !xs_dev || !ys_dev))
        return afx_fail(AFX_E_ARG, "null array", 0);
    if (!w_scratch_dev || !w_scratch_dev[0] || !gemm_workspace_dev || !aligned16(w_scratch_dev[0]) ||
        (w_scratch_dev[1] && !aligned16(w_scratch_dev[1])))
        return afx_fail(AFX_E_ARG, "16-byte aligned scratch and a workspace are needed", 0);
    for (uint32_t i = 0; i < count; ++i) {
        const afx_status st = check_product(descs[i], containers_dev[i], rows[i], cols[i], xs_dev[i], n_tokens, ys_dev[i]);
        if (st != AFX_OK) return st;
    }
    cublasHandle_t h;
    afx_status st = handle_for_current_device(&h);
    if (st != AFX_OK) return st;
    cudaStream_t rs = reinterpret_cast<cudaStream_t>(restore_stream);
    cudaStream_t gs = reinterpret_cast<cudaStream_t>(gemm_stream);
    if (!w_scratch_dev[1]) {
        // every matrix restored in one launch into w_scratch_dev[0] (back to
        // back, each at a 256-byte boundary), then the products in order
        std::vector<void*> outs(count);
        uint64_t off = 0;
        for (uint32_t i = 0; i < count; ++i) {
            outs[i] = w_scratch_dev[0] + off / 2;
            off += (descs[i].n * 2 + 255) / 256 * 256;
        }
        st = afx_decode_batch(descs, containers_dev, outs.data(), count, gemm_stream, status_dev);
        if (st != AFX_OK) return st;
        for (uint32_t i = 0; i < count; ++i) {
            st = product(h, static_cast<const uint16_t*>(outs[i]), xs_dev[i], ys_dev[i], rows[i], cols[i], n_tokens,
                         descs[i].format, gemm_workspace_dev, gs);
            if (st != AFX_OK) return st;
        }
        return AFX_OK;
    }
    Events restored, consumed, entry;
    if (!restored.create(count ? count : 1) || !consumed.create(2) || !entry.create(1))
        return afx_fail(AFX_E_CUDA, "cudaEventCreateWithFlags", static_cast<int>(cudaGetLastError()));
    // products that an earlier call queued may still read the scratch buffers
    AFX_PF_CUDA(cudaEventRecord(entry.ev[0], gs), "cudaEventRecord");
    AFX_PF_CUDA(cudaStreamWaitEvent(rs, entry.ev[0], 0), "cudaStreamWaitEvent");
    for (uint32_t i = 0; i < count; ++i) {
        const uint32_t k = i % 2;
        if (i >= 2) AFX_PF_CUDA(cudaStreamWaitEvent(rs, consumed.ev[k], 0), "cudaStreamWaitEvent");
        st = afx_decode(&descs[i], containers_dev[i], w_scratch_dev[k], restore_stream, status_dev);
        if (st != AFX_OK) return st;
        AFX_PF_CUDA(cudaEventRecord(restored.ev[i], rs), "cudaEventRecord");
        AFX_PF_CUDA(cudaStreamWaitEvent(gs, restored.ev[i], 0), "cudaStreamWaitEvent");
        st = product(h, w_scratch_dev[k], xs_dev[i], ys_dev[i], rows[i], cols[i], n_tokens, descs[i].format,
                     gemm_workspace_dev, gs);
        if (st != AFX_OK) return st;
        AFX_PF_CUDA(cudaEventRecord(consumed.ev[k], gs), "cudaEventRecord");
    }
    return AFX_OK;
}
