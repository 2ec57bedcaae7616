// Bounded host wait and status read-back.
//
// The library never blocks the host on its own: every call enqueues work
// and returns.  A caller that must know when that work is done, and
// whether the kernels flagged a corrupt container, calls afx_sync: it
// records an event behind the queued work and polls it against a
// wall-clock limit, so a stream that never finishes turns into
// AFX_E_TIMEOUT instead of a host thread that hangs.  The pages have no
// counterpart; this is the library's failure detection.
#include <cuda_runtime.h>

#include <chrono>
#include <cstdint>
#include <thread>

#include "afx_internal.h"

namespace {

// Polls ev until it completes, for at most `limit` (no limit when
// unlimited).  Returns AFX_OK, AFX_E_TIMEOUT or AFX_E_CUDA.
afx_status poll_event(cudaEvent_t ev, std::chrono::steady_clock::time_point deadline, bool unlimited) {
    for (unsigned spins = 0;; ++spins) {
        const cudaError_t q = cudaEventQuery(ev);
        if (q == cudaSuccess) return AFX_OK;
        if (q != cudaErrorNotReady) return afx_fail(AFX_E_CUDA, "cudaEventQuery", q);
        if (!unlimited && std::chrono::steady_clock::now() >= deadline) return AFX_E_TIMEOUT;
        if (spins < 64)
            std::this_thread::yield();
        else
            std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

struct Event {
    cudaEvent_t ev = nullptr;
    ~Event() {
        if (ev) cudaEventDestroy(ev);
    }
};

}  // namespace

extern "C" afx_status afx_sync(afx_stream_t stream, uint32_t timeout_ms, const int32_t* status_dev,
                               int32_t* status_out) {
    if (status_out) *status_out = 0;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool unlimited = timeout_ms == 0;
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
    Event done;
    cudaError_t e = cudaEventCreateWithFlags(&done.ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return afx_fail(AFX_E_CUDA, "cudaEventCreateWithFlags", e);
    e = cudaEventRecord(done.ev, s);
    if (e != cudaSuccess) return afx_fail(AFX_E_CUDA, "cudaEventRecord", e);
    afx_status st = poll_event(done.ev, deadline, unlimited);
    if (st != AFX_OK || !status_dev) return st;
    // the queued work is done: read the status word behind it, still bounded
    int32_t word = 0;
    e = cudaMemcpyAsync(&word, status_dev, sizeof word, cudaMemcpyDefault, s);
    if (e != cudaSuccess) return afx_fail(AFX_E_CUDA, "cudaMemcpyAsync", e);
    e = cudaEventRecord(done.ev, s);
    if (e != cudaSuccess) return afx_fail(AFX_E_CUDA, "cudaEventRecord", e);
    st = poll_event(done.ev, deadline, unlimited);
    if (st != AFX_OK) return st;
    if (status_out) *status_out = word;
    return word != 0 ? AFX_E_CORRUPT : AFX_OK;
}
