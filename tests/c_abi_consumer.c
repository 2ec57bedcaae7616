/*
 * A plain C program that uses libafx through include/afx.h alone: the test
 * that the boundary is a C ABI (no C++, no Python, no torch types).
 *
 * Host part (always): builds a code for a few thousand BF16 weights, plans
 * and writes the container, parses its header back and compares the two
 * descriptions, and asks the residency planner for a placement.
 * Device part (argument "gpu"): copies the container to device memory with
 * the CUDA runtime, restores it with afx_decode, waits with afx_sync and
 * compares every weight.
 * Prints "ok" and exits 0 on success; prints the failing step otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "afx.h"

#ifdef AFX_CONSUMER_GPU
#include <cuda_runtime.h>
#endif

#define N 5000u

static int fail(const char* what, int status) {
    printf("failed: %s (status %d: %s)\n", what, status, afx_status_string((afx_status)status));
    return 1;
}

/* A deterministic mix of BF16 patterns: a few common exponents, every sign
   and mantissa, some zeros. */
static void make_weights(uint16_t* w, uint32_t n) {
    uint32_t x = 12345u;
    for (uint32_t i = 0; i < n; ++i) {
        x = x * 1664525u + 1013904223u;
        const uint32_t exponent = 118u + ((x >> 8) % 7u);
        const uint32_t sign = (x >> 20) & 1u, mantissa = (x >> 24) & 0x7Fu;
        w[i] = (uint16_t)(i % 97u == 0u ? 0u : (sign << 15) | (exponent << 7) | mantissa);
    }
}

int main(int argc, char** argv) {
    static uint16_t w[N];
    make_weights(w, N);

    afx_code code;
    afx_status st = afx_build_code(w, N, AFX_MAX_CODE_LEN, &code);
    if (st != AFX_OK) return fail("afx_build_code", st);
    afx_desc desc;
    st = afx_encode_bound(N, &code, 0, 0, &desc);
    if (st != AFX_OK) return fail("afx_encode_bound", st);
    uint8_t* container = (uint8_t*)malloc(desc.container_bytes);
    if (!container) return fail("malloc", 0);
    st = afx_encode(w, N, &code, &desc, container, desc.container_bytes);
    if (st != AFX_OK) return fail("afx_encode", st);
    afx_desc parsed;
    st = afx_parse_header(container, desc.container_bytes, &parsed);
    if (st != AFX_OK) return fail("afx_parse_header", st);
    if (memcmp(&parsed, &desc, sizeof desc) != 0) return fail("parsed description differs", 0);
    if (desc.format != AFX_FMT_BF16 || desc.n != N) return fail("description fields", 0);

    afx_plan_tensor tensors[2] = {{2u * N, desc.container_bytes}, {2u * N, desc.container_bytes}};
    afx_plan_rates rates = {200.0, 2000.0, 1u, 0u};
    uint32_t placement[2];
    double step_ms = -1.0;
    uint64_t resident = 0;
    st = afx_plan_residency(tensors, 2, 4u * N, &rates, placement, &step_ms, &resident);
    if (st != AFX_OK) return fail("afx_plan_residency", st);
    if (resident > 4u * N || step_ms < 0.0) return fail("plan result", 0);

    if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
#ifdef AFX_CONSUMER_GPU
        void *dev_container = NULL, *dev_out = NULL, *dev_status = NULL;
        if (cudaMalloc(&dev_container, desc.container_bytes) != cudaSuccess ||
            cudaMalloc(&dev_out, 2u * N) != cudaSuccess || cudaMalloc(&dev_status, sizeof(int32_t)) != cudaSuccess)
            return fail("cudaMalloc", 0);
        if (cudaMemcpy(dev_container, container, desc.container_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemset(dev_status, 0, sizeof(int32_t)) != cudaSuccess)
            return fail("cudaMemcpy", 0);
        st = afx_decode(&desc, dev_container, dev_out, NULL, (int32_t*)dev_status);
        if (st != AFX_OK) return fail("afx_decode", st);
        int32_t word = -1;
        st = afx_sync(NULL, 10000u, (const int32_t*)dev_status, &word);
        if (st != AFX_OK || word != 0) return fail("afx_sync", st);
        static uint16_t back[N];
        if (cudaMemcpy(back, dev_out, 2u * N, cudaMemcpyDeviceToHost) != cudaSuccess) return fail("cudaMemcpy back", 0);
        if (memcmp(back, w, sizeof back) != 0) return fail("restored weights differ", 0);
        cudaFree(dev_container);
        cudaFree(dev_out);
        cudaFree(dev_status);
#else
        return fail("built without the CUDA runtime", 0);
#endif
    }
    free(container);
    printf("ok\n");
    return 0;
}
