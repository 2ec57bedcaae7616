// Internal declarations shared by the afx host and device translation units.
#pragma once

#include <stdint.h>

#include "../../include/afx.h"

#define AFX_MAGIC 0x31584641u

// Decoder geometry: one CTA thread per chunk, so a block is one CTA tile.
#define AFX_DECODE_THREADS 512

#ifdef __cplusplus
// GEMV workspace: per sub-tile of 32 chunks (16 per block), its first
// weight index and two row partials per batch row.
inline uint64_t afx_gemv_workspace_bytes(uint64_t n_blocks, uint32_t batch) {
    uint64_t b = n_blocks * 16ull * (sizeof(uint64_t) + 2ull * batch * sizeof(float));
    return b < 16 ? 16 : (b + 15) / 16 * 16;
}
#endif

#ifdef __cplusplus
extern "C" {
#endif

// Checks that a description is self-consistent (geometry, section layout,
// code lengths).  Returns AFX_OK, AFX_E_ARG or AFX_E_FORMAT.
__attribute__((visibility("hidden"))) afx_status afx_check_desc(const afx_desc* d);

// Records a message for afx_last_error() on this thread and returns status.
__attribute__((visibility("hidden"))) afx_status afx_fail(afx_status status, const char* what, int cuda_error);

#ifdef __cplusplus
}
#endif
