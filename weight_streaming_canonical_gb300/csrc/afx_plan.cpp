// Residency planning: where each tensor lives during inference on one GPU.
//
// "Why Weight Offloading Slows Inference", section "Lossless compression:
// fewer bytes to read, more work to unpack": a step pays for the bytes it
// reads plus t_unpack (Eq. (1)), and streaming compressed weights pays only
// when (S - S_disk) / b > t_unpack (Eq. (2)).  "Memory requirements of
// language model inference on a consumer GPU", section "Loading one part of
// the model at a time": what does not fit in device memory is loaded when
// it is needed.
//
// Each tensor has four placements, each a (resident bytes, seconds per
// step) pair; the plan minimises the sum of the per-step costs with the
// resident bytes within the budget.  That is a multiple-choice knapsack,
// solved exactly by dynamic programming over memory counted in whole units
// of budget / U (sizes rounded up, so a plan always fits).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <vector>

#include "afx_internal.h"

namespace {

constexpr uint32_t kMaxTensors = 65536;
constexpr uint64_t kMaxUnits = 65536;         // memory resolution: budget / 65536
constexpr uint64_t kMaxCells = uint64_t{1} << 25;  // tensors x units kept for the backtrack

struct Option {
    uint64_t units;
    double ms;
    uint32_t placement;
};

}  // namespace

extern "C" afx_status afx_plan_residency(const afx_plan_tensor* tensors, uint32_t n, uint64_t device_budget_bytes,
                                         const afx_plan_rates* rates, uint32_t* placement_out, double* step_ms_out,
                                         uint64_t* resident_bytes_out) {
    if (!tensors || !rates || !placement_out || n == 0 || n > kMaxTensors) return AFX_E_ARG;
    if (!(rates->link_gbs > 0) || !(rates->restore_gbs > 0) || !std::isfinite(rates->link_gbs) ||
        !std::isfinite(rates->restore_gbs))
        return AFX_E_ARG;
    // memory units: fine enough to tell the tensors apart, coarse enough
    // that tensors x units fits the backtrack table
    const uint64_t units_cap = std::max<uint64_t>(1, std::min<uint64_t>(kMaxUnits, kMaxCells / n));
    const uint64_t unit = std::max<uint64_t>(1, (device_budget_bytes + units_cap - 1) / units_cap);
    const uint64_t cap = device_budget_bytes / unit;  // whole units within the budget
    const double b = rates->link_gbs * 1e6, r = rates->restore_gbs * 1e6;  // bytes per ms

    // options of each tensor: the two resident ones and the better streamed one
    std::vector<Option> opts(static_cast<size_t>(n) * 3);
    for (uint32_t i = 0; i < n; ++i) {
        const double S = static_cast<double>(tensors[i].decoded_bytes);
        const double C = static_cast<double>(tensors[i].compressed_bytes);
        const double t_unpack = S / r;
        const double stream_c = rates->overlapped ? std::max(C / b, t_unpack) : C / b + t_unpack;
        const double stream_raw = S / b;
        Option* o = &opts[static_cast<size_t>(i) * 3];
        o[0] = {(tensors[i].decoded_bytes + unit - 1) / unit, 0.0, AFX_RESIDENT_DECODED};
        o[1] = {(tensors[i].compressed_bytes + unit - 1) / unit, t_unpack, AFX_RESIDENT_COMPRESSED};
        // Eq. (2): stream the container only when that beats the raw copy
        o[2] = stream_c < stream_raw ? Option{0, stream_c, AFX_STREAM_COMPRESSED}
                                     : Option{0, stream_raw, AFX_STREAM_RAW};
    }

    // best[m]: least time of the tensors so far within m units; choice[i][m]
    // the option tensor i takes there
    std::vector<double> best(cap + 1, 0.0), next(cap + 1);
    std::vector<uint8_t> choice(static_cast<size_t>(n) * (cap + 1));
    for (uint32_t i = 0; i < n; ++i) {
        const Option* o = &opts[static_cast<size_t>(i) * 3];
        uint8_t* ch = &choice[static_cast<size_t>(i) * (cap + 1)];
        for (uint64_t m = 0; m <= cap; ++m) {
            double t = best[m] + o[2].ms;
            uint8_t k = 2;
            for (uint8_t j = 0; j < 2; ++j) {
                if (o[j].units > m) continue;
                const double tj = best[m - o[j].units] + o[j].ms;
                if (tj < t) {
                    t = tj;
                    k = j;
                }
            }
            next[m] = t;
            ch[m] = k;
        }
        best.swap(next);
    }
    // walk back from the full budget
    uint64_t m = cap, resident = 0;
    for (uint32_t i = n; i-- > 0;) {
        const uint8_t k = choice[static_cast<size_t>(i) * (cap + 1) + m];
        const Option& o = opts[static_cast<size_t>(i) * 3 + k];
        placement_out[i] = o.placement;
        m -= o.units;
        if (o.placement == AFX_RESIDENT_DECODED) resident += tensors[i].decoded_bytes;
        if (o.placement == AFX_RESIDENT_COMPRESSED) resident += tensors[i].compressed_bytes;
    }
    if (step_ms_out) *step_ms_out = best[cap];
    if (resident_bytes_out) *resident_bytes_out = resident;
    return AFX_OK;
}
