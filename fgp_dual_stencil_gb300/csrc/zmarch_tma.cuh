// ZMARCH_TMA variant: x-y tile marching along z with TMA-staged planes.
// (Interface only; the kernel is not built yet, so the variant reports
// itself unsupported.)
#pragma once

#include "fgp_kernels.cuh"

namespace tvfgp {

struct ZmarchPlan {
    int ok;
};

struct ZmarchArgs {
    StepArgs a;
    int *err;
};

inline int zmarch_plan(int, int, int, ZmarchPlan *plan)
{
    plan->ok = 0;
    return 0;
}
inline bool zmarch_supported(int, int, int) { return false; }
inline const void *zmarch_kernel() { return nullptr; }
inline int zmarch_threads() { return 0; }
inline dim3 zmarch_grid(const ZmarchPlan &) { return dim3(1, 1, 1); }
inline size_t zmarch_smem_bytes() { return 0; }
inline void zmarch_fill(const ZmarchPlan &, const StepArgs &a, int *err, ZmarchArgs &za)
{
    za.a = a;
    za.err = err;
}

}  // namespace tvfgp
