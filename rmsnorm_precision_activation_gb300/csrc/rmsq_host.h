// rmsq_host.h -- host-side plumbing shared by the library's translation units: the launch plan
// and the per-mode dispatch entry points (each mode's kernels live in their own .cu file so the
// build compiles them in parallel).
#pragma once

#include <cuda_runtime.h>

#include "rmsq_device.cuh"

namespace rmsq {

struct Plan {
    int mode;          // MODE_*
    int dt;            // DT_*
    bool res;          // residual present
    int vpt;           // 16-byte vectors per thread per row: 1, 2, 4 or 8
    int sched;         // SCHED_PIPE, SCHED_REG, SCHED_WARP or SCHED_CLUSTER
    int threads;       // CTA size (multiple of 32); SCHED_WARP: 32 x rows in flight per CTA
    int stages;        // ring depth (SCHED_PIPE: per CTA, SCHED_WARP: per warp)
    int smem;          // dynamic shared memory bytes
    int ctas_per_sm;   // cap on resident CTAs per SM (0: occupancy limit)
    bool w16;          // 16-bit input and weight_offset 0: products from packed halves
    int cluster = 1;   // SCHED_CLUSTER: CTAs per cluster (each takes 1/cluster of every row)
};

// Launch `fn` (a rmsq_row_kernel instantiation) with the plan: sets the dynamic shared memory
// limit once per function and device, sizes a persistent grid of CTAs per SM x SMs (no more CTAs
// than it takes to give each one a row; a row-per-warp CTA takes one row per warp).
cudaError_t run_kernel(const void* fn, const Plan& plan, const Params& p, cudaStream_t stream);

// Per-mode dispatch on (dtype, residual, vpt, schedule). Each quantisation mode's kernels are
// split over two translation units, rmsq_<mode>.cu (no residual) and rmsq_<mode>_res.cu, so
// the build compiles them in parallel (the amax pre-pass likewise).
cudaError_t dispatch_fp8_plain(const Plan& plan, const Params& p, cudaStream_t stream);
cudaError_t dispatch_fp8_res(const Plan& plan, const Params& p, cudaStream_t stream);
cudaError_t dispatch_nvfp4_plain(const Plan& plan, const Params& p, cudaStream_t stream);
cudaError_t dispatch_nvfp4_res(const Plan& plan, const Params& p, cudaStream_t stream);
cudaError_t dispatch_mxfp4_plain(const Plan& plan, const Params& p, cudaStream_t stream);
cudaError_t dispatch_mxfp4_res(const Plan& plan, const Params& p, cudaStream_t stream);
cudaError_t dispatch_amax_plain(const Plan& plan, const Params& p, cudaStream_t stream);
cudaError_t dispatch_amax_res(const Plan& plan, const Params& p, cudaStream_t stream);

inline cudaError_t dispatch_fp8(const Plan& pl, const Params& p, cudaStream_t st)
{
    return pl.res ? dispatch_fp8_res(pl, p, st) : dispatch_fp8_plain(pl, p, st);
}
inline cudaError_t dispatch_nvfp4(const Plan& pl, const Params& p, cudaStream_t st)
{
    return pl.res ? dispatch_nvfp4_res(pl, p, st) : dispatch_nvfp4_plain(pl, p, st);
}
inline cudaError_t dispatch_mxfp4(const Plan& pl, const Params& p, cudaStream_t st)
{
    return pl.res ? dispatch_mxfp4_res(pl, p, st) : dispatch_mxfp4_plain(pl, p, st);
}
inline cudaError_t dispatch_amax(const Plan& pl, const Params& p, cudaStream_t st)
{
    return pl.res ? dispatch_amax_res(pl, p, st) : dispatch_amax_plain(pl, p, st);
}

// Instantiates the dispatch switch of one mode, for one residual case (RESV), inside a .cu file.
#define RMSQ_DEFINE_DISPATCH_FOR(NAME, MODE, RESV) RMSQ_DEFINE_DISPATCH_IMPL(NAME, MODE, !(RESV), RESV)
#define RMSQ_DEFINE_DISPATCH_IMPL(NAME, MODE, PLAIN_OK, RES_OK)                                  \
    template <int DT, bool RES, int VPT, int SCHED, bool W16>                                     \
    static cudaError_t NAME##_go(const Plan& pl, const Params& p, cudaStream_t st)                \
    {                                                                                             \
        return run_kernel(                                                                        \
            reinterpret_cast<const void*>(&rmsq_row_kernel<DT, RES, MODE, VPT, SCHED, W16>), pl,  \
            p, st);                                                                               \
    }                                                                                             \
    template <int DT, bool RES, int VPT, int SCHED>                                               \
    static cudaError_t NAME##_w16(const Plan& pl, const Params& p, cudaStream_t st)               \
    {                                                                                             \
        if constexpr (DT != DT_F32) {                                                             \
            if (pl.w16) return NAME##_go<DT, RES, VPT, SCHED, true>(pl, p, st);                   \
        }                                                                                         \
        return NAME##_go<DT, RES, VPT, SCHED, false>(pl, p, st);                                  \
    }                                                                                             \
    template <int DT, bool RES, int VPT>                                                          \
    static cudaError_t NAME##_sched(const Plan& pl, const Params& p, cudaStream_t st)             \
    {                                                                                             \
        switch (pl.sched) {                                                                       \
        case SCHED_PIPE: return NAME##_w16<DT, RES, VPT, SCHED_PIPE>(pl, p, st);                  \
        case SCHED_WARP: return NAME##_w16<DT, RES, VPT, SCHED_WARP>(pl, p, st);                  \
        case SCHED_CLUSTER:                                                                       \
            if constexpr (VPT >= 4) return NAME##_w16<DT, RES, VPT, SCHED_CLUSTER>(pl, p, st);    \
            return cudaErrorInvalidConfiguration;                                                 \
        default: return NAME##_w16<DT, RES, VPT, SCHED_REG>(pl, p, st);                           \
        }                                                                                         \
    }                                                                                             \
    template <int DT, bool RES>                                                                   \
    static cudaError_t NAME##_vpt(const Plan& pl, const Params& p, cudaStream_t st)               \
    {                                                                                             \
        switch (pl.vpt) {                                                                         \
        case 1: return NAME##_sched<DT, RES, 1>(pl, p, st);                                       \
        case 2: return NAME##_sched<DT, RES, 2>(pl, p, st);                                       \
        case 4: return NAME##_sched<DT, RES, 4>(pl, p, st);                                       \
        default: return NAME##_sched<DT, RES, 8>(pl, p, st);                                      \
        }                                                                                         \
    }                                                                                             \
    template <int DT>                                                                             \
    static cudaError_t NAME##_res(const Plan& pl, const Params& p, cudaStream_t st)               \
    {                                                                                             \
        if (pl.res) {                                                                             \
            if constexpr (RES_OK) return NAME##_vpt<DT, true>(pl, p, st);                         \
        } else {                                                                                  \
            if constexpr (PLAIN_OK) return NAME##_vpt<DT, false>(pl, p, st);                      \
        }                                                                                         \
        return cudaErrorInvalidValue;                                                             \
    }                                                                                             \
    cudaError_t NAME(const Plan& pl, const Params& p, cudaStream_t st)                            \
    {                                                                                             \
        switch (pl.dt) {                                                                          \
        case DT_BF16: return NAME##_res<DT_BF16>(pl, p, st);                                      \
        case DT_FP16: return NAME##_res<DT_FP16>(pl, p, st);                                      \
        default: return NAME##_res<DT_F32>(pl, p, st);                                            \
        }                                                                                         \
    }

}  // namespace rmsq
