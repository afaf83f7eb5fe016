// launch.cuh -- host-side launch of one tile-kernel instantiation.
#pragma once

#include <atomic>

#include "kernel.cuh"

namespace mx {

// Launch mxfp8_tile_kernel<OP, MODE> (activation ACT, evaluated by the
// policy policy_of picks) on `grid` CTAs.  The dynamic shared memory limit of
// the instantiation is raised once per device.
template <int OP, int MODE, int ACT, bool GRP>
cudaError_t launch_tiles(const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,
                         cudaStream_t stream, int device)
{
    constexpr int kTM = TuningFor<OP, MODE, ACT, GRP>::kTM;
    constexpr int kStages = TuningFor<OP, MODE, ACT, GRP>::kStages;
    constexpr int kCtas = TuningFor<OP, MODE, ACT, GRP>::kCtas;
    constexpr int kGroup = TuningFor<OP, MODE, ACT, GRP>::kGroup;
    constexpr int kPol = policy_of<OP, MODE, ACT, GRP>();
    constexpr size_t kSmem = smem_bytes<OP, kTM, kStages, kGroup, GRP>();
    constexpr size_t kStatic = static_smem_bytes<OP, kPol>();
    static_assert(kSmem + kStatic <= 227 * 1024, "shared memory per CTA");
    static_assert(kCtas * (kSmem + kStatic + 1024) <= 228 * 1024, "shared memory per SM");
    auto kern = mxfp8_tile_kernel<OP, MODE, kTM, kStages, kCtas, kGroup, kPol, GRP>;
    static std::atomic<unsigned long long> attr_done{0};
    const unsigned long long bit = 1ull << (device & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmem));
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    void *args[] = {const_cast<CUtensorMap *>(&maps[0]), const_cast<CUtensorMap *>(&maps[1]),
                    const_cast<CUtensorMap *>(&maps[2]), const_cast<KernelArgs *>(&a)};
    return cudaLaunchKernel(reinterpret_cast<const void *>(kern), dim3(grid),
                            dim3((warps_of<kTM>() + 1) * 32), args, kSmem, stream);
}

// tile rows, resident CTAs per SM and row-scale group of the instantiation
// the host will launch (GEGLU's backward "both" with plain scales has its
// own)
struct LaunchShape {
    int tile_rows, ctas_per_sm, group;
};
template <int OP, int MODE, int ACT, bool GRP>
constexpr LaunchShape shape_of()
{
    using T = TuningFor<OP, MODE, ACT, GRP>;
    return {T::kTM, T::kCtas, T::kGroup};
}
inline LaunchShape launch_shape(int op, int mode, int act, bool grouped)
{
    if (act == kGelu && op == kBwd && mode == kBoth && !grouped) return shape_of<kBwd, kBoth, kGelu, false>();
    switch (op * 4 + mode) {
    case kQuant * 4 + kRow: return shape_of<kQuant, kRow, kSilu, false>();
    case kQuant * 4 + kCol: return shape_of<kQuant, kCol, kSilu, false>();
    case kQuant * 4 + kBoth: return shape_of<kQuant, kBoth, kSilu, false>();
    case kFwd * 4 + kRow: return shape_of<kFwd, kRow, kSilu, false>();
    case kFwd * 4 + kCol: return shape_of<kFwd, kCol, kSilu, false>();
    case kFwd * 4 + kBoth: return shape_of<kFwd, kBoth, kSilu, false>();
    case kBwd * 4 + kRow: return shape_of<kBwd, kRow, kSilu, false>();
    case kBwd * 4 + kCol: return shape_of<kBwd, kCol, kSilu, false>();
    default: return shape_of<kBwd, kBoth, kSilu, false>();
    }
}

// per-op (and activation) dispatch over the scale mode, one translation unit
// each
#define MX_DECLARE_LAUNCH(NAME)                                                                  \
    cudaError_t NAME(int mode, const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,      \
                     cudaStream_t stream, int device);                                           \
    cudaError_t NAME##_grouped(int mode, const CUtensorMap (&maps)[3], const KernelArgs &a,      \
                               int grid, cudaStream_t stream, int device);
MX_DECLARE_LAUNCH(launch_quant)
MX_DECLARE_LAUNCH(launch_fwd)
MX_DECLARE_LAUNCH(launch_bwd)
MX_DECLARE_LAUNCH(launch_fwd_gelu)
MX_DECLARE_LAUNCH(launch_bwd_gelu)
#undef MX_DECLARE_LAUNCH

// one translation unit per (op, activation) and per plain / grouped scales
#define MX_DEFINE_LAUNCH(NAME, OP, ACT, GRP)                                                     \
    cudaError_t NAME(int mode, const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,      \
                     cudaStream_t stream, int device)                                            \
    {                                                                                            \
        switch (mode) {                                                                          \
        case kRow: return launch_tiles<OP, kRow, ACT, GRP>(maps, a, grid, stream, device);       \
        case kCol: return launch_tiles<OP, kCol, ACT, GRP>(maps, a, grid, stream, device);       \
        case kBoth: return launch_tiles<OP, kBoth, ACT, GRP>(maps, a, grid, stream, device);     \
        default: return cudaErrorInvalidValue;                                                   \
        }                                                                                        \
    }

}  // namespace mx
