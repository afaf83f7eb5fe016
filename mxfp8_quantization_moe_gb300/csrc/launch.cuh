// launch.cuh -- host-side launch of one tile-kernel instantiation.
#pragma once

#include <atomic>

#include "kernel.cuh"

namespace mx {

// Launch mxfp8_tile_kernel<OP, MODE> on `grid` CTAs.  The dynamic shared
// memory limit of the instantiation is raised once per device.
template <int OP, int MODE>
cudaError_t launch_tiles(const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,
                         cudaStream_t stream, int device)
{
    constexpr int kTM = Tuning<OP, MODE>::kTM;
    constexpr int kStages = Tuning<OP, MODE>::kStages;
    constexpr size_t kSmem = smem_bytes<OP, kTM, kStages>();
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    auto kern = mxfp8_tile_kernel<OP, MODE, kTM, kStages>;
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

// tile rows of the instantiation the host will launch
inline int tile_rows(int op, int mode)
{
    switch (op * 4 + mode) {
    case kQuant * 4 + kRow: return Tuning<kQuant, kRow>::kTM;
    case kQuant * 4 + kCol: return Tuning<kQuant, kCol>::kTM;
    case kQuant * 4 + kBoth: return Tuning<kQuant, kBoth>::kTM;
    case kFwd * 4 + kRow: return Tuning<kFwd, kRow>::kTM;
    case kFwd * 4 + kCol: return Tuning<kFwd, kCol>::kTM;
    case kFwd * 4 + kBoth: return Tuning<kFwd, kBoth>::kTM;
    case kBwd * 4 + kRow: return Tuning<kBwd, kRow>::kTM;
    case kBwd * 4 + kCol: return Tuning<kBwd, kCol>::kTM;
    default: return Tuning<kBwd, kBoth>::kTM;
    }
}

// per-op dispatch over the scale mode (one translation unit per op)
cudaError_t launch_quant(int mode, const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,
                         cudaStream_t stream, int device);
cudaError_t launch_fwd(int mode, const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,
                       cudaStream_t stream, int device);
cudaError_t launch_bwd(int mode, const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,
                       cudaStream_t stream, int device);

#define MX_DEFINE_LAUNCH(NAME, OP)                                                               \
    cudaError_t NAME(int mode, const CUtensorMap (&maps)[3], const KernelArgs &a, int grid,      \
                     cudaStream_t stream, int device)                                            \
    {                                                                                            \
        switch (mode) {                                                                          \
        case kRow: return launch_tiles<OP, kRow>(maps, a, grid, stream, device);                 \
        case kCol: return launch_tiles<OP, kCol>(maps, a, grid, stream, device);                 \
        case kBoth: return launch_tiles<OP, kBoth>(maps, a, grid, stream, device);               \
        default: return cudaErrorInvalidValue;                                                   \
        }                                                                                        \
    }

}  // namespace mx
