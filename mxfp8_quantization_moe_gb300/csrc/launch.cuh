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
    constexpr int kStages = Tuning<OP>::kStages;
    constexpr size_t kSmem = smem_bytes<OP, kStages>();
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    auto kern = mxfp8_tile_kernel<OP, MODE, kStages>;
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
                            dim3((kWarps + 1) * 32), args, kSmem, stream);
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
