// ops_bwd_grouped.cu -- instantiations of the tile kernel for the bwd op
// (rowwise, colwise and both scale modes) with per-group blocked scales.
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_bwd_grouped, kBwd, kSilu, true)
}  // namespace mx
