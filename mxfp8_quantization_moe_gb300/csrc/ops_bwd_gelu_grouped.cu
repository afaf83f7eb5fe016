// ops_bwd_gelu_grouped.cu -- instantiations of the tile kernel for the bwd op with the GEGLU
// activation
// (rowwise, colwise and both scale modes) with per-group blocked scales.
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_bwd_gelu_grouped, kBwd, kGelu, true)
}  // namespace mx
