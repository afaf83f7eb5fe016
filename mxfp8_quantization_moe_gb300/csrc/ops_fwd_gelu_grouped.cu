// ops_fwd_gelu_grouped.cu -- instantiations of the tile kernel for the fwd op with the GEGLU
// activation
// (rowwise, colwise and both scale modes) with per-group blocked scales.
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_fwd_gelu_grouped, kFwd, kGelu, true)
}  // namespace mx
