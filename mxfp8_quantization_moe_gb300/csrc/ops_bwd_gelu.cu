// ops_bwd_gelu.cu -- instantiations of the tile kernel for the bwd op with the GEGLU
// activation
// (rowwise, colwise and both scale modes; plain or blocked scales).
#include "launch.cuh"

namespace mx {
MX_DEFINE_LAUNCH(launch_bwd_gelu, kBwd, kGelu, false)
}  // namespace mx
